"""Host-side tests of the C ABI (no GPU): the library builds for sm_103a, loads, exports every
function include/twell.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from activation_sparse_ffn_gate_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "twell.h")).read()
    return sorted(set(re.findall(r"TWELL_API\s+[\w\s\*]+?\b(twell_\w+)\s*\(", src)))


def test_header_declarations_are_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.EXPORTS)


def test_built_for_sm103a_only():
    out = os.popen(f"cuobjdump --list-elf {binding.LIB_PATH} 2>/dev/null").read()
    if not out:
        pytest.skip("cuobjdump not available")
    archs = set(re.findall(r"sm_(\d+a?)", out))
    assert archs == {"103a"}, archs


def test_status_strings(lib):
    for code in range(8):
        assert lib.twell_status_string(code)
    assert lib.twell_status_string(99) == b"unknown status"


def test_sizes(lib):
    assert lib.twell_packed_vals_bytes(8192, 5632, 128, binding.TWELL_BF16) == 8192 * 44 * 128 * 2
    assert lib.twell_packed_vals_bytes(10, 300, 256, binding.TWELL_F32) == 10 * 2 * 256 * 4
    assert lib.twell_packed_idx_bytes(10, 300, 64) == 10 * 5 * 64
    assert lib.twell_packed_cnt_bytes(10, 300, 64) == 10 * 5 * 2
    assert lib.twell_packed_vals_bytes(10, 0, 64, 0) == 0
    assert lib.twell_packed_vals_bytes(-1, 10, 64, 0) == 0


def _packed(N=4, f=256, T=128, dtype=0, ptr=4096):
    return binding._Packed(N, f, T, T, dtype, ptr, ptr, ptr)


ALIGNED = ctypes.c_void_p(1 << 20)
STATUS = ctypes.c_void_p(1 << 21)


def test_gate_pack_rejects_bad_arguments(lib):
    p = _packed()
    call = lambda **kw: lib.twell_gate_pack(  # noqa: E731
        kw.get("x", ALIGNED), kw.get("w", ALIGNED), kw.get("N", 4), kw.get("d", 64), kw.get("f", 256),
        kw.get("T", 128), kw.get("dt", 0), ctypes.byref(kw.get("p", p)), None, 0, kw.get("st", STATUS), None)
    assert call(x=None) == 1
    assert call(w=None) == 1
    assert call(st=None) == 1
    assert call(d=60) == 1  # d not a multiple of 8
    assert call(N=-1) == 1
    assert call(f=0) == 1
    assert call(x=ctypes.c_void_p((1 << 20) + 2)) == 1  # misaligned
    assert call(T=100, p=_packed(T=100)) == 2  # unsupported tile width
    assert call(p=_packed(f=255)) == 1  # descriptor shape mismatch
    assert call(dt=7) == 2
    assert call(dt=1) == 1  # fp32 inputs with bf16 packed values
    bad = _packed()
    bad.cap = 64
    assert call(p=bad) == 1
    null_vals = _packed()
    null_vals.vals = None
    assert call(p=null_vals) == 1


def test_fused_rejects_bad_arguments(lib):
    p = _packed()
    need = lib.twell_workspace_bytes(1, 4, 64, 256, 128, 0, 0)  # TWELL_OP_FFN_FUSED_FWD
    call = lambda **kw: lib.twell_ffn_fused_fwd(  # noqa: E731
        ALIGNED, ALIGNED, ALIGNED, ctypes.byref(kw.get("p", p)), kw.get("N", 4), kw.get("d", 64),
        kw.get("f", 256), kw.get("dt", 0), kw.get("y", ALIGNED), kw.get("ws", ALIGNED), kw.get("ws_bytes", need),
        STATUS, None)
    assert call(y=None) == 1
    assert call(ws=None) == 7  # TWELL_ERR_WORKSPACE: the work counter is required
    assert call(ws_bytes=need - 1) == 7
    assert call(N=0, p=_packed(N=0), ws=None, ws_bytes=0) == 0  # an empty batch needs no workspace
    assert call(N=5) == 1
    assert call(d=12) == 1
    assert call(y=ctypes.c_void_p((1 << 20) + 8)) == 1
    assert call(dt=1) == 1  # fp32 inputs need fp32 packed values
    assert call(dt=5) == 2


def test_compaction_calls_reject_bad_arguments(lib):
    p = _packed()
    assert lib.twell_column_activity(ctypes.byref(p), None, STATUS, None) == 1
    assert lib.twell_column_activity(ctypes.byref(p), ALIGNED, None, None) == 1
    bad = _packed()
    bad.cap = 64
    assert lib.twell_column_activity(ctypes.byref(bad), ALIGNED, STATUS, None) == 1
    rows = ALIGNED
    assert lib.twell_gather_rows(ALIGNED, 10, rows, 4, 4, 0, ALIGNED, STATUS, None) == 1  # 8-byte rows
    assert lib.twell_gather_rows(ALIGNED, 10, rows, 4, 8, 0, ctypes.c_void_p((1 << 20) + 8), STATUS, None) == 1
    assert lib.twell_gather_rows(None, 10, rows, 4, 8, 0, ALIGNED, STATUS, None) == 1
    assert lib.twell_gather_rows(ALIGNED, 10, rows, 4, 8, 7, ALIGNED, STATUS, None) == 2
    assert lib.twell_gather_rows(None, 10, None, 0, 8, 0, None, STATUS, None) == 0  # nothing to gather


def test_pack_unpack_reject_bad_arguments(lib):
    p = _packed()
    assert lib.twell_pack_from_gate(None, 4, 256, 128, 0, ctypes.byref(p), STATUS, None) == 1
    assert lib.twell_pack_from_gate(ALIGNED, 4, 256, 64, 0, ctypes.byref(p), STATUS, None) == 1
    assert lib.twell_unpack(ctypes.byref(p), None, STATUS, None) == 1
    assert lib.twell_gate_gemm(ALIGNED, ALIGNED, 4, 64, 250, ALIGNED, STATUS, None) == 1  # f % 4


def test_read_status_rejects_null(lib):
    assert lib.twell_read_status(None, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        binding._lib_backup = binding._lib
        try:
            binding._lib = None
            binding.load(str(tmp_path / "missing.so"))
        finally:
            binding._lib = binding._lib_backup


def test_fused_workspace_grows_with_rows_and_width(lib):
    """The fused walk's workspace holds a 256-byte header, three row lists of N entries and, for
    split rows, item records and fp32 partial rows of width d; its size depends on N, d and f."""
    ws = lambda N, d, f=5632: lib.twell_workspace_bytes(1, N, d, f, 128, 0, 0)  # noqa: E731
    item = lambda d: 32 + 4 * d  # noqa: E731  (item record, split-row record, partial row)
    assert ws(1, 64) > 256
    assert ws(8192, 2048) > ws(4096, 2048) > ws(64, 2048)
    assert ws(8192, 2560) > ws(8192, 2048)
    # item slots: N/8 within [4096, 16384], at most N * ceil(f / 4) (items of at least 4 nonzeros), at least 64
    assert ws(8192, 2048) >= 4096 * item(2048) + 3 * 8192 * 4
    assert ws(1, 2048, 64) < 64 * item(2048) + 4096  # at least 64 slots
    assert ws(1 << 20, 1024) < ws(1 << 20, 2048) < 16384 * item(2048) + 3 * (1 << 20) * 4 + 4096
    assert ws(1 << 20, 2048) >= 16384 * item(2048)
    assert all(ws(N, 1024) % 256 == 0 for N in (1, 7, 100, 8192))


def test_union_rejects_bad_arguments(lib):
    p = _packed()
    need = lib.twell_workspace_bytes(5, 4, 64, 256, 128, 0, 0)  # TWELL_OP_FFN_UNION_FWD
    assert need >= 4 * 256 * 2 + 4 * 256 // 8  # H [N, f_pad] fp16 and the keep masks [N, f_pad / 32] words
    call = lambda **kw: lib.twell_ffn_union_fwd(  # noqa: E731
        ALIGNED, ALIGNED, ALIGNED, ctypes.byref(kw.get("p", p)), kw.get("N", 4), kw.get("d", 64),
        kw.get("f", 256), kw.get("dt", 0), kw.get("y", ALIGNED), kw.get("ws", ALIGNED), kw.get("ws_bytes", need),
        STATUS, None)
    assert call(y=None) == 1
    assert call(ws=None) == 7
    assert call(ws_bytes=need - 1) == 7
    assert call(dt=1) == 2  # bf16 only
    assert call(d=12) == 1
    assert call(N=5) == 1  # the TwELL describes 4 rows
    assert call(N=0, p=_packed(N=0), ws=None, ws_bytes=0) == 0
    assert call(y=ctypes.c_void_p((1 << 20) + 8)) == 1


def test_gate_union_rejects_bad_arguments(lib):
    p = _packed()
    need = lib.twell_workspace_bytes(8, 4, 64, 256, 128, 0, 0)  # TWELL_OP_FFN_GATE_UNION_FWD
    assert need >= 4 * 256 * 2  # H [N, f_pad] fp16
    assert lib.twell_workspace_bytes(8, 3, 64, 1000, 128, 0, 0) >= 3 * 1024 * 2  # f_pad = 1024
    # up to 512 tokens the down product adds its split partials on chip: H alone; from 513 tokens the
    # SM-pair down GEMM's fp32 partials (up to 2048 rows of d_model) come on top
    h = lambda N: (N * 5632 * 2 + 255) // 256 * 256  # noqa: E731
    assert lib.twell_workspace_bytes(8, 512, 2048, 5632, 128, 0, 0) == h(512)
    assert lib.twell_workspace_bytes(8, 513, 2048, 5632, 128, 0, 0) >= h(513) + 2048 * 2048 * 4
    assert lib.twell_workspace_bytes(5, 512, 2048, 5632, 128, 0, 0) < lib.twell_workspace_bytes(5, 513, 2048, 5632, 128, 0, 0)
    call = lambda **kw: lib.twell_ffn_gate_union_fwd(  # noqa: E731
        ALIGNED, kw.get("wg", ALIGNED), ALIGNED, kw.get("wd", ALIGNED), kw.get("N", 4), kw.get("d", 64),
        kw.get("f", 256), kw.get("T", 128), kw.get("dt", 0), ctypes.byref(kw.get("p", p)), kw.get("y", ALIGNED),
        kw.get("ws", ALIGNED), kw.get("ws_bytes", need), STATUS, None)
    assert call(wg=None) == 1
    assert call(wd=None) == 1
    assert call(y=None) == 1
    assert call(ws=None) == 7
    assert call(ws_bytes=need - 1) == 7
    assert call(dt=1) == 2  # bf16 only
    assert call(T=256, p=_packed(T=256)) == 2  # the tile holds 128 units: T = 64 or 128
    assert call(T=64) == 1  # the TwELL's tile is 128
    assert call(d=12) == 1
    assert call(f=252, p=_packed(f=252)) == 1  # f a multiple of 8
    assert call(N=5) == 1  # the TwELL describes 4 rows
    assert call(N=0, p=_packed(N=0), ws=None, ws_bytes=0) == 0
    assert call(y=ctypes.c_void_p((1 << 20) + 8)) == 1


def test_fused_f16down_rejects_bad_arguments(lib):
    p = _packed()
    need = lib.twell_workspace_bytes(1, 4, 512, 256, 128, 0, 0)  # TWELL_OP_FFN_FUSED_FWD
    call = lambda **kw: lib.twell_ffn_fused_fwd_f16down(  # noqa: E731
        ALIGNED, ALIGNED, kw.get("wd", ALIGNED), ctypes.byref(kw.get("p", p)), kw.get("N", 4), kw.get("d", 512),
        kw.get("f", 256), kw.get("y", ALIGNED), kw.get("ws", ALIGNED), kw.get("ws_bytes", need), STATUS, None)
    assert call(wd=None) == 1
    assert call(y=None) == 1
    assert call(ws=None) == 7
    assert call(ws_bytes=need - 1) == 7
    assert call(d=640) == 2  # a multiple of 256 in [512, 3072] only
    assert call(d=256) == 2
    assert call(d=3328) == 2
    assert call(d=12) == 1
    assert call(N=5) == 1  # the TwELL describes 4 rows
    assert call(N=0, p=_packed(N=0), ws=None, ws_bytes=0) == 0
    assert call(y=ctypes.c_void_p((1 << 20) + 8)) == 1


def test_decode_rejects_bad_arguments(lib):
    p = _packed()
    need = lib.twell_workspace_bytes(6, 4, 512, 256, 128, 0, 0)  # TWELL_OP_FFN_DECODE
    assert need >= 4 * 4 * 512 * 4  # a partial row per (CTA, token): 2 * ceil(256 / 128) CTAs
    assert lib.twell_workspace_bytes(6, 4, 512, 256, 0, 0, 0) == 0  # the tile width sizes it
    call = lambda **kw: lib.twell_ffn_decode(  # noqa: E731
        ALIGNED, ALIGNED, kw.get("wu", ALIGNED), ALIGNED, kw.get("N", 4), kw.get("d", 512), kw.get("f", 256),
        kw.get("T", 128), ctypes.byref(kw.get("p", p)), kw.get("y", ALIGNED), kw.get("ws", ALIGNED),
        kw.get("ws_bytes", need), STATUS, None)
    assert call(wu=None) == 1
    assert call(y=None) == 1
    assert call(ws=None) == 7
    assert call(ws_bytes=need - 1) == 7
    assert call(N=17, p=_packed(N=17)) == 2  # at most 16 tokens
    assert call(d=72) == 2  # d_model a multiple of 64
    assert call(d=4160) == 2  # at most 4096
    assert call(d=100) == 1
    assert call(T=32, p=_packed(T=32)) == 2
    assert call(N=5) == 1  # the TwELL describes 4 rows
    assert call(T=64) == 1  # the TwELL's tile is 128
    assert call(N=0, p=_packed(N=0), ws=None, ws_bytes=0) == 0
    assert call(y=ctypes.c_void_p((1 << 20) + 8)) == 1


def test_convert_f16_rejects_bad_arguments(lib):
    assert lib.twell_convert_f16(ALIGNED, ALIGNED, -1, STATUS, None) == 1
    assert lib.twell_convert_f16(ALIGNED, ALIGNED, 16, None, None) == 1
    assert lib.twell_convert_f16(None, ALIGNED, 16, STATUS, None) == 1
    assert lib.twell_convert_f16(ALIGNED, None, 16, STATUS, None) == 1
    assert lib.twell_convert_f16(None, None, 0, STATUS, None) == 0


def test_wait_probe_rejects_bad_limits(lib):
    assert lib.twell_wait_probe(0, 0, STATUS, None) == 1
    assert lib.twell_wait_probe(0, 10001, STATUS, None) == 1
    assert lib.twell_wait_probe(1, 50, None, None) == 1
