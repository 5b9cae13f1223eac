"""Thin ctypes binding over libtwell_gb300.so (the C ABI declared in include/twell.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels. PyTorch
provides device memory and the current CUDA stream. The functions carry the C names; each
allocates its outputs with torch when they are not given, passes raw device pointers and the
current stream, and raises TwellError on a non-OK status. There is no fallback: without the
built library every call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtwell_gb300.so")

TWELL_OK = 0
TWELL_ERR_UNSUPPORTED = 2
TWELL_BF16 = 0
TWELL_F32 = 1
(OP_GATE_PACK, OP_FFN_FUSED_FWD, OP_HYBRID_FWD, OP_HYBRID_BWD, OP_HYBRID_ROUTE, OP_FFN_UNION_FWD, OP_FFN_DECODE,
 OP_FFN_TILE_UNION_FWD, OP_FFN_GATE_UNION_FWD) = range(9)
DECODE_MAX_N = 16  # twell_ffn_decode takes batches of at most this many tokens
STATUS_NAMES = {0: "TWELL_OK", 1: "TWELL_ERR_INVALID", 2: "TWELL_ERR_UNSUPPORTED", 3: "TWELL_ERR_BACKUP_FULL",
                4: "TWELL_ERR_TIMEOUT", 5: "TWELL_ERR_DEVICE_CHECK", 6: "TWELL_ERR_CUDA",
                7: "TWELL_ERR_WORKSPACE"}

# Every function the header declares; the CPU tests check that the library exports each one.
EXPORTS = ("twell_packed_vals_bytes", "twell_packed_idx_bytes", "twell_packed_cnt_bytes", "twell_workspace_bytes",
           "twell_gate_pack", "twell_ffn_fused_fwd", "twell_ffn_union_fwd", "twell_hybrid_fwd", "twell_hybrid_bwd", "twell_unpack",
           "twell_pack_from_gate", "twell_hybrid_route_from_gate", "twell_hybrid_route_noalloc",
           "twell_gate_gemm", "twell_gemm_test", "twell_column_activity", "twell_gather_rows",
           "twell_read_status", "twell_status_string", "twell_device_info", "twell_wait_probe",
           "twell_ffn_fused_fwd_f16down", "twell_convert_f16", "twell_ffn_decode", "twell_ffn_tile_union_fwd",
           "twell_count_nonzeros", "twell_convert_f16_transposed", "twell_ffn_gate_union_fwd")


class TwellError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_status_string(code)})")


class _Packed(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("n_cols", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("cap", ctypes.c_int32), ("dtype", ctypes.c_int), ("vals", ctypes.c_void_p),
                ("idx", ctypes.c_void_p), ("cnt", ctypes.c_void_p)]


class _Hybrid(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("n_cols", ctypes.c_int32), ("K", ctypes.c_int32),
                ("backup_cap", ctypes.c_int32), ("dtype", ctypes.c_int), ("a", ctypes.c_void_p),
                ("u", ctypes.c_void_p), ("col", ctypes.c_void_p), ("cnt", ctypes.c_void_p),
                ("backup_rows", ctypes.c_void_p), ("n_backup", ctypes.c_void_p), ("A_b", ctypes.c_void_p),
                ("U_b", ctypes.c_void_p), ("l1", ctypes.c_void_p), ("dev_status", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with activation_sparse_ffn_gate_gb300.build.build()")
            lib = ctypes.CDLL(path)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            st = ctypes.c_int
            sig = {
                "twell_packed_vals_bytes": (sz, [i32, i32, i32, ctypes.c_int]),
                "twell_packed_idx_bytes": (sz, [i32, i32, i32]),
                "twell_packed_cnt_bytes": (sz, [i32, i32, i32]),
                "twell_workspace_bytes": (sz, [ctypes.c_int, i32, i32, i32, i32, i32, i32]),
                "twell_gate_pack": (st, [vp, vp, i32, i32, i32, i32, ctypes.c_int, ctypes.POINTER(_Packed), vp, sz,
                                         vp, vp]),
                "twell_ffn_fused_fwd": (st, [vp, vp, vp, ctypes.POINTER(_Packed), i32, i32, i32, ctypes.c_int, vp, vp,
                                             sz, vp, vp]),
                "twell_ffn_union_fwd": (st, [vp, vp, vp, ctypes.POINTER(_Packed), i32, i32, i32, ctypes.c_int, vp, vp,
                                             sz, vp, vp]),
                "twell_ffn_gate_union_fwd": (st, [vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                                  ctypes.POINTER(_Packed), vp, vp, sz, vp, vp]),
                "twell_ffn_tile_union_fwd": (st, [vp, vp, vp, ctypes.POINTER(_Packed), i32, i32, i32, vp, vp, sz,
                                                  vp, vp]),
                "twell_wait_probe": (st, [i32, i32, vp, vp]),
                "twell_ffn_fused_fwd_f16down": (st, [vp, vp, vp, ctypes.POINTER(_Packed), i32, i32, i32, vp, vp, sz,
                                                     vp, vp]),
                "twell_convert_f16": (st, [vp, vp, ctypes.c_int64, vp, vp]),
                "twell_convert_f16_transposed": (st, [vp, vp, i32, i32, vp, vp]),
                "twell_ffn_decode": (st, [vp, vp, vp, vp, i32, i32, i32, i32, ctypes.POINTER(_Packed), vp, vp, sz,
                                          vp, vp]),
                "twell_hybrid_fwd": (st, [vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                          ctypes.POINTER(_Hybrid), vp, vp, sz, vp]),
                "twell_hybrid_bwd": (st, [vp, vp, vp, vp, ctypes.POINTER(_Hybrid), vp, i32, i32, i32, ctypes.c_float,
                                          vp, vp, vp, vp, vp, sz, vp]),
                "twell_unpack": (st, [ctypes.POINTER(_Packed), vp, vp, vp]),
                "twell_pack_from_gate": (st, [vp, i32, i32, i32, ctypes.c_int, ctypes.POINTER(_Packed), vp, vp]),
                "twell_hybrid_route_from_gate": (st, [vp, i32, i32, i32, ctypes.c_int, ctypes.POINTER(_Hybrid), vp,
                                                      sz, vp]),
                "twell_hybrid_route_noalloc": (st, [ctypes.POINTER(_Packed), i32, ctypes.POINTER(_Hybrid), vp]),
                "twell_gate_gemm": (st, [vp, vp, i32, i32, i32, vp, vp, vp]),
                "twell_column_activity": (st, [ctypes.POINTER(_Packed), vp, vp, vp]),
                "twell_count_nonzeros": (st, [ctypes.POINTER(_Packed), vp, vp, vp]),
                "twell_gather_rows": (st, [vp, i32, vp, i32, i32, ctypes.c_int, vp, vp, vp]),
                "twell_gemm_test": (st, [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
                "twell_read_status": (st, [vp, vp]),
                "twell_status_string": (ctypes.c_char_p, [ctypes.c_int]),
                "twell_device_info": (st, [ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _status_string(code: int) -> str:
    try:
        return load().twell_status_string(code).decode()
    except Exception:  # the library itself failed to load
        return "?"


def _check(code: int, where: str):
    if code != TWELL_OK:
        raise TwellError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return TWELL_BF16
    if dt == torch.float32:
        return TWELL_F32
    raise TypeError(f"unsupported element type {dt}")


_status_bufs = {}


def status_buffer(device=None) -> torch.Tensor:
    """The per-device int32 status word the binding passes as dev_status."""
    dev = torch.device(device if device is not None else torch.cuda.current_device())
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    buf = _status_bufs.get(dev.index)
    if buf is None:
        buf = torch.zeros(1, dtype=torch.int32, device=dev)
        _status_bufs[dev.index] = buf
    return buf


_fused_ws = {}


def fused_workspace(N: int, d: int, f: int, device=None, stream=None) -> torch.Tensor:
    """The workspace twell_ffn_fused_fwd needs for N rows, d_model d, d_ff f (work counter, split
    plan and the partial rows of split rows), one per device and stream, grown on demand: calls on
    one stream run one after the other, so they can share it."""
    dev = torch.device(device if device is not None else torch.cuda.current_device())
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    key = (dev.index, _stream(stream).value or 0)
    n = int(load().twell_workspace_bytes(OP_FFN_FUSED_FWD, N, d, f, 8, 0, 0))
    buf = _fused_ws.get(key)
    if buf is None or buf.numel() < n:
        buf = torch.empty(n, dtype=torch.uint8, device=dev)
        _fused_ws[key] = buf
    return buf


def twell_read_status(status: Optional[torch.Tensor] = None, stream=None, reset: bool = True) -> int:
    """Synchronise the stream and return the device status code (optionally clearing it)."""
    status = status if status is not None else status_buffer()
    code = load().twell_read_status(_ptr(status), _stream(stream))
    if reset and code != TWELL_OK:
        status.zero_()
    return code


def twell_wait_probe(arrive: bool, limit_ms: int, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Run the library's bounded mbarrier wait on its own (test export): with arrive=False it runs
    out after limit_ms and records TWELL_ERR_TIMEOUT in the status word."""
    _check(load().twell_wait_probe(1 if arrive else 0, int(limit_ms), _ptr(status if status is not None else
                                                                             status_buffer()), _stream(stream)),
           "twell_wait_probe")


def check_device_status(where: str = "device", status: Optional[torch.Tensor] = None, stream=None):
    _check(twell_read_status(status, stream), where)


# ------------------------------------------------------------------------------------------ TwELL

@dataclasses.dataclass
class TwELL:
    """A TwELL matrix in device memory (see twell_packed in include/twell.h)."""

    n_rows: int
    n_cols: int
    tile: int
    vals: torch.Tensor  # [n_rows, nt, tile] element type
    idx: torch.Tensor  # [n_rows, nt, tile] uint8
    cnt: torch.Tensor  # [n_rows, nt] int16 storage of uint16 counts

    @property
    def nt(self) -> int:
        return -(-self.n_cols // self.tile)

    @property
    def dtype(self) -> torch.dtype:
        return self.vals.dtype

    @staticmethod
    def empty(n_rows, n_cols, tile, dtype=torch.bfloat16, device=None):
        nt = -(-n_cols // tile)
        device = device or torch.device("cuda", torch.cuda.current_device())
        return TwELL(n_rows, n_cols, tile,
                     torch.empty((n_rows, nt, tile), dtype=dtype, device=device),
                     torch.empty((n_rows, nt, tile), dtype=torch.uint8, device=device),
                     torch.empty((n_rows, nt), dtype=torch.int16, device=device))

    def counts(self) -> torch.Tensor:
        """Counts as non-negative integers (int32)."""
        return self.cnt.to(torch.int32) & 0xFFFF

    def c_struct(self) -> _Packed:
        return _Packed(self.n_rows, self.n_cols, self.tile, self.tile, _dtype_code(self.vals.dtype),
                       self.vals.data_ptr(), self.idx.data_ptr(), self.cnt.data_ptr())


def twell_gate_pack(x: torch.Tensor, Wg_s: torch.Tensor, T: int = 128, out: Optional[TwELL] = None,
                    status: Optional[torch.Tensor] = None, stream=None,
                    vals_dtype: torch.dtype = torch.float32) -> TwELL:
    """Gate GEMM with the ReLU + TwELL pack epilogue: returns the TwELL of ReLU(x Wg_s^T).

    The packed values keep the fp32 accumulator by default (vals_dtype=torch.bfloat16 rounds them)."""
    N, d = x.shape
    f = Wg_s.shape[0]
    out = out if out is not None else TwELL.empty(N, f, T, vals_dtype, x.device)
    s = out.c_struct()
    _check(load().twell_gate_pack(_ptr(x), _ptr(Wg_s), N, d, f, T, _dtype_code(x.dtype), ctypes.byref(s), None, 0,
                                  _ptr(status if status is not None else status_buffer(x.device)), _stream(stream)),
           "twell_gate_pack")
    return out


def twell_ffn_fused_fwd(x: torch.Tensor, Wu_s: torch.Tensor, Wd_s: torch.Tensor, a: TwELL,
                        y: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        stream=None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Fused up+down projection over the packed nonzeros: y = (a * (x Wu_s^T)) Wd_s."""
    N, d = x.shape
    f = Wu_s.shape[0]
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    ws = ws if ws is not None else fused_workspace(N, d, f, x.device, stream)
    s = a.c_struct()
    _check(load().twell_ffn_fused_fwd(_ptr(x), _ptr(Wu_s), _ptr(Wd_s), ctypes.byref(s), N, d, f,
                                      _dtype_code(x.dtype), _ptr(y), _ptr(ws), ws.numel(),
                                      _ptr(status if status is not None else status_buffer(x.device)),
                                      _stream(stream)),
           "twell_ffn_fused_fwd")
    return y


def twell_convert_f16(src: torch.Tensor, out: Optional[torch.Tensor] = None, status=None,
                      stream=None) -> torch.Tensor:
    """A bf16 tensor converted to fp16 by the library (e.g. Wd_s for twell_ffn_fused_fwd_f16down)."""
    if src.dtype != torch.bfloat16 or not src.is_contiguous():
        raise ValueError("src must be a contiguous bf16 tensor")
    out = out if out is not None else torch.empty(src.shape, dtype=torch.float16, device=src.device)
    _check(load().twell_convert_f16(_ptr(src), _ptr(out), src.numel(),
                                    _ptr(status if status is not None else status_buffer(src.device)),
                                    _stream(stream)),
           "twell_convert_f16")
    return out


def twell_convert_f16_transposed(src: torch.Tensor, out: Optional[torch.Tensor] = None, status=None,
                                 stream=None) -> torch.Tensor:
    """The transpose of a 2-D bf16 tensor converted to fp16 by the library (e.g. Wd_s [f, d] -> Wd16t_s
    [d, f] for twell_ffn_union_fwd)."""
    if src.dtype != torch.bfloat16 or src.dim() != 2 or not src.is_contiguous():
        raise ValueError("src must be a contiguous 2-D bf16 tensor")
    rows, cols = src.shape
    out = out if out is not None else torch.empty((cols, rows), dtype=torch.float16, device=src.device)
    _check(load().twell_convert_f16_transposed(_ptr(src), _ptr(out), rows, cols,
                                               _ptr(status if status is not None else status_buffer(src.device)),
                                               _stream(stream)),
           "twell_convert_f16_transposed")
    return out


def twell_ffn_fused_fwd_f16down(x: torch.Tensor, Wu_s: torch.Tensor, Wd16_s: torch.Tensor, a: TwELL,
                                y: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                stream=None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """twell_ffn_fused_fwd with Wd_s given in fp16 (twell_convert_f16) and the down projection in fp16."""
    if Wd16_s.dtype != torch.float16:
        raise ValueError("Wd16_s must be fp16")
    N, d = x.shape
    f = Wu_s.shape[0]
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    ws = ws if ws is not None else fused_workspace(N, d, f, x.device, stream)
    s = a.c_struct()
    _check(load().twell_ffn_fused_fwd_f16down(_ptr(x), _ptr(Wu_s), _ptr(Wd16_s), ctypes.byref(s), N, d, f,
                                              _ptr(y), _ptr(ws), ws.numel(),
                                              _ptr(status if status is not None else status_buffer(x.device)),
                                              _stream(stream)),
           "twell_ffn_fused_fwd_f16down")
    return y


class StreamedFFN:
    """The sparse inference FFN over a sequence of batches held in pinned host memory, with each
    batch's copy to the device and its result's copy back overlapped with the neighbouring batches'
    compute: host-to-device copies on one stream, gate + walk (or union path) on a second,
    device-to-host copies on a third, ordered by events, with two device buffers of x and of y
    used in turn. A serving loop so keeps the copy engines and the SMs busy at the same time; the
    kernels and their results are those of ffn_forward."""

    def __init__(self, Wg_s: torch.Tensor, Wu_s: torch.Tensor, Wd_s: torch.Tensor, N: int, T: int = 128,
                 path: str = "walk", vals_dtype: torch.dtype = torch.float32, status: Optional[torch.Tensor] = None,
                 Wd16_s: Optional[torch.Tensor] = None, Wd16t_s: Optional[torch.Tensor] = None):
        dev = Wg_s.device
        f, d = Wg_s.shape
        self.W, self.T, self.path, self.status, self.N, self.d = (Wg_s, Wu_s, Wd_s), T, path, status, N, d
        self.Wd16, self.Wd16t = Wd16_s, Wd16t_s
        self.copy_in, self.compute, self.copy_out = (torch.cuda.Stream(dev) for _ in range(3))
        self.x = [torch.empty((N, d), dtype=Wg_s.dtype, device=dev) for _ in range(2)]
        self.y = [torch.empty((N, d), dtype=Wg_s.dtype, device=dev) for _ in range(2)]
        self.packed = TwELL.empty(N, f, T, vals_dtype, dev)
        self.x_in = [torch.cuda.Event() for _ in range(2)]    # x[b] holds the batch
        self.done = [torch.cuda.Event() for _ in range(2)]    # x[b] read, y[b] written
        self.y_out = [torch.cuda.Event() for _ in range(2)]   # y[b] copied to the host
        self.count = 0

    def submit(self, x_host: torch.Tensor, y_host: torch.Tensor):
        """Queue one batch: x_host [N, d] pinned input, y_host a pinned output of the same shape (valid
        once the copy-out stream has passed it, e.g. after torch.cuda.synchronize())."""
        if tuple(x_host.shape) != (self.N, self.d) or tuple(y_host.shape) != (self.N, self.d):
            raise ValueError("batch shape differs from the pipeline's")
        b, later = self.count % 2, self.count >= 2
        with torch.cuda.stream(self.copy_in):
            if later:
                self.copy_in.wait_event(self.done[b])  # batch count-2 is done reading x[b]
            self.x[b].copy_(x_host, non_blocking=True)
            self.x_in[b].record(self.copy_in)
        with torch.cuda.stream(self.compute):
            self.compute.wait_event(self.x_in[b])
            if later:
                self.compute.wait_event(self.y_out[b])  # y[b] of batch count-2 is on the host
            ffn_forward(self.x[b], *self.W, T=self.T, packed=self.packed, y=self.y[b], status=self.status,
                        stream=self.compute, path=self.path, Wd16_s=self.Wd16, Wd16t_s=self.Wd16t)
            self.done[b].record(self.compute)
        with torch.cuda.stream(self.copy_out):
            self.copy_out.wait_event(self.done[b])
            y_host.copy_(self.y[b], non_blocking=True)
            self.y_out[b].record(self.copy_out)
        self.count += 1


_union_ws = {}


def twell_ffn_union_fwd(x: torch.Tensor, Wu_s: torch.Tensor, Wd16t_s: torch.Tensor, a: TwELL,
                        y: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        stream=None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The same y as twell_ffn_fused_fwd, as two tensor-core GEMMs over all of d_ff (for dense layers);
    Wd16t_s [d, f] is Wd_s transposed and converted by twell_convert_f16_transposed."""
    N, d = x.shape
    f = Wu_s.shape[0]
    if Wd16t_s.dtype != torch.float16 or tuple(Wd16t_s.shape) != (d, f) or not Wd16t_s.is_contiguous():
        raise ValueError("Wd16t_s must be a contiguous fp16 [d_model, d_ff] tensor "
                         "(twell_convert_f16_transposed of Wd_s)")
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    if ws is None:
        n = twell_workspace_bytes(OP_FFN_UNION_FWD, N, d, f)
        key = (x.device.index, _stream(stream).value or 0)
        ws = _union_ws.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.empty(n, dtype=torch.uint8, device=x.device)
            _union_ws[key] = ws
    s = a.c_struct()
    _check(load().twell_ffn_union_fwd(_ptr(x), _ptr(Wu_s), _ptr(Wd16t_s), ctypes.byref(s), N, d, f,
                                      _dtype_code(x.dtype), _ptr(y), _ptr(ws), ws.numel(),
                                      _ptr(status if status is not None else status_buffer(x.device)),
                                      _stream(stream)),
           "twell_ffn_union_fwd")
    return y


def twell_ffn_gate_union_fwd(x: torch.Tensor, Wg_s: torch.Tensor, Wu_s: torch.Tensor, Wd16t_s: torch.Tensor,
                             T: int = 128, out: Optional[TwELL] = None, y: Optional[torch.Tensor] = None,
                             status: Optional[torch.Tensor] = None, stream=None, ws: Optional[torch.Tensor] = None,
                             vals_dtype: torch.dtype = torch.float32):
    """twell_gate_pack and twell_ffn_union_fwd with the gate and up projections in one tensor-core
    GEMM: returns (y, the TwELL of ReLU(x Wg_s^T)). T = 64 or 128."""
    N, d = x.shape
    f = Wu_s.shape[0]
    if Wd16t_s.dtype != torch.float16 or tuple(Wd16t_s.shape) != (d, f) or not Wd16t_s.is_contiguous():
        raise ValueError("Wd16t_s must be a contiguous fp16 [d_model, d_ff] tensor "
                         "(twell_convert_f16_transposed of Wd_s)")
    out = out if out is not None else TwELL.empty(N, f, T, vals_dtype, x.device)
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    if ws is None:
        n = twell_workspace_bytes(OP_FFN_GATE_UNION_FWD, N, d, f)
        key = (x.device.index, _stream(stream).value or 0)
        ws = _union_ws.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
            _union_ws[key] = ws
    s = out.c_struct()
    _check(load().twell_ffn_gate_union_fwd(_ptr(x), _ptr(Wg_s), _ptr(Wu_s), _ptr(Wd16t_s), N, d, f, T,
                                           _dtype_code(x.dtype), ctypes.byref(s), _ptr(y), _ptr(ws), ws.numel(),
                                           _ptr(status if status is not None else status_buffer(x.device)),
                                           _stream(stream)),
           "twell_ffn_gate_union_fwd")
    return y, out


_tile_union_ws = {}


def twell_ffn_tile_union_fwd(x: torch.Tensor, Wu_s: torch.Tensor, Wd16_s: torch.Tensor, a: TwELL,
                             y: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                             stream=None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The same y as twell_ffn_fused_fwd, as tensor-core GEMMs over each 128-token tile's union of kept
    units (gathered weight rows); Wd16_s is Wd_s converted by twell_convert_f16."""
    N, d = x.shape
    f = Wu_s.shape[0]
    if Wd16_s.dtype != torch.float16:
        raise ValueError("Wd16_s must be fp16 (twell_convert_f16 of Wd_s)")
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    if ws is None:
        n = twell_workspace_bytes(OP_FFN_TILE_UNION_FWD, N, d, f)
        key = (x.device.index, _stream(stream).value or 0)
        ws = _tile_union_ws.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.empty(n, dtype=torch.uint8, device=x.device)
            _tile_union_ws[key] = ws
    s = a.c_struct()
    _check(load().twell_ffn_tile_union_fwd(_ptr(x), _ptr(Wu_s), _ptr(Wd16_s), ctypes.byref(s), N, d, f, _ptr(y),
                                           _ptr(ws), ws.numel(),
                                           _ptr(status if status is not None else status_buffer(x.device)),
                                           _stream(stream)),
           "twell_ffn_tile_union_fwd")
    return y


_decode_ws = {}


def twell_ffn_decode(x: torch.Tensor, Wg_s: torch.Tensor, Wu_s: torch.Tensor, Wd_s: torch.Tensor, T: int = 128,
                     packed: Optional[TwELL] = None, y: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None, ws: Optional[torch.Tensor] = None,
                     vals_dtype: torch.dtype = torch.float32):
    """The whole layer for at most DECODE_MAX_N tokens in two launches; returns (y, packed TwELL)."""
    N, d = x.shape
    f = Wg_s.shape[0]
    packed = packed if packed is not None else TwELL.empty(N, f, T, vals_dtype, x.device)
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    if ws is None:
        n = twell_workspace_bytes(OP_FFN_DECODE, N, d, f, T)
        key = (x.device.index, _stream(stream).value or 0)
        ws = _decode_ws.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
            _decode_ws[key] = ws
    s = packed.c_struct()
    _check(load().twell_ffn_decode(_ptr(x), _ptr(Wg_s), _ptr(Wu_s), _ptr(Wd_s), N, d, f, T, ctypes.byref(s),
                                   _ptr(y), _ptr(ws), ws.numel(),
                                   _ptr(status if status is not None else status_buffer(x.device)),
                                   _stream(stream)),
           "twell_ffn_decode")
    return y, packed


# Density (kept fraction of d_ff per token) above which the union path beats the walk, measured with
# the whole layer on the 1.5B-like shapes (d_model 2048, d_ff 5632, 8192 tokens, T = 128, L2 flushed; ms):
#   density                               0.1%    0.5%    1%      2%      5%      10%     50%
#   walk (gate + pack, then the walk)     0.188   0.324   0.465   0.782   1.723   3.320   15.27
#   union (gate + up in one GEMM, down)   0.309   0.313   0.313   0.317   0.321   0.340   0.571
#   tile union (gate, then gathered)      0.236   0.378   0.481   0.586   0.688   0.790   1.623
#   dense cuBLAS FFN                      0.365   0.366   0.367   0.366   0.366   0.366   0.369
# The walk's time grows about linearly with the density, so the two cross near 0.45%. On the
# 1.5B-like layer (0.5% kept) the union path is also the faster of the two for every batch of 32 to
# 4096 tokens (us; dense in brackets; up to 128 tokens the union path's products run transposed):
#   tokens      32     64     128    256    512    1024   2048    4096
#   walk        37.7   38.3   46.1   51.5   65.9   89.1   121.2   185.3
#   union       26.7   28.7   32.5   36.4   48.5   65.0   90.0    165.5
#   dense      (31.7) (30.6) (32.7) (36.3) (46.5) (67.3) (111.2) (191.8)
# so batches of up to 4096 tokens switch a little lower, and smaller batches lower still; up to
# UNION_ANY_DENSITY_MAX_N tokens the union path is taken at every density. Uniform layers of those
# shapes at 0.1% / 0.25% kept:
#   64 tokens:  walk 30.8 / 33.0, union 26.8 / 27.3, dense 27.0 / 27.5
#   128 tokens: walk 33.1 / 36.7, union 31.1 / 30.8, dense 29.9 / 29.4
#   256 tokens: walk 34.0 / 43.0, union 34.4 / 34.8, dense 32.8 / 32.9  (cross near 0.1%)
#   512 tokens: walk 38.4 / 51.1, union 48.8 / 48.7, dense 45.6 / 45.3  (cross near 0.22%)
# The gathered tile-union path is never the fastest under these densities; it stays available as path
# "tile_union".
UNION_MIN_DENSITY = 0.0045
UNION_MIN_DENSITY_SMALL_BATCH = 0.004
SMALL_BATCH_MAX_N = 4096
UNION_ANY_DENSITY_MAX_N = 128
# (largest batch, density from which the union path is taken) for batches between those sizes
UNION_MIN_DENSITY_BY_BATCH = ((256, 0.001), (512, 0.002))


def choose_path(n_tokens: int, density: Optional[float]) -> str:
    """The policy of ffn_forward(path="auto"): decode for at most DECODE_MAX_N tokens; the union path
    up to UNION_ANY_DENSITY_MAX_N tokens; above that the walk below a density that grows with the
    batch (UNION_MIN_DENSITY_BY_BATCH, then UNION_MIN_DENSITY_SMALL_BATCH up to SMALL_BATCH_MAX_N
    tokens, then UNION_MIN_DENSITY) or without a density estimate, the union path (gate and up
    projection in one GEMM, down GEMM over all of d_ff) from it on."""
    if n_tokens <= DECODE_MAX_N:
        return "decode"
    if n_tokens <= UNION_ANY_DENSITY_MAX_N:
        return "union"
    limit = UNION_MIN_DENSITY_SMALL_BATCH if n_tokens <= SMALL_BATCH_MAX_N else UNION_MIN_DENSITY
    for max_n, d in UNION_MIN_DENSITY_BY_BATCH:
        if n_tokens <= max_n:
            limit = d
            break
    if density is None or density < limit:
        return "walk"
    return "union"


def ffn_forward(x, Wg_s, Wu_s, Wd_s, T: int = 128, packed: Optional[TwELL] = None, y=None, status=None, stream=None,
                vals_dtype: torch.dtype = torch.float32, path: str = "walk", Wd16_s: Optional[torch.Tensor] = None,
                density: Optional[float] = None, Wd16t_s: Optional[torch.Tensor] = None):
    """The sparse inference FFN: twell_gate_pack, then twell_ffn_fused_fwd (path "walk"),
    twell_ffn_union_fwd (path "union", with Wd16t_s = twell_convert_f16_transposed(Wd_s); for
    T = 64 or 128 as twell_ffn_gate_union_fwd, gate and up projection in one GEMM) or
    twell_ffn_tile_union_fwd (path "tile_union", with Wd16_s = twell_convert_f16(Wd_s)); path
    "decode" runs twell_ffn_decode (at most DECODE_MAX_N tokens). Path "auto" follows choose_path
    with `density`, the kept fraction of the previous batch (twell_count_nonzeros / (N * d_ff));
    without Wd16t_s it stays on the walk."""
    if path == "auto":
        path = choose_path(x.shape[0], density)
        if path == "union" and Wd16t_s is None:
            path = "walk"
        if path == "decode":
            try:
                return twell_ffn_decode(x, Wg_s, Wu_s, Wd_s, T, packed=packed, y=y, status=status, stream=stream,
                                        vals_dtype=vals_dtype)[0]
            except TwellError as e:
                if e.code != TWELL_ERR_UNSUPPORTED:
                    raise
            path = "walk"
    if path == "decode":
        return twell_ffn_decode(x, Wg_s, Wu_s, Wd_s, T, packed=packed, y=y, status=status, stream=stream,
                                vals_dtype=vals_dtype)[0]
    if path == "union" and Wd16t_s is None:
        raise ValueError('path "union" needs Wd16t_s (twell_convert_f16_transposed(Wd_s))')
    if path == "union" and T in (64, 128):
        return twell_ffn_gate_union_fwd(x, Wg_s, Wu_s, Wd16t_s, T, out=packed, y=y, status=status, stream=stream,
                                        vals_dtype=vals_dtype)[0]
    a = twell_gate_pack(x, Wg_s, T, out=packed, status=status, stream=stream, vals_dtype=vals_dtype)
    if path == "union":
        return twell_ffn_union_fwd(x, Wu_s, Wd16t_s, a, y=y, status=status, stream=stream)
    if path == "tile_union":
        if Wd16_s is None:
            raise ValueError('path "tile_union" needs Wd16_s (twell_convert_f16(Wd_s))')
        return twell_ffn_tile_union_fwd(x, Wu_s, Wd16_s, a, y=y, status=status, stream=stream)
    if path != "walk":
        raise ValueError(f"unknown path {path!r}")
    return twell_ffn_fused_fwd(x, Wu_s, Wd_s, a, y=y, status=status, stream=stream)


def twell_unpack(a: TwELL, out: Optional[torch.Tensor] = None, status=None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty((a.n_rows, a.n_cols), dtype=a.dtype, device=a.vals.device)
    s = a.c_struct()
    _check(load().twell_unpack(ctypes.byref(s), _ptr(out),
                               _ptr(status if status is not None else status_buffer(out.device)), _stream(stream)),
           "twell_unpack")
    return out


def twell_column_activity(a: TwELL, counts: Optional[torch.Tensor] = None, status=None, stream=None) -> torch.Tensor:
    """Per-column count of the rows of `a` that keep the column (added to `counts`, zeros if None)."""
    counts = counts if counts is not None else torch.zeros(a.n_cols, dtype=torch.int32, device=a.vals.device)
    s = a.c_struct()
    _check(load().twell_column_activity(ctypes.byref(s), _ptr(counts),
                                        _ptr(status if status is not None else status_buffer(counts.device)),
                                        _stream(stream)),
           "twell_column_activity")
    return counts


def twell_count_nonzeros(a: TwELL, total: Optional[torch.Tensor] = None, status=None, stream=None) -> torch.Tensor:
    """Device int64 [1]: the number of kept entries of `a` (added to `total`, zeros if None)."""
    total = total if total is not None else torch.zeros(1, dtype=torch.int64, device=a.vals.device)
    s = a.c_struct()
    _check(load().twell_count_nonzeros(ctypes.byref(s), _ptr(total),
                                       _ptr(status if status is not None else status_buffer(total.device)),
                                       _stream(stream)),
           "twell_count_nonzeros")
    return total


def twell_gather_rows(src: torch.Tensor, rows: torch.Tensor, out: Optional[torch.Tensor] = None, status=None,
                      stream=None) -> torch.Tensor:
    """out[i] = src[rows[i]] (rows: int32 device tensor)."""
    n_src, d = src.shape
    n = rows.numel()
    out = out if out is not None else torch.empty((n, d), dtype=src.dtype, device=src.device)
    _check(load().twell_gather_rows(_ptr(src), n_src, _ptr(rows), n, d, _dtype_code(src.dtype), _ptr(out),
                                    _ptr(status if status is not None else status_buffer(src.device)),
                                    _stream(stream)),
           "twell_gather_rows")
    return out


def live_columns(counts: torch.Tensor) -> torch.Tensor:
    """Ascending int32 indices (on the counts' device) of the columns that fired at least once;
    computed on the host, once per model."""
    import numpy as np
    live = np.flatnonzero(counts.cpu().numpy() > 0).astype(np.int32)
    return torch.from_numpy(live).to(counts.device)


def compact_weights(Wg_s, Wu_s, Wd_s, live: torch.Tensor, status=None, stream=None):
    """The rows of Wg_s, Wu_s, Wd_s of the live hidden units, in the order of `live`."""
    return tuple(twell_gather_rows(W, live, status=status, stream=stream) for W in (Wg_s, Wu_s, Wd_s))


def twell_pack_from_gate(G: torch.Tensor, T: int = 128, out: Optional[TwELL] = None, status=None,
                         stream=None) -> TwELL:
    N, f = G.shape
    out = out if out is not None else TwELL.empty(N, f, T, G.dtype, G.device)
    s = out.c_struct()
    _check(load().twell_pack_from_gate(_ptr(G), N, f, T, _dtype_code(G.dtype), ctypes.byref(s),
                                       _ptr(status if status is not None else status_buffer(G.device)),
                                       _stream(stream)),
           "twell_pack_from_gate")
    return out


def twell_gate_gemm(x: torch.Tensor, Wg_s: torch.Tensor, out: Optional[torch.Tensor] = None, status=None,
                    stream=None) -> torch.Tensor:
    N, d = x.shape
    f = Wg_s.shape[0]
    out = out if out is not None else torch.empty((N, f), dtype=torch.float32, device=x.device)
    _check(load().twell_gate_gemm(_ptr(x), _ptr(Wg_s), N, d, f, _ptr(out),
                                  _ptr(status if status is not None else status_buffer(x.device)), _stream(stream)),
           "twell_gate_gemm")
    return out


def twell_workspace_bytes(op: int, N: int, d: int, f: int, tile: int = 128, K: int = 0, backup_cap: int = 0) -> int:
    return int(load().twell_workspace_bytes(op, N, d, f, tile, K, backup_cap))


def twell_device_info():
    sm, ma, mi = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().twell_device_info(ctypes.byref(sm), ctypes.byref(ma), ctypes.byref(mi)), "twell_device_info")
    return sm.value, ma.value, mi.value


def twell_gemm_test(A: torch.Tensor, B: torch.Tensor, a_mn: bool, b_mn: bool, status=None, stream=None) -> torch.Tensor:
    """C = A_logical @ B_logical (fp32) where A is [M,K] (or [K,M] if a_mn) and B is [N,K] (or [K,N] if b_mn)."""
    M = A.shape[1] if a_mn else A.shape[0]
    K = A.shape[0] if a_mn else A.shape[1]
    N = B.shape[1] if b_mn else B.shape[0]
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(load().twell_gemm_test(_ptr(A), _ptr(B), M, N, K, int(a_mn), int(b_mn), _ptr(C),
                                  _ptr(status if status is not None else status_buffer(A.device)), _stream(stream)),
           "twell_gemm_test")
    return C


# ------------------------------------------------------------------------------------------ hybrid format

@dataclasses.dataclass
class Hybrid:
    """A hybrid sparse-block / dense-backup context in device memory (twell_hybrid in include/twell.h)."""

    n_rows: int
    n_cols: int
    K: int
    backup_cap: int
    a: torch.Tensor  # [N, K] fp32
    u: torch.Tensor  # [N, K] fp32
    col: torch.Tensor  # [N, K] int16 storage of uint16 columns
    cnt: torch.Tensor  # [N] int16 storage of uint16 counts (0xFFFF = backup row)
    backup_rows: torch.Tensor  # [cap] int32
    n_backup: torch.Tensor  # [1] int32
    A_b: torch.Tensor  # [cap, f] fp32
    U_b: torch.Tensor  # [cap, f] fp32
    l1: torch.Tensor  # [1] fp32
    status: torch.Tensor  # [1] int32

    @staticmethod
    def empty(n_rows, n_cols, K, backup_cap, device=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        cap = max(int(backup_cap), 0)
        z = dict(device=device)
        return Hybrid(n_rows, n_cols, K, cap,
                      torch.empty((n_rows, K), dtype=torch.float32, **z),
                      torch.empty((n_rows, K), dtype=torch.float32, **z),
                      torch.empty((n_rows, K), dtype=torch.int16, **z),
                      torch.empty((n_rows,), dtype=torch.int16, **z),
                      torch.empty((max(cap, 1),), dtype=torch.int32, **z),
                      torch.zeros((1,), dtype=torch.int32, **z),
                      torch.empty((max(cap, 1), n_cols), dtype=torch.float32, **z),
                      torch.empty((max(cap, 1), n_cols), dtype=torch.float32, **z),
                      torch.zeros((1,), dtype=torch.float32, **z),
                      torch.zeros((1,), dtype=torch.int32, **z))

    def counts(self) -> torch.Tensor:
        return self.cnt.to(torch.int32) & 0xFFFF

    def cols(self) -> torch.Tensor:
        return self.col.to(torch.int32) & 0xFFFF

    def c_struct(self) -> _Hybrid:
        def ptr(t):
            return t.data_ptr() if t is not None else None
        return _Hybrid(self.n_rows, self.n_cols, self.K, self.backup_cap, TWELL_BF16, ptr(self.a), ptr(self.u),
                       ptr(self.col), ptr(self.cnt), ptr(self.backup_rows), ptr(self.n_backup), ptr(self.A_b),
                       ptr(self.U_b), ptr(self.l1), ptr(self.status))


def _workspace(op, N, d, f, K, cap, device, ws=None):
    nbytes = twell_workspace_bytes(op, N, d, f, 0, K, cap)
    if ws is not None and ws.numel() >= nbytes:
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def twell_hybrid_route_from_gate(G: torch.Tensor, K: int, backup_cap: int, ctx: Optional[Hybrid] = None, ws=None,
                                 stream=None) -> Hybrid:
    N, f = G.shape
    ctx = ctx if ctx is not None else Hybrid.empty(N, f, K, backup_cap, G.device)
    ws = _workspace(OP_HYBRID_ROUTE, N, 8, f, K, ctx.backup_cap, G.device, ws)
    s = ctx.c_struct()
    _check(load().twell_hybrid_route_from_gate(_ptr(G), N, f, K, TWELL_BF16, ctypes.byref(s), _ptr(ws), ws.numel(),
                                               _stream(stream)), "twell_hybrid_route_from_gate")
    return ctx


def twell_hybrid_fwd(x, Wg_s, Wu_s, Wd_s, K: int, backup_cap: int, l1_coef: float = 2e-5,
                     ctx: Optional[Hybrid] = None, y=None, ws=None, stream=None):
    """Hybrid-format training forward: returns (y, ctx)."""
    N, d = x.shape
    f = Wg_s.shape[0]
    ctx = ctx if ctx is not None else Hybrid.empty(N, f, K, backup_cap, x.device)
    y = y if y is not None else torch.empty((N, d), dtype=x.dtype, device=x.device)
    ws = _workspace(OP_HYBRID_FWD, N, d, f, K, ctx.backup_cap, x.device, ws)
    s = ctx.c_struct()
    _check(load().twell_hybrid_fwd(_ptr(x), _ptr(Wg_s), _ptr(Wu_s), _ptr(Wd_s), N, d, f, K, ctypes.c_float(l1_coef),
                                   TWELL_BF16, ctypes.byref(s), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "twell_hybrid_fwd")
    return y, ctx


def twell_hybrid_bwd(x, Wg_s, Wu_s, Wd_s, ctx: Hybrid, dy, l1_coef: float = 2e-5, dx=None, dWg_s=None, dWu_s=None,
                     dWd_s=None, ws=None, stream=None):
    """Hybrid-format training backward: returns (dx, dWg_s, dWu_s, dWd_s), all fp32."""
    N, d = x.shape
    f = Wg_s.shape[0]
    dx = dx if dx is not None else torch.empty((N, d), dtype=torch.float32, device=x.device)
    dWg_s = dWg_s if dWg_s is not None else torch.empty((f, d), dtype=torch.float32, device=x.device)
    dWu_s = dWu_s if dWu_s is not None else torch.empty((f, d), dtype=torch.float32, device=x.device)
    dWd_s = dWd_s if dWd_s is not None else torch.empty((f, d), dtype=torch.float32, device=x.device)
    ws = _workspace(OP_HYBRID_BWD, N, d, f, ctx.K, ctx.backup_cap, x.device, ws)
    s = ctx.c_struct()
    _check(load().twell_hybrid_bwd(_ptr(x), _ptr(Wg_s), _ptr(Wu_s), _ptr(Wd_s), ctypes.byref(s), _ptr(dy), N, d, f,
                                   ctypes.c_float(l1_coef), _ptr(dx), _ptr(dWg_s), _ptr(dWu_s), _ptr(dWd_s), _ptr(ws),
                                   ws.numel(), _stream(stream)), "twell_hybrid_bwd")
    return dx, dWg_s, dWu_s, dWd_s


def twell_hybrid_route_noalloc(a: TwELL, K: int, ctx: Hybrid, stream=None) -> Hybrid:
    """Route a packed TwELL (fp32 values, tile 128) into `ctx` with no workspace and no allocation
    in the library (see twell_hybrid_route_noalloc in include/twell.h for who needs this)."""
    sa, sc = a.c_struct(), ctx.c_struct()
    _check(load().twell_hybrid_route_noalloc(ctypes.byref(sa), K, ctypes.byref(sc), _stream(stream)),
           "twell_hybrid_route_noalloc")
    return ctx
