"""GPU parity of twell_ffn_gate_union_fwd (gate and up projection in one tcgen05 GEMM on SM pairs,
the TwELL packed and h = a * u formed in its epilogue, then the fp16 down GEMM) through the C ABI.

- the TwELL it writes: bit-exact against the oracle's pack on integer-valued x and Wg_s (exact
  fp32 accumulation in any order) and bit-identical to twell_gate_pack's, for T = 64 / 128, fp32
  and bf16 values, ragged last tiles, d_ff whose 128-unit blocks overrun f_pad (f = 1032);
- y against the fp64 oracle (rel-Frobenius <= 5e-3, max-abs <= 2e-2 x RMS per row) on ragged
  batches, the sweep shapes (sampled rows) and the full-size 1.5B-like / 2B-like layers
  (sampled rows plus the densest rows);
- batches of at most 1024 tokens, whose down GEMM splits K into fp32 partials added in order;
- batches of at most 128 tokens, on the kernels with the weights on the MMA's M side (N = 32 / 64 /
  128 token columns, a cluster pair per 128-unit tile, the down product's K split over a cluster):
  every N up to and across those widths, T = 64 / 128, d_model not a multiple of 128, d_ff whose
  last 128-unit block is mostly past d_ff, every unit kept, no unit kept, the same bits twice;
- edge cases: zero density (y == 0, no entries), every unit kept, N = 1 / 7, an empty batch,
  T = 256 refused, the same bits on a second call.
"""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_ffn_gate_gb300 import binding, build, synthetic
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_dev):
    build.build()
    binding.load()
    binding.status_buffer(cuda_dev).zero_()
    yield
    assert binding.twell_read_status() == 0, "device status was raised"


def _to(dev, a, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)


def _run(dev, t, T, vals_dtype=torch.float32):
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y, tw = binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, T, vals_dtype=vals_dtype)
    torch.cuda.synchronize()
    return y, tw


def _compare_packed(tw, vals, idx, cnt, exact_vals):
    np.testing.assert_array_equal(tw.counts().cpu().numpy(), cnt.astype(np.int64))
    T = vals.shape[2]
    mask = np.arange(T)[None, None, :] < cnt[:, :, None]
    np.testing.assert_array_equal(tw.idx.cpu().numpy()[mask], idx[mask])
    np.testing.assert_array_equal(tw.vals.double().cpu().numpy()[mask], exact_vals[mask])


@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("N,d,f", [(300, 136, 704), (257, 256, 1032), (64, 512, 1000), (1, 256, 1024),
                                   (513, 512, 1280)])
def test_gate_union_twell_bit_exact_and_y(cuda_dev, T, N, d, f, vals_dtype):
    """Integer x and Wg_s: the packed TwELL is the oracle's exactly (values rounded to bf16 when
    asked) and the same as twell_gate_pack's; y matches the oracle's walk of that TwELL."""
    rng = np.random.default_rng(T + N + f)
    x = rng.integers(-1, 2, (N, d)).astype(np.float32)
    x[:, 0] = 1.0
    Wg = rng.integers(-1, 2, (f, d)).astype(np.float32)
    Wg[:, 0] = rng.integers(-6, 2, f)
    Wu = synthetic.round_bf16_np((rng.standard_normal((f, d)) / np.sqrt(d)).astype(np.float32))
    Wd = synthetic.round_bf16_np((rng.standard_normal((f, d)) / np.sqrt(f)).astype(np.float32))
    t = {"x": _to(cuda_dev, x), "Wg_s": _to(cuda_dev, Wg), "Wu_s": _to(cuda_dev, Wu), "Wd_s": _to(cuda_dev, Wd)}
    y, tw = _run(cuda_dev, t, T, vals_dtype)
    G = oracle.gate(x, Wg)  # exact integers
    vals, idx, cnt = oracle.twell_pack(G, T)
    exact = vals if vals_dtype == torch.float32 else oracle.round_bf16(vals)
    _compare_packed(tw, vals, idx, cnt, exact)
    assert cnt.sum() > 0
    ref_tw = binding.twell_gate_pack(t["x"], t["Wg_s"], T, vals_dtype=vals_dtype)
    assert torch.equal(tw.cnt, ref_tw.cnt)
    assert torch.equal(binding.twell_unpack(tw), binding.twell_unpack(ref_tw))
    y_ref = oracle.twell_walk(exact, idx, cnt, T, x.astype(np.float64), Wu.astype(np.float64), Wd.astype(np.float64))
    assert_close(y.double().cpu().numpy(), y_ref, f"gate union int T={T} N={N} f={f} {vals_dtype}")


@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("p", [0.01, 0.05, 0.3])
def test_gate_union_random_ragged(cuda_dev, p, T):
    L = synthetic.uniform_layer(300, 512, 1000, T, p, seed=int(p * 1000) + T)
    y, _ = _run(cuda_dev, L.torch_inputs(cuda_dev), T)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"gate union p={p} T={T}")


def test_gate_union_small_batches(cuda_dev):
    for N in (1, 7):
        L = synthetic.uniform_layer(N, 512, 1024, 128, 0.05, seed=N + 70)
        y, _ = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
        assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"gate union N={N}")


def test_gate_union_zero_density(cuda_dev):
    L = synthetic.uniform_layer(260, 512, 1024, 128, 0.02, seed=4)
    L.Wg_s[:, 0] = -1e4  # no gate fires
    y, tw = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    assert int(tw.counts().sum().item()) == 0
    assert torch.count_nonzero(y).item() == 0


def test_gate_union_every_unit_kept(cuda_dev):
    L = synthetic.uniform_layer(256, 512, 768, 128, 0.5, seed=5)
    L.Wg_s[:, 0] = 1e4
    y, tw = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    assert int(tw.counts().sum().item()) == 256 * 768
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "gate union all kept")


def test_gate_union_empty_batch_and_refused_tile(cuda_dev):
    L = synthetic.uniform_layer(4, 512, 1024, 128, 0.02, seed=1)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y, tw = binding.twell_ffn_gate_union_fwd(t["x"][:0], t["Wg_s"], t["Wu_s"], Wd16t, 128)
    assert y.shape == (0, 512) and tw.cnt.shape == (0, 8)
    with pytest.raises(binding.TwellError) as e:
        binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, 256)
    assert e.value.code == 2  # TWELL_ERR_UNSUPPORTED


def test_gate_union_repeatable_and_agrees_with_the_two_call_union(cuda_dev):
    """A second call gives the same bits; twell_gate_pack + twell_ffn_union_fwd (a rounded to fp16
    before the product) agrees within the parity bounds, and ffn_forward(path="union") is this call."""
    L = synthetic.uniform_layer(640, 512, 1280, 128, 0.03, seed=12)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y1, tw1 = binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, 128)
    y2, tw2 = binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, 128)
    assert torch.equal(y1, y2) and torch.equal(tw1.cnt, tw2.cnt)
    y3 = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128, path="union", Wd16t_s=Wd16t)
    assert torch.equal(y1, y3)
    a = binding.twell_gate_pack(t["x"], t["Wg_s"], 128)
    y4 = binding.twell_ffn_union_fwd(t["x"], t["Wu_s"], Wd16t, a)
    ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s)
    assert_close(y1.double().cpu().numpy(), ref, "gate union")
    assert_close(y4.double().cpu().numpy(), ref, "two-call union")


def _sampled_rows(N, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, N - 1], rng.choice(N, n, replace=False), np.asarray(extra, dtype=np.int64)]))


@pytest.mark.parametrize("p,N", [(0.005, 1024), (0.01, 1024), (0.02, 1024), (0.1, 1024), (0.5, 1024),
                                 (0.01, 8192), (0.02, 8192), (0.05, 8192)])
def test_gate_union_sweep_shapes_sampled(cuda_dev, p, N):
    """The sweep's shapes (d_model 2048, d_ff 5632, T = 128) at N = 1024 and, for 1%, 2% and 5%, at
    the sweep's full 8192 tokens, on sampled rows."""
    L = synthetic.sweep_point(p, 128, N=N)
    y, _ = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    rows = _sampled_rows(L.N, 16, seed=int(p * 1e4))
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"gate union sweep p={p} N={N}")


@pytest.mark.parametrize("which", ["1.5b", "2b"])
def test_gate_union_full_size_layers_sampled(cuda_dev, which):
    """The bench's workloads at full size on sampled rows plus the eight densest rows."""
    L = synthetic.layer_1p5b() if which == "1.5b" else synthetic.layer_2b()
    y, tw = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    longest = torch.argsort(tw.counts().sum(1), descending=True)[:8].cpu().numpy()
    rows = _sampled_rows(L.N, 24, seed=2, extra=longest)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"gate union {which}")


@pytest.mark.parametrize("N", [17, 64, 256, 512, 1024])
def test_gate_union_small_batches_split_down_gemm(cuda_dev, N):
    """Batches of at most 1024 tokens split the down GEMM's K into fp32 partials that a second kernel
    adds in order: the 1.5B-like layer's shapes, every row (N <= 256) or sampled rows plus the densest,
    against the oracle; the two-call union path on the same TwELL agrees as well."""
    L = synthetic.layer_1p5b(N=N)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y, tw = binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, 128)
    y2 = binding.twell_ffn_union_fwd(t["x"], t["Wu_s"], Wd16t, tw)
    longest = torch.argsort(tw.counts().sum(1), descending=True)[:4].cpu().numpy()
    rows = np.arange(N) if N <= 256 else _sampled_rows(N, 24, seed=N, extra=longest)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    sel = torch.from_numpy(rows).to(cuda_dev)
    assert_close(y[sel].double().cpu().numpy(), y_ref, f"gate union split N={N}")
    assert_close(y2[sel].double().cpu().numpy(), y_ref, f"two-call union split N={N}")


@pytest.mark.parametrize("N", [100, 1024, 1025])
def test_union_split_boundary_and_partial_tiles(cuda_dev, N):
    """The down GEMM splits K for at most 1024 tokens and not above; d_model 576 leaves a partial
    256-column tile in every split, d_ff 1000 a partial K range. Both union entry points against the
    oracle on every row (N = 100) or sampled rows."""
    L = synthetic.uniform_layer(N, 576, 1000, 128, 0.03, seed=N + 3)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y, tw = binding.twell_ffn_gate_union_fwd(t["x"], t["Wg_s"], t["Wu_s"], Wd16t, 128)
    y2 = binding.twell_ffn_union_fwd(t["x"], t["Wu_s"], Wd16t, tw)
    rows = np.arange(N) if N <= 128 else _sampled_rows(N, 40, seed=N)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    sel = torch.from_numpy(rows).to(cuda_dev)
    assert_close(y[sel].double().cpu().numpy(), y_ref, f"gate union d=576 N={N}")
    assert_close(y2[sel].double().cpu().numpy(), y_ref, f"two-call union d=576 N={N}")


def _int_layer(N, d, f, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-1, 2, (N, d)).astype(np.float32)
    x[:, 0] = 1.0
    Wg = rng.integers(-1, 2, (f, d)).astype(np.float32)
    Wg[:, 0] = rng.integers(-6, 2, f)
    Wu = synthetic.round_bf16_np((rng.standard_normal((f, d)) / np.sqrt(d)).astype(np.float32))
    Wd = synthetic.round_bf16_np((rng.standard_normal((f, d)) / np.sqrt(f)).astype(np.float32))
    return x, Wg, Wu, Wd


@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("N,d,f", [(1, 512, 1000), (31, 136, 1032), (32, 512, 1000), (33, 576, 1032),
                                   (64, 136, 704), (65, 512, 1000), (100, 576, 1032), (127, 256, 1024),
                                   (128, 512, 1280)])
def test_gate_union_small_batch_kernels(cuda_dev, T, N, d, f):
    """Batches of at most 128 tokens (the transposed gate + up and down kernels): on integer x and
    Wg_s the TwELL is the oracle's bit for bit (fp32 values) and twell_gate_pack's; y matches the
    oracle's walk of that TwELL on every row, repeats bit for bit, and the bf16-value TwELL matches
    the oracle's rounded values."""
    x, Wg, Wu, Wd = _int_layer(N, d, f, seed=N * 7 + f + T)
    t = {"x": _to(cuda_dev, x), "Wg_s": _to(cuda_dev, Wg), "Wu_s": _to(cuda_dev, Wu), "Wd_s": _to(cuda_dev, Wd)}
    G = oracle.gate(x, Wg)
    vals, idx, cnt = oracle.twell_pack(G, T)
    assert cnt.sum() > 0
    for vdt in (torch.float32, torch.bfloat16):
        y, tw = _run(cuda_dev, t, T, vdt)
        exact = vals if vdt == torch.float32 else oracle.round_bf16(vals)
        _compare_packed(tw, vals, idx, cnt, exact)
        ref_tw = binding.twell_gate_pack(t["x"], t["Wg_s"], T, vals_dtype=vdt)
        assert torch.equal(tw.cnt, ref_tw.cnt)
        assert torch.equal(binding.twell_unpack(tw), binding.twell_unpack(ref_tw))
        y_ref = oracle.twell_walk(exact, idx, cnt, T, x.astype(np.float64), Wu.astype(np.float64),
                                  Wd.astype(np.float64))
        assert_close(y.double().cpu().numpy(), y_ref, f"gate union small N={N} d={d} f={f} T={T} {vdt}")
        y2, tw2 = _run(cuda_dev, t, T, vdt)
        assert torch.equal(y, y2) and torch.equal(tw.cnt, tw2.cnt)


@pytest.mark.parametrize("N", [40, 128])
def test_gate_union_small_batch_all_and_none_kept(cuda_dev, N):
    """Every unit kept (each T-tile count T, h everywhere) and no unit kept (y exactly 0)."""
    L = synthetic.uniform_layer(N, 512, 1000, 128, 0.5, seed=N)
    L.Wg_s[:, 0] = 1e4
    y, tw = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    assert int(tw.counts().sum().item()) == N * 1000
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"small all kept N={N}")
    L.Wg_s[:, 0] = -1e4
    y, tw = _run(cuda_dev, L.torch_inputs(cuda_dev), 128)
    assert int(tw.counts().sum().item()) == 0 and torch.count_nonzero(y).item() == 0
