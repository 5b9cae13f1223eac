"""GPU parity of the inference path against the fp64 oracle, through the C ABI.

- twell_gate_gemm (tcgen05 main loop, plain epilogue) vs exact integer products and fp64 matmul;
- twell_pack_from_gate / twell_unpack: bit-exact against the oracle's TwELL pack;
- twell_gate_pack (tcgen05 + ReLU/TwELL epilogue): bit-exact on integer-valued inputs, where
  the fp32 accumulator is exact in any order;
- twell_ffn_fused_fwd on an oracle-packed TwELL, and the whole path (gate_pack + fused), within
  rel-Frobenius <= 5e-3 and max-abs <= 2e-2 * RMS(ref) of the fp64 oracle;
- the full-size 1.5B-like and 2B-like layers in the launch configuration the bench times,
  checked on sampled rows;
- edge cases: empty batch, zero density, full density, rows longer than one list window.
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


def _int_layer(N, d, f, seed, bias_lo=-6, bias_hi=2):
    """Integer-valued x and Wg_s: every product and partial sum is exact in fp32 and bf16 holds
    every input exactly."""
    rng = np.random.default_rng(seed)
    x = rng.integers(-1, 2, (N, d)).astype(np.float32)
    x[:, 0] = 1.0
    W = rng.integers(-1, 2, (f, d)).astype(np.float32)
    W[:, 0] = rng.integers(bias_lo, bias_hi, f)
    return x, W


def _to(dev, a, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)


def _compare_packed(tw, vals, idx, cnt, exact_vals=None):
    """Compare a device TwELL with an oracle pack: counts, indices and values of slots < cnt."""
    g_cnt = tw.counts().cpu().numpy()
    np.testing.assert_array_equal(g_cnt, cnt.astype(np.int64))
    g_idx = tw.idx.cpu().numpy()
    g_val = tw.vals.double().cpu().numpy()
    ref_vals = vals if exact_vals is None else exact_vals
    N, nt, T = vals.shape
    mask = np.arange(T)[None, None, :] < cnt[:, :, None]
    np.testing.assert_array_equal(g_idx[mask], idx[mask])
    np.testing.assert_array_equal(g_val[mask], ref_vals[mask])


# ------------------------------------------------------------------------------------------ GEMM

@pytest.mark.parametrize("N,d,f", [(128, 64, 256), (300, 136, 700), (1000, 520, 1284), (64, 2048, 256)])
def test_gate_gemm_integer_exact(cuda_dev, N, d, f):
    x, W = _int_layer(N, d, f, seed=N + d)
    G = binding.twell_gate_gemm(_to(cuda_dev, x), _to(cuda_dev, W))
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    np.testing.assert_array_equal(G.double().cpu().numpy(), ref)


def test_gate_gemm_random_vs_fp64(cuda_dev):
    L = synthetic.uniform_layer(384, 1024, 1536, 128, 0.01, seed=5)
    G = binding.twell_gate_gemm(_to(cuda_dev, L.x), _to(cuda_dev, L.Wg_s)).double().cpu().numpy()
    ref = oracle.gate(L.x, L.Wg_s)
    assert np.abs(G - ref).max() <= 1e-4 * np.abs(ref).max()


# ------------------------------------------------------------------------------------------ pack

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,N,f", [(64, 77, 300), (128, 130, 1024), (256, 33, 700), (128, 5, 5632)])
def test_pack_from_gate_bit_exact(cuda_dev, dtype, T, N, f):
    rng = np.random.default_rng(T * N + f)
    G = (rng.standard_normal((N, f)) - 1.5).astype(np.float32)
    G[0] = -1.0
    G[1 % N] = 1.0
    G[2 % N, ::4] = -0.0
    if dtype == torch.bfloat16:
        G = synthetic.round_bf16_np(G)
    tw = binding.twell_pack_from_gate(_to(cuda_dev, G, dtype), T)
    vals, idx, cnt = oracle.twell_pack(G.astype(np.float64), T)
    _compare_packed(tw, vals, idx, cnt)
    dense = binding.twell_unpack(tw).double().cpu().numpy()
    assert np.array_equal(dense, np.where(G > 0, G, 0).astype(np.float64))


def test_pack_empty_batch(cuda_dev):
    G = torch.zeros((0, 256), dtype=torch.bfloat16, device=cuda_dev)
    tw = binding.twell_pack_from_gate(G, 128)
    assert tw.cnt.shape == (0, 2)


# ------------------------------------------------------------------------------------------ gate + pack

@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("N,d,f", [(300, 136, 700), (257, 256, 1024), (64, 2048, 5632), (1, 512, 1000),
                                   (200, 256, 1024)])
def test_gate_pack_integer_bit_exact(cuda_dev, T, N, d, f, vals_dtype):
    """Bit-exact TwELL pack from the gate GEMM epilogue, on SM-pair 256 x 256 tiles (N > 256) and on
    single-SM 128 x T tiles (batches of up to 256 tokens)."""
    x, W = _int_layer(N, d, f, seed=T + N)
    tw = binding.twell_gate_pack(_to(cuda_dev, x), _to(cuda_dev, W), T, vals_dtype=vals_dtype)
    G = oracle.gate(x, W)  # exact integers
    vals, idx, cnt = oracle.twell_pack(G, T)
    exact = vals if vals_dtype == torch.float32 else oracle.round_bf16(vals)
    _compare_packed(tw, vals, idx, cnt, exact_vals=exact)
    assert cnt.sum() > 0


@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("N,d,f", [(1, 2048, 5632), (2, 64, 300), (7, 512, 1000), (8, 1024, 777), (9, 256, 1024),
                                   (16, 4096, 520), (17, 512, 1000)])
def test_gate_pack_small_batch_bit_exact(cuda_dev, T, N, d, f, vals_dtype):
    """Batches of up to 16 tokens run the cluster-pair GEMV kernel (two CTAs per column tile, the
    tile's halves exchanged through distributed shared memory); 17 tokens the 128 x T tile GEMM.
    Bit-exact on integer inputs, with ragged last tiles, and the same bits on a second call."""
    x, W = _int_layer(N, d, f, seed=3 * T + N)
    xt, Wt = _to(cuda_dev, x), _to(cuda_dev, W)
    tw = binding.twell_gate_pack(xt, Wt, T, vals_dtype=vals_dtype)
    G = oracle.gate(x, W)
    vals, idx, cnt = oracle.twell_pack(G, T)
    exact = vals if vals_dtype == torch.float32 else oracle.round_bf16(vals)
    _compare_packed(tw, vals, idx, cnt, exact_vals=exact)
    assert cnt.sum() > 0
    tw2 = binding.twell_gate_pack(xt, Wt, T, vals_dtype=vals_dtype)
    assert torch.equal(tw.cnt, tw2.cnt) and torch.equal(binding.twell_unpack(tw), binding.twell_unpack(tw2))


def test_gate_pack_small_batch_random_matches_oracle(cuda_dev):
    """Random bf16 decode batch of the 1.5B-like layer: kept set and values against fp64 away from
    zero, and the fp32 sums equal to the large-batch tile GEMM's within fp32 rounding."""
    L = synthetic.layer_1p5b(N=12)
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    dense = binding.twell_unpack(tw).double().cpu().numpy()
    G = oracle.gate(L.x, L.Wg_s)
    big = np.abs(G) > 1e-3
    assert np.array_equal(dense[big] > 0, G[big] > 0)
    np.testing.assert_allclose(dense[big], np.maximum(G[big], 0), rtol=1e-5, atol=2e-5)
    # the same rows inside a 300-token batch go through the tile GEMM
    x_big = torch.cat([t["x"], t["x"][:1].expand(288, -1)]).contiguous()
    dense_big = binding.twell_unpack(binding.twell_gate_pack(x_big, t["Wg_s"], L.T))[:12].double().cpu().numpy()
    both = big & (dense > 0)
    np.testing.assert_allclose(dense[both], dense_big[both], rtol=1e-5, atol=2e-5)


@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
def test_gate_pack_random_matches_oracle_away_from_zero(cuda_dev, vals_dtype):
    """On random bf16 layers the kept set can differ from fp64 only where |g| is at the fp32
    accumulation-error level."""
    L = synthetic.uniform_layer(512, 1024, 2048, 128, 0.02, seed=9)
    tw = binding.twell_gate_pack(_to(cuda_dev, L.x), _to(cuda_dev, L.Wg_s), L.T, vals_dtype=vals_dtype)
    dense = binding.twell_unpack(tw).double().cpu().numpy()
    G = oracle.gate(L.x, L.Wg_s)
    ref = np.where(G > 0, G, 0.0)
    big = np.abs(G) > 1e-3
    assert np.array_equal(dense[big] > 0, ref[big] > 0)
    if vals_dtype == torch.float32:
        np.testing.assert_allclose(dense[big], ref[big], rtol=1e-5, atol=2e-5)
    else:
        # fp32 and fp64 accumulators may round to neighbouring bf16 values: one bf16 ulp (2^-7 relative)
        np.testing.assert_allclose(dense[big], oracle.round_bf16(ref[big]), rtol=2 ** -7, atol=2e-5)


def test_gate_pack_f32_path(cuda_dev):
    L = synthetic.tiny_fp32()
    tw = binding.twell_gate_pack(_to(cuda_dev, L.x, torch.float32), _to(cuda_dev, L.Wg_s, torch.float32), L.T)
    dense = binding.twell_unpack(tw).double().cpu().numpy()
    G = oracle.gate(L.x, L.Wg_s)
    big = np.abs(G) > 1e-4
    assert np.array_equal(dense[big] > 0, G[big] > 0)
    # fp32 accumulation of terms of size ~1 (with cancellation against the bias): ~1e-6 absolute
    np.testing.assert_allclose(dense[big], np.maximum(G[big], 0), rtol=1e-5, atol=2e-5)


# ------------------------------------------------------------------------------------------ fused up+down

def _fused_from_oracle_pack(dev, L, dt, vals_dt=None):
    """Run the fused kernel on the oracle's own gate activations, packed on the device."""
    vals_dt = vals_dt or dt
    G = oracle.gate(L.x, L.Wg_s)
    Ga = np.where(G > 0, G, 0.0)
    Gs = synthetic.round_bf16_np(Ga.astype(np.float32)) if vals_dt == torch.bfloat16 else Ga.astype(np.float32)
    tw = binding.twell_pack_from_gate(_to(dev, Gs, vals_dt), L.T)
    t = L.torch_inputs(dev, dt)
    y = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    vals, idx, cnt = oracle.twell_pack(Gs.astype(np.float64), L.T)
    y_ref = oracle.twell_walk(vals, idx, cnt, L.T, L.x, L.Wu_s, L.Wd_s)
    return y.double().cpu().numpy(), y_ref


def test_fused_tiny_fp32(cuda_dev):
    L = synthetic.tiny_fp32()
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.float32)
    rel, mx = assert_close(y, y_ref, "fused fp32")
    assert rel < 1e-5


@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [64, 128, 256])
def test_fused_bf16_small(cuda_dev, T, vals_dtype):
    L = synthetic.uniform_layer(200, 512, 1000, T, 0.03, seed=T)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.bfloat16, vals_dtype)
    assert_close(y, y_ref, f"fused bf16 T={T}")


def test_fused_wide_model_two_chunks_per_thread(cuda_dev):
    """d_model = 5120: more 16-byte chunks than consumer threads (two chunks per thread)."""
    L = synthetic.uniform_layer(64, 5120, 768, 128, 0.03, seed=6)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.bfloat16, torch.float32)
    assert_close(y, y_ref, "fused d=5120")


@pytest.mark.parametrize("d,dt", [(64, torch.bfloat16), (512, torch.bfloat16), (1024, torch.bfloat16),
                                  (1280, torch.bfloat16), (1536, torch.bfloat16), (2048, torch.bfloat16),
                                  (2560, torch.bfloat16), (3072, torch.bfloat16), (4096, torch.bfloat16),
                                  (1000, torch.bfloat16), (1024, torch.float32), (2048, torch.float32)])
def test_fused_every_row_layout(cuda_dev, d, dt):
    """Every (chunks per lane, warps per row) layout the fused kernel dispatches to, with a ragged
    last tile (f = 1000) and more rows than resident warps."""
    L = synthetic.uniform_layer(1500 if d <= 2048 else 600, d, 1000, 128, 0.02, seed=d, bf16=dt == torch.bfloat16)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, dt, torch.float32)
    assert_close(y, y_ref, f"fused d={d} {dt}")


def test_fused_mostly_empty_rows(cuda_dev):
    """About one nonzero per row: most metadata segments are empty rows (y = 0) or hold one entry."""
    L = synthetic.uniform_layer(2000, 512, 1000, 128, 0.0008, seed=8)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.bfloat16)
    assert (np.abs(y_ref).sum(1) == 0).sum() > 500
    assert_close(y, y_ref, "fused mostly empty rows")
    assert np.array_equal(np.abs(y).sum(1) == 0, np.abs(y_ref).sum(1) == 0)


def test_fused_reports_corrupt_entries(cuda_dev):
    """A count above the tile width, an in-tile index >= T and a column >= d_ff are reported as
    TWELL_ERR_DEVICE_CHECK and contribute nothing; the other rows are unaffected."""
    L = synthetic.uniform_layer(64, 256, 1000, 128, 0.05, seed=9, bf16=False)
    G = oracle.gate(L.x, L.Wg_s)
    vals, idx, cnt = oracle.twell_pack(np.where(G > 0, G, 0.0), L.T)
    assert cnt[0, 0] > 0 and cnt[1, 0] > 0 and cnt[2, 7] > 0
    bad_vals, bad_idx, bad_cnt = vals.copy(), idx.copy(), cnt.copy()
    bad_cnt[0, 0] = L.T + 5  # count above the tile width: the tile is dropped
    bad_idx[1, 0, 0] = L.T + 3  # in-tile index past the tile
    bad_idx[2, 7, 0] = 110  # column 7*128 + 110 = 1006 >= d_ff = 1000
    clean_vals, clean_cnt = vals.copy(), cnt.copy()
    clean_cnt[0, 0] = 0
    clean_vals[1, 0, 0] = 0.0
    clean_vals[2, 7, 0] = 0.0
    y_ref = oracle.twell_walk(clean_vals, idx, clean_cnt, L.T, L.x, L.Wu_s, L.Wd_s)
    nt = cnt.shape[1]
    tw = binding.TwELL(L.N, L.f, L.T, _to(cuda_dev, np.nan_to_num(bad_vals), torch.float32),
                       torch.from_numpy(bad_idx).to(cuda_dev),
                       torch.from_numpy(bad_cnt.astype(np.int16)).to(cuda_dev).reshape(L.N, nt))
    t = L.torch_inputs(cuda_dev, torch.float32)
    y = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    assert binding.twell_read_status(reset=True) == 5  # TWELL_ERR_DEVICE_CHECK
    rel, mx = assert_close(y.double().cpu().numpy(), y_ref, "fused with corrupt entries")
    assert rel < 1e-5


def test_fused_long_rows_cross_list_windows(cuda_dev):
    """Rows with more nonzeros than one list window (256) and than the slot ring."""
    L = synthetic.uniform_layer(24, 256, 2048, 128, 0.5, seed=4)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.bfloat16)
    assert_close(y, y_ref, "fused long rows")


def _long_row_layer(N, d, f, seed, base=0.008):
    """Per-token density (lognormal spread, ten times denser sequence starts): rows from none to
    over a thousand nonzeros, so the fused walk cuts the long rows into items."""
    return synthetic.per_token_layer(N, d, f, 128, seed, base=base, normalise=True, seq_len=128, first=4)


@pytest.mark.parametrize("d", [512, 2048, 2560])
def test_fused_splits_long_rows(cuda_dev, d):
    """Long rows are walked as several items (here of at most 32 nonzeros: 1500 rows are a small
    batch) whose fp32 partial rows the last one to finish adds up in item order: the result
    matches the oracle and repeats bit for bit."""
    L = _long_row_layer(1500, d, 3072, seed=d + 11)
    G = oracle.gate(L.x, L.Wg_s)
    nnz = (G > 0).sum(1)
    assert (nnz > 128).sum() >= 20 and nnz.max() > 600
    Ga = np.where(G > 0, G, 0.0).astype(np.float32)
    tw = binding.twell_pack_from_gate(_to(cuda_dev, Ga, torch.float32), L.T)
    t = L.torch_inputs(cuda_dev)
    y1 = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    y2 = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    assert torch.equal(y1, y2)
    vals, idx, cnt = oracle.twell_pack(Ga.astype(np.float64), L.T)
    y_ref = oracle.twell_walk(vals, idx, cnt, L.T, L.x, L.Wu_s, L.Wd_s)
    y = y1.double().cpu().numpy()
    assert_close(y, y_ref, f"fused split rows d={d}")
    assert_close(y[nnz > 128], y_ref[nnz > 128], f"fused, the split rows alone, d={d}")


def test_fused_split_item_list_full(cuda_dev):
    """More long rows than the item list holds (1024 items; 100 rows of ~300 nonzeros in items of 4
    want ~7,700): the rows that find no room are walked whole, the others split; every row matches
    the oracle."""
    L = synthetic.uniform_layer(100, 2048, 3072, 128, 0.1, seed=21)
    y, y_ref = _fused_from_oracle_pack(cuda_dev, L, torch.bfloat16, torch.float32)
    assert_close(y, y_ref, "fused split, item list full")


@pytest.mark.parametrize("N", [1, 3, 64])
def test_small_batch_decode(cuda_dev, N):
    """Decoding a few tokens of the 1.5B-like layer (d_model 2048, d_ff 5632, ~29 nonzeros per
    token): each row's nonzeros are spread over items of 4 nonzeros on different warps; gate + pack
    and the walk end to end against the oracle, and a second call repeats bit for bit."""
    L = synthetic.layer_1p5b(N=N)
    t = L.torch_inputs(cuda_dev)
    y1 = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T)
    y2 = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T)
    assert torch.equal(y1, y2)
    assert_close(y1.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"decode N={N}")


def test_streamed_batches_match_ffn_forward(cuda_dev):
    """binding.StreamedFFN (copies overlapped with compute on three streams, double-buffered device
    buffers) returns, for five different host batches, exactly what ffn_forward returns for each."""
    L = synthetic.uniform_layer(5 * 256, 512, 1024, 128, 0.02, seed=41)
    t = L.torch_inputs(cuda_dev)
    pipe = binding.StreamedFFN(t["Wg_s"], t["Wu_s"], t["Wd_s"], 256, T=L.T)
    xs = [t["x"][256 * i:256 * (i + 1)].cpu().pin_memory() for i in range(5)]
    ys = [torch.empty((256, L.d), dtype=torch.bfloat16).pin_memory() for _ in range(5)]
    for xh, yh in zip(xs, ys):
        pipe.submit(xh, yh)
    torch.cuda.synchronize()
    for i in range(5):
        ref = binding.ffn_forward(t["x"][256 * i:256 * (i + 1)].contiguous(), t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T)
        assert torch.equal(ys[i], ref.cpu()), i


# ------------------------------------------------------------------------------------------ union path

@pytest.mark.parametrize("N", [7, 300])
@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
def test_union_small_ragged(cuda_dev, vals_dtype, N):
    """twell_ffn_union_fwd on an oracle-packed TwELL with a ragged last tile (d_ff = 1000), for a
    batch that fills part of one 128-row tile and for one that spans three."""
    L = synthetic.uniform_layer(N, 512, 1000, 128, 0.05, seed=31 + N)
    G = oracle.gate(L.x, L.Wg_s)
    Ga = np.where(G > 0, G, 0.0)
    Gs = synthetic.round_bf16_np(Ga.astype(np.float32)) if vals_dtype == torch.bfloat16 else Ga.astype(np.float32)
    tw = binding.twell_pack_from_gate(_to(cuda_dev, Gs, vals_dtype), L.T)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    y = binding.twell_ffn_union_fwd(t["x"], t["Wu_s"], Wd16t, tw).double().cpu().numpy()
    vals, idx, cnt = oracle.twell_pack(Gs.astype(np.float64), L.T)
    assert_close(y, oracle.twell_walk(vals, idx, cnt, L.T, L.x, L.Wu_s, L.Wd_s), f"union {vals_dtype}")


@pytest.mark.parametrize("T", [64, 256])
def test_union_other_tile_widths(cuda_dev, T):
    """The union path reads TwELL tiles of 64 and 256 columns (d_ff 1000: a ragged last tile)."""
    L = synthetic.uniform_layer(200, 512, 1000, T, 0.04, seed=T + 5)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=T, path="union",
                            Wd16t_s=binding.twell_convert_f16_transposed(t["Wd_s"]))
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"union T={T}")


def test_step_replays_from_a_cuda_graph(cuda_dev):
    """Gate + pack and the walk captured once into a CUDA graph (the library allocates nothing and
    its work counters are reset by a memset node inside the graph), then replayed on new inputs
    copied into the same buffers: each replay gives what a direct call gives."""
    L = synthetic.uniform_layer(512, 512, 1024, 128, 0.02, seed=44)
    t = L.torch_inputs(cuda_dev)
    x = t["x"].clone()
    packed = binding.TwELL.empty(L.N, L.f, L.T, torch.float32, cuda_dev)
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up call on the capture stream (workspace allocated here)
        binding.ffn_forward(x, t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T, packed=packed, y=y)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.ffn_forward(x, t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T, packed=packed, y=y)
    rng = np.random.default_rng(5)
    for _ in range(3):
        xn = synthetic.round_bf16_np(rng.standard_normal((L.N, L.d)).astype(np.float32))
        xn[:, 0] = 1.0
        x.copy_(torch.from_numpy(xn).to(cuda_dev, torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        ref = binding.ffn_forward(x.clone(), t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T)
        assert torch.equal(y, ref)
    assert binding.twell_read_status() == 0


def test_streamed_batches_union_path(cuda_dev):
    """StreamedFFN on the union path returns what ffn_forward(path="union") returns."""
    L = synthetic.uniform_layer(3 * 128, 512, 1024, 128, 0.05, seed=43)
    t = L.torch_inputs(cuda_dev)
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    pipe = binding.StreamedFFN(t["Wg_s"], t["Wu_s"], t["Wd_s"], 128, T=L.T, path="union", Wd16t_s=Wd16t)
    xs = [t["x"][128 * i:128 * (i + 1)].cpu().pin_memory() for i in range(3)]
    ys = [torch.empty((128, L.d), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    for xh, yh in zip(xs, ys):
        pipe.submit(xh, yh)
    torch.cuda.synchronize()
    for i in range(3):
        ref = binding.ffn_forward(t["x"][128 * i:128 * (i + 1)].contiguous(), t["Wg_s"], t["Wu_s"], t["Wd_s"],
                                  T=L.T, path="union", Wd16t_s=Wd16t)
        assert torch.equal(ys[i], ref.cpu()), i


@pytest.mark.parametrize("p", [0.01, 0.05, 0.5])
def test_union_sweep_shapes_end_to_end_sampled(cuda_dev, p):
    """The union path end to end (gate + pack, then the two GEMMs) at the sweep's shapes
    (d_model 2048, d_ff 5632, N = 1024) on sampled rows, against the oracle."""
    L = synthetic.sweep_point(p, 128, N=1024)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128, path="union",
                            Wd16t_s=binding.twell_convert_f16_transposed(t["Wd_s"]))
    rows = _sampled_rows(L.N, 12, seed=3)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"union p={p}")


def test_fused_zero_density_is_exact_zero(cuda_dev):
    L = synthetic.uniform_layer(130, 256, 512, 128, 0.02, seed=1)
    L.Wg_s[:, 0] = -1e4
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128)
    assert torch.count_nonzero(y).item() == 0


def test_fused_empty_batch(cuda_dev):
    L = synthetic.uniform_layer(4, 256, 512, 128, 0.02, seed=1)
    t = L.torch_inputs(cuda_dev)
    x = t["x"][:0]
    y = binding.ffn_forward(x, t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128)
    assert y.shape == (0, 256)


# ------------------------------------------------------------------------------------------ dead-column compaction

def test_column_activity_matches_oracle_counts(cuda_dev):
    """Per-column keep counts of a device TwELL equal the oracle's count of g > 0, exactly."""
    L = synthetic.uniform_layer(700, 512, 1000, 128, 0.03, seed=21, dead_frac=0.3)
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    counts = binding.twell_column_activity(tw)
    dense = binding.twell_unpack(tw).double().cpu().numpy()
    np.testing.assert_array_equal(counts.cpu().numpy(), (dense > 0).sum(0))
    G = oracle.gate(L.x, L.Wg_s)
    assert (counts.cpu().numpy() == 0).sum() >= 300  # the dead columns never fire
    big = np.abs(G) > 1e-2  # away from the accumulation-order threshold both agree
    np.testing.assert_array_equal(((G > 0) & big).sum(0) <= counts.cpu().numpy(), True)
    np.testing.assert_array_equal(counts.cpu().numpy() <= ((G > 0) | ~big).sum(0), True)
    twice = binding.twell_column_activity(tw, counts=counts.clone())
    np.testing.assert_array_equal(twice.cpu().numpy(), 2 * counts.cpu().numpy())


def test_gather_rows_copies_and_checks(cuda_dev):
    src = torch.randn(50, 64, device=cuda_dev).to(torch.bfloat16)
    rows = torch.tensor([3, 0, 49, 7, 7], dtype=torch.int32, device=cuda_dev)
    out = binding.twell_gather_rows(src, rows)
    assert torch.equal(out, src[rows.long()])
    bad = torch.tensor([1, 50, 2], dtype=torch.int32, device=cuda_dev)
    out = binding.twell_gather_rows(src, bad)
    assert binding.twell_read_status(reset=True) == 5  # TWELL_ERR_DEVICE_CHECK
    assert torch.equal(out[0], src[1]) and torch.equal(out[2], src[2])
    assert torch.count_nonzero(out[1]).item() == 0


def test_compacted_layer_gives_the_same_y(cuda_dev):
    """Live columns from a calibration batch, weights gathered to them: y is bit-identical to the
    uncompacted layer on a different batch (1.5B-like shapes, 30% dead columns, N = 1024), and
    matches the fp64 oracle's dense layer over all d_ff units (the dropped ones included) on every
    row."""
    L = synthetic.layer_1p5b(N=1024)
    t = L.torch_inputs(cuda_dev)
    x_cal = torch.from_numpy(synthetic.calibration_tokens(L, 2048, seed=77)).to(cuda_dev, torch.bfloat16)
    counts = binding.twell_column_activity(binding.twell_gate_pack(x_cal, t["Wg_s"], L.T))
    live = binding.live_columns(counts)
    assert 0.68 * L.f <= live.numel() <= 0.72 * L.f
    Wg_c, Wu_c, Wd_c = binding.compact_weights(t["Wg_s"], t["Wu_s"], t["Wd_s"], live)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    y = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    # the batch's active units are among the calibration's live ones
    active = binding.twell_column_activity(tw).cpu().numpy() > 0
    assert not (active & (counts.cpu().numpy() == 0)).any()
    y_c = binding.ffn_forward(t["x"], Wg_c, Wu_c, Wd_c, T=L.T)
    assert torch.equal(y_c, y)
    assert_close(y_c.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "compacted layer vs oracle")


# ------------------------------------------------------------------------------------------ end to end

def test_end_to_end_tiny_fp32(cuda_dev):
    L = synthetic.tiny_fp32()
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T).double().cpu().numpy()
    assert_close(y, oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "tiny fp32 end to end")


def test_end_to_end_bf16_values(cuda_dev):
    """bf16-rounded packed values: one more rounding, still inside the bounds."""
    L = synthetic.uniform_layer(333, 512, 1280, 128, 0.01, seed=3)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128, vals_dtype=torch.bfloat16)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "end to end, bf16 values")


@pytest.mark.parametrize("p", [0.005, 0.05, 1.0])
def test_end_to_end_bf16_density(cuda_dev, p):
    L = synthetic.uniform_layer(333, 512, 1280, 128, min(p, 0.999), seed=int(p * 1000))
    if p == 1.0:
        L.Wg_s[:, 0] = 1e4  # every gate on: the plain ReLU FFN with a = g
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128).double().cpu().numpy()
    assert_close(y, oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"end to end p={p}")


def _sampled_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, 2, 3, N - 1], rng.choice(N, n, replace=False)]))


@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("p", [0.001, 0.05, 0.5])
def test_sweep_shapes_end_to_end_sampled(cuda_dev, p, T):
    """The density x tile-width sweep's shapes (d_model 2048, d_ff 5632, uniform density p) at
    N = 1024, end to end (gate + pack, fused walk), on sampled rows."""
    L = synthetic.sweep_point(p, T, N=1024)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=T)
    rows = _sampled_rows(L.N, 12, seed=T)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"sweep p={p} T={T}")


def test_sweep_point_full_size_sampled(cuda_dev):
    """One sweep point at the bench's full size (N = 8192, p = 1%, T = 256), on sampled rows."""
    L = synthetic.sweep_point(0.01, 256)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=256)
    rows = _sampled_rows(L.N, 16, seed=5)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, "sweep p=1% T=256 full size")


@pytest.mark.parametrize("which", ["1.5b", "2b"])
def test_full_size_layers_sampled(cuda_dev, which):
    """The bench's workloads at full size, in the bench's launch configuration, on sampled rows."""
    L = synthetic.layer_1p5b() if which == "1.5b" else synthetic.layer_2b()
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    y = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    torch.cuda.synchronize()
    # sampled rows plus the eight longest ones (on the 2B-like layer those are split into items)
    longest = torch.argsort(tw.counts().sum(1), descending=True)[:8].cpu().numpy()
    rows = np.unique(np.concatenate([_sampled_rows(L.N, 24, seed=1), longest]))
    y_ref, G, _ = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows, return_gu=True)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, which)
    # the row counts agree with the oracle's except where |g| is at the accumulation-error level
    cnt = tw.counts()[torch.from_numpy(rows).to(cuda_dev)].sum(1).cpu().numpy()
    lo = (G > 1e-2).sum(1)
    hi = (G > -1e-2).sum(1)
    assert np.all(cnt >= lo) and np.all(cnt <= hi)
