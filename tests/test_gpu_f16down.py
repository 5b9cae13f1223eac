"""GPU parity of the fused walk with its down projection in fp16 (twell_ffn_fused_fwd_f16down) and
of the bf16 -> fp16 weight conversion (twell_convert_f16), through the C ABI.

- twell_convert_f16: bit-exact against IEEE round-to-nearest-even (numpy's float16 cast) over
  normal, subnormal and out-of-range magnitudes; an overflow is reported as TWELL_ERR_DEVICE_CHECK;
- the walk against the fp64 oracle (which uses the bf16 weights: the fp16 copy holds the same
  values), within the parity bounds, for every d_model the bulk kernel dispatches, with a ragged
  last tile, split long rows (repeating bit for bit), decoding batches and the full 1.5B-like layer.
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


def _walk_f16(dev, L, vals_dt=torch.float32):
    """The f16down walk on the oracle's own gate activations, packed on the device, and the oracle's y."""
    G = oracle.gate(L.x, L.Wg_s)
    Ga = np.where(G > 0, G, 0.0).astype(np.float32)
    if vals_dt == torch.bfloat16:
        Ga = synthetic.round_bf16_np(Ga)
    tw = binding.twell_pack_from_gate(torch.from_numpy(Ga).to(device=dev, dtype=vals_dt), L.T)
    t = L.torch_inputs(dev)
    Wd16 = binding.twell_convert_f16(t["Wd_s"])
    y = binding.twell_ffn_fused_fwd_f16down(t["x"], t["Wu_s"], Wd16, tw)
    vals, idx, cnt = oracle.twell_pack(Ga.astype(np.float64), L.T)
    y_ref = oracle.twell_walk(vals, idx, cnt, L.T, L.x, L.Wu_s, L.Wd_s)
    return y, y_ref, (t, tw, Wd16)


def test_convert_f16_round_to_nearest_even(cuda_dev):
    rng = np.random.default_rng(3)
    mags = np.concatenate([rng.normal(0, 0.02, 20000),                       # weight-like
                           2.0 ** rng.uniform(-30, -14, 5000) * rng.choice([-1, 1], 5000),  # fp16 subnormal range
                           2.0 ** rng.uniform(-14, 15.99, 5000) * rng.choice([-1, 1], 5000),
                           [0.0, -0.0, 65280.0, -65280.0, 2.0 ** -17, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    src = torch.from_numpy(mags.astype(np.float32)).to(torch.bfloat16)
    want = src.float().numpy().astype(np.float16)
    got = binding.twell_convert_f16(src.to(cuda_dev)).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # exact for every bf16 value of magnitude >= 2^-17
    big = np.abs(src.float().numpy()) >= 2.0 ** -17
    assert np.array_equal(got[big].astype(np.float32), src.float().numpy()[big])
    assert binding.twell_read_status() == 0


@pytest.mark.parametrize("shape", [(1000, 576), (37, 45), (1, 8), (5632, 2048)])
def test_convert_f16_transposed_is_the_transpose(cuda_dev, shape):
    """twell_convert_f16_transposed gives, bit for bit, the transpose of numpy's round-to-nearest-even
    fp16 conversion, for shapes that are and are not multiples of its 32 x 32 tile."""
    rng = np.random.default_rng(shape[0])
    src = torch.from_numpy(rng.normal(0, 0.02, shape).astype(np.float32)).to(torch.bfloat16)
    src[0, 0] = 2.0 ** -20  # an fp16 subnormal
    want = np.ascontiguousarray(src.float().numpy().astype(np.float16).T)
    got = binding.twell_convert_f16_transposed(src.to(cuda_dev)).cpu().numpy()
    assert got.shape == (shape[1], shape[0])
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    assert binding.twell_read_status() == 0


def test_convert_f16_transposed_reports_overflow(cuda_dev):
    src = torch.tensor([[1.0, 65536.0], [-1e6, 3.0]], dtype=torch.bfloat16, device=cuda_dev)
    got = binding.twell_convert_f16_transposed(src).cpu().float().numpy()
    assert binding.twell_read_status(reset=True) == 5  # TWELL_ERR_DEVICE_CHECK
    assert got[0, 0] == 1.0 and got[1, 1] == 3.0 and np.isposinf(got[1, 0]) and np.isneginf(got[0, 1])


def test_convert_f16_reports_overflow(cuda_dev):
    src = torch.tensor([1.0, 65536.0, -1e6, 3.0], dtype=torch.bfloat16, device=cuda_dev)
    got = binding.twell_convert_f16(src).cpu().float().numpy()
    assert binding.twell_read_status(reset=True) == 5  # TWELL_ERR_DEVICE_CHECK
    assert got[0] == 1.0 and got[3] == 3.0 and np.isposinf(got[1]) and np.isneginf(got[2])


@pytest.mark.parametrize("d", [512, 768, 1024, 1280, 1536, 2048, 2560, 3072])
def test_f16down_every_bulk_width(cuda_dev, d):
    """Every d_model the bulk kernel dispatches, with a ragged last tile (f = 1000) and more rows
    than resident warps."""
    L = synthetic.uniform_layer(1500 if d <= 2048 else 600, d, 1000, 128, 0.02, seed=d + 5)
    y, y_ref, _ = _walk_f16(cuda_dev, L)
    assert_close(y.double().cpu().numpy(), y_ref, f"f16down d={d}")


@pytest.mark.parametrize("T", [64, 256])
def test_f16down_tile_widths_bf16_values(cuda_dev, T):
    L = synthetic.uniform_layer(300, 1024, 1000, T, 0.03, seed=T)
    y, y_ref, _ = _walk_f16(cuda_dev, L, torch.bfloat16)
    assert_close(y.double().cpu().numpy(), y_ref, f"f16down T={T}")


def test_f16down_split_rows_repeat_bit_for_bit(cuda_dev):
    """Rows from none to over a thousand nonzeros: the long ones are split into items and their fp32
    partial rows summed in item order, so a second call gives the same bits."""
    L = synthetic.per_token_layer(1500, 2048, 3072, 128, 17, base=0.008, normalise=True, seq_len=128, first=4)
    y1, y_ref, (t, tw, Wd16) = _walk_f16(cuda_dev, L)
    nnz = tw.counts().sum(1).cpu().numpy()
    assert (nnz > 128).sum() >= 20
    y2 = binding.twell_ffn_fused_fwd_f16down(t["x"], t["Wu_s"], Wd16, tw)
    assert torch.equal(y1, y2)
    y = y1.double().cpu().numpy()
    assert_close(y, y_ref, "f16down split rows")
    assert_close(y[nnz > 128], y_ref[nnz > 128], "f16down, the split rows alone")


def test_f16down_zero_density_is_exact_zero(cuda_dev):
    L = synthetic.uniform_layer(200, 512, 1000, 128, 0.02, seed=4)
    L.Wg_s[:, 0] = -1e4  # x[:, 0] = 1: every gate entry is negative
    y, y_ref, _ = _walk_f16(cuda_dev, L)
    assert not np.any(y_ref) and not torch.any(y)


@pytest.mark.parametrize("N", [1, 3, 64])
def test_f16down_decode(cuda_dev, N):
    """Decoding a few tokens of the 1.5B-like layer: gate + pack on the device, then the walk."""
    L = synthetic.layer_1p5b(N=N)
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    y = binding.twell_ffn_fused_fwd_f16down(t["x"], t["Wu_s"], binding.twell_convert_f16(t["Wd_s"]), tw)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"f16down decode N={N}")


def test_f16down_full_size_1p5b_sampled(cuda_dev):
    """The 1.5B-like layer (N = 8192) in the launch configuration the bench times, on sampled rows
    plus the eight longest."""
    L = synthetic.layer_1p5b()
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], L.T)
    y = binding.twell_ffn_fused_fwd_f16down(t["x"], t["Wu_s"], binding.twell_convert_f16(t["Wd_s"]), tw)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    longest = torch.argsort(tw.counts().sum(1), descending=True)[:8].cpu().numpy()
    rows = np.unique(np.concatenate([[0, L.N - 1], rng.choice(L.N, 24, replace=False), longest]))
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, "f16down 1.5b full size")
