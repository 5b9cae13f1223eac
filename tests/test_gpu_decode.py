"""GPU parity of the fused decode path (twell_ffn_decode: gate + pack + per-tile walk in one cluster
kernel, the partial rows summed in a fixed order by a second) against the fp64 oracle, through the C ABI.

- the TwELL it writes is the one twell_gate_pack writes, bit for bit, and on integer inputs the
  oracle's pack exactly;
- y within the parity bounds of the oracle, for 1 to 16 tokens, tile widths 64, 128, 256, fp32 and
  bf16 values, d_model 512 to 4096 (multiples of 64, not only of 256) and ragged last tiles;
- y the same bit for bit on a second call; zero density gives y = 0 exactly.
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


def _same_twell(a, b):
    assert torch.equal(a.cnt, b.cnt)
    assert torch.equal(binding.twell_unpack(a), binding.twell_unpack(b))


@pytest.mark.parametrize("vals_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 2, 5, 8, 9, 16])
def test_decode_1p5b_matches_oracle(cuda_dev, N, T, vals_dtype):
    """The 1.5B-like layer (d_model 2048, d_ff 5632, ~29 nonzeros per token) at decode batch sizes."""
    L = synthetic.layer_1p5b(N=N)
    t = L.torch_inputs(cuda_dev)
    y, tw = binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T, vals_dtype=vals_dtype)
    _same_twell(tw, binding.twell_gate_pack(t["x"], t["Wg_s"], T, vals_dtype=vals_dtype))
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"decode N={N} T={T}")
    y2, _ = binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T, vals_dtype=vals_dtype)
    assert torch.equal(y, y2)
    # the two-call path on the same TwELL agrees to fp32 summation order
    y_walk = binding.twell_ffn_fused_fwd(t["x"], t["Wu_s"], t["Wd_s"], tw)
    assert_close(y.double().cpu().numpy(), y_walk.double().cpu().numpy(), f"decode vs walk N={N} T={T}")


@pytest.mark.parametrize("N,d,f,T", [(3, 512, 1000, 128), (16, 576, 1000, 64), (7, 1024, 3000, 256),
                                     (12, 2560, 6912, 128), (16, 4096, 1500, 128), (1, 64, 300, 64)])
def test_decode_other_shapes(cuda_dev, N, d, f, T):
    L = synthetic.uniform_layer(N, d, f, T, 0.02, seed=N + d)
    t = L.torch_inputs(cuda_dev)
    y, tw = binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T)
    _same_twell(tw, binding.twell_gate_pack(t["x"], t["Wg_s"], T))
    assert tw.counts().sum().item() > 0
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"decode {N},{d},{f},{T}")


def test_decode_integer_inputs_pack_exactly(cuda_dev):
    """Integer-valued x and weights: every sum is exact in fp32, so the TwELL equals the oracle's
    pack bit for bit and y equals the oracle's y rounded once to bf16."""
    rng = np.random.default_rng(5)
    N, d, f, T = 11, 256, 700, 128
    x = rng.integers(-1, 2, (N, d)).astype(np.float32)
    x[:, 0] = 1.0
    Wg = rng.integers(-1, 2, (f, d)).astype(np.float32)
    Wg[:, 0] = rng.integers(-6, 2, f)
    Wu = rng.integers(-1, 2, (f, d)).astype(np.float32)
    Wd = rng.integers(-1, 2, (f, d)).astype(np.float32)
    to = lambda a: torch.from_numpy(a).to(cuda_dev, torch.bfloat16)  # noqa: E731
    y, tw = binding.twell_ffn_decode(to(x), to(Wg), to(Wu), to(Wd), T)
    G = oracle.gate(x, Wg)
    vals, idx, cnt = oracle.twell_pack(G, T)
    np.testing.assert_array_equal(tw.counts().cpu().numpy(), cnt.astype(np.int64))
    np.testing.assert_array_equal(binding.twell_unpack(tw).double().cpu().numpy(), np.maximum(G, 0))
    y_ref = oracle.ffn(x, Wg, Wu, Wd)
    assert np.abs(y_ref).max() < 2 ** 24
    np.testing.assert_array_equal(y.double().cpu().numpy(), oracle.round_bf16(y_ref))


def test_decode_zero_density_and_empty(cuda_dev):
    L = synthetic.uniform_layer(6, 512, 1000, 128, 0.02, seed=4)
    L.Wg_s[:, 0] = -1e4  # x[:, 0] = 1: every gate entry is negative
    t = L.torch_inputs(cuda_dev)
    y, tw = binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], 128)
    assert tw.counts().sum().item() == 0 and torch.count_nonzero(y).item() == 0
    y0, _ = binding.twell_ffn_decode(t["x"][:0], t["Wg_s"], t["Wu_s"], t["Wd_s"], 128)
    assert y0.shape == (0, 512)


def test_decode_unsupported_shape_falls_back(cuda_dev):
    """d_model above 4096 is outside the decode kernel's range: the call says so before launching,
    and the auto path falls back to gate + walk."""
    L = synthetic.uniform_layer(4, 4608, 1000, 128, 0.02, seed=8)
    t = L.torch_inputs(cuda_dev)
    with pytest.raises(binding.TwellError) as e:
        binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], 128)
    assert e.value.code == binding.TWELL_ERR_UNSUPPORTED
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=128, path="auto")
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "auto fallback")


def test_ffn_forward_auto_path(cuda_dev):
    L = synthetic.layer_1p5b(N=4)
    t = L.torch_inputs(cuda_dev)
    y_auto = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T, path="auto")
    y_dec, _ = binding.twell_ffn_decode(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], L.T)
    assert torch.equal(y_auto, y_dec)
