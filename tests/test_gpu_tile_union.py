"""GPU parity of twell_ffn_tile_union_fwd (tensor-core GEMMs over each 128-token tile's union of
kept units, with gathered weight rows) against the fp64 oracle, through the C ABI.

Cases: ragged token counts (a last tile of 44 rows), tile widths 64 / 128 / 256, fp32 and bf16
packed values, d_model not a multiple of 256 (a partial N-block in the down GEMM), d_ff not a
multiple of 256 (a partial union block), zero density (y == 0 exactly), every unit kept, the sweep
shapes at N = 1024, and the 1.5B-like / 2B-like layers at full size on sampled rows (the densest
rows included). Tolerances as everywhere: rel-Frobenius <= 5e-3, max-abs <= 2e-2 x RMS per row.
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


def _run(dev, L, T=None, vals_dtype=torch.float32):
    t = L.torch_inputs(dev)
    T = T or L.T
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], T, vals_dtype=vals_dtype)
    Wd16 = binding.twell_convert_f16(t["Wd_s"])
    y = binding.twell_ffn_tile_union_fwd(t["x"], t["Wu_s"], Wd16, tw)
    torch.cuda.synchronize()
    return y, tw, t


@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("p", [0.01, 0.05])
def test_tile_union_small_ragged(cuda_dev, p, T):
    L = synthetic.uniform_layer(300, 512, 1280, T, p, seed=int(p * 1000) + T)
    y, _, _ = _run(cuda_dev, L)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"tile union p={p} T={T}")


def test_tile_union_bf16_values_partial_blocks(cuda_dev):
    """bf16 packed values; d_model 576 (the down GEMM's last N-block has 64 of 256 columns) and
    d_ff 1000 (the union's last block is partial)."""
    L = synthetic.uniform_layer(200, 576, 1000, 128, 0.02, seed=9)
    y, _, _ = _run(cuda_dev, L, vals_dtype=torch.bfloat16)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "tile union bf16 values")


def test_tile_union_zero_density(cuda_dev):
    L = synthetic.uniform_layer(260, 512, 1024, 128, 0.02, seed=4)
    L.Wg_s[:, 0] = -1e4  # no gate fires: every union is empty
    y, tw, _ = _run(cuda_dev, L)
    assert int(tw.counts().sum().item()) == 0
    assert torch.count_nonzero(y).item() == 0


def test_tile_union_every_unit_kept(cuda_dev):
    """Every gate on: the union of every tile is all of d_ff and y is the plain ReLU FFN with a = g."""
    L = synthetic.uniform_layer(256, 512, 768, 128, 0.5, seed=5)
    L.Wg_s[:, 0] = 1e4
    y, _, _ = _run(cuda_dev, L)
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "tile union all kept")


def test_tile_union_matches_the_walk_on_one_row_tiles(cuda_dev):
    """Batches below one tile (N = 1, 7, 129): the union path and the walk agree with the oracle."""
    for N in (1, 7, 129):
        L = synthetic.uniform_layer(N, 512, 1024, 128, 0.03, seed=N)
        y, tw, t = _run(cuda_dev, L)
        assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), f"tile union N={N}")


def test_tile_union_empty_batch(cuda_dev):
    L = synthetic.uniform_layer(4, 512, 1024, 128, 0.02, seed=1)
    t = L.torch_inputs(cuda_dev)
    x = t["x"][:0]
    tw = binding.twell_gate_pack(x, t["Wg_s"], 128)
    y = binding.twell_ffn_tile_union_fwd(x, t["Wu_s"], binding.twell_convert_f16(t["Wd_s"]), tw)
    assert y.shape == (0, 512)


def _sampled_rows(N, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, N - 1], rng.choice(N, n, replace=False), np.asarray(extra, dtype=np.int64)]))


@pytest.mark.parametrize("p", [0.001, 0.005, 0.01, 0.02, 0.1])
def test_tile_union_sweep_shapes_sampled(cuda_dev, p):
    """The sweep's shapes (d_model 2048, d_ff 5632, T = 128) at N = 1024, on sampled rows."""
    L = synthetic.sweep_point(p, 128, N=1024)
    y, _, _ = _run(cuda_dev, L)
    rows = _sampled_rows(L.N, 16, seed=int(p * 1e4))
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"tile union sweep p={p}")


@pytest.mark.parametrize("which", ["1.5b", "2b"])
def test_tile_union_full_size_layers_sampled(cuda_dev, which):
    """The bench's workloads at full size on sampled rows plus the eight densest rows."""
    L = synthetic.layer_1p5b() if which == "1.5b" else synthetic.layer_2b()
    y, tw, _ = _run(cuda_dev, L)
    longest = torch.argsort(tw.counts().sum(1), descending=True)[:8].cpu().numpy()
    rows = _sampled_rows(L.N, 24, seed=2, extra=longest)
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    assert_close(y[torch.from_numpy(rows).to(cuda_dev)].double().cpu().numpy(), y_ref, f"tile union {which}")


def test_count_nonzeros_matches_the_counts(cuda_dev):
    L = synthetic.uniform_layer(300, 512, 1280, 128, 0.03, seed=17)
    t = L.torch_inputs(cuda_dev)
    tw = binding.twell_gate_pack(t["x"], t["Wg_s"], 128)
    total = binding.twell_count_nonzeros(tw)
    assert int(total.item()) == int(tw.counts().sum().item())
    binding.twell_count_nonzeros(tw, total=total)  # adds to what is there
    assert int(total.item()) == 2 * int(tw.counts().sum().item())


def test_auto_path_follows_the_density(cuda_dev):
    """ffn_forward(path="auto"): with a density above the crossover and the transposed fp16 Wd_s the
    union path runs (same y as calling it directly), below it the walk; without Wd16t_s the walk.
    The tile-union path is called by name."""
    L = synthetic.uniform_layer(400, 512, 1280, 128, 0.03, seed=23)
    t = L.torch_inputs(cuda_dev)
    Wd16 = binding.twell_convert_f16(t["Wd_s"])
    Wd16t = binding.twell_convert_f16_transposed(t["Wd_s"])
    args = (t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"])
    y_union = binding.ffn_forward(*args, T=128, path="union", Wd16t_s=Wd16t)
    y_tu = binding.ffn_forward(*args, T=128, path="tile_union", Wd16_s=Wd16)
    y_walk = binding.ffn_forward(*args, T=128, path="walk")
    y_auto_hi = binding.ffn_forward(*args, T=128, path="auto", Wd16t_s=Wd16t, density=0.03)
    y_auto_lo = binding.ffn_forward(*args, T=128, path="auto", Wd16t_s=Wd16t, density=0.001)
    y_auto_no16 = binding.ffn_forward(*args, T=128, path="auto", Wd16_s=Wd16, density=0.03)
    assert torch.equal(y_auto_hi, y_union)
    assert torch.equal(y_auto_lo, y_walk)
    assert torch.equal(y_auto_no16, y_walk)
    ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s)
    assert_close(y_tu.double().cpu().numpy(), ref, "tile union")
    assert_close(y_union.double().cpu().numpy(), ref, "union")
    for path in ("tile_union", "union"):
        with pytest.raises(ValueError):
            binding.ffn_forward(*args, T=128, path=path)
