"""GPU parity of the hybrid (sparse block + dense backup) training path against the fp64 oracle.

- twell_gemm_test: the tcgen05 GEMM used for the backup rows, for all four operand layouts,
  exact on integer-valued inputs (fp32 accumulation is exact there);
- twell_hybrid_route_from_gate: bit-exact routing against the oracle's hybrid_route on the same
  gate matrix (sparse block, backup rows in ascending order, dense backup rows), incl. K = 0,
  K >= d_ff and a backup buffer that is too small;
- twell_hybrid_fwd / twell_hybrid_bwd: y, the L1 term, dx, dWg, dWu, dWd against the oracle's
  dense definition (rel-Frobenius <= 5e-3, max-abs <= 2e-2 * RMS per output row), on small layers
  and on sampled rows / hidden units of the full-size training layer.
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


def _to(dev, a, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)


# ------------------------------------------------------------------------------------------ GEMM

@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 264, 136), (384, 520, 1000), (64, 8, 8)])
def test_gemm_layouts_integer_exact(cuda_dev, a_mn, b_mn, M, N, K):
    rng = np.random.default_rng(M + N + K + 2 * a_mn + b_mn)
    A = rng.integers(-2, 3, (M, K)).astype(np.float32)
    B = rng.integers(-2, 3, (K, N)).astype(np.float32)
    A_st = A.T.copy() if a_mn else A  # [K, M] if MN-major
    B_st = B if b_mn else B.T.copy()  # [N, K] if K-major
    C = binding.twell_gemm_test(_to(cuda_dev, A_st), _to(cuda_dev, B_st), bool(a_mn), bool(b_mn))
    np.testing.assert_array_equal(C.double().cpu().numpy(), A.astype(np.float64) @ B.astype(np.float64))
    assert binding.twell_read_status() == 0


# ------------------------------------------------------------------------------------------ routing

def _gate_with_row_spread(N, f, seed):
    rng = np.random.default_rng(seed)
    dens = np.minimum(0.002 * np.exp(1.3 * rng.standard_normal(N)), 0.8)
    dens[::17] *= 20
    G = np.where(rng.random((N, f)) < np.minimum(dens, 0.9)[:, None], rng.random((N, f)) + 0.01,
                 -rng.random((N, f)))
    G[3] = -1.0
    return synthetic.round_bf16_np(G.astype(np.float32))


def _check_route(ctx, R, K, cap, G):
    hcnt = ctx.counts().cpu().numpy()
    np.testing.assert_array_equal(hcnt, R["hcnt"].astype(np.int64))
    light = R["hcnt"] != 0xFFFF
    if K > 0:
        np.testing.assert_array_equal(ctx.cols().cpu().numpy()[light], R["hcol"][light].astype(np.int64))
        np.testing.assert_array_equal(ctx.a.double().cpu().numpy()[light], R["hval_a"][light])
    nb = int(ctx.n_backup.item())
    assert nb == R["n_backup"]
    s = min(nb, cap)
    np.testing.assert_array_equal(ctx.backup_rows[:s].cpu().numpy(), R["brows"][:s])
    np.testing.assert_array_equal(ctx.A_b[:s].double().cpu().numpy(), R["A_b"][:s])


@pytest.mark.parametrize("K", [0, 4, 16, 64, 3000])
def test_route_bit_exact(cuda_dev, K):
    N, f = 700, 2048
    G = _gate_with_row_spread(N, f, K)
    R = oracle.hybrid_route(G.astype(np.float64), K)
    cap = max(R["n_backup"], 1)
    ctx = binding.twell_hybrid_route_from_gate(_to(cuda_dev, G), K, cap)
    assert binding.twell_read_status(ctx.status) == 0
    _check_route(ctx, R, K, cap, G)
    if K == 0:
        assert R["n_backup"] == (G > 0).any(1).sum()
    if K >= f:
        assert R["n_backup"] == 0


def test_route_backup_full_is_reported(cuda_dev):
    N, f, K = 500, 1024, 4
    G = _gate_with_row_spread(N, f, 7)
    R = oracle.hybrid_route(G.astype(np.float64), K)
    assert R["n_backup"] > 10
    cap = R["n_backup"] // 2
    ctx = binding.twell_hybrid_route_from_gate(_to(cuda_dev, G), K, cap)
    code = binding.twell_read_status(ctx.status)
    assert code == 3  # TWELL_ERR_BACKUP_FULL
    _check_route(ctx, R, K, cap, G)


# ------------------------------------------------------------------------------------------ forward / backward

def _run_hybrid(dev, L, cap):
    t = L.torch_inputs(dev)
    y, ctx = binding.twell_hybrid_fwd(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], L.K, cap, L.l1_coef)
    dx, dWg, dWu, dWd = binding.twell_hybrid_bwd(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], ctx, t["dy"], L.l1_coef)
    torch.cuda.synchronize()
    return y, ctx, dx, dWg, dWu, dWd


@pytest.mark.parametrize("K,base", [(16, 0.01), (4, 0.02), (64, 0.02)])
def test_hybrid_small_all_outputs(cuda_dev, K, base):
    L = synthetic.small_train(seed=K, N=300, d=256, f=1024, K=K, base=base, bf16=True)
    _check_all_outputs(cuda_dev, L)


@pytest.mark.parametrize("d", [512, 1024, 2048, 2560])
def test_hybrid_tensor_core_light_rows(cuda_dev, d):
    """Every d_model the tensor-core light-row walk serves, with light rows longer than one
    32-entry segment, light rows without entries and backup rows: all outputs against the oracle."""
    L = synthetic.small_train(seed=d, N=400, d=d, f=2048, K=48, base=0.012, bf16=True)
    L.x[[5, 17, 200], 0] = 50.0  # threshold far above every gate: rows without entries
    nnz = (oracle.gate(L.x, L.Wg_s) > 0).sum(1)
    assert (nnz == 0).sum() >= 3 and ((nnz > 32) & (nnz <= 48)).sum() >= 5
    _check_all_outputs(cuda_dev, L)


def _check_all_outputs(cuda_dev, L):
    K = L.K
    G = oracle.gate(L.x, L.Wg_s)
    n_over = ((G > 0).sum(1) > K).sum()
    assert n_over > 0  # the dense backup path is exercised
    y, ctx, dx, dWg, dWu, dWd = _run_hybrid(cuda_dev, L, cap=n_over + 8)
    assert binding.twell_read_status(ctx.status) == 0
    nb = int(ctx.n_backup.item())
    assert abs(nb - n_over) <= 2  # rows at the K boundary may flip on |g| at rounding level
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s)
    assert_close(y.double().cpu().numpy(), y_ref, "hybrid y")
    l1_ref = oracle.l1(L.x, L.Wg_s, L.Wu_s, L.l1_coef)
    assert abs(ctx.l1.item() - l1_ref) <= 5e-3 * abs(l1_ref)
    dx_ref = oracle.ffn_bwd_rows(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef)
    assert_close(dx.double().cpu().numpy(), dx_ref, "hybrid dx")
    rg, ru, rd = oracle.ffn_bwd_cols(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef)
    live = np.abs(rd).sum(1) > 0  # hidden units that fire somewhere
    for name, got, ref in (("dWg", dWg, rg), ("dWu", dWu, ru), ("dWd", dWd, rd)):
        g = got.double().cpu().numpy()
        # units that never fire in fp64 may fire at rounding level in fp32: then only tiny values
        assert np.abs(g[~live]).max(initial=0.0) <= 1e-3 * np.sqrt((ref[live] ** 2).mean()), name
        assert_close(g[live], ref[live], "hybrid " + name)


def test_hybrid_no_backup_rows(cuda_dev):
    """K large enough that every row is light: the dense path is skipped entirely."""
    L = synthetic.small_train(seed=3, N=130, d=256, f=512, K=512, base=0.01, bf16=True)
    y, ctx, dx, dWg, dWu, dWd = _run_hybrid(cuda_dev, L, cap=4)
    assert int(ctx.n_backup.item()) == 0
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "y")
    assert_close(dx.double().cpu().numpy(), oracle.ffn_bwd_rows(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef), "dx")


def test_hybrid_all_rows_backup(cuda_dev):
    """K = 0: every row with a nonzero goes to the dense backup (tensor-core path only)."""
    L = synthetic.small_train(seed=5, N=200, d=256, f=512, K=0, base=0.01, bf16=True)
    y, ctx, dx, dWg, dWu, dWd = _run_hybrid(cuda_dev, L, cap=200)
    assert binding.twell_read_status(ctx.status) == 0
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "y")
    assert_close(dx.double().cpu().numpy(), oracle.ffn_bwd_rows(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef), "dx")
    rg, ru, rd = oracle.ffn_bwd_cols(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef)
    live = np.abs(rd).sum(1) > 0
    for name, got, ref in (("dWg", dWg, rg), ("dWu", dWu, ru), ("dWd", dWd, rd)):
        assert_close(got.double().cpu().numpy()[live], ref[live], name)


def _heaviest_units(dev, L, n):
    """The n hidden units kept by the most tokens (from the library's own gate pack and column
    counts: a choice of what to check, not an expected value)."""
    t = L.torch_inputs(dev)
    counts = binding.twell_column_activity(binding.twell_gate_pack(t["x"], t["Wg_s"], 128))
    return torch.argsort(counts, descending=True)[:n].cpu().numpy()


def _check_sampled(cuda_dev, L, cap, overflow_lo, overflow_hi, n_rows, n_cols, seed):
    """y, dx on sampled rows (backup rows forced in) and dWg, dWu, dWd on sampled and on the
    heaviest hidden units, against the oracle."""
    y, ctx, dx, dWg, dWu, dWd = _run_hybrid(cuda_dev, L, cap=cap)
    assert binding.twell_read_status(ctx.status) == 0
    nb = int(ctx.n_backup.item())
    assert overflow_lo * L.N <= nb <= overflow_hi * L.N, nb / L.N
    rng = np.random.default_rng(seed)
    brows = ctx.backup_rows[:nb].cpu().numpy()
    rows = np.unique(np.concatenate([[0, 1, L.N - 1], rng.choice(L.N, n_rows, replace=False), brows[:6]]))
    y_ref = oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows)
    sel = torch.from_numpy(rows).to(cuda_dev)
    assert_close(y[sel].double().cpu().numpy(), y_ref, "y (sampled rows)")
    dx_ref = oracle.ffn_bwd_rows(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef, rows=rows)
    assert_close(dx[sel].double().cpu().numpy(), dx_ref, "dx (sampled rows)")
    heavy = _heaviest_units(cuda_dev, L, n_cols)
    cols = np.unique(np.concatenate([rng.choice(L.f, n_cols, replace=False), heavy]))
    rg, ru, rd = oracle.ffn_bwd_cols(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef, cols=cols)
    csel = torch.from_numpy(cols).to(cuda_dev)
    for name, got, ref in (("dWg", dWg, rg), ("dWu", dWu, ru), ("dWd", dWd, rd)):
        assert_close(got[csel].double().cpu().numpy(), ref, name + " (sampled and heaviest hidden units)")
    return ctx, nb


def test_hybrid_full_size_training_layer_sampled(cuda_dev):
    """The 2B-like training step (N=16384, d=2560, f=6912, K=64) on sampled rows and hidden units
    (8 random, 8 kept by the most tokens)."""
    _check_sampled(cuda_dev, synthetic.train_2b(), 2048, 0.01, 0.04, 12, 8, seed=3)


def test_hybrid_full_size_literal_density_sampled(cuda_dev):
    """The training step on the 2B-like layer's own generator (mean density 0.5%, lognormal per
    token, 10x on the first four positions of each sequence): ~13% of rows overflow K = 64, so the
    dense backup carries the heavy case. Sampled rows (backup rows forced in) and hidden units."""
    _check_sampled(cuda_dev, synthetic.train_2b(literal=True), 16384 // 4, 0.08, 0.2, 10, 8, seed=4)


def test_hybrid_training_layer_full_width_l1_and_all_rows(cuda_dev):
    """The 2B-like training layer's widths (d=2560, f=6912, K=64) on N = 2048 tokens: the L1 term
    against the oracle's (reduced over all N*f hidden activations), y and dx on sampled rows
    (backup rows forced in), and the weight gradients of the 8 heaviest units."""
    L = synthetic.train_2b(N=2048)
    y, ctx, dx, dWg, dWu, dWd = _run_hybrid(cuda_dev, L, cap=2048 // 4)
    assert binding.twell_read_status(ctx.status) == 0
    nb = int(ctx.n_backup.item())
    assert nb > 0
    l1_ref = oracle.l1(L.x, L.Wg_s, L.Wu_s, L.l1_coef)
    assert abs(ctx.l1.item() - l1_ref) <= 5e-3 * abs(l1_ref), (ctx.l1.item(), l1_ref)
    rng = np.random.default_rng(8)
    brows = ctx.backup_rows[:nb].cpu().numpy()
    rows = np.unique(np.concatenate([rng.choice(L.N, 64, replace=False), brows[:16]]))
    sel = torch.from_numpy(rows).to(cuda_dev)
    assert_close(y[sel].double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s, rows=rows), "y (sampled rows)")
    dx_ref = oracle.ffn_bwd_rows(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef, rows=rows)
    assert_close(dx[sel].double().cpu().numpy(), dx_ref, "dx (sampled rows)")
    cols = _heaviest_units(cuda_dev, L, 8)
    rg, ru, rd = oracle.ffn_bwd_cols(L.x, L.Wg_s, L.Wu_s, L.Wd_s, L.dy, L.l1_coef, cols=cols)
    csel = torch.from_numpy(cols).to(cuda_dev)
    for name, got, ref in (("dWg", dWg, rg), ("dWu", dWu, ru), ("dWd", dWd, rd)):
        assert_close(got[csel].double().cpu().numpy(), ref, name + " (heaviest hidden units)")
