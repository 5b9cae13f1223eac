"""Pins for the fp64 CPU oracle (no GPU).

Each oracle function is checked against something other than itself: a hand-worked example
(tests/golden/hand_worked_2x2x3.json), library routines (torch's bf16 conversion), invariants
and closed forms (homogeneity, permutation and split equivariance, zero density, exact
unpack(pack) identity, routing rules), brute force with an independently written numpy
construction on tiny inputs, and central finite differences of the forward for the backward.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_ffn_gate_gb300 import synthetic

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked_2x2x3.json")))


def _arr(k):
    return np.array(GOLD[k], dtype=np.float64)


# ----------------------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(0)
    mags = rng.uniform(-140, 128, 20000)
    v = (rng.choice([-1.0, 1.0], 20000) * np.exp2(mags)).astype(np.float32)
    # exact ties between neighbouring bf16 values, at several exponents, both parities
    m = rng.integers(0, 128, 4000)
    e = rng.integers(-133, 120, 4000)
    ties = (((128 + m) * 2 + 1) * np.exp2(e - 8.0)).astype(np.float32)
    sub = (rng.integers(1, 2 ** 23, 2000) * np.exp2(-149.0)).astype(np.float32)  # fp32 subnormals
    allv = np.concatenate([v, ties, -ties, sub, -sub,
                           np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 1e-45], np.float32)])
    lib = torch.from_numpy(allv).to(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.round_bf16(allv.astype(np.float64))
    assert np.array_equal(np.signbit(ours), np.signbit(lib))
    np.testing.assert_array_equal(ours, lib)


def test_round_bf16_closed_forms():
    r = oracle.round_bf16
    one_ulp = 2.0 ** -7
    # a tie between 1 and 1+2^-7 goes to the even mantissa (1.0); just above the tie goes up
    assert r(np.array([1 + 2 ** -8]))[0] == 1.0
    assert r(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 1 + one_ulp
    assert r(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 * one_ulp  # tie, odd below -> even above
    assert r(np.array([-9999.0]))[0] == -9984.0
    assert r(np.array([2.0 ** -133]))[0] == 2.0 ** -133  # smallest bf16 subnormal
    assert r(np.array([2.0 ** -134]))[0] == 0.0  # tie with zero -> even (zero)
    assert math.isinf(r(np.array([2.0 ** 128]))[0])
    for k in range(-20, 9):  # integers up to 256 are exact
        assert r(np.array([float(k)]))[0] == k


# ----------------------------------------------------------------------------- dense layer

def test_ffn_hand_worked():
    y, G, U = oracle.ffn(_arr("x"), _arr("Wg_s"), _arr("Wu_s"), _arr("Wd_s"), return_gu=True)
    np.testing.assert_array_equal(G, _arr("G"))
    np.testing.assert_array_equal(U, _arr("U"))
    np.testing.assert_array_equal(y, _arr("y"))
    np.testing.assert_array_equal(oracle.gate(_arr("x"), _arr("Wg_s")), _arr("G"))
    np.testing.assert_array_equal(oracle.ffn(_arr("x"), _arr("Wg_s"), _arr("Wu_s"), _arr("Wd_s"),
                                             rows=[1]), _arr("y")[1:2])


def _rand_layer(seed=0, N=9, d=7, f=13):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, d)), rng.standard_normal((f, d)), rng.standard_normal((f, d)),
            rng.standard_normal((f, d)))


def test_ffn_invariants():
    x, Wg, Wu, Wd = _rand_layer()
    y = oracle.ffn(x, Wg, Wu, Wd)
    assert np.abs(y).max() > 0.1
    # positive homogeneity of ReLU in Wg, linearity in Wu and in Wd
    np.testing.assert_allclose(oracle.ffn(x, 2.5 * Wg, Wu, Wd), 2.5 * y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.ffn(x, Wg, -3.0 * Wu, Wd), -3.0 * y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.ffn(x, Wg, Wu, 0.5 * Wd), 0.5 * y, rtol=1e-12, atol=1e-12)
    # a negative gate scale changes the support: result differs
    assert not np.allclose(oracle.ffn(x, -Wg, Wu, Wd), -y)
    # hidden units are interchangeable: permuting rows of all three weights leaves y unchanged
    p = np.random.default_rng(1).permutation(Wg.shape[0])
    np.testing.assert_allclose(oracle.ffn(x, Wg[p], Wu[p], Wd[p]), y, rtol=1e-12, atol=1e-12)
    # tokens are independent: permuting tokens permutes y
    q = np.random.default_rng(2).permutation(x.shape[0])
    np.testing.assert_allclose(oracle.ffn(x[q], Wg, Wu, Wd), y[q], rtol=1e-12, atol=1e-12)
    # the hidden dimension splits additively
    s = 5
    y2 = oracle.ffn(x, Wg[:s], Wu[:s], Wd[:s]) + oracle.ffn(x, Wg[s:], Wu[s:], Wd[s:])
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-12)
    # zero density: a hugely negative bias column switches every gate off -> y == 0 exactly
    x1 = x.copy()
    x1[:, 0] = 1.0
    Wg1 = Wg.copy()
    Wg1[:, 0] = -1e6
    assert np.array_equal(oracle.ffn(x1, Wg1, Wu, Wd), np.zeros_like(y))
    # all gates on: then y is the (unmasked) bilinear form; check it on one scalar hidden unit
    Wg1[:, 0] = 1e6
    y_on = oracle.ffn(x1, Wg1[:1], Wu[:1], Wd[:1])
    g = x1 @ Wg1[0]
    u = x1 @ Wu[0]
    np.testing.assert_allclose(y_on, np.outer(g * u, Wd[0]), rtol=1e-12)


def test_ffn_rows_subset_matches_full():
    x, Wg, Wu, Wd = _rand_layer(3)
    y = oracle.ffn(x, Wg, Wu, Wd)
    rows = [8, 0, 3, 3]
    np.testing.assert_array_equal(oracle.ffn(x, Wg, Wu, Wd, rows=rows), y[rows])


# ----------------------------------------------------------------------------- TwELL

def test_pack_hand_worked():
    vals, idx, cnt = oracle.twell_pack(_arr("G"), 2)
    gold = GOLD["twell_T2"]
    np.testing.assert_array_equal(cnt, np.array(gold["cnt"]))
    for key, v in gold["vals"].items():
        r, t = map(int, key.split(","))
        n = len(v)
        np.testing.assert_array_equal(vals[r, t, :n], v)
        np.testing.assert_array_equal(idx[r, t, :n], gold["idx"][key])
    # slots past cnt are never written
    assert np.isnan(vals[0, 1]).all() and (idx[0, 1] == 0xFF).all()
    assert np.isnan(vals[1, 0, 1:]).all()


def _brute_pack(G, T):
    """Independent construction: np.nonzero per tile."""
    N, f = G.shape
    nt = -(-f // T)
    out = {}
    for r in range(N):
        for t in range(nt):
            seg = G[r, t * T:min(f, (t + 1) * T)]
            k = np.nonzero(seg > 0)[0]
            out[(r, t)] = (k, seg[k])
    return out


@pytest.mark.parametrize("T,f", [(64, 300), (128, 1024), (256, 700), (2, 5)])
def test_pack_bruteforce_and_invariants(T, f):
    rng = np.random.default_rng(T + f)
    N = 37
    G = rng.standard_normal((N, f)) - 1.2
    G[0] = -1.0  # empty row
    G[1] = 1.0  # full row
    G[2, ::3] = -0.0  # negative zeros are not kept
    G[3, :] = 0.0
    vals, idx, cnt = oracle.twell_pack(G, T)
    nt = -(-f // T)
    assert cnt.shape == (N, nt)
    brute = _brute_pack(G, T)
    for (r, t), (k, v) in brute.items():
        c = cnt[r, t]
        assert c == len(k)
        np.testing.assert_array_equal(idx[r, t, :c], k)
        np.testing.assert_array_equal(vals[r, t, :c], v)
    # per-row counts sum to the row's nonzero count; indices ascending and inside the tile
    np.testing.assert_array_equal(cnt.sum(1), (G > 0).sum(1))
    for r in range(N):
        for t in range(nt):
            c = cnt[r, t]
            assert np.all(np.diff(idx[r, t, :c].astype(int)) > 0)
            assert np.all(t * T + idx[r, t, :c].astype(int) < f)
    # unpack(pack(ReLU(G))) == ReLU(G) exactly
    dense = oracle.twell_unpack(vals, idx, cnt, f, T)
    assert np.array_equal(dense, np.where(G > 0, G, 0.0))
    assert cnt[0].sum() == 0 and cnt[1].sum() == f and cnt[3].sum() == 0


def test_walk_equals_dense_definition():
    L = synthetic.tiny_fp32()
    x, Wg, Wu, Wd = (L.x.astype(np.float64), L.Wg_s.astype(np.float64), L.Wu_s.astype(np.float64),
                     L.Wd_s.astype(np.float64))
    y, G, _ = oracle.ffn(x, Wg, Wu, Wd, return_gu=True)
    vals, idx, cnt = oracle.twell_pack(G, L.T)
    yw = oracle.twell_walk(vals, idx, cnt, L.T, x, Wu, Wd)
    rel = np.linalg.norm(yw - y) / np.linalg.norm(y)
    assert rel <= 1e-12
    # hand example through the walk
    v2, i2, c2 = oracle.twell_pack(_arr("G"), 2)
    np.testing.assert_array_equal(oracle.twell_walk(v2, i2, c2, 2, _arr("x"), _arr("Wu_s"), _arr("Wd_s")),
                                  _arr("y"))


# ----------------------------------------------------------------------------- hybrid routing

def test_route_hand_worked():
    r2 = oracle.hybrid_route(_arr("G"), 2)
    g2 = GOLD["hybrid_K2"]
    np.testing.assert_array_equal(r2["hcnt"], g2["hcnt"])
    np.testing.assert_array_equal(r2["hcol"], g2["hcol"])
    np.testing.assert_array_equal(r2["hval_a"], g2["hval_a"])
    assert r2["n_backup"] == 0
    r1 = oracle.hybrid_route(_arr("G"), 1)
    g1 = GOLD["hybrid_K1"]
    np.testing.assert_array_equal(r1["hcnt"], g1["hcnt"])
    np.testing.assert_array_equal(r1["brows"], g1["brows"])
    np.testing.assert_array_equal(r1["A_b"], g1["A_b"])
    assert r1["n_backup"] == 2


@pytest.mark.parametrize("K", [0, 1, 5, 16, 2000])
def test_route_invariants(K):
    rng = np.random.default_rng(K)
    N, f = 120, 700
    dens = np.exp(rng.standard_normal(N)) * 0.01
    G = np.where(rng.random((N, f)) < dens[:, None], rng.random((N, f)) + 0.1, -rng.random((N, f)))
    G[5] = -1.0  # empty row
    nnz = (G > 0).sum(1)
    R = oracle.hybrid_route(G, K)
    over = nnz > K
    # each row is in exactly one of block / backup; the backup holds exactly the rows with nnz > K
    assert R["n_backup"] == over.sum()
    np.testing.assert_array_equal(R["brows"], np.nonzero(over)[0])  # ascending row order
    np.testing.assert_array_equal(R["hcnt"][over], 0xFFFF)
    np.testing.assert_array_equal(R["hcnt"][~over], nnz[~over])
    for i, r in enumerate(R["brows"]):
        np.testing.assert_array_equal(R["A_b"][i], np.maximum(G[r], 0.0))
    for r in np.nonzero(~over)[0]:
        c = nnz[r]
        cols = np.nonzero(G[r] > 0)[0]
        np.testing.assert_array_equal(R["hcol"][r, :c], cols)
        np.testing.assert_array_equal(R["hval_a"][r, :c], G[r, cols])
        assert np.all(R["hval_a"][r, c:] == 0.0) and np.all(R["hcol"][r, c:] == 0)
        assert not np.any(np.signbit(R["hval_a"][r, c:]))
    if K == 0:
        assert R["n_backup"] == (nnz > 0).sum()
    if K >= f:
        assert R["n_backup"] == 0


def test_route_backup_capacity_counts_all():
    G = np.ones((6, 4))
    G[2] = -1
    R = oracle.hybrid_route(G, 1, backup_cap=3)
    assert R["n_backup"] == 5
    np.testing.assert_array_equal(R["brows"], [0, 1, 3])


# ----------------------------------------------------------------------------- L1 and backward

def test_l1_hand_worked():
    assert oracle.l1(_arr("x"), _arr("Wg_s"), _arr("Wu_s"), 1.0) == GOLD["sum_abs_h"] / 6.0
    assert oracle.l1(_arr("x"), _arr("Wg_s"), _arr("Wu_s"), 6.0) == GOLD["grads_lambda6"]["l1"]


@pytest.mark.parametrize("key,lam", [("grads_lambda0", 0.0), ("grads_lambda6", 6.0)])
def test_backward_hand_worked(key, lam):
    g = GOLD[key]
    args = (_arr("x"), _arr("Wg_s"), _arr("Wu_s"), _arr("Wd_s"), _arr("dy"), lam)
    np.testing.assert_array_equal(oracle.ffn_bwd_rows(*args), g["dx"])
    dWg, dWu, dWd = oracle.ffn_bwd_cols(*args)
    np.testing.assert_array_equal(dWg, g["dWg_s"])
    np.testing.assert_array_equal(dWu, g["dWu_s"])
    np.testing.assert_array_equal(dWd, g["dWd_s"])


def _loss(x, Wg, Wu, Wd, dy, lam):
    return float((oracle.ffn(x, Wg, Wu, Wd) * dy).sum()) + oracle.l1(x, Wg, Wu, lam)


@pytest.mark.parametrize("lam", [0.0, 0.7])
def test_backward_central_differences(lam):
    """Gradients of L = <y, dy> + lam * mean|h| against central differences of the forward."""
    rng = np.random.default_rng(11)
    N, d, f = 6, 5, 9
    x, Wg, Wu, Wd = _rand_layer(11, N, d, f)
    dy = rng.standard_normal((N, d))
    G = x @ Wg.T
    U = x @ Wu.T
    # stay away from the kinks of ReLU (g = 0) and |h| (u = 0 where g > 0)
    assert np.abs(G).min() > 1e-3 and np.abs(U[G > 0]).min() > 1e-3
    dx = oracle.ffn_bwd_rows(x, Wg, Wu, Wd, dy, lam)
    dWg, dWu, dWd = oracle.ffn_bwd_cols(x, Wg, Wu, Wd, dy, lam)
    eps = 1e-6
    for name, arr, grad in (("x", x, dx), ("Wg", Wg, dWg), ("Wu", Wu, dWu), ("Wd", Wd, dWd)):
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            keep = arr[i]
            arr[i] = keep + eps
            lp = _loss(x, Wg, Wu, Wd, dy, lam)
            arr[i] = keep - eps
            lm = _loss(x, Wg, Wu, Wd, dy, lam)
            arr[i] = keep
            num[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=name)


def test_backward_subsets_match_full():
    rng = np.random.default_rng(5)
    x, Wg, Wu, Wd = _rand_layer(5, 8, 6, 10)
    dy = rng.standard_normal((8, 6))
    dx = oracle.ffn_bwd_rows(x, Wg, Wu, Wd, dy, 0.3)
    np.testing.assert_array_equal(oracle.ffn_bwd_rows(x, Wg, Wu, Wd, dy, 0.3, rows=[7, 2]), dx[[7, 2]])
    full = oracle.ffn_bwd_cols(x, Wg, Wu, Wd, dy, 0.3)
    part = oracle.ffn_bwd_cols(x, Wg, Wu, Wd, dy, 0.3, cols=[9, 0])
    for a, b in zip(full, part):
        np.testing.assert_array_equal(a[[9, 0]], b)


def test_backward_torch_autograd_crosscheck():
    """Extra cross-check against torch fp64 autograd of the dense formula (a library routine)."""
    rng = np.random.default_rng(7)
    x, Wg, Wu, Wd = _rand_layer(7, 10, 8, 12)
    dy = rng.standard_normal((10, 8))
    lam = 0.37
    t = [torch.tensor(a, requires_grad=True) for a in (x, Wg, Wu, Wd)]
    G = t[0] @ t[1].T
    H = torch.relu(G) * (t[0] @ t[2].T)
    L = ((H @ t[3]) * torch.tensor(dy)).sum() + lam * H.abs().mean()
    L.backward()
    dx = oracle.ffn_bwd_rows(x, Wg, Wu, Wd, dy, lam)
    dWg, dWu, dWd = oracle.ffn_bwd_cols(x, Wg, Wu, Wd, dy, lam)
    for ours, ref in ((dx, t[0].grad), (dWg, t[1].grad), (dWu, t[2].grad), (dWd, t[3].grad)):
        np.testing.assert_allclose(ours, ref.numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------- synthetic inputs

def test_tiny_layer_density_matches_construction():
    """The 2%-density tiny layer realises P(g > 0) = Phi(-tau) within a 4-sigma binomial band."""
    L = synthetic.tiny_fp32()
    G = oracle.gate(L.x, L.Wg_s)
    n = G.size
    p = 0.02
    k = (G > 0).sum()
    assert abs(k - n * p) <= 4 * math.sqrt(n * p * (1 - p))


def test_1p5b_layer_statistics():
    """29 nonzeros per token (pulsen ¶4) and 30% dead columns (pulsen ¶5), on a row sample."""
    L = synthetic.layer_1p5b(N=256)
    G = torch.from_numpy(L.x).double() @ torch.from_numpy(L.Wg_s).double().T
    nnz = (G > 0).sum(1).double()
    assert abs(nnz.mean().item() - 29.0) < 4 * math.sqrt(29.0 / 256)
    dead = (L.Wg_s[:, 0] < -9000).sum()
    assert dead == round(0.3 * L.f)
    assert not (G[:, torch.from_numpy(L.Wg_s[:, 0] < -9000)] > 0).any()


def test_train_layer_overflow_fraction():
    """About 1-3% of rows overflow K = 64 under the training generator (2B shapes)."""
    L = synthetic.train_2b(N=2048)
    G = torch.from_numpy(L.x).double() @ torch.from_numpy(L.Wg_s).double().T
    nnz = (G > 0).sum(1)
    frac = (nnz > L.K).double().mean().item()
    assert 0.01 <= frac <= 0.04, frac
