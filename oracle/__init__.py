"""fp64 CPU oracle for the activation-sparse gated FFN, TwELL and the hybrid format.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The library under
``activation_sparse_ffn_gate_gb300`` never imports it, and it imports nothing from there.

The arithmetic lives in ``twell_oracle.c`` (plain C loops in fp64). This module only marshals
numpy arrays into it and builds it with gcc on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twell_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

i64 = ctypes.c_int64
dbl = ctypes.c_double
vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile twell_oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_round_bf16.restype = dbl
            lib.oracle_round_bf16.argtypes = [dbl]
            lib.oracle_round_bf16_array.argtypes = [i64, vp, vp]
            lib.oracle_gate_rows.argtypes = [i64, vp, i64, i64, vp, vp, vp]
            lib.oracle_ffn_rows.argtypes = [i64, vp, i64, i64, vp, vp, vp, vp, vp, vp, vp]
            lib.oracle_twell_pack.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_twell_unpack.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_twell_walk.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp]
            lib.oracle_hybrid_route.argtypes = [i64, i64, i64, vp, i64, vp, vp, vp, vp, vp, vp]
            lib.oracle_l1.restype = dbl
            lib.oracle_l1.argtypes = [i64, i64, i64, dbl, vp, vp, vp]
            lib.oracle_ffn_bwd_rows.argtypes = [i64, vp, i64, i64, i64, dbl, vp, vp, vp, vp, vp, vp]
            lib.oracle_ffn_bwd_cols.argtypes = [i64, vp, i64, i64, i64, dbl, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.oracle_set_threads.argtypes = [i64]
            lib.oracle_max_threads.restype = i64
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, n):
    if rows is None:
        rows = np.arange(n, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= n):
        raise IndexError("row index out of range")
    return rows


# ------------------------------------------------------------------------------ rounding

def round_bf16(a):
    """Round fp64 values to the nearest bf16 value, ties to even (returned as fp64)."""
    a = _f64(a)
    out = np.empty_like(a)
    _load().oracle_round_bf16_array(a.size, _ptr(a), _ptr(out))
    return out


# ------------------------------------------------------------------------------ dense layer

def set_threads(n: int) -> None:
    """Threads the oracle's OpenMP loops use from now on (for timing: per-row results do not depend on it;
    the order in which the L1 sum adds its per-thread parts does)."""
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gate(x, Wg_s, rows=None):
    """G[rows] = x[rows] Wg_s^T in fp64."""
    x, Wg_s = _f64(x), _f64(Wg_s)
    (N, d), f = x.shape, Wg_s.shape[0]
    rows = _rows(rows, N)
    G = np.empty((rows.size, f))
    _load().oracle_gate_rows(rows.size, _ptr(rows), d, f, _ptr(x), _ptr(Wg_s), _ptr(G))
    return G


def ffn(x, Wg_s, Wu_s, Wd_s, rows=None, return_gu=False):
    """y[rows] of the ReLU-gated FFN, in fp64; optionally also G and U of those rows."""
    x, Wg_s, Wu_s, Wd_s = map(_f64, (x, Wg_s, Wu_s, Wd_s))
    (N, d), f = x.shape, Wg_s.shape[0]
    rows = _rows(rows, N)
    y = np.empty((rows.size, d))
    G = np.empty((rows.size, f)) if return_gu else None
    U = np.empty((rows.size, f)) if return_gu else None
    _load().oracle_ffn_rows(rows.size, _ptr(rows), d, f, _ptr(x), _ptr(Wg_s), _ptr(Wu_s), _ptr(Wd_s),
                            _ptr(y), _ptr(G) if return_gu else None, _ptr(U) if return_gu else None)
    return (y, G, U) if return_gu else y


# ------------------------------------------------------------------------------ TwELL

def twell_pack(G, T):
    """TwELL pack of G [N, f]: returns (vals [N, nt, T] fp64, idx [N, nt, T] u8, cnt [N, nt] u16).

    Slots past cnt are NaN in vals and 0xFF in idx (never written by the pack)."""
    G = _f64(G)
    N, f = G.shape
    nt = -(-f // T)
    vals = np.full((N, nt, T), np.nan)
    idx = np.full((N, nt, T), 0xFF, dtype=np.uint8)
    cnt = np.zeros((N, nt), dtype=np.uint16)
    _load().oracle_twell_pack(N, f, T, _ptr(G), _ptr(vals), _ptr(idx), _ptr(cnt))
    return vals, idx, cnt


def twell_unpack(vals, idx, cnt, f, T):
    vals = _f64(vals)
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    cnt = np.ascontiguousarray(cnt, dtype=np.uint16)
    N = cnt.shape[0]
    dense = np.empty((N, f))
    _load().oracle_twell_unpack(N, f, T, _ptr(vals), _ptr(idx), _ptr(cnt), _ptr(dense))
    return dense


def twell_walk(vals, idx, cnt, T, x, Wu_s, Wd_s):
    """y from a TwELL matrix of gate activations by the fused up+down walk (fp64)."""
    vals = _f64(vals)
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    cnt = np.ascontiguousarray(cnt, dtype=np.uint16)
    x, Wu_s, Wd_s = map(_f64, (x, Wu_s, Wd_s))
    N, d = x.shape
    f = Wu_s.shape[0]
    y = np.empty((N, d))
    _load().oracle_twell_walk(N, d, f, T, _ptr(vals), _ptr(idx), _ptr(cnt), _ptr(x), _ptr(Wu_s),
                              _ptr(Wd_s), _ptr(y))
    return y


# ------------------------------------------------------------------------------ hybrid format

def hybrid_route(G, K, backup_cap=None):
    """Hybrid routing of G [N, f] with capacity K.

    Returns dict(hval_a [N,K], hcol [N,K] u16, hcnt [N] u16, brows [n_stored] i32,
    n_backup int, A_b [n_stored, f]). Slots of overflow rows are NaN / 0xFFFF (not written)."""
    G = _f64(G)
    N, f = G.shape
    cap = N if backup_cap is None else int(backup_cap)
    hval_a = np.full((N, K), np.nan)
    hcol = np.full((N, K), 0xFFFF, dtype=np.uint16)
    hcnt = np.zeros(N, dtype=np.uint16)
    brows = np.full(max(cap, 1), -1, dtype=np.int32)
    nb = np.zeros(1, dtype=np.int32)
    A_b = np.full((max(cap, 1), f), np.nan)
    _load().oracle_hybrid_route(N, f, K, _ptr(G), cap, _ptr(hval_a), _ptr(hcol), _ptr(hcnt),
                                _ptr(brows), _ptr(nb), _ptr(A_b))
    n = int(nb[0])
    s = min(n, cap)
    return dict(hval_a=hval_a, hcol=hcol, hcnt=hcnt, brows=brows[:s].copy(), n_backup=n,
                A_b=A_b[:s].copy())


def l1(x, Wg_s, Wu_s, lam):
    """lam * mean|h| over all N*f hidden activations."""
    x, Wg_s, Wu_s = map(_f64, (x, Wg_s, Wu_s))
    (N, d), f = x.shape, Wg_s.shape[0]
    return float(_load().oracle_l1(N, d, f, lam, _ptr(x), _ptr(Wg_s), _ptr(Wu_s)))


def ffn_bwd_rows(x, Wg_s, Wu_s, Wd_s, dy, lam, rows=None):
    """dx[rows] of L = <y, dy> + lam * mean|h| (fp64)."""
    x, Wg_s, Wu_s, Wd_s, dy = map(_f64, (x, Wg_s, Wu_s, Wd_s, dy))
    (N, d), f = x.shape, Wg_s.shape[0]
    rows = _rows(rows, N)
    dx = np.empty((rows.size, d))
    _load().oracle_ffn_bwd_rows(rows.size, _ptr(rows), N, d, f, lam, _ptr(x), _ptr(Wg_s), _ptr(Wu_s),
                                _ptr(Wd_s), _ptr(dy), _ptr(dx))
    return dx


def ffn_bwd_cols(x, Wg_s, Wu_s, Wd_s, dy, lam, cols=None):
    """(dWg_s[cols], dWu_s[cols], dWd_s[cols]) of L = <y, dy> + lam * mean|h| (fp64)."""
    x, Wg_s, Wu_s, Wd_s, dy = map(_f64, (x, Wg_s, Wu_s, Wd_s, dy))
    (N, d), f = x.shape, Wg_s.shape[0]
    cols = _rows(cols, f)
    dWg = np.empty((cols.size, d))
    dWu = np.empty((cols.size, d))
    dWd = np.empty((cols.size, d))
    _load().oracle_ffn_bwd_cols(cols.size, _ptr(cols), N, d, f, lam, _ptr(x), _ptr(Wg_s), _ptr(Wu_s),
                                _ptr(Wd_s), _ptr(dy), _ptr(dWg), _ptr(dWu), _ptr(dWd))
    return dWg, dWu, dWd
