"""Seeded synthetic layers for the activation-sparse gated FFN.

This module only builds inputs. It holds none of the layer's arithmetic (no gate, no
packing, no FFN product): both the CUDA path and the CPU oracle take their inputs from
here, and from nowhere else.

The pages measure on trained 0.5B-2B models over fineweb (pulsen.vercel.app, "Sakana AI og
NVIDIA introduserer TwELL", paragraphs 1 and 4), which are not available here. These seeded
layers stand in for them. They copy the statistics the pages report: about 29 nonzero gate
activations per token out of d_ff, i.e. ~99.5% sparsity (pulsen, paragraph 4); more than 30% of
gate columns permanently dead (pulsen, paragraph 5); 5 vs 500 active neurons between tokens
(Tencent Cloud article "一文读懂 NVIDIA 与 Sakana AI 联手打造的稀疏 LLM 黑科技", §3); and the first
tokens of a sequence being the densest (same article, §5).

Construction, shared by every preset (weights are stored one row per hidden unit, [d_ff, d_model]):

* ``x[:, 1:] ~ N(0, 1)`` and ``x[:, 0]`` is a bias feature (1, or a per-token threshold).
* ``Wg_s, Wu_s ~ N(0, 1/d_model)`` and ``Wd_s ~ N(0, 1/d_ff)``: std = 1/sqrt(fan_in).
* All values are drawn in float32 and rounded to bf16 (round to nearest even), except in the
  fp32 preset.
* ``sigma_j = sqrt(sum_{i>=1} Wg_s[j, i]^2)`` from the rounded weights, and the bias column
  ``Wg_s[j, 0] = -tau * sigma_j``. The gate pre-activation of a token is then
  ``g ~ N(-tau*sigma_j, sigma_j^2)`` and ``P(g > 0) = Phi(-tau)``, so ``tau = Phi^{-1}(1 - p)``
  sets the density ``p``.
"""
from __future__ import annotations

import dataclasses
import math
from statistics import NormalDist
from typing import Optional

import numpy as np
import torch

_ND = NormalDist()


def tau_for_density(p: float) -> float:
    """Threshold tau with P(N(0,1) > tau) = p."""
    return _ND.inv_cdf(1.0 - p)


def round_bf16_np(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) and return them as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


@dataclasses.dataclass
class Layer:
    """One synthetic FFN layer plus the token batch it is run on.

    All arrays are float32 and hold values exactly representable in ``dtype``.
    """

    name: str
    N: int
    d: int
    f: int
    T: int
    dtype: str  # "bf16" or "f32"
    x: np.ndarray  # [N, d]
    Wg_s: np.ndarray  # [f, d]
    Wu_s: np.ndarray  # [f, d]
    Wd_s: np.ndarray  # [f, d]
    dy: Optional[np.ndarray] = None  # [N, d] upstream gradient (training presets)
    K: Optional[int] = None  # hybrid per-row capacity (training presets)
    l1_coef: float = 2e-5
    target_density: float = 0.0
    recipe: str = ""

    def torch_inputs(self, device, dtype=None):
        dt = dtype or (torch.bfloat16 if self.dtype == "bf16" else torch.float32)
        out = {k: torch.from_numpy(getattr(self, k)).to(device=device, dtype=dt).contiguous()
               for k in ("x", "Wg_s", "Wu_s", "Wd_s")}
        if self.dy is not None:
            out["dy"] = torch.from_numpy(self.dy).to(device=device, dtype=dt).contiguous()
        return out


def _weights(rng, d, f, bf16):
    Wg = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / math.sqrt(d))
    Wu = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / math.sqrt(d))
    Wd = rng.standard_normal((f, d), dtype=np.float32) * np.float32(1.0 / math.sqrt(f))
    if bf16:
        Wg, Wu, Wd = round_bf16_np(Wg), round_bf16_np(Wu), round_bf16_np(Wd)
    return Wg, Wu, Wd


def _sigma(Wg):
    w = Wg[:, 1:].astype(np.float64)
    return np.sqrt((w * w).sum(axis=1))


def _finish(a, bf16):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return round_bf16_np(a) if bf16 else a


def uniform_layer(N, d, f, T, p, seed, bf16=True, dead_frac=0.0, target_nnz=None, name="uniform"):
    """Layer with one threshold for every live column.

    ``dead_frac`` of the columns (the first ones of a seeded permutation) get the bias -1e4,
    so they never fire. If ``target_nnz`` is given, live columns use p = target_nnz / n_live.
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, d), dtype=np.float32)
    x[:, 0] = 1.0
    Wg, Wu, Wd = _weights(rng, d, f, bf16)
    n_dead = int(round(dead_frac * f))
    perm = rng.permutation(f)
    dead = perm[:n_dead]
    if target_nnz is not None:
        p = target_nnz / (f - n_dead)
    tau = tau_for_density(p)
    sig = _sigma(Wg)
    Wg[:, 0] = (-tau * sig).astype(np.float32)
    Wg[dead, 0] = -1e4
    recipe = (f"x[:,0]=1, x[:,1:]~N(0,1); W~N(0,1/fan_in); Wg_s[j,0]=-tau*sigma_j with tau={tau:.4f} "
              f"(p={p:.5f} per live column); {n_dead} dead columns with Wg_s[j,0]=-1e4; seed {seed}")
    return Layer(name=name, N=N, d=d, f=f, T=T, dtype="bf16" if bf16 else "f32",
                 x=_finish(x, bf16), Wg_s=_finish(Wg, bf16), Wu_s=Wu, Wd_s=Wd,
                 target_density=p * (f - n_dead) / f, recipe=recipe)


def per_token_layer(N, d, f, T, seed, base=0.005, normalise=True, seq_len=1024, first=4,
                    first_mult=10.0, sigma_ln=0.8, cap=0.5, bf16=True, name="per_token"):
    """Layer whose density varies per token: lognormal multiplier, denser sequence starts.

    w_r = exp(sigma_ln * z_r) (z ~ N(0,1)), times ``first_mult`` for the first ``first``
    positions of each ``seq_len``-token sequence. p_r = min(base * w_r / mean(w), cap) when
    ``normalise`` (so the mean density is ``base``), else p_r = min(base * w_r, cap).
    The threshold moves into the token: x[r, 0] = tau_r and Wg_s[j, 0] = -sigma_j.
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, d), dtype=np.float32)
    Wg, Wu, Wd = _weights(rng, d, f, bf16)
    z = rng.standard_normal(N)
    w = np.exp(sigma_ln * z)
    w[(np.arange(N) % seq_len) < first] *= first_mult
    p = base * w / w.mean() if normalise else base * w
    p = np.minimum(p, cap)
    tau = np.array([tau_for_density(float(q)) for q in p])
    x[:, 0] = tau.astype(np.float32)
    sig = _sigma(Wg)
    Wg[:, 0] = (-sig).astype(np.float32)
    recipe = (f"x[:,1:]~N(0,1); W~N(0,1/fan_in); per-token density p_r=min({base}*w_r"
              f"{'/mean(w)' if normalise else ''},{cap}), w_r=exp({sigma_ln} z_r) x{first_mult} for the first "
              f"{first} positions of each {seq_len}-token sequence; x[r,0]=tau_r, Wg_s[j,0]=-sigma_j; seed {seed}")
    return Layer(name=name, N=N, d=d, f=f, T=T, dtype="bf16" if bf16 else "f32",
                 x=_finish(x, bf16), Wg_s=_finish(Wg, bf16), Wu_s=Wu, Wd_s=Wd,
                 target_density=float(p.mean()), recipe=recipe)


def calibration_tokens(L: Layer, N: int, seed: int) -> np.ndarray:
    """Another batch of tokens for layer L, drawn like L's own x (x[:,0] = 1, x[:,1:] ~ N(0,1),
    rounded to L's dtype); for layers whose bias feature is x[:,0] = 1 (uniform_layer)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, L.d), dtype=np.float32)
    x[:, 0] = 1.0
    return _finish(x, L.dtype == "bf16")


# --------------------------------------------------------------------------- presets

SWEEP_DENSITIES = (0.001, 0.005, 0.01, 0.02, 0.05, 0.10, 0.50)
SWEEP_TILES = (64, 128, 256)


def tiny_fp32(seed=0):
    """64 tokens, d_model 256, d_ff 1024, T 128, fp32, 2% gate density."""
    return uniform_layer(64, 256, 1024, 128, 0.02, seed, bf16=False, name="tiny_fp32_64x256x1024")


def layer_1p5b(seed=1, N=8192):
    """1.5B-like inference layer: 8192 tokens, d_model 2048, d_ff 5632, T 128, bf16,
    about 29 nonzeros per token, 30% dead columns."""
    return uniform_layer(N, 2048, 5632, 128, None, seed, bf16=True, dead_frac=0.3,
                         target_nnz=29.0, name=f"layer1.5b_N{N}_d2048_f5632_T128")


def layer_2b(seed=2, N=16384):
    """2B-like inference layer: 16384 tokens, d_model 2560, d_ff 6912, T 128, bf16, mean density
    0.5% with a lognormal(0, 0.8) per-token multiplier and 10x density on the first 4 positions of
    each 1024-token sequence."""
    return per_token_layer(N, 2560, 6912, 128, seed, base=0.005, normalise=True,
                           name=f"layer2b_N{N}_d2560_f6912_T128")


def sweep_point(p, T, seed=3, N=8192):
    """Density-sweep point on the 1.5B-like shapes: uniform density p, tile width T."""
    return uniform_layer(N, 2048, 5632, T, p, seed, bf16=True,
                         name=f"sweep_p{p:g}_T{T}_N{N}_d2048_f5632")


def train_2b(seed=4, N=16384, literal=False):
    """Hybrid training step on the 2B-like shapes, K = 64, L1 coefficient 2e-5, dy ~ N(0,1).

    The default scales the per-token density so that about 2% of rows overflow K (median density
    0.18%, un-normalised lognormal); ``literal=True`` keeps the 0.5%-mean generator of the 2B
    inference layer, under which far more rows overflow.
    """
    if literal:
        L = per_token_layer(N, 2560, 6912, 128, seed, base=0.005, normalise=True,
                            name=f"train2b_literal_N{N}_d2560_f6912_K64")
    else:
        L = per_token_layer(N, 2560, 6912, 128, seed, base=0.0018, normalise=False,
                            name=f"train2b_N{N}_d2560_f6912_K64")
    rng = np.random.default_rng(seed + 1000)
    L.dy = round_bf16_np(rng.standard_normal((N, L.d), dtype=np.float32))
    L.K = 64
    L.l1_coef = 2e-5
    return L


def small_train(seed=0, N=200, d=256, f=1024, K=16, base=0.01, bf16=False, name=None):
    """Small training layer (for tests): per-token density with a heavy tail so that some rows
    overflow the capacity K."""
    L = per_token_layer(N, d, f, 128, seed, base=base, normalise=True, seq_len=64, first=2,
                        bf16=bf16, name=name or f"small_train_N{N}_d{d}_f{f}_K{K}")
    rng = np.random.default_rng(seed + 1000)
    dy = rng.standard_normal((N, d), dtype=np.float32)
    L.dy = round_bf16_np(dy) if bf16 else dy
    L.K = K
    return L
