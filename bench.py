#!/usr/bin/env python3
"""Benchmark of the sparse inference FFN layer (TwELL) on GB300.

One step = the whole inference hot path over one batch of tokens: twell_gate_pack (tcgen05 gate
GEMM with the ReLU + TwELL pack epilogue) followed by twell_ffn_fused_fwd (fused up+down walk
over the packed nonzeros), both through the C ABI. The workload is the 1.5B-like layer:
N = 8192 tokens, d_model = 2048, d_ff = 5632, T = 128, bf16 with fp32 accumulation, ~29 nonzero
gate activations per token, 30% dead columns (seed 1). Inputs are resident in HBM; the 129 MB L2
is flushed (256 MiB write) before every timed step.

Prints ONE JSON line. Beside tokens/s it reports the dominant kernel's roofline fraction, the
layer roofline of the method's byte model, the speedup over a dense cuBLAS bf16 FFN of the same
shape, an end-to-end figure with host buffers, and the fp64 CPU oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --sweep     # density x tile-width sweep, the 2B-like layer, decode batches: one line each
N > 1 is launched with torchrun: every rank runs its own batch (weak scaling, no collective on
the data path; a barrier and a max over ranks of the timed region only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse FFN tokens/s per layer on 1 GB300; % of roofline; speedup vs dense FFN"
NOMINAL_HBM = 8.0e12  # bytes/s: the rough HBM3e figure the layer's target is stated against
# L2 -> shared-memory rate of random 4 KB weight rows from an L2-resident 46 MB table, moved with
# cp.async.bulk by every warp's own two-slot ring (8-16 warps per SM), measured on this GPU type by a
# probe program (not part of the product): 20.1-20.6 TB/s. The walk's gathers are bounded by it.
L2_GATHER_GBS = 20600.0
L2_GATHER_KIND = ("probe: cp.async.bulk of 4 KB rows from an L2-resident table, one ring per warp, "
                  "8-16 warps per SM (20.1-20.6 TB/s); not in MEASURED_PEAKS.json")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--no-train", action="store_true", help="skip the hybrid training-step measurement")
    p.add_argument("--no-f16down", action="store_true",
                   help="skip the sub-entry of the walk with its down projection in fp16")
    p.add_argument("--train-steps", type=int, default=20)
    p.add_argument("--config", type=int, choices=[1, 2], default=1,
                   help="workload of the main line: 1 = the 1.5B-like layer (default), 2 = the 2B-like layer "
                        "(N=16384, d_model 2560, d_ff 6912, lognormal per-token density; no dead-column step)")
    p.add_argument("--path", choices=["walk", "union", "tile_union"], default="walk",
                   help="the step: gate + pack then the fused walk (default); the union path "
                        "(twell_ffn_gate_union_fwd: gate and up projection in one GEMM, then the down GEMM over all "
                        "of d_ff); or gate + pack then the tile-union GEMMs (twell_ffn_tile_union_fwd); the last two "
                        "with Wd_s converted to fp16 once outside the timed region")
    p.add_argument("--tokens", type=int, default=None,
                   help="batch size of the --config layer's main line (default: the layer's own, 8192 / 16384)")
    p.add_argument("--density", type=float, default=None,
                   help="run the main line on the sweep's uniform-density layer (N=8192, d_model 2048, d_ff 5632, "
                        "T=128) with this kept fraction instead of the --config layer")
    p.add_argument("--train-only", action="store_true",
                   help="only the hybrid training step against the dense cuBLAS step (one JSON line)")
    p.add_argument("--sweep", action="store_true",
                   help="density x tile-width sweep on the 1.5B-like shapes, the 2B-like layer and small decode "
                        "batches of the 1.5B-like layer, against dense cuBLAS (one JSON line per point; not the "
                        "default bench line)")
    p.add_argument("--sweep-iters", type=int, default=15)
    p.add_argument("--sweep-only", default="", help="with --sweep: only the points whose label contains this text")
    return p.parse_args()


def max_over_ranks(value, dist, device):
    """Largest value over the ranks of the process group (the timed region ends when the slowest
    rank ends), or the value itself without a group."""
    if dist is None:
        return value
    import torch
    tt = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tt.item()


def weak_scaling_rate(tokens_per_rank, ms_per_step, world):
    """Whole-job tokens/s when every rank processes its own batch of tokens_per_rank per step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------ oracle (CPU)

def oracle_sparse_rows(L, rows):
    """The fp64 oracle's sparse path on the given token rows: gate -> TwELL pack -> walk."""
    import numpy as np

    import oracle
    G = oracle.gate(L.x, L.Wg_s, rows=rows)
    vals, idx, cnt = oracle.twell_pack(G, L.T)
    return oracle.twell_walk(vals, idx, cnt, L.T, L.x[rows].astype(np.float64), L.Wu_s, L.Wd_s)


def cpu_oracle_rate(L, target_s=4.0, max_rows=4096):
    """Tokens/s of the oracle's sparse path on a bounded row sample sized to take ~target_s."""
    import numpy as np
    rng = np.random.default_rng(123)
    n = 8
    while True:
        rows = rng.choice(L.N, n, replace=False)
        t0 = time.perf_counter()
        oracle_sparse_rows(L, rows)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= max_rows:
            return n / dt, n, dt
        n = min(max_rows, max(n * 2, int(n * target_s / max(dt, 1e-3))))


# ------------------------------------------------------------------------------------ reference arm

def run_reference(a, rank, world):
    if rank != 0:
        return
    import numpy as np

    from activation_sparse_ffn_gate_gb300 import synthetic
    L = synthetic.layer_1p5b()
    rng = np.random.default_rng(7)
    # calibrate one row, then size each step's sample so the whole run ends within a few minutes
    t0 = time.perf_counter()
    oracle_sparse_rows(L, rng.choice(L.N, 4, replace=False))
    per_row = (time.perf_counter() - t0) / 4
    budget = 120.0
    S = int(max(1, min(512, budget / max(1, a.steps + a.warmup) / per_row)))
    for _ in range(a.warmup):
        oracle_sparse_rows(L, rng.choice(L.N, S, replace=False))
    t0 = time.perf_counter()
    for _ in range(a.steps):
        oracle_sparse_rows(L, rng.choice(L.N, S, replace=False))
    dt = time.perf_counter() - t0
    value = a.steps * S / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt / a.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": L.name, "N": L.N, "d_model": L.d, "d_ff": L.f, "T": L.T},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                         "sample": f"{S} random token rows of the {L.N}-token batch per step (fp64 gate, TwELL pack, "
                                   f"fused walk)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------ our arm

def _source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "gate": ["activation_sparse_ffn_gate_gb300/csrc/twell_gemm.cuh", "activation_sparse_ffn_gate_gb300/csrc/twell_gate.cu",
             "activation_sparse_ffn_gate_gb300/csrc/twell_common.cuh"],
    "fused": ["activation_sparse_ffn_gate_gb300/csrc/twell_ffn.cu", "activation_sparse_ffn_gate_gb300/csrc/twell_common.cuh",
              "activation_sparse_ffn_gate_gb300/csrc/twell_mma.cuh"],
}


def _traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))[kernel]
    except Exception:
        return None
    if rec.get("source_hash") != _source_hash(KERNEL_SOURCES[kernel]):
        return None
    return rec.get("bytes_per_launch")


def _union_down_launches(N, d, sm_count):
    """Launches of the union path's down product, by the library's host rule: one kernel up to 512
    tokens (K split over a cluster, partials added on chip); the SM-pair GEMM and a reduction of its
    K-split partials up to 1024; above that the GEMM, plus a reduction of the K halves when the
    partial last wave of 256 x 256 tiles is split (it fills at most half the SM pairs, at most 40
    tiles)."""
    if N <= 512:
        return 1
    if N <= 1024:
        return 2
    pairs = sm_count // 2
    units = -(-N // 256) * -(-d // 256)
    tail = units % pairs
    return 2 if (units > pairs and 0 < tail and 2 * tail <= pairs and tail <= 40) else 1


def run_ours(a, rank, world):
    import numpy as np
    import torch

    from activation_sparse_ffn_gate_gb300 import binding, build, synthetic
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # every rank its own batch (weak scaling)
    if a.density is not None:
        L = synthetic.sweep_point(a.density, 128, seed=3 + rank)
    else:
        kw = {} if a.tokens is None else {"N": a.tokens}
        L = synthetic.layer_1p5b(seed=1 + rank, **kw) if a.config == 1 else synthetic.layer_2b(seed=2 + rank, **kw)
    main_cfg1 = a.density is None and a.config == 1 and a.tokens is None
    t = L.torch_inputs(dev)
    x, Wg, Wu, Wd = t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"]
    N, d, f, T = L.N, L.d, L.f, L.T
    status = binding.status_buffer(dev)
    status.zero_()
    packed = binding.TwELL.empty(N, f, T, torch.float32, dev)  # fp32 packed gate values
    y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    Wd16 = binding.twell_convert_f16(Wd, status=status, stream=stream) if a.path == "tile_union" else None
    Wd16t = binding.twell_convert_f16_transposed(Wd, status=status, stream=stream) if a.path == "union" else None

    # the union path with T = 64 or 128 is one call: gate and up projection in one GEMM, then the down GEMM
    gate_union = a.path == "union" and T in (64, 128)

    def first():
        if gate_union:
            binding.twell_ffn_gate_union_fwd(x, Wg, Wu, Wd16t, T, out=packed, y=y, status=status, stream=stream)
        else:
            binding.twell_gate_pack(x, Wg, T, out=packed, status=status, stream=stream)

    def second():
        if gate_union:
            return
        if a.path == "tile_union":
            binding.twell_ffn_tile_union_fwd(x, Wu, Wd16, packed, y=y, status=status, stream=stream)
        elif a.path == "union":
            binding.twell_ffn_union_fwd(x, Wu, Wd16t, packed, y=y, status=status, stream=stream)
        else:
            binding.twell_ffn_fused_fwd(x, Wu, Wd, packed, y=y, status=status, stream=stream)

    def step():
        first()
        second()

    for _ in range(a.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    binding.check_device_status("warmup", status)

    clk = ClockSampler(dev.index)
    clk.start()
    time.sleep(0.6)  # let nvidia-smi start sampling
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(a.steps):
        flush.fill_(1)
        e0, e1, e2 = ev[i]
        e0.record(stream)
        first()
        e1.record(stream)
        second()
        e2.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk.stop()
    binding.check_device_status("timed region", status)
    t_gate = [e0.elapsed_time(e1) for e0, e1, _ in ev]
    t_fused = [e1.elapsed_time(e2) for _, e1, e2 in ev]
    t_step = sum(t_gate) + sum(t_fused)  # ms over K steps, L2 flushes excluded
    t_step = max_over_ranks(t_step, dist, dev)
    ms_step = t_step / a.steps
    value = weak_scaling_rate(N, ms_step, world)

    # the same step without the L2 flush in between (weights and x may stay L2-resident)
    warm_steps = max(10, min(a.steps, 200))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step()
    w0.record(stream)
    for _ in range(warm_steps):
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = max_over_ranks(w0.elapsed_time(w1) / warm_steps, dist, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---- realised sparsity and the union of active weight rows per 128-token tile (byte model)
    dense_a = binding.twell_unpack(packed)
    active = dense_a != 0
    nnz = active.sum().item()
    tiles = (N + 127) // 128
    union = sum(int(active[i * 128:(i + 1) * 128].any(0).sum().item()) for i in range(tiles))
    distinct = int(active.any(0).sum().item())  # units some token of the batch keeps
    del dense_a, active
    twell_bytes = N * (f // T) * 2 + nnz * 5  # counts + packed (fp32 value, u8 index) entries
    peaks, peak_kind = _peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    gate_flops = 2.0 * N * d * f
    bytes_layer = (N * d * 2) + (f * d * 2) + union * 2 * d * 2 + (N * d * 2)
    t_roof = max(gate_flops / tc, bytes_layer / hbm)
    t_roof_nominal = max(gate_flops / tc, bytes_layer / NOMINAL_HBM)
    # stricter model: every active weight row read once per layer (the rows stay in L2)
    bytes_strict = (N * d * 2) + (f * d * 2) + distinct * 2 * d * 2 + (N * d * 2)
    t_roof_strict = max(gate_flops / tc, bytes_strict / hbm)
    # per-kernel algorithmic work
    fused_bytes = (N * d * 2) + union * 2 * d * 2 + (N * d * 2) + twell_bytes
    mg, mf = sum(t_gate) / a.steps, sum(t_fused) / a.steps
    second_name = {"walk": "twell_ffn_fused_fwd", "union": "twell_ffn_union_fwd",
                   "tile_union": "twell_ffn_tile_union_fwd"}[a.path]
    first_name = "twell_ffn_gate_union_fwd" if gate_union else "twell_gate_pack"
    if gate_union:
        # one call: the gate + up GEMM (2 * N * d * 2 f FLOPs, the TwELL packed in its epilogue) and
        # the down GEMM over f rounded up to 64 (2 * N * f_pad * d)
        gu_flops = 4.0 * N * d * f + 2.0 * N * ((f + 63) // 64 * 64) * d
        ach = gu_flops / (mg * 1e-3) / 1e12
        roof = {"kernel": first_name, "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": None,
                "algorithmic_flops": gu_flops, "ms_per_launch": mg,
                "peak_kind": peak_kind + " bf16_tflops (burst; the down GEMM runs fp16, the same rate)",
                "note": "whole call (gate + up GEMM with the pack and h = a * u in its epilogue, then the "
                        "down GEMM) against the three products' FLOPs: all of d_ff, the dense regime"}
    elif a.path != "walk" and mf >= mg:
        # the up and down GEMMs: over each 128-token tile's union (2 * 128 * |U_m| * d FLOPs each per
        # tile), or over all of d_ff rounded up to 64 for the union path
        tu_flops = 4.0 * 128 * union * d if a.path == "tile_union" else 4.0 * N * ((f + 63) // 64 * 64) * d
        ach = tu_flops / (mf * 1e-3) / 1e12
        roof = {"kernel": second_name, "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": None,
                "algorithmic_flops": tu_flops, "ms_per_launch": mf,
                "peak_kind": peak_kind + " bf16_tflops (burst; the down GEMM runs fp16, the same rate)",
                "note": "whole call (expand, up and down GEMMs; the tile unions first on the tile-union path) "
                        "against the two GEMMs' FLOPs"}
    elif mf >= mg:
        # The walk moves, per kept entry, the unit's rows of Wu_s and Wd_s (2 * d * 2 B) from L2 into
        # shared memory, plus x_r once per row: these gathers, not HBM, bound it (ncu: DRAM ~9% busy).
        gathered = nnz * 2 * d * 2 + N * d * 2
        ach_l2 = gathered / (mf * 1e-3) / 1e9
        ach = fused_bytes / (mf * 1e-3) / 1e9
        roof = {"kernel": "twell_ffn_fused_fwd", "bound": "l2", "achieved": ach_l2, "peak": L2_GATHER_GBS,
                "unit": "GB/s", "frac": ach_l2 / L2_GATHER_GBS,
                "traffic": _traffic("fused") if main_cfg1 else None,
                "algorithmic_bytes": gathered, "ms_per_launch": mf,
                "peak_kind": L2_GATHER_KIND,
                "limiter": "L2 -> SM gathers of weight rows and the per-nonzero instruction chain (latency; "
                           "ncu: issue ~30% active, tensor pipe ~42%, DRAM ~9% of peak)",
                "hbm_byte_model": {"bytes": fused_bytes, "achieved_gbs": ach,
                                   "frac_measured_hbm": ach / peaks["hbm_gbs"],
                                   "frac_nominal_hbm": ach * 1e9 / NOMINAL_HBM,
                                   "definition": "x + y + the union of active Wu/Wd rows per 128-token tile + "
                                                 "TwELL, charged at HBM rate (the method's byte model; the "
                                                 "union rows are L2 hits, so this is not an HBM-bound figure)"}}
    else:
        ach = gate_flops / (mg * 1e-3) / 1e12
        roof = {"kernel": "twell_gate_pack", "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                "traffic": _traffic("gate") if main_cfg1 else None,
                "algorithmic_flops": gate_flops, "ms_per_launch": mg, "peak_kind": peak_kind + " bf16_tflops (burst)"}

    # ---- dense cuBLAS bf16 FFN of the same shape (best of two formulations)
    dense = None
    if not a.no_dense:
        Wgu = torch.cat([Wg, Wu], 0)

        def dense_a_():
            g = x @ Wg.T
            u = x @ Wu.T
            return (torch.relu(g) * u) @ Wd

        def dense_b_():
            gu = x @ Wgu.T
            g, u = gu[:, :f], gu[:, f:]
            return (torch.relu(g) * u) @ Wd

        best = {}
        for name, fn in (("three_gemms", dense_a_), ("fused_gate_up_gemm", dense_b_)):
            for _ in range(5):
                flush.fill_(1)
                fn()
            ts = []
            for _ in range(30):
                flush.fill_(1)
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record()
                fn()
                s1.record()
                torch.cuda.synchronize()
                ts.append(s0.elapsed_time(s1))
            best[name] = statistics.median(ts)
        bname = min(best, key=best.get)
        dense = {"ms": best[bname], "formulation": bname, "all_ms": best, "speedup": best[bname] / ms_step}

    # ---- end to end through the public API with host buffers (pinned H2D of x, D2H of y, every
    # step): binding.StreamedFFN overlaps each step's copies with its neighbours' compute (copy-in,
    # compute and copy-out streams, double-buffered device x and y); the serial figure runs the
    # three one after the other on one stream.
    xh = x.cpu().pin_memory()
    yh = torch.empty((N, d), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)
    e2e_steps = max(10, min(a.steps, 200))
    for _ in range(3):
        xd.copy_(xh, non_blocking=True)
        binding.ffn_forward(xd, Wg, Wu, Wd, T, packed=packed, y=y, status=status, stream=stream, path=a.path,
                            Wd16_s=Wd16, Wd16t_s=Wd16t)
        yh.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(e2e_steps):
        xd.copy_(xh, non_blocking=True)
        binding.ffn_forward(xd, Wg, Wu, Wd, T, packed=packed, y=y, status=status, stream=stream, path=a.path,
                            Wd16_s=Wd16, Wd16t_s=Wd16t)
        yh.copy_(y, non_blocking=True)
    s1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = s0.elapsed_time(s1) / e2e_steps
    pipe = binding.StreamedFFN(Wg, Wu, Wd, N, T=T, status=status, path=a.path, Wd16_s=Wd16, Wd16t_s=Wd16t)
    for _ in range(3):
        pipe.submit(xh, yh)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(pipe.copy_in)
    for _ in range(e2e_steps):
        pipe.submit(xh, yh)
    s1.record(pipe.copy_out)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / e2e_steps
    binding.check_device_status("e2e", status)

    # ---- dead-column compaction (the 1.5B-like layer: 30% of its units never fire; the 2B-like layer
    # has none by construction)
    def medians_gate_walk(gate, walk, n):
        """Median gate + pack and walk times over n steps, L2 flushed before each."""
        cg, cf = [], []
        for _ in range(n):
            flush.fill_(1)
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            gate()
            e1.record(stream)
            walk()
            e2.record(stream)
            cg.append((e0, e1))
            cf.append((e1, e2))
        torch.cuda.synchronize()
        return (statistics.median(u.elapsed_time(v) for u, v in cg),
                statistics.median(u.elapsed_time(v) for u, v in cf))

    compacted = None
    Wu_c = Wd_c = Wg_c = packed_c = None
    if main_cfg1 and a.path == "walk":
        x_cal = torch.from_numpy(synthetic.calibration_tokens(L, N, seed=1000 + rank)).to(dev, torch.bfloat16)
        counts = binding.twell_column_activity(binding.twell_gate_pack(x_cal, Wg, T, status=status), status=status)
        live = binding.live_columns(counts)
        Wg_c, Wu_c, Wd_c = binding.compact_weights(Wg, Wu, Wd, live, status=status)
        f_c = live.numel()
        packed_c = binding.TwELL.empty(N, f_c, T, torch.float32, dev)
        y_c = torch.empty_like(y)
        del x_cal
        binding.twell_gate_pack(x, Wg, T, out=packed, status=status, stream=stream)
        binding.twell_ffn_fused_fwd(x, Wu, Wd, packed, y=y, status=status, stream=stream)
        binding.twell_gate_pack(x, Wg_c, T, out=packed_c, status=status, stream=stream)
        binding.twell_ffn_fused_fwd(x, Wu_c, Wd_c, packed_c, y=y_c, status=status, stream=stream)
        torch.cuda.synchronize()
        identical = bool(torch.equal(y, y_c))
        c_steps = max(10, min(a.steps, 200))
        mcg, mcf = medians_gate_walk(
            lambda: binding.twell_gate_pack(x, Wg_c, T, out=packed_c, status=status, stream=stream),
            lambda: binding.twell_ffn_fused_fwd(x, Wu_c, Wd_c, packed_c, y=y_c, status=status, stream=stream),
            c_steps)
        binding.check_device_status("compacted", status)
        compacted = {"live_cols": f_c, "dead_cols": f - f_c, "calibration": f"{N} other tokens (seed {1000 + rank})",
                     "ms_gate_pack": mcg, "ms_fused": mcf, "ms_per_step": mcg + mcf,
                     "tokens_per_s": N / ((mcg + mcf) * 1e-3), "y_bit_identical": identical,
                     "speedup_vs_dense": (dense["ms"] / (mcg + mcf)) if dense else None,
                     "note": "dead-column compaction (units that never fired in the calibration batch are dropped "
                             "from Wg_s, Wu_s, Wd_s once); medians over the steps, L2 flushed"}

    # ---- the walk with its down projection in fp16 (Wd_s converted once; h rounded once to fp16)
    f16 = None
    if not a.no_f16down and a.path == "walk":
        n16 = max(10, min(a.steps, 200))
        Wd16 = binding.twell_convert_f16(Wd, status=status, stream=stream)
        y16 = torch.empty_like(y)
        binding.twell_gate_pack(x, Wg, T, out=packed, status=status, stream=stream)
        binding.twell_ffn_fused_fwd(x, Wu, Wd, packed, y=y, status=status, stream=stream)
        binding.twell_ffn_fused_fwd_f16down(x, Wu, Wd16, packed, y=y16, status=status, stream=stream)
        torch.cuda.synchronize()
        diff = (y16.float() - y.float()).norm().item() / max(y.float().norm().item(), 1e-30)
        g16, w16 = medians_gate_walk(
            lambda: binding.twell_gate_pack(x, Wg, T, out=packed, status=status, stream=stream),
            lambda: binding.twell_ffn_fused_fwd_f16down(x, Wu, Wd16, packed, y=y16, status=status, stream=stream),
            n16)
        binding.check_device_status("f16down", status)
        f16 = {"ms_gate_pack": g16, "ms_walk": w16, "ms_per_step": g16 + w16, "tokens_per_s": N / ((g16 + w16) * 1e-3),
               "walk_roofline_frac": (fused_bytes / (w16 * 1e-3)) / 1e9 / peaks["hbm_gbs"],
               "speedup_vs_dense": (dense["ms"] / (g16 + w16)) if dense else None,
               "rel_fro_vs_bf16_walk": diff,
               "note": "twell_ffn_fused_fwd_f16down: Wd_s converted once to fp16 (exact for these weights), h "
                       "rounded once to fp16 (11 significant bits) instead of a bf16 hi + lo pair; medians, L2 "
                       "flushed; not the headline (the headline walk keeps every operand in bf16)"}
        if Wd_c is not None:
            Wd16_c = binding.twell_convert_f16(Wd_c, status=status, stream=stream)
            gc, wc = medians_gate_walk(
                lambda: binding.twell_gate_pack(x, Wg_c, T, out=packed_c, status=status, stream=stream),
                lambda: binding.twell_ffn_fused_fwd_f16down(x, Wu_c, Wd16_c, packed_c, y=y_c, status=status,
                                                            stream=stream),
                n16)
            binding.check_device_status("f16down compacted", status)
            f16["compacted"] = {"ms_per_step": gc + wc, "tokens_per_s": N / ((gc + wc) * 1e-3),
                                "speedup_vs_dense": (dense["ms"] / (gc + wc)) if dense else None}
            del Wd16_c
        del Wd16, y16

    # ---- the union path on the same workload (gate and up projection in one GEMM, fp16 down GEMM),
    # and on the compacted weights: the layer's other path, beside the walk
    union_sub = None
    if not a.no_f16down and a.path == "walk" and T in (64, 128):
        nu = max(10, min(a.steps, 200))
        Wd16t_m = binding.twell_convert_f16_transposed(Wd, status=status, stream=stream)
        yu = torch.empty_like(y)
        gu_ms, _ = medians_gate_walk(
            lambda: binding.twell_ffn_gate_union_fwd(x, Wg, Wu, Wd16t_m, T, out=packed, y=yu, status=status,
                                                     stream=stream),
            lambda: None, nu)
        binding.check_device_status("union", status)
        union_sub = {"ms_per_step": gu_ms, "tokens_per_s": N / (gu_ms * 1e-3),
                     "speedup_vs_dense": (dense["ms"] / gu_ms) if dense else None,
                     "note": "twell_ffn_gate_union_fwd on the same batch (the TwELL packed in the gate + up GEMM's "
                             "epilogue, h in fp16, down GEMM over all of d_ff); medians, L2 flushed"}
        if Wd_c is not None:
            # the union path wants d_ff a multiple of 8: pad the live units with zero rows (g = 0 is
            # never kept, so y is unchanged)
            f_c = Wg_c.shape[0]
            pad = (f_c + 7) // 8 * 8 - f_c
            Wg_p, Wu_p, Wd_p = (torch.cat([w, w.new_zeros((pad, d))]) for w in (Wg_c, Wu_c, Wd_c))
            Wd16t_c = binding.twell_convert_f16_transposed(Wd_p, status=status, stream=stream)
            packed_p = binding.TwELL.empty(N, f_c + pad, T, torch.float32, dev)
            yc = torch.empty_like(y)
            gc_ms, _ = medians_gate_walk(
                lambda: binding.twell_ffn_gate_union_fwd(x, Wg_p, Wu_p, Wd16t_c, T, out=packed_p, y=yc,
                                                         status=status, stream=stream),
                lambda: None, nu)
            binding.check_device_status("union compacted", status)
            union_sub["compacted"] = {"ms_per_step": gc_ms, "tokens_per_s": N / (gc_ms * 1e-3), "units": f_c + pad,
                                      "speedup_vs_dense": (dense["ms"] / gc_ms) if dense else None}
            del Wd16t_c, yc, Wg_p, Wu_p, Wd_p, packed_p
        del Wd16t_m, yu
    del packed_c, Wg_c, Wu_c, Wd_c

    train = None
    if not a.no_train:
        train = train_step_measure(a, dev, flush, peaks)
        lit = train_step_measure(a, dev, flush, peaks, literal=True)
        train["literal"] = {k: lit[k] for k in ("workload", "ms", "tokens_per_s", "backup_rows", "backup_frac",
                                                 "dense_cublas_ms", "speedup_vs_dense")}
        train["literal"]["note"] = ("the 2B-like layer's own generator (0.5% mean density, lognormal per token, 10x "
                                    "on each sequence's first four tokens): ~13% of rows overflow K = 64")

    cpu = None
    if not a.no_cpu_baseline:
        import oracle
        oracle.set_threads(_cores())
        rate, n_rows, secs = cpu_oracle_rate(L)
        cpu = {"value": rate, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
               "sample": f"{n_rows} random token rows of the {N}-token batch (fp64 gate GEMV, TwELL pack, fused "
                         f"walk), {secs:.1f} s wall"}
        oracle.set_threads(1)
        rate1, n1, secs1 = cpu_oracle_rate(L, target_s=2.0, max_rows=512)
        oracle.set_threads(_cores())
        cpu["one_core"] = {"value": rate1, "unit": "tokens/s", "cores": 1,
                           "sample": f"{n1} random token rows, {secs1:.1f} s wall"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": L.name, "N": N, "d_model": d, "d_ff": f, "T": T, "tokens_per_gpu": N,
                   "nnz_per_token": nnz / N, "density": nnz / (N * f), "l2": "flushed before every step (256 MiB write)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "roofline": roof,
        "layer_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step, "bytes": bytes_layer,
                           "gate_flops": gate_flops, "union_cols_per_128_tokens": union / tiles,
                           "definition": "max(gate FLOPs / bf16 peak, (x + Wg + union of active Wu/Wd rows per "
                                         "128-token tile + y) / HBM peak), peaks measured (MEASURED_PEAKS.json)",
                           "frac_nominal_hbm": t_roof_nominal * 1e3 / ms_step,
                           "nominal_hbm_gbs": NOMINAL_HBM / 1e9,
                           "t_roof_strict_ms": t_roof_strict * 1e3, "frac_strict": t_roof_strict * 1e3 / ms_step,
                           "distinct_active_units": distinct,
                           "definition_strict": "every active weight row read once per layer: max(gate FLOPs / bf16 "
                                                "peak, (x + Wg + distinct active Wu/Wd rows + y) / HBM peak)"},
        "kernels_ms": {first_name: mg} if gate_union else {"twell_gate_pack": mg, second_name: mf},
        "compacted": compacted,
        "union": union_sub,
        "f16down": f16,
        "warm": {"ms_per_step": warm_ms, "tokens_per_s": weak_scaling_rate(N, warm_ms, world),
                 "l2": "not flushed between steps"},
        "vs_dense_cublas": dense,
        "train_step": train,
        "cpu_baseline": cpu,
        "e2e": {"value": N / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": N * d * 2,
                "d2h_bytes_per_step": N * d * 2, "ms_per_step": e2e_ms,
                "how": "binding.StreamedFFN: each step's pinned H2D copy and D2H copy overlap the neighbouring "
                       "steps' layer calls (three streams, double-buffered device x and y)",
                "serial": {"value": N / (e2e_serial_ms * 1e-3), "ms_per_step": e2e_serial_ms,
                           "how": "copy in, the layer, copy out one after the other on one stream"}},
        # per step: gate + pack, then the walk's zeroing, plan and walk; or the union path's gate + up
        # GEMM (or gate + pack, expand and up GEMM) and its down product; or the tile-union path's gate,
        # union bits, prefix, work list, expand, up and down GEMMs
        "gpu_launches": (((1 if gate_union else 3)
                          + _union_down_launches(N, d, torch.cuda.get_device_properties(dev).multi_processor_count))
                         if a.path == "union"
                         else {"walk": 4, "tile_union": 7}[a.path]) * a.steps,
        "path": a.path,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def hybrid_context_bytes(N, f, K, cap_rows, value_bytes=4):
    """Activation memory the hybrid backward reads from the forward, per layer (x is common to the
    hybrid and the dense step): a and u (value_bytes each; fp32 as the kernels store them) and the
    int16 column at each of the N * K block slots, the int16 row counts, the int32 backup list and
    the backup rows' dense a and u ([cap_rows, d_ff], value_bytes each)."""
    return N * K * (2 * value_bytes + 2) + N * 2 + cap_rows * 4 + 2 * cap_rows * f * value_bytes


def dense_context_bytes(N, f):
    """The dense step's saved gate pre-activation and up projection, [N, d_ff] bf16 each."""
    return 2 * N * f * 2


def train_step_measure(a, dev, flush, peaks, literal=False):
    """The hybrid training step on the 2B-like layer (N=16384, d=2560, f=6912, K=64, L1 2e-5):
    twell_hybrid_fwd + twell_hybrid_bwd, against a dense cuBLAS bf16 step of the same layer. The
    backup buffers are sized from the routed count of a first step (the count plus 12.5%), as a
    training loop sizes them from the previous step."""
    import torch

    from activation_sparse_ffn_gate_gb300 import binding, synthetic
    L = synthetic.train_2b(literal=literal)
    t = L.torch_inputs(dev)
    x, Wg, Wu, Wd, dy = t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], t["dy"]
    N, d, f, K = L.N, L.d, L.f, L.K
    # a first forward with room for every row sizes the buffers
    probe = binding.Hybrid.empty(N, f, K, N, dev)
    ws0 = torch.empty(binding.twell_workspace_bytes(binding.OP_HYBRID_FWD, N, d, f, 0, K, N), dtype=torch.uint8,
                      device=dev)
    y0 = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    binding.twell_hybrid_fwd(x, Wg, Wu, Wd, K, N, L.l1_coef, ctx=probe, y=y0, ws=ws0)
    routed = int(probe.n_backup.item())
    del probe, ws0, y0
    torch.cuda.empty_cache()
    cap = max(16, routed + routed // 8)
    ctx = binding.Hybrid.empty(N, f, K, cap, dev)
    ws_f = torch.empty(binding.twell_workspace_bytes(binding.OP_HYBRID_FWD, N, d, f, 0, K, cap), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(binding.twell_workspace_bytes(binding.OP_HYBRID_BWD, N, d, f, 0, K, cap), dtype=torch.uint8,
                       device=dev)
    y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((N, d), dtype=torch.float32, device=dev)
    dW = [torch.empty((f, d), dtype=torch.float32, device=dev) for _ in range(3)]

    def step():
        binding.twell_hybrid_fwd(x, Wg, Wu, Wd, K, cap, L.l1_coef, ctx=ctx, y=y, ws=ws_f)
        binding.twell_hybrid_bwd(x, Wg, Wu, Wd, ctx, dy, L.l1_coef, dx=dx, dWg_s=dW[0], dWu_s=dW[1], dWd_s=dW[2],
                                 ws=ws_b)

    def dense():
        g = x @ Wg.T
        u = x @ Wu.T
        a_ = torch.relu(g)
        h = a_ * u
        yd = h @ Wd
        dh = dy @ Wd.T + L.l1_coef / (N * f) * torch.sign(h)
        du = dh * a_
        dg = dh * u * (g > 0)
        dxd = du @ Wu + dg @ Wg
        return yd, dxd, h.T @ dy, du.T @ x, dg.T @ x

    def timed(fn, n):
        for _ in range(3):
            flush.fill_(1)
            fn()
        ts = []
        for _ in range(n):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    ms = timed(step, a.train_steps)
    code = binding.twell_read_status(ctx.status)
    if code != 0:
        raise RuntimeError(f"hybrid training step reported status {code}")
    ms_dense = timed(dense, max(5, a.train_steps // 2))
    nb = int(ctx.n_backup.item())
    act = {"hybrid_bytes_as_run": hybrid_context_bytes(N, f, K, cap), "backup_cap_as_run": cap, "backup_rows": nb,
           "hybrid_bytes_exact": hybrid_context_bytes(N, f, K, nb), "dense_bytes": dense_context_bytes(N, f),
           "ratio_dense_over_hybrid": dense_context_bytes(N, f) / hybrid_context_bytes(N, f, K, cap),
           "hybrid_bytes_if_bf16_storage": hybrid_context_bytes(N, f, K, cap, value_bytes=2),
           "note": "what the backward reads from the forward per layer: the hybrid context with a, u, A_b, U_b "
                   "in fp32 as the kernels store them (backup buffers sized from the routed count + 12.5%); "
                   "dense = g and u, [N, d_ff] bf16 each; hybrid_bytes_if_bf16_storage is the format's size "
                   "with those four in bf16 (arithmetic, not what the kernels store)"}
    name = "train2b_literal" if literal else "train2b"
    return {"workload": f"{name}_N{N}_d{d}_f{f}_K{K} (hybrid fwd + bwd, L1 {L.l1_coef})", "ms": ms,
            "tokens_per_s": N / (ms * 1e-3), "backup_rows": nb, "backup_frac": nb / N,
            "dense_cublas_ms": ms_dense, "speedup_vs_dense": ms_dense / ms,
            "activation_memory": act, "launches_per_step": 25, "l2": "flushed before every step"}


def run_train_only(a):
    """The training-step measurement alone, as one JSON line."""
    import torch

    from activation_sparse_ffn_gate_gb300 import binding, build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    train = train_step_measure(a, dev, flush, _peaks())
    train["literal"] = train_step_measure(a, dev, flush, _peaks(), literal=True)
    print(json.dumps({"train_step": train}), flush=True)


def run_sweep(a):
    """Density x tile-width sweep on the 1.5B-like shapes (N=8192, d=2048, f=5632, uniform density
    p, no dead columns) and the 2B-like layer, each against a dense cuBLAS bf16 FFN of the same
    shape. One JSON line per point; L2 flushed before every timed iteration, median of the rest."""
    import torch

    from activation_sparse_ffn_gate_gb300 import binding, build, synthetic
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    status = binding.status_buffer(dev)
    status.zero_()

    def timed(fn, n):
        for _ in range(3):
            flush.fill_(1)
            fn()
        ts = []
        for _ in range(n):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def timed_in_graph(fn, n, rounds=3):
        """Device time of fn for small decode batches, which run for tens of microseconds: the
        event clock resolves only ~2 us here, so fn is captured after an L2 flush into one CUDA
        graph, a flush alone into another, each graph is replayed n times between one pair of
        events, and the difference per replay is fn's time (L2 still flushed before every call).
        Median of `rounds` such measurements."""
        def capture(body):
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                body()
            torch.cuda.current_stream().wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body()
            torch.cuda.synchronize()
            return g

        def body_fn():
            flush.fill_(1)
            fn()

        g_fn, g_fl = capture(body_fn), capture(lambda: flush.fill_(1))

        def total(g):
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        return statistics.median((total(g_fn) - total(g_fl)) / n for _ in range(rounds))

    points = [(p, T) for T in synthetic.SWEEP_TILES for p in synthetic.SWEEP_DENSITIES]
    layers = [(f"sweep p={p:g} T={T}", lambda p=p, T=T: synthetic.sweep_point(p, T)) for p, T in points]
    layers.append(("layer2b", synthetic.layer_2b))
    layers += [(f"batch N={n}", lambda n=n: synthetic.layer_1p5b(N=n))
               for n in (1, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)]
    layers = [(label, make) for label, make in layers if a.sweep_only in label]
    for label, make in layers:
        L = make()
        t = L.torch_inputs(dev)
        x, Wg, Wu, Wd = t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"]
        packed = binding.TwELL.empty(L.N, L.f, L.T, torch.float32, dev)
        y = torch.empty((L.N, L.d), dtype=torch.bfloat16, device=dev)
        binding.twell_gate_pack(x, Wg, L.T, out=packed, status=status)
        nnz = int(packed.counts().sum().item())
        n_it = a.sweep_iters if nnz / L.N < 400 else max(3, a.sweep_iters // 3)
        gate_fn = lambda: binding.twell_gate_pack(x, Wg, L.T, out=packed, status=status)  # noqa: E731
        fused_fn = lambda: binding.twell_ffn_fused_fwd(x, Wu, Wd, packed, y=y, status=status)  # noqa: E731
        Wd16 = binding.twell_convert_f16(Wd, status=status)
        Wd16t = binding.twell_convert_f16_transposed(Wd, status=status)
        union_fn = lambda: binding.twell_ffn_union_fwd(x, Wu, Wd16t, packed, y=y, status=status)  # noqa: E731
        gu_fn = (lambda: binding.twell_ffn_gate_union_fwd(x, Wg, Wu, Wd16t, L.T, out=packed, y=y,  # noqa: E731
                                                          status=status)) if L.T in (64, 128) else None
        f16_fn = lambda: binding.twell_ffn_fused_fwd_f16down(x, Wu, Wd16, packed, y=y, status=status)  # noqa: E731
        tu_fn = lambda: binding.twell_ffn_tile_union_fwd(x, Wu, Wd16, packed, y=y, status=status)  # noqa: E731

        def dense_fn():
            return (torch.relu(x @ Wg.T) * (x @ Wu.T)) @ Wd

        use_graphs = label.startswith("batch")
        if use_graphs:
            ms_gate = timed_in_graph(gate_fn, 50)
            ms_fused = timed_in_graph(fused_fn, 50)
            ms_union = timed_in_graph(union_fn, 50)
            ms_gu = timed_in_graph(gu_fn, 50) if gu_fn else None
            ms_f16 = timed_in_graph(f16_fn, 50)
            ms_tu = timed_in_graph(tu_fn, 50)
            ms_dense = timed_in_graph(dense_fn, 50)
        else:
            ms_gate = timed(gate_fn, n_it)
            ms_fused = timed(fused_fn, n_it)
            ms_union = timed(union_fn, max(3, min(n_it, 15)))
            ms_gu = timed(gu_fn, max(3, min(n_it, 15))) if gu_fn else None
            ms_f16 = timed(f16_fn, n_it)
            ms_tu = timed(tu_fn, n_it)
            ms_dense = timed(dense_fn, n_it)
        decode = None
        if L.N <= binding.DECODE_MAX_N:
            packed_d = binding.TwELL.empty(L.N, L.f, L.T, torch.float32, dev)
            y_d = torch.empty_like(y)
            decode_fn = lambda: binding.twell_ffn_decode(x, Wg, Wu, Wd, L.T, packed=packed_d, y=y_d,  # noqa: E731
                                                         status=status)
            decode_fn()
            fused_fn()
            torch.cuda.synchronize()
            rel = ((y_d.float() - y.float()).norm() / y.float().norm().clamp_min(1e-30)).item()
            ms_d = timed_in_graph(decode_fn, 50) if use_graphs else timed(decode_fn, n_it)
            decode = {"ms": ms_d, "tokens_per_s": L.N / (ms_d * 1e-3), "speedup_vs_dense": ms_dense / ms_d,
                      "rel_fro_vs_two_call_path": rel,
                      "how": "twell_ffn_decode: gate + pack + per-tile walk in one cluster kernel, partial rows "
                             "summed in a fixed order by a second kernel"}
        binding.check_device_status(label, status)
        ms = ms_gate + ms_fused
        ms_u2 = ms_gate + ms_union
        ms_u = ms_gu if ms_gu is not None else ms_u2  # the union path as ffn_forward runs it
        ms_t = ms_gate + ms_tu
        best = min((("walk", ms), ("union", ms_u), ("tile_union", ms_t)), key=lambda kv: kv[1])[0]
        auto = binding.choose_path(L.N, nnz / (L.N * L.f))
        ms_auto = {"decode": None, "walk": ms, "tile_union": ms_t, "union": ms_u}[auto]
        if ms_auto is None:
            ms_auto = decode["ms"] if decode else ms
        print(json.dumps({"sweep": label, "workload": L.name, "N": L.N, "d_model": L.d, "d_ff": L.f, "T": L.T,
                          "density": nnz / (L.N * L.f), "nnz_per_token": nnz / L.N, "ms_gate_pack": ms_gate,
                          "ms_fused": ms_fused, "ms_sparse": ms, "tokens_per_s": L.N / (ms * 1e-3),
                          "ms_dense_cublas": ms_dense, "speedup_vs_dense": ms_dense / ms,
                          "ms_union": ms_union, "ms_sparse_union_two_call": ms_u2, "ms_gate_union": ms_gu,
                          "ms_sparse_union": ms_u, "speedup_union_vs_dense": ms_dense / ms_u,
                          "ms_tile_union": ms_tu, "ms_sparse_tile_union": ms_t,
                          "speedup_tile_union_vs_dense": ms_dense / ms_t,
                          "faster_path": best, "speedup_faster_path_vs_dense": ms_dense / min(ms, ms_u, ms_t),
                          "auto_path": auto, "speedup_auto_vs_dense": ms_dense / ms_auto,
                          "f16down": {"ms_walk": ms_f16, "ms_step": ms_gate + ms_f16,
                                      "speedup_vs_dense": ms_dense / (ms_gate + ms_f16)},
                          "decode": decode,
                          "cuda_graphs": use_graphs, "l2": "flushed before every iteration",
                          "timing": ("per call: (50 replays of a graph [L2 flush + call] - 50 replays of a graph "
                                     "[L2 flush]) / 50, median of 3" if use_graphs else
                                     f"CUDA events around each call, median of {n_it}")}), flush=True)
        del t, x, Wg, Wu, Wd, Wd16, Wd16t, packed, y
        binding._tile_union_ws.clear()
        torch.cuda.empty_cache()


def main():
    a = _args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", a.gpus if a.gpus == 1 else 1))
    if a.sweep:
        if rank == 0:
            run_sweep(a)
        return
    if a.train_only:
        if rank == 0:
            run_train_only(a)
        return
    if a.impl == "reference":
        run_reference(a, rank, world)
    else:
        run_ours(a, rank, world)


if __name__ == "__main__":
    main()
