"""The activation-memory figures the bench reports for the hybrid training step (no GPU): the byte
count is the size of the context binding.Hybrid allocates, and the dense comparison is g and u."""
import importlib.util
import os

import torch

from activation_sparse_ffn_gate_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_memory", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_hybrid_context_bytes_is_what_the_context_holds():
    bench = _bench()
    for N, f, K, cap in ((64, 300, 8, 5), (1024, 6912, 64, 446), (7, 128, 0, 1)):
        ctx = binding.Hybrid.empty(N, f, K, cap, device=torch.device("cpu"))
        held = sum(t.numel() * t.element_size() for t in (ctx.a, ctx.u, ctx.col, ctx.cnt, ctx.backup_rows, ctx.A_b, ctx.U_b))
        assert bench.hybrid_context_bytes(N, f, K, cap) == held


def test_dense_context_and_the_ratio_at_the_training_layer():
    bench = _bench()
    N, f, K = 16384, 6912, 64
    assert bench.dense_context_bytes(N, f) == 2 * N * f * 2 == 452_984_832
    # 397 backup rows (2.4%): the context is ~14x smaller than g and u; in bf16 storage ~24x
    assert 13 < bench.dense_context_bytes(N, f) / bench.hybrid_context_bytes(N, f, K, 397) < 15
    assert bench.hybrid_context_bytes(N, f, K, 397, value_bytes=2) < bench.hybrid_context_bytes(N, f, K, 397) * 0.6
