"""The bench's multi-rank timing (no GPU): world-size 2 over gloo on CPU.

Under torchrun every rank times its own batch; the job's time per step is the largest over the
ranks, and the whole-job rate is world * tokens per rank / that time (weak scaling)."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    local_ms = 10.0 + 3.0 * rank  # rank 1 is the slow one
    m = b.max_over_ranks(local_ms, dist, torch.device("cpu"))
    q.put((rank, m, b.weak_scaling_rate(8192, m, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    for _, m, v in out:
        assert m == pytest.approx(13.0)  # every rank sees the slowest rank's time
        assert v == pytest.approx(2 * 8192 / 13.0e-3)


def test_single_rank_needs_no_group():
    b = _bench()
    assert b.max_over_ranks(7.5, None, torch.device("cpu")) == 7.5
    assert b.weak_scaling_rate(8192, 0.5, 1) == pytest.approx(8192 / 0.5e-3)
