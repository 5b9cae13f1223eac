"""Failure detection on the GPU without faulting or hanging it (GPU).

Every wait inside the library's kernels (TMA stages, tensor-memory accumulators, the walk's bulk-copy
slots) is bounded: past its limit the waiting thread records TWELL_ERR_TIMEOUT in the status word and
the kernel winds down and returns. twell_wait_probe runs that same bounded wait on an mbarrier that
nothing ever arrives on, so the timeout path is taken on purpose; the context must stay usable.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_ffn_gate_gb300 import binding, build, synthetic
from parity import assert_close

pytestmark = pytest.mark.gpu

TWELL_ERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_dev):
    build.build()
    binding.load()


def test_wait_that_completes_reports_nothing(cuda_dev):
    status = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    binding.twell_wait_probe(True, 50, status=status)
    assert binding.twell_read_status(status) == 0


def test_wait_that_never_completes_times_out_and_the_context_survives(cuda_dev):
    status = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.twell_wait_probe(False, 50, status=status)
    code = binding.twell_read_status(status, reset=False)
    dt = time.perf_counter() - t0
    assert code == TWELL_ERR_TIMEOUT
    assert 0.045 <= dt < 5.0, dt  # gave up after the 50 ms limit, not before and not much later
    status.zero_()
    # the device still runs kernels correctly afterwards
    L = synthetic.uniform_layer(256, 512, 1024, 128, 0.02, seed=12)
    t = L.torch_inputs(cuda_dev)
    y = binding.ffn_forward(t["x"], t["Wg_s"], t["Wu_s"], t["Wd_s"], T=L.T, status=status)
    assert binding.twell_read_status(status) == 0
    assert_close(y.double().cpu().numpy(), oracle.ffn(L.x, L.Wg_s, L.Wu_s, L.Wd_s), "after a timed-out wait")
