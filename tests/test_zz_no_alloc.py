"""The allocation-free routing entry point, against the ordinary one (GPU).

twell_hybrid_route_noalloc serves callers that cannot allocate device memory or hand the library a
workspace -- for example code inside a framework whose caching allocator owns every device
allocation, or a plug-in host whose interface carries only inputs and outputs. It routes an already
packed TwELL matrix using only a fixed scratch array inside the library. Here it must give exactly
the routing of twell_hybrid_route_from_gate on the same gate matrix, on two calls in a row: the
second call starts with the first call's block counts still in the shared array, and must not
depend on them (it rewrites every entry it reads before reading it). The second call also leaves
the context's u and U_b null, which routing never writes.
"""
import numpy as np
import pytest
import torch

from activation_sparse_ffn_gate_gb300 import binding, build, synthetic

pytestmark = pytest.mark.gpu


def _gate(N, f, seed):
    rng = np.random.default_rng(seed)
    dens = np.minimum(0.003 * np.exp(1.2 * rng.standard_normal(N)), 0.7)
    dens[::13] *= 15
    G = np.where(rng.random((N, f)) < np.minimum(dens, 0.9)[:, None], rng.random((N, f)) + 0.01,
                 -rng.random((N, f)))
    return synthetic.round_bf16_np(G.astype(np.float32))


def _same_routing(a, b):
    hc = a.counts().cpu().numpy()
    np.testing.assert_array_equal(hc, b.counts().cpu().numpy())
    light = hc != 0xFFFF
    np.testing.assert_array_equal(a.cols().cpu().numpy()[light], b.cols().cpu().numpy()[light])
    np.testing.assert_array_equal(a.a.cpu().numpy()[light], b.a.cpu().numpy()[light])
    n = int(a.n_backup.item())
    assert n == int(b.n_backup.item())
    s = min(n, a.backup_cap)
    np.testing.assert_array_equal(a.backup_rows[:s].cpu().numpy(), b.backup_rows[:s].cpu().numpy())
    np.testing.assert_array_equal(a.A_b[:s].cpu().numpy(), b.A_b[:s].cpu().numpy())
    return n


def test_noalloc_route_matches_the_workspace_route_twice(cuda_dev):
    build.build()
    binding.load()
    K = 16
    seen = []
    for call, (N, f, seed) in enumerate([(900, 2048, 11), (333, 1024, 12)]):
        G = torch.from_numpy(_gate(N, f, seed)).to(cuda_dev)
        ref = binding.twell_hybrid_route_from_gate(G.to(torch.bfloat16), K, backup_cap=N)
        packed = binding.twell_pack_from_gate(G.to(torch.float32), 128)
        ctx = binding.Hybrid.empty(N, f, K, N, cuda_dev)
        if call == 1:
            ctx.u = ctx.U_b = None  # not written by routing: a caller need not provide them
        binding.twell_hybrid_route_noalloc(packed, K, ctx)
        assert binding.twell_read_status(ctx.status) == 0
        assert binding.twell_read_status(ref.status) == 0
        n = _same_routing(ctx, ref)
        assert n > 0, "the dense backup is exercised"
        seen.append(n)
    assert len(seen) == 2


def test_noalloc_route_rejects_too_many_rows(cuda_dev):
    build.build()
    binding.load()
    N, f = 1_048_577, 128
    fake = binding.TwELL(N, f, 128, torch.empty(16, device=cuda_dev), torch.empty(16, dtype=torch.uint8, device=cuda_dev),
                         torch.empty(16, dtype=torch.int16, device=cuda_dev))
    ctx = binding.Hybrid.empty(1, f, 4, 1, cuda_dev)
    ctx.n_rows = N
    with pytest.raises(binding.TwellError) as e:
        binding.twell_hybrid_route_noalloc(fake, 4, ctx)
    assert e.value.code == 2  # TWELL_ERR_UNSUPPORTED, before anything is launched
