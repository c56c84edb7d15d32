"""qgemm_moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin whose framework owns all device memory, a decode loop in which an
allocation may synchronise the device) get the same routing kernels with their scratch in
a static device array of the library.  This file sorts last so that a run stopping at its
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import synth


def _lib():
    import moe_qw_repack_gb300.qw as Q
    return Q


def _route_with_workspace(Q, lg, T, E, k):
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    sp = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, k)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_route(lg, T, E, k, ids, sp, off, ws, n)
    torch.cuda.synchronize()
    return ids.cpu(), sp.cpu(), off.cpu()


def _route_noalloc_c_abi(Q, lg, T, E, k):
    """Call the C entry point directly through ctypes."""
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    sp = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = Q.LIB.qgemm_moe_route_noalloc(
        ctypes.c_void_p(lg.data_ptr()), T, E, k, ctypes.c_void_p(ids.data_ptr()),
        ctypes.c_void_p(sp.data_ptr()), ctypes.c_void_p(off.data_ptr()),
        ctypes.c_void_p(err.data_ptr()), stream)
    assert status == Q.QW_OK, Q.status_str(status)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ids.cpu(), sp.cpu(), off.cpu()


@pytest.mark.gpu
def test_noalloc_route_matches_workspace_route_on_two_calls_in_a_row():
    Q = _lib()
    # two different routings back to back; the second reuses the scratch the first left
    for (T, E, k, cfg) in [(4096, 256, 8, 3), (300, 1000, 32, 7)]:
        lg = torch.from_numpy(synth.router_logits(T, E, cfg_id=cfg)).cuda()
        want = _route_with_workspace(Q, lg, T, E, k)
        got = _route_noalloc_c_abi(Q, lg, T, E, k)
        for g, w in zip(got, want):  # routing is integer work: bit-exact
            assert torch.equal(g, w)


def test_noalloc_route_rejects_requests_beyond_its_scratch():
    """ceil(T*k/256) * E int32 must fit in the 1 MiB static scratch; the check happens on
    the host before any device work, so this runs without a GPU."""
    Q = _lib()
    T, E, k = 8192, 1024, 32  # 1024 chunks x 1024 experts x 4 B = 4 MiB
    assert Q.qgemm_moe_route_workspace_size(T, E, k) > (1 << 20)
    fake = 1 << 20  # never dereferenced
    status = Q.LIB.qgemm_moe_route_noalloc(fake, T, E, k, fake, fake, fake, None, None)
    assert status == Q.QW_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_route_matches_the_oracle():
    """The routing the no-alloc entry point returns is the oracle's, bit for bit (heavy
    ties included), on consecutive calls that reuse the shared scratch."""
    import numpy as np
    from oracle import moe as OM
    Q = _lib()
    rng = np.random.default_rng(17)
    cases = [(synth.router_logits(16, 128, cfg_id=4), 8),
             (rng.integers(-2, 3, (300, 40)).astype(np.float32), 6),
             (synth.router_logits(2048, 128, cfg_id=5), 8)]
    for logits, k in cases:
        T, E = logits.shape
        got = _route_noalloc_c_abi(Q, torch.from_numpy(logits).cuda(), T, E, k)
        rids, _, roff, rsp = OM.route(logits, k)
        assert np.array_equal(got[0].numpy(), rids)
        assert np.array_equal(got[1].numpy(), rsp)
        assert np.array_equal(got[2].numpy(), roff)
