"""Grouped-MoE GEMMs at the full workload sizes, inputs drawn on the device.

The kernels run the whole problem; the float64 oracle checks sampled output rows (first,
last and middle row of sampled non-empty experts, always including the largest and the
smallest) against sampled columns, and the routing bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import moe as OM
from oracle import qgemm as OQ
from qwtest import host, moe_pipeline, qw, sample_rows_per_expert, u16_view

pytestmark = pytest.mark.gpu


def _cols(N, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(40), np.arange(N - 40, N),
                                     rng.choice(N, 96, replace=False)]))


def _check(r, rows, cols, oracle_rows):
    C = u16_view(r["C"])[rows][:, cols]
    R, S = oracle_rows
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, f"worst |err|/bound {ratio:.3g}, rel frob {frob:.3g}"


def _expert_of(off, rows):
    return np.searchsorted(off, rows, side="right") - 1


def test_config4_moe_w4a8_full_size():
    """E=256, top-8, T=4096, K=7168 -> N=4096 (fused gate+up), MXFP4 x MXFP8 group-32."""
    Q = qw()
    E, T, K, N, k = 256, 4096, 7168, 4096, 8
    r = moe_pipeline(Q.QW_A_MXFP8_G32, Q.QW_W_MXFP4_G32, E, T, K, N, k, cfg_id=3)
    r["route"]()
    r["permute"]()
    r["gemm"]()
    assert Q.qw_read_error(r["err"]) == 0
    off, sp = host(r["offsets"]), host(r["sorted_pairs"])
    _, _, roff, rsp = OM.route(r["logits"], k)
    assert np.array_equal(off, roff) and np.array_equal(sp, rsp)
    # every active expert, its first and last row (and a middle one)
    rows = sample_rows_per_expert(off, per_expert=3, max_experts=None, seed=1)
    assert np.unique(_expert_of(off, rows)).size == np.count_nonzero(np.diff(off))
    cols = _cols(N, 2)
    tok = sp[rows] // k
    A, Asf = host(r["A"])[tok], host(r["A_sf"])[tok]
    exp = _expert_of(off, rows)
    ct = torch.from_numpy(cols).cuda()
    R = np.zeros((rows.size, cols.size))
    S = np.zeros_like(R)
    for e in np.unique(exp):
        sel = np.nonzero(exp == e)[0]
        w = host(r["w_canon"][int(e)].index_select(0, ct))
        sf = host(r["s_canon"][int(e)].index_select(0, ct))
        R[sel], S[sel] = OQ.gemm_w4a8(A[sel], Asf[sel], OF.unpack_e2m1_bytes(w, K), sf)
    _check(r, rows, cols, (R, S))


def _w4a16_case(T, up, bits=4):
    Q = qw()
    import synth.device as sd
    E, k = 128, 8
    K, N = (4096, 1280) if up else (640, 4096)
    x_sorted = None if up else sd.bf16_activations(T * k, K, cfg_id=40 + T)
    wfmt = Q.QW_W_INT4_G128_BF16 if bits == 4 else Q.QW_W_INT3_G128_BF16
    r = moe_pipeline(Q.QW_A_BF16, wfmt, E, T, K, N, k, cfg_id=4, bits=bits, x_sorted=x_sorted)
    r["route"]()
    r["permute"]()
    r["gemm"]()
    assert Q.qw_read_error(r["err"]) == 0
    off, sp = host(r["offsets"]), host(r["sorted_pairs"])
    rows = sample_rows_per_expert(off, per_expert=3, max_experts=16, seed=T)
    cols = _cols(N, T)
    if up:
        A = host(r["A"]).view(np.uint16)[sp[rows] // k]
    else:
        A = host(x_sorted).view(np.uint16)[rows]
    exp = _expert_of(off, rows)
    ct = torch.from_numpy(cols).cuda()
    R = np.zeros((rows.size, cols.size))
    S = np.zeros_like(R)
    for e in np.unique(exp):
        sel = np.nonzero(exp == e)[0]
        w = host(r["w_canon"][int(e)].index_select(0, ct)).view(np.uint32)
        s = host(r["s_canon"][int(e)].index_select(0, ct)).view(np.uint16)
        q = OF.unpack_int4(w, K) if bits == 4 else OF.unpack_int3(w, K)
        R[sel], S[sel] = OQ.gemm_w4a16(A[sel], q, s)
    _check(r, rows, cols, (R, S))


@pytest.mark.parametrize("T", [1, 16, 256, 2048, 8192])
def test_config5_moe_w4a16_up_projection(T):
    """E=128, top-8, hidden 4096 -> gate+up 1280, INT4 group-128, token sweep."""
    _w4a16_case(T, up=True)


@pytest.mark.parametrize("T", [1, 16, 256, 2048, 8192])
def test_config5_moe_w4a16_down_projection(T):
    """Down projection 640 -> 4096 (K not a multiple of 256) on a per-pair input."""
    _w4a16_case(T, up=False)


def test_config5_moe_w3a16_up_projection_t16():
    _w4a16_case(16, up=True, bits=3)
