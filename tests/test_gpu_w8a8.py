"""W8A8 (MXFP8 weights x MXFP8 activations, group-32 E8M0) on the block-scaled tcgen05
kernel, against the float64 oracle; repack round trip bit for bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from oracle import moe as OM
from qwtest import dense_w4a8, dev, host, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def _check(C, p, bias=None):
    R, S = OQ.gemm_w8a8(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], bias_bits=bias)
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (128, 256, 128), (200, 384, 512),
                                   (300, 1000, 1024)])
def test_w8a8_shapes(M, N, K):
    Q = qw()
    p = synth.w8a8_problem(M, N, K, cfg_id=600 + M)
    _check(dense_w4a8(p, wfmt=Q.QW_W_MXFP8_G32), p)


def test_w8a8_k_not_multiple_of_128_and_bias():
    Q = qw()
    p = synth.w8a8_problem(130, 260, 96, cfg_id=650, bias=True)
    C = dense_w4a8(p, bias=p["bias"][0], wfmt=Q.QW_W_MXFP8_G32)
    _check(C, p, bias=p["bias"][0])


def test_w8a8_full_size_sampled_rows():
    """(4096, 14336, 4096): the whole GEMM on the GPU, 64 sampled rows checked."""
    Q = qw()
    M, N, K = 4096, 14336, 4096
    p = synth.w8a8_problem(M, N, K, cfg_id=660)
    C = dense_w4a8(p, wfmt=Q.QW_W_MXFP8_G32)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(1).choice(M, 62, False)]))
    R, S = OQ.gemm_w8a8(p["A"][rows], p["A_sf"][rows], p["w_canon"][0], p["s_canon"][0])
    ok, ratio, frob = OQ.check_bf16_result(C[rows], R, S)
    assert ok, (ratio, frob)


def test_mxfp8_repack_round_trip_and_nan_flag():
    Q = qw()
    E, N, K = 2, 200, 96
    p = synth.w8a8_problem(1, N, K, E=E, cfg_id=670)
    d, wp, sp = repack(Q.QW_W_MXFP8_G32, E, N, K, p["w_canon"], p["s_canon"])
    assert d.N_pad == 256 and d.K_pad == 128 and d.w_bytes == E * 256 * 128
    wc = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty((E, N, K // 32), dtype=torch.uint8, device="cuda")
    Q.qw_unpack(d, wp, sp, wc, sc)
    assert np.array_equal(host(wc), p["w_canon"]) and np.array_equal(host(sc), p["s_canon"])
    bad = p["w_canon"].copy()
    bad[1, 7, 33] = 0xFF  # E4M3 NaN
    wp2, sp2 = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(bad), dev(p["s_canon"]), wp2, sp2, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


def test_w8a8_grouped_moe_small():
    Q = qw()
    E, T, K, N, k = 8, 40, 256, 384, 2
    p = synth.w8a8_problem(T, N, K, E=E, cfg_id=680)
    logits = synth.router_logits(T, E, cfg_id=680)
    d, wp, sp = repack(Q.QW_W_MXFP8_G32, E, N, K, p["w_canon"], p["s_canon"])
    P = T * k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    spairs = torch.empty((P,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, k)
    rws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_route(dev(logits), T, E, k, ids, spairs, off, rws, n)
    A, Asf = dev(p["A"]), dev(p["A_sf"])
    As = torch.empty((P, K), dtype=torch.uint8, device="cuda")
    Asf_s = torch.empty((P, K // 32), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_permute(Q.QW_A_MXFP8_G32, A, Asf, K, spairs, P, k, As, Asf_s)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_MXFP8_G32, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, Q.QW_A_MXFP8_G32, As, Asf_s, off, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    roff, rsp = host(off), host(spairs)
    tok = rsp // k
    e_of = np.searchsorted(roff, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        R, S = OQ.gemm_w8a8(p["A"][tok[sel]], p["A_sf"][tok[sel]], p["w_canon"][e],
                            p["s_canon"][e])
        ok, ratio, frob = OQ.check_bf16_result(Cn[sel], R, S)
        assert ok, (e, ratio, frob)
