"""Asymmetric INT4 (unsigned codes, a BF16 scale and a zero point per group of 128:
w = s (q - z)) through every W4A16 path - staged decode GEMV, register-ring GEMV, grouped
TMA-ring GEMV and the tcgen05 kernel - against the float64 oracle; repack round trip bit for
bit; with every zero point 8 the results equal the symmetric INT4 kernels' bit for bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import moe as OM
from oracle import qgemm as OQ
from qwtest import dense_w4a16, dev, host, qw, repack, route, u16_view

pytestmark = pytest.mark.gpu


def dense_zp(p, bias=None):
    Q = qw()
    N, K = p["N"], p["K"]
    d, wp, sp = repack(Q.QW_W_UINT4ZP_G128_BF16, 1, N, K, p["w_canon"], p["s_canon"])
    M = p["A"].shape[0]
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, dev(p["A"].view(np.int16)), None, b, C, M, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


@pytest.mark.parametrize("M,N,K", [(1, 200, 512), (1, 8192, 4096), (3, 40, 384), (8, 256, 1024),
                                   (13, 96, 256), (48, 384, 1024), (300, 1280, 640)])
def test_zp_dense_paths(M, N, K):
    """M = 1 over 32 M weights: staged GEMV; other M <= 16: register ring; M > 16: tcgen05."""
    p = synth.w4a16_zp_problem(M, N, K, cfg_id=800 + M)
    C = dense_zp(p)
    R, S = OQ.w4a16_zp_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K)
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("M", [5, 64])
def test_zp_bias(M):
    p = synth.w4a16_zp_problem(M, 72, 256, cfg_id=850 + M, bias=True)
    C = dense_zp(p, bias=p["bias"][0])
    R, S = OQ.w4a16_zp_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 256,
                                      bias_bits=p["bias"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


def _as_zero_point_8(p, N, K):
    q = OF.unpack_int4(p["w_canon"][0], K).astype(np.int64) + 8
    words = np.ascontiguousarray(synth.pack_nibbles(q.astype(np.uint8))).view("<u4")
    sz = p["s_canon"][0].astype(np.uint32) | np.uint32(8 << 16)
    return dict(A=p["A"], w_canon=words[None].astype(np.uint32), s_canon=sz[None], N=N, K=K)


@pytest.mark.parametrize("M,N,K", [(5, 100, 256), (40, 256, 512)])
def test_zp_with_zero_point_8_equals_symmetric_int4(M, N, K):
    """q + 8 with z = 8 is the symmetric code: same kernels' arithmetic, same bits."""
    p = synth.w4a16_problem(M, N, K, bits=4, cfg_id=860 + M)
    C_sym = dense_w4a16(p)
    assert np.array_equal(dense_zp(_as_zero_point_8(p, N, K)), C_sym)


def test_zp_with_zero_point_8_single_token():
    """Single-token decode: symmetric INT4 runs the FP16-operand decode kernel and the
    asymmetric format the staged BF16 kernel, so the two round differently; with z = 8 both
    match the same oracle result."""
    M, N, K = 1, 8192, 4096
    p = synth.w4a16_problem(M, N, K, bits=4, cfg_id=861)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, 4)
    for C in (dense_w4a16(p), dense_zp(_as_zero_point_8(p, N, K))):
        ok, ratio, frob = OQ.check_bf16_result(C, R, S)
        assert ok, (ratio, frob)


def test_zp_repack_round_trip_and_value_flag():
    Q = qw()
    E, N, K = 3, 40, 384
    p = synth.w4a16_zp_problem(1, N, K, E=E, cfg_id=870)
    d, wp, sp = repack(Q.QW_W_UINT4ZP_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
    assert d.s_expert_stride == 2 * 256 * ((3 * 48 * 2 + 255) // 256)
    wc = torch.empty((E, N, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((E, N, K // 128), dtype=torch.int32, device="cuda")
    Q.qw_unpack(d, wp, sp, wc, sc)
    assert np.array_equal(host(wc).view(np.uint32), p["w_canon"])
    assert np.array_equal(host(sc).view(np.uint32), p["s_canon"])
    bad = p["s_canon"].copy()
    bad[2, 5, 1] = (bad[2, 5, 1] & 0xFFFF) | (16 << 16)  # zero point 16
    wp2, sp2 = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(p["w_canon"]), dev(bad), wp2, sp2, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


@pytest.mark.parametrize("T", [12, 32])
def test_zp_grouped_moe(T):
    """E = 8 top-8: 12 rows per expert (grouped TMA-ring GEMV) and 32 (tcgen05)."""
    Q = qw()
    E, K, N, k = 8, 512, 256, 8
    p = synth.w4a16_zp_problem(T, N, K, E=E, cfg_id=880 + T)
    logits = synth.router_logits(T, E, cfg_id=880 + T)
    d, wp, sp = repack(Q.QW_W_UINT4ZP_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
    ids, spairs, off = route(logits, k)
    P = T * k
    A = dev(p["A"].view(np.int16))
    As = torch.empty((P, K), dtype=torch.int16, device="cuda")
    sp_dev, off_dev = dev(spairs.astype(np.int32)), dev(off.astype(np.int32))
    Q.qgemm_moe_permute(Q.QW_A_BF16, A, None, K, sp_dev, P, k, As, None)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, Q.QW_A_BF16, As, None, off_dev, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    tok = spairs // k
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        R, S = OQ.w4a16_zp_from_canonical(p["A"][tok[sel]], p["w_canon"][e], p["s_canon"][e], K)
        ok, ratio, frob = OQ.check_bf16_result(Cn[sel], R, S)
        assert ok, (e, ratio, frob)
