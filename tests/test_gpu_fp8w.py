"""FP8-weight WnA16 (E4M3 codes with a BF16 scale per group of 128, BF16 activations)
through every W4A16-family path - staged decode GEMV, register-ring GEMV, grouped TMA-ring
GEMV and the tcgen05 kernel - against the float64 oracle; repack round trip bit for bit;
on E4M3 codes of integers the results equal the INT4 kernels' bit for bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import qgemm as OQ
from qwtest import dense_fp8w, dense_w4a16, dev, host, qw, repack, route, u16_view

pytestmark = pytest.mark.gpu


def _e4m3_of_ints(q):
    t = torch.from_numpy(np.asarray(q, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("M,N,K", [(1, 200, 512), (1, 8192, 4096), (3, 40, 384), (8, 256, 1024),
                                   (13, 96, 256), (16, 264, 640), (48, 384, 1024),
                                   (300, 1280, 640), (130, 136, 128)])
def test_fp8w_dense_paths(M, N, K):
    """M = 1 over 32 M weights: staged GEMV; other M <= 16: register ring; M > 16: tcgen05.
    Ragged N (not a multiple of 16 / 128) and K of one to eight groups."""
    p = synth.fp8w_problem(M, N, K, cfg_id=900 + M)
    C = dense_fp8w(p)
    R, S = OQ.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("M", [1, 5, 64])
def test_fp8w_bias(M):
    p = synth.fp8w_problem(M, 72, 256, cfg_id=950 + M, bias=True)
    C = dense_fp8w(p, bias=p["bias"][0])
    R, S = OQ.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], p["bias"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("M,N,K", [(17, 100, 256), (40, 256, 512), (200, 136, 384)])
def test_fp8w_on_integer_codes_equals_int4(M, N, K):
    """E4M3 codes of the INT4 weights -7..7 on the tcgen05 path, where the INT4 kernel
    removes the excess exactly in BF16 before the MMA: the same operands in the same order,
    so the same bits.  (The INT4 GEMVs subtract the excess after the MMA, a different
    rounding; the oracle checks those paths.)"""
    p = synth.w4a16_problem(M, N, K, bits=4, cfg_id=960 + M)
    C_int4 = dense_w4a16(p)
    q = OF.unpack_int4(p["w_canon"][0], K)
    pf = dict(A=p["A"], w_canon=_e4m3_of_ints(q)[None], s_canon=p["s_canon"], N=N, K=K)
    assert np.array_equal(dense_fp8w(pf), C_int4)


def test_fp8w_full_size_decode_sampled():
    """(1, 14336, 4096): the decode shape of the bench, every output checked."""
    p = synth.fp8w_problem(1, 14336, 4096, cfg_id=970)
    C = dense_fp8w(p)
    R, S = OQ.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


def test_fp8w_repack_round_trip_and_nan_flag():
    Q = qw()
    E, N, K = 3, 40, 384
    p = synth.fp8w_problem(1, N, K, E=E, cfg_id=975)
    d, wp, sp = repack(Q.QW_W_FP8E4M3_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
    assert d.N_pad == 48 and d.w_bytes == E * 3 * 3 * 2048 and d.group == 128
    wc = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty((E, N, K // 128), dtype=torch.int16, device="cuda")
    Q.qw_unpack(d, wp, sp, wc, sc)
    assert np.array_equal(host(wc), p["w_canon"])
    assert np.array_equal(host(sc).view(np.uint16), p["s_canon"])
    for nan in (0x7F, 0xFF):
        bad = p["w_canon"].copy()
        bad[2, 39, 383] = nan
        wp2, sp2 = Q.empty_packed(d)
        err = Q.new_error_flag()
        Q.qw_repack(d, dev(bad), dev(p["s_canon"]), wp2, sp2, err)
        assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


def test_fp8w_packed_layout_of_one_block():
    """Byte b of word 2s + j of lane 4g + t is the code of row g + 8 (b >> 1) at
    k = 16s + 4t + 2j + (b & 1) - read back from the packed buffer for one block."""
    Q = qw()
    N, K = 16, 128
    codes = np.zeros((1, N, K), np.uint8)
    rng = np.random.default_rng(3)
    codes[0] = rng.integers(0, 0x7F, (N, K), dtype=np.uint8)
    d, wp, sp = repack(Q.QW_W_FP8E4M3_G128_BF16, 1, N, K, codes,
                       np.full((1, N, 1), 0x3F80, np.uint16))
    words = host(wp)[:2048].view("<u4").reshape(32, 16)
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        for u in range(16):
            s, j = u >> 1, u & 1
            for b in range(4):
                row, k = g + 8 * (b >> 1), 16 * s + 4 * t + 2 * j + (b & 1)
                assert (int(words[lane, u]) >> (8 * b)) & 0xFF == codes[0, row, k]


@pytest.mark.parametrize("T", [12, 32])
def test_fp8w_grouped_moe(T):
    """E = 8 top-8: 12 rows per expert (grouped TMA-ring GEMV) and 32 (tcgen05)."""
    Q = qw()
    E, K, N, k = 8, 512, 264, 8
    p = synth.fp8w_problem(T, N, K, E=E, cfg_id=980 + T)
    logits = synth.router_logits(T, E, cfg_id=980 + T)
    d, wp, sp = repack(Q.QW_W_FP8E4M3_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
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
        R, S = OQ.fp8w_from_canonical(p["A"][tok[sel]], p["w_canon"][e], p["s_canon"][e])
        ok, ratio, frob = OQ.check_bf16_result(Cn[sel], R, S)
        assert ok, (e, ratio, frob)
