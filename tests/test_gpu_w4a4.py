"""W4A4 (NVFP4 weights x NVFP4 activations: E2M1 with an unsigned E4M3 scale per 16) on the
block-scaled tcgen05 kernel (kind::mxf4nvf4, scale_vec::4X), against the float64 oracle;
repack round trip bit for bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import qgemm as OQ
from qwtest import dev, host, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def dense_w4a4(p, bias=None):
    Q = qw()
    N, K = p["N"], p["K"]
    d, wp, sp = repack(Q.QW_W_NVFP4_G16, 1, N, K, p["w_canon"], p["s_canon"])
    M = p["A"].shape[0]
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_NVFP4_G16, M)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_NVFP4_G16, dev(p["A"]), dev(p["A_sf"]), b, C, M, ws, wsn,
                  err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


def _oracle(p, rows=None, bias=None):
    return OQ.w4a4_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], p["K"],
                                  bias_bits=bias, rows=rows)


def test_w4a4_single_tile_integer_exact():
    """Unit scales and integer-valued E2M1 codes: one 128 x 256 x 256 tile is exact."""
    rng = np.random.default_rng(8)
    M, N, K = 128, 256, 256
    ints = [0, 2, 4, 5, 10, 12, 13]  # E2M1 codes of 0, 1, 2, 3, -1, -2, -3
    A = synth.pack_nibbles(rng.choice(ints, (M, K)).astype(np.uint8))
    W = synth.pack_nibbles(rng.choice(ints, (N, K)).astype(np.uint8))
    p = dict(A=A, A_sf=np.full((M, K // 16), 0x38, np.uint8), w_canon=W[None],
             s_canon=np.full((1, N, K // 16), 0x38, np.uint8), N=N, K=K)
    C = dense_w4a4(p)
    R, _ = _oracle(p)
    assert np.array_equal(C, synth.to_bf16_bits(R)), f"{np.sum(C != synth.to_bf16_bits(R))} differ"


def test_w4a4_distinct_scale_per_16_group():
    """Power-of-two scales that differ for every 16-group and row: an exact result, so a
    scale read from the wrong group, row or MMA shows up as a mismatch."""
    rng = np.random.default_rng(9)
    M, N, K = 128, 256, 512
    ints = [0, 2, 4, 5, 10, 12, 13]
    A = synth.pack_nibbles(rng.choice(ints, (M, K)).astype(np.uint8))
    W = synth.pack_nibbles(rng.choice(ints, (N, K)).astype(np.uint8))
    pow2 = lambda e: ((e + 7) << 3).astype(np.uint8)  # noqa: E731  E4M3 code of 2^e
    Asf = pow2(rng.integers(-3, 4, (M, K // 16)))
    Wsf = pow2(rng.integers(-3, 4, (N, K // 16)))
    p = dict(A=A, A_sf=Asf, w_canon=W[None], s_canon=Wsf[None], N=N, K=K)
    C = dense_w4a4(p)
    R, _ = _oracle(p)
    assert np.array_equal(C, synth.to_bf16_bits(R)), f"{np.sum(C != synth.to_bf16_bits(R))} differ"


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 300, 512), (64, 264, 320),
                                   (1, 256, 256), (384, 3072, 1024)])
def test_w4a4_shapes(M, N, K):
    p = synth.w4a4_problem(M, N, K, cfg_id=700 + M)
    C = dense_w4a4(p)
    R, S = _oracle(p)
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


def test_w4a4_bias_and_k_not_multiple_of_256():
    p = synth.w4a4_problem(130, 260, 96, cfg_id=750, bias=True)
    C = dense_w4a4(p, bias=p["bias"][0])
    R, S = _oracle(p, bias=p["bias"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


def test_w4a4_full_size_sampled_rows():
    """(4096, 14336, 4096): the whole GEMM on the GPU, 64 sampled rows checked."""
    M, N, K = 4096, 14336, 4096
    p = synth.w4a4_problem(M, N, K, cfg_id=760)
    C = dense_w4a4(p)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(2).choice(M, 62, False)]))
    R, S = _oracle(p, rows=rows)
    ok, ratio, frob = OQ.check_bf16_result(C[rows], R, S)
    assert ok, (ratio, frob)


def test_nvfp4_repack_round_trip_and_scale_flags():
    Q = qw()
    E, N, K = 2, 200, 96
    p = synth.w4a4_problem(1, N, K, E=E, cfg_id=770)
    d, wp, sp = repack(Q.QW_W_NVFP4_G16, E, N, K, p["w_canon"], p["s_canon"])
    assert d.N_pad == 256 and d.K_pad == 256 and d.group == 16
    assert d.w_bytes == E * 256 * 128 and d.s_bytes == E * 2 * 1 * 2048
    wc = torch.empty((E, N, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((E, N, K // 16), dtype=torch.uint8, device="cuda")
    Q.qw_unpack(d, wp, sp, wc, sc)
    assert np.array_equal(host(wc), p["w_canon"]) and np.array_equal(host(sc), p["s_canon"])
    for bad_code in (0xB8, 0x7F):  # a negative scale, the NaN code
        bad = p["s_canon"].copy()
        bad[1, 7, 3] = bad_code
        wp2, sp2 = Q.empty_packed(d)
        err = Q.new_error_flag()
        Q.qw_repack(d, dev(p["w_canon"]), dev(bad), wp2, sp2, err)
        assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


def test_w4a4_grouped_moe_small():
    Q = qw()
    E, T, K, N, k = 8, 40, 512, 384, 2
    p = synth.w4a4_problem(T, N, K, E=E, cfg_id=780)
    logits = synth.router_logits(T, E, cfg_id=780)
    d, wp, sp = repack(Q.QW_W_NVFP4_G16, E, N, K, p["w_canon"], p["s_canon"])
    P = T * k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    spairs = torch.empty((P,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, k)
    rws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_route(dev(logits), T, E, k, ids, spairs, off, rws, n)
    A, Asf = dev(p["A"]), dev(p["A_sf"])
    As = torch.empty((P, K // 2), dtype=torch.uint8, device="cuda")
    Asf_s = torch.empty((P, K // 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_permute(Q.QW_A_NVFP4_G16, A, Asf, K, spairs, P, k, As, Asf_s)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_NVFP4_G16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, Q.QW_A_NVFP4_G16, As, Asf_s, off, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    Ci = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    Q.qgemm_moe_grouped_indexed(d, wp, sp, Q.QW_A_NVFP4_G16, A, Asf, T, spairs, k, off, P, None,
                                Ci, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    assert np.array_equal(u16_view(C), u16_view(Ci))
    roff, rsp = host(off), host(spairs)
    tok = rsp // k
    e_of = np.searchsorted(roff, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    a_codes = OF.unpack_e2m1_bytes(p["A"], K)
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        R, S = OQ.gemm_w4a4(a_codes[tok[sel]], p["A_sf"][tok[sel]],
                            OF.unpack_e2m1_bytes(p["w_canon"][e], K), p["s_canon"][e])
        ok, ratio, frob = OQ.check_bf16_result(Cn[sel], R, S)
        assert ok, (e, ratio, frob)
