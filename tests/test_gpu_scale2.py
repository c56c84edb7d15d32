"""Second-level scales (QW_W_SCALE2: an FP32 scale per output channel and expert applied to
the finished sum before the bias) through every GEMM path, against the oracle's
apply_scale2; with every scale 1.0 (what qw_repack leaves) the results equal the base
format's bit for bit; the packed plane round-trips and rejects non-finite scales."""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from qwtest import dev, host, qw, route, u16_view

pytestmark = pytest.mark.gpu


def _problem(kind, M, N, K, E=1, cfg_id=0):
    Q = qw()
    if kind in (4, 3, 2):
        p = synth.w4a16_problem(M, N, K, bits=kind, E=E, cfg_id=cfg_id)
        wfmt = {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16, 2: Q.QW_W_INT2_G128_BF16}[kind]
        return p, wfmt, Q.QW_A_BF16
    if kind == "fp8":
        return synth.fp8w_problem(M, N, K, E=E, cfg_id=cfg_id), Q.QW_W_FP8E4M3_G128_BF16, Q.QW_A_BF16
    if kind == "w4a8":
        return synth.w4a8_problem(M, N, K, E=E, cfg_id=cfg_id), Q.QW_W_MXFP4_G32, Q.QW_A_MXFP8_G32
    if kind == "w8a8":
        return synth.w8a8_problem(M, N, K, E=E, cfg_id=cfg_id), Q.QW_W_MXFP8_G32, Q.QW_A_MXFP8_G32
    return synth.w4a4_problem(M, N, K, E=E, cfg_id=cfg_id), Q.QW_W_NVFP4_G16, Q.QW_A_NVFP4_G16


def _oracle(kind, p, e, rows, K):
    """(R, absum) without bias for expert e and activation rows `rows`."""
    A = p["A"][rows]
    if kind in (4, 3, 2):
        return OQ.w4a16_from_canonical(A, p["w_canon"][e], p["s_canon"][e], K, kind)
    if kind == "fp8":
        return OQ.fp8w_from_canonical(A, p["w_canon"][e], p["s_canon"][e])
    if kind == "w4a8":
        return OQ.w4a8_from_canonical(A, p["A_sf"][rows], p["w_canon"][e], p["s_canon"][e], K)
    if kind == "w8a8":
        return OQ.gemm_w8a8(A, p["A_sf"][rows], p["w_canon"][e], p["s_canon"][e])
    return OQ.w4a4_from_canonical(A, p["A_sf"][rows], p["w_canon"][e], p["s_canon"][e], K)


def _pack(wfmt, E, N, K, p, t=None, flag=True):
    Q = qw()
    d = Q.qw_repack_query(wfmt | (Q.QW_W_SCALE2 if flag else 0), E, N, K)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(p["w_canon"]), dev(p["s_canon"]), wp, sp, err)
    if t is not None:
        Q.qw_repack_scale2(d, dev(t), sp, err)
    assert Q.qw_read_error(err) == 0
    return d, wp, sp


def _dense(afmt, d, wp, sp, p, bias=None):
    Q = qw()
    M, N = p["A"].shape[0], d.N
    A = dev(p["A"].view(np.int16)) if afmt == Q.QW_A_BF16 else dev(p["A"])
    Asf = None if afmt == Q.QW_A_BF16 else dev(p["A_sf"])
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, afmt, M)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, afmt, A, Asf, b, C, M, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


def _scales(E, N, seed):
    rng = np.random.default_rng(seed)
    t = rng.uniform(0.25, 4.0, (E, N)) * np.where(rng.random((E, N)) < 0.2, -1.0, 1.0)
    return t.astype(np.float32)


# (kind, M, N, K): the staged decode GEMV, the register ring, tcgen05 W4A16, FP8 weights,
# the W4A8 GEMV and block-scaled GEMMs of the three MX kinds
DENSE = [(4, 1, 8192, 4096), (4, 5, 200, 512), (3, 12, 136, 384), (4, 48, 264, 640),
         ("fp8", 40, 136, 256), ("w4a8", 1, 512, 1024), ("w4a8", 200, 264, 512),
         ("w8a8", 130, 256, 256), ("w4a4", 129, 256, 512)]


@pytest.mark.parametrize("kind,M,N,K", DENSE)
def test_scale2_of_ones_equals_the_base_format(kind, M, N, K):
    p, wfmt, afmt = _problem(kind, M, N, K, cfg_id=1100 + M)
    bias = synth.to_bf16_bits(np.random.default_rng(M).normal(size=N))
    C0 = _dense(afmt, *_pack(wfmt, 1, N, K, p, flag=False), p, bias)
    C1 = _dense(afmt, *_pack(wfmt, 1, N, K, p, flag=True), p, bias)
    assert np.array_equal(C0, C1)


@pytest.mark.parametrize("kind,M,N,K", DENSE)
def test_scale2_dense_against_the_oracle(kind, M, N, K):
    p, wfmt, afmt = _problem(kind, M, N, K, cfg_id=1150 + M)
    t = _scales(1, N, 1150 + M)
    bias = synth.to_bf16_bits(np.random.default_rng(M + 1).normal(size=N))
    C = _dense(afmt, *_pack(wfmt, 1, N, K, p, t=t), p, bias)
    R, S = _oracle(kind, p, 0, np.arange(M), K)
    R, S = OQ.apply_scale2(R, S, t[0], bias)
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("kind,T", [(4, 12), (4, 32), ("fp8", 12), ("w4a8", 40)])
def test_scale2_grouped_per_expert(kind, T):
    """E = 8 top-8 with a different t per expert: grouped GEMV (12 rows per expert), tcgen05
    W4A16 (32) and the block-scaled GEMM; the W4A8 case also runs the indexed call."""
    Q = qw()
    E, K, N, k = 8, 512, 264, 8
    p, wfmt, afmt = _problem(kind, T, N, K, E=E, cfg_id=1200 + T)
    t = _scales(E, N, 1200 + T)
    d, wp, sp = _pack(wfmt, E, N, K, p, t=t)
    logits = synth.router_logits(T, E, cfg_id=1200 + T)
    ids, spairs, off = route(logits, k)
    P = T * k
    sp_dev, off_dev = dev(spairs.astype(np.int32)), dev(off.astype(np.int32))
    if afmt == Q.QW_A_BF16:
        A, Asf = dev(p["A"].view(np.int16)), None
        As, Asf_s = torch.empty((P, K), dtype=torch.int16, device="cuda"), None
    else:
        A, Asf = dev(p["A"]), dev(p["A_sf"])
        As = torch.empty((P, K), dtype=torch.uint8, device="cuda")
        Asf_s = torch.empty((P, K // 32), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_permute(afmt, A, Asf, K, sp_dev, P, k, As, Asf_s)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, afmt, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, afmt, As, Asf_s, off_dev, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    outs = [u16_view(C)]
    if kind == "w4a8":
        Ci = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
        Q.qgemm_moe_grouped_indexed(d, wp, sp, afmt, A, Asf, T, sp_dev, k, off_dev, P, None, Ci,
                                    ws, wsn, err)
        assert Q.qw_read_error(err) == 0
        outs.append(u16_view(Ci))
    tok = spairs // k
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1
    for Cn in outs:
        for e in np.unique(e_of):
            sel = np.nonzero(e_of == e)[0]
            R, S = _oracle(kind, p, e, tok[sel], K)
            R, S = OQ.apply_scale2(R, S, t[e])
            ok, ratio, frob = OQ.check_bf16_result(Cn[sel], R, S)
            assert ok, (e, ratio, frob)


def test_scale2_round_trip_and_non_finite_flag():
    Q = qw()
    E, N, K = 3, 200, 256
    p, wfmt, _ = _problem(4, 1, N, K, E=E, cfg_id=1250)
    t = _scales(E, N, 1250)
    d, wp, sp = _pack(wfmt, E, N, K, p, t=t)
    back = torch.empty((E, N), dtype=torch.float32, device="cuda")
    Q.qw_unpack_scale2(d, sp, back)
    assert np.array_equal(host(back), t)
    d1, wp1, sp1 = _pack(wfmt, E, N, K, p)  # qw_repack alone leaves 1.0
    Q.qw_unpack_scale2(d1, sp1, back)
    assert np.array_equal(host(back), np.ones((E, N), np.float32))
    for bad_v in (np.nan, np.inf):
        bad = t.copy()
        bad[1, 7] = bad_v
        err = Q.new_error_flag()
        Q.qw_repack_scale2(d, dev(bad), sp, err)
        assert Q.qw_read_error(err) == Q.QW_ERR_VALUE
