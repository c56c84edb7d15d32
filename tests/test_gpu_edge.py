"""Degenerate and boundary cases through the C ABI: no rows, one output channel, one scale
group, all-zero weights or scales (the output is the bias exactly), for every weight format."""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from qwtest import dev, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def _problem(kind, M, N, K, cfg_id):
    Q = qw()
    if kind in (4, 3, 2):
        p = synth.w4a16_problem(M, N, K, bits=kind, cfg_id=cfg_id)
        return p, {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16,
                   2: Q.QW_W_INT2_G128_BF16}[kind], Q.QW_A_BF16
    if kind == "zp":
        return synth.w4a16_zp_problem(M, N, K, cfg_id=cfg_id), Q.QW_W_UINT4ZP_G128_BF16, Q.QW_A_BF16
    if kind == "fp8":
        return synth.fp8w_problem(M, N, K, cfg_id=cfg_id), Q.QW_W_FP8E4M3_G128_BF16, Q.QW_A_BF16
    if kind == "w4a8":
        return synth.w4a8_problem(M, N, K, cfg_id=cfg_id), Q.QW_W_MXFP4_G32, Q.QW_A_MXFP8_G32
    if kind == "w8a8":
        return synth.w8a8_problem(M, N, K, cfg_id=cfg_id), Q.QW_W_MXFP8_G32, Q.QW_A_MXFP8_G32
    return synth.w4a4_problem(M, N, K, cfg_id=cfg_id), Q.QW_W_NVFP4_G16, Q.QW_A_NVFP4_G16


def _run(d, wp, sp, afmt, p, M, bias=None, fill=-1):
    Q = qw()
    A = dev(p["A"].view(np.int16)) if afmt == Q.QW_A_BF16 else dev(p["A"])
    Asf = None if afmt == Q.QW_A_BF16 else dev(p["A_sf"])
    C = torch.full((max(M, 1), d.N), fill, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, afmt, max(M, 1))
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, afmt, A, Asf, b, C, M, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


KINDS = [4, 3, 2, "zp", "fp8", "w4a8", "w8a8", "w4a4"]


@pytest.mark.parametrize("kind", KINDS)
def test_zero_rows_is_a_no_op(kind):
    p, wfmt, afmt = _problem(kind, 4, 64, 256, cfg_id=1300)
    d, wp, sp = repack(wfmt, 1, 64, 256, p["w_canon"], p["s_canon"])
    C = _run(d, wp, sp, afmt, p, 0)
    assert np.all(C == 0xFFFF)  # untouched


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M", [1, 40])
def test_one_output_channel_and_minimal_k(kind, M):
    """N = 1 (the rest of the 16- or 128-row padding is zero codes) and the smallest K of the
    format: one BF16 scale group, or one 32/16-element MX group."""
    K = {"w4a8": 32, "w8a8": 32, "w4a4": 32}.get(kind, 128)
    p, wfmt, afmt = _problem(kind, M, 1, K, cfg_id=1310 + M)
    d, wp, sp = repack(wfmt, 1, 1, K, p["w_canon"], p["s_canon"])
    bias = synth.to_bf16_bits(np.array([0.75]))
    C = _run(d, wp, sp, afmt, p, M, bias)
    if kind in (4, 3, 2):
        R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, kind, bias)
    elif kind == "zp":
        R, S = OQ.w4a16_zp_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bias)
    elif kind == "fp8":
        R, S = OQ.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], bias)
    elif kind == "w4a8":
        R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K, bias)
    elif kind == "w8a8":
        R, S = OQ.gemm_w8a8(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], bias)
    else:
        R, S = OQ.w4a4_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K, bias)
    # one output per row: the element-wise bound is the meaningful one here
    ok_elem = np.all(np.abs(OQ.F.decode_bf16(C) - R) <= 2.0 ** -7 * S + 1e-6)
    assert ok_elem


@pytest.mark.parametrize("kind", [4, 3, "fp8", "w4a8"])
@pytest.mark.parametrize("M", [1, 12, 64])
def test_zero_scales_give_the_bias_exactly(kind, M):
    """Every group scale zero (BF16 0, or E8M0 with the smallest code for MX: not zero, so
    MX uses zero codes instead): the output is the BF16 bias, bit for bit."""
    N, K = 136, 512
    p, wfmt, afmt = _problem(kind, M, N, K, cfg_id=1330 + M)
    if kind == "w4a8":
        p = dict(p, w_canon=np.zeros_like(p["w_canon"]))
    else:
        p = dict(p, s_canon=np.zeros_like(p["s_canon"]))
    d, wp, sp = repack(wfmt, 1, N, K, p["w_canon"], p["s_canon"])
    bias = synth.to_bf16_bits(np.random.default_rng(M).normal(size=N))
    C = _run(d, wp, sp, afmt, p, M, bias)
    assert np.array_equal(C, np.broadcast_to(bias, (M, N)))


def test_grouped_with_no_rows_is_a_no_op():
    Q = qw()
    E, N, K = 4, 64, 256
    p = synth.w4a16_problem(1, N, K, bits=4, E=E, cfg_id=1350)
    d, wp, sp = repack(Q.QW_W_INT4_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
    off = torch.zeros((E + 1,), dtype=torch.int32, device="cuda")
    C = torch.full((1, N), -1, dtype=torch.int16, device="cuda")
    A = torch.zeros((1, K), dtype=torch.int16, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, Q.QW_A_BF16, A, None, off, 0, None, C, None, 0, err)
    assert Q.qw_read_error(err) == 0
    assert np.all(u16_view(C) == 0xFFFF)
