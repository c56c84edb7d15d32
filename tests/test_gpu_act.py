"""Activation-side MoE steps on the GPU against the float64 oracle (oracle/act.py):
MXFP8 quantizer bit for bit, SiLU*mul within one BF16 ulp, the top-k combine within the
GEMM tolerance; plus BF16 activations -> MXFP8 -> W4A8 GEMM end to end."""
import numpy as np
import pytest
import torch

import synth
from oracle import act as OA
from oracle import formats as OF
from oracle import moe as OM
from oracle import qgemm as OQ
from qwtest import dev, host, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def _activations(rows, K, seed):
    """BF16 activations with varied per-row magnitudes, an all-zero group, BF16
    subnormals, values that saturate and exact E4M3 ties."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (rows, K)) * np.exp2(rng.integers(-40, 40, (rows, 1)))
    x[0, :32] = 0.0
    if rows > 1:
        x[1, :32] = np.exp2(-130.0) * rng.integers(-3, 4, 32)          # subnormals
    if rows > 2:
        x[2, :8] = [256.0, 264.0, 272.0, 304.0, 480.0, -460.0, -2.0 ** -140, 1.0]  # ties, sat
    return synth.to_bf16_bits(x)


def _quantize(bits):
    Q = qw()
    rows, K = bits.shape
    A = dev(bits.view(np.int16))
    q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qw_quantize_mxfp8(A, rows, K, q, sf, err)
    assert Q.qw_read_error(err) == 0
    return host(q), host(sf)


@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (37, 640), (64, 4096), (5, 7168)])
def test_quantize_mxfp8_bit_exact(rows, K):
    bits = _activations(max(rows, 3), K, seed=rows * 7 + K)[:rows]
    q, sf = _quantize(bits)
    rq, rsf = OA.quantize_mxfp8(bits)
    assert np.array_equal(sf, rsf)
    assert np.array_equal(q, rq)


def test_quantize_mxfp8_full_size_moe_activations():
    """T=4096 tokens x hidden 7168 (the E=256 MoE workload's activations), every element."""
    bits = _activations(4096, 7168, seed=99)
    q, sf = _quantize(bits)
    rq, rsf = OA.quantize_mxfp8(bits)
    assert np.array_equal(sf, rsf) and np.array_equal(q, rq)


def test_quantize_mxfp8_flags_non_finite():
    Q = qw()
    bits = _activations(4, 64, seed=3)
    bits[2, 40] = 0x7F80  # +inf
    A = dev(bits.view(np.int16))
    q = torch.empty((4, 64), dtype=torch.uint8, device="cuda")
    sf = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qw_quantize_mxfp8(A, 4, 64, q, sf, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


def test_bf16_activations_through_mxfp8_into_w4a8():
    """BF16 activations -> qw_quantize_mxfp8 -> W4A8 GEMM, against the oracle's own
    quantizer and GEMM on the same BF16 input."""
    Q = qw()
    M, N, K = 200, 384, 512
    rng = np.random.default_rng(21)
    x = synth.to_bf16_bits(rng.normal(0, 1, (M, K)))
    p = synth.w4a8_problem(M, N, K, cfg_id=55)
    d, wp, sp = repack(Q.QW_W_MXFP4_G32, 1, N, K, p["w_canon"], p["s_canon"])
    A = dev(x.view(np.int16))
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sf = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qw_quantize_mxfp8(A, M, K, q, sf, err)
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    Q.qgemm_dense(d, wp, sp, Q.QW_A_MXFP8_G32, q, sf, None, C, M, None, 0, err)
    assert Q.qw_read_error(err) == 0
    rq, rsf = OA.quantize_mxfp8(x)
    R, S = OQ.gemm_w4a8(rq, rsf, OF.unpack_e2m1_bytes(p["w_canon"][0], K), p["s_canon"][0])
    ok, ratio, frob = OQ.check_bf16_result(u16_view(C), R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("rows,I", [(1, 8), (7, 640), (300, 640), (64, 2048)])
def test_silu_mul_within_one_bf16_ulp(rows, I):
    Q = qw()
    rng = np.random.default_rng(rows + I)
    gu = synth.to_bf16_bits(rng.normal(0, 3, (rows, 2 * I)))
    Y = torch.empty((rows, I), dtype=torch.int16, device="cuda")
    Q.qw_silu_mul(dev(gu.view(np.int16)), rows, I, Y)
    got = u16_view(Y)
    ref = OA.silu_mul(gu)
    g, r = OF.decode_bf16(got), OF.decode_bf16(ref)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
    assert np.all(np.abs(g - r) <= ulp), np.max(np.abs(g - r) / ulp)
    assert np.mean(got == ref) > 0.99  # FP32 evaluation differs only at rounding boundaries


@pytest.mark.parametrize("T,E,k,N", [(1, 8, 2, 8), (37, 16, 4, 640), (512, 128, 8, 4096)])
def test_moe_combine(T, E, k, N):
    Q = qw()
    rng = np.random.default_rng(T + E)
    logits = synth.router_logits(T, E, cfg_id=T)
    lg = dev(logits)
    P = T * k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    spt = torch.empty((P,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, k)
    rws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_route(lg, T, E, k, ids, spt, off, rws, n)
    Y = synth.to_bf16_bits(rng.normal(0, 1, (P, N)))
    out = torch.empty((T, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_moe_combine_workspace_size(T, k)
    ws = torch.empty(wsn, dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_combine(dev(Y.view(np.int16)), spt, ids, lg, T, E, k, N, out, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    _, R, S = OA.combine(Y, host(spt), host(ids), logits)
    ok, ratio, frob = OQ.check_bf16_result(u16_view(out), R, S)
    assert ok, (ratio, frob)


def test_moe_combine_flags_bad_pairs():
    Q = qw()
    T, E, k, N = 4, 8, 2, 16
    spt = dev(np.array([0, 1, 2, 3, 4, 5, 6, 99], dtype=np.int32))  # 99 is out of range
    ids = dev(np.zeros((T, k), dtype=np.int32))
    lg = dev(np.zeros((T, E), dtype=np.float32))
    Y = torch.zeros((T * k, N), dtype=torch.int16, device="cuda")
    out = torch.empty((T, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_moe_combine_workspace_size(T, k)
    ws = torch.zeros(wsn, dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_combine(Y, spt, ids, lg, T, E, k, N, out, ws, wsn, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_INVALID_ARG
