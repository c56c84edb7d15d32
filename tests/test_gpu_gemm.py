"""Dense GEMM parity on the GPU against the float64 oracle.

Tolerance (the spec acceptance rule): per element |C - R| <= 2^-7 sum_k |a_k w_k| + 1e-6
and ||C - R||_F <= 2e-3 ||R||_F.
"""
import numpy as np
import pytest

import synth
from oracle import qgemm as OQ
from qwtest import dense_w4a16, dense_w4a8

pytestmark = pytest.mark.gpu


def assert_parity(C, R, absum, what=""):
    ok, ratio, frob = OQ.check_bf16_result(C, R, absum)
    assert ok, f"{what}: worst |err|/bound = {ratio:.3g}, rel frob = {frob:.3g}"


# ----------------------------------------------------------------------------- W4A16 small M
@pytest.mark.parametrize("bits", [4, 3, 2])
@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (3, 40, 384), (8, 2048, 2048), (13, 96, 256),
                                   (16, 200, 640), (16, 128, 1024)])
def test_w4a16_small_shapes(bits, M, N, K):
    """M <= 16 runs the split-K tensor-core GEMV (one or two 8-row token slices)."""
    p = synth.w4a16_problem(M, N, K, bits=bits, cfg_id=100 + M)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    assert_parity(C, R, S, f"W{bits}A16 {M}x{N}x{K}")


@pytest.mark.parametrize("bits", [4, 3])
def test_w4a16_bias(bits):
    p = synth.w4a16_problem(5, 72, 256, bits=bits, cfg_id=120, bias=True)
    C = dense_w4a16(p, bias=p["bias"][0])
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 256, bits,
                                   bias_bits=p["bias"][0])
    assert_parity(C, R, S, "bias")


def test_config1_dense_w4a16_m8():
    """M=8, N=K=2048 INT4 group-128 (the small oracle-checkable workload), every output."""
    p = synth.w4a16_problem(8, 2048, 2048, bits=4, cfg_id=0)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 2048, 4)
    assert_parity(C, R, S, "config 1")


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336), (4096, 4096)])
def test_config3_m1_decode_full(bits, N, K):
    """M=1 decode GEMV sweep at full size, every output element."""
    p = synth.w4a16_problem(1, N, K, bits=bits, cfg_id=2)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    assert_parity(C, R, S, f"config 3 W{bits} {N}x{K}")


@pytest.mark.parametrize("bits", [4, 3, 2])
def test_m1_staged_kernel_ragged_n_odd_groups_bias(bits):
    """Single-token decode over a matrix large enough for the staged-activation kernel, with
    N not a multiple of 16, an odd group count (33: the last warp of a CTA gets no group) and
    a bias."""
    N, K = 8200, 4224
    p = synth.w4a16_problem(1, N, K, bits=bits, cfg_id=121, bias=True)
    C = dense_w4a16(p, bias=p["bias"][0])
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits,
                                   bias_bits=p["bias"][0])
    assert_parity(C, R, S, f"M=1 W{bits} {N}x{K} bias")


# ----------------------------------------------------------------------------- W4A8
def test_w4a8_single_tile_integer_exact():
    """All scales 2^0 and small integer codes: one 128 x 256 x 128 tile must be exact."""
    rng = np.random.default_rng(7)
    M, N, K = 128, 256, 128
    int_e4m3 = [0x00, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0xC4]  # 0, 1, 2, 3, -1, -2, -3
    int_e2m1 = [0, 2, 4, 5, 10, 12, 13]                   # 0, 1, 2, 3, -1, -2, -3
    A = rng.choice(int_e4m3, (M, K)).astype(np.uint8)
    W = rng.choice(int_e2m1, (N, K)).astype(np.uint8)
    p = dict(A=A, A_sf=np.full((M, K // 32), 127, np.uint8), w_canon=synth.pack_nibbles(W)[None],
             s_canon=np.full((1, N, K // 32), 127, np.uint8), N=N, K=K)
    C = dense_w4a8(p)
    R, S = OQ.gemm_w4a8(A, p["A_sf"], W, p["s_canon"][0])
    Cv = synth.to_bf16_bits(R)
    assert np.array_equal(C, Cv), f"{np.sum(C != Cv)} of {C.size} differ"


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 256, 512), (256, 512, 256),
                                   (1, 256, 128), (200, 300, 256), (129, 640, 4096),
                                   (384, 3072, 1024)])
def test_w4a8_shapes(M, N, K):
    p = synth.w4a8_problem(M, N, K, cfg_id=200 + M)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    assert_parity(C, R, S, f"W4A8 {M}x{N}x{K}")


def test_w4a8_k_not_multiple_of_128_and_bias():
    p = synth.w4a8_problem(70, 264, 96, cfg_id=230, bias=True)
    C = dense_w4a8(p, bias=p["bias"][0])
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 96,
                                  bias_bits=p["bias"][0])
    assert_parity(C, R, S, "W4A8 K=96 + bias")


# ----------------------------------------------------------------------------- W4A8 small M
@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_w4a8_gemv_integer_exact(M):
    """M <= 8 runs the streaming W4A8 GEMV; with unit scales and small integer codes every
    group sum is an exact integer, so the output equals the oracle's BF16 rounding."""
    rng = np.random.default_rng(70 + M)
    N, K = 272, 384
    int_e4m3 = [0x00, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0xC4]  # 0, 1, 2, 3, -1, -2, -3
    int_e2m1 = [0, 2, 4, 5, 10, 12, 13]                   # 0, 1, 2, 3, -1, -2, -3
    A = rng.choice(int_e4m3, (M, K)).astype(np.uint8)
    W = rng.choice(int_e2m1, (N, K)).astype(np.uint8)
    p = dict(A=A, A_sf=np.full((M, K // 32), 127, np.uint8), w_canon=synth.pack_nibbles(W)[None],
             s_canon=np.full((1, N, K // 32), 127, np.uint8), N=N, K=K)
    C = dense_w4a8(p)
    R, S = OQ.gemm_w4a8(A, p["A_sf"], W, p["s_canon"][0])
    assert np.array_equal(C, synth.to_bf16_bits(R))


@pytest.mark.parametrize("M,N,K", [(1, 144, 32), (3, 264, 96), (8, 1000, 640), (2, 130, 4096),
                                   (7, 4096, 1024)])
def test_w4a8_gemv_shapes(M, N, K):
    """Ragged N (padded to 128 rows), K not a multiple of 128 and group counts that leave
    some warps of a CTA without work.  (With only a few dozen outputs the Frobenius bound
    can fail for the correctly rounded BF16 result itself - e.g. 16 outputs of K = 32 -
    so the smallest case keeps 144.)"""
    p = synth.w4a8_problem(M, N, K, cfg_id=240 + M)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    assert_parity(C, R, S, f"W4A8 GEMV {M}x{N}x{K}")


def test_w4a8_gemv_largest_staging():
    """M = 8 at the largest K whose staged activations the GEMV takes (176 groups: 95.7 KB of
    FP16 fragments and scales, one CTA per SM beside its rings): seven warps stream 24
    groups each, the last 8."""
    p = synth.w4a8_problem(8, 272, 5632, cfg_id=255)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 5632)
    assert_parity(C, R, S, "W4A8 GEMV M=8 K=5632")


def test_w4a8_gemv_bias_and_wide_scales():
    """Bias, and E8M0 scales over a wide range (2^-47 .. 2^43) on both sides, so group
    products span ~2^-94 .. 2^86 (inside BF16's range)."""
    p = synth.w4a8_problem(4, 520, 512, cfg_id=250, bias=True, sf_lo=80, sf_hi=170)
    C = dense_w4a8(p, bias=p["bias"][0])
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 512,
                                  bias_bits=p["bias"][0])
    assert_parity(C, R, S, "W4A8 GEMV bias, wide scales")


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_w4a8_gemv_m1_decode_full(N, K):
    """Single-token W4A8 decode at full size, every output element."""
    p = synth.w4a8_problem(1, N, K, cfg_id=260)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    assert_parity(C, R, S, f"W4A8 M=1 {N}x{K}")


def test_w4a8_last_wave_shape_bias_ragged_and_repeatable():
    """A dense W4A8 call whose 10 x 16 tiles leave a last wave of 8 tiles for 152 SMs, with
    bias and ragged N, K = 8192: every element against the oracle, with and without the
    workspace the call asks for, and twice: the results are the same bits every time."""
    p = synth.w4a8_problem(1280, 4000, 8192, cfg_id=270, bias=True)
    C1 = dense_w4a8(p, bias=p["bias"][0])
    C2 = dense_w4a8(p, bias=p["bias"][0])
    C0 = dense_w4a8(p, bias=p["bias"][0], workspace=False)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 8192,
                                  bias_bits=p["bias"][0])
    assert_parity(C1, R, S, "W4A8 1280 x 4000 x 8192")
    assert np.array_equal(C1, C2) and np.array_equal(C1, C0)


def test_config2a_w4a8_full():
    """(M,N,K) = (4096, 3072, 4096) MXFP4 x MXFP8 group-32, every output element."""
    p = synth.w4a8_problem(4096, 3072, 4096, cfg_id=1)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 4096)
    assert_parity(C, R, S, "config 2a")


def test_config2b_w4a8_full_size_sampled_rows():
    """(4096, 14336, 4096): the kernel runs the full problem; the oracle checks 384 sampled
    rows (three from every 128-row tile) against all 14336 columns."""
    p = synth.w4a8_problem(4096, 14336, 4096, cfg_id=1)
    C = dense_w4a8(p)
    rows = np.concatenate([np.array([0, 61, 127]) + 128 * i for i in range(32)])
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], 4096,
                                  rows=rows)
    assert_parity(C[rows], R, S, "config 2b")


# ----------------------------------------------------------------------------- W4A16 large M
@pytest.mark.parametrize("bits", [4, 3, 2])
@pytest.mark.parametrize("M,N,K", [(17, 96, 256), (33, 200, 640), (64, 128, 1024),
                                   (65, 40, 128), (128, 128, 256), (130, 48, 256),
                                   (257, 200, 640), (300, 1280, 4096), (129, 4096, 640)])
def test_w4a16_tensor_core_shapes(bits, M, N, K):
    """M > 16 runs the tcgen05 path: dequantized BF16 weights written into tensor memory."""
    p = synth.w4a16_problem(M, N, K, bits=bits, cfg_id=400 + M)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    assert_parity(C, R, S, f"W{bits}A16 TC {M}x{N}x{K}")


def test_w4a16_tensor_core_bias():
    p = synth.w4a16_problem(150, 96, 384, bits=4, cfg_id=430, bias=True)
    C = dense_w4a16(p, bias=p["bias"][0])
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 384, 4,
                                   bias_bits=p["bias"][0])
    assert_parity(C, R, S, "W4A16 TC bias")


def test_w4a16_tensor_core_large_sampled_rows():
    """(4096, 4096, 4096) INT4 on the tensor-core path; 256 sampled rows checked in full."""
    p = synth.w4a16_problem(4096, 4096, 4096, bits=4, cfg_id=431)
    C = dense_w4a16(p)
    rows = np.concatenate([np.array([0, 77, 127]) + 128 * i for i in range(32)])
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 4096, 4, rows=rows)
    assert_parity(C[rows], R, S, "W4A16 TC 4096^3")
