"""Pins for the oracle GEMMs (CPU only): exact integer dot products, exact rational
brute force on tiny shapes, and planted mistakes that the pins must catch."""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import qgemm as Q
import synth


def bf16_bits_of(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float64))


# ----------------------------------------------------------------------------- W4A16
def test_w4a16_exact_integer_dot():
    """All scales 1.0 and integer activations (|a| <= 256 is exact in BF16): the float64
    result must equal the int64 dot product exactly.  Shapes are non-square."""
    rng = np.random.default_rng(10)
    M, N, K = 5, 7, 384
    a = rng.integers(-256, 257, (M, K))
    q = rng.integers(-7, 8, (N, K))
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)  # BF16 1.0
    R, absum = Q.gemm_w4a16(bf16_bits_of(a), q, s)
    assert np.array_equal(R, (a @ q.T).astype(np.float64))
    assert np.array_equal(absum, (np.abs(a) @ np.abs(q).T).astype(np.float64))


def test_w4a16_exact_from_canonical_int3_and_int4():
    rng = np.random.default_rng(11)
    M, N, K = 3, 6, 256
    a = rng.integers(-100, 101, (M, K))
    for bits, qmax, pack in ((4, 7, synth.pack_int4), (3, 3, synth.pack_int3)):
        q = rng.integers(-qmax, qmax + 1, (N, K))
        s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
        R, _ = Q.w4a16_from_canonical(bf16_bits_of(a), pack(q), s, K, bits)
        assert np.array_equal(R, (a @ q.T).astype(np.float64))


def _exact_w4a16(a_bits, q, s_bits, group=128):
    """Exact rational evaluation; BF16 widened through torch (a library routine)."""
    a = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    s = torch.from_numpy(s_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    M, K = a.shape
    N = q.shape[0]
    R = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(a[m, k]) * int(q[n, k]) * Fraction(s[n, k // group])
            R[m][n] = acc
    return R


def test_w4a16_fraction_brute_force_groups():
    rng = np.random.default_rng(12)
    M, N, K = 2, 3, 256  # two groups of 128
    a_bits = bf16_bits_of(rng.standard_normal((M, K)))
    q = rng.integers(-7, 8, (N, K))
    s_bits = bf16_bits_of(rng.uniform(0.005, 0.02, (N, K // 128)))
    R, absum = Q.gemm_w4a16(a_bits, q, s_bits)
    ex = _exact_w4a16(a_bits, q, s_bits)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(R[m, n]) - ex[m][n]) <= Fraction(2.0 ** -50) * Fraction(absum[m, n])


def test_w4a16_bias_added():
    rng = np.random.default_rng(13)
    a = rng.integers(-8, 9, (2, 128))
    q = rng.integers(-7, 8, (3, 128))
    s = np.full((3, 1), 0x3F80, dtype=np.uint16)
    b = bf16_bits_of([0.5, -2.0, 3.25])
    R, _ = Q.gemm_w4a16(bf16_bits_of(a), q, s, b)
    assert np.array_equal(R, a @ q.T + np.array([0.5, -2.0, 3.25])[None, :])


# ----------------------------------------------------------------------------- W4A8
E4M3_INT = {}  # integer value -> E4M3 code, built from torch's decoder (a library routine)
for _c in range(256):
    if (_c & 0x7F) == 0x7F:
        continue
    _v = float(torch.tensor([_c], dtype=torch.uint8).view(torch.float8_e4m3fn).double())
    if _v == int(_v) and abs(_v) <= 16 and not (_v == 0 and _c != 0):
        E4M3_INT[int(_v)] = _c
E2M1_INT = {0: 0, 1: 2, 2: 4, 3: 5, 4: 6, 6: 7, -1: 10, -2: 12, -3: 13, -4: 14, -6: 15}


def test_w4a8_exact_integer_dot():
    """Scale bytes 127 (2^0) and integer-valued E4M3 / E2M1 codes: exact int64 match."""
    rng = np.random.default_rng(20)
    M, N, K = 4, 6, 96
    av = rng.integers(-16, 17, (M, K))
    wv = rng.choice(list(E2M1_INT), (N, K))
    a_codes = np.vectorize(E4M3_INT.get)(av).astype(np.uint8)
    w_codes = np.vectorize(E2M1_INT.get)(wv).astype(np.uint8)
    R, absum = Q.gemm_w4a8(a_codes, np.full((M, K // 32), 127, np.uint8),
                           w_codes, np.full((N, K // 32), 127, np.uint8))
    assert np.array_equal(R, (av @ wv.T).astype(np.float64))
    assert np.array_equal(absum, (np.abs(av) @ np.abs(wv).T).astype(np.float64))


def test_w4a8_power_of_two_scales_exact():
    """Per-group scale exponents: R = sum_g 2^(ea_g + ew_g - 254) * (int dot of group g)."""
    rng = np.random.default_rng(21)
    M, N, K = 3, 5, 128
    av = rng.integers(-16, 17, (M, K))
    wv = rng.choice(list(E2M1_INT), (N, K))
    ea = rng.integers(118, 127, (M, K // 32))
    ew = rng.integers(118, 127, (N, K // 32))
    R, _ = Q.gemm_w4a8(np.vectorize(E4M3_INT.get)(av).astype(np.uint8), ea.astype(np.uint8),
                       np.vectorize(E2M1_INT.get)(wv).astype(np.uint8), ew.astype(np.uint8))
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for g in range(K // 32):
                d = int(av[m, 32 * g:32 * g + 32] @ wv[n, 32 * g:32 * g + 32])
                exact += Fraction(d) * Fraction(2) ** (int(ea[m, g]) + int(ew[n, g]) - 254)
            assert Fraction(R[m, n]) == exact


def test_w4a8_fraction_brute_force_random_codes():
    """Random codes over the whole E4M3 / E2M1 ranges, exact rationals via torch decoding."""
    rng = np.random.default_rng(22)
    M, N, K = 2, 3, 64
    a_codes = synth.to_e4m3_codes(rng.standard_normal((M, K)) * 30)
    w_codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    a_sf = rng.integers(118, 127, (M, K // 32)).astype(np.uint8)
    w_sf = rng.integers(118, 127, (N, K // 32)).astype(np.uint8)
    R, absum = Q.gemm_w4a8(a_codes, a_sf, w_codes, w_sf)
    a = torch.from_numpy(a_codes).view(torch.float8_e4m3fn).double().numpy()
    from test_oracle_formats import e2m1_closed_form
    for m in range(M):
        for n in range(N):
            ex = sum(Fraction(a[m, k]) * Fraction(math.ldexp(1, int(a_sf[m, k // 32]) - 127))
                     * Fraction(e2m1_closed_form(int(w_codes[n, k])))
                     * Fraction(math.ldexp(1, int(w_sf[n, k // 32]) - 127)) for k in range(K))
            assert abs(Fraction(R[m, n]) - ex) <= Fraction(2.0 ** -50) * Fraction(absum[m, n])


def test_w4a8_from_canonical_nibble_order():
    """k even in the low nibble: a weight row [1, 6, 0, ...] packs as byte 0x72."""
    K = 32
    w = np.zeros((1, K // 2), np.uint8)
    w[0, 0] = 0x72  # k0 = code 2 (1.0), k1 = code 7 (6.0)
    a = np.zeros((1, K), np.uint8)
    a[0, 0] = E4M3_INT[3]
    a[0, 1] = E4M3_INT[5]
    sf = np.full((1, 1), 127, np.uint8)
    R, _ = Q.w4a8_from_canonical(a, sf, w, sf, K)
    assert R[0, 0] == 3 * 1 + 5 * 6


# ----------------------------------------------------------------------------- acceptance checker
def test_check_bf16_result_accepts_rounded_and_rejects_wrong():
    rng = np.random.default_rng(30)
    R = rng.standard_normal((16, 16)) * 10
    absum = np.abs(R) * 4 + 1
    ok, ratio, frob = Q.check_bf16_result(bf16_bits_of(R), R, absum)
    assert ok and ratio < 0.5
    bad = R.copy()
    bad[3, 4] += 0.2 * absum[3, 4]
    ok, _, _ = Q.check_bf16_result(bf16_bits_of(bad), R, absum)
    assert not ok


# ----------------------------------------------------------------------------- planted mistakes
def test_planted_wrong_e2m1_entry_is_caught(monkeypatch):
    from test_oracle_formats import e2m1_closed_form
    bad = F._E2M1_MAG.copy()
    bad[5] = 2.5  # should be 3.0
    monkeypatch.setattr(F, "_E2M1_MAG", bad)
    got = F.decode_e2m1(np.arange(16))
    assert not np.array_equal(got, [e2m1_closed_form(c) for c in range(16)])


def test_planted_wrong_group_size_is_caught(monkeypatch):
    orig = Q.dequant_mx

    def wrong_group(codes, sf, decode):  # scale group 64 instead of 32
        v = decode(codes)
        return v * np.repeat(F.decode_e8m0(sf), 64, axis=-1)[..., :v.shape[-1]]

    monkeypatch.setattr(Q, "dequant_mx", wrong_group)
    with pytest.raises(AssertionError):
        test_w4a8_power_of_two_scales_exact()
    monkeypatch.setattr(Q, "dequant_mx", orig)


def test_planted_transposed_operand_is_caught(monkeypatch):
    def transposed(A_bits, q, s_bits, bias_bits=None, group=128):
        a = F.decode_bf16(A_bits)
        w = Q.dequant_int_weights(q, s_bits, group)
        return (a @ w.T)[:, ::-1], np.abs(a) @ np.abs(w).T  # columns in the wrong order

    monkeypatch.setattr(Q, "gemm_w4a16", transposed)
    with pytest.raises(AssertionError):
        test_w4a16_exact_integer_dot()


def test_w8a8_exact_integer_dot():
    """Integer-valued E4M3 codes with unit scales: an exact integer dot product."""
    rng = np.random.default_rng(31)
    M, N, K = 3, 4, 64
    ints = rng.integers(-16, 17, (M, K))
    wint = rng.integers(-16, 17, (N, K))
    enc = {v: c for c, v in enumerate(F.decode_e4m3(np.arange(127))) if float(v).is_integer()}
    code = lambda v: (enc[abs(int(v))] | (0x80 if v < 0 else 0))  # noqa: E731
    A = np.vectorize(code)(ints).astype(np.uint8)
    W = np.vectorize(code)(wint).astype(np.uint8)
    ones_a = np.full((M, K // 32), 127, np.uint8)
    ones_w = np.full((N, K // 32), 127, np.uint8)
    R, S = Q.gemm_w8a8(A, ones_a, W, ones_w)
    assert np.array_equal(R, (ints @ wint.T).astype(np.float64))


def test_w8a8_equals_w4a8_on_e2m1_values():
    """E2M1 values are E4M3 values: re-encoding the E2M1 weights as E4M3 codes (with the
    E4M3 encoder of oracle/act) must give the W4A8 result exactly."""
    from oracle import act as OA
    rng = np.random.default_rng(32)
    M, N, K = 5, 7, 96
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0
    Asf = rng.integers(118, 127, (M, K // 32)).astype(np.uint8)
    w4 = rng.integers(0, 16, (N, K))
    wsf = rng.integers(118, 127, (N, K // 32)).astype(np.uint8)
    w8 = OA.encode_e4m3(F.decode_e2m1(w4))
    R4, S4 = Q.gemm_w4a8(A, Asf, w4, wsf)
    R8, S8 = Q.gemm_w8a8(A, Asf, w8, wsf)
    assert np.array_equal(R4, R8) and np.array_equal(S4, S8)


# ----------------------------------------------------------------------------- W4A4 (NVFP4)
E4M3_ONE = 0x38  # 1.0
E2M1_INT = {0: 0, 1: 2, 2: 4, 3: 5, 4: 6, 6: 7}  # integer magnitude -> E2M1 code


def _e2m1_int_codes(rng, shape):
    mags = rng.choice([0, 1, 2, 3, 4, 6], shape)
    neg = rng.integers(0, 2, shape).astype(bool)
    codes = np.vectorize(lambda v: E2M1_INT[int(v)])(mags).astype(np.uint8)
    return np.where(neg, codes | 8, codes).astype(np.uint8), np.where(neg, -mags, mags)


def test_w4a4_exact_integer_dot():
    """Unit scales and integer-valued E2M1 codes: an exact integer dot product."""
    rng = np.random.default_rng(41)
    M, N, K = 3, 5, 64
    A, ai = _e2m1_int_codes(rng, (M, K))
    W, wi = _e2m1_int_codes(rng, (N, K))
    R, S = Q.gemm_w4a4(A, np.full((M, K // 16), E4M3_ONE, np.uint8), W,
                       np.full((N, K // 16), E4M3_ONE, np.uint8))
    assert np.array_equal(R, (ai @ wi.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(ai) @ np.abs(wi).T).astype(np.float64))


def test_w4a4_equals_w4a8_with_power_of_two_scales():
    """E2M1 values are E4M3 values and a power-of-two E4M3 scale is an E8M0 scale: with
    both 16-groups of every 32-group sharing one such scale, W4A4 must equal W4A8 on the
    same values exactly."""
    from oracle import act as OA
    rng = np.random.default_rng(42)
    M, N, K = 4, 6, 128
    A4 = rng.integers(0, 16, (M, K)).astype(np.uint8)
    W4 = rng.integers(0, 16, (N, K)).astype(np.uint8)
    ea = rng.integers(-6, 8, (M, K // 32))          # exponents representable as E4M3 normals
    ew = rng.integers(-6, 8, (N, K // 32))
    e4m3_pow2 = lambda e: ((e + 7) << 3).astype(np.uint8)  # noqa: E731  (sign 0, mantissa 0)
    Asf16 = np.repeat(e4m3_pow2(ea), 2, axis=1)
    Wsf16 = np.repeat(e4m3_pow2(ew), 2, axis=1)
    assert np.array_equal(F.decode_e4m3(Asf16), np.repeat(np.exp2(ea), 2, axis=1))
    R4, S4 = Q.gemm_w4a4(A4, Asf16, W4, Wsf16)
    A8 = OA.encode_e4m3(F.decode_e2m1(A4))
    R8, S8 = Q.gemm_w4a8(A8, (ea + 127).astype(np.uint8), W4, (ew + 127).astype(np.uint8))
    assert np.array_equal(R4, R8) and np.array_equal(S4, S8)


def test_w4a4_fraction_brute_force_groups():
    """Random codes and random finite E4M3 scales, exact rationals, three 16-groups."""
    rng = np.random.default_rng(43)
    M, N, K = 2, 3, 48
    A = rng.integers(0, 16, (M, K)).astype(np.uint8)
    W = rng.integers(0, 16, (N, K)).astype(np.uint8)
    Asf = rng.integers(0, 0x7F, (M, K // 16)).astype(np.uint8)
    Wsf = rng.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)
    R, absum = Q.gemm_w4a4(A, Asf, W, Wsf)
    from test_oracle_formats import e2m1_closed_form
    a_s = torch.from_numpy(Asf).view(torch.float8_e4m3fn).double().numpy()
    w_s = torch.from_numpy(Wsf).view(torch.float8_e4m3fn).double().numpy()
    for m in range(M):
        for n in range(N):
            ex = sum(Fraction(e2m1_closed_form(int(A[m, k]))) * Fraction(a_s[m, k // 16])
                     * Fraction(e2m1_closed_form(int(W[n, k]))) * Fraction(w_s[n, k // 16])
                     for k in range(K))
            assert abs(Fraction(R[m, n]) - ex) <= Fraction(2.0 ** -50) * Fraction(absum[m, n])


def test_w4a4_from_canonical_nibble_order():
    """Even k in the low nibble on both operands: A row bytes [0x52] (k0 = 1.0, k1 = 3.0)
    times W row bytes [0x74] (k0 = 2.0, k1 = 6.0) = 1*2 + 3*6."""
    K = 16
    A = np.zeros((1, K // 2), np.uint8)
    A[0, 0] = 0x52
    W = np.zeros((1, K // 2), np.uint8)
    W[0, 0] = 0x74
    one = np.full((1, 1), E4M3_ONE, np.uint8)
    R, _ = Q.w4a4_from_canonical(A, one, W, one, K)
    assert R[0, 0] == 1 * 2 + 3 * 6


def test_w4a4_rejects_negative_and_nan_scales():
    A = np.zeros((1, 16), np.uint8)
    for bad in (0x80 | E4M3_ONE, 0x7F):
        with pytest.raises(F.FormatError):
            Q.gemm_w4a4(A, np.full((1, 1), bad, np.uint8), A, np.full((1, 1), E4M3_ONE, np.uint8))


def test_planted_wrong_nvfp4_group_is_caught(monkeypatch):
    orig = Q.dequant_nv

    def wrong_group(codes, sf, group=16):  # each 16-group takes its neighbour's scale
        return orig(codes, np.roll(np.asarray(sf), 1, axis=-1), group=group)

    monkeypatch.setattr(Q, "dequant_nv", wrong_group)
    with pytest.raises(AssertionError):
        test_w4a4_fraction_brute_force_groups()


# ----------------------------------------------------------------------------- W4A16 zero points
def test_w4a16_zp_exact_integer_dot():
    """Unit scales: sum_k a (q - z) with integer activations is an exact integer."""
    rng = np.random.default_rng(51)
    M, N, K = 3, 4, 256
    a = rng.integers(-20, 21, (M, K))
    q = rng.integers(0, 16, (N, K))
    z = rng.integers(0, 16, (N, K // 128))
    A = synth.to_bf16_bits(a.astype(np.float64))
    one = synth.to_bf16_bits(np.ones((N, K // 128)))
    R, S = Q.gemm_w4a16_zp(A, q, one, z)
    want = a @ (q - np.repeat(z, 128, axis=1)).T
    assert np.array_equal(R, want.astype(np.float64))


def test_w4a16_zp_with_zero_point_8_is_the_symmetric_code():
    """q - 8 is the two's-complement INT4 value of the excess code: with z = 8 everywhere
    the asymmetric GEMM must equal the symmetric one on q - 8 exactly."""
    p = synth.w4a16_problem(5, 40, 384, bits=4, cfg_id=52)
    q_signed = F.unpack_int4(p["w_canon"][0], 384).astype(np.int64)
    R1, S1 = Q.gemm_w4a16(p["A"], q_signed, p["s_canon"][0])
    R2, S2 = Q.gemm_w4a16_zp(p["A"], q_signed + 8, p["s_canon"][0],
                             np.full((40, 3), 8, np.int64))
    assert np.array_equal(R1, R2) and np.array_equal(S1, S2)


def test_w4a16_zp_fraction_brute_force_and_canonical_words():
    """Packed words (unsigned nibbles, scale + zero-point group words) decoded by the
    canonical driver against exact rationals on a tiny shape with two groups."""
    p = synth.w4a16_zp_problem(2, 3, 256, cfg_id=53)
    R, absum = Q.w4a16_zp_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], 256)
    a = F.decode_bf16(p["A"])
    words = p["w_canon"][0]
    sz = p["s_canon"][0].astype(np.int64)
    for m in range(2):
        for n in range(3):
            ex = Fraction(0)
            for k in range(256):
                q = (int(words[n, k // 8]) >> (4 * (k % 8))) & 0xF
                g = k // 128
                s = Fraction(float(F.decode_bf16(np.uint16(sz[n, g] & 0xFFFF))))
                z = (int(sz[n, g]) >> 16) & 0xFF
                ex += Fraction(float(a[m, k])) * (q - z) * s
            assert abs(Fraction(R[m, n]) - ex) <= Fraction(2.0 ** -50) * Fraction(absum[m, n])


def test_split_zp_scales_rejects_bad_words():
    with pytest.raises(F.FormatError):
        F.split_zp_scales(np.array([0x3F80 | (16 << 16)], np.uint32))
    with pytest.raises(F.FormatError):
        F.split_zp_scales(np.array([0x3F80 | (1 << 24)], np.uint32))
    s, z = F.split_zp_scales(np.array([0x3F80 | (15 << 16)], np.uint32))
    assert s[0] == 0x3F80 and z[0] == 15


def test_w4a16_int2_from_canonical_exact():
    """INT2 words through the canonical driver: unit scales and integer activations give the
    exact integer product of the codes decoded bit by bit here."""
    rng = np.random.default_rng(54)
    M, N, K = 3, 5, 256
    q = rng.integers(-1, 2, (N, K))
    a = rng.integers(-9, 10, (M, K))
    words = np.zeros((N, K // 16), np.uint32)
    for n in range(N):
        for k in range(K):
            words[n, k // 16] |= np.uint32((int(q[n, k]) & 3) << (2 * (k % 16)))
    one = synth.to_bf16_bits(np.ones((N, K // 128)))
    R, _ = Q.w4a16_from_canonical(synth.to_bf16_bits(a.astype(np.float64)), words, one, K, 2)
    assert np.array_equal(R, (a @ q.T).astype(np.float64))


# ----------------------------------------------------------------------------- FP8 weights
def _e4m3_codes_torch(x):
    """E4M3 codes by PyTorch's float8_e4m3fn cast (independent of the oracle's decoder)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _e4m3_values_torch(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_fp8w_equals_w4a16_on_integer_codes():
    """E4M3 codes of the integers -7..7 are exact: the FP8-weight GEMM must equal the W4A16
    GEMM on those integers bit for bit, with the same BF16 group scales and bias."""
    p = synth.w4a16_problem(4, 24, 384, bits=4, cfg_id=60, bias=True)
    q = F.unpack_int4(p["w_canon"][0], 384).astype(np.int64)
    codes = _e4m3_codes_torch(q)
    R1, S1 = Q.gemm_w4a16(p["A"], q, p["s_canon"][0], p["bias"][0])
    R2, S2 = Q.gemm_w8a16_fp8(p["A"], codes, p["s_canon"][0], p["bias"][0])
    assert np.array_equal(R1, R2) and np.array_equal(S1, S2)


def test_fp8w_fraction_brute_force_with_subnormal_codes():
    """Random codes over every finite E4M3 code (subnormals included), two groups with
    different scales: exact rationals from PyTorch's E4M3 values."""
    rng = np.random.default_rng(61)
    M, N, K = 2, 3, 256
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    codes = rng.choice(finite, (N, K))
    codes[0, :16] = np.arange(16, dtype=np.uint8)  # zero and the subnormal / small codes
    s = synth.to_bf16_bits(rng.uniform(0.25, 4.0, (N, K // 128)))
    a = synth.to_bf16_bits(rng.normal(size=(M, K)))
    R, absum = Q.fp8w_from_canonical(a, codes, s)
    wv = _e4m3_values_torch(codes)
    av, sv = F.decode_bf16(a), F.decode_bf16(s)
    for m in range(M):
        for n in range(N):
            ex = sum(Fraction(float(av[m, k])) * Fraction(float(wv[n, k])) *
                     Fraction(float(sv[n, k // 128])) for k in range(K))
            assert abs(Fraction(R[m, n]) - ex) <= Fraction(2.0 ** -50) * Fraction(absum[m, n])


def test_fp8w_from_canonical_rows_and_cols():
    p = synth.fp8w_problem(6, 20, 256, cfg_id=62, bias=True)
    R, S = Q.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], p["bias"][0])
    rows, cols = np.array([1, 4]), np.array([0, 7, 19])
    R2, S2 = Q.fp8w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], p["bias"][0],
                                   rows=rows, cols=cols)
    assert np.array_equal(R[np.ix_(rows, cols)], R2) and np.array_equal(S[np.ix_(rows, cols)], S2)


def test_fp8w_rejects_nan_codes():
    codes = np.zeros((2, 128), np.uint8)
    codes[1, 5] = 0xFF
    with pytest.raises(F.FormatError):
        Q.gemm_w8a16_fp8(synth.to_bf16_bits(np.ones((1, 128))), codes,
                         synth.to_bf16_bits(np.ones((2, 1))))


def test_planted_subnormal_e4m3_decode_is_caught(monkeypatch):
    """A decoder that treats exponent 0 as normal must fail the brute-force pin."""
    good = F.decode_e4m3

    def bad(codes):
        c = np.asarray(codes).astype(np.int64)
        v = good(codes)
        e, m = (c >> 3) & 0xF, c & 7
        wrong = (1.0 + m / 8.0) * 2.0 ** -7 * np.where((c >> 7) & 1, -1.0, 1.0)
        return np.where((e == 0) & (m != 0), wrong, v)

    monkeypatch.setattr(F, "decode_e4m3", bad)
    with pytest.raises(AssertionError):
        test_fp8w_fraction_brute_force_with_subnormal_codes()


# ----------------------------------------------------------------------------- second-level scales
def test_scale2_of_ones_is_the_identity():
    p = synth.w4a16_problem(3, 20, 256, bits=4, cfg_id=63, bias=True)
    q = F.unpack_int4(p["w_canon"][0], 256)
    R, S = Q.gemm_w4a16(p["A"], q, p["s_canon"][0])
    Rb, Sb = Q.gemm_w4a16(p["A"], q, p["s_canon"][0], p["bias"][0])
    R2, S2 = Q.apply_scale2(R, S, np.ones(20, np.float32), p["bias"][0])
    assert np.array_equal(R2, Rb) and np.array_equal(S2, Sb)


def test_scale2_equals_scaled_weights_exactly():
    """Integer activations, unit group scales and power-of-two t per channel: t * (a w) must
    equal a (t w) exactly, with t folded into the weights of an independent integer GEMM;
    N != M so a t applied along the wrong axis cannot broadcast."""
    rng = np.random.default_rng(64)
    M, N, K = 3, 7, 256
    a = rng.integers(-50, 51, (M, K))
    q = rng.integers(-7, 8, (N, K))
    e = rng.integers(-6, 7, N)
    t = np.ldexp(np.ones(N, np.float32), e).astype(np.float32) * np.where(rng.random(N) < 0.3, -1, 1)
    R, S = Q.gemm_w4a16(bf16_bits_of(a), q, np.full((N, 2), 0x3F80, np.uint16))
    R2, S2 = Q.apply_scale2(R, S, t)
    want = (a.astype(np.float64) @ (q.astype(np.float64) * t[:, None].astype(np.float64)).T)
    assert np.array_equal(R2, want)
    assert np.array_equal(S2, np.abs(a) @ np.abs(q * t[:, None].astype(np.float64)).T)


def test_scale2_applies_before_the_bias_and_rejects_non_finite():
    R = np.array([[2.0, 4.0]])
    S = np.array([[2.0, 4.0]])
    b = bf16_bits_of(np.array([1.0, -1.0]))
    R2, S2 = Q.apply_scale2(R, S, np.array([0.5, 3.0], np.float32), b)
    assert np.array_equal(R2, np.array([[2.0, 11.0]])) and np.array_equal(S2, np.array([[2.0, 13.0]]))
    with pytest.raises(F.FormatError):
        Q.apply_scale2(R, S, np.array([1.0, np.inf], np.float32))
