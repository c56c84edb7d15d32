"""Pins for the oracle's FP4-weight and INT1 WnA16 GEMMs and the INT1 unpacking (CPU only).

The announcement (spke.com, section "WnA16") lists INT1 and FP4 among the weight types of
its WnA16 kernels.  Readings: FP4 weights are E2M1 codes (OCP MX v1.0 element values) with
the integer formats' BF16 scale per 128 along K; INT1 is sign quantisation, bit b standing
for the weight 2b - 1.  Each function is pinned to something other than itself: hand-written
words, exact integer dot products, an exact rational brute force with the E2M1 values
written out here as fractions, and planted mistakes that must be caught.
"""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import qgemm as Q
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int1_words.txt")

# E2M1 magnitudes written out independently of the oracle's table (OCP MX v1.0: exponent
# bias 1, one mantissa bit, e = 0 subnormal)
E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
        Fraction(4), Fraction(6)]


def e2m1_exact(code):
    v = E2M1[code & 7]
    return -v if code & 8 else v


def bf16_exact(bits):
    return Fraction(float(torch.tensor([int(bits) << 16], dtype=torch.int64)
                          .to(torch.int32).view(torch.float32).item()))


def golden_int1():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        word, vals = line.split(":")
        rows.append((int(word, 16), [int(v) for v in vals.split()]))
    return rows


# ----------------------------------------------------------------------------- INT1
def test_unpack_int1_golden():
    for word, vals in golden_int1():
        got = F.unpack_int1(np.array([word], dtype=np.uint32), 32)
        assert got.tolist() == vals, hex(word)


def test_unpack_int1_random_against_bit_strings():
    rng = np.random.default_rng(61)
    words = rng.integers(0, 2 ** 32, (5, 4), dtype=np.uint64).astype(np.uint32)
    got = F.unpack_int1(words, 128)
    for r in range(5):
        bits = "".join(format(int(w), "032b")[::-1] for w in words[r])  # bit i first
        assert got[r].tolist() == [1 if b == "1" else -1 for b in bits]


def test_int1_exact_integer_dot():
    """Unit scales and integer activations: the result is the int64 dot with +-1 weights."""
    rng = np.random.default_rng(62)
    M, N, K = 3, 7, 256
    a = rng.integers(-200, 201, (M, K))
    q = 2 * rng.integers(0, 2, (N, K)) - 1
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
    R, _ = Q.w4a16_from_canonical(synth.to_bf16_bits(a.astype(np.float64)), synth.pack_int1(q),
                                  s, K, 1)
    assert np.array_equal(R, (a @ q.T).astype(np.float64))


def test_int1_fraction_brute_force_with_group_scales():
    rng = np.random.default_rng(63)
    M, N, K = 2, 3, 256
    p = synth.w4a16_problem(M, N, K, bits=1, cfg_id=64)
    R, _ = Q.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, 1)
    words = p["w_canon"][0]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                b = (int(words[n, k // 32]) >> (k % 32)) & 1
                acc += bf16_exact(p["A"][m, k]) * (2 * b - 1) * bf16_exact(p["s_canon"][0][n, k // 128])
            assert Fraction(R[m, n]) == acc


def test_planted_int1_bit_order_is_caught(monkeypatch):
    """Reading the bits from the top of the word instead of the bottom breaks the golden."""
    true = F.unpack_int1

    def reversed_bits(words, K):
        w = np.asarray(words).astype(np.uint32)
        rev = np.zeros_like(w)
        for i in range(32):
            rev |= ((w >> np.uint32(i)) & np.uint32(1)) << np.uint32(31 - i)
        return true(rev, K)
    monkeypatch.setattr(F, "unpack_int1", reversed_bits)
    with pytest.raises(AssertionError):
        test_unpack_int1_golden()


# ----------------------------------------------------------------------------- FP4 weights
def test_fp4w_exact_integer_valued_codes():
    """Codes of integer E2M1 values (0, +-1, +-2, +-3, +-4, +-6), unit scales and integer
    activations: an exact int64 dot."""
    rng = np.random.default_rng(65)
    M, N, K = 4, 9, 384
    int_codes = np.array([0, 2, 4, 5, 6, 7, 8, 10, 12, 13, 14, 15], dtype=np.uint8)
    codes = int_codes[rng.integers(0, int_codes.size, (N, K))]
    vals = np.array([int(e2m1_exact(int(c))) for c in codes.reshape(-1)]).reshape(N, K)
    a = rng.integers(-100, 101, (M, K))
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
    R, _ = Q.fp4w_from_canonical(synth.to_bf16_bits(a.astype(np.float64)),
                                 synth.pack_nibbles(codes), s, K)
    assert np.array_equal(R, (a @ vals.T).astype(np.float64))


def test_fp4w_fraction_brute_force_all_codes():
    """Every one of the sixteen codes, BF16 activations and scales: exact rationals."""
    M, N, K = 2, 16, 256
    p = synth.fp4w_problem(M, N, K, cfg_id=66)
    codes = p["codes"][0].copy()
    codes[:, :16] = np.arange(16, dtype=np.uint8)[None, :]  # all codes on every row
    R, _ = Q.fp4w_from_canonical(p["A"], synth.pack_nibbles(codes), p["s_canon"][0], K)
    for m in range(M):
        for n in range(N):
            acc = sum(bf16_exact(p["A"][m, k]) * e2m1_exact(int(codes[n, k])) *
                      bf16_exact(p["s_canon"][0][n, k // 128]) for k in range(K))
            assert Fraction(R[m, n]) == acc


def test_fp4w_nibble_order():
    """Even k sits in the low nibble: one byte 0x21 puts code 1 (0.5) at k = 0 and code 2
    (1.0) at k = 1, so activations (4, 1) give 3 and the swapped order 4.5."""
    K = 128
    w = np.zeros((1, K // 2), dtype=np.uint8)
    w[0, 0] = 0x21
    a = np.zeros((1, K))
    a[0, 0], a[0, 1] = 4.0, 1.0
    s = np.full((1, 1), 0x3F80, dtype=np.uint16)
    R, _ = Q.fp4w_from_canonical(synth.to_bf16_bits(a), w, s, K)
    assert R[0, 0] == 3.0


def test_planted_wrong_e2m1_entry_is_caught(monkeypatch):
    wrong = F._E2M1_MAG.copy()
    wrong[5] = 2.5  # 3.0 written as 2.5
    monkeypatch.setattr(F, "_E2M1_MAG", wrong)
    with pytest.raises(AssertionError):
        test_fp4w_fraction_brute_force_all_codes()
