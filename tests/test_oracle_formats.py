"""Pins for the oracle's format decoders (CPU only)."""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats as F


# ----------------------------------------------------------------------------- E2M1
def e2m1_closed_form(code: int) -> float:
    """OCP MX v1.0 FP4 E2M1 from its float definition: bias 1, subnormal at e == 0."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def test_e2m1_all_codes_match_float_definition():
    got = F.decode_e2m1(np.arange(16))
    want = np.array([e2m1_closed_form(c) for c in range(16)])
    assert np.array_equal(got, want)
    # the value set the MX spec lists, both signs
    assert sorted(set(np.abs(got).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_golden_bytes():
    for ln in read_golden("e2m1_bytes.txt"):
        byte_s, vals = ln.split(":")
        byte = int(byte_s, 16)
        want = [float(v) for v in vals.split()]
        codes = F.unpack_e2m1_bytes(np.array([[byte]], dtype=np.uint8), 2)[0]
        got = F.decode_e2m1(codes)
        assert got.tolist() == want, ln
        assert [math.copysign(1, g) for g in got] == [math.copysign(1, w) for w in want]


# ----------------------------------------------------------------------------- E4M3
def test_e4m3_all_finite_codes_match_torch():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.decode_e4m3(codes)
    assert np.array_equal(got, want)
    assert got.max() == 448.0 and got.min() == -448.0
    assert np.min(np.abs(got[got != 0])) == 2.0 ** -9


@pytest.mark.parametrize("nan_code", [0x7F, 0xFF])
def test_e4m3_nan_rejected(nan_code):
    with pytest.raises(F.FormatError):
        F.decode_e4m3([nan_code])


# ----------------------------------------------------------------------------- E8M0
def test_e8m0_matches_ldexp_and_torch():
    codes = np.arange(255, dtype=np.uint8)
    got = F.decode_e8m0(codes)
    assert np.array_equal(got, np.array([math.ldexp(1.0, int(c) - 127) for c in codes]))
    if hasattr(torch, "float8_e8m0fnu"):
        t = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(got, t)
    with pytest.raises(F.FormatError):
        F.decode_e8m0([255])


# ----------------------------------------------------------------------------- BF16
def test_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 4096).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite only
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.decode_bf16(bits), want)


# ----------------------------------------------------------------------------- INT4 / INT3
def test_int4_golden_words():
    for ln in read_golden("int4_words.txt"):
        w, vals = ln.split(":")
        got = F.unpack_int4(np.array([int(w, 16)], dtype=np.uint32), 8)
        assert got.tolist() == [int(v) for v in vals.split()], ln


def test_int4_minus8_rejected():
    with pytest.raises(F.FormatError):
        F.unpack_int4(np.array([0x00000008], dtype=np.uint32), 8)


def test_int3_golden_stream():
    for ln in read_golden("int3_stream.txt"):
        ws, vals = ln.split(":")
        words = np.array([[int(x, 16) for x in ws.split()]], dtype=np.uint32)
        got = F.unpack_int3(words, 32)
        assert got.tolist() == [int(v) for v in vals.split()], ln


def _int3_words_by_bitstring(values):
    """Independent construction: concatenate 3-bit two's-complement fields LSB first."""
    bits = "".join(format(v & 7, "03b")[::-1] for v in values)  # LSB-first per field
    return [int(bits[32 * w:32 * (w + 1)][::-1], 2) for w in range(3)]


def test_int3_random_vs_bitstring_construction():
    rng = np.random.default_rng(1)
    for _ in range(50):
        vals = rng.integers(-3, 4, 32).tolist()
        words = np.array([_int3_words_by_bitstring(vals)], dtype=np.uint32)
        assert F.unpack_int3(words, 32).tolist() == vals


def test_int3_minus4_rejected():
    words = np.array([_int3_words_by_bitstring([-4] + [0] * 31)], dtype=np.uint32)
    with pytest.raises(F.FormatError):
        F.unpack_int3(words, 32)


def _int2_word_by_bitstring(values):
    """Independent construction: 2-bit two's-complement fields, LSB first."""
    bits = "".join(format(v & 3, "02b")[::-1] for v in values)
    return int(bits[::-1], 2)


def test_int2_hand_word():
    # [1, -1, 0, 1, 0 ...]: fields 01, 11, 00, 01 -> 0b01_00_11_01 = 0x4D
    vals = [1, -1, 0, 1] + [0] * 12
    assert _int2_word_by_bitstring(vals) == 0x4D
    assert F.unpack_int2(np.array([0x4D], dtype=np.uint32), 16).tolist() == vals


def test_int2_random_vs_bitstring_construction():
    rng = np.random.default_rng(2)
    for _ in range(50):
        vals = rng.integers(-1, 2, 32).tolist()
        words = np.array([[_int2_word_by_bitstring(vals[:16]), _int2_word_by_bitstring(vals[16:])]],
                         dtype=np.uint32)
        assert F.unpack_int2(words, 32).tolist() == [vals]


def test_int2_minus2_rejected():
    with pytest.raises(F.FormatError):
        F.unpack_int2(np.array([0x2], dtype=np.uint32), 16)


# ----------------------------------------------------------------------------- e0m equivalence
@pytest.mark.parametrize("bits", [8, 4, 3])
def test_e0m_value_set_equals_symmetric_int(bits):
    """spke.com announcement, section "量子化サポート": the zero-exponent float of a bit
    width has exactly the values of the symmetric INT of that width without its minimum
    (INT8 without -128 and float8e0m7 both cover -127..127)."""
    m = bits - 1
    lo, hi = -(1 << m), (1 << m) - 1  # two's-complement range
    sym = set(range(lo + 1, hi + 1))  # minimum excluded
    e0m_values = set(F.e0m_decode(np.arange(1 << bits), m).tolist())
    assert e0m_values == sym
    # the two encodings agree on every value (the -0 e0m code also decodes to 0)
    q = np.arange(lo + 1, hi + 1)
    assert np.array_equal(F.e0m_decode(F.e0m_encode(q, m), m), q)
    with pytest.raises(F.FormatError):
        F.e0m_encode([lo], m)
