"""Oracle format decoders (float64, CPU).  Test infrastructure only.

The pages name the formats (INT4/INT3 symmetric with group scales, MXFP4 = E2M1
with E8M0 group-32 scales, MXFP8 = E4M3 with E8M0 group-32 scales; spke.com
Humming announcement, sections "WnA16" and "W8A8 / W4A8 / W4A4"; aireiter.com,
"H100 group-32 W4A8") but do not print their bit layouts.  The readings used here
are the OCP Microscaling v1.0 / OFP8 definitions, and for the packed integer
words the layouts fixed by the library's header (8 INT4 per uint32 with element
8j+i at bits [4i,4i+4) of word j; INT3 as a 96-bit little-endian stream per 32
elements; E2M1 two per byte, even k in the low nibble).

Pins (tests/test_oracle_formats.py):
  decode_e2m1   closed-form E2M1 float definition, all 16 codes
  decode_e4m3   torch.float8_e4m3fn -> float64 for all 254 finite codes
  decode_e8m0   torch.float8_e8m0fnu -> float64 and math.ldexp, all 255 codes
  decode_bf16   torch.bfloat16 -> float64
  unpack_int4   hand-written words in tests/golden/int4_words.txt
  unpack_int3   hand-written stream in tests/golden/int3_stream.txt + bit-string build
  unpack_e2m1_bytes  hand-written bytes in tests/golden/e2m1_bytes.txt
  unpack_int1   hand-written words in tests/golden/int1_words.txt, random words against a
                bit-string construction
  e0m_encode / e0m_decode  the zero-exponent-float equivalence of the spke.com page,
                section "量子化サポート" (INT8 without -128 == float8e0m7 value set)
"""
from __future__ import annotations

import numpy as np


class FormatError(ValueError):
    """A code outside the format's valid set (NaN encodings, the excluded INT minimum)."""


# E2M1 magnitudes by the low three code bits [e1 e0 m]: exponent bias 1, one mantissa
# bit, e == 0 is subnormal (OCP MX v1.0, FP4 E2M1).  No inf / NaN encodings exist.
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def decode_e2m1(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64)
    mag = _E2M1_MAG[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def decode_e4m3(codes) -> np.ndarray:
    """OFP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits.  e == 0 is
    subnormal (m/8 * 2^-6).  S.1111.111 is NaN (rejected); there is no infinity."""
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    if np.any((e == 15) & (m == 7)):
        raise FormatError("E4M3 NaN code")
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    mag = np.where(e == 0, sub, normal)
    return np.where(s == 1, -mag, mag)


def decode_e8m0(codes) -> np.ndarray:
    """E8M0 scale: byte e -> 2^(e - 127); 0xFF is NaN (rejected)."""
    c = np.asarray(codes).astype(np.int64)
    if np.any(c == 255):
        raise FormatError("E8M0 NaN code")
    return np.exp2(c.astype(np.float64) - 127.0)


def decode_bf16(bits) -> np.ndarray:
    """BF16 bits are the top half of an IEEE binary32; widen exactly."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def unpack_int4(words, K: int) -> np.ndarray:
    """uint32 [..., K/8] -> int8 [..., K]; two's-complement nibbles, -8 rejected."""
    w = np.asarray(words).astype(np.uint32)
    assert w.shape[-1] * 8 == K
    out = np.empty((*w.shape[:-1], K), dtype=np.int8)
    for i in range(8):
        nib = ((w >> np.uint32(4 * i)) & np.uint32(0xF)).astype(np.int16)
        out[..., i::8] = np.where(nib >= 8, nib - 16, nib)
    if np.any(out == -8):
        raise FormatError("INT4 code -8 is outside the symmetric range")
    return out


def unpack_int2(words, K: int) -> np.ndarray:
    """uint32 [..., K/16] -> int8 [..., K]; element k = 16j + i at bits [2i, 2i + 2) of
    word j, two's complement; -2 rejected (the symmetric range is {-1, 0, 1})."""
    w = np.asarray(words).astype(np.uint32)
    assert w.shape[-1] * 16 == K
    out = np.empty((*w.shape[:-1], K), dtype=np.int8)
    for i in range(16):
        f = ((w >> np.uint32(2 * i)) & np.uint32(3)).astype(np.int16)
        out[..., i::16] = np.where(f >= 2, f - 4, f)
    if np.any(out == -2):
        raise FormatError("INT2 code -2 is outside the symmetric range")
    return out


def unpack_int1(words, K: int) -> np.ndarray:
    """uint32 [..., K/32] -> int8 [..., K] in {-1, +1}; element k = 32j + i is bit i of
    word j, and bit b stands for the weight 2b - 1.

    Reading: the announcement (section "WnA16") lists INT1 among the weight types without
    defining it.  A one-bit two's-complement integer without its minimum (the rule the
    other symmetric widths follow) would hold only 0, so INT1 is read as sign
    quantisation: the two codes are -1 and +1 and the group scale sets the magnitude."""
    w = np.asarray(words).astype(np.uint32)
    assert w.shape[-1] * 32 == K
    out = np.empty((*w.shape[:-1], K), dtype=np.int8)
    for i in range(32):
        b = ((w >> np.uint32(i)) & np.uint32(1)).astype(np.int8)
        out[..., i::32] = 2 * b - 1
    return out


def unpack_uint4(words, K: int) -> np.ndarray:
    """uint32 [..., K/8] -> int16 [..., K] in [0, 15]; element k = 8j + i at bits
    [4i, 4i + 4) of word j (the INT4 packing, read unsigned)."""
    w = np.asarray(words).astype(np.uint32)
    assert w.shape[-1] * 8 == K
    out = np.empty((*w.shape[:-1], K), dtype=np.int16)
    for i in range(8):
        out[..., i::8] = ((w >> np.uint32(4 * i)) & np.uint32(0xF)).astype(np.int16)
    return out


def split_zp_scales(words):
    """Asymmetric INT4 group words uint32 [..., G]: bits 0-15 the BF16 scale, bits 16-23
    the zero point (0..15), bits 24-31 zero -> (scale BF16 bits uint16, zero point int16)."""
    w = np.asarray(words).astype(np.uint32)
    z = ((w >> np.uint32(16)) & np.uint32(0xFF)).astype(np.int16)
    if np.any((w >> np.uint32(24)) != 0) or np.any(z > 15):
        raise FormatError("zero point outside [0, 15]")
    return (w & np.uint32(0xFFFF)).astype(np.uint16), z


def unpack_int3(words, K: int) -> np.ndarray:
    """uint32 [..., K/32, 3] -> int8 [..., K]; element i of each 32-block at stream
    bits [3i, 3i+3) of the 96-bit little-endian stream (word 0 = bits 0..31);
    two's complement, -4 rejected."""
    w = np.asarray(words).astype(np.uint64)
    assert w.shape[-1] == 3 and w.shape[-2] * 32 == K
    stream96 = [w[..., 0], w[..., 1], w[..., 2]]
    out = np.empty((*w.shape[:-2], K // 32, 32), dtype=np.int8)
    for i in range(32):
        v = np.zeros(w.shape[:-1], dtype=np.uint64)
        for b in range(3):
            bit = 3 * i + b
            word, off = divmod(bit, 32)
            v |= ((stream96[word] >> np.uint64(off)) & np.uint64(1)) << np.uint64(b)
        vi = v.astype(np.int16)
        out[..., i] = np.where(vi >= 4, vi - 8, vi)
    out = out.reshape(*w.shape[:-2], K)
    if np.any(out == -4):
        raise FormatError("INT3 code -4 is outside the symmetric range")
    return out


def unpack_e2m1_bytes(packed, K: int) -> np.ndarray:
    """uint8 [..., K/2] -> 4-bit codes [..., K]; even k in the low nibble."""
    p = np.asarray(packed).astype(np.uint8)
    assert p.shape[-1] * 2 == K
    out = np.empty((*p.shape[:-1], K), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e0m_encode(q, mbits: int) -> np.ndarray:
    """Symmetric integer in [-(2^m - 1), 2^m - 1] -> code of a float with zero
    exponent bits and m mantissa bits: sign bit above the magnitude bits."""
    q = np.asarray(q).astype(np.int64)
    lim = (1 << mbits) - 1
    if np.any(np.abs(q) > lim):
        raise FormatError("value outside the symmetric range of e0m%d" % mbits)
    return ((q < 0).astype(np.int64) << mbits) | np.abs(q)


def e0m_decode(code, mbits: int) -> np.ndarray:
    """e0m code -> its value in units of the mantissa LSB: (-1)^s * m."""
    c = np.asarray(code).astype(np.int64)
    mag = c & ((1 << mbits) - 1)
    return np.where((c >> mbits) & 1, -mag, mag)
