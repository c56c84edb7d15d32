"""Oracle GEMMs (float64, CPU).  Test infrastructure only.

What the quantized GEMMs compute (spke.com Humming announcement, section
"フォーマットとアーキテクチャを横断して共有されるCUDAコンポーネント": dequantization and
scaling are part of the kernel computation, scale and bias may be fused into the
output stage; section "WnA16": low-bit weights times 16-bit activations; section
"W8A8 / W4A8 / W4A4": MX block-scaled weights and activations):

  W4A16:  R[m,n] = sum_k a[m,k] * q[n,k] * s[n, k // G]            (+ bias[n])
  W4A16 with zero points (asymmetric INT4, the section "背景"'s symmetric / asymmetric
  quantization): R[m,n] = sum_k a[m,k] * (q[n,k] - z[n, k // G]) * s[n, k // G],
          q and z unsigned 4-bit                                    (+ bias[n])
  FP8-weight WnA16 (the section "WnA16"'s floating-point weights up to FP8; E4M3 codes
  with the same BF16 group-128 scales as the integer formats):
          R[m,n] = sum_k a[m,k] * e4m3(w[n,k]) * s[n, k // G]          (+ bias[n])
  FP4-weight WnA16 (the same section's FP4 weights; E2M1 codes with the BF16 group-128
  scales of the integer formats):
          R[m,n] = sum_k a[m,k] * e2m1(w[n,k]) * s[n, k // G]          (+ bias[n])
  INT1 WnA16 (the same section's INT1; sign quantisation, w = s * (2b - 1)):
          R[m,n] = sum_k a[m,k] * (2 b[n,k] - 1) * s[n, k // G]        (+ bias[n])
  W4A8:   R[m,n] = sum_k e4m3(a[m,k]) 2^(sa[m,k//32]-127)
                          * e2m1(w[n,k]) 2^(sw[n,k//32]-127)      (+ bias[n])
  W4A4:   R[m,n] = sum_k e2m1(a[m,k]) e4m3(sa[m,k//16])
                          * e2m1(w[n,k]) e4m3(sw[n,k//16])        (+ bias[n])
          (NVFP4 x NVFP4, the section's W4A4 / "NVFP4 x NVFP4 W4A4": E2M1 elements
          with an unsigned E4M3 scale per 16 along K; the format's per-tensor FP32
          factors are a plain multiplier of the result: apply_scale2 with equal t)

Second-level scales (section "統一されたquantization表現": the quantization description
carries them as a parameter of its own): an FP32 scale t per output channel on top of
the format's group scales, applied to the finished sum before the bias:
          R'[m,n] = t[n] * R[m,n] + bias[n]    (apply_scale2)

Every operand is decoded exactly into float64 and the sum over k is a float64
matrix product (a library matmul used as one step, no blocking or reordering
beyond it).  Weights are [N][K] (out x in), activations [M][K], results [M][N].

Pins (tests/test_oracle_gemm.py): exact int64 dot products when every scale is
1.0 and every operand an integer; exact rational (fractions.Fraction) brute force
on tiny shapes with several groups; non-square shapes so that a transposed
operand or a wrong group index changes the result; FP8-weight: equality with the W4A16
GEMM on E4M3 codes of integers, and exact rationals over every finite E4M3 code from
PyTorch's float8_e4m3fn values.  FP4-weight and INT1 (tests/test_oracle_fp4_int1.py):
exact int64 dot products on integer-valued codes, exact rationals over all sixteen E2M1
codes, hand-written INT1 words, and planted mistakes.
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def dequant_int_weights(q, s_bits, group: int = 128) -> np.ndarray:
    """q [..., N, K] integers, s_bits [..., N, K/group] BF16 bits -> float64."""
    q = np.asarray(q).astype(np.float64)
    s = F.decode_bf16(s_bits)
    return q * np.repeat(s, group, axis=-1)


def dequant_mx(codes, sf, decode) -> np.ndarray:
    """Element codes [..., R, K] with E8M0 scales [..., R, K/32] -> float64."""
    v = decode(codes)
    return v * np.repeat(F.decode_e8m0(sf), 32, axis=-1)


def gemm_w4a16(A_bits, q, s_bits, bias_bits=None, group: int = 128):
    """A_bits [M][K] BF16, q [N][K] ints, s_bits [N][K/group] BF16 -> (R, absum)."""
    a = F.decode_bf16(A_bits)
    w = dequant_int_weights(q, s_bits, group)
    r = a @ w.T
    absum = np.abs(a) @ np.abs(w).T
    if bias_bits is not None:
        b = F.decode_bf16(bias_bits)
        r = r + b[None, :]
        absum = absum + np.abs(b)[None, :]
    return r, absum


def gemm_w4a16_zp(A_bits, q, s_bits, z, bias_bits=None, group: int = 128):
    """A_bits [M][K] BF16, q [N][K] unsigned codes, s_bits [N][K/group] BF16 scales, z
    [N][K/group] zero points -> (R, absum) of w = s * (q - z)."""
    qz = np.asarray(q).astype(np.int64) - np.repeat(np.asarray(z).astype(np.int64), group, axis=-1)
    return gemm_w4a16(A_bits, qz, s_bits, bias_bits, group)


def gemm_w8a16_fp8(A_bits, w_codes, s_bits, bias_bits=None, group: int = 128):
    """A_bits [M][K] BF16, w_codes [N][K] E4M3, s_bits [N][K/group] BF16 -> (R, absum) of
    w = e4m3(code) * s: the W4A16 product with decoded E4M3 values in place of integers."""
    return gemm_w4a16(A_bits, F.decode_e4m3(w_codes), s_bits, bias_bits, group)


def gemm_w4a16_fp4(A_bits, w_codes, s_bits, bias_bits=None, group: int = 128):
    """A_bits [M][K] BF16, w_codes [N][K] E2M1 codes, s_bits [N][K/group] BF16 -> (R, absum)
    of w = e2m1(code) * s: the W4A16 product with decoded E2M1 values in place of integers."""
    return gemm_w4a16(A_bits, F.decode_e2m1(w_codes), s_bits, bias_bits, group)


def apply_scale2(R, absum, t, bias_bits=None):
    """Second-level scales: R and absum of a GEMM computed without bias, t float32 [N] ->
    (t[n] * R + bias[n], |t[n]| * absum + |bias[n]|)."""
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    if not np.all(np.isfinite(t)):
        raise F.FormatError("non-finite second-level scale")
    r = np.asarray(R) * t[None, :]
    a = np.asarray(absum) * np.abs(t)[None, :]
    if bias_bits is not None:
        b = F.decode_bf16(bias_bits)
        r = r + b[None, :]
        a = a + np.abs(b)[None, :]
    return r, a


def gemm_w4a8(A_codes, A_sf, w_codes, w_sf, bias_bits=None):
    """A_codes [M][K] E4M3, A_sf [M][K/32] E8M0, w_codes [N][K] E2M1 (4-bit codes),
    w_sf [N][K/32] E8M0 -> (R, absum)."""
    a = dequant_mx(A_codes, A_sf, F.decode_e4m3)
    w = dequant_mx(w_codes, w_sf, F.decode_e2m1)
    r = a @ w.T
    absum = np.abs(a) @ np.abs(w).T
    if bias_bits is not None:
        b = F.decode_bf16(bias_bits)
        r = r + b[None, :]
        absum = absum + np.abs(b)[None, :]
    return r, absum


def gemm_w8a8(A_codes, A_sf, w_codes, w_sf, bias_bits=None):
    """MXFP8 x MXFP8: A_codes [M][K] E4M3, A_sf [M][K/32] E8M0, w_codes [N][K] E4M3 byte
    codes, w_sf [N][K/32] E8M0 -> (R, absum).  The pages' "W8A8" MX kind (spke.com
    announcement, "W8A8 / W4A8 / W4A4")."""
    a = dequant_mx(A_codes, A_sf, F.decode_e4m3)
    w = dequant_mx(w_codes, w_sf, F.decode_e4m3)
    r = a @ w.T
    absum = np.abs(a) @ np.abs(w).T
    if bias_bits is not None:
        b = F.decode_bf16(bias_bits)
        r = r + b[None, :]
        absum = absum + np.abs(b)[None, :]
    return r, absum


def dequant_nv(codes, sf, group: int = 16) -> np.ndarray:
    """E2M1 codes [..., R, K] with E4M3 block scales [..., R, K/16] -> float64.  The
    scale is unsigned: a set sign bit or the NaN code is a FormatError."""
    sfa = np.asarray(sf).astype(np.int64)
    if np.any((sfa & 0x80) != 0) or np.any((sfa & 0x7F) == 0x7F):
        raise F.FormatError("NVFP4 scale must be a finite non-negative E4M3 code")
    return F.decode_e2m1(codes) * np.repeat(F.decode_e4m3(sfa), group, axis=-1)


def gemm_w4a4(A_codes, A_sf, w_codes, w_sf, bias_bits=None):
    """NVFP4 x NVFP4: A_codes [M][K] and w_codes [N][K] E2M1 4-bit codes, A_sf [M][K/16]
    and w_sf [N][K/16] E4M3 scale codes -> (R, absum)."""
    a = dequant_nv(A_codes, A_sf)
    w = dequant_nv(w_codes, w_sf)
    r = a @ w.T
    absum = np.abs(a) @ np.abs(w).T
    if bias_bits is not None:
        b = F.decode_bf16(bias_bits)
        r = r + b[None, :]
        absum = absum + np.abs(b)[None, :]
    return r, absum


# --------------------------------------------------------------- canonical-input drivers
def w4a16_from_canonical(A_bits, w_canon, s_canon, K, bits, bias_bits=None, rows=None, cols=None):
    """Unpack canonical packed words (one expert) and run :func:`gemm_w4a16`.
    ``rows`` / ``cols`` optionally select a sample of output rows / columns."""
    q = {4: F.unpack_int4, 3: F.unpack_int3, 2: F.unpack_int2, 1: F.unpack_int1}[bits](w_canon, K)
    A = np.asarray(A_bits)
    s = np.asarray(s_canon)
    if rows is not None:
        A = A[rows]
    if cols is not None:
        q, s = q[cols], s[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    return gemm_w4a16(A, q, s, bias_bits)


def fp4w_from_canonical(A_bits, w_canon, s_canon, K, bias_bits=None, rows=None, cols=None):
    """E2M1 codes two per byte [N][K/2] (even k in the low nibble) and BF16 group-128
    scales of one expert -> :func:`gemm_w4a16_fp4`."""
    codes = F.unpack_e2m1_bytes(w_canon, K)
    A = np.asarray(A_bits)
    s = np.asarray(s_canon)
    if rows is not None:
        A = A[rows]
    if cols is not None:
        codes, s = codes[cols], s[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    return gemm_w4a16_fp4(A, codes, s, bias_bits)


def fp8w_from_canonical(A_bits, w_canon, s_canon, bias_bits=None, rows=None, cols=None):
    """E4M3 codes [N][K] and BF16 group scales of one expert -> :func:`gemm_w8a16_fp8`
    (canonical FP8 codes are already one byte per weight)."""
    A = np.asarray(A_bits)
    w, s = np.asarray(w_canon), np.asarray(s_canon)
    if rows is not None:
        A = A[rows]
    if cols is not None:
        w, s = w[cols], s[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    return gemm_w8a16_fp8(A, w, s, bias_bits)


def w4a16_zp_from_canonical(A_bits, w_canon, sz_canon, K, bias_bits=None, rows=None,
                            cols=None):
    """Unsigned INT4 words and (scale, zero point) group words of one expert ->
    :func:`gemm_w4a16_zp`."""
    q = F.unpack_uint4(w_canon, K)
    s, z = F.split_zp_scales(sz_canon)
    A = np.asarray(A_bits)
    if rows is not None:
        A = A[rows]
    if cols is not None:
        q, s, z = q[cols], s[cols], z[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    return gemm_w4a16_zp(A, q, s, z, bias_bits)


def w4a8_from_canonical(A_codes, A_sf, w_canon, w_sf, K, bias_bits=None, rows=None, cols=None):
    w = np.asarray(w_canon)
    sf = np.asarray(w_sf)
    A, Asf = np.asarray(A_codes), np.asarray(A_sf)
    if rows is not None:
        A, Asf = A[rows], Asf[rows]
    if cols is not None:
        w, sf = w[cols], sf[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    codes = F.unpack_e2m1_bytes(w, K)
    return gemm_w4a8(A, Asf, codes, sf, bias_bits)


def w4a4_from_canonical(A_packed, A_sf, w_canon, w_sf, K, bias_bits=None, rows=None, cols=None):
    """Packed E2M1 activations [M][K/2] and weights [N][K/2] (even k in the low nibble)
    with their E4M3 scales -> :func:`gemm_w4a4`."""
    w, sf = np.asarray(w_canon), np.asarray(w_sf)
    A, Asf = np.asarray(A_packed), np.asarray(A_sf)
    if rows is not None:
        A, Asf = A[rows], Asf[rows]
    if cols is not None:
        w, sf = w[cols], sf[cols]
        bias_bits = None if bias_bits is None else np.asarray(bias_bits)[cols]
    return gemm_w4a4(F.unpack_e2m1_bytes(A, K), Asf, F.unpack_e2m1_bytes(w, K), sf, bias_bits)


# --------------------------------------------------------------- acceptance test
def check_bf16_result(C_bits, R, absum, elem_rel=2.0 ** -7, elem_abs=1e-6, frob_rel=2e-3):
    """Per-element |C - R| <= elem_rel * sum_k |a_k w_k| + elem_abs and
    ||C - R||_F <= frob_rel * ||R||_F.  Returns (ok, worst_ratio, frob)."""
    C = F.decode_bf16(C_bits)
    err = np.abs(C - R)
    bound = elem_rel * absum + elem_abs
    ratio = float(np.max(err / bound)) if err.size else 0.0
    nr = float(np.linalg.norm(R))
    frob = float(np.linalg.norm(C - R) / nr) if nr > 0 else float(np.linalg.norm(C - R))
    ok = bool(np.all(np.isfinite(C)) and ratio <= 1.0 and frob <= frob_rel)
    return ok, ratio, frob
