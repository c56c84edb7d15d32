"""Oracle for the activation-side MoE steps (float64, CPU).  Test infrastructure only.

These are the steps either side of the quantized GEMMs in a MoE layer that the pages
time together with them (spke.com Humming announcement: the MoE benchmark times
"gate-up + down" as one unit, section "パフォーマンス"; serving uses token-wise FP8 /
MXFP8 activations, sections "W8A8 / W4A8 / W4A4" and the closing FAQ on choosing MXFP8
activations).  The pages do not spell the steps out; the readings are:

  quantize_mxfp8  OCP Microscaling v1.0 conversion of a group of 32 values to MXFP8:
                  shared exponent X = floor(log2(max|v|)) - 8 (8 = the exponent of the
                  largest E4M3 power of two), clamped to the E8M0 range; elements
                  v / 2^X rounded to nearest-even E4M3 and saturated to +-448 (the
                  format has no infinity).  An all-zero group gets the scale code 0.
  silu_mul        y = silu(g) * u with g the first and u the second half of each row of
                  the fused gate+up projection (the intermediate-640 workload's N = 1280
                  = 2 x 640), silu(g) = g / (1 + exp(-g)); BF16 round-to-nearest-even.
  combine         out[t] = sum_j w[t][j] * Y[row of pair (t, j)], the weights the softmax
                  over token t's k selected router logits (the renormalised top-k of a
                  softmax router); BF16 round-to-nearest-even.

Pins (tests/test_oracle_act.py):
  encode_e4m3      every finite code round-trips; random values against a brute-force
                   nearest-even search over all 254 finite values; torch.float8_e4m3fn
                   casts of in-range values; saturation above 448
  quantize_mxfp8   hand-computed groups in tests/golden/mxfp8_groups.txt; exact
                   reconstruction of representable inputs; the scale rule
                   256 <= amax / 2^X < 512; the element error bound
  round_bf16       torch.bfloat16 casts (round-to-nearest-even) of random float64 values
  silu_mul         torch's float64 silu; silu(0) = 0
  combine          brute force over explicit loops on tiny inputs; k = 1 is the inverse
                   permutation
"""
from __future__ import annotations

import numpy as np

from .formats import FormatError, decode_bf16, decode_e4m3

# All non-negative finite E4M3 values, by code (0..126; 127 is NaN).
_E4M3_POS = decode_e4m3(np.arange(127))


def encode_e4m3(x) -> np.ndarray:
    """float64 -> E4M3 code: round to nearest, ties to the even code, saturate to 448.
    The sign is kept (a negative value that rounds to zero gives -0, code 0x80)."""
    v = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(v)):
        raise FormatError("non-finite value")
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def quantize_mxfp8(x_bits, group: int = 32):
    """BF16 bits [rows][K] -> (E4M3 codes uint8 [rows][K], E8M0 scales uint8 [rows][K/32])."""
    x = decode_bf16(np.asarray(x_bits).view(np.uint16))
    rows, K = x.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    if np.any(~np.isfinite(x)):
        raise FormatError("non-finite activation")
    g = x.reshape(rows, K // group, group)
    amax = np.abs(g).max(axis=2)
    _, p = np.frexp(amax)              # amax = m 2^p, m in [0.5, 1): floor(log2) = p - 1
    X = np.where(amax > 0, p - 1 - 8, -127)
    X = np.clip(X, -127, 127)
    codes = encode_e4m3(g / np.exp2(X)[..., None])
    return codes.reshape(rows, K), (X + 127).astype(np.uint8)


def round_bf16(x) -> np.ndarray:
    """float64 -> BF16 bits, round to nearest even (finite, normal-range inputs)."""
    v = np.asarray(x, dtype=np.float64)
    m, p = np.frexp(v)                 # v = m 2^p, |m| in [0.5, 1)
    r = np.rint(m * 256.0)             # 8 significant bits, ties to even
    q = np.ldexp(r, p - 8)             # exactly representable in float32 and BF16
    return (q.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def silu_mul(gate_up_bits) -> np.ndarray:
    """BF16 bits [rows][2I] -> BF16 bits [rows][I]: silu(first half) * second half."""
    gu = decode_bf16(np.asarray(gate_up_bits).view(np.uint16))
    half = gu.shape[1] // 2
    g, u = gu[:, :half], gu[:, half:]
    return round_bf16(g / (1.0 + np.exp(-g)) * u)


def combine_weights(logits, topk_ids) -> np.ndarray:
    """Softmax over each token's selected logits: float64 [T][k]."""
    lg = np.asarray(logits, dtype=np.float64)
    sel = np.take_along_axis(lg, np.asarray(topk_ids, dtype=np.int64), axis=1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def combine(Y_bits, sorted_pairs, topk_ids, logits):
    """Weighted sum of each token's k expert rows.  Y rows are in sorted-pair order
    (row i holds pair sorted_pairs[i] = t * k + j).  Returns (BF16 bits [T][N], the float64
    result and the sum of |w y| per element for the tolerance check)."""
    Y = decode_bf16(np.asarray(Y_bits).view(np.uint16))
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    pos = np.empty(T * k, dtype=np.int64)
    pos[np.asarray(sorted_pairs, dtype=np.int64)] = np.arange(T * k)
    w = combine_weights(logits, ids)
    rows = Y[pos.reshape(T, k)]                     # [T][k][N]
    R = np.einsum("tk,tkn->tn", w, rows)
    S = np.einsum("tk,tkn->tn", np.abs(w), np.abs(rows))
    return round_bf16(R), R, S
