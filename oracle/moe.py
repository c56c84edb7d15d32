"""Oracle MoE routing and grouped GEMM (CPU).  Test infrastructure only.

The pages describe MoE execution where tokens spread over several experts and
each expert's load varies (spke.com Humming announcement, "背景" and "WnA16": the
Indexed and Grouped paths; "フォーマットとアーキテクチャを横断して共有される
CUDAコンポーネント": each GEMM type has its own scheduling).  They do not print the
router; the reading used here (top-k by logit, no softmax inside the GEMM) is:

  1. topk_ids[t] = the k experts with the largest float32 logit, in descending
     logit order; equal logits go to the lower expert index.
  2. counts[e] = number of (t, j) with topk_ids[t, j] == e; offsets = exclusive
     prefix sum of counts, length E + 1.
  3. The pairs p = t * k + j are ordered by (expert, p): sorted_pairs[r] is the
     pair that lands in row r of the expert-contiguous ("Grouped") layout.

Grouped GEMM: row r of the output is pair p = sorted_pairs[r] with expert e (the
segment containing r); R[r, :] = x_r @ W_e^T with x_r the row's input.

Pins (tests/test_oracle_route.py): brute-force full sort per token written with
Python's sorted(); torch.topk + a stable argsort on tie-free logits; a hand-built
tie case with its expected order in tests/golden/route_ties.txt.
"""
from __future__ import annotations

import numpy as np

from . import qgemm


def route_topk(logits, k: int) -> np.ndarray:
    """float32 [T][E] -> int32 [T][k]."""
    x = np.asarray(logits, dtype=np.float32)
    T, E = x.shape
    idx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary -> sort by -logit, then by expert index
    order = np.lexsort((idx, -x.astype(np.float64)), axis=1)
    return order[:, :k].astype(np.int32)


def route_sort(topk_ids, E: int):
    """-> counts [E], offsets [E+1], sorted_pairs [T*k] (all int32)."""
    ids = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    counts = np.bincount(ids, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    sorted_pairs = np.argsort(ids, kind="stable")
    return counts.astype(np.int32), offsets.astype(np.int32), sorted_pairs.astype(np.int32)


def route(logits, k: int):
    ids = route_topk(logits, k)
    counts, offsets, sorted_pairs = route_sort(ids, np.asarray(logits).shape[1])
    return ids, counts, offsets, sorted_pairs


def expert_of_rows(offsets) -> np.ndarray:
    off = np.asarray(offsets, dtype=np.int64)
    E = off.size - 1
    return np.repeat(np.arange(E), np.diff(off))


def grouped_w4a16(A_sorted_bits, offsets, q, s_bits, bias_bits=None, rows=None, cols=None):
    """A_sorted_bits [P][K] BF16 (already in sorted-row order), q [E][N][K] ints,
    s_bits [E][N][K/128] -> (R [len(rows)][len(cols)], absum) for the sampled rows."""
    P = np.asarray(A_sorted_bits).shape[0]
    rows = np.arange(P) if rows is None else np.asarray(rows)
    exp = expert_of_rows(offsets)[rows]
    N = np.asarray(q).shape[1]
    cols = np.arange(N) if cols is None else np.asarray(cols)
    R = np.zeros((rows.size, cols.size))
    S = np.zeros((rows.size, cols.size))
    for e in np.unique(exp):
        sel = np.nonzero(exp == e)[0]
        b = None if bias_bits is None else np.asarray(bias_bits)[e][cols]
        r, s = qgemm.gemm_w4a16(np.asarray(A_sorted_bits)[rows[sel]], np.asarray(q)[e][cols],
                                np.asarray(s_bits)[e][cols], b)
        R[sel], S[sel] = r, s
    return R, S


def grouped_w4a8(A_sorted, A_sf_sorted, offsets, w_codes, w_sf, bias_bits=None, rows=None, cols=None):
    """A_sorted [P][K] E4M3 codes, A_sf_sorted [P][K/32], w_codes [E][N][K] 4-bit codes,
    w_sf [E][N][K/32] -> (R, absum) for the sampled rows / columns."""
    P = np.asarray(A_sorted).shape[0]
    rows = np.arange(P) if rows is None else np.asarray(rows)
    exp = expert_of_rows(offsets)[rows]
    N = np.asarray(w_codes).shape[1]
    cols = np.arange(N) if cols is None else np.asarray(cols)
    R = np.zeros((rows.size, cols.size))
    S = np.zeros((rows.size, cols.size))
    for e in np.unique(exp):
        sel = np.nonzero(exp == e)[0]
        b = None if bias_bits is None else np.asarray(bias_bits)[e][cols]
        r, s = qgemm.gemm_w4a8(np.asarray(A_sorted)[rows[sel]], np.asarray(A_sf_sorted)[rows[sel]],
                               np.asarray(w_codes)[e][cols], np.asarray(w_sf)[e][cols], b)
        R[sel], S[sel] = r, s
    return R, S
