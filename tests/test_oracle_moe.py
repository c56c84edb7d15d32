"""Pins for the oracle's grouped-MoE helpers (CPU only).

expert_of_rows, grouped_w4a16 and grouped_w4a8 are what the grouped GPU kernels are
judged against, so each is pinned to something other than itself:
  - a hand-written offsets vector with empty experts at the start, in the middle and at
    the end, and its row -> expert list (tests/golden/grouped_rows.txt);
  - a brute force that finds each row's expert by scanning the offsets in plain Python and
    evaluates that row alone with the (separately pinned) dense oracle GEMM;
  - exact integer results with unit scales, each row against its own expert's int64 dot;
  - a planted mistake (the expert list rolled by one row) that these pins must catch.
The reading (spke.com Humming announcement, "WnA16", Grouped MoE layout): expert e owns
rows offsets[e] .. offsets[e+1]-1.
"""
import os

import numpy as np
import pytest

from oracle import formats as OF
from oracle import moe as OM
from oracle import qgemm as OQ
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "grouped_rows.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(v) for v in rest]
    return vals


def _scan_expert(offsets, r):
    """The expert whose segment holds row r, by a plain scan over the offsets."""
    for e in range(len(offsets) - 1):
        if offsets[e] <= r < offsets[e + 1]:
            return e
    raise AssertionError(f"row {r} is in no segment")


def test_expert_of_rows_golden():
    g = _golden()
    got = OM.expert_of_rows(np.array(g["offsets"]))
    assert got.tolist() == g["expert"]
    assert len(got) == g["offsets"][-1] == len(g["rows"])
    assert all(_scan_expert(g["offsets"], r) == e for r, e in zip(g["rows"], g["expert"]))


def test_expert_of_rows_brute_force_random_segments():
    rng = np.random.default_rng(41)
    for E in (1, 2, 9, 64):
        counts = rng.integers(0, 5, E) * (rng.random(E) < 0.6)  # many empty experts
        offsets = np.concatenate([[0], np.cumsum(counts)])
        got = OM.expert_of_rows(offsets)
        assert got.tolist() == [_scan_expert(offsets.tolist(), r) for r in range(offsets[-1])]


def _w4a16_case(cfg):
    g = _golden()
    off = np.array(g["offsets"], dtype=np.int32)
    E, P, N, K = len(off) - 1, int(off[-1]), 24, 256
    p = synth.w4a16_problem(P, N, K, bits=4, E=E, cfg_id=cfg)
    q = OF.unpack_int4(p["w_canon"], K)  # [E][N][K]
    return off, p["A"], q, p["s_canon"]


def _w4a8_case(cfg):
    g = _golden()
    off = np.array(g["offsets"], dtype=np.int32)
    E, P, N, K = len(off) - 1, int(off[-1]), 24, 128
    p = synth.w4a8_problem(P, N, K, E=E, cfg_id=cfg)
    codes = OF.unpack_e2m1_bytes(p["w_canon"], K)
    return off, p["A"], p["A_sf"], codes, p["s_canon"]


def _brute_w4a16(off, A, q, s, rows, cols):
    R = np.zeros((len(rows), len(cols)))
    for i, r in enumerate(rows):
        e = _scan_expert(off.tolist(), int(r))
        R[i], _ = OQ.gemm_w4a16(A[r:r + 1], q[e][cols], s[e][cols])
    return R


def _brute_w4a8(off, A, Asf, codes, sf, rows, cols):
    R = np.zeros((len(rows), len(cols)))
    for i, r in enumerate(rows):
        e = _scan_expert(off.tolist(), int(r))
        R[i], _ = OQ.gemm_w4a8(A[r:r + 1], Asf[r:r + 1], codes[e][cols], sf[e][cols])
    return R


def test_grouped_w4a16_equals_per_row_brute_force():
    off, A, q, s = _w4a16_case(501)
    P, N = A.shape[0], q.shape[1]
    R, S = OM.grouped_w4a16(A, off, q, s)
    assert np.array_equal(R, _brute_w4a16(off, A, q, s, np.arange(P), np.arange(N)))
    assert np.all(S > 0)
    # the sampled form (rows and columns in any order) the full-size GPU tests use
    rows, cols = np.array([8, 0, 4, 3, 5]), np.array([23, 0, 7])
    Rs, _ = OM.grouped_w4a16(A, off, q, s, rows=rows, cols=cols)
    assert np.array_equal(Rs, _brute_w4a16(off, A, q, s, rows, cols))


def test_grouped_w4a8_equals_per_row_brute_force():
    off, A, Asf, codes, sf = _w4a8_case(502)
    P, N = A.shape[0], codes.shape[1]
    R, _ = OM.grouped_w4a8(A, Asf, off, codes, sf)
    assert np.array_equal(R, _brute_w4a8(off, A, Asf, codes, sf, np.arange(P), np.arange(N)))
    rows, cols = np.array([2, 7, 3]), np.array([5, 1, 22, 9])
    Rs, _ = OM.grouped_w4a8(A, Asf, off, codes, sf, rows=rows, cols=cols)
    assert np.array_equal(Rs, _brute_w4a8(off, A, Asf, codes, sf, rows, cols))


def test_grouped_w4a16_exact_integers_per_expert():
    """Unit scales and integer activations: row r must equal the int64 dot of its
    activations with its own expert's codes (expert found by scanning the offsets)."""
    g = _golden()
    off = np.array(g["offsets"])
    E, P, N, K = len(off) - 1, int(off[-1]), 5, 256
    rng = np.random.default_rng(43)
    a = rng.integers(-200, 201, (P, K))
    q = rng.integers(-7, 8, (E, N, K))
    s = np.full((E, N, K // 128), 0x3F80, dtype=np.uint16)  # BF16 1.0
    R, _ = OM.grouped_w4a16(synth.to_bf16_bits(a.astype(np.float64)), off, q, s)
    for r in range(P):
        e = _scan_expert(off.tolist(), r)
        assert np.array_equal(R[r], (a[r] @ q[e].T).astype(np.float64)), r


def test_planted_wrong_expert_is_caught(monkeypatch):
    """Roll the oracle's row -> expert list by one row: the brute-force pins must fail."""
    off, A, q, s = _w4a16_case(503)
    true_rows = OM.expert_of_rows
    monkeypatch.setattr(OM, "expert_of_rows", lambda o: np.roll(true_rows(o), 1))
    P, N = A.shape[0], q.shape[1]
    R, _ = OM.grouped_w4a16(A, off, q, s)
    assert not np.array_equal(R, _brute_w4a16(off, A, q, s, np.arange(P), np.arange(N)))
    offm, Am, Asf, codes, sf = _w4a8_case(504)
    Rm, _ = OM.grouped_w4a8(Am, Asf, offm, codes, sf)
    assert not np.array_equal(
        Rm, _brute_w4a8(offm, Am, Asf, codes, sf, np.arange(Am.shape[0]), np.arange(codes.shape[1])))
    g = _golden()
    assert OM.expert_of_rows(np.array(g["offsets"])).tolist() != g["expert"]
