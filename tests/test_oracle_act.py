"""Pins of the activation-side oracle (oracle/act.py) against things other than itself."""
import numpy as np
import pytest
import torch

import synth
from conftest import read_golden
from oracle import act as OA
from oracle import formats as OF


def _fval(tok):
    return float.fromhex(tok) if tok.lstrip("-").startswith("0x") else float(tok)


# ----------------------------------------------------------------------------- E4M3 encoder
def test_e4m3_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = OF.decode_e4m3(codes)
    back = OA.encode_e4m3(vals)
    # +0 and -0 both decode to 0.0; -0.0 keeps its sign bit
    assert np.array_equal(back, codes)


def test_e4m3_nearest_even_brute_force():
    rng = np.random.default_rng(11)
    table = OF.decode_e4m3(np.arange(127))
    x = np.concatenate([rng.uniform(0, 448, 4000), rng.uniform(0, 2 ** -5, 1000),
                        (table[:-1] + table[1:]) / 2])          # include every midpoint
    got = OA.encode_e4m3(x)
    for xi, ci in zip(x, got):
        d = np.abs(table - xi)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert ci == want, (xi, ci, want)


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(12)
    x = rng.normal(0, 60, 20000).clip(-448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(OA.encode_e4m3(x), ref)


def test_e4m3_saturates():
    assert list(OA.encode_e4m3([448.0, 449.0, 1e6, -1e6])) == [126, 126, 126, 254]


# ----------------------------------------------------------------------------- MXFP8 quantizer
def _golden_groups():
    lines = read_golden("mxfp8_groups.txt")
    groups = []
    for i in range(0, len(lines), 3):
        xs, ss, qs = lines[i].split()[1:], lines[i + 1].split()[1:], lines[i + 2].split()[1:]
        x = np.zeros(32)
        for j in range(0, len(xs), 2):
            x[int(xs[j])] = _fval(xs[j + 1])
        q = np.zeros(32, dtype=np.uint8)
        for j in range(0, len(qs), 2):
            q[int(qs[j])] = int(qs[j + 1])
        groups.append((x, int(ss[0]), q))
    return groups


def test_mxfp8_hand_computed_groups():
    groups = _golden_groups()
    assert len(groups) == 6
    x = np.stack([g[0] for g in groups])
    bits = synth.to_bf16_bits(x)
    assert np.array_equal(OF.decode_bf16(bits), x)  # the fixture values are exact in BF16
    codes, sf = OA.quantize_mxfp8(bits)
    assert list(sf[:, 0]) == [g[1] for g in groups]
    for r, g in enumerate(groups):
        assert np.array_equal(codes[r], g[2]), r


def test_mxfp8_exact_reconstruction_of_representable_inputs():
    rng = np.random.default_rng(13)
    rows, K = 16, 256
    codes = rng.integers(0, 256, (rows, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x20
    # force each group's largest magnitude into [256, 448] so the scale rule recovers X
    codes[:, ::32] = 0x78 | (rng.integers(0, 7, (rows, K // 32)).astype(np.uint8))
    X = rng.integers(-20, 10, (rows, K // 32))
    vals = OF.decode_e4m3(codes) * np.exp2(np.repeat(X, 32, axis=1))
    bits = synth.to_bf16_bits(vals)
    assert np.array_equal(OF.decode_bf16(bits), vals)
    q, sf = OA.quantize_mxfp8(bits)
    assert np.array_equal(sf.astype(np.int64) - 127, X)
    assert np.array_equal(OF.decode_e4m3(q), OF.decode_e4m3(codes))


def test_mxfp8_scale_rule_and_error_bound():
    rng = np.random.default_rng(14)
    x = rng.normal(0, 3, (32, 512)) * np.exp2(rng.integers(-30, 30, (32, 1)))
    bits = synth.to_bf16_bits(x)
    xv = OF.decode_bf16(bits).reshape(32, 16, 32)
    q, sf = OA.quantize_mxfp8(bits)
    scale = np.exp2(sf.astype(np.float64) - 127)
    amax = np.abs(xv).max(axis=2)
    assert np.all((amax / scale >= 256) & (amax / scale < 512))
    deq = OF.decode_e4m3(q).reshape(32, 16, 32) * scale[..., None]
    v = np.abs(xv) / scale[..., None]
    # not saturated: within half a step of E4M3 at that magnitude (3 mantissa bits)
    step = np.where(v >= 2 ** -6, np.exp2(np.floor(np.log2(np.maximum(v, 2 ** -6))) - 3), 2 ** -9)
    ok = v <= 448
    assert np.all(np.abs(deq - xv)[ok] <= (0.5 * step * scale[..., None])[ok] * (1 + 1e-12))
    assert np.all(np.abs(deq)[~ok] == 448 * np.broadcast_to(scale[..., None], deq.shape)[~ok])


def test_mxfp8_rejects_non_finite():
    bits = synth.to_bf16_bits(np.zeros((1, 32)))
    bits[0, 3] = 0x7FC0  # NaN
    with pytest.raises(OF.FormatError):
        OA.quantize_mxfp8(bits)


# ----------------------------------------------------------------------------- BF16 rounding, SiLU
def test_round_bf16_matches_torch():
    rng = np.random.default_rng(15)
    x = rng.normal(0, 1, 20000) * np.exp2(rng.integers(-60, 60, 20000))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(OA.round_bf16(x), ref)


def test_silu_mul_matches_torch_float64():
    rng = np.random.default_rng(16)
    gu = synth.to_bf16_bits(rng.normal(0, 3, (8, 2 * 96)))
    v = OF.decode_bf16(gu)
    g, u = torch.from_numpy(v[:, :96]), torch.from_numpy(v[:, 96:])
    ref = (torch.nn.functional.silu(g) * u).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(OA.silu_mul(gu), ref.view(np.uint16))
    zero = synth.to_bf16_bits(np.array([[0.0, 5.0]]))
    assert OF.decode_bf16(OA.silu_mul(zero))[0, 0] == 0.0


# ----------------------------------------------------------------------------- combine
def test_combine_brute_force_loops():
    rng = np.random.default_rng(17)
    T, E, k, N = 5, 6, 3, 7
    logits = rng.normal(0, 1, (T, E))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    sp = rng.permutation(T * k)                      # any order of the pairs
    Y = synth.to_bf16_bits(rng.normal(0, 1, (T * k, N)))
    yv = OF.decode_bf16(Y)
    out, R, S = OA.combine(Y, sp, ids, logits)
    for t in range(T):
        sel = [logits[t, ids[t, j]] for j in range(k)]
        m = max(sel)
        e = [np.exp(s - m) for s in sel]
        w = [ei / sum(e) for ei in e]
        for n in range(N):
            acc = 0.0
            for j in range(k):
                row = int(np.flatnonzero(sp == t * k + j)[0])
                acc += w[j] * yv[row, n]
            assert abs(R[t, n] - acc) <= 1e-12 * (1 + abs(acc))
    assert np.allclose(OA.combine_weights(logits, ids).sum(axis=1), 1.0)


def test_combine_k1_is_the_inverse_permutation():
    rng = np.random.default_rng(18)
    T, E, N = 9, 4, 5
    ids = rng.integers(0, E, (T, 1))
    sp = rng.permutation(T)
    Y = synth.to_bf16_bits(rng.normal(0, 1, (T, N)))
    out, _, _ = OA.combine(Y, sp, ids, rng.normal(0, 1, (T, E)))
    for i, pair in enumerate(sp):
        assert np.array_equal(out[pair], Y[i])
