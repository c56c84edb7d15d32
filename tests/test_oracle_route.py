"""Pins for the oracle router (CPU only)."""
import numpy as np
import torch

from conftest import read_golden
from oracle import moe
import synth


def _parse_ties():
    d = {"logits": [], "topk": []}
    for ln in read_golden("route_ties.txt"):
        key, *vals = ln.split()
        if key in ("logits", "topk"):
            d[key].append([float(v) for v in vals])
        else:
            d[key] = [int(v) for v in vals]
    return d


def test_route_tie_golden():
    g = _parse_ties()
    logits = np.array(g["logits"], dtype=np.float32)
    ids, counts, offsets, sp = moe.route(logits, g["k"][0])
    assert ids.tolist() == [[int(v) for v in r] for r in g["topk"]]
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert sp.tolist() == g["sorted_pairs"]


def test_topk_brute_force_sorted():
    rng = np.random.default_rng(3)
    T, E, k = 7, 12, 4
    logits = rng.integers(-3, 4, (T, E)).astype(np.float32)  # many ties
    ids = moe.route_topk(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        assert ids[t].tolist() == order[:k]


def test_route_matches_torch_on_tie_free_logits():
    logits = synth.router_logits(64, 32, cfg_id=99)
    k = 8
    ids, counts, offsets, sp = moe.route(logits, k)
    tv, ti = torch.topk(torch.from_numpy(logits), k, dim=1, sorted=True)
    assert np.array_equal(ids, ti.numpy())
    flat = torch.from_numpy(ids.reshape(-1).astype(np.int64))
    assert np.array_equal(sp, torch.sort(flat, stable=True).indices.numpy())
    assert np.array_equal(counts, torch.bincount(flat, minlength=32).numpy())
    assert offsets[0] == 0 and offsets[-1] == 64 * k


def test_sorted_pairs_is_a_stable_permutation():
    logits = synth.router_logits(50, 16, cfg_id=98)
    ids, counts, offsets, sp = moe.route(logits, 3)
    assert sorted(sp.tolist()) == list(range(150))
    flat = ids.reshape(-1)
    for e in range(16):
        seg = sp[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
