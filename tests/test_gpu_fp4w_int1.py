"""FP4-weight WnA16 (E2M1 codes, BF16 scale per 128) and INT1 WnA16 (sign codes, bit b =
weight 2b - 1, BF16 scale per 128) through every W4A16-family path - single-token decode
kernel, staged GEMV, register-ring GEMV, grouped TMA-ring GEMV and the tcgen05 kernel -
against the float64 oracle; repack round trip bit for bit; the packed layout of one block
read back against the header's formula, written out here."""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from qwtest import dev, host, qw, repack, route, u16_view

pytestmark = pytest.mark.gpu


def _fmt(kind):
    Q = qw()
    return Q.QW_W_FP4E2M1_G128_BF16 if kind == "fp4" else Q.QW_W_INT1_G128_BF16


def _problem(kind, M, N, K, E=1, cfg_id=0, bias=False):
    if kind == "fp4":
        return synth.fp4w_problem(M, N, K, E=E, cfg_id=cfg_id, bias=bias)
    return synth.w4a16_problem(M, N, K, bits=1, E=E, cfg_id=cfg_id, bias=bias)


def _oracle(kind, p, A, e=0, bias=None):
    if kind == "fp4":
        return OQ.fp4w_from_canonical(A, p["w_canon"][e], p["s_canon"][e], p["K"], bias)
    return OQ.w4a16_from_canonical(A, p["w_canon"][e], p["s_canon"][e], p["K"], 1, bias)


def _dense(kind, p, bias=None):
    Q = qw()
    N, K = p["N"], p["K"]
    d, wp, sp = repack(_fmt(kind), 1, N, K, p["w_canon"], p["s_canon"])
    M = p["A"].shape[0]
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, dev(p["A"].view(np.int16)), None, b, C, M, ws, wsn,
                  err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


@pytest.mark.parametrize("kind", ["fp4", "int1"])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 4096), (1, 4104, 14336), (1, 1032, 640),
                                   (3, 264, 384), (8, 256, 1024), (13, 296, 256),
                                   (16, 264, 640), (48, 384, 1024), (300, 1280, 640),
                                   (130, 136, 128)])
def test_dense_paths(kind, M, N, K):
    """M = 1: the decode kernel (K = 640 has no split with whole ring batches: staged GEMV);
    other M <= 16: register ring; M > 16: tcgen05.  Ragged N and K of one to 112 groups."""
    p = _problem(kind, M, N, K, cfg_id=1100 + M)
    C = _dense(kind, p)
    R, S = _oracle(kind, p, p["A"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("kind", ["fp4", "int1"])
@pytest.mark.parametrize("M", [1, 5, 64])
def test_bias(kind, M):
    p = _problem(kind, M, 1000, 256, cfg_id=1150 + M, bias=True)
    C = _dense(kind, p, bias=p["bias"][0])
    R, S = _oracle(kind, p, p["A"], bias=p["bias"][0])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("kind", ["fp4", "int1"])
def test_repack_round_trip(kind):
    Q = qw()
    E, N, K = 3, 40, 384
    p = _problem(kind, 1, N, K, E=E, cfg_id=1170)
    d, wp, sp = repack(_fmt(kind), E, N, K, p["w_canon"], p["s_canon"])
    blk = 1024 if kind == "fp4" else 256
    assert d.N_pad == 48 and d.w_bytes == E * 3 * 3 * blk and d.group == 128
    if kind == "fp4":
        wc = torch.empty((E, N, K // 2), dtype=torch.uint8, device="cuda")
    else:
        wc = torch.empty((E, N, K // 32), dtype=torch.int32, device="cuda")
    sc = torch.empty((E, N, K // 128), dtype=torch.int16, device="cuda")
    Q.qw_unpack(d, wp, sp, wc, sc)
    got = host(wc) if kind == "fp4" else host(wc).view(np.uint32)
    assert np.array_equal(got, p["w_canon"])
    assert np.array_equal(host(sc).view(np.uint16), p["s_canon"])


def test_int1_packed_layout_of_one_block():
    """Register r of MMA step s for lane 4g + t (rows g + 8 (r & 1), k = 16s + 4t + 2 (r >> 1)
    + h) at bit 4 (s % 4) + r + 16h of word s / 4 - read back for one 16 x 128 block."""
    Q = qw()
    N, K = 16, 128
    rng = np.random.default_rng(7)
    signs = 2 * rng.integers(0, 2, (1, N, K)) - 1
    d, wp, sp = repack(Q.QW_W_INT1_G128_BF16, 1, N, K, synth.pack_int1(signs),
                       np.full((1, N, 1), 0x3F80, np.uint16))
    words = host(wp)[:256].view("<u4").reshape(32, 2)
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        for s in range(8):
            for r in range(4):
                for h in range(2):
                    row, k = g + 8 * (r & 1), 16 * s + 4 * t + 2 * (r >> 1) + h
                    bit = (int(words[lane, s // 4]) >> (4 * (s % 4) + r + 16 * h)) & 1
                    assert 2 * bit - 1 == signs[0, row, k]


def test_fp4_packed_layout_of_one_block():
    """Byte r of word s of lane 4g + t holds the codes of row g + 8 (r & 1) at
    k = 16s + 4t + 2 (r >> 1) (low nibble) and k + 1 (high nibble)."""
    Q = qw()
    N, K = 16, 128
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 16, (1, N, K)).astype(np.uint8)
    d, wp, sp = repack(Q.QW_W_FP4E2M1_G128_BF16, 1, N, K, synth.pack_nibbles(codes),
                       np.full((1, N, 1), 0x3F80, np.uint16))
    words = host(wp)[:1024].view("<u4").reshape(32, 8)
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        for s in range(8):
            for r in range(4):
                row, k = g + 8 * (r & 1), 16 * s + 4 * t + 2 * (r >> 1)
                byte = (int(words[lane, s]) >> (8 * r)) & 0xFF
                assert byte & 0xF == codes[0, row, k] and byte >> 4 == codes[0, row, k + 1]


@pytest.mark.parametrize("kind", ["fp4", "int1"])
@pytest.mark.parametrize("T", [1, 12, 32])
def test_grouped_moe(kind, T):
    """E = 8 top-8: 1 and 12 rows per expert (grouped TMA-ring GEMV), 32 (tcgen05)."""
    Q = qw()
    E, K, N, k = 8, 512, 264, 8
    p = _problem(kind, T, N, K, E=E, cfg_id=1180 + T)
    logits = synth.router_logits(T, E, cfg_id=1180 + T)
    d, wp, sp = repack(_fmt(kind), E, N, K, p["w_canon"], p["s_canon"])
    ids, spairs, off = route(logits, k)
    P = T * k
    A = dev(p["A"].view(np.int16))
    As = torch.empty((P, K), dtype=torch.int16, device="cuda")
    sp_dev, off_dev = dev(spairs.astype(np.int32)), dev(off.astype(np.int32))
    Q.qgemm_moe_permute(Q.QW_A_BF16, A, None, K, sp_dev, P, k, As, None)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp, Q.QW_A_BF16, As, None, off_dev, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    tok = spairs // k
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    Rall, Sall = np.zeros((P, N)), np.zeros((P, N))
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        Rall[sel], Sall[sel] = _oracle(kind, p, p["A"][tok[sel]], e=e)
    ok, ratio, frob = OQ.check_bf16_result(Cn, Rall, Sall)
    assert ok, (ratio, frob)
