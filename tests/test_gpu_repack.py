"""Repack / unpack on the GPU: bit-exact round trips and device-detected value errors."""
import numpy as np
import pytest
import torch

import synth
from qwtest import dev, host, qw

pytestmark = pytest.mark.gpu


def roundtrip(wfmt, E, N, K, w_canon, s_canon):
    Q = qw()
    d = Q.qw_repack_query(wfmt, E, N, K)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(w_canon), dev(s_canon), wp, sp, err)
    assert Q.qw_read_error(err) == 0
    wc2 = torch.zeros(w_canon.nbytes, dtype=torch.uint8, device="cuda")
    sc2 = torch.zeros(s_canon.nbytes, dtype=torch.uint8, device="cuda")
    Q.qw_unpack(d, wp, sp, wc2, sc2, err)
    assert Q.qw_read_error(err) == 0
    return host(wc2), host(sc2), d, wp, sp


@pytest.mark.parametrize("bits", [4, 3, 2])
@pytest.mark.parametrize("E,N,K", [(1, 2048, 2048), (3, 40, 384), (2, 1280, 4096), (1, 16, 128)])
def test_int_roundtrip_bit_exact(bits, E, N, K):
    p = synth.w4a16_problem(1, N, K, bits=bits, E=E, cfg_id=50 + bits)
    wfmt = {4: 0, 3: 1, 2: 6}[bits]
    wc2, sc2, _, _, _ = roundtrip(wfmt, E, N, K, p["w_canon"], p["s_canon"])
    assert np.array_equal(wc2, p["w_canon"].reshape(-1).view(np.uint8))
    assert np.array_equal(sc2, p["s_canon"].reshape(-1).view(np.uint8))


@pytest.mark.parametrize("E,N,K", [(1, 3072, 4096), (2, 300, 96), (4, 640, 7168), (1, 1, 32)])
def test_mxfp4_roundtrip_bit_exact(E, N, K):
    p = synth.w4a8_problem(1, N, K, E=E, cfg_id=60)
    wc2, sc2, d, wp, sp = roundtrip(2, E, N, K, p["w_canon"], p["s_canon"])
    assert np.array_equal(wc2, p["w_canon"].reshape(-1))
    assert np.array_equal(sc2, p["s_canon"].reshape(-1))
    # padding: zero codes, scale 127
    wpk = host(wp).reshape(E, d.N_pad, d.K_pad // 2)
    assert np.all(wpk[:, N:, :] == 0) and np.all(wpk[:, :N, K // 2:] == 0)


def test_int4_packed_codes_are_excess8_fragments():
    """One 16 x 128 block: word (lane, step) nibble i holds q[row][k] + 8 with the m16n8k16
    fragment mapping row = g + 8(r & 1), k = 16s + 4t + 2(r >> 1) + h (r = i & 3, h = i >> 2)."""
    rng = np.random.default_rng(5)
    q = rng.integers(-7, 8, (1, 16, 128))
    s = synth.to_bf16_bits(np.ones((1, 16, 1)))
    Q = qw()
    d = Q.qw_repack_query(0, 1, 16, 128)
    wp, sp = Q.empty_packed(d)
    Q.qw_repack(d, dev(synth.pack_int4(q)), dev(s), wp, sp)
    words = host(wp).view(np.uint32).reshape(32, 8)
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for step in range(8):
            for i in range(8):
                r, h = i & 3, i >> 2
                row, k = g + 8 * (r & 1), 16 * step + 4 * t + 2 * (r >> 1) + h
                assert (words[lane, step] >> (4 * i)) & 0xF == q[0, row, k] + 8


def test_int3_packed_codes_are_three_bit_fields():
    """One 16 x 128 block: the lane's six words (4 at lane*16, 2 at 512 + lane*8) hold
    u = q + 4 of pair j = 4s + r (rows g + 8(r & 1), k = 16s + 4t + 2(r >> 1) + h) at
    bits 3(j % 5) + 16h of word j / 5 for j < 30, and bit i of u at bit 15 + 16h of word
    i (j = 30) or 3 + i (j = 31)."""
    rng = np.random.default_rng(7)
    q = rng.integers(-3, 4, (1, 16, 128))
    s = synth.to_bf16_bits(np.ones((1, 16, 1)))
    Q = qw()
    d = Q.qw_repack_query(1, 1, 16, 128)
    wp, sp = Q.empty_packed(d)
    Q.qw_repack(d, dev(synth.pack_int3(q)), dev(s), wp, sp)
    raw = host(wp).view(np.uint32)
    assert raw.size == 192
    for lane in range(32):
        g, t = lane // 4, lane % 4
        w = [int(x) for x in raw[lane * 4:lane * 4 + 4]] + \
            [int(x) for x in raw[128 + lane * 2:128 + lane * 2 + 2]]
        for step in range(8):
            for r in range(4):
                j = 4 * step + r
                for h in range(2):
                    row, k = g + 8 * (r & 1), 16 * step + 4 * t + 2 * (r >> 1) + h
                    if j < 30:
                        u = (w[j // 5] >> (3 * (j % 5) + 16 * h)) & 7
                    else:
                        b = 0 if j == 30 else 3
                        u = sum(((w[b + i] >> (15 + 16 * h)) & 1) << i for i in range(3))
                    assert u == q[0, row, k] + 4, (lane, step, r, h)


def test_int2_packed_codes_are_two_bit_fields():
    """One 16 x 128 block: word s // 2 of lane l holds u = q + 2 of pair (s, r) at bits
    2(4(s % 2) + r) + 16h, the (row, k) assignment as for INT4."""
    rng = np.random.default_rng(8)
    q = rng.integers(-1, 2, (1, 16, 128))
    s = synth.to_bf16_bits(np.ones((1, 16, 1)))
    Q = qw()
    d = Q.qw_repack_query(6, 1, 16, 128)
    wp, sp = Q.empty_packed(d)
    Q.qw_repack(d, dev(synth.pack_int2(q)), dev(s), wp, sp)
    words = host(wp).view(np.uint32).reshape(32, 4)
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for step in range(8):
            for r in range(4):
                for h in range(2):
                    row, k = g + 8 * (r & 1), 16 * step + 4 * t + 2 * (r >> 1) + h
                    u = (int(words[lane, step // 2]) >> (2 * (4 * (step % 2) + r) + 16 * h)) & 3
                    assert u == q[0, row, k] + 2, (lane, step, r, h)


def test_value_errors_flagged():
    Q = qw()
    # INT4 code -8
    q = np.zeros((1, 16, 128), np.int64)
    q[0, 3, 77] = -8
    d = Q.qw_repack_query(0, 1, 16, 128)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(synth.pack_int4(q)), dev(np.zeros((1, 16, 1), np.uint16)), wp, sp, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE
    # INT3 code -4
    d = Q.qw_repack_query(1, 1, 16, 128)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(synth.pack_int3(q // 2)), dev(np.zeros((1, 16, 1), np.uint16)), wp, sp, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE
    # E8M0 0xFF
    p = synth.w4a8_problem(1, 128, 128, cfg_id=61)
    sf = p["s_canon"].copy()
    sf[0, 5, 2] = 0xFF
    d = Q.qw_repack_query(2, 1, 128, 128)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(p["w_canon"]), dev(sf), wp, sp, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE


def test_bounded_wait_reports_timeout():
    """A wait on a barrier nothing arrives on gives up and reports; the context stays usable."""
    Q = qw()
    err = Q.new_error_flag()
    Q.qw_test_wait_timeout(err, 20_000_000)  # 20 ms
    assert Q.qw_read_error(err) == Q.QW_ERR_TIMEOUT
    x = torch.ones(4, device="cuda")
    assert float((x + 1).sum()) == 8.0


def test_int2_minus2_flagged():
    Q = qw()
    N, K = 16, 128
    p = synth.w4a16_problem(1, N, K, bits=2, cfg_id=59)
    bad = p["w_canon"].copy()
    bad[0, 3, 2] = (bad[0, 3, 2] & ~np.uint32(3 << 6)) | np.uint32(2 << 6)  # element 35 = -2
    d = Q.qw_repack_query(Q.QW_W_INT2_G128_BF16, 1, N, K)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, dev(bad), dev(p["s_canon"]), wp, sp, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_VALUE
