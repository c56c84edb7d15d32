"""Packed layouts read back from the device buffers against the byte formulas of
include/qw.h, written out independently here: the INT block order over several blocks,
groups and experts with the BF16 scale plane, the MX scale-chunk image (512 bytes per 128
rows x 4 groups) and the NVFP4 chunk of four 512-byte images (2048 bytes per 128 rows x 16
groups)."""
import numpy as np
import pytest

import synth
from qwtest import dev, host, qw, repack

pytestmark = pytest.mark.gpu


def test_int4_block_order_over_groups_blocks_and_experts_and_scale_plane():
    """Expert e, group G, block nb: the 1 KiB block at e * w_expert_stride +
    (G * N_pad / 16 + nb) * 1024 holds rows 16 nb .. 16 nb + 15, k = 128 G .. 128 G + 127 in
    the fragment order; scales BF16 at e * s_expert_stride + (G * N_pad + n) * 2."""
    Q = qw()
    E, N, K = 2, 40, 384  # N_pad 48: three blocks, the last one ragged; three groups
    rng = np.random.default_rng(21)
    q = rng.integers(-7, 8, (E, N, K))
    s = rng.integers(0x3C00, 0x4100, (E, N, K // 128)).astype(np.uint16)
    d, wp, sp = repack(Q.QW_W_INT4_G128_BF16, E, N, K, synth.pack_int4(q), s)
    W = host(wp).view(np.uint8)
    S = host(sp).view(np.uint8)
    nblk = d.N_pad // 16
    for e in range(E):
        for G in range(K // 128):
            for nb in range(nblk):
                base = e * d.w_expert_stride + (G * nblk + nb) * 1024
                words = W[base:base + 1024].view("<u4").reshape(32, 8)
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    for st in range(8):
                        for i in range(8):
                            r, h = i & 3, i >> 2
                            row = 16 * nb + g + 8 * (r & 1)
                            k = 128 * G + 16 * st + 4 * t + 2 * (r >> 1) + h
                            want = q[e, row, k] + 8 if row < N else 8  # padding rows: q = 0
                            assert (int(words[lane, st]) >> (4 * i)) & 0xF == want
            plane = S[e * d.s_expert_stride + G * d.N_pad * 2:
                      e * d.s_expert_stride + (G + 1) * d.N_pad * 2].view("<u2")
            assert np.array_equal(plane[:N], s[e, :, G])


def _mx_scale_byte_offset(r, g, K_pad):
    """MXFP4 / MXFP8 scales: chunk (r / 128, g / 4) at ((r / 128) * (K_pad / 128) + g / 4) *
    512, byte (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4."""
    return ((r // 128) * (K_pad // 128) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4


def test_mx_scale_chunk_image():
    Q = qw()
    N, K = 200, 224  # N_pad 256, K_pad 256: two row chunks, two group chunks, padding
    rng = np.random.default_rng(22)
    codes = rng.integers(0, 256, (1, N, K // 2)).astype(np.uint8)
    sf = rng.integers(100, 140, (1, N, K // 32)).astype(np.uint8)
    d, wp, sp = repack(Q.QW_W_MXFP4_G32, 1, N, K, codes, sf)
    S = host(sp).view(np.uint8)
    assert d.s_bytes == (d.N_pad // 128) * (d.K_pad // 128) * 512
    seen = np.zeros(d.s_bytes, bool)
    for r in range(d.N_pad):
        for g in range(d.K_pad // 32):
            off = _mx_scale_byte_offset(r, g, d.K_pad)
            want = sf[0, r, g] if (r < N and g < K // 32) else 127  # padding: scale 1
            assert S[off] == want, (r, g)
            seen[off] = True
    assert seen.all()  # the formula covers every byte exactly once


def _nv_scale_byte_offset(r, g, K_pad):
    """NVFP4 scales: chunk (r / 128, g / 16) at ((r / 128) * (K_pad / 256) + g / 16) * 2048,
    byte ((g % 16) / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4."""
    return (((r // 128) * (K_pad // 256) + g // 16) * 2048 + ((g % 16) // 4) * 512 +
            (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4)


def test_nvfp4_scale_chunk_four_images():
    Q = qw()
    N, K = 136, 416  # N_pad 256, K_pad 512
    rng = np.random.default_rng(23)
    codes = rng.integers(0, 256, (1, N, K // 2)).astype(np.uint8)
    sf = rng.integers(0x28, 0x48, (1, N, K // 16)).astype(np.uint8)
    d, wp, sp = repack(Q.QW_W_NVFP4_G16, 1, N, K, codes, sf)
    S = host(sp).view(np.uint8)
    assert d.s_bytes == (d.N_pad // 128) * (d.K_pad // 256) * 2048
    seen = np.zeros(d.s_bytes, bool)
    for r in range(d.N_pad):
        for g in range(d.K_pad // 16):
            off = _nv_scale_byte_offset(r, g, d.K_pad)
            want = sf[0, r, g] if (r < N and g < K // 16) else 0x38  # padding: scale 1
            assert S[off] == want, (r, g)
            seen[off] = True
    assert seen.all()
