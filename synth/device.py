"""Seeded synthetic inputs drawn directly on the GPU, for workloads too large to draw on
the host in reasonable time (the grouped-MoE weights run to several GB).

The draws use PyTorch's own seeded CUDA generator (Philox); the distributions are those of
``synth.gen`` (uniform codes, uniform integers, normals cast with PyTorch's round-to-
nearest-even conversions) but the values differ from the host streams.  Like ``synth.gen``
this module holds no dequantization, GEMM or routing arithmetic; the oracle reads back
whatever part of these tensors it checks.
"""
from __future__ import annotations

import torch

from .gen import BASE_SEED


def _gen(cfg_id: int, tensor_id: int, seed: int = BASE_SEED) -> torch.Generator:
    g = torch.Generator(device="cuda")
    g.manual_seed((seed + cfg_id) * 1000003 + tensor_id)
    return g


def mxfp4_weights(E, N, K, *, cfg_id, seed=BASE_SEED, sf_lo=118, sf_hi=126):
    """E2M1 codes uniform over the 16 codes, packed two per byte ([E][N][K/2] uint8), and
    E8M0 group-32 scales uniform in [sf_lo, sf_hi] ([E][N][K/32] uint8)."""
    w = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, device="cuda",
                      generator=_gen(cfg_id, 31, seed))
    s = torch.randint(sf_lo, sf_hi + 1, (E, N, K // 32), dtype=torch.uint8, device="cuda",
                      generator=_gen(cfg_id, 32, seed))
    return w, s


def mxfp8_activations(M, K, *, cfg_id, seed=BASE_SEED, sf_lo=118, sf_hi=126):
    """E4M3 codes of N(0,1) samples ([M][K] uint8) and E8M0 group-32 scales."""
    x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=_gen(cfg_id, 33, seed))
    a = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    s = torch.randint(sf_lo, sf_hi + 1, (M, K // 32), dtype=torch.uint8, device="cuda",
                      generator=_gen(cfg_id, 34, seed))
    return a, s


def int_weights(E, N, K, *, bits, cfg_id, seed=BASE_SEED, scale_lo=0.005, scale_hi=0.02):
    """Symmetric INT4 (U{-7..7}) or INT3 (U{-3..3}) codes in the canonical packing and BF16
    group-128 scales U[scale_lo, scale_hi].  INT4: [E][N][K/8] int32 words, element 8j+i at
    bits [4i, 4i+4); INT3: [E][N][K/32][3] int32 words, a 96-bit little-endian stream."""
    qmax = 7 if bits == 4 else 3
    q = torch.randint(-qmax, qmax + 1, (E, N, K), dtype=torch.int32, device="cuda",
                      generator=_gen(cfg_id, 35 + bits, seed))
    u = q & (0xF if bits == 4 else 0x7)
    if bits == 4:
        u = u.view(E, N, K // 8, 8)
        w = torch.zeros((E, N, K // 8), dtype=torch.int64, device="cuda")
        for i in range(8):
            w |= u[..., i].to(torch.int64) << (4 * i)
    else:
        u = u.view(E, N, K // 32, 32).to(torch.int64)
        lo = torch.zeros((E, N, K // 32), dtype=torch.int64, device="cuda")  # bits 0..62
        hi = torch.zeros((E, N, K // 32), dtype=torch.int64, device="cuda")  # bits 63..95
        for i in range(32):
            b = 3 * i
            if b + 3 <= 63:
                lo |= u[..., i] << b
            else:
                hi |= u[..., i] << (b - 63)  # stream bit 63 + j at bit j of `hi`
        w0 = lo & 0xFFFFFFFF
        w1 = ((lo >> 32) & 0x7FFFFFFF) | ((hi & 1) << 31)
        w2 = (hi >> 1) & 0xFFFFFFFF
        w = torch.stack([w0, w1, w2], dim=-1)
    w = w.to(torch.int64).bitwise_and(0xFFFFFFFF)
    w = torch.where(w >= 2 ** 31, w - 2 ** 32, w).to(torch.int32)
    sc = torch.rand((E, N, K // 128), dtype=torch.float64, device="cuda",
                    generator=_gen(cfg_id, 40, seed))
    s = (scale_lo + (scale_hi - scale_lo) * sc).to(torch.bfloat16).view(torch.int16)
    return w, s


def bf16_activations(M, K, *, cfg_id, seed=BASE_SEED):
    x = torch.randn((M, K), dtype=torch.float32, device="cuda", generator=_gen(cfg_id, 41, seed))
    return x.to(torch.bfloat16).view(torch.int16)
