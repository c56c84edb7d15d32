"""Counter-based splitmix64 streams and canonical-layout packing of synthetic data.

Random numbers
--------------
Every tensor gets its own stream, keyed by ``(seed, tensor_id)``.  Element ``i``
(1-based) of a stream is ``mix64(key + i * GAMMA)`` with the splitmix64 constants
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators", 2014):
GAMMA = 0x9E3779B97F4A7C15, and ``mix64`` the published finaliser
``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
z ^= z >> 31``.  The key itself is ``mix64(seed * GAMMA + tensor_id)``.

* uniform integers in [lo, hi]: Lemire's multiply-shift on each 32-bit half of a
  draw (high half first),
* uniform reals in [0, 1): the top 53 bits times 2^-53,
* normals: Box-Muller on two consecutive uniforms (cos and sin branch).

Canonical layouts (the library's input formats)
------------------------------------------------
* INT4: ``[..., N, K/8]`` uint32; element ``k = 8j + i`` sits at bits ``[4i, 4i+4)``
  of word ``j``, two's complement.
* INT3: ``[..., N, K/32, 3]`` uint32 forming a 96-bit little-endian stream per
  32 elements; element ``i`` sits at stream bits ``[3i, 3i+3)``, two's complement.
* E2M1: ``[..., N, K/2]`` uint8; even ``k`` in the low nibble.
* E8M0 / E4M3 / BF16: one code per element, row-major.

Casts of real samples to BF16 and E4M3 codes use PyTorch's own round-to-nearest-even
conversions (a library routine); E4M3 samples are clamped to +-448 first.
"""
from __future__ import annotations

import numpy as np
import torch

BASE_SEED = 20261202

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


class Stream:
    """One splitmix64 counter stream; successive draws continue the counter."""

    def __init__(self, seed: int, tensor_id: int):
        with np.errstate(over="ignore"):
            k = np.array([seed], dtype=np.uint64) * _GAMMA + np.uint64(tensor_id)
        self.key = _mix64(k)[0]
        self.counter = 0

    def u64(self, n: int) -> np.ndarray:
        idx = np.arange(self.counter + 1, self.counter + 1 + n, dtype=np.uint64)
        self.counter += n
        with np.errstate(over="ignore"):
            return _mix64(self.key + idx * _GAMMA)


def stream(cfg_id: int, tensor_id: int, seed: int = BASE_SEED) -> Stream:
    """Stream for one tensor of one workload: seed ``seed + cfg_id``."""
    return Stream(seed + cfg_id, tensor_id)


# ----------------------------------------------------------------------------- draws
_CHUNK = 1 << 24  # draws per chunk (keeps the uint64 temporaries small)


def _chunks(n):
    for lo in range(0, n, _CHUNK):
        yield lo, min(n, lo + _CHUNK)


def uniform_int(st: Stream, shape, lo: int, hi: int) -> np.ndarray:
    """Two draws per 64-bit output: element 2j from its high 32 bits, 2j+1 from its low
    32 bits, each mapped to [lo, hi] by Lemire's multiply-shift."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    out = np.empty(n + 1, dtype=np.int64 if (hi > 127 or lo < -128) else np.int16)
    for a, b in _chunks(n):
        z = st.u64((b - a + 1) // 2)
        with np.errstate(over="ignore"):
            hi32 = ((z >> np.uint64(32)) * span) >> np.uint64(32)
            lo32 = ((z & np.uint64(0xFFFFFFFF)) * span) >> np.uint64(32)
        out[a:a + 2 * z.size:2] = hi32.astype(np.int64) + lo
        out[a + 1:a + 2 * z.size:2] = lo32.astype(np.int64) + lo
    return out[:n].reshape(shape)


def uniform(st: Stream, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for a, b in _chunks(n):
        u = (st.u64(b - a) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        out[a:b] = lo + (hi - lo) * u
    return out.reshape(shape)


def normal(st: Stream, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n + 1, dtype=np.float64)
    for a, b in _chunks(n):
        m = b - a
        pairs = (m + 1) // 2
        u = (st.u64(2 * pairs) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1 = 1.0 - u[0::2]  # (0, 1]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        out[a:a + 2 * pairs:2] = r * np.cos(2.0 * np.pi * u2)
        out[a + 1:a + 2 * pairs:2] = r * np.sin(2.0 * np.pi * u2)
    return (std * out[:n]).reshape(shape)


def random_bytes(st: Stream, n: int) -> np.ndarray:
    out = np.empty(((n + 7) // 8) * 8, dtype=np.uint8)
    nw = out.size // 8
    for a, b in _chunks(nw):
        out[8 * a:8 * b] = st.u64(b - a).view(np.uint8)
    return out[:n]


# ----------------------------------------------------------------------------- casts
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    x = np.clip(np.asarray(x, dtype=np.float64), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


# ----------------------------------------------------------------------------- packing
def pack_int4(codes: np.ndarray) -> np.ndarray:
    """int codes in [-8, 7], shape [..., K] (K % 8 == 0) -> uint32 [..., K/8]."""
    c = np.asarray(codes)
    assert c.shape[-1] % 8 == 0
    nib = (c.astype(np.int8).view(np.uint8) & np.uint8(0xF))
    # two nibbles per byte (even k low), four bytes per little-endian word
    return np.ascontiguousarray(pack_nibbles(nib)).view("<u4").astype(np.uint32, copy=False)


def pack_int2(codes: np.ndarray) -> np.ndarray:
    """int codes in [-2, 1], shape [..., K] (K % 16 == 0) -> uint32 [..., K/16]; element
    k = 16j + i at bits [2i, 2i + 2) of word j."""
    c = np.asarray(codes).astype(np.int64) & 3
    assert c.shape[-1] % 16 == 0
    c = c.reshape(*c.shape[:-1], c.shape[-1] // 16, 16).astype(np.uint64)
    w = np.zeros(c.shape[:-1], dtype=np.uint64)
    for i in range(16):
        w |= c[..., i] << np.uint64(2 * i)
    return w.astype(np.uint32)


def pack_int3(codes: np.ndarray) -> np.ndarray:
    """int codes in [-4, 3], shape [..., K] (K % 32 == 0) -> uint32 [..., K/32, 3]."""
    c = np.asarray(codes, dtype=np.int64)
    K = c.shape[-1]
    assert K % 32 == 0
    f = (c & 0x7).astype(np.uint64).reshape(*c.shape[:-1], K // 32, 32)
    lo = np.zeros(f.shape[:-1], dtype=np.uint64)  # stream bits 0..63
    hi = np.zeros(f.shape[:-1], dtype=np.uint64)  # stream bits 64..95
    for i in range(32):
        b = 3 * i
        if b + 3 <= 64:
            lo |= f[..., i] << np.uint64(b)
        if b + 3 > 64 and b < 64:  # element 21 straddles bit 64
            lo |= (f[..., i] << np.uint64(b)) & np.uint64(0xFFFFFFFFFFFFFFFF)
            hi |= f[..., i] >> np.uint64(64 - b)
        if b >= 64:
            hi |= f[..., i] << np.uint64(b - 64)
    out = np.empty((*f.shape[:-1], 3), dtype=np.uint32)
    out[..., 0] = (lo & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    out[..., 1] = (lo >> np.uint64(32)).astype(np.uint32)
    out[..., 2] = (hi & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return out


def pack_int1(signs: np.ndarray) -> np.ndarray:
    """weights in {-1, +1}, shape [..., K] (K % 32 == 0) -> uint32 [..., K/32]; element
    k = 32j + i is bit i of word j, set for +1."""
    b = (np.asarray(signs).astype(np.int64) > 0).astype(np.uint64)
    assert b.shape[-1] % 32 == 0
    b = b.reshape(*b.shape[:-1], b.shape[-1] // 32, 32)
    w = np.zeros(b.shape[:-1], dtype=np.uint64)
    for i in range(32):
        w |= b[..., i] << np.uint64(i)
    return w.astype(np.uint32)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [..., K] (K even) -> uint8 [..., K/2], even k in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


# ----------------------------------------------------------------------------- problems
def w4a16_problem(M, N, K, *, bits=4, E=1, cfg_id=0, seed=BASE_SEED,
                  scale_lo=0.005, scale_hi=0.02, bias=False):
    """Group-128 symmetric INT weights with BF16 scales and BF16 N(0,1) activations."""
    if bits == 1:  # INT1: the two codes -1 and +1, equally likely
        q = (2 * uniform_int(stream(cfg_id, 1, seed), (E, N, K), 0, 1) - 1).astype(np.int8)
    else:
        qmax = {4: 7, 3: 3, 2: 1}[bits]
        q = uniform_int(stream(cfg_id, 1, seed), (E, N, K), -qmax, qmax).astype(np.int8)
    s = to_bf16_bits(uniform(stream(cfg_id, 2, seed), (E, N, K // 128), scale_lo, scale_hi))
    a = to_bf16_bits(normal(stream(cfg_id, 3, seed), (M, K)))
    w = {4: pack_int4, 3: pack_int3, 2: pack_int2, 1: pack_int1}[bits](q)
    out = dict(A=a, q=q, w_canon=w, s_canon=s, E=E, N=N, K=K, M=M, bits=bits)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 4, seed), (E, N)))
    return out


def fp4w_problem(M, N, K, *, E=1, cfg_id=0, seed=BASE_SEED, scale_lo=0.005, scale_hi=0.02,
                 bias=False):
    """FP4-weight WnA16: E2M1 codes uniform over the 16 codes (two per byte, even k in the
    low nibble), BF16 scales per 128 along K, BF16 N(0,1) activations."""
    codes = uniform_int(stream(cfg_id, 1, seed), (E, N, K), 0, 15).astype(np.uint8)
    s = to_bf16_bits(uniform(stream(cfg_id, 2, seed), (E, N, K // 128), scale_lo, scale_hi))
    a = to_bf16_bits(normal(stream(cfg_id, 3, seed), (M, K)))
    out = dict(A=a, codes=codes, w_canon=pack_nibbles(codes), s_canon=s, E=E, N=N, K=K, M=M)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 4, seed), (E, N)))
    return out


def w4a16_zp_problem(M, N, K, *, E=1, cfg_id=0, seed=BASE_SEED, scale_lo=0.005,
                     scale_hi=0.02, bias=False):
    """Group-128 asymmetric INT4 weights: unsigned codes uniform in [0, 15], a BF16 scale
    U[scale_lo, scale_hi] and a zero point uniform in [0, 15] per group, packed as
    uint32 group words (scale bits 0-15, zero point bits 16-23); BF16 N(0,1) activations."""
    q = uniform_int(stream(cfg_id, 30, seed), (E, N, K), 0, 15).astype(np.uint8)
    s = to_bf16_bits(uniform(stream(cfg_id, 31, seed), (E, N, K // 128), scale_lo, scale_hi))
    z = uniform_int(stream(cfg_id, 32, seed), (E, N, K // 128), 0, 15).astype(np.uint32)
    a = to_bf16_bits(normal(stream(cfg_id, 33, seed), (M, K)))
    w = np.ascontiguousarray(pack_nibbles(q)).view("<u4").astype(np.uint32, copy=False)
    sz = (s.astype(np.uint32) | (z << np.uint32(16))).astype(np.uint32)
    out = dict(A=a, w_canon=w, s_canon=sz, E=E, N=N, K=K, M=M, bits=4, zp=True)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 34, seed), (E, N)))
    return out


def fp8w_problem(M, N, K, *, E=1, cfg_id=0, seed=BASE_SEED, scale_lo=0.005, scale_hi=0.02,
                 bias=False):
    """FP8-weight WnA16: E4M3 codes of N(0,1) samples times 2^u, u uniform in [-10, 6] per
    element (clipped to +-448), so the codes span every E4M3 exponent, subnormals included;
    a BF16 scale U[scale_lo, scale_hi] per group of 128 along K; BF16 N(0,1) activations."""
    mag = np.exp2(uniform(stream(cfg_id, 44, seed), (E * N, K), -10.0, 6.0))
    w = to_e4m3_codes(normal(stream(cfg_id, 40, seed), (E * N, K)) * mag).reshape(E, N, K)
    s = to_bf16_bits(uniform(stream(cfg_id, 41, seed), (E, N, K // 128), scale_lo, scale_hi))
    a = to_bf16_bits(normal(stream(cfg_id, 42, seed), (M, K)))
    out = dict(A=a, w_canon=w, s_canon=s, E=E, N=N, K=K, M=M, fp8=True)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 43, seed), (E, N)))
    return out


def w4a8_problem(M, N, K, *, E=1, cfg_id=1, seed=BASE_SEED, sf_lo=118, sf_hi=126,
                 bias=False):
    """MXFP4 weights (uniform over the 16 E2M1 codes) and MXFP8 activations
    (E4M3 codes of N(0,1) samples), both with group-32 E8M0 scales uniform in
    [sf_lo, sf_hi]."""
    nib = random_bytes(stream(cfg_id, 11, seed), E * N * K // 2)
    w_canon = nib.reshape(E, N, K // 2)
    w_sf = uniform_int(stream(cfg_id, 12, seed), (E, N, K // 32), sf_lo, sf_hi).astype(np.uint8)
    a = to_e4m3_codes(normal(stream(cfg_id, 13, seed), (M, K)))
    a_sf = uniform_int(stream(cfg_id, 14, seed), (M, K // 32), sf_lo, sf_hi).astype(np.uint8)
    out = dict(A=a, A_sf=a_sf, w_canon=w_canon, s_canon=w_sf, E=E, N=N, K=K, M=M)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 15, seed), (E, N)))
    return out


def w8a8_problem(M, N, K, *, E=1, cfg_id=1, seed=BASE_SEED, sf_lo=118, sf_hi=126,
                 bias=False):
    """MXFP8 weights and activations: E4M3 codes of N(0,1) samples with group-32 E8M0
    scales uniform in [sf_lo, sf_hi]."""
    w = to_e4m3_codes(normal(stream(cfg_id, 16, seed), (E * N, K))).reshape(E, N, K)
    w_sf = uniform_int(stream(cfg_id, 17, seed), (E, N, K // 32), sf_lo, sf_hi).astype(np.uint8)
    a = to_e4m3_codes(normal(stream(cfg_id, 13, seed), (M, K)))
    a_sf = uniform_int(stream(cfg_id, 14, seed), (M, K // 32), sf_lo, sf_hi).astype(np.uint8)
    out = dict(A=a, A_sf=a_sf, w_canon=w, s_canon=w_sf, E=E, N=N, K=K, M=M)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 15, seed), (E, N)))
    return out


def w4a4_problem(M, N, K, *, E=1, cfg_id=1, seed=BASE_SEED, sf_lo=0x28, sf_hi=0x48,
                 bias=False):
    """NVFP4 weights and activations: E2M1 codes uniform over the 16 codes (random
    nibbles, even k in the low nibble) with one unsigned E4M3 scale per 16 along K, its code
    uniform in [sf_lo, sf_hi] (0x28..0x48 = 0.125 .. 4.0)."""
    w = random_bytes(stream(cfg_id, 23, seed), E * N * K // 2).reshape(E, N, K // 2)
    w_sf = uniform_int(stream(cfg_id, 24, seed), (E, N, K // 16), sf_lo, sf_hi).astype(np.uint8)
    a = random_bytes(stream(cfg_id, 25, seed), M * K // 2).reshape(M, K // 2)
    a_sf = uniform_int(stream(cfg_id, 26, seed), (M, K // 16), sf_lo, sf_hi).astype(np.uint8)
    out = dict(A=a, A_sf=a_sf, w_canon=w, s_canon=w_sf, E=E, N=N, K=K, M=M)
    if bias:
        out["bias"] = to_bf16_bits(normal(stream(cfg_id, 27, seed), (E, N)))
    return out


def unpack_nibbles_layout(w_canon: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles` (a layout helper for test inputs, no decoding)."""
    lo = w_canon & 0xF
    hi = w_canon >> 4
    out = np.empty((*w_canon.shape[:-1], w_canon.shape[-1] * 2), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def router_logits(T, E, *, cfg_id=3, seed=BASE_SEED, bias_std=1.5):
    """Router logits N(0,1) plus a per-expert bias N(0, bias_std), float32 [T][E]."""
    b = normal(stream(cfg_id, 21, seed), (E,), bias_std)
    x = normal(stream(cfg_id, 22, seed), (T, E))
    return (x + b[None, :]).astype(np.float32)


__all__ = [
    "BASE_SEED", "Stream", "stream", "uniform_int", "uniform", "normal", "random_bytes",
    "to_bf16_bits", "to_e4m3_codes", "pack_int4", "pack_int3", "pack_int2", "pack_int1",
    "pack_nibbles", "unpack_nibbles_layout", "w4a16_problem", "w4a16_zp_problem",
    "fp8w_problem", "fp4w_problem", "w4a8_problem",
    "w8a8_problem",
    "w4a4_problem",
    "router_logits",
]
