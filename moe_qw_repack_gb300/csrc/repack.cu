// repack.cu - preprocessing: validate, pad and repack canonical weights and scales
// into the layouts the GEMM kernels stream (spke.com Humming announcement, section
// "ワークロードごとのチューニングとJITコンパイル": preprocessing validates parameters,
// pads dimensions and repacks tensors for the target kernel), plus the exact inverse.
//
// Integer weights are rewritten as excess codes (q + 2^(b-1)): the zero-exponent
// value set of section "量子化サポート" shifted so that the code drops directly into
// a BF16 mantissa next to a fixed exponent.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

// ----------------------------------------------------------------------------- INT4
// Canonical nibble of (row n, column k): two's complement, word k/8, bits 4*(k%8).
__device__ __forceinline__ uint32_t int4_canon_nib(const uint32_t* wc, int32_t K, int64_t n,
                                                   int32_t k) {
  return (wc[n * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xFu;
}

// Mapping of one packed INT4 word (lane l, step s of a 16 x 128 block) to the weights it
// holds: nibble i feeds register r = i & 3 of the m16n8k16 A fragment, half h = i >> 2;
// row = g + 8 * (r & 1), k = 16s + 4t + 2 * (r >> 1) + h, g = l / 4, t = l % 4.
// Word s thus holds rows g and g + 8 at the four k's 16s + 4t .. 16s + 4t + 3.  The
// synchronous MMA does not care which real k sits in which of its k slots as long as the
// B operand agrees (lane t's activations for step s are 8 contiguous bytes), and the same
// four registers are exactly what tcgen05.st.16x256b puts at TMEM lanes g, g + 8 and
// columns 8s + 2t, 8s + 2t + 1 - the tensor-core path stores decoded words as they are.
__device__ __forceinline__ void int4_nib_pos(int l, int s, int i, int& row, int& k) {
  const int g = l >> 2, t = l & 3, r = i & 3, h = i >> 2;
  row = g + 8 * (r & 1);
  k = 16 * s + 4 * t + 2 * (r >> 1) + h;
}

// `unsigned_codes`: the asymmetric format's q in [0, 15] is packed as it is (its zero point
// plays the excess); otherwise the symmetric q becomes the excess-8 code q + 8.
__global__ void repack_int4_kernel(const uint32_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K, int32_t* err,
                                   bool unsigned_codes) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 256;
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    int64_t rem = idx % per_expert;
    const int64_t blk = rem / 256;  // G * (N_pad/16) + nb
    const int w = (int)(rem % 256);
    const int lane = w / 8, s = w % 8;
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const uint32_t* wce = wc + e * (int64_t)N * (K / 8);
    uint32_t out = 0;
    for (int i = 0; i < 8; ++i) {
      int row, k;
      int4_nib_pos(lane, s, i, row, k);
      const int64_t n = (int64_t)nb * 16 + row;
      uint32_t nib = 0;  // q = 0 for padding rows
      if (n < N) {
        nib = int4_canon_nib(wce, K, n, G * 128 + k);
        if (!unsigned_codes && nib == 8u) {  // -8 is outside the symmetric range
          set_error(err, QW_ERR_VALUE);
          nib = 0;
        }
      } else if (!unsigned_codes) {
        nib = 0;
      }
      out |= ((unsigned_codes ? nib : (nib ^ 8u)) & 0xFu) << (4 * i);
    }
    wp[idx] = out;
  }
}

__global__ void unpack_int4_kernel(const uint32_t* __restrict__ wp, uint32_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                   bool unsigned_codes) {
  // one thread per canonical word (8 consecutive k of one row)
  const int64_t per_expert = (int64_t)N * (K / 8);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 8);
    const int k0 = (int)(rem % (K / 8)) * 8;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 256;
    uint32_t out = 0;
    for (int j = 0; j < 8; ++j) {
      const int k = k0 + j;
      const int G = k / 128, kk = k % 128;
      const int nb = (int)(n / 16), row = (int)(n % 16);
      // invert int4_nib_pos: row = g + 8(r&1), kk = 16s + 4t + 2(r>>1) + h
      const int g = row & 7, r0 = row >> 3, t = (kk >> 2) & 3, s = kk >> 4;
      const int r1 = (kk >> 1) & 1, h = kk & 1;
      const int lane = g * 4 + t, i = (r0 | (r1 << 1)) + 4 * h;
      const uint32_t word = wpe[((int64_t)G * (N_pad / 16) + nb) * 256 + lane * 8 + s];
      const uint32_t code = (word >> (4 * i)) & 0xFu;
      out |= ((unsigned_codes ? code : (code ^ 8u)) & 0xFu) << (4 * j);
    }
    wc[idx] = out;
  }
}

// ----------------------------------------------------------------------------- INT3
__device__ __forceinline__ int32_t int3_canon(const uint32_t* wc, int32_t K, int64_t n, int32_t k) {
  const uint32_t* blk = wc + (n * (K / 32) + k / 32) * 3;
  const int bit = 3 * (k % 32);
  const int w = bit / 32, off = bit % 32;
  uint32_t v = blk[w] >> off;
  if (off > 29) v |= blk[w + 1] << (32 - off);
  v &= 7u;
  return (v >= 4u) ? (int32_t)v - 8 : (int32_t)v;
}

// Packed INT3 of lane l, step s, register r, half h (same (row, k) as the INT4 words:
// row g + 8 (r & 1), k 16s + 4t + 2 (r >> 1) + h), u = q + 4 in three bits.  The lane's six
// words (four in the first 512 bytes of the block, two in the last 256) each hold five
// registers: register j = 4s + r < 30 is field j % 5 of word j / 5, u at bits
// 3 (j % 5) + 16 h, so that one shift and one logic op give a BF16 pair, as for INT4.
// The two registers left over use the spare bit 15 + 16 h of each word: bit i of u is in
// word i (j = 30) or word 3 + i (j = 31).
__global__ void repack_int3_kernel(const uint32_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K, int32_t* err) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 32;  // (block, lane)
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t blk = rem / 32;
    const int lane = (int)(rem % 32);
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const uint32_t* wce = wc + e * (int64_t)N * (K / 32) * 3;
    uint32_t W[6] = {0, 0, 0, 0, 0, 0};
    const int g = lane >> 2, t = lane & 3;
    for (int s = 0; s < 8; ++s)
      for (int r = 0; r < 4; ++r)
        for (int h = 0; h < 2; ++h) {
          const int row = g + 8 * (r & 1);
          const int k = G * 128 + 16 * s + 4 * t + 2 * (r >> 1) + h;
          const int64_t n = (int64_t)nb * 16 + row;
          int32_t q = 0;
          if (n < N) {
            q = int3_canon(wce, K, n, k);
            if (q == -4) {
              set_error(err, QW_ERR_VALUE);
              q = 0;
            }
          }
          const uint32_t u = (uint32_t)(q + 4);
          const int j = 4 * s + r;
          if (j < 30) {
            W[j / 5] |= u << (3 * (j % 5) + 16 * h);
          } else {
            const int b = j == 30 ? 0 : 3;
            for (int i = 0; i < 3; ++i) W[b + i] |= ((u >> i) & 1u) << (15 + 16 * h);
          }
        }
    uint32_t* out = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 192 + blk * 192;
    for (int i = 0; i < 4; ++i) out[lane * 4 + i] = W[i];
    for (int i = 0; i < 2; ++i) out[128 + lane * 2 + i] = W[4 + i];
  }
}

__global__ void unpack_int3_kernel(const uint32_t* __restrict__ wp, uint32_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  // one thread per canonical 32-element block (3 words)
  const int64_t per_expert = (int64_t)N * (K / 32);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 32);
    const int k0 = (int)(rem % (K / 32)) * 32;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 192;
    uint32_t w3[3] = {0, 0, 0};
    for (int j = 0; j < 32; ++j) {
      const int k = k0 + j;
      const int G = k / 128, kk = k % 128;
      const int nb = (int)(n / 16), row = (int)(n % 16);
      const int t = (kk >> 2) & 3, s = kk >> 4, h = kk & 1;
      const int g = row & 7, r = (row >> 3) | (((kk >> 1) & 1) << 1);
      const int lane = g * 4 + t;
      const uint32_t* blk = wpe + ((int64_t)G * (N_pad / 16) + nb) * 192;
      const int jr = 4 * s + r;  // the lane's register; its words as in repack_int3_kernel
      uint32_t u = 0;
      if (jr < 30) {
        const int wi = jr / 5;
        const uint32_t x = wi < 4 ? blk[lane * 4 + wi] : blk[128 + lane * 2 + (wi - 4)];
        u = (x >> (3 * (jr % 5) + 16 * h)) & 7u;
      } else {
        const int b = jr == 30 ? 0 : 3;
        for (int i = 0; i < 3; ++i) {
          const int wi = b + i;
          const uint32_t x = wi < 4 ? blk[lane * 4 + wi] : blk[128 + lane * 2 + (wi - 4)];
          u |= ((x >> (15 + 16 * h)) & 1u) << i;
        }
      }
      const uint32_t code = (uint32_t)((int32_t)u - 4) & 7u;  // back to two's complement
      const int bit = 3 * j;
      w3[bit / 32] |= code << (bit % 32);
      if (bit % 32 > 29) w3[bit / 32 + 1] |= code >> (32 - bit % 32);
    }
    uint32_t* o = wc + idx * 3;
    o[0] = w3[0];
    o[1] = w3[1];
    o[2] = w3[2];
  }
}

// ----------------------------------------------------------------------------- INT2
// Packed INT2 of lane l, step s, register r, half h (the INT4 (row, k) assignment): word s/2
// of the lane's four keeps u = q + 2 at bits 2 * (4 * (s % 2) + r) + 16 h.
__global__ void repack_int2_kernel(const uint32_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K, int32_t* err) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 32;  // (block, lane)
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t blk = rem / 32;
    const int lane = (int)(rem % 32);
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const uint32_t* wce = wc + e * (int64_t)N * (K / 16);
    uint32_t lo[4] = {0, 0, 0, 0};
    const int g = lane >> 2, t = lane & 3;
    for (int s = 0; s < 8; ++s)
      for (int r = 0; r < 4; ++r)
        for (int h = 0; h < 2; ++h) {
          const int row = g + 8 * (r & 1);
          const int k = G * 128 + 16 * s + 4 * t + 2 * (r >> 1) + h;
          const int64_t n = (int64_t)nb * 16 + row;
          int32_t q = 0;
          if (n < N) {
            const uint32_t f = (wce[n * (K / 16) + k / 16] >> (2 * (k % 16))) & 3u;
            q = f >= 2u ? (int32_t)f - 4 : (int32_t)f;
            if (q == -2) {  // outside the symmetric range
              set_error(err, QW_ERR_VALUE);
              q = 0;
            }
          }
          lo[s / 2] |= (uint32_t)(q + 2) << (2 * (4 * (s % 2) + r) + 16 * h);
        }
    uint32_t* out = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 128 + blk * 128;
    for (int i = 0; i < 4; ++i) out[lane * 4 + i] = lo[i];
  }
}

__global__ void unpack_int2_kernel(const uint32_t* __restrict__ wp, uint32_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  // one thread per canonical word (16 consecutive k of one row)
  const int64_t per_expert = (int64_t)N * (K / 16);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 16);
    const int k0 = (int)(rem % (K / 16)) * 16;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 128;
    uint32_t out = 0;
    for (int j = 0; j < 16; ++j) {
      const int k = k0 + j;
      const int G = k / 128, kk = k % 128;
      const int nb = (int)(n / 16), row = (int)(n % 16);
      const int t = (kk >> 2) & 3, s = kk >> 4, h = kk & 1;
      const int g = row & 7, r = (row >> 3) | (((kk >> 1) & 1) << 1);
      const uint32_t L = wpe[((int64_t)G * (N_pad / 16) + nb) * 128 + (g * 4 + t) * 4 + s / 2];
      const uint32_t u = (L >> (2 * (4 * (s % 2) + r) + 16 * h)) & 3u;
      out |= ((u - 2u) & 3u) << (2 * j);  // back to two's complement
    }
    wc[idx] = out;
  }
}

// ----------------------------------------------------------------------------- FP8 weights
// Packed FP8 (E4M3) weights: byte b of word u = 2s + j of lane l = 4g + t holds the code of
// row g + 8 (b >> 1), k = 16s + 4t + 2j + (b & 1) - the INT4 (row, k) assignment with one
// byte per weight, so each 16-bit half decodes to one BF16 pair of the m16n8k16 A fragment
// (and of the 16-lane TMEM store).  NaN codes (0x7F, 0xFF) are value errors, packed as 0.
__global__ void repack_fp8w_kernel(const uint8_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K, int32_t* err) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 512;  // words
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t blk = rem / 512;
    const int w = (int)(rem % 512);
    const int lane = w >> 4, u = w & 15;
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const int g = lane >> 2, t = lane & 3, s = u >> 1, j = u & 1;
    const uint8_t* wce = wc + e * (int64_t)N * K;
    uint32_t out = 0;
    for (int b = 0; b < 4; ++b) {
      const int64_t n = (int64_t)nb * 16 + g + 8 * (b >> 1);
      const int k = G * 128 + 16 * s + 4 * t + 2 * j + (b & 1);
      uint32_t c = 0;  // padding rows: zero
      if (n < N) {
        c = wce[n * K + k];
        if ((c & 0x7Fu) == 0x7Fu) {
          set_error(err, QW_ERR_VALUE);
          c = 0;
        }
      }
      out |= c << (8 * b);
    }
    wp[idx] = out;
  }
}

__global__ void unpack_fp8w_kernel(const uint32_t* __restrict__ wp, uint32_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  // one thread per 4 consecutive canonical codes of one row (k0 % 4 == 0)
  const int64_t per_expert = (int64_t)N * (K / 4);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 4);
    const int k0 = (int)(rem % (K / 4)) * 4;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 512;
    const int G = k0 / 128, kk = k0 % 128;
    const int nb = (int)(n / 16), row = (int)(n % 16);
    const int g = row & 7, hi = row >> 3, t = (kk >> 2) & 3, s = kk >> 4;
    const uint32_t* lw = wpe + ((int64_t)G * (N_pad / 16) + nb) * 512 + (g * 4 + t) * 16 + 2 * s;
    uint32_t out = 0;
    for (int i = 0; i < 4; ++i) {  // k0 + i: word 2s + (i >> 1), byte 2 hi + (i & 1)
      const uint32_t c = (lw[i >> 1] >> (8 * (2 * hi + (i & 1)))) & 0xFFu;
      out |= c << (8 * i);
    }
    wc[idx] = out;
  }
}

// ----------------------------------------------------------------------------- INT1
// Packed INT1 (sign codes, bit b = weight 2b - 1): 256-byte blocks of 32 lanes x 2 words.
// Register r of MMA step s (rows g + 8 (r & 1), k = 16s + 4t + 2 (r >> 1) + h) keeps its two
// bits at bit 4 (s % 4) + r + 16h of word s / 4: one shift moves both to the sign positions
// 15 and 31 of a BF16 (or FP16) pair.
__global__ void repack_int1_kernel(const uint32_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 64;  // words
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t blk = rem / 64;
    const int w = (int)(rem % 64);
    const int lane = w >> 1, half = w & 1;  // word `half` holds steps 4 half .. 4 half + 3
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const int g = lane >> 2, t = lane & 3;
    const uint32_t* wce = wc + e * (int64_t)N * (K / 32);
    uint32_t out = 0;
    for (int s4 = 0; s4 < 4; ++s4)
      for (int r = 0; r < 4; ++r)
        for (int h = 0; h < 2; ++h) {
          const int s = 4 * half + s4;
          const int64_t n = (int64_t)nb * 16 + g + 8 * (r & 1);
          const int k = G * 128 + 16 * s + 4 * t + 2 * (r >> 1) + h;
          // padding rows: bit 0 (weight -1 times a zero scale)
          const uint32_t b = n < N ? (wce[n * (K / 32) + k / 32] >> (k % 32)) & 1u : 0u;
          out |= b << (4 * s4 + r + 16 * h);
        }
    wp[idx] = out;
  }
}

__global__ void unpack_int1_kernel(const uint32_t* __restrict__ wp, uint32_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  // one thread per canonical word (32 consecutive k of one row)
  const int64_t per_expert = (int64_t)N * (K / 32);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 32);
    const int k0 = (int)(rem % (K / 32)) * 32;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 64;
    uint32_t out = 0;
    for (int j = 0; j < 32; ++j) {
      const int k = k0 + j;
      const int G = k / 128, kk = k % 128;
      const int nb = (int)(n / 16), row = (int)(n % 16);
      const int g = row & 7, t = (kk >> 2) & 3, s = kk >> 4, h = kk & 1;
      const int r = (row >> 3) | (((kk >> 1) & 1) << 1);
      const uint32_t W = wpe[((int64_t)G * (N_pad / 16) + nb) * 64 + (g * 4 + t) * 2 + s / 4];
      out |= ((W >> (4 * (s % 4) + r + 16 * h)) & 1u) << j;
    }
    wc[idx] = out;
  }
}

// ----------------------------------------------------------------------------- FP4 weights
// Packed FP4 (E2M1) weights: the INT4 block of 1 KiB (32 lanes x 8 words, word s = MMA step
// s), but byte r of a word holds register r - the codes at k = 16s + 4t + 2 (r >> 1) and
// k + 1 of row g + 8 (r & 1), the first in the low nibble - so one hardware conversion
// (cvt.rn.f16x2.e2m1x2) turns a byte into the register's FP16 pair.  Every code is valid.
__global__ void repack_fp4w_kernel(const uint8_t* __restrict__ wc, uint32_t* __restrict__ wp,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  const int64_t per_expert = (int64_t)(K / 128) * (N_pad / 16) * 256;  // words
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t blk = rem / 256;
    const int w = (int)(rem % 256);
    const int lane = w / 8, s = w % 8;
    const int G = (int)(blk / (N_pad / 16));
    const int nb = (int)(blk % (N_pad / 16));
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* wce = wc + e * (int64_t)N * (K / 2);
    uint32_t out = 0;
    for (int r = 0; r < 4; ++r) {
      const int64_t n = (int64_t)nb * 16 + g + 8 * (r & 1);
      const int k = G * 128 + 16 * s + 4 * t + 2 * (r >> 1);  // even: one canonical byte
      const uint32_t byte = n < N ? wce[n * (K / 2) + k / 2] : 0u;  // padding rows: 0
      out |= byte << (8 * r);
    }
    wp[idx] = out;
  }
}

__global__ void unpack_fp4w_kernel(const uint32_t* __restrict__ wp, uint8_t* __restrict__ wc,
                                   int32_t E, int32_t N, int32_t N_pad, int32_t K) {
  // one thread per canonical byte (k, k + 1 of one row, k even)
  const int64_t per_expert = (int64_t)N * (K / 2);
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t n = rem / (K / 2);
    const int k = (int)(rem % (K / 2)) * 2;
    const uint32_t* wpe = wp + e * (int64_t)(K / 128) * (N_pad / 16) * 256;
    const int G = k / 128, kk = k % 128;
    const int nb = (int)(n / 16), row = (int)(n % 16);
    const int g = row & 7, t = (kk >> 2) & 3, s = kk >> 4;
    const int r = (row >> 3) | (((kk >> 1) & 1) << 1);
    const uint32_t W = wpe[((int64_t)G * (N_pad / 16) + nb) * 256 + (g * 4 + t) * 8 + s];
    wc[idx] = (uint8_t)((W >> (8 * r)) & 0xFFu);
  }
}

// ----------------------------------------------------------------------------- second-level scales
// FP32 [E][N] <-> the packed plane [E][N_pad] (padding channels 0; a non-finite t is a value
// error, packed as 0).
__global__ void scale2_fill_kernel(float* __restrict__ tp, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    tp[i] = 1.0f;
}
__global__ void scale2_repack_kernel(const float* __restrict__ tc, float* __restrict__ tp,
                                     int32_t E, int32_t N, int32_t N_pad, int32_t* err) {
  const int64_t total = (int64_t)E * N_pad;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / N_pad;
    const int n = (int)(i % N_pad);
    float v = 0.f;
    if (n < N) {
      v = tc[e * N + n];
      if (!isfinite(v)) {
        set_error(err, QW_ERR_VALUE);
        v = 0.f;
      }
    }
    tp[i] = v;
  }
}
__global__ void scale2_unpack_kernel(const float* __restrict__ tp, float* __restrict__ tc,
                                     int32_t E, int32_t N, int32_t N_pad) {
  const int64_t total = (int64_t)E * N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x)
    tc[i] = tp[(i / N) * N_pad + i % N];
}

// ----------------------------------------------------------------------------- INT scales
// canonical [E][N][K/128] <-> packed [E][K/128][N_pad] (zero padded)
// Experts sit `estride` halfwords apart (the descriptor's scale stride: G * N_pad rounded up
// to 256 bytes).
__global__ void repack_int_scales_kernel(const uint16_t* __restrict__ sc, uint16_t* __restrict__ sp,
                                         int32_t E, int32_t N, int32_t N_pad, int32_t G,
                                         int64_t estride) {
  const int64_t total = (int64_t)E * G * N_pad;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)G * N_pad);
    const int64_t rem = idx % ((int64_t)G * N_pad);
    const int g = (int)(rem / N_pad);
    const int n = (int)(rem % N_pad);
    sp[e * estride + rem] = (n < N) ? sc[(e * N + n) * G + g] : (uint16_t)0;
  }
}
__global__ void unpack_int_scales_kernel(const uint16_t* __restrict__ sp, uint16_t* __restrict__ sc,
                                         int32_t E, int32_t N, int32_t N_pad, int32_t G,
                                         int64_t estride) {
  const int64_t total = (int64_t)E * N * G;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)N * G);
    const int64_t rem = idx % ((int64_t)N * G);
    const int n = (int)(rem / G);
    const int g = (int)(rem % G);
    sc[idx] = sp[e * estride + (int64_t)g * N_pad + n];
  }
}

// Asymmetric INT4 group words (BF16 scale | zero point << 16) -> the scale plane [G][N_pad]
// and the plane of BF16 128 + z (0x4300 | z, exact), per expert at `plane` halfwords apart.
__global__ void repack_zp_scales_kernel(const uint32_t* __restrict__ sc, uint16_t* __restrict__ sp,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t G,
                                        int64_t plane, int32_t* err) {
  const int64_t total = (int64_t)E * G * N_pad;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)G * N_pad);
    const int64_t rem = idx % ((int64_t)G * N_pad);
    const int g = (int)(rem / N_pad);
    const int n = (int)(rem % N_pad);
    uint32_t w = 0;
    if (n < N) {
      w = sc[(e * N + n) * G + g];
      if ((w >> 20) != 0) {  // zero point above 15 or stray high bits
        set_error(err, QW_ERR_VALUE);
        w &= 0xFFFFu;
      }
    }
    uint16_t* spe = sp + e * 2 * plane;
    spe[rem] = (uint16_t)(w & 0xFFFFu);
    spe[plane + rem] = (uint16_t)(0x4300u | (w >> 16));
  }
}
__global__ void unpack_zp_scales_kernel(const uint16_t* __restrict__ sp, uint32_t* __restrict__ sc,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t G,
                                        int64_t plane) {
  const int64_t total = (int64_t)E * N * G;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)N * G);
    const int64_t rem = idx % ((int64_t)N * G);
    const int n = (int)(rem / G);
    const int g = (int)(rem % G);
    const uint16_t* spe = sp + e * 2 * plane;
    const int64_t at = (int64_t)g * N_pad + n;
    sc[idx] = (uint32_t)spe[at] | ((uint32_t)(spe[plane + at] & 0xFFu) << 16);
  }
}

// ----------------------------------------------------------------------------- MXFP4
// codes: canonical [E][N][K/2] -> packed [E][N_pad][K_pad/2], 4 bytes per thread
__global__ void repack_mxfp4_codes_kernel(const uint8_t* __restrict__ wc, uint8_t* __restrict__ wp,
                                          int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                          int32_t K_pad) {
  const int64_t wpr = K_pad / 8;  // packed words per row
  const int64_t total = (int64_t)E * N_pad * wpr;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t er = idx / wpr;  // e * N_pad + n
    const int64_t e = er / N_pad;
    const int64_t n = er % N_pad;
    const int64_t b0 = (idx % wpr) * 4;  // byte within the packed row
    uint32_t v = 0;
    if (n < N) {
      const uint8_t* src = wc + (e * N + n) * (int64_t)(K / 2);
      for (int j = 0; j < 4; ++j)
        if (b0 + j < K / 2) v |= (uint32_t)src[b0 + j] << (8 * j);
    }
    reinterpret_cast<uint32_t*>(wp)[idx] = v;
  }
}
__global__ void unpack_mxfp4_codes_kernel(const uint8_t* __restrict__ wp, uint8_t* __restrict__ wc,
                                          int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                          int32_t K_pad) {
  const int64_t total = (int64_t)E * N * (K / 2);
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t er = idx / (K / 2);
    const int64_t e = er / N, n = er % N;
    const int64_t b = idx % (K / 2);
    wc[idx] = wp[(e * N_pad + n) * (int64_t)(K_pad / 2) + b];
  }
}

// ----------------------------------------------------------------------------- MXFP8
// codes: canonical [E][N][K] -> packed [E][N_pad][K_pad], 4 bytes per thread; E4M3 NaN
// codes (0x7F, 0xFF) are value errors and packed as 0
__global__ void repack_mxfp8_codes_kernel(const uint8_t* __restrict__ wc, uint8_t* __restrict__ wp,
                                          int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                          int32_t K_pad, int32_t* err) {
  const int64_t wpr = K_pad / 4;  // packed words per row
  const int64_t total = (int64_t)E * N_pad * wpr;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t er = idx / wpr;
    const int64_t e = er / N_pad;
    const int64_t n = er % N_pad;
    const int64_t b0 = (idx % wpr) * 4;
    uint32_t v = 0;
    if (n < N) {
      const uint8_t* src = wc + (e * N + n) * (int64_t)K;
      for (int j = 0; j < 4; ++j)
        if (b0 + j < K) {
          uint32_t c = src[b0 + j];
          if ((c & 0x7Fu) == 0x7Fu) {
            set_error(err, QW_ERR_VALUE);
            c = 0;
          }
          v |= c << (8 * j);
        }
    }
    reinterpret_cast<uint32_t*>(wp)[idx] = v;
  }
}
__global__ void unpack_mxfp8_codes_kernel(const uint8_t* __restrict__ wp, uint8_t* __restrict__ wc,
                                          int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                          int32_t K_pad) {
  const int64_t total = (int64_t)E * N * K;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t er = idx / K;
    const int64_t e = er / N, n = er % N;
    const int64_t b = idx % K;
    wc[idx] = wp[(e * N_pad + n) * (int64_t)K_pad + b];
  }
}

// Offset of scale (row r, group g) in the 128 x 4 chunked layout of one expert.
__device__ __forceinline__ int64_t sf_chunk_offset(int64_t r, int g, int K_pad) {
  return ((r / 128) * (K_pad / 128) + g / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4;
}

__global__ void repack_mx_scales_kernel(const uint8_t* __restrict__ sc, uint8_t* __restrict__ sp,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                        int32_t K_pad, int32_t* err) {
  const int Gp = K_pad / 32, Gc = K / 32;
  const int64_t per_expert = (int64_t)N_pad * Gp;
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t r = rem / Gp;
    const int g = (int)(rem % Gp);
    uint8_t v = 127;  // scale 1 for padding
    if (r < N && g < Gc) {
      v = sc[(e * N + r) * Gc + g];
      if (v == 0xFF) {
        set_error(err, QW_ERR_VALUE);
        v = 127;
      }
    }
    sp[e * per_expert + sf_chunk_offset(r, g, K_pad)] = v;
  }
}
__global__ void unpack_mx_scales_kernel(const uint8_t* __restrict__ sp, uint8_t* __restrict__ sc,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                        int32_t K_pad) {
  const int Gp = K_pad / 32, Gc = K / 32;
  const int64_t total = (int64_t)E * N * Gc;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)N * Gc);
    const int64_t rem = idx % ((int64_t)N * Gc);
    const int64_t r = rem / Gc;
    const int g = (int)(rem % Gc);
    sc[idx] = sp[e * (int64_t)N_pad * Gp + sf_chunk_offset(r, g, K_pad)];
  }
}

// ----------------------------------------------------------------------------- NVFP4
// Offset of scale (row r, group g of 16) in the 128-row x 16-group chunked layout of one
// expert: four 512-byte images per chunk, one per 64-k MMA, each in the image layout of
// the E8M0 chunks (lane r % 32, column (r % 128) / 32, byte g % 4).
__device__ __forceinline__ int64_t nv_sf_offset(int64_t r, int g, int K_pad) {
  return ((r / 128) * (K_pad / 256) + g / 16) * 2048 + ((g % 16) / 4) * 512 + (r % 32) * 16 +
         ((r % 128) / 32) * 4 + g % 4;
}

__global__ void repack_nv_scales_kernel(const uint8_t* __restrict__ sc, uint8_t* __restrict__ sp,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                        int32_t K_pad, int32_t* err) {
  const int Gp = K_pad / 16, Gc = K / 16;
  const int64_t per_expert = (int64_t)N_pad * Gp;
  const int64_t total = per_expert * E;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / per_expert;
    const int64_t rem = idx % per_expert;
    const int64_t r = rem / Gp;
    const int g = (int)(rem % Gp);
    uint8_t v = 0x38;  // scale 1 for padding
    if (r < N && g < Gc) {
      v = sc[(e * N + r) * Gc + g];
      if ((v & 0x80) || v == 0x7F) {  // unsigned scale: no sign, no NaN
        set_error(err, QW_ERR_VALUE);
        v = 0x38;
      }
    }
    sp[e * per_expert + nv_sf_offset(r, g, K_pad)] = v;
  }
}

__global__ void unpack_nv_scales_kernel(const uint8_t* __restrict__ sp, uint8_t* __restrict__ sc,
                                        int32_t E, int32_t N, int32_t N_pad, int32_t K,
                                        int32_t K_pad) {
  const int Gp = K_pad / 16, Gc = K / 16;
  const int64_t total = (int64_t)E * N * Gc;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = idx / ((int64_t)N * Gc);
    const int64_t rem = idx % ((int64_t)N * Gc);
    const int64_t r = rem / Gc;
    const int g = (int)(rem % Gc);
    sc[idx] = sp[e * (int64_t)N_pad * Gp + nv_sf_offset(r, g, K_pad)];
  }
}

// An empty kernel launched in plain stream order after the repack kernels.  The small-M
// GEMVs are programmatic dependents of the kernel before them and read packed weights and
// scales before their griddepcontrol.wait; with this kernel between, the kernel right
// before a GEMV that directly follows qw_repack is this one, which began only after every
// repack kernel had finished and its writes were visible.
__global__ void stream_order_kernel() {}

int grid_for(int64_t total, int threads) {
  int64_t b = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 32;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

qw_status launch_scale2_fill(float* t_packed, int64_t n, cudaStream_t st) {
  scale2_fill_kernel<<<grid_for(n, 256), 256, 0, st>>>(t_packed, n);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}
qw_status launch_scale2_repack(const float* t_canon, float* t_packed, int32_t E, int32_t N,
                               int32_t N_pad, int32_t* err, cudaStream_t st) {
  scale2_repack_kernel<<<grid_for((int64_t)E * N_pad, 256), 256, 0, st>>>(t_canon, t_packed, E,
                                                                          N, N_pad, err);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}
qw_status launch_scale2_unpack(const float* t_packed, float* t_canon, int32_t E, int32_t N,
                               int32_t N_pad, cudaStream_t st) {
  scale2_unpack_kernel<<<grid_for((int64_t)E * N, 256), 256, 0, st>>>(t_packed, t_canon, E, N,
                                                                       N_pad);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_repack(const qw_packed_desc& d, const void* w_canon, const void* s_canon,
                        void* w_packed, void* s_packed, int32_t* err, cudaStream_t st) {
  const int T = 256;
  switch (d.wfmt) {
    case QW_W_INT4_G128_BF16:
    case QW_W_UINT4ZP_G128_BF16: {
      const bool zp = d.wfmt == QW_W_UINT4ZP_G128_BF16;
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 256;
      repack_int4_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K, err, zp);
      if (zp) {
        const int64_t ts = (int64_t)d.E * (d.K / 128) * d.N_pad;
        repack_zp_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
            (const uint32_t*)s_canon, (uint16_t*)s_packed, d.E, d.N, d.N_pad, d.K / 128,
            (int64_t)(d.s_expert_stride / 4), err);
      }
      break;
    }
    case QW_W_INT2_G128_BF16: {
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 32;
      repack_int2_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K, err);
      break;
    }
    case QW_W_FP8E4M3_G128_BF16: {
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 512;
      repack_fp8w_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint8_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K, err);
      break;
    }
    case QW_W_INT1_G128_BF16: {
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 64;
      repack_int1_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_FP4E2M1_G128_BF16: {
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 256;
      repack_fp4w_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint8_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_INT3_G128_BF16: {
      const int64_t tw = (int64_t)d.E * (d.K / 128) * (d.N_pad / 16) * 32;
      repack_int3_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_canon,
                                                        (uint32_t*)w_packed, d.E, d.N, d.N_pad,
                                                        d.K, err);
      break;
    }
    case QW_W_MXFP4_G32:
    case QW_W_MXFP8_G32: {
      if (d.wfmt == QW_W_MXFP4_G32) {
        const int64_t tw = (int64_t)d.E * d.N_pad * (d.K_pad / 8);
        repack_mxfp4_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
            (const uint8_t*)w_canon, (uint8_t*)w_packed, d.E, d.N, d.N_pad, d.K, d.K_pad);
      } else {
        const int64_t tw = (int64_t)d.E * d.N_pad * (d.K_pad / 4);
        repack_mxfp8_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
            (const uint8_t*)w_canon, (uint8_t*)w_packed, d.E, d.N, d.N_pad, d.K, d.K_pad, err);
      }
      const int64_t ts = (int64_t)d.E * d.N_pad * (d.K_pad / 32);
      repack_mx_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
          (const uint8_t*)s_canon, (uint8_t*)s_packed, d.E, d.N, d.N_pad, d.K, d.K_pad, err);
      break;
    }
    case QW_W_NVFP4_G16: {
      const int64_t tw = (int64_t)d.E * d.N_pad * (d.K_pad / 8);
      repack_mxfp4_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
          (const uint8_t*)w_canon, (uint8_t*)w_packed, d.E, d.N, d.N_pad, d.K, d.K_pad);
      const int64_t ts = (int64_t)d.E * d.N_pad * (d.K_pad / 16);
      repack_nv_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
          (const uint8_t*)s_canon, (uint8_t*)s_packed, d.E, d.N, d.N_pad, d.K, d.K_pad, err);
      break;
    }
    default:
      return QW_ERR_UNSUPPORTED;
  }
  if (d.wfmt == QW_W_INT4_G128_BF16 || d.wfmt == QW_W_INT3_G128_BF16 ||
      d.wfmt == QW_W_INT2_G128_BF16 || d.wfmt == QW_W_FP8E4M3_G128_BF16 ||
      d.wfmt == QW_W_INT1_G128_BF16 || d.wfmt == QW_W_FP4E2M1_G128_BF16) {
    const int64_t ts = (int64_t)d.E * (d.K / 128) * d.N_pad;
    repack_int_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
        (const uint16_t*)s_canon, (uint16_t*)s_packed, d.E, d.N, d.N_pad, d.K / 128,
        (int64_t)(d.s_expert_stride / 2));
  }
  stream_order_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_unpack(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                        void* w_canon, void* s_canon, int32_t* err, cudaStream_t st) {
  (void)err;
  const int T = 256;
  switch (d.wfmt) {
    case QW_W_INT4_G128_BF16:
    case QW_W_UINT4ZP_G128_BF16: {
      const bool zp = d.wfmt == QW_W_UINT4ZP_G128_BF16;
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 8);
      unpack_int4_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint32_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K, zp);
      if (zp) {
        const int64_t ts = (int64_t)d.E * d.N * (d.K / 128);
        unpack_zp_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
            (const uint16_t*)s_packed, (uint32_t*)s_canon, d.E, d.N, d.N_pad, d.K / 128,
            (int64_t)(d.s_expert_stride / 4));
      }
      break;
    }
    case QW_W_INT2_G128_BF16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 16);
      unpack_int2_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint32_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_FP8E4M3_G128_BF16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 4);
      unpack_fp8w_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint32_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_INT1_G128_BF16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 32);
      unpack_int1_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint32_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_FP4E2M1_G128_BF16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 2);
      unpack_fp4w_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint8_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_INT3_G128_BF16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 32);
      unpack_int3_kernel<<<grid_for(tw, T), T, 0, st>>>((const uint32_t*)w_packed,
                                                        (uint32_t*)w_canon, d.E, d.N, d.N_pad,
                                                        d.K);
      break;
    }
    case QW_W_MXFP4_G32:
    case QW_W_MXFP8_G32: {
      if (d.wfmt == QW_W_MXFP4_G32) {
        const int64_t tw = (int64_t)d.E * d.N * (d.K / 2);
        unpack_mxfp4_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
            (const uint8_t*)w_packed, (uint8_t*)w_canon, d.E, d.N, d.N_pad, d.K, d.K_pad);
      } else {
        const int64_t tw = (int64_t)d.E * d.N * d.K;
        unpack_mxfp8_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
            (const uint8_t*)w_packed, (uint8_t*)w_canon, d.E, d.N, d.N_pad, d.K, d.K_pad);
      }
      const int64_t ts = (int64_t)d.E * d.N * (d.K / 32);
      unpack_mx_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
          (const uint8_t*)s_packed, (uint8_t*)s_canon, d.E, d.N, d.N_pad, d.K, d.K_pad);
      break;
    }
    case QW_W_NVFP4_G16: {
      const int64_t tw = (int64_t)d.E * d.N * (d.K / 2);
      unpack_mxfp4_codes_kernel<<<grid_for(tw, T), T, 0, st>>>(
          (const uint8_t*)w_packed, (uint8_t*)w_canon, d.E, d.N, d.N_pad, d.K, d.K_pad);
      const int64_t ts = (int64_t)d.E * d.N * (d.K / 16);
      unpack_nv_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
          (const uint8_t*)s_packed, (uint8_t*)s_canon, d.E, d.N, d.N_pad, d.K, d.K_pad);
      break;
    }
    default:
      return QW_ERR_UNSUPPORTED;
  }
  if (d.wfmt == QW_W_INT4_G128_BF16 || d.wfmt == QW_W_INT3_G128_BF16 ||
      d.wfmt == QW_W_INT2_G128_BF16 || d.wfmt == QW_W_FP8E4M3_G128_BF16 ||
      d.wfmt == QW_W_INT1_G128_BF16 || d.wfmt == QW_W_FP4E2M1_G128_BF16) {
    const int64_t ts = (int64_t)d.E * d.N * (d.K / 128);
    unpack_int_scales_kernel<<<grid_for(ts, T), T, 0, st>>>(
        (const uint16_t*)s_packed, (uint16_t*)s_canon, d.E, d.N, d.N_pad, d.K / 128,
        (int64_t)(d.s_expert_stride / 2));
  }
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
