// act.cu - the activation-side steps of a quantized MoE layer around the GEMMs:
//   - BF16 -> MXFP8 (E4M3 codes + E8M0 group-32 scales) activation quantizer, the input
//     format of the W4A8 GEMM (spke.com Humming announcement, "W8A8 / W4A8 / W4A4": MXFP8
//     activations);
//   - SiLU * mul over the fused gate+up projection output;
//   - the top-k weighted combine of each token's expert rows.
// All three are streaming, HBM-bound passes: one thread moves 16 bytes of BF16 at a time,
// in registers, with no shared memory.
//
// Quantizer (OCP Microscaling v1.0 conversion): per group of 32 values the shared exponent
// is X = floor(log2(max |v|)) - 8 (8 = exponent of the largest E4M3 power of two), clamped
// to [-127, 127]; elements are v * 2^-X rounded to nearest-even E4M3 and saturated to
// +-448 by the hardware conversion (cvt.rn.satfinite); an all-zero group gets scale byte 0.
// The exponent comes from the integer bits of max |v| (exact), and v * 2^-X is exact in
// FP32, so every rounding decision is the single E4M3 rounding.
#include <cuda_bf16.h>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// two FP32 values -> two E4M3 codes, x0 in the low byte (round to nearest even, saturate)
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x1), "f"(x0));
  return d;
}

// One thread = 8 consecutive BF16 values; 4 threads = one group of 32 (K % 32 == 0, so a
// group never straddles rows and its four threads sit in the same warp).
__global__ void quantize_mxfp8_kernel(const uint4* __restrict__ A, int64_t n8, uint2* __restrict__ Q,
                                      uint8_t* __restrict__ SF, int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // every thread of a warp runs the same number of iterations (n8 % 4 == 0, stride % 32 == 0)
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i - (threadIdx.x & 31) < n8;
       i += stride) {
    const bool live = i < n8;
    uint4 v = live ? __ldg(A + i) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t amax = 0;  // max |v| as BF16 bits (finite values order like their bit patterns)
    bool finite = true;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = w[j] & 0x7FFFu, hi = (w[j] >> 16) & 0x7FFFu;
      finite = finite && lo < 0x7F80u && hi < 0x7F80u;
      amax = max(amax, max(lo, hi));
    }
    if (!finite) set_error(err, QW_ERR_VALUE);
    amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    int X = -127;
    if (amax != 0) {
      const int ef = (int)(amax >> 7), mant = (int)(amax & 0x7F);
      const int fl = ef > 0 ? ef - 127 : -133 + (31 - __clz(mant));  // floor(log2 max|v|)
      X = max(-127, min(127, fl - 8));
    }
    const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, X in [-127, 126]
    uint2 q;
    q.x = e4m3x2(bf16_lo(w[0]) * inv, bf16_hi(w[0]) * inv) |
          (e4m3x2(bf16_lo(w[1]) * inv, bf16_hi(w[1]) * inv) << 16);
    q.y = e4m3x2(bf16_lo(w[2]) * inv, bf16_hi(w[2]) * inv) |
          (e4m3x2(bf16_lo(w[3]) * inv, bf16_hi(w[3]) * inv) << 16);
    if (live) {
      Q[i] = q;
      if ((i & 3) == 0) SF[i >> 2] = (uint8_t)(X + 127);
    }
  }
}

// One thread = 8 outputs of one row: y = silu(g) * u, g the first half, u the second half.
__global__ void silu_mul_kernel(const uint16_t* __restrict__ GU, int64_t rows, int32_t I,
                                uint16_t* __restrict__ Y) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int32_t per_row = I / 8;
  const int64_t total = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row;
    const int32_t c = (int32_t)(i - r * per_row) * 8;
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(GU + r * 2 * I + c));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(GU + r * 2 * I + I + c));
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float g0 = bf16_lo(gw[j]), g1 = bf16_hi(gw[j]);
      const float y0 = g0 / (1.f + expf(-g0)) * bf16_lo(uw[j]);
      const float y1 = g1 / (1.f + expf(-g1)) * bf16_hi(uw[j]);
      __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
      o[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(Y + r * I + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// position of every pair in the sorted order: inv[sorted_pairs[i]] = i
__global__ void invert_pairs_kernel(const int32_t* __restrict__ sp, int64_t P,
                                    int32_t* __restrict__ inv, int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < P;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t pair = __ldg(sp + i);
    if (pair < 0 || pair >= P) {
      set_error(err, QW_ERR_INVALID_ARG);
      continue;
    }
    inv[pair] = (int32_t)i;
  }
}

// out[t][n] = sum_j w[t][j] Y[inv[t k + j]][n], w = softmax of token t's k selected logits.
// One CTA per token; a thread owns 8 consecutive columns at a time.  With `inv` null (small
// batches) the CTA finds its k rows itself by scanning the sorted pair list, which saves
// the inversion launch.
__global__ void combine_kernel(const uint16_t* __restrict__ Y, const int32_t* __restrict__ inv,
                               const int32_t* __restrict__ sp, const int32_t* __restrict__ ids,
                               const float* __restrict__ logits, int32_t E, int32_t k, int32_t N,
                               int64_t P, uint16_t* __restrict__ out, int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  __shared__ float w[32];
  __shared__ int32_t row[32];
  if (!inv) {
    if (threadIdx.x < 32) row[threadIdx.x] = -1;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < P; i += blockDim.x) {
      const int32_t pair = __ldg(sp + i);
      if (pair < 0 || pair >= P) {
        set_error(err, QW_ERR_INVALID_ARG);
        continue;
      }
      if (pair / k == t) row[pair - t * k] = (int32_t)i;
    }
    __syncthreads();
  }
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    float l = -INFINITY;
    int32_t r = 0;
    if (j < k) {
      const int32_t e = __ldg(ids + t * k + j);
      const bool ok_e = e >= 0 && e < E;
      if (!ok_e) set_error(err, QW_ERR_INVALID_ARG);
      l = ok_e ? __ldg(logits + t * E + e) : 0.f;
      r = inv ? __ldg(inv + t * k + j) : row[j];
      if (r < 0 || r >= P) {
        set_error(err, QW_ERR_INVALID_ARG);
        r = 0;
      }
    }
    float m = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float ex = j < k ? expf(l - m) : 0.f;
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    w[j] = ex / s;
    row[j] = r;
  }
  __syncthreads();
  for (int32_t c = threadIdx.x * 8; c < N; c += blockDim.x * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(Y + (int64_t)row[j] * N + c));
      const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
      const float wj = w[j];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = fmaf(wj, bf16_lo(yw[q]), acc[2 * q]);
        acc[2 * q + 1] = fmaf(wj, bf16_hi(yw[q]), acc[2 * q + 1]);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(out + t * N + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// pairs up to which the combine scans the sorted pair list per token instead of inverting it
constexpr int64_t kCombineScanPairs = 2048;

unsigned stream_grid(int64_t work_items, int threads) {
  const int64_t want = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

qw_status launch_quantize_mxfp8(const void* A, int64_t rows, int32_t K, void* Q, void* SF,
                                int32_t* err, cudaStream_t st) {
  const int64_t n8 = rows * (int64_t)(K / 8);
  (void)launch_pdl(quantize_mxfp8_kernel, dim3(stream_grid(n8, 256)), dim3(256), 0, st, static_cast<const uint4*>(A), n8, static_cast<uint2*>(Q), static_cast<uint8_t*>(SF), err);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_silu_mul(const void* GU, int64_t rows, int32_t I, void* Y, cudaStream_t st) {
  (void)launch_pdl(silu_mul_kernel, dim3(stream_grid(rows * (int64_t)(I / 8), 256)), dim3(256), 0, st, static_cast<const uint16_t*>(GU), rows, I, static_cast<uint16_t*>(Y));
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_moe_combine(const void* Y, const int32_t* sorted_pairs, const int32_t* topk_ids,
                             const float* logits, int32_t T, int32_t E, int32_t topk, int32_t N,
                             void* out, int32_t* inv, int32_t* err, cudaStream_t st) {
  const int64_t P = (int64_t)T * topk;
  // decode-sized batches: each token's CTA scans the pair list itself (no inversion launch)
  const bool scan = P <= kCombineScanPairs;
  if (!scan) {
    (void)launch_pdl(invert_pairs_kernel, dim3(stream_grid(P, 256)), dim3(256), 0, st, sorted_pairs, P, inv, err);
    if (cudaGetLastError() != cudaSuccess) return QW_ERR_CUDA;
  }
  int threads = (N / 8 + 31) / 32 * 32;
  if (threads > 512) threads = 512;
  if (threads < 32) threads = 32;
  (void)launch_pdl(combine_kernel, dim3((unsigned)T), dim3(threads), 0, st, static_cast<const uint16_t*>(Y),
                                                   scan ? nullptr : inv, sorted_pairs, topk_ids,
                                                   logits, E, topk, N, P,
                                                   static_cast<uint16_t*>(out), err);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
