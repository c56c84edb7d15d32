// diag.cu - reference points the kernels are measured against; no method arithmetic.
//  - A plain streaming read: the same bytes read with 16-byte loads by a full grid, folded
//    into one word per CTA (written out so the loads cannot be dropped).
//  - The tcgen05 MMA issue rate: one CTA per SM, one thread issuing back-to-back MMAs of the
//    kind and shape a tensor-core GEMM uses, on zero operands, timed from the first issue to
//    the completion seen through a commit.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kReadUnroll = 4;  // 16-byte loads in flight per thread

// `chained`: loads go before griddepcontrol.wait (only the one output word waits), as a
// programmatic dependent launch allows for a kernel that reads nothing its predecessor wrote.
template <bool CHAINED>
__global__ void __launch_bounds__(256) stream_read_kernel(const uint4* __restrict__ src, uint64_t n16,
                                                          uint32_t* __restrict__ sink) {
  if (CHAINED) pdl_launch_dependents();
  uint32_t acc = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
  for (; i + (kReadUnroll - 1) * stride < n16; i += kReadUnroll * stride) {
    uint4 v[kReadUnroll];
#pragma unroll
    for (int u = 0; u < kReadUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kReadUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  __shared__ uint32_t part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (CHAINED) pdl_wait();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a ^= part[w];
    sink[blockIdx.x] = a;
  }
}

// ---------------------------------------------------------------- tcgen05 MMA issue rate
constexpr int kProbeABox = 128 * 128;  // 128 rows x 128 bytes (one swizzle atom per row)
constexpr int kProbeBBox = 256 * 128;  // up to 256 rows x 128 bytes
constexpr int kProbeOperands = 2 * kProbeABox + 2 * kProbeBBox;
// one A and two B scale images (128 rows x 4 groups, 512 B each), or (wide copies) the same
// with every 32-row image repeated for the four lane quarters: 2 KiB of A and 4 KiB of B
constexpr int kProbeSf = 6 * 1024;
// 120 KiB of shared memory: one probe CTA per SM (two would share its tensor core)
constexpr size_t kProbeSmem = 120 * 1024;
static_assert(kProbeOperands + kProbeSf + 64 + 1024 <= (int)kProbeSmem, "probe layout");
constexpr uint32_t kProbeACol = 256;   // A operand in TMEM (the W4A16 form): 64 columns
// scale factors: A 4 columns, B 8 columns per stage; four stages rotate through 48 columns
// (as the GEMM's ring does, so a copy never overwrites columns an MMA in flight reads)
constexpr uint32_t kProbeSfCol = 320;

template <int MODE>
__global__ void __launch_bounds__(128, 1)
    mma_probe_kernel(int n, int iters, int random, uint64_t* __restrict__ out, int32_t* err) {
  extern __shared__ uint8_t probe_raw[];
  uint8_t* sA = reinterpret_cast<uint8_t*>(((uintptr_t)probe_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sB = sA + 2 * kProbeABox;
  uint8_t* sSF = sB + 2 * kProbeBBox;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sSF + kProbeSf);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  const int warp = threadIdx.x >> 5;

  // zero operands (BF16, E4M3 and E2M1 zeros), or (random) hashed bits, finite by their
  // masks: BF16 with the top exponent bit clear (magnitudes below 2), E4M3 bytes with the
  // lowest exponent bit clear (never the NaN code); scale bytes 127 (2^0)
  const uint32_t mask = (MODE == QW_MMA_PROBE_F16_TMEM_A || MODE == QW_MMA_PROBE_F16_SMEM)
                            ? 0xBF7FBF7Fu
                            : 0xF7F7F7F7u;
  for (int i = threadIdx.x; i < kProbeOperands / 4; i += blockDim.x) {
    uint32_t h = (uint32_t)i * 0x9E3779B1u + 0x7F4A7C15u;  // a multiplicative hash of i
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    reinterpret_cast<uint32_t*>(sA)[i] = random ? (h & mask) : 0u;
  }
  // scale bytes 1.0: E8M0 127, or (4X kind) unsigned E4M3 0x38
  constexpr bool NV = MODE == QW_MMA_PROBE_MXF4NVF4 || MODE == QW_MMA_PROBE_MXF4NVF4_CP;
  for (int i = threadIdx.x; i < kProbeSf / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sSF)[i] = NV ? 0x38383838u : 0x7F7F7F7Fu;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();  // the tensor core reads what the threads wrote
  if (warp == 0) {
    tmem_alloc(slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *slot;

  if (threadIdx.x == 0) {
    // kind::f16: FP32 accumulator, A = B = BF16, K-major, N at bit 17, M = 128 at bit 24;
    // kind::mxf8f6f4: A = E4M3, B = E2M1, UE8M0 scales, N = 256, M = 128, the scale byte of
    // each 32-k MMA selected at bits 4 and 29
    const uint32_t id_f16 =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (8u << 24);
    const uint32_t id_mx = (5u << 10) | (32u << 17) | (1u << 23) | (8u << 24);
    // kind::mxf4nvf4: A = B = E2M1 packed, UE4M3 scales (bit 23 clear), N = 256, M = 128
    const uint32_t id_nv = (1u << 7) | (1u << 10) | (32u << 17) | (8u << 24);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB), sf0 = smem_u32(sSF);
    auto issue = [&](int i) {
      if constexpr (MODE == QW_MMA_PROBE_F16_TMEM_A || MODE == QW_MMA_PROBE_F16_SMEM) {
        const int s = i & 7;  // 16-k step of a 128-k group (two 64-k boxes)
        const uint64_t bd = smem_desc(b0 + (s >> 2) * kProbeBBox + (s & 3) * 32, 16, 1024, 2);
        if constexpr (MODE == QW_MMA_PROBE_F16_TMEM_A)
          tc_mma_f16_tmem_a(tbase, tbase + kProbeACol + 8 * s, bd, id_f16, s != 0 ? 1u : 0u);
        else
          tc_mma_f16(tbase, smem_desc(a0 + (s >> 2) * kProbeABox + (s & 3) * 32, 16, 1024, 2),
                     bd, id_f16, s != 0 ? 1u : 0u);
      } else if constexpr (NV) {
        // one 64-k MMA per 32 bytes of each row: four per 256-k stage, which copies twelve
        // scale images (A: one per MMA, B: two 128-row chunks per MMA) into 48 columns that
        // rotate over four stages
        const int kk = i & 3;
        const uint32_t sfc = tbase + kProbeSfCol + 48u * (uint32_t)((i >> 2) & 3);
        if (MODE == QW_MMA_PROBE_MXF4NVF4_CP && kk == 0) {
#pragma unroll
          for (int img = 0; img < 4; ++img) {
            tc_cp_32x128b_warpx4(sfc + 4 * img, smem_desc(sf0 + img * 512, 0, 128, 0));
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tc_cp_32x128b_warpx4(sfc + 16 + 8 * img + 4 * c,
                                   smem_desc(sf0 + 2048 + (c * 4 + img) * 512, 0, 128, 0));
          }
        }
        tc_mma_mxf4nvf4_4x(tbase, smem_desc(a0 + kk * 32, 16, 1024, 2),
                           smem_desc(b0 + kk * 32, 16, 1024, 2), id_nv, sfc + 4 * kk,
                           sfc + 16 + 8 * kk, i != 0 ? 1u : 0u);
      } else {
        const int kk = i & 3;  // 32-k MMA of a 128-k stage
        const uint32_t sfc = tbase + kProbeSfCol + 12u * (uint32_t)((i >> 2) & 3);
        // scale columns of the next stage (copies issued a stage ahead of their MMAs)
        const uint32_t sfn = tbase + kProbeSfCol + 12u * (uint32_t)(((i >> 2) + 1) & 3);
        if (MODE == QW_MMA_PROBE_MXF8F6F4_CP && kk == 0) {
          // the stage's scale images, as the W4A8 GEMM copies them
          tc_cp_32x128b_warpx4(sfc, smem_desc(sf0, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfc + 4, smem_desc(sf0 + 512, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfc + 8, smem_desc(sf0 + 1024, 0, 128, 0));
        }
        if (MODE == QW_MMA_PROBE_MXF8F6F4_CP_AHEAD && kk == 0) {
          // the same three copies, into the next stage's columns
          tc_cp_32x128b_warpx4(sfn, smem_desc(sf0, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfn + 4, smem_desc(sf0 + 512, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfn + 8, smem_desc(sf0 + 1024, 0, 128, 0));
        }
        if (MODE == QW_MMA_PROBE_MXF8F6F4_CP_WIDE && kk == 0) {
          // A's 4 columns in one 128-lane copy, B's 8 columns in another (rows of 32 bytes:
          // two 16-byte core-matrix columns 128 bytes apart, 8-row groups 256 bytes apart)
          tc_cp_128x128b(sfc, smem_desc(sf0, 0, 128, 0));
          tc_cp_128x256b(sfc + 4, smem_desc(sf0 + 2048, 128, 256, 0));
        }
        tc_mma_mxf8f6f4(tbase, smem_desc(a0 + kk * 32, 16, 1024, 2),
                        smem_desc(b0 + kk * 32, 16, 1024, 2),
                        id_mx | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), sfc, sfc + 4,
                        i != 0 ? 1u : 0u);
      }
    };
    for (int i = 0; i < 64; ++i) issue(i);  // warm-up
    tc_commit(bar);
    bool ok = mbar_wait(bar, 0, abort_flag, err);
    const uint64_t c0 = clock64(), t0 = globaltimer_ns();
    for (int i = 0; ok && i < iters; ++i) issue(i);
    tc_commit(bar);
    ok = mbar_wait(bar, 1, abort_flag, err) && ok;
    const uint64_t c1 = clock64(), t1 = globaltimer_ns();
    out[2 * blockIdx.x] = ok ? c1 - c0 : 0;
    out[2 * blockIdx.x + 1] = ok ? t1 - t0 : 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int MODE>
qw_status launch_probe_mode(int n, int iters, int random, uint64_t* out, int32_t* err, int grid,
                            cudaStream_t st) {
  static const cudaError_t attr = cudaFuncSetAttribute(
      mma_probe_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProbeSmem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  mma_probe_kernel<MODE><<<grid, 128, kProbeSmem, st>>>(n, iters, random, out, err);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace

qw_status launch_mma_probe(int mode, int n, int iters, uint64_t* out, int32_t* err,
                           cudaStream_t st) {
  const int random = (mode & QW_MMA_PROBE_RANDOM) != 0;
  mode &= ~QW_MMA_PROBE_RANDOM;
  int grid = device_sm_count();
  if (grid > QW_MMA_PROBE_MAX_CTAS) grid = QW_MMA_PROBE_MAX_CTAS;
  switch (mode) {
    case QW_MMA_PROBE_F16_TMEM_A:
      return launch_probe_mode<QW_MMA_PROBE_F16_TMEM_A>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_F16_SMEM:
      return launch_probe_mode<QW_MMA_PROBE_F16_SMEM>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_MXF8F6F4:
      return launch_probe_mode<QW_MMA_PROBE_MXF8F6F4>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_MXF8F6F4_CP:
      return launch_probe_mode<QW_MMA_PROBE_MXF8F6F4_CP>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_MXF8F6F4_CP_AHEAD:
      return launch_probe_mode<QW_MMA_PROBE_MXF8F6F4_CP_AHEAD>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_MXF4NVF4:
      return launch_probe_mode<QW_MMA_PROBE_MXF4NVF4>(n, iters, random, out, err, grid, st);
    case QW_MMA_PROBE_MXF4NVF4_CP:
      return launch_probe_mode<QW_MMA_PROBE_MXF4NVF4_CP>(n, iters, random, out, err, grid, st);
    default:
      return launch_probe_mode<QW_MMA_PROBE_MXF8F6F4_CP_WIDE>(n, iters, random, out, err, grid, st);
  }
}

qw_status launch_stream_read(const void* src, uint64_t bytes, uint32_t* sink, bool chained,
                             cudaStream_t st) {
  // a full grid: every SM holds eight CTAs of 256 threads (the thread limit)
  int64_t grid = (int64_t)device_sm_count() * 8;
  if (grid > QW_STREAM_READ_SINK_WORDS) grid = QW_STREAM_READ_SINK_WORDS;
  const uint4* p = static_cast<const uint4*>(src);
  if (chained)
    return launch_pdl(stream_read_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, p,
                      bytes / 16, sink);
  stream_read_kernel<false><<<(unsigned)grid, 256, 0, st>>>(p, bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
