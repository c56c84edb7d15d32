// gemv_w4a8.cu - small-M W4A8 path: MXFP4 weights (E2M1 codes, E8M0 scale per 32 along K)
// times MXFP8 activations (E4M3 codes, E8M0 scale per 32) for at most 8 token rows.
//
// What it computes (spke.com Humming announcement, "W8A8 / W4A8 / W4A4": MX formats with
// group-32 E8M0 scales on both operands; OCP Microscaling v1.0 defines the element values):
//     C[m][n] = bf16( sum_g 2^(sa[m][g] - 127) 2^(sw[n][g] - 127)
//                           sum_{k in g} e4m3(a[m][k]) e2m1(w[n][k])  + bias[n] )
// At a handful of token rows the block-scaled tensor-core GEMM leaves most of its 128-row
// tile empty and streams every weight tile from few SMs; this path streams the packed
// weights once across all SMs instead (HBM-bound, like the W4A16 GEMV).
//
// Decode: every E2M1 and E4M3 value is exact in FP16 (E4M3 spans 2^-9 .. 448), so one
// hardware conversion per pair (cvt.rn.f16x2.e2m1x2 / .e4m3x2) feeds a synchronous FP16
// MMA with FP32 accumulation: the products are exact and each group's sum is one FP32
// accumulation; the two group scales multiply it in FP32.
//
// Layout: the packed weights are the block-scaled GEMM's (row-major codes, N padded to 128
// rows and K to 128), so one repack serves both paths.  A scale group of 32 k is two MMA
// steps; lane (g, t) of a warp takes k = 8t .. 8t + 7 of the group (4 code bytes) for
// weight rows g and g + 8, and the same k of token row g for the B fragment - any fixed
// assignment of k to MMA slots gives the same sum, as long as both operands use it.
// Work item = 16 weight rows over all of K; the 8 warps of a CTA split the groups and meet
// in shared memory (fixed-order sum).  Each warp streams its groups through its own ring of
// two shared-memory stages, one TMA box of 16 rows x 128 bytes (eight groups) each, stored
// with the 128-byte swizzle so that the lanes' 4-byte fragment reads (word t of chunk j of
// rows g and g + 8) fall in 32 different banks; lane 0 refills a slot as soon as the warp
// has read it.  (Reading the fragments straight from global memory, 4 bytes per lane from
// 8 rows at a time, used half of every 32-byte sector per instruction: 2.2x the sector
// traffic.)  The activations are staged once per warp, already decoded (FP16 B fragments
// and FP32 scales in shared memory).  Launched as a programmatic dependent: only weights
// and their scales are read before griddepcontrol.wait.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kW8Warps = 8;
constexpr int kW8StageGroups = 8;                       // scale groups per ring stage
constexpr int kW8StageBytes = 16 * kW8StageGroups * 16;  // one TMA box: 16 rows x 128 bytes
// ring stages per warp: measured on GB300 (M = 1, 14336 x 4096 / 4096 x 14336 / 4096 x
// 4096), two stages ran 9.4 / 10.5 / 4.3 us, three 10.4 / 10.9 / 4.6, four 10.8 / 11.1 / 4.3
constexpr int kW8MaxStages = 2;

// two E8M0 scales (the low 16 bits of `pair`) -> 2^(s - 127) as a BF16 pair, exactly (the
// smallest, 2^-127, is a BF16 subnormal)
__device__ __forceinline__ uint32_t e8m0x2_to_bf16x2(uint32_t pair) {
  uint32_t d;
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(d) : "h"((uint16_t)pair));
  return d;
}
// two E4M3 codes (the low 16 bits of `pair`, first code in the low byte) -> FP16 pair
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)pair));
  return d;
}
// E8M0 byte -> 2^(s - 127) as FP32 (s = 0 is the subnormal 2^-127; 0xFF never reaches here:
// repack and the callers' quantizer reject it)
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  return __uint_as_float(s ? (s << 23) : 0x00400000u);
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct W4A8GemvParams {
  const uint8_t* sp;   // E8M0 in 512-byte chunks of 128 rows x 4 groups
  const uint8_t* A;    // E4M3 [M][K]
  const uint8_t* Asf;  // E8M0 [M][K / 32]
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K, K_pad, M;
  int32_t gpw;          // scale groups per warp, a multiple of kW8StageGroups
  int32_t stages;       // ring stages per warp (kW8MaxStages)
  const float* scale2;  // second-level scales [N_pad] or null
  int32_t* err;         // QW_ERR_TIMEOUT if a ring wait gives up
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// ONE: a single token row (only the D fragment's column 0 is ever stored: lanes t = 0 keep
// rows g and g + 8; the other columns' scale work is skipped)
template <bool ONE>
__global__ void __launch_bounds__(kW8Warps * 32, 2)
    gemv_w4a8_kernel(const __grid_constant__ CUtensorMap tmW, const W4A8GemvParams p) {
  __shared__ float red[2][kW8Warps * 128];
  __shared__ uint64_t full[kW8Warps][kW8MaxStages];
  __shared__ int abort_flag;
  extern __shared__ uint8_t w8_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.stages;
  const int G = p.K >> 5;
  const uint32_t nblocks = (uint32_t)(p.N_pad >> 4);
  const int g0 = min(G, warp * p.gpw);
  const int cnt = min(G, g0 + p.gpw) - g0;  // this warp's groups per item (may be 0)
  const int nst = (cnt + kW8StageGroups - 1) / kW8StageGroups;  // its stages per item
  const uint32_t my_items =
      blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint32_t total = my_items * (uint32_t)nst;  // the warp's stage sequence
  // the warps' rings (1 KiB aligned: the 128-byte swizzle repeats every 1 KiB), then the
  // staged activations
  const uint32_t pad = (1024u - (smem_u32(w8_smem) & 1023u)) & 1023u;
  uint8_t* ring = w8_smem + pad + (size_t)warp * S * kW8StageBytes;
  uint8_t* act = w8_smem + pad + (size_t)kW8Warps * S * kW8StageBytes;
  uint64_t* bar = full[warp];
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // issue cursor: the next stage to copy (item, stage within the item, ring slot); every
  // lane advances it, lane 0 issues the copy
  uint32_t i_it = 0;
  int i_c = 0, i_s = 0;
  uint32_t issued = 0;
  auto issue_next = [&]() {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[i_s], kW8StageBytes);
      tma_load_2d(ring + i_s * kW8StageBytes, &tmW, &bar[i_s], (g0 + kW8StageGroups * i_c) * 16,
                  (int32_t)((blockIdx.x + i_it * gridDim.x) * 16));
    }
    ++issued;
    if (++i_c == nst) {
      i_c = 0;
      ++i_it;
    }
    if (++i_s == S) i_s = 0;
  };
  // scale cursor: the next stage whose scale words are loaded.  Row g's word of groups
  // 4Q .. 4Q + 3 sits at srow + 512 Q; row g + 8's 128 bytes after it (rows g and g + 8 of
  // a 16-row block share their 32-row lane group)
  uint32_t s_q = 0, s_it = 0;
  int s_c = 0;
  const uint8_t* srow = nullptr;
  auto load_scales_next = [&](uint32_t (&w)[4]) {
    if (s_q >= total) return;
    ++s_q;
    if (s_c == 0) {
      const int64_t row = (int64_t)(blockIdx.x + s_it * gridDim.x) * 16 + g;
      srow = p.sp + (row >> 7) * (int64_t)(p.K_pad >> 7) * 512 + (row & 31) * 16 +
             ((row & 127) >> 5) * 4;
    }
    const int gb = g0 + kW8StageGroups * s_c;
    const uint8_t* a = srow + (gb >> 2) * 512;
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(a));
    w[1] = __ldg(reinterpret_cast<const uint32_t*>(a + 128));
    if (gb + 4 < g0 + cnt) {
      w[2] = __ldg(reinterpret_cast<const uint32_t*>(a + 512));
      w[3] = __ldg(reinterpret_cast<const uint32_t*>(a + 640));
    }
    if (++s_c == nst) {
      s_c = 0;
      ++s_it;
    }
  };

  // weights do not depend on the previous kernel: the first stages stream before the wait
  while (issued < total && issued < (uint32_t)S) issue_next();
  uint32_t sc_a[4] = {0u, 0u, 0u, 0u}, sc_b[4] = {0u, 0u, 0u, 0u};
  load_scales_next(sc_a);

  // ---- activations (the previous kernel's output may be A): each warp stages its own
  // groups once, decoded - B fragments as FP16 pairs [group][row][t][4 x f16x2] and the
  // scales as FP32 [group][8 tokens] (tokens past M get 0: never stored)
  pdl_wait();
  const int KG = p.K >> 5;
  float* fa = reinterpret_cast<float*>(act + (size_t)G * p.M * 64);
  for (int q = lane; q < cnt * p.M * 4; q += 32) {
    const int tt = q & 3, m = (q >> 2) % p.M, gl = (q >> 2) / p.M;
    const int gg = g0 + gl;
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(p.A + (int64_t)m * p.K + gg * 32 + 8 * tt));
    const uint4 v = make_uint4(e4m3x2_to_f16x2(x.x), e4m3x2_to_f16x2(x.x >> 16),
                               e4m3x2_to_f16x2(x.y), e4m3x2_to_f16x2(x.y >> 16));
    *reinterpret_cast<uint4*>(act + ((gg * p.M + m) * 4 + tt) * 16) = v;
  }
  for (int q = lane; q < cnt * 8; q += 32) {
    const int tok = q & 7, gg = g0 + (q >> 3);
    fa[gg * 8 + tok] = tok < p.M ? e8m0_to_f32(__ldg(p.Asf + (int64_t)tok * KG + gg)) : 0.f;
  }
  __syncwarp();
  // B operand: token row g (rows past M read row 0; their results are never stored); the
  // D fragment's columns are tokens 2t and 2t + 1
  const uint32_t act_lane = smem_u32(act) + (uint32_t)(((g < p.M ? g : 0) * 4 + t) * 16);
  const uint32_t grp_stride = (uint32_t)p.M * 64;
  const uint32_t fa_lane = smem_u32(fa) + (uint32_t)(2 * t * 4);
  // lane (g, t) reads word t of 16-byte chunk j of rows g and g + 8 of a slot; the TMA's
  // 128-byte swizzle stores chunk j of row r at chunk j ^ (r % 8)
  const uint32_t ring_lane = smem_u32(ring) + (uint32_t)(g * 128 + 4 * t);

  bool ok = true;       // warp-uniform
  uint32_t done = 0;    // stages whose copies have landed
  int w_s = 0;          // ring slot of the stage being consumed
  uint32_t w_ph = 0;    // and the phase it completes
  // one group: MMAs over its 32 k, then the two scales
  auto group = [&](uint32_t slot, int j, int gg, const uint32_t (&cur)[4], float (&acc)[4]) {
    const uint32_t off = (uint32_t)((j ^ g) << 4);
    const uint32_t wa = lds32(slot + off), wb = lds32(slot + 1024u + off);
    uint4 x;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                 : "r"(act_lane + (uint32_t)gg * grp_stride));
    uint2 f2;
    if constexpr (ONE) {
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(f2.x) : "r"(fa_lane + (uint32_t)gg * 32));
      f2.y = 0u;
    } else {
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                   : "=r"(f2.x), "=r"(f2.y)
                   : "r"(fa_lane + (uint32_t)gg * 32));
    }
    float pr[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t ca[4], cb[4];  // FP16 pairs of the code bytes of rows g and g + 8
    e2m1x8_to_f16x2(wa, ca);
    e2m1x8_to_f16x2(wb, cb);
#pragma unroll
    for (int st = 0; st < 2; ++st) {  // code bytes 2st, 2st + 1 of each row
      const uint32_t a[4] = {ca[2 * st], cb[2 * st], ca[2 * st + 1], cb[2 * st + 1]};
      mma_f16_16816(pr, a, st ? x.z : x.x, st ? x.w : x.y);
    }
    // this group's byte of each row's scale word, both converted at once
    const uint32_t swa = cur[(j >> 2) * 2], swb = cur[(j >> 2) * 2 + 1];
    const uint32_t sbyte = (uint32_t)(j & 3);
    const uint32_t wsc = e8m0x2_to_bf16x2(__byte_perm(swa, swb, sbyte | ((4u + sbyte) << 4)));
    const float fw0 = __uint_as_float(wsc << 16);
    const float fw1 = __uint_as_float(wsc & 0xFFFF0000u);
    const float fa0 = __uint_as_float(f2.x), fa1 = __uint_as_float(f2.y);
    if constexpr (ONE) {
      acc[0] = fmaf(pr[0] * fw0, fa0, acc[0]);
      acc[2] = fmaf(pr[2] * fw1, fa0, acc[2]);
    } else {
      acc[0] = fmaf(pr[0] * fw0, fa0, acc[0]);
      acc[1] = fmaf(pr[1] * fw0, fa1, acc[1]);
      acc[2] = fmaf(pr[2] * fw1, fa0, acc[2]);
      acc[3] = fmaf(pr[3] * fw1, fa1, acc[3]);
    }
  };
  // one stage: wait for its slot, its groups' MMAs, refill the slot with the next stage to
  // copy; `cur` holds this stage's scale words, `nxt` receives the next stage's
  auto stage = [&](int c, const uint32_t (&cur)[4], uint32_t (&nxt)[4], float (&acc)[4]) {
    load_scales_next(nxt);
    if (ok) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[w_s], w_ph, abort, p.err));
      if (ok) ++done;
    }
    if (ok) {
      const uint32_t slot = ring_lane + (uint32_t)(w_s * kW8StageBytes);
      const int gb = g0 + kW8StageGroups * c;
      const int ng = min(kW8StageGroups, g0 + cnt - gb);
      if (ng == kW8StageGroups) {
#pragma unroll
        for (int j = 0; j < kW8StageGroups; ++j) group(slot, j, gb + j, cur, acc);
      } else {
#pragma unroll
        for (int j = 0; j < kW8StageGroups; ++j)
          if (j < ng) group(slot, j, gb + j, cur, acc);
      }
    }
    if (++w_s == S) {
      w_s = 0;
      w_ph ^= 1u;
    }
    // every lane has read the slot: it takes the next stage to copy
    __syncwarp();
    if (ok && issued < total) issue_next();
  };

  uint32_t q = 0;
  for (uint32_t it = 0; it < my_items; ++it) {
    const uint32_t nb = blockIdx.x + it * gridDim.x;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < nst; ++c, ++q) {
      if (q & 1u)
        stage(c, sc_b, sc_a, acc);
      else
        stage(c, sc_a, sc_b, acc);
    }

    // split-K reduction over the CTA's warps, fixed order; one barrier per item
    float* rb = red[it & 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) rb[(warp * 4 + i) * 32 + lane] = acc[i];
    __syncthreads();
    for (int o = threadIdx.x; o < 16 * p.M; o += kW8Warps * 32) {
      const int nl = o & 15, m = o >> 4;
      const int l = (nl & 7) * 4 + (m >> 1), i = (nl >> 3) * 2 + (m & 1);
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kW8Warps; ++w2) v += rb[(w2 * 4 + i) * 32 + l];
      const int n = (int)nb * 16 + nl;
      if (n < p.N) {
        if (p.scale2) v *= __ldg(p.scale2 + n);
        if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + n) << 16);
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        p.C[(int64_t)m * p.N + n] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
  }
  // a wait that gave up leaves copies in flight: let them land before shared memory goes
  if (!ok && lane == 0) {
    for (uint32_t qq = done; qq < issued; ++qq) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bar[qq % (uint32_t)S], (qq / (uint32_t)S) & 1u))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 w8_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

qw_status launch_gemv_w4a8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* A_sf, const void* bias, const float* scale2,
                           void* C, int M, int32_t* err, cudaStream_t st) {
  if (M < 1 || M > kW4A8GemvRows || d.E != 1 || d.wfmt != QW_W_MXFP4_G32 ||
      w4a8_gemv_smem_bytes(d.K, M) > kW4A8GemvMaxSmem)
    return QW_ERR_UNSUPPORTED;
  auto enc = w8_encode_fn();
  if (!enc) return QW_ERR_CUDA;
  // the packed codes as [N_pad rows][K_pad / 2 bytes]; a box is 16 rows x 128 bytes (eight
  // groups of 32 codes), stored with the 128-byte swizzle
  CUtensorMap tmW;
  {
    cuuint64_t gdim[2] = {(cuuint64_t)(d.K_pad / 2), (cuuint64_t)d.N_pad};
    cuuint64_t gstr[1] = {(cuuint64_t)(d.K_pad / 2)};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w_packed), gdim, gstr, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QW_ERR_ALIGNMENT;
  }
  W4A8GemvParams p{};
  p.sp = static_cast<const uint8_t*>(s_packed);
  p.A = static_cast<const uint8_t*>(A);
  p.Asf = static_cast<const uint8_t*>(A_sf);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.K_pad = d.K_pad;
  p.M = M;
  p.scale2 = scale2;
  p.err = err;
  const int G = d.K / kMxGroup;
  p.gpw = ((G + kW8Warps - 1) / kW8Warps + kW8StageGroups - 1) / kW8StageGroups * kW8StageGroups;
  p.stages = kW8MaxStages;
  const size_t act = w4a8_gemv_smem_bytes(d.K, M);
  auto kern = M == 1 ? gemv_w4a8_kernel<true> : gemv_w4a8_kernel<false>;
  const size_t smem = act + 1024 + (size_t)kW8Warps * p.stages * kW8StageBytes;
  const int max_dyn =
      (int)(kW4A8GemvMaxSmem + 1024 + (size_t)kW8Warps * kW8MaxStages * kW8StageBytes);
  static const cudaError_t attr =
      cudaFuncSetAttribute(gemv_w4a8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           max_dyn) == cudaSuccess
          ? cudaFuncSetAttribute(gemv_w4a8_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn)
          : cudaErrorInvalidValue;
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kW8Warps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t items = d.N_pad / 16;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kW8Warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmW, p) != cudaSuccess) return QW_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
