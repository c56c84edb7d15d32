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
// in shared memory (fixed-order sum).  Each warp keeps the next 16 groups' code words in a
// register ring (4 KiB per warp in flight) and stages its groups' activations once, already
// decoded (FP16 B fragments and FP32 scales in shared memory), so the inner loop is two
// shared loads, eight conversions and two MMAs per group.  Launched as a programmatic
// dependent: only weights and their scales are read before griddepcontrol.wait.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kW8Warps = 8;
constexpr int kW8Ring = 16;  // scale groups per batch (two code words per group and lane)

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
  const uint8_t* wp;   // codes [N_pad][K_pad / 2]
  const uint8_t* sp;   // E8M0 in 512-byte chunks of 128 rows x 4 groups
  const uint8_t* A;    // E4M3 [M][K]
  const uint8_t* Asf;  // E8M0 [M][K / 32]
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K, K_pad, M;
  int32_t gpw;  // scale groups per warp, a multiple of 4
  const float* scale2;  // second-level scales [N_pad] or null
};

// Byte offset of the 4 scales (row r, groups 4q .. 4q + 3) in the chunked layout.
__device__ __forceinline__ int64_t sf_word_offset(int64_t r, int q, int K_pad) {
  return ((r >> 7) * (K_pad >> 7) + q) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
}

__global__ void __launch_bounds__(kW8Warps * 32, 2) gemv_w4a8_kernel(const W4A8GemvParams p) {
  constexpr int R = kW8Ring;
  __shared__ float red[2][kW8Warps * 128];
  extern __shared__ uint4 w8_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.K >> 5;
  const uint32_t nblocks = (uint32_t)(p.N_pad >> 4);
  const int g0 = min(G, warp * p.gpw);
  const int cnt = min(G, g0 + p.gpw) - g0;  // this warp's groups per item (may be 0)
  const int nbat = (cnt + R - 1) / R;
  const int64_t row_bytes = p.K_pad >> 1;
  const uint32_t my_items =
      blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  pdl_launch_dependents();

  // ring: code words of rows g and g + 8 for the batch's groups, and their scale words
  uint32_t wr[R][2];
  uint32_t sw[R / 4][2];
  const uint8_t* rw = nullptr;  // row g's code bytes at the refilling batch's first group
  int rg = 0;                   // first group of the refilling batch
  int rng = 0;                  // its group count (0: nothing left)
  int64_t rrow = 0;             // row g of the refilling batch's item
  uint32_t nx_it = 0;
  int nx_c = 0;
  auto point = [&](uint32_t it, int c) {
    rng = 0;
    if (it < my_items && c < nbat) {
      const uint32_t nb = blockIdx.x + it * gridDim.x;
      rg = g0 + R * c;
      rrow = (int64_t)nb * 16 + g;
      rw = p.wp + rrow * row_bytes + rg * 16 + 4 * t;
      rng = min(R, g0 + cnt - rg);
    }
  };
  auto advance = [&]() {
    if (++nx_c == nbat) {
      nx_c = 0;
      ++nx_it;
    }
    point(nx_it, nx_c);
  };
  // slot j's code words; scale word b covers slots 4b .. 4b + 3 (rg is a multiple of 4)
  auto refill_w = [&](int j) {
    if (j < rng) {
      wr[j][0] = __ldcs(reinterpret_cast<const uint32_t*>(rw + j * 16));
      wr[j][1] = __ldcs(reinterpret_cast<const uint32_t*>(rw + 8 * row_bytes + j * 16));
    }
  };
  auto refill_s = [&](int b) {
    if (4 * b < rng) {
      const int q = (rg >> 2) + b;
      sw[b][0] = __ldg(reinterpret_cast<const uint32_t*>(p.sp + sf_word_offset(rrow, q, p.K_pad)));
      sw[b][1] =
          __ldg(reinterpret_cast<const uint32_t*>(p.sp + sf_word_offset(rrow + 8, q, p.K_pad)));
    }
  };
  point(0, 0);
#pragma unroll
  for (int j = 0; j < R; ++j) refill_w(j);
#pragma unroll
  for (int b = 0; b < R / 4; ++b) refill_s(b);
  advance();

  // ---- activations (the previous kernel's output may be A): each warp stages its own
  // groups once, decoded - B fragments as FP16 pairs [group][row][t][4 x f16x2] and the
  // scales as FP32 [group][8 tokens] (tokens past M get 0: never stored)
  pdl_wait();
  const int KG = p.K >> 5;
  uint8_t* act = reinterpret_cast<uint8_t*>(w8_smem);
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

  for (uint32_t it = 0; it < my_items; ++it) {
    const uint32_t nb = blockIdx.x + it * gridDim.x;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < nbat; ++c) {
      const int gb = g0 + R * c;
      const int ng = min(R, g0 + cnt - gb);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (j < ng) {
          const int gg = gb + j;
          uint4 x;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                       : "r"(act_lane + (uint32_t)gg * grp_stride));
          uint2 f2;
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                       : "=r"(f2.x), "=r"(f2.y)
                       : "r"(fa_lane + (uint32_t)gg * 32));
          const uint32_t wa = wr[j][0], wb = wr[j][1];
          const uint32_t swa = sw[j >> 2][0], swb = sw[j >> 2][1];
          // slot j (and after its last group, scale word j / 4) is free: start loading the
          // next batch's
          refill_w(j);
          if ((j & 3) == 3) refill_s(j >> 2);
          float pr[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t ca[4], cb[4];  // FP16 pairs of the code bytes of rows g and g + 8
          e2m1x8_to_f16x2(wa, ca);
          e2m1x8_to_f16x2(wb, cb);
#pragma unroll
          for (int st = 0; st < 2; ++st) {  // code bytes 2st, 2st + 1 of each row
            const uint32_t a[4] = {ca[2 * st], cb[2 * st], ca[2 * st + 1], cb[2 * st + 1]};
            mma_f16_16816(pr, a, st ? x.z : x.x, st ? x.w : x.y);
          }
          // this group's byte of each row's scale word (gb % 4 == 0), both converted at once
          const uint32_t sbyte = (uint32_t)(j & 3);
          const uint32_t wsc = e8m0x2_to_bf16x2(__byte_perm(swa, swb, sbyte | ((4u + sbyte) << 4)));
          const float fw0 = __uint_as_float(wsc << 16);
          const float fw1 = __uint_as_float(wsc & 0xFFFF0000u);
          const float fa0 = __uint_as_float(f2.x), fa1 = __uint_as_float(f2.y);
          acc[0] = fmaf(pr[0] * fw0, fa0, acc[0]);
          acc[1] = fmaf(pr[1] * fw0, fa1, acc[1]);
          acc[2] = fmaf(pr[2] * fw1, fa0, acc[2]);
          acc[3] = fmaf(pr[3] * fw1, fa1, acc[3]);
        }
      }
      // slots and scale words the loop did not reach
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (j >= ng) refill_w(j);
#pragma unroll
      for (int b = 0; b < R / 4; ++b)
        if (4 * b + 3 >= ng) refill_s(b);
      advance();
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
}

}  // namespace

qw_status launch_gemv_w4a8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* A_sf, const void* bias, const float* scale2,
                           void* C, int M, cudaStream_t st) {
  if (M < 1 || M > kW4A8GemvRows || d.E != 1 || d.wfmt != QW_W_MXFP4_G32 ||
      w4a8_gemv_smem_bytes(d.K, M) > kW4A8GemvMaxSmem)
    return QW_ERR_UNSUPPORTED;
  W4A8GemvParams p{};
  p.wp = static_cast<const uint8_t*>(w_packed);
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
  const int G = d.K / kMxGroup;
  p.gpw = ((G + kW8Warps - 1) / kW8Warps + 3) / 4 * 4;
  auto kern = gemv_w4a8_kernel;
  const size_t smem = w4a8_gemv_smem_bytes(d.K, M);
  static const cudaError_t attr = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kW4A8GemvMaxSmem);
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
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return QW_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
