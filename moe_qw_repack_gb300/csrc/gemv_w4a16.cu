// gemv_w4a16.cu - small-M W4A16 path: weights streamed once from HBM with 128-bit
// coalesced loads, dequantized in registers and multiplied on the tensor cores.
//
// What it computes (spke.com Humming announcement, "WnA16"; "フォーマットとアーキテクチャ
// を横断して共有されるCUDAコンポーネント": dequantization and scaling inside the kernel,
// bias fused into the output stage):
//     C[m][n] = bf16( sum_g s[n][g] * sum_{k in g} a[m][k] * q[n][k]  + bias[n] )
//
// Design (GB300).  At M <= 64 the work is bound by HBM: 0.5 (INT4) or 0.375 (INT3) bytes
// per weight against 2M flops, so what matters is keeping enough bytes in flight per SM
// (bandwidth x latency / SMs, about 40 KB).  A work item is one 16-row block of N (and up
// to 8 x MCH token rows); its CTA of W warps splits K, each warp owning up to MAXG scale
// groups at a time whose packed words it loads all at once (16-byte loads, 512 contiguous
// bytes per warp and load), so a CTA has about W x MAXG KB in flight and several CTAs stay
// resident per SM.  Each lane loads exactly its own m16n8k16 A-fragments (the repack
// stored them in that order), turns excess codes into BF16 with one logic op and one
// subtract per two weights (code | 0x4300 is the BF16 number 128 + code), and issues
// mma.sync with up to 8 tokens per MMA as the B operand.  Per-group sums stay in FP32 and
// are scaled by the BF16 group scale in FP32; the warps' partial sums are reduced through
// shared memory in a fixed order (deterministic).  The tensor pipe is mostly idle at these
// sizes, so the synchronous MMA is the natural instruction.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

// warps per CTA at most: 16, or 8 when 32+ token rows per item need the registers
constexpr int max_warps(int mch) { return mch >= 4 ? 8 : 16; }

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// Excess-8 INT4 word (fragment order) -> four BF16x2 A-fragment registers.
__device__ __forceinline__ void dq_int4(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t magic = 0x43004300u;  // BF16 pair (128, 128)
  const uint32_t bias = 0x43084308u;   // BF16 pair (136, 136)
  a[0] = bf16x2_sub((w & 0x000F000Fu) | magic, bias);
  a[1] = bf16x2_sub(((w >> 4) & 0x000F000Fu) | magic, bias);
  a[2] = bf16x2_sub(((w >> 8) & 0x000F000Fu) | magic, bias);
  a[3] = bf16x2_sub(((w >> 12) & 0x000F000Fu) | magic, bias);
}

// Excess-4 INT3, k16 step S of the group: low two bits from lo-plane word S/2, third bit
// from hi-plane word S/4 -> four BF16x2 registers.
template <int S>
__device__ __forceinline__ void dq_int3(uint32_t L, uint32_t H, uint32_t (&a)[4]) {
  const uint32_t magic = 0x43004300u;
  const uint32_t bias = 0x43044304u;  // BF16 pair (132, 132)
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int ls = 2 * (4 * (S & 1) + r);
    const int hs = 4 * (S & 3) + r;
    const uint32_t lo = (L >> ls) & 0x00030003u;
    const uint32_t hi = ((H >> hs) & 0x00010001u) << 2;
    a[r] = bf16x2_sub(lo | hi | magic, bias);
  }
}

template <int BITS, int S>
__device__ __forceinline__ void decode_step(const uint32_t (&w)[8], uint32_t (&a)[4]) {
  if constexpr (BITS == 4) {
    dq_int4(w[S], a);
  } else {
    dq_int3<S>(w[S / 2], w[4 + S / 4], a);  // INT3: w[0..3] lo plane, w[4..5] hi plane
  }
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packed words of one 16 x 128 block for this lane (INT4: 8 words; INT3: 4 + 2 words).
template <int BITS>
__device__ __forceinline__ void load_block(const uint32_t* blk, int lane, uint32_t (&w)[8]) {
  if constexpr (BITS == 4) {
    const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2);
    const uint4 v1 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2 + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else {
    const uint4 lo = __ldcs(reinterpret_cast<const uint4*>(blk) + lane);
    const uint2 hi = __ldcs(reinterpret_cast<const uint2*>(blk + 128) + lane);
    w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
    w[4] = hi.x; w[5] = hi.y; w[6] = 0; w[7] = 0;
  }
}

struct Params {
  const uint32_t* wp;
  const uint16_t* sp;
  const uint16_t* A;
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K;
  int64_t M;             // dense rows (unused when grouped)
  const int32_t* queue;  // grouped tile queue or null
  int64_t w_estride_words, s_estride;
  int32_t gpw;           // scale groups per warp
};

// One work item = (expert e, 16-row block nb, token rows [rb, re)), re - rb <= 8 * MCH.
template <int BITS, int MCH, int MAXG>
__global__ void __launch_bounds__(max_warps(MCH) * 32)
    gemv_w4a16_kernel(const Params p) {
  constexpr int BLK_WORDS = (BITS == 4 ? 1024 : 768) / 4;
  extern __shared__ float red[];  // [W][MCH][4][32]
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nblocks = p.N_pad / 16;
  const int G = p.K / 128;
  // item counts stay below 2^31 (checked on the host): 32-bit index arithmetic
  const uint32_t n_items = p.queue ? (uint32_t)__ldg(p.queue) * (uint32_t)nblocks
                                   : (uint32_t)nblocks * (uint32_t)((p.M + 8 * MCH - 1) / (8 * MCH));
  const int g0 = min(G, warp * p.gpw), g1 = min(G, g0 + p.gpw);

  for (uint32_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    int e = 0;
    const uint32_t tile = item / (uint32_t)nblocks;
    const int nb = (int)(item - tile * (uint32_t)nblocks);
    int64_t rb, re;
    if (p.queue) {
      e = __ldg(p.queue + 1 + 3 * tile);
      rb = __ldg(p.queue + 2 + 3 * tile);
      re = __ldg(p.queue + 3 + 3 * tile);
    } else {
      rb = (int64_t)tile * (8 * MCH);
      re = min64(p.M, rb + 8 * MCH);
    }
    const uint32_t* wpe = p.wp + e * p.w_estride_words + (int64_t)nb * BLK_WORDS;
    const uint16_t* spe = p.sp + e * p.s_estride + (int64_t)nb * 16;
    const int64_t wstride_g = (int64_t)nblocks * BLK_WORDS;  // words between groups

    // B operand: lane (g, t) needs token rb + 8c + g at k = 32t + 4s .. +3 of each group
    // (8 contiguous bytes per MMA step, 64 per group); rows past the tile read row rb
    // and are zeroed
    const uint16_t* arow[MCH];
    bool aval[MCH];
#pragma unroll
    for (int c = 0; c < MCH; ++c) {
      const int64_t r = rb + 8 * c + g;
      aval[c] = r < re;
      arow[c] = p.A + (aval[c] ? r : rb) * (int64_t)p.K + 32 * t;
    }
    float acc[MCH][4];
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[c][j] = 0.f;

    for (int gb = g0; gb < g1; gb += MAXG) {
      // every load of the batch is issued before any of its data is used
      uint32_t wv[MAXG][8];
      uint32_t sv[MAXG][2];
#pragma unroll
      for (int j = 0; j < MAXG; ++j) {
        if (gb + j < g1) {
          load_block<BITS>(wpe + (gb + j) * wstride_g, lane, wv[j]);
          sv[j][0] = __ldg(spe + (int64_t)(gb + j) * p.N_pad + g);
          sv[j][1] = __ldg(spe + (int64_t)(gb + j) * p.N_pad + g + 8);
        }
      }
#pragma unroll
      for (int j = 0; j < MAXG; ++j) {
        if (gb + j < g1) {
          const int kbase = (gb + j) * 128;
          uint32_t bv[MCH == 1 ? 16 : 1];  // one token row: the group's B words, loaded at once
          if constexpr (MCH == 1) {
            const uint4* q = reinterpret_cast<const uint4*>(arow[0] + kbase);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 x = __ldg(q + v);
              bv[4 * v] = aval[0] ? x.x : 0u;
              bv[4 * v + 1] = aval[0] ? x.y : 0u;
              bv[4 * v + 2] = aval[0] ? x.z : 0u;
              bv[4 * v + 3] = aval[0] ? x.w : 0u;
            }
          }
          float part[MCH][4];
#pragma unroll
          for (int c = 0; c < MCH; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[c][i] = 0.f;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint32_t a[4];
            switch (s) {
              case 0: decode_step<BITS, 0>(wv[j], a); break;
              case 1: decode_step<BITS, 1>(wv[j], a); break;
              case 2: decode_step<BITS, 2>(wv[j], a); break;
              case 3: decode_step<BITS, 3>(wv[j], a); break;
              case 4: decode_step<BITS, 4>(wv[j], a); break;
              case 5: decode_step<BITS, 5>(wv[j], a); break;
              case 6: decode_step<BITS, 6>(wv[j], a); break;
              default: decode_step<BITS, 7>(wv[j], a); break;
            }
#pragma unroll
            for (int c = 0; c < MCH; ++c) {
              uint32_t b0, b1;
              if constexpr (MCH == 1) {
                b0 = bv[2 * s];
                b1 = bv[2 * s + 1];
              } else {
                const uint2 x = __ldg(reinterpret_cast<const uint2*>(arow[c] + kbase + 4 * s));
                b0 = aval[c] ? x.x : 0u;
                b1 = aval[c] ? x.y : 0u;
              }
              mma_bf16_16816(part[c], a, b0, b1);
            }
          }
          const float s_lo = __uint_as_float(sv[j][0] << 16);
          const float s_hi = __uint_as_float(sv[j][1] << 16);
#pragma unroll
          for (int c = 0; c < MCH; ++c) {
            acc[c][0] = fmaf(s_lo, part[c][0], acc[c][0]);
            acc[c][1] = fmaf(s_lo, part[c][1], acc[c][1]);
            acc[c][2] = fmaf(s_hi, part[c][2], acc[c][2]);
            acc[c][3] = fmaf(s_hi, part[c][3], acc[c][3]);
          }
        }
      }
    }

    // split-K reduction over the CTA's warps, fixed order
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * MCH + c) * 4 + i) * 32 + lane] = acc[c][i];
    __syncthreads();
    for (int o = threadIdx.x; o < MCH * 4 * 32; o += blockDim.x) {
      float v = 0.f;
      for (int w = 0; w < W; ++w) v += red[w * MCH * 128 + o];
      // fragment (lane l, register i) -> weight row gg + 8 (i >> 1), token 2 tt + (i & 1)
      const int c = o / 128, i = (o / 32) % 4, l = o % 32;
      const int gg = l >> 2, tt = l & 3;
      const int n = nb * 16 + gg + 8 * (i >> 1);
      const int64_t r = rb + 8 * c + 2 * tt + (i & 1);
      if (n < p.N && r < re) {
        if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + (int64_t)e * p.N + n) << 16);
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        p.C[r * p.N + n] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
    __syncthreads();
  }
}

template <int BITS, int MCH, int MAXG>
qw_status launch_variant(const Params& p, int warps, int64_t max_items, cudaStream_t st) {
  auto kern = gemv_w4a16_kernel<BITS, MCH, MAXG>;
  const size_t smem = (size_t)warps * MCH * 128 * sizeof(float);
  static const cudaError_t attr = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_warps(MCH) * MCH * 128 * 4);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, warps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, warps * 32, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

template <int BITS, int MCH>
qw_status launch_bits_mch(const Params& p, int warps, int maxg, int64_t max_items,
                          cudaStream_t st) {
  if (maxg <= 2) return launch_variant<BITS, MCH, 2>(p, warps, max_items, st);
  if (maxg <= 4) return launch_variant<BITS, MCH, 4>(p, warps, max_items, st);
  return launch_variant<BITS, MCH, 8>(p, warps, max_items, st);
}

int mch_for_rows(int64_t rows) { return rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8; }

int mch_for(const qw_packed_desc& d, int64_t rows, bool grouped) {
  if (!grouped) return mch_for_rows(rows);
  return mch_for_rows((rows + d.E - 1) / d.E);  // average rows per expert
}

}  // namespace

uint64_t gemv_w4a16_workspace(const qw_packed_desc& d, int64_t max_rows) {
  // only grouped calls need device memory of their own: the tile queue
  if (d.E <= 1) return 0;
  return tile_queue_bytes(d.E, max_rows, 8 * mch_for(d, max_rows, true));
}

qw_status launch_gemv_w4a16(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                            const void* A, const void* bias, void* C, const RowSet& rs,
                            void* ws, uint64_t ws_bytes, int32_t* err, cudaStream_t st) {
  const bool grouped = rs.offsets != nullptr;
  const int mch = mch_for(d, rs.rows, grouped);
  const int G = d.K / 128;
  // warps per CTA: about four scale groups (4 KB of INT4) per warp
  int warps = G / 4;
  if (warps < 1) warps = 1;
  if (warps > max_warps(mch)) warps = max_warps(mch);
  const int gpw = (G + warps - 1) / warps;
  const int maxg = gpw <= 2 ? 2 : gpw <= 4 ? 4 : 8;

  Params p{};
  p.wp = static_cast<const uint32_t*>(w_packed);
  p.sp = static_cast<const uint16_t*>(s_packed);
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.M = rs.rows;
  p.w_estride_words = (int64_t)(d.w_expert_stride / 4);
  p.s_estride = (int64_t)(d.s_expert_stride / 2);
  p.gpw = gpw;
  const int64_t nblocks = d.N_pad / 16;
  int64_t max_items = nblocks * ((rs.rows + 8 * mch - 1) / (8 * mch));
  if (grouped) {
    const uint64_t need = tile_queue_bytes(rs.E, rs.rows, 8 * mch);
    if (ws == nullptr || ws_bytes < need) return QW_ERR_WORKSPACE;
    int32_t* queue = static_cast<int32_t*>(ws);
    const int64_t max_entries = (int64_t)(need / 4 - 1) / 3;
    const qw_status s =
        launch_build_tile_queue(rs.offsets, rs.E, 8 * mch, rs.rows, queue, max_entries, err, st);
    if (s != QW_OK) return s;
    p.queue = queue;
    max_items = max_entries * nblocks;
  }
  if (max_items > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  const bool int4 = d.wfmt == QW_W_INT4_G128_BF16;
  switch (mch) {
    case 1:
      return int4 ? launch_bits_mch<4, 1>(p, warps, maxg, max_items, st)
                  : launch_bits_mch<3, 1>(p, warps, maxg, max_items, st);
    case 2:
      return int4 ? launch_bits_mch<4, 2>(p, warps, maxg, max_items, st)
                  : launch_bits_mch<3, 2>(p, warps, maxg, max_items, st);
    case 4:
      return int4 ? launch_bits_mch<4, 4>(p, warps, maxg, max_items, st)
                  : launch_bits_mch<3, 4>(p, warps, maxg, max_items, st);
    default:
      return int4 ? launch_bits_mch<4, 8>(p, warps, maxg, max_items, st)
                  : launch_bits_mch<3, 8>(p, warps, maxg, max_items, st);
  }
}

}  // namespace qw
