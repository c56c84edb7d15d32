// gemv_w4a16.cu - small-M W4A16 path: weights streamed once from HBM with 128-bit
// coalesced loads, dequantized in registers and multiplied on the tensor cores.
//
// What it computes (spke.com Humming announcement, "WnA16"; "フォーマットとアーキテクチャ
// を横断して共有されるCUDAコンポーネント": dequantization and scaling inside the kernel,
// bias fused into the output stage):
//     C[m][n] = bf16( sum_g s[n][g] * sum_{k in g} a[m][k] * q[n][k]  + bias[n] )
//
// Design (GB300): one 16-row block of N per work item; the CTA's warps split K and
// reduce through shared memory in a fixed order (deterministic).  Each lane loads the
// packed words of exactly its own m16n8k16 A-fragment (the repack put them in that
// order), turns excess codes into BF16 with one logic op + one subtract per two weights
// (code | 0x4300 = 128 + u, then - (128 + 2^(b-1))), and issues mma.sync with the
// activations as the 8-column B operand (up to 8 rows per MMA, MCH chunks of 8 rows
// reuse the decoded weights).  Per-group partial sums stay in FP32 registers and are
// scaled by the BF16 group scale in FP32.  At these sizes the kernel is bound by HBM,
// not by the tensor pipe, so the legacy synchronous MMA is the natural instruction.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

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

// Excess-4 INT3, step s of the group: low two bits from lo word s/2, third bit from
// hi word s/4 -> four BF16x2 registers.
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

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kPF = 4;  // groups per prefetch batch

template <int BITS>
struct GroupWords;
template <>
struct GroupWords<4> {
  uint4 w0, w1;  // 8 words: k16 steps 0..7
};
template <>
struct GroupWords<3> {
  uint4 lo;  // 4 lo-plane words
  uint2 hi;  // 2 hi-plane words
};

template <int BITS>
__device__ __forceinline__ void load_group(GroupWords<BITS>& gw, const uint32_t* blk, int lane);
template <>
__device__ __forceinline__ void load_group<4>(GroupWords<4>& gw, const uint32_t* blk, int lane) {
  const uint4* p = reinterpret_cast<const uint4*>(blk) + lane * 2;
  gw.w0 = __ldcs(p);
  gw.w1 = __ldcs(p + 1);
}
template <>
__device__ __forceinline__ void load_group<3>(GroupWords<3>& gw, const uint32_t* blk, int lane) {
  gw.lo = __ldcs(reinterpret_cast<const uint4*>(blk) + lane);
  gw.hi = __ldcs(reinterpret_cast<const uint2*>(blk + 128) + lane);
}

template <int BITS, int S>
__device__ __forceinline__ void decode_step(const GroupWords<BITS>& gw, uint32_t (&a)[4]);
template <int S>
__device__ __forceinline__ void decode_step4(const GroupWords<4>& gw, uint32_t (&a)[4]) {
  const uint32_t w = (S < 4) ? (S == 0 ? gw.w0.x : S == 1 ? gw.w0.y : S == 2 ? gw.w0.z : gw.w0.w)
                             : (S == 4 ? gw.w1.x : S == 5 ? gw.w1.y : S == 6 ? gw.w1.z : gw.w1.w);
  dq_int4(w, a);
}
template <int S>
__device__ __forceinline__ void decode_step3(const GroupWords<3>& gw, uint32_t (&a)[4]) {
  const uint32_t L = (S / 2 == 0) ? gw.lo.x : (S / 2 == 1) ? gw.lo.y : (S / 2 == 2) ? gw.lo.z : gw.lo.w;
  const uint32_t H = (S / 4 == 0) ? gw.hi.x : gw.hi.y;
  dq_int3<S>(L, H, a);
}

// One work item = (expert e, 16-row block nb, rows [rb, re)), re - rb <= 8 * MCH.
template <int BITS, int MCH, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    gemv_w4a16_kernel(const uint32_t* __restrict__ wp, const uint16_t* __restrict__ sp,
                      const uint16_t* __restrict__ A, const uint16_t* __restrict__ bias,
                      uint16_t* __restrict__ C, int32_t N, int32_t N_pad, int32_t K, int64_t M,
                      const int32_t* __restrict__ queue, int64_t w_estride_words,
                      int64_t s_estride) {
  constexpr int BLK_WORDS = (BITS == 4 ? 1024 : 768) / 4;
  __shared__ float red[WARPS][MCH][4][32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nblocks = N_pad / 16;
  const int G = K / 128;
  const int64_t n_items =
      queue ? (int64_t)__ldg(queue) * nblocks : (int64_t)nblocks * ((M + 8 * MCH - 1) / (8 * MCH));

  // this warp's K slice, in groups
  const int gpw = (G + WARPS - 1) / WARPS;
  const int g0 = min(G, warp * gpw), g1 = min(G, g0 + gpw);

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    int e = 0, nb;
    int64_t rb, re;
    if (queue) {
      const int64_t tile = item / nblocks;
      nb = (int)(item % nblocks);
      e = __ldg(queue + 1 + 3 * tile);
      rb = __ldg(queue + 2 + 3 * tile);
      re = __ldg(queue + 3 + 3 * tile);
    } else {
      nb = (int)(item % nblocks);
      rb = (item / nblocks) * (8 * MCH);
      re = min64(M, rb + 8 * MCH);
    }
    const uint32_t* wpe = wp + e * w_estride_words + (int64_t)nb * BLK_WORDS;
    const uint16_t* spe = sp + e * s_estride + (int64_t)nb * 16;
    const int64_t wstride_g = (int64_t)nblocks * BLK_WORDS;  // words between groups

    // activation rows of this lane's B fragments
    const uint16_t* arow[MCH];
    bool aval[MCH];
#pragma unroll
    for (int c = 0; c < MCH; ++c) {
      const int64_t r = rb + 8 * c + g;
      aval[c] = r < re;
      arow[c] = A + (aval[c] ? r : 0) * (int64_t)K + 2 * t;
    }

    float acc[MCH][4];
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;

    GroupWords<BITS> cur[kPF], nxt[kPF];
    uint16_t scur[kPF][2], snxt[kPF][2];
    auto load_batch = [&](int gb, GroupWords<BITS>(&dst)[kPF], uint16_t(&sdst)[kPF][2]) {
#pragma unroll
      for (int j = 0; j < kPF; ++j) {
        const int gg = gb + j;
        if (gg < g1) {
          load_group<BITS>(dst[j], wpe + gg * wstride_g, lane);
          sdst[j][0] = __ldg(spe + (int64_t)gg * N_pad + g);
          sdst[j][1] = __ldg(spe + (int64_t)gg * N_pad + g + 8);
        }
      }
    };
    load_batch(g0, cur, scur);
    for (int gb = g0; gb < g1; gb += kPF) {
      if (gb + kPF < g1) load_batch(gb + kPF, nxt, snxt);
#pragma unroll
      for (int j = 0; j < kPF; ++j) {
        const int gg = gb + j;
        if (gg < g1) {
          float part[MCH][4];
#pragma unroll
          for (int c = 0; c < MCH; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[c][i] = 0.f;
          const int kbase = gg * 128;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint32_t a[4];
            if constexpr (BITS == 4) {
              switch (s) {
                case 0: decode_step4<0>(cur[j], a); break;
                case 1: decode_step4<1>(cur[j], a); break;
                case 2: decode_step4<2>(cur[j], a); break;
                case 3: decode_step4<3>(cur[j], a); break;
                case 4: decode_step4<4>(cur[j], a); break;
                case 5: decode_step4<5>(cur[j], a); break;
                case 6: decode_step4<6>(cur[j], a); break;
                default: decode_step4<7>(cur[j], a); break;
              }
            } else {
              switch (s) {
                case 0: decode_step3<0>(cur[j], a); break;
                case 1: decode_step3<1>(cur[j], a); break;
                case 2: decode_step3<2>(cur[j], a); break;
                case 3: decode_step3<3>(cur[j], a); break;
                case 4: decode_step3<4>(cur[j], a); break;
                case 5: decode_step3<5>(cur[j], a); break;
                case 6: decode_step3<6>(cur[j], a); break;
                default: decode_step3<7>(cur[j], a); break;
              }
            }
#pragma unroll
            for (int c = 0; c < MCH; ++c) {
              uint32_t b0 = 0, b1 = 0;
              if (aval[c]) {
                const uint16_t* p = arow[c] + kbase + 16 * s;
                b0 = __ldg(reinterpret_cast<const uint32_t*>(p));
                b1 = __ldg(reinterpret_cast<const uint32_t*>(p + 8));
              }
              mma_bf16_16816(part[c], a, b0, b1);
            }
          }
          const float s_lo = __uint_as_float((uint32_t)scur[j][0] << 16);
          const float s_hi = __uint_as_float((uint32_t)scur[j][1] << 16);
#pragma unroll
          for (int c = 0; c < MCH; ++c) {
            acc[c][0] = fmaf(s_lo, part[c][0], acc[c][0]);
            acc[c][1] = fmaf(s_lo, part[c][1], acc[c][1]);
            acc[c][2] = fmaf(s_hi, part[c][2], acc[c][2]);
            acc[c][3] = fmaf(s_hi, part[c][3], acc[c][3]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kPF; ++j) {
        cur[j] = nxt[j];
        scur[j][0] = snxt[j][0];
        scur[j][1] = snxt[j][1];
      }
    }

    // split-K reduction over the CTA's warps, fixed order
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[warp][c][i][lane] = acc[c][i];
    __syncthreads();
    for (int o = threadIdx.x; o < MCH * 4 * 32; o += WARPS * 32) {
      const int c = o / 128, i = (o / 32) % 4, l = o % 32;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) v += red[w][c][i][l];
      // fragment (lane l, register i) -> weight row gg + 8 * (i >> 1), token 2 tt + (i & 1)
      const int gg = l >> 2, tt = l & 3;
      const int n = nb * 16 + gg + 8 * (i >> 1);
      const int64_t r = rb + 8 * c + 2 * tt + (i & 1);
      if (n < N && r < re) {
        if (bias) v += __uint_as_float((uint32_t)__ldg(bias + (int64_t)e * N + n) << 16);
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        C[r * N + n] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
    __syncthreads();
  }
}

template <int BITS, int MCH>
void launch_variant(const qw_packed_desc& d, const void* wp, const void* sp, const void* A,
                    const void* bias, void* C, const RowSet& rs, const int32_t* queue,
                    int64_t max_items, cudaStream_t st) {
  constexpr int WARPS = 8;
  const int sms = device_sm_count();
  int64_t grid = max_items;
  const int64_t cap = (int64_t)sms * 2;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const int64_t wes = (int64_t)(d.w_expert_stride / 4);
  const int64_t ses = (int64_t)(d.s_expert_stride / 2);
  gemv_w4a16_kernel<BITS, MCH, WARPS><<<(unsigned)grid, WARPS * 32, 0, st>>>(
      (const uint32_t*)wp, (const uint16_t*)sp, (const uint16_t*)A, (const uint16_t*)bias,
      (uint16_t*)C, d.N, d.N_pad, d.K, rs.rows, queue, wes, ses);
}

}  // namespace

uint64_t gemv_w4a16_workspace(const qw_packed_desc& d, int64_t max_rows) {
  // grouped calls keep their tile queue in the workspace
  return d.E > 1 ? tile_queue_bytes(d.E, max_rows, 8) : 0;
}

qw_status launch_gemv_w4a16(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                            const void* A, const void* bias, void* C, const RowSet& rs,
                            void* ws, uint64_t ws_bytes, int32_t* err, cudaStream_t st) {
  const int64_t nblocks = d.N_pad / 16;
  if (rs.offsets == nullptr) {
    // dense: chunks of up to 64 rows reuse each decoded weight fragment
    const int64_t rows = rs.rows;
    auto go = [&](auto bits_tag) {
      constexpr int B = decltype(bits_tag)::value;
      if (rows <= 8)
        launch_variant<B, 1>(d, w_packed, s_packed, A, bias, C, rs, nullptr, nblocks, st);
      else if (rows <= 16)
        launch_variant<B, 2>(d, w_packed, s_packed, A, bias, C, rs, nullptr, nblocks, st);
      else if (rows <= 32)
        launch_variant<B, 4>(d, w_packed, s_packed, A, bias, C, rs, nullptr, nblocks, st);
      else
        launch_variant<B, 8>(d, w_packed, s_packed, A, bias, C, rs, nullptr,
                             nblocks * ((rows + 63) / 64), st);
    };
    if (d.wfmt == QW_W_INT4_G128_BF16)
      go(std::integral_constant<int, 4>{});
    else
      go(std::integral_constant<int, 3>{});
  } else {
    // grouped: tiles of <= 8 rows per expert from the device tile queue
    const uint64_t need = tile_queue_bytes(rs.E, rs.rows, 8);
    if (ws == nullptr || ws_bytes < need) return QW_ERR_WORKSPACE;
    int32_t* queue = static_cast<int32_t*>(ws);
    const int64_t max_entries = (int64_t)(need / 4 - 1) / 3;
    qw_status s = launch_build_tile_queue(rs.offsets, rs.E, 8, queue, max_entries, err, st);
    if (s != QW_OK) return s;
    const int64_t max_items = max_entries * nblocks;
    if (d.wfmt == QW_W_INT4_G128_BF16)
      launch_variant<4, 1>(d, w_packed, s_packed, A, bias, C, rs, queue, max_items, st);
    else
      launch_variant<3, 1>(d, w_packed, s_packed, A, bias, C, rs, queue, max_items, st);
  }
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
