// gemv_w4a16.cu - small-M W4A16 path: the packed weights stream once from HBM through a
// deep shared-memory ring (bulk copies), are dequantized in registers and multiplied on
// the tensor cores.
//
// What it computes (spke.com Humming announcement, "WnA16"; "フォーマットとアーキテクチャ
// を横断して共有されるCUDAコンポーネント": dequantization and scaling inside the kernel,
// bias fused into the output stage):
//     C[m][n] = bf16( sum_g s[n][g] * sum_{k in g} a[m][k] * q[n][k]  + bias[n] )
//
// Design (GB300).  At M <= 64 the work is bound by HBM: 0.5 (INT4) or 0.375 (INT3) bytes
// per weight against 2M flops.  Two things decide the speed: enough bytes in flight per SM
// at every moment, and few issued instructions per weight (measured: the SM's issue slots,
// not DRAM, limited the first versions of this kernel).
//   - A work item is one 16-row block of N (times up to 8 x MCH token rows) over the whole
//     of K; the 8 warps of a CTA split its scale groups into contiguous ranges and meet in
//     shared memory at the end of the item (fixed-order sum: deterministic, no workspace).
//   - A warp walks its (item, batch of NB groups) sequence with the next batch's packed
//     words already loading into registers: each slot of the register ring is refilled
//     (16-byte streaming loads of the lane's own fragment words, which the repack stored
//     contiguously) right after the group in it is taken for compute, across item
//     boundaries, so loads stay in flight while the CTA computes and reduces.
//   - Codes become BF16 with one logic op per two weights: code | 0x4300 is the BF16 number
//     128 + code.  With up to 16 token rows the MMA takes these biased values as they are
//     and one extra MMA per step against an all-ones fragment yields the activation sums,
//     so the group sum is P - (128 + excess) * sum(a) in FP32 (no BF16 subtracts); with
//     more rows the bias is subtracted in BF16 (exact, small integers).  Per-group sums are
//     scaled by the BF16 group scale in FP32.
// The tensor pipe is mostly idle at these sizes, so the synchronous MMA is the natural
// instruction.  No thread waits on another CTA or on a flag.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kWarps = 8;        // warps per CTA (split K of one item)
// resident CTAs per SM a variant is built for (token rows cost registers)
__host__ __device__ constexpr int ctas_per_sm(int mch) { return 2; }

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// (a & b) | c in one logic instruction (written out so the compiler cannot split it)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Step S of a group -> four BF16x2 A-fragment registers holding 128 + code.
// INT4: word S of the lane's eight, nibble pairs at shifts 0, 4, 8, 12 (one shift and one
// logic op per pair).  INT3: low two bits from lo-plane word S/2, third bit from hi-plane
// word S/4 (two shifts and two logic ops per pair).
template <int BITS, int S>
__device__ __forceinline__ void biased_step(const uint32_t (&w)[8], uint32_t (&a)[4]) {
  const uint32_t magic = 0x43004300u;  // BF16 pair (128, 128)
  if constexpr (BITS == 4) {
    const uint32_t x = w[S];
    a[0] = and_or(x, 0x000F000Fu, magic);
    a[1] = and_or(x >> 4, 0x000F000Fu, magic);
    a[2] = and_or(x >> 8, 0x000F000Fu, magic);
    a[3] = and_or(x >> 12, 0x000F000Fu, magic);
  } else {
    const uint32_t L = w[S / 2], H = w[4 + S / 4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int ls = 2 * (4 * (S & 1) + r);
      const int hs = 4 * (S & 3) + r;  // hi bit to bit 2 of each half
      const uint32_t hb = hs >= 2 ? H >> (hs - 2) : H << (2 - hs);
      a[r] = and_or(hb, 0x00040004u, and_or(L >> ls, 0x00030003u, magic));
    }
  }
}

template <int BITS>
__device__ __forceinline__ void biased(int s, const uint32_t (&w)[8], uint32_t (&a)[4]) {
  switch (s) {
    case 0: biased_step<BITS, 0>(w, a); break;
    case 1: biased_step<BITS, 1>(w, a); break;
    case 2: biased_step<BITS, 2>(w, a); break;
    case 3: biased_step<BITS, 3>(w, a); break;
    case 4: biased_step<BITS, 4>(w, a); break;
    case 5: biased_step<BITS, 5>(w, a); break;
    case 6: biased_step<BITS, 6>(w, a); break;
    default: biased_step<BITS, 7>(w, a); break;
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

template <int BITS>
struct Geo {
  static constexpr int BLK = BITS == 4 ? 1024 : 768;   // one 16 x 128 block
  static constexpr int WPG = BITS == 4 ? 8 : 6;        // words per lane and group
  static constexpr float BIAS = BITS == 4 ? 136.f : 132.f;  // 128 + excess
};

// groups per batch = register ring depth (token rows cost registers)
__host__ __device__ constexpr int batch_groups(int mch) { return mch >= 4 ? 2 : 4; }

struct Params {
  const uint8_t* wp;
  const uint16_t* sp;
  const uint16_t* A;
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K;
  int64_t M;             // dense rows (unused when grouped)
  const int32_t* queue;  // grouped tile queue or null
  int64_t w_estride, s_estride;  // bytes, BF16 elements
  int32_t gpw;           // scale groups per warp
};

// One work item = (expert e, 16-row block nb, token rows [rb, re)), re - rb <= 8 * MCH.
template <int MCH>
__device__ __forceinline__ void item_of(const Params& p, uint32_t item, uint32_t nblocks, int& e,
                                        int& nb, int64_t& rb, int64_t& re) {
  const uint32_t tile = item / nblocks;
  nb = (int)(item - tile * nblocks);
  if (p.queue) {
    e = __ldg(p.queue + 1 + 3 * tile);
    rb = __ldg(p.queue + 2 + 3 * tile);
    re = __ldg(p.queue + 3 + 3 * tile);
  } else {
    e = 0;
    rb = (int64_t)tile * (8 * MCH);
    re = min64(p.M, rb + 8 * MCH);
  }
}

// The lane's packed words of one 16 x 128 block (INT4: 8 words; INT3: 4 lo + 2 hi words).
template <int BITS>
__device__ __forceinline__ void load_words(const uint8_t* blk, int lane,
                                           uint32_t (&w)[Geo<BITS>::WPG]) {
  if constexpr (BITS == 4) {
    const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2);
    const uint4 v1 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2 + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else {
    const uint4 lo = __ldcs(reinterpret_cast<const uint4*>(blk) + lane);
    const uint2 hi = __ldcs(reinterpret_cast<const uint2*>(blk + 512) + lane);
    w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
    w[4] = hi.x; w[5] = hi.y;
  }
}

// Where batch `qb` of a warp's sequence lives: item ordinal it, first group gb.
struct BatchPtr {
  const uint8_t* w;   // block (g = gb) of the item's 16-row block
  const uint16_t* s;  // scales of rows nb*16 + lane/4 (+ 8) at group gb
  int ng;             // groups in the batch (0: past the end)
};

template <int BITS, int MCH, int NB>
__device__ __forceinline__ BatchPtr batch_ptr(const Params& p, uint32_t qb, uint32_t total,
                                              uint32_t nbat, int g0, int cnt, uint32_t nblocks,
                                              int g) {
  BatchPtr b{nullptr, nullptr, 0};
  if (qb >= total) return b;
  const uint32_t it = qb / nbat;
  const int bi = (int)(qb - it * nbat);
  int e, nb;
  int64_t rb, re;
  item_of<MCH>(p, blockIdx.x + it * gridDim.x, nblocks, e, nb, rb, re);
  const int gb = g0 + bi * NB;
  b.ng = min(NB, g0 + cnt - gb);
  b.w = p.wp + e * p.w_estride + ((int64_t)gb * nblocks + nb) * Geo<BITS>::BLK;
  b.s = p.sp + e * p.s_estride + (int64_t)gb * p.N_pad + nb * 16 + g;
  return b;
}

// Step S of a group -> four BF16x2 A-fragment registers holding 128 + code.
template <int BITS>
__device__ __forceinline__ void biased_all(const uint32_t (&w)[Geo<BITS>::WPG], int s,
                                           uint32_t (&a)[4]) {
  uint32_t w8[8];
#pragma unroll
  for (int i = 0; i < Geo<BITS>::WPG; ++i) w8[i] = w[i];
#pragma unroll
  for (int i = Geo<BITS>::WPG; i < 8; ++i) w8[i] = 0;
  biased<BITS>(s, w8, a);
}

template <int BITS, int MCH>
__global__ void __launch_bounds__(kWarps * 32, ctas_per_sm(MCH))
    gemv_w4a16_kernel(const Params p) {
  using GE = Geo<BITS>;
  constexpr int WPG = GE::WPG;
  constexpr int NB = batch_groups(MCH);
  extern __shared__ float red[];  // [warp][MCH][4][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t nblocks = (uint32_t)(p.N_pad / 16);
  const int G = p.K / 128;
  // item counts stay below 2^31 (checked on the host): 32-bit index arithmetic
  const uint32_t n_items = p.queue ? (uint32_t)__ldg(p.queue) * nblocks
                                   : nblocks * (uint32_t)((p.M + 8 * MCH - 1) / (8 * MCH));
  const uint32_t my_items =
      blockIdx.x < n_items ? (n_items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int g0 = min(G, warp * p.gpw);
  const int cnt = min(G, g0 + p.gpw) - g0;  // this warp's groups per item (may be 0)
  const uint32_t nbat = (uint32_t)((cnt + NB - 1) / NB);
  const uint32_t total = my_items * nbat;
  const int64_t gstride_w = (int64_t)nblocks * GE::BLK;  // bytes between groups

  // register ring: the batch being computed next
  uint32_t wb[NB][WPG];
  uint32_t sc[NB];  // BF16 scales of rows g (low half) and g + 8 (high half)
  // refills walk the next batch's groups in slot order with running pointers
  const uint8_t* rw = nullptr;
  const uint16_t* rsc = nullptr;
  int rng = 0;
  auto refill = [&](int j) {
    if (j < rng) {
      load_words<BITS>(rw, lane, wb[j]);
      sc[j] = __byte_perm(__ldg(rsc), __ldg(rsc + 8), 0x5410);
      rw += gstride_w;
      rsc += p.N_pad;
    }
  };
  {
    const BatchPtr b0 = batch_ptr<BITS, MCH, NB>(p, 0, total, nbat, g0, cnt, nblocks, g);
    rw = b0.w;
    rsc = b0.s;
    rng = b0.ng;
#pragma unroll
    for (int j = 0; j < NB; ++j) refill(j);
  }

  uint32_t qb = 0;
  for (uint32_t it = 0; it < my_items; ++it) {
    int e, nb;
    int64_t rb, re;
    item_of<MCH>(p, blockIdx.x + it * gridDim.x, nblocks, e, nb, rb, re);
    // B operand: lane (g, t) reads token rb + 8c + g at k = 16s + 4t .. 16s + 4t + 3 for
    // MMA step s (8 bytes); rows past the tile read row rb (their results land in outputs
    // nobody stores)
    const uint16_t* arow[MCH];
#pragma unroll
    for (int c = 0; c < MCH; ++c) {
      const int64_t r = rb + 8 * c + g;
      arow[c] = p.A + (r < re ? r : rb) * (int64_t)p.K + 4 * t;
    }
    float acc[MCH][4];
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[c][j] = 0.f;

    for (uint32_t bi = 0; bi < nbat; ++bi, ++qb) {
      const int gb = g0 + (int)bi * NB;
      const int ng = min(NB, g0 + cnt - gb);
      {
        const BatchPtr nx = batch_ptr<BITS, MCH, NB>(p, qb + 1, total, nbat, g0, cnt, nblocks, g);
        rw = nx.w;
        rsc = nx.s;
        rng = nx.ng;
      }
      const uint16_t* abase[MCH];
#pragma unroll
      for (int c = 0; c < MCH; ++c) abase[c] = arow[c] + gb * 128;
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if (j < ng) {
          // the previous group is done: its slot starts loading the next batch's group
          if (j > 0) refill(j - 1);
          const uint32_t(&w)[WPG] = wb[j];
          const float s_lo = __uint_as_float(sc[j] << 16);
          const float s_hi = __uint_as_float(sc[j] & 0xFFFF0000u);
          if constexpr (MCH <= 2) {
            const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
            float pr[MCH][4], sm[MCH][4];
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i) pr[c][i] = sm[c][i] = 0.f;
            if constexpr (MCH == 1) {
              const uint2* qa = reinterpret_cast<const uint2*>(abase[0] + j * 128);
#pragma unroll
              for (int st = 0; st < 8; ++st) {
                const uint2 x = __ldg(qa + 4 * st);  // k = 16 st + 4t .. + 3
                uint32_t a[4];
                biased_all<BITS>(w, st, a);
                mma_bf16_16816(pr[0], a, x.x, x.y);
                mma_bf16_16816(sm[0], ones, x.x, x.y);
              }
            } else {
#pragma unroll
              for (int s = 0; s < 8; ++s) {
                uint32_t a[4];
                biased_all<BITS>(w, s, a);
#pragma unroll
                for (int c = 0; c < MCH; ++c) {
                  const uint2 x = __ldg(reinterpret_cast<const uint2*>(abase[c] + j * 128 + 16 * s));
                  mma_bf16_16816(pr[c], a, x.x, x.y);
                  mma_bf16_16816(sm[c], ones, x.x, x.y);
                }
              }
            }
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                acc[c][i] = fmaf(i < 2 ? s_lo : s_hi, fmaf(-GE::BIAS, sm[c][i], pr[c][i]),
                                 acc[c][i]);
          } else {
            const uint32_t bias2 = BITS == 4 ? 0x43084308u : 0x43044304u;  // BF16 pair of BIAS
            float part[MCH][4];
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i) part[c][i] = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              uint32_t a[4];
              biased_all<BITS>(w, s, a);
#pragma unroll
              for (int r = 0; r < 4; ++r) a[r] = bf16x2_sub(a[r], bias2);  // exact
#pragma unroll
              for (int c = 0; c < MCH; ++c) {
                const uint2 x = __ldg(reinterpret_cast<const uint2*>(abase[c] + j * 128 + 16 * s));
                mma_bf16_16816(part[c], a, x.x, x.y);
              }
            }
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                acc[c][i] = fmaf(i < 2 ? s_lo : s_hi, part[c][i], acc[c][i]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (j >= ng - 1) refill(j);  // slots not refilled inside the loop
    }

    // split-K reduction over the CTA's warps, fixed order
#pragma unroll
    for (int c = 0; c < MCH; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * MCH + c) * 4 + i) * 32 + lane] = acc[c][i];
    __syncthreads();
    for (int o = threadIdx.x; o < MCH * 128; o += kWarps * 32) {
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) v += red[w2 * MCH * 128 + o];
      // fragment (lane l, register i) -> weight row gq + 8 (i >> 1), token 2 tt + (i & 1)
      const int c = o >> 7, i = (o >> 5) & 3, l = o & 31;
      const int gq = l >> 2, tt = l & 3;
      const int n = nb * 16 + gq + 8 * (i >> 1);
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

template <int BITS, int MCH>
qw_status launch_variant(const Params& p, int64_t size_items, cudaStream_t st) {
  auto kern = gemv_w4a16_kernel<BITS, MCH>;
  const size_t smem = (size_t)kWarps * MCH * 128 * sizeof(float);
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > size_items) grid = size_items;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kWarps * 32, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
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
  Params p{};
  p.wp = static_cast<const uint8_t*>(w_packed);
  p.sp = static_cast<const uint16_t*>(s_packed);
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.M = rs.rows;
  p.w_estride = (int64_t)d.w_expert_stride;
  p.s_estride = (int64_t)(d.s_expert_stride / 2);
  p.gpw = (G + kWarps - 1) / kWarps;
  const int64_t nblocks = d.N_pad / 16;
  int64_t max_items = nblocks * ((rs.rows + 8 * mch - 1) / (8 * mch));
  int64_t size_items = max_items;  // what the grid is sized for
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
    // the tile count is only known on the device; size the grid for its bound (each
    // non-empty expert adds at most one ragged tile)
    const int64_t active = rs.rows < rs.E ? rs.rows : rs.E;
    size_items = nblocks * ((rs.rows + 8 * mch - 1) / (8 * mch) + active);
    if (size_items > max_items) size_items = max_items;
  }
  if (max_items > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  (void)err;
  const bool int4 = d.wfmt == QW_W_INT4_G128_BF16;
  switch (mch) {
    case 1: return int4 ? launch_variant<4, 1>(p, size_items, st) : launch_variant<3, 1>(p, size_items, st);
    case 2: return int4 ? launch_variant<4, 2>(p, size_items, st) : launch_variant<3, 2>(p, size_items, st);
    case 4: return int4 ? launch_variant<4, 4>(p, size_items, st) : launch_variant<3, 4>(p, size_items, st);
    default: return int4 ? launch_variant<4, 8>(p, size_items, st) : launch_variant<3, 8>(p, size_items, st);
  }
}

}  // namespace qw
