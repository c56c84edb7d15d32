// gemv_w4a16.cu - small-M W4A16 path: the packed weights stream once from HBM, are
// dequantized in registers and multiplied on the tensor cores.  Three kernels share the
// decode and MMA code: a staged-activation kernel for single-token decode over large
// matrices, a register-ring kernel for the other dense calls and a TMA-ring kernel for
// grouped (MoE) calls.  All three are launched as programmatic dependents of the previous
// kernel on the stream (griddepcontrol): back-to-back GEMVs overlap one launch's ramp-up
// with the previous one's tail, and only weights are read before the wait.
//
// What it computes (spke.com Humming announcement, "WnA16"; "フォーマットとアーキテクチャ
// を横断して共有されるCUDAコンポーネント": dequantization and scaling inside the kernel,
// bias fused into the output stage):
//     C[m][n] = bf16( sum_g s[n][g] * sum_{k in g} a[m][k] * q[n][k]  + bias[n] )
//
// Design (GB300).  At M <= 16 the work is bound by HBM: 0.5 (INT4) or 0.375 (INT3) bytes
// per weight against 2M flops.  Two things decide the speed: enough bytes in flight per SM
// at every moment (HBM latency under load is microseconds), and few issued instructions
// per weight (the SM's issue slots, not DRAM, limited the first versions of this kernel).
// A work item is one 16-row block of N (times up to 8 x MCH token rows) over the whole of
// K; the warps of a CTA split its scale groups and meet in shared memory at the end of the
// item (fixed-order sum: deterministic, no workspace).
//   - Dense (gemv_reg_kernel): 8 warps per CTA each own a contiguous range of groups and
//     walk their (item, batch of 4 groups) sequence with the next batch's packed words
//     already loading into a register ring (16-byte loads of the lane's own fragment
//     words), refilled across item boundaries.
//   - Single-token decode (gemv_m8_kernel): as the register ring, plus activations staged
//     in shared memory in B-fragment order and per-group activation sums, which replace the
//     all-ones MMA below (fewer issued instructions per weight: the decode GEMV is bound by
//     issue slots as much as by HBM).
//   - Grouped (gemv_tma_kernel): one producer thread per CTA streams an item's groups
//     eight at a time: a 4-D tensor map views the packed weights as [expert][group][16-row
//     block][1 KiB], so one TMA copy brings 8 groups of a block (8 KiB; 1 KiB copies
//     measured far below HBM speed on this GPU, 4-8 KiB ones reach it) plus a 3-D copy of
//     their scales into a 4-stage ring; four consumer warps take two groups of every stage
//     (every consumer visits every stage in order, so the barrier phase parity cannot
//     alias).  With MoE tiles of a few rows and short K (e.g. 640) this keeps more bytes in
//     flight than the register ring; with dense shapes of few items the register ring's
//     finer split of K wins (both measured).
// Codes become BF16 with one shift and one logic op per two weights: code | 0x4300 is the
// BF16 number 128 + code.  With up to 16 token rows the MMA takes these biased values as they are and
// one extra MMA per step against an all-ones fragment yields the activation sums, so the
// group sum is P - (128 + excess) * sum(a) in FP32 (no BF16 subtracts); with more rows the
// bias is subtracted in BF16 (exact, small integers).  Per-group sums are scaled by the
// BF16 group scale in FP32.  The tensor pipe is mostly idle at these sizes, so the
// synchronous MMA is the natural instruction.  No thread waits on another CTA; every
// mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

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

// (a & b) | c in one logic instruction (written out so the compiler cannot split it)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Step S of a group -> four BF16x2 A-fragment registers holding 128 + code.
// INT4: word S of the lane's eight, nibble pairs at shifts 0, 4, 8, 12 (one shift and one
// logic op per pair).  INT3: register j = 4S + r is the 3-bit field j % 5 of word j / 5
// (one shift and one logic op, like INT4), except j = 30, 31, gathered from the spare bit
// 15 + 16h of words 0..2 and 3..5.  INT2: 2-bit fields of word S/2 at 2 (4 (S & 1) + r).
template <int BITS, int S>
__device__ __forceinline__ void biased_step(const uint32_t (&w)[8], uint32_t (&a)[4]) {
  const uint32_t magic = 0x43004300u;  // BF16 pair (128, 128)
  if constexpr (BITS == 4) {
    const uint32_t x = w[S];
    a[0] = and_or(x, 0x000F000Fu, magic);
    a[1] = and_or(x >> 4, 0x000F000Fu, magic);
    a[2] = and_or(x >> 8, 0x000F000Fu, magic);
    a[3] = and_or(x >> 12, 0x000F000Fu, magic);
  } else if constexpr (BITS == 2) {
    const uint32_t L = w[S / 2];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = and_or(L >> (2 * (4 * (S & 1) + r)), 0x00030003u, magic);
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * S + r;
      if (j < 30) {
        a[r] = and_or(w[j / 5] >> (3 * (j % 5)), 0x00070007u, magic);
      } else {
        const int b = j == 30 ? 0 : 3;
        a[r] = and_or(w[b + 2] >> 13, 0x00040004u,
                      and_or(w[b + 1] >> 14, 0x00020002u, and_or(w[b] >> 15, 0x00010001u, magic)));
      }
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

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint64_t* bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint64_t* bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// ---------------------------------------------------------------- register-ring kernel (dense)
constexpr int kWarps = 8;        // warps per CTA (split K of one item)
// resident CTAs per SM a variant is built for (token rows cost registers)
__host__ __device__ constexpr int ctas_per_sm(int mch) { return 2; }

// Format codes (the BITS template argument): 4, 3, 2, 1 for INT4 / INT3 / INT2 / INT1, 8 for
// E4M3 weights, kBitsFp4 for E2M1 weights.
template <int BITS>
struct Geo {
  static constexpr int BLK = wna16_block_bytes(BITS);        // one 16 x 128 block
  static constexpr int WPG = BLK / 128;                      // words per lane and group
  // values decoded as they are (E4M3, E2M1, INT1 +-1): no excess to remove
  static constexpr bool FP = BITS == 8 || BITS == kBitsFp4 || BITS == 1;
  static constexpr float BIAS = FP ? 0.f : 128.f + (1 << (BITS - 1));  // 128 + excess
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
  int64_t zplane;        // asymmetric INT4: BF16 elements from a scale to its 128 + z
  const float* scale2;   // second-level scales [E][N_pad] or null
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

// The lane's packed words of one 16 x 128 block (INT4: 8 words; INT3: 4 + 2 words;
// INT2: 4 words; E4M3: 16 words).
template <int BITS>
__device__ __forceinline__ void load_words(const uint8_t* blk, int lane,
                                           uint32_t (&w)[Geo<BITS>::WPG]) {
  if constexpr (BITS == 4) {
    const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2);
    const uint4 v1 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2 + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else if constexpr (BITS == 2) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(blk) + lane);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 4 + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  } else if constexpr (BITS == kBitsFp4) {
    const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2);
    const uint4 v1 = __ldcs(reinterpret_cast<const uint4*>(blk) + lane * 2 + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else if constexpr (BITS == 1) {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(blk) + lane);
    w[0] = v.x; w[1] = v.y;
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

// Values decoded as they are (no excess), step s of a group -> four BF16x2 A-fragment
// registers.  E4M3: words 2s (rows g, g + 8 at k + 0/1) and 2s + 1 (at k + 2/3).  E2M1:
// byte r of word s is register r (one hardware conversion to FP16, then to BF16).  INT1:
// register r's two bits are bits 4 (s % 4) + r and 16 + 4 (s % 4) + r of word s / 4.
template <int BITS, int NW>
__device__ __forceinline__ void direct_step(const uint32_t (&w)[NW], int s, uint32_t (&a)[4]) {
  if constexpr (BITS == 8) {
    a[0] = e4m3x2_to_bf16x2(w[2 * s]);
    a[1] = e4m3x2_to_bf16x2(w[2 * s] >> 16);
    a[2] = e4m3x2_to_bf16x2(w[2 * s + 1]);
    a[3] = e4m3x2_to_bf16x2(w[2 * s + 1] >> 16);
  } else if constexpr (BITS == kBitsFp4) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[s], h);
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = f16x2_to_bf16x2(h[r]);
  } else {
    static_assert(BITS == 1, "direct decode of E4M3, E2M1 or INT1");
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = int1_pair(w[s >> 2], 4 * (s & 3) + r, 0x3F803F80u);
  }
}

// Step S of a group -> four BF16x2 A-fragment registers holding 128 + code (integer
// formats) or the decoded values (E4M3, E2M1, INT1).
template <int BITS>
__device__ __forceinline__ void biased_all(const uint32_t (&w)[Geo<BITS>::WPG], int s,
                                           uint32_t (&a)[4]) {
  if constexpr (Geo<BITS>::FP) {
    direct_step<BITS>(w, s, a);
  } else {
    uint32_t w8[8];
#pragma unroll
    for (int i = 0; i < Geo<BITS>::WPG; ++i) w8[i] = w[i];
#pragma unroll
    for (int i = Geo<BITS>::WPG; i < 8; ++i) w8[i] = 0;
    biased<BITS>(s, w8, a);
  }
}

// Step s of a group from a lane's words held in an array of any length (the TMA ring's
// consumers keep 8 words for the integer formats, 16 for E4M3).
template <int BITS, int NW>
__device__ __forceinline__ void decode_step(const uint32_t (&w)[NW], int s, uint32_t (&a)[4]) {
  if constexpr (Geo<BITS>::FP) {
    static_assert(BITS != 8 || NW == 16, "E4M3 blocks hold 16 words per lane");
    direct_step<BITS>(w, s, a);
  } else {
    static_assert(NW == 8, "integer words are passed as 8");
    biased<BITS>(s, w, a);
  }
}

template <int BITS, int MCH, bool ZP>
__global__ void __launch_bounds__(kWarps * 32, ctas_per_sm(MCH))
    gemv_reg_kernel(const Params p) {
  using GE = Geo<BITS>;
  constexpr int WPG = GE::WPG;
  // E4M3 groups are twice the bytes: half the ring depth in the same registers
  constexpr int NB = WPG > 8 ? (batch_groups(MCH) + 1) / 2 : batch_groups(MCH);
  extern __shared__ float red[];  // [warp][MCH][4][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t nblocks = (uint32_t)(p.N_pad / 16);
  const int G = p.K / 128;
  // The tile queue is the previous kernel's output: with a queue, nothing (not even the
  // item count) is read before the wait; dense calls prefetch weights before it.
  if (p.queue) pdl_wait();
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
  uint32_t zc[NB];  // asymmetric INT4: BF16 128 + z of rows g and g + 8
  // refills walk the next batch's groups in slot order with running pointers
  const uint8_t* rw = nullptr;
  const uint16_t* rsc = nullptr;
  int rng = 0;
  auto refill = [&](int j) {
    if (j < rng) {
      load_words<BITS>(rw, lane, wb[j]);
      sc[j] = __byte_perm(__ldg(rsc), __ldg(rsc + 8), 0x5410);
      if constexpr (ZP) zc[j] = __byte_perm(__ldg(rsc + p.zplane), __ldg(rsc + p.zplane + 8), 0x5410);
      rw += gstride_w;
      rsc += p.N_pad;
    }
  };
  pdl_launch_dependents();
  {
    const BatchPtr b0 = batch_ptr<BITS, MCH, NB>(p, 0, total, nbat, g0, cnt, nblocks, g);
    rw = b0.w;
    rsc = b0.s;
    rng = b0.ng;
#pragma unroll
    for (int j = 0; j < NB; ++j) refill(j);
  }
  // activations, bias and the output belong to the stream's order from here on
  pdl_wait();

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
                if constexpr (!GE::FP) mma_bf16_16816(sm[0], ones, x.x, x.y);
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
                  if constexpr (!GE::FP) mma_bf16_16816(sm[c], ones, x.x, x.y);
                }
              }
            }
            // the excess of rows g and g + 8: 128 + excess, or (asymmetric) 128 + z
            const float b_lo = ZP ? __uint_as_float(zc[j] << 16) : GE::BIAS;
            const float b_hi = ZP ? __uint_as_float(zc[j] & 0xFFFF0000u) : GE::BIAS;
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                acc[c][i] = fmaf(i < 2 ? s_lo : s_hi, fmaf(i < 2 ? -b_lo : -b_hi, sm[c][i], pr[c][i]),
                                 acc[c][i]);
          } else {
            static_assert(!ZP, "the asymmetric format runs with at most 16 token rows");
            const uint32_t bias2 = 0x43004300u + 0x10001u * (1u << (BITS - 1));  // BF16 pair of BIAS
            float part[MCH][4];
#pragma unroll
            for (int c = 0; c < MCH; ++c)
#pragma unroll
              for (int i = 0; i < 4; ++i) part[c][i] = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              uint32_t a[4];
              biased_all<BITS>(w, s, a);
              if constexpr (!GE::FP) {
#pragma unroll
                for (int r = 0; r < 4; ++r) a[r] = bf16x2_sub(a[r], bias2);  // exact
              }
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
        if (p.scale2) v *= __ldg(p.scale2 + (int64_t)e * p.N_pad + n);
        if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + (int64_t)e * p.N + n) << 16);
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        p.C[r * p.N + n] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
    __syncthreads();
  }
}

template <int BITS, int MCH, bool ZP>
qw_status launch_reg_variant(const Params& p, int64_t size_items, cudaStream_t st) {
  auto kern = gemv_reg_kernel<BITS, MCH, ZP>;
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
  return launch_pdl(kern, (unsigned)grid, kWarps * 32, smem, st, p);
}


// ---------------------------------------------------------------- dense kernel, M <= 8
// One token tile of at most 8 rows.  After griddepcontrol.wait the CTA stages the
// activations once, in the order the MMA's B fragments read them ([group][step pair][row][t]
// 16-byte chunks: one conflict-free 16-byte shared load feeds two MMA steps), together with
// every row's sum over every scale group.  With those sums known the biased codes need no
// all-ones MMA: the group sum is P - (128 + excess) * sum(a), one MMA per step.  The weights
// stream through each warp's register ring as in gemv_reg_kernel; batch pointers advance
// incrementally (no division per batch).  Items are 16-row blocks; the CTA's warps split
// the scale groups and meet in a double-buffered shared reduction (one barrier per item).
constexpr int kM8Warps = 8;
constexpr int kM8Ring = 4;  // groups per batch = register ring depth
// largest shared-memory footprint sent to the kernel: two CTAs per SM still fit
constexpr size_t kM8MaxSmem = 96 * 1024;
// smallest matrix (N x K weights) sent to it
constexpr int64_t kM8MinWeights = int64_t(1) << 25;

struct M8Params {
  const uint8_t* wp;
  const uint16_t* sp;
  const uint16_t* A;
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K, M;  // M <= 8
  int32_t gpw;             // scale groups per warp
  int64_t zplane;          // asymmetric INT4: BF16 elements from a scale to its 128 + z
  const float* scale2;     // second-level scales [N_pad] or null
};

__host__ __device__ constexpr size_t m8_act_bytes(int K, int M) {
  return (size_t)(K / 128) * 4 * M * 64;
}
constexpr size_t m8_smem_bytes(int K, int M) {
  return m8_act_bytes(K, M) + (size_t)(K / 128) * 8 * 4 + 2 * kM8Warps * 4 * 32 * 4;
}

template <int BITS, bool ZP>
__global__ void __launch_bounds__(kM8Warps * 32, 2) gemv_m8_kernel(const M8Params p) {
  using GE = Geo<BITS>;
  constexpr int WPG = GE::WPG;
  constexpr int R = GE::WPG > 8 ? kM8Ring / 2 : kM8Ring;  // E4M3: twice the words per group
  extern __shared__ uint4 m8_smem[];
  const int G = p.K >> 7;
  uint8_t* act = reinterpret_cast<uint8_t*>(m8_smem);
  float* gsum = reinterpret_cast<float*>(act + m8_act_bytes(p.K, p.M));  // [G][8 tokens]
  float* red = gsum + G * 8;                                               // [2][warp][4][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t nblocks = (uint32_t)(p.N_pad >> 4);
  const int g0 = min(G, warp * p.gpw);
  const int cnt = min(G, g0 + p.gpw) - g0;  // this warp's groups per item (may be 0)
  const int nbat = (cnt + R - 1) / R;
  const int64_t gstride = (int64_t)nblocks * GE::BLK;  // bytes between groups of a block
  const uint32_t my_items =
      blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  pdl_launch_dependents();

  // register ring and the running pointers of the batch that refills it
  uint32_t wb[R][WPG];
  uint32_t sc[R];
  uint32_t zc[R];  // asymmetric INT4: BF16 128 + z of rows g and g + 8
  const uint8_t* rw = nullptr;
  const uint16_t* rs = nullptr;
  int rng = 0;                    // groups in the refilling batch
  uint32_t nx_it = 0;             // (item, chunk) of the refilling batch
  int nx_c = 0;
  auto point = [&](uint32_t it, int c) {
    rng = 0;
    if (it < my_items && c < nbat) {
      const uint32_t nb = blockIdx.x + it * gridDim.x;
      const int gb = g0 + R * c;
      rw = p.wp + ((int64_t)gb * nblocks + nb) * GE::BLK;
      rs = p.sp + (int64_t)gb * p.N_pad + nb * 16 + g;
      rng = min(R, g0 + cnt - gb);
    }
  };
  auto advance = [&]() {
    if (++nx_c == nbat) {
      nx_c = 0;
      ++nx_it;
    }
    point(nx_it, nx_c);
  };
  auto refill = [&](int j) {
    if (j < rng) {
      load_words<BITS>(rw + j * gstride, lane, wb[j]);
      const uint16_t* q = rs + (int64_t)j * p.N_pad;
      sc[j] = __byte_perm(__ldg(q), __ldg(q + 8), 0x5410);
      if constexpr (ZP) zc[j] = __byte_perm(__ldg(q + p.zplane), __ldg(q + p.zplane + 8), 0x5410);
    }
  };
  point(0, 0);
#pragma unroll
  for (int j = 0; j < R; ++j) refill(j);
  advance();

  // ---- activations and group sums (the previous kernel's output may be A).  Each warp
  // stages the chunks of its own groups (all loads first), so it only waits for itself.
  pdl_wait();
  {
    const int per_row = cnt * 16;      // 16-byte chunks of one row in this warp's groups
    const int nchunk = p.M * per_row;  // a multiple of 16
    for (int b0 = 0; b0 < nchunk; b0 += 32 * 8) {
      uint4 v[8];
      int rowv[8], k0v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = b0 + 32 * u + lane;
        const int row = p.M == 1 ? 0 : q / per_row;  // no division for single-token decode
        const int k0 = g0 * 128 + (q - row * per_row) * 8;
        rowv[u] = row;
        k0v[u] = k0;
        v[u] = q < nchunk ? __ldg(reinterpret_cast<const uint4*>(p.A + (int64_t)row * p.K + k0))
                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = b0 + 32 * u + lane;
        if (b0 + 32 * u >= nchunk) break;  // warp-uniform
        const int row = rowv[u], k0 = k0v[u];
        const int gg = k0 >> 7, st = (k0 >> 4) & 7, tt = (k0 >> 2) & 3;
        if (q < nchunk) {
          uint8_t* dst = act + ((gg * 4 + (st >> 1)) * p.M + row) * 64 + tt * 16 + (st & 1) * 8;
          *reinterpret_cast<uint2*>(dst) = make_uint2(v[u].x, v[u].y);
          *reinterpret_cast<uint2*>(dst + 16) = make_uint2(v[u].z, v[u].w);
        }
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float sum = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h)
          sum += __uint_as_float(w4[h] << 16) + __uint_as_float(w4[h] & 0xFFFF0000u);
        // the 16 chunks of one (row, group) sit in 16 consecutive lanes
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (q < nchunk && (lane & 15) == 0) gsum[gg * 8 + row] = sum;
      }
    }
    for (int i = lane; i < cnt * 8; i += 32)
      if ((i & 7) >= p.M) gsum[g0 * 8 + i] = 0.f;  // token columns past M (never stored)
  }
  __syncwarp();

  const uint32_t act_lane = smem_u32(act) + (uint32_t)(((g < p.M ? g : 0) * 4 + t) * 16);
  const uint32_t jj_stride = (uint32_t)p.M * 64;  // bytes between step pairs
  const uint32_t gsum_lane = smem_u32(gsum) + (uint32_t)(2 * t * 4);
  for (uint32_t it = 0; it < my_items; ++it) {
    const uint32_t nb = blockIdx.x + it * gridDim.x;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < nbat; ++c) {
      const int gb = g0 + R * c;
      const int ng = min(R, g0 + cnt - gb);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (j < ng) {
          if (j > 0) refill(j - 1);  // slot j - 1 is free: next batch's group j - 1
          const int gg = gb + j;
          const uint32_t ab = act_lane + (uint32_t)gg * 4 * jj_stride;
          float pr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint4 x = lds128(ab + jj * jj_stride);
            uint32_t a[4];
            biased_all<BITS>(wb[j], 2 * jj, a);
            mma_bf16_16816(pr, a, x.x, x.y);
            biased_all<BITS>(wb[j], 2 * jj + 1, a);
            mma_bf16_16816(pr, a, x.z, x.w);
          }
          const uint2 sm2 = lds64(gsum_lane + (uint32_t)gg * 32);
          const float sm0 = __uint_as_float(sm2.x), sm1 = __uint_as_float(sm2.y);
          const float s_lo = __uint_as_float(sc[j] << 16);
          const float s_hi = __uint_as_float(sc[j] & 0xFFFF0000u);
          // the excess of rows g and g + 8: 128 + excess, or (asymmetric) 128 + z
          const float b_lo = ZP ? __uint_as_float(zc[j] << 16) : GE::BIAS;
          const float b_hi = ZP ? __uint_as_float(zc[j] & 0xFFFF0000u) : GE::BIAS;
          acc[0] = fmaf(s_lo, fmaf(-b_lo, sm0, pr[0]), acc[0]);
          acc[1] = fmaf(s_lo, fmaf(-b_lo, sm1, pr[1]), acc[1]);
          acc[2] = fmaf(s_hi, fmaf(-b_hi, sm0, pr[2]), acc[2]);
          acc[3] = fmaf(s_hi, fmaf(-b_hi, sm1, pr[3]), acc[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (j >= ng - 1) refill(j);  // slots not refilled inside the loop
      advance();
    }

    // split-K reduction over the CTA's warps, fixed order; one barrier per item
    float* rb = red + (it & 1) * (kM8Warps * 128);
#pragma unroll
    for (int i = 0; i < 4; ++i) rb[(warp * 4 + i) * 32 + lane] = acc[i];
    __syncthreads();
    for (int o = threadIdx.x; o < 16 * p.M; o += kM8Warps * 32) {
      const int nl = o & 15, m = o >> 4;
      const int l = (nl & 7) * 4 + (m >> 1), i = (nl >> 3) * 2 + (m & 1);
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kM8Warps; ++w2) v += rb[(w2 * 4 + i) * 32 + l];
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

template <int BITS, bool ZP>
qw_status launch_m8_variant(const M8Params& p, cudaStream_t st) {
  auto kern = gemv_m8_kernel<BITS, ZP>;
  const size_t smem = m8_smem_bytes(p.K, p.M);
  // one attribute call sized for the largest staging this kernel is sent (see the dispatch)
  static const cudaError_t attr = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kM8MaxSmem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kM8Warps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t items = p.N_pad / 16;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, (unsigned)grid, kM8Warps * 32, smem, st, p);
}

// ---------------------------------------------------------------- single-token decode, INT4
// M = 1 over symmetric INT4 weights: the same packed words and (16-row block, scale group)
// work as gemv_m8_kernel, rebuilt around fewer issued instructions per 1 KiB group.
//  - FP16 operands.  With the FP16 pattern 0x6400 (the number 1024, unit in the last place
//    1) one masking op turns the nibbles at bits 0-3 and 16-19 of a word into 1024 + u and
//    the nibbles at bits 4-7 and 20-23, left in place, into 1024 + 16 u: one shift per four
//    fragment registers instead of three.  In the packed words the in-place nibbles are
//    exactly the registers of rows g + 8, so rows g hold 1032 + q and rows g + 8 hold
//    16 (72 + q) (u = q + 8): the two halves of a block differ by a row factor that goes
//    out with the excess after the MMA.
//  - Activations are staged once per CTA as FP16, each scale group multiplied by the power
//    of two 2^f that puts its largest magnitude in [2^14, 2^15).  That is exact (a BF16
//    value times a power of two is an FP16 number) except for values 2^28 or more below the
//    group maximum, which round to FP16 subnormals.  Beside each group sit its constants
//    (2^-f, 2^-f / 16, -1032 * 2^-f * S, -72 * 2^-f * S), S the sum of its FP16 values,
//    so that per group two FMAs remove the excess and two apply the weight scales:
//      sum_k q a = 2^-f (P_g - 1032 S)   (rows g),   2^-f (P_g+8 / 16 - 72 S)   (rows g + 8).
//  - Only token 0 exists: the lanes with t = 0 carry the outputs (fragment registers 0 and
//    2); the other columns of the MMA are never read.
// A CTA's warps split the scale groups of a block (gpw groups each, a whole number of ring
// batches) and meet in shared memory once per block; CTAs take blocks round-robin.  Each
// thread may use 128 registers: measured on GB300 (14336 x 4096), the schedule the compiler
// builds with that budget streams 1.25x faster than the same code held to 64 or 80 registers
// (which would let more CTAs share an SM), and splitting a block's K over several CTAs (slice
// sums in the workspace, last arrival adds them) was slower at every shape tried.
constexpr int kDecRing = 4;                 // groups per warp in flight (register ring)
constexpr int kDecMaxWarps = 16;            // 512 threads x 128 registers fill an SM
constexpr int kDecMaxGpw = 16;              // groups per warp the staging is sized for
constexpr size_t kDecMaxSmem = 100 * 1024;  // largest staging sent to the decode kernel

struct DecParams {
  const uint8_t* wp;
  const uint16_t* sp;
  const uint16_t* A;
  const uint16_t* bias;
  const float* scale2;  // second-level scales [N_pad] or null
  uint16_t* C;
  int32_t N, N_pad, K;
  int32_t gpw;          // scale groups per warp (a multiple of kDecRing, at most kDecMaxGpw)
  // K split across CTAs (S > 1): a cluster of S CTAs takes one block, CTA rank r its slice r
  // (gs = warps x gpw groups); rank 0 adds the slice sums in rank order through distributed
  // shared memory and applies scale2 and bias
  int32_t S, gs;
};

// shared memory: FP16 activations [group][step pair][t][16 B] and the group constants
// (float4), then the reduction [2][warp][16] floats (and, split, the CTA's 16 slice sums)
__host__ __device__ constexpr size_t dec_smem_bytes(int groups, int warps, bool split = false) {
  return (size_t)groups * (256 + 16) + 2 * (size_t)warps * 16 * 4 + (split ? 16 * 4 : 0);
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// SPLIT: the cluster form (one slice of one block per CTA); otherwise whole blocks per CTA
// (compiled without any of the split's code).
template <int BITS, int R, bool SPLIT>
__global__ void __launch_bounds__(kDecMaxWarps * 32, 1) gemv_decode_kernel(const DecParams p) {
  using GE = Geo<BITS>;
  constexpr int WPG = GE::WPG;        // packed words per lane and group
  // FP16 operands for INT4 (the in-place nibble trick), E2M1 (hardware conversion) and
  // INT1 (sign pairs); BF16 for INT3 and INT2
  constexpr bool F16 = BITS == 4 || BITS == kBitsFp4 || BITS == 1;
  extern __shared__ uint4 dec_smem[];
  const int warps = (int)(blockDim.x >> 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.K >> 7;
  const uint32_t nblocks = (uint32_t)(p.N_pad >> 4);
  const int S = SPLIT ? p.S : 1;
  const uint32_t my_items =
      S > 1 ? (blockIdx.x < nblocks * (uint32_t)S ? 1u : 0u)
            : (blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0);
  // the warp's first group (its slice's first group plus its share)
  const int wg0 = (S > 1 ? (int)(blockIdx.x % (uint32_t)S) * p.gs : 0) + warp * p.gpw;
  auto block_of = [&](uint32_t it) -> uint32_t {
    return S > 1 ? blockIdx.x / (uint32_t)S : blockIdx.x + it * gridDim.x;
  };
  const uint32_t gstride = nblocks * (uint32_t)GE::BLK;  // bytes between groups of a block
  uint8_t* act = reinterpret_cast<uint8_t*>(dec_smem);  // [G][4][4][16 B]
  // staged groups: the whole K, or the CTA's slice (indexed from its first group gbase)
  const int gbase = S > 1 ? (int)(blockIdx.x % (uint32_t)S) * p.gs : 0;
  const int gstaged = S > 1 ? p.gs : G;
  float4* gconst = reinterpret_cast<float4*>(act + (size_t)gstaged * 256);
  float* red = reinterpret_cast<float*>(gconst + gstaged);  // [2][warps][16]
  float* cpart = red + 2 * warps * 16;                        // split: this CTA's slice sums

  pdl_launch_dependents();

  // ---- register ring: the packed words and scales of R consecutive groups of an item
  uint32_t wb[R][WPG];
  uint32_t sl_[R], sh_[R];  // BF16 scale bits of rows g and g + 8
  // byte offset of (item it, the warp's first group) and its scale index
  auto unit_w = [&](uint32_t it) {
    return block_of(it) * (uint32_t)GE::BLK + (uint32_t)wg0 * gstride;
  };
  auto unit_s = [&](uint32_t it) {
    return (uint32_t)wg0 * (uint32_t)p.N_pad + block_of(it) * 16u + (uint32_t)g;
  };
  auto load = [&](int r, uint32_t woff, uint32_t soff) {
    load_words<BITS>(p.wp + woff, lane, wb[r]);
    sl_[r] = __ldg(p.sp + soff);
    sh_[r] = __ldg(p.sp + soff + 8);
  };
  // weights and scales are never written by the kernel before this one on the stream (a
  // documented precondition): the first batch streams before the wait
  if (my_items > 0) {
    const uint32_t w0 = unit_w(0), s0 = unit_s(0);
#pragma unroll
    for (int r = 0; r < R; ++r)
      load(r, w0 + (uint32_t)r * gstride, s0 + (uint32_t)r * (uint32_t)p.N_pad);
  }

  // ---- activations of the warp's groups as B fragments, and their constants.  A half warp
  // covers one group; up to four chunks per lane load before any is converted.
  pdl_wait();
  {
    constexpr int kBatch = 4;
    const int nchunk = p.gpw * 16;         // 16-byte chunks (8 BF16) of the warp's groups
    const int iters = (nchunk + 31) >> 5;  // per lane
    for (int u0 = 0; u0 < iters; u0 += kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (u0 + u < iters) {
          const int q = lane + 32 * (u0 + u);
          const int gl = wg0 + (q >> 4), c = q & 15;  // group, chunk
          v[u] = q < nchunk ? __ldg(reinterpret_cast<const uint4*>(p.A + gl * 128 + c * 8))
                            : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (u0 + u < iters) {
          const int q = lane + 32 * (u0 + u);
          const int gl = wg0 + (q >> 4), c = q & 15;
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          uint32_t h[4];
          float sum = 0.f;
          int f = 0;
          if constexpr (F16) {
            // group maximum magnitude: BF16 magnitudes order like their bit patterns
            uint32_t m = __vmaxu2(__vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                                  __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu));
            m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            const int ex = (int)(m >> 7);  // biased exponent of the maximum
            f = min(141 - ex, 126);        // 2^f puts the maximum in [2^14, 2^15)
            const float up = __uint_as_float((uint32_t)(127 + f) << 23);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              h[i] = f16x2_of(__uint_as_float(w4[i] << 16) * up,
                              __uint_as_float(w4[i] & 0xFFFF0000u) * up);
              const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
              sum += back.x + back.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              h[i] = w4[i];
              sum += __uint_as_float(w4[i] << 16) + __uint_as_float(w4[i] & 0xFFFF0000u);
            }
          }
          // chunk c holds k = 8c .. 8c + 7: step c / 2, lanes t = 2 (c & 1) and 2 (c & 1) + 1
          if (q < nchunk) {
            uint8_t* dst =
                act + (((gl - gbase) * 4 + (c >> 2)) * 4 + 2 * (c & 1)) * 16 + ((c >> 1) & 1) * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(h[0], h[1]);
            *reinterpret_cast<uint2*>(dst + 16) = make_uint2(h[2], h[3]);
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
          if ((lane & 15) == 0 && q < nchunk) {
            if constexpr (BITS == 4) {
              const float e = __uint_as_float((uint32_t)(127 - f) << 23);  // 2^-f
              gconst[gl - gbase] = make_float4(e, e * 0.0625f, -1032.f * e * sum, -72.f * e * sum);
            } else if constexpr (F16) {
              const float e = __uint_as_float((uint32_t)(127 - f) << 23);  // 2^-f, no excess
              gconst[gl - gbase] = make_float4(e, e, 0.f, 0.f);
            } else {
              // biased codes 128 + excess + q on both row halves
              gconst[gl - gbase] = make_float4(1.f, 1.f, -GE::BIAS * sum, -GE::BIAS * sum);
            }
          }
        }
    }
  }
  __syncwarp();

  const uint32_t act_lane = smem_u32(act) + (uint32_t)((wg0 - gbase) * 256 + t * 16);
  const uint32_t const_base = smem_u32(gconst) + (uint32_t)(wg0 - gbase) * 16;
  for (uint32_t it = 0; it < my_items; ++it) {
    const uint32_t nb = block_of(it);
    const uint32_t wit = unit_w(it), sit = unit_s(it);
    const uint32_t wnx = unit_w(it + 1), snx = unit_s(it + 1);
    const bool has_next = it + 1 < my_items;
    float acc_lo = 0.f, acc_hi = 0.f;
    for (int jb = 0; jb < p.gpw; jb += R) {
      // the ring's next batch: (it, jb + R ..) or the next item's first R groups
      const bool same = jb + R < p.gpw;
      const uint32_t nw = same ? wit + (uint32_t)(jb + R) * gstride : wnx;
      const uint32_t ns = same ? sit + (uint32_t)(jb + R) * (uint32_t)p.N_pad : snx;
      const bool more = same || has_next;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = jb + r;
        const uint32_t ab = act_lane + (uint32_t)j * 256u;
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint4 x = lds128(ab + jj * 64);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t a[4];
            if constexpr (BITS == 4) {
              const uint32_t wv = wb[r][2 * jj + h2];
              const uint32_t ws = wv >> 8;
              a[0] = and_or(wv, 0x000F000Fu, 0x64006400u);
              a[1] = and_or(wv, 0x00F000F0u, 0x64006400u);
              a[2] = and_or(ws, 0x000F000Fu, 0x64006400u);
              a[3] = and_or(ws, 0x00F000F0u, 0x64006400u);
              mma_f16_16816(pr, a, h2 ? x.z : x.x, h2 ? x.w : x.y);
            } else if constexpr (BITS == kBitsFp4) {
              e2m1x8_to_f16x2(wb[r][2 * jj + h2], a);  // byte i of the word is register i
              mma_f16_16816(pr, a, h2 ? x.z : x.x, h2 ? x.w : x.y);
            } else if constexpr (BITS == 1) {
              const int s2 = 2 * jj + h2;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                a[q] = int1_pair(wb[r][s2 >> 2], 4 * (s2 & 3) + q, 0x3C003C00u);
              mma_f16_16816(pr, a, h2 ? x.z : x.x, h2 ? x.w : x.y);
            } else {
              biased_all<BITS>(wb[r], 2 * jj + h2, a);
              mma_bf16_16816(pr, a, h2 ? x.z : x.x, h2 ? x.w : x.y);
            }
          }
        }
        float4 c4;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(c4.x), "=f"(c4.y), "=f"(c4.z), "=f"(c4.w)
                     : "r"(const_base + (uint32_t)j * 16u));
        const float s_lo = __uint_as_float(sl_[r] << 16);
        const float s_hi = __uint_as_float(sh_[r] << 16);
        acc_lo = fmaf(s_lo, fmaf(pr[0], c4.x, c4.z), acc_lo);
        acc_hi = fmaf(s_hi, fmaf(pr[2], c4.y, c4.w), acc_hi);
        // the slot is free: load the ring's next group into it
        if (more) load(r, nw + (uint32_t)r * gstride, ns + (uint32_t)r * (uint32_t)p.N_pad);
      }
    }

    // ---- the CTA's warps meet: fixed-order sum of their 16 rows; one barrier per item
    float* rb = red + (it & 1) * (warps * 16);
    if (t == 0) {
      rb[warp * 16 + g] = acc_lo;
      rb[warp * 16 + g + 8] = acc_hi;
    }
    __syncthreads();
    if (warp == 0 && lane < 16) {
      float v = 0.f;
      for (int w2 = 0; w2 < warps; ++w2) v += rb[w2 * 16 + lane];
      const int n = (int)nb * 16 + lane;
      if (S > 1) {
        cpart[lane] = v;  // this slice's sums, read by the cluster's rank 0 below
      } else if (n < p.N) {
        if (p.scale2) v *= __ldg(p.scale2 + n);
        if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + n) << 16);
        __nv_bfloat16 hb = __float2bfloat16_rn(v);
        p.C[n] = *reinterpret_cast<uint16_t*>(&hb);
      }
    }
  }
  if (S > 1) {
    // the cluster's S CTAs hold one block's slice sums: rank 0 adds them in rank order
    // (deterministic) from the CTAs' shared memory; every thread of every CTA takes both
    // cluster barriers (each CTA has exactly one item), the second keeping the peers'
    // shared memory alive until rank 0 has read it
    cluster_sync();
    if (cluster_ctarank() == 0 && warp == 0 && lane < 16) {
      const uint32_t own = smem_u32(cpart + lane);
      float v = 0.f;
      for (int r = 0; r < S; ++r) v += ld_shared_cluster_f32(mapa_shared(own, (uint32_t)r));
      const int n = (int)(blockIdx.x / (uint32_t)S) * 16 + lane;
      if (n < p.N) {
        if (p.scale2) v *= __ldg(p.scale2 + n);
        if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + n) << 16);
        __nv_bfloat16 hb = __float2bfloat16_rn(v);
        p.C[n] = *reinterpret_cast<uint16_t*>(&hb);
      }
    }
    cluster_sync();
  }
}

// How a decode call is split: warps per CTA (each streaming gpw groups of every block the
// CTA takes) and resident CTAs per SM.
struct DecPlan {
  int warps = 0, gpw = 0, per_sm = 0;  // warps == 0: no plan (the shape goes to gemv_m8_kernel)
  int S = 1;                           // K slices per block, one CTA each (1: no split)
};
constexpr int kDecMaxSlices = 8;  // a slice per CTA of a cluster (portable cluster size)

// The split with the most warps per SM (16 at 128 registers each), ties to more warps per
// CTA (fewer blocks per SM to wait on); measured best at K = 4096 (8 warps x 4 groups, two
// CTAs per SM) and K = 14336 (14 warps x 8 groups, one CTA per SM).
DecPlan decode_plan(int K) {
  DecPlan best;
  const int G = K / 128;
  for (int warps = 1; warps <= kDecMaxWarps; ++warps) {
    if (G % warps) continue;
    const int gpw = G / warps;
    if (gpw % kDecRing || gpw > kDecMaxGpw) continue;
    if (dec_smem_bytes(G, warps) > kDecMaxSmem) continue;
    const int per_sm = kDecMaxWarps / warps;
    const int score = warps * per_sm;
    if (best.warps == 0 || score > best.warps * best.per_sm ||
        (score == best.warps * best.per_sm && warps > best.warps)) {
      best.warps = warps;
      best.gpw = gpw;
      best.per_sm = per_sm;
    }
  }
  return best;
}

// Shapes with fewer 16-row blocks than SMs leave SMs idle when every CTA takes whole blocks:
// split each block's K into S slices (a cluster of S CTAs, one slice each, the slice sums
// added through distributed shared memory) when that puts CTAs on more SMs and fills more of their warp slots over the waves (CTAs
// of `warps` warps, 16 / warps of them per SM).  Measured on GB300 (M = 1, INT4): 1024 x
// 32768 and 512 x 16384 ran at half a plain streaming read unsplit.
DecPlan decode_plan_for(int K, int64_t nblocks, int sms) {
  DecPlan best = decode_plan(K);
  // measured: a split pays at 32 blocks x 128 groups and 64 x 256 (the CTAs' streams are
  // long enough to cover the cluster's set-up), not at 64 x 64 or 128 x 64..128
  if (best.warps == 0 || 2 * nblocks > sms || K / 128 < 128) return best;
  const int G = K / 128;
  auto score = [&](int64_t ctas, int warps, int per_sm) {
    const int64_t slots = (int64_t)sms * per_sm;
    const int64_t waves = (ctas + slots - 1) / slots;
    const double busy = (double)(ctas < sms ? ctas : sms) / sms;  // SMs with a CTA
    return busy + (double)(ctas * warps) / (double)(waves * sms * kDecMaxWarps);
  };
  double best_score = score(nblocks, best.warps, best.per_sm);
  for (int S = 2; S <= kDecMaxSlices; ++S) {
    if (G % S) continue;
    const int gs = G / S;
    for (int warps = 1; warps <= kDecMaxWarps; ++warps) {
      if (gs % warps) continue;
      const int gpw = gs / warps;
      if (gpw % kDecRing || gpw > kDecMaxGpw) continue;
      if (dec_smem_bytes(gs, warps, true) > kDecMaxSmem) continue;
      const int per_sm = kDecMaxWarps / warps;
      const double sc = score(nblocks * S, warps, per_sm);
      if (sc > best_score + 1e-9) {
        best.warps = warps;
        best.gpw = gpw;
        best.per_sm = per_sm;
        best.S = S;
        best_score = sc;
      }
    }
  }
  return best;
}

template <int BITS>
qw_status launch_decode_variant(const qw_packed_desc& d, const DecPlan& pl, const DecParams& p,
                                cudaStream_t st);

qw_status launch_decode_plan(const qw_packed_desc& d, const DecPlan& pl, const void* w_packed,
                             const void* s_packed, const void* A, const void* bias,
                             const float* scale2, void* C, cudaStream_t st) {
  if (pl.warps == 0) return QW_ERR_UNSUPPORTED;
  DecParams p{};
  p.wp = static_cast<const uint8_t*>(w_packed);
  p.sp = static_cast<const uint16_t*>(s_packed);
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.scale2 = scale2;
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.gpw = pl.gpw;
  p.S = pl.S;
  p.gs = pl.warps * pl.gpw;
  switch (d.wfmt) {
    case QW_W_INT4_G128_BF16: return launch_decode_variant<4>(d, pl, p, st);
    case QW_W_INT3_G128_BF16: return launch_decode_variant<3>(d, pl, p, st);
    case QW_W_INT2_G128_BF16: return launch_decode_variant<2>(d, pl, p, st);
    case QW_W_INT1_G128_BF16: return launch_decode_variant<1>(d, pl, p, st);
    default: return launch_decode_variant<kBitsFp4>(d, pl, p, st);
  }
}

qw_status launch_decode(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                        const void* A, const void* bias, const float* scale2, void* C,
                        cudaStream_t st) {
  const DecPlan pl = decode_plan_for(d.K, d.N_pad / 16, device_sm_count());
  const qw_status s = launch_decode_plan(d, pl, w_packed, s_packed, A, bias, scale2, C, st);
  // a cluster of pl.S CTAs that cannot be placed: the unsplit schedule
  if (s == QW_ERR_UNSUPPORTED && pl.S > 1)
    return launch_decode_plan(d, decode_plan(d.K), w_packed, s_packed, A, bias, scale2, C, st);
  return s;
}

template <int BITS>
qw_status launch_decode_variant(const qw_packed_desc& d, const DecPlan& pl, const DecParams& p,
                                cudaStream_t st) {
  auto kern = gemv_decode_kernel<BITS, kDecRing, false>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecMaxSmem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  const int64_t items = d.N_pad / 16;
  if (pl.S > 1) {
    auto skern = gemv_decode_kernel<BITS, kDecRing, true>;
    static const cudaError_t sattr =
        cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecMaxSmem);
    if (sattr != cudaSuccess) return QW_ERR_CUDA;
    const size_t smem = dec_smem_bytes(p.gs, pl.warps, true);
    // one cluster of S CTAs per block, launched as a programmatic dependent like the rest
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(items * pl.S));
    cfg.blockDim = dim3((unsigned)(pl.warps * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)pl.S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, skern, &cfg) != cudaSuccess || clusters < 1) {
      (void)cudaGetLastError();
      return QW_ERR_UNSUPPORTED;
    }
    if (cudaLaunchKernelEx(&cfg, skern, p) != cudaSuccess) return QW_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
  }
  const size_t smem = dec_smem_bytes(d.K / 128, pl.warps);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, pl.warps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  if (per_sm > pl.per_sm) per_sm = pl.per_sm;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, (unsigned)grid, pl.warps * 32, smem, st, p);
}

// Dense single-token symmetric INT4 / INT3 / INT2 / INT1 and E2M1 calls the decode kernel takes (32-bit
// offsets into the packed buffers; a split with a whole number of ring batches per warp).
bool decode_eligible(const qw_packed_desc& d, const void* A) {
  if (d.wfmt != QW_W_INT4_G128_BF16 && d.wfmt != QW_W_INT3_G128_BF16 &&
      d.wfmt != QW_W_INT2_G128_BF16 && d.wfmt != QW_W_INT1_G128_BF16 &&
      d.wfmt != QW_W_FP4E2M1_G128_BF16)
    return false;
  if ((reinterpret_cast<uintptr_t>(A) & 15) != 0) return false;
  if (d.w_expert_stride >= (uint64_t(1) << 32)) return false;
  if ((uint64_t)(d.K / 128) * (uint64_t)d.N_pad >= (uint64_t(1) << 31)) return false;
  return decode_plan(d.K).warps != 0;
}

// ---------------------------------------------------------------- TMA-ring kernel
constexpr int kStageGroups = 8;  // scale groups per stage (one TMA copy)

// Shape of a TMA-ring launch: consumer warps, ring stages, resident CTAs per SM.
template <int CONS_, int STAGES_, int CTAS_>
struct Ring {
  static constexpr int CONS = CONS_, STAGES = STAGES_, CTAS = CTAS_;
  static constexpr int THREADS = (CONS + 1) * 32;
  static constexpr int GPC = kStageGroups / CONS;  // groups of a stage per consumer
  static_assert(kStageGroups % CONS == 0, "consumers split a stage evenly");
};
// grouped (MoE) calls: many short items, several CTAs per SM
using GroupedRing = Ring<4, 4, 4>;
// E4M3 weights: 16 KiB stages, three CTAs per SM fit
using GroupedRing8 = Ring<4, 4, 3>;

template <int BITS, bool ZP>
struct TmaGeo {
  static constexpr int BLK = wna16_block_bytes(BITS);  // one 16 x 128 block
  static constexpr int W_STAGE = kStageGroups * BLK;
  static constexpr int S_STAGE = kStageGroups * 16 * 2;  // BF16 scales of 16 rows x 8 groups
  // asymmetric INT4: the same rows and groups of BF16 128 + z follow the scales
  static constexpr int STAGE = W_STAGE + S_STAGE * (ZP ? 2 : 1);
  static constexpr bool FP = Geo<BITS>::FP;  // values decoded as they are: no excess
  static constexpr float BIAS = Geo<BITS>::BIAS;
};

template <int BITS, int MCH, class R, bool ZP>
constexpr size_t tma_smem_bytes() {
  return 128 + (size_t)R::STAGES * TmaGeo<BITS, ZP>::STAGE + 2 * 8 * R::STAGES +
         (size_t)R::CONS * MCH * 128 * 4 + 16;
}

struct TmaParams {
  const uint16_t* A;
  const uint16_t* bias;
  uint16_t* C;
  int32_t N, N_pad, K;
  int64_t M;             // dense rows (unused when grouped)
  const int32_t* queue;  // grouped tile queue or null
  int32_t* err;
  const float* scale2;   // second-level scales [E][N_pad] or null
};

// One work item = (expert e, 16-row block nb, token rows [rb, re)), re - rb <= 8 * MCH.
template <int MCH>
__device__ __forceinline__ void tma_item_of(const TmaParams& p, uint32_t item, uint32_t nblocks, int& e,
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

template <int BITS, int MCH, class R, bool ZP>
__global__ void __launch_bounds__(R::THREADS, R::CTAS)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmZ, const TmaParams p) {
  using GE = TmaGeo<BITS, ZP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + R::STAGES * GE::STAGE);
  uint64_t* empty = full + R::STAGES;
  float* red = reinterpret_cast<float*>(empty + R::STAGES);  // [consumer][MCH][4][32]
  volatile int* flags = reinterpret_cast<volatile int*>(red + R::CONS * MCH * 128);
  // flags[0]: abort; flags[1]: abort as seen at the end of the current item

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < R::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], R::CONS);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const uint32_t nblocks = (uint32_t)(p.N_pad / 16);
  const int G = p.K / 128;
  const int chunks = (G + kStageGroups - 1) / kStageGroups;  // stages per item
  // Work items.  The tile queue (and so its count) is the previous kernel's output: every
  // role reads it only after its griddepcontrol.wait.  Item counts stay below 2^31
  // (checked on the host): 32-bit index arithmetic.
  auto count_items = [&]() -> uint32_t {
    return p.queue ? (uint32_t)__ldg(p.queue) * nblocks
                   : nblocks * (uint32_t)((p.M + 8 * MCH - 1) / (8 * MCH));
  };
  volatile int* abort_flag = flags;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmS);
      // dense calls stream weights at once; the tile queue is the previous kernel's output
      if (p.queue) pdl_wait();
      const uint32_t n_items = count_items();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // per stage: used, phase of its last copy
      bool ok = true;
      for (uint32_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        int e, nb;
        int64_t rb, re;
        tma_item_of<MCH>(p, item, nblocks, e, nb, rb, re);
        for (int c = 0; c < chunks; ++c) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = smem_u32(ring + stage * GE::STAGE);
          mbar_arrive_expect_tx(&full[stage], GE::STAGE);
          tma_load_4d(dst, &tmW, &full[stage], 0, nb, c * kStageGroups, e);
          tma_load_3d(dst + GE::W_STAGE, &tmS, &full[stage], nb * 16, c * kStageGroups, e);
          if constexpr (ZP)
            tma_load_3d(dst + GE::W_STAGE + GE::S_STAGE, &tmZ, &full[stage], nb * 16,
                        c * kStageGroups, e);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == R::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // let every copy issued here land before the CTA's shared memory goes away
      for (int s = 0; s < R::STAGES; ++s)
        if (issued & (1u << s)) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], (issued_phase >> s) & 1u))
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int g = lane >> 2, t = lane & 3;
    pdl_wait();  // activations, queue, bias and output
    const uint32_t n_items = count_items();
    const uint32_t ring_base = smem_u32(ring);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (uint32_t item = blockIdx.x; item < n_items; item += gridDim.x) {
      int e, nb;
      int64_t rb, re;
      tma_item_of<MCH>(p, item, nblocks, e, nb, rb, re);
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
        for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;

      for (int ch = 0; ch < chunks; ++ch) {
        if (ok && !mbar_wait(&full[stage], phase, abort_flag, p.err)) ok = false;
        if (ok) {
          const uint32_t sbase = ring_base + stage * GE::STAGE;
#pragma unroll
          for (int jj = 0; jj < R::GPC; ++jj) {
            const int j = R::GPC * cw + jj;  // group within the stage
            const int gg = ch * kStageGroups + j;
            if (gg < G) {
              const uint32_t blk = sbase + j * GE::BLK;
              uint32_t w[BITS == 8 ? 16 : 8];
              if constexpr (BITS == 4 || BITS == kBitsFp4) {
                const uint4 v0 = lds128(blk + lane * 32), v1 = lds128(blk + lane * 32 + 16);
                w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
                w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
              } else if constexpr (BITS == 1) {
                const uint2 v = lds64(blk + lane * 8);
                w[0] = v.x; w[1] = v.y;
                w[2] = w[3] = w[4] = w[5] = w[6] = w[7] = 0;
              } else if constexpr (BITS == 2) {
                const uint4 v = lds128(blk + lane * 16);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
                w[4] = w[5] = w[6] = w[7] = 0;
              } else if constexpr (BITS == 8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint4 v = lds128(blk + lane * 64 + 16 * i);
                  w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                }
              } else {
                const uint4 lo = lds128(blk + lane * 16);
                const uint2 hi = lds64(blk + 512 + lane * 8);
                w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
                w[4] = hi.x; w[5] = hi.y; w[6] = 0; w[7] = 0;
              }
              // BF16 scales of rows g (low half) and g + 8 (high half) of this group
              const uint32_t srow = sbase + GE::W_STAGE + j * 32;
              const uint32_t sc = __byte_perm(lds32(srow + (g & ~1) * 2),
                                              lds32(srow + ((g + 8) & ~1) * 2),
                                              (g & 1) ? 0x7632 : 0x5410);
              const float s_lo = __uint_as_float(sc << 16);
              const float s_hi = __uint_as_float(sc & 0xFFFF0000u);
              // the excess of rows g and g + 8: 128 + excess, or (asymmetric) 128 + z
              float b_lo = GE::BIAS, b_hi = GE::BIAS;
              if constexpr (ZP) {
                const uint32_t zrow = srow + GE::S_STAGE;
                const uint32_t zc = __byte_perm(lds32(zrow + (g & ~1) * 2),
                                                lds32(zrow + ((g + 8) & ~1) * 2),
                                                (g & 1) ? 0x7632 : 0x5410);
                b_lo = __uint_as_float(zc << 16);
                b_hi = __uint_as_float(zc & 0xFFFF0000u);
              }
              const int koff = gg * 128;
              if constexpr (MCH <= 2) {
                const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
                float pr[MCH][4], sm[MCH][4];
#pragma unroll
                for (int c = 0; c < MCH; ++c)
#pragma unroll
                  for (int i = 0; i < 4; ++i) pr[c][i] = sm[c][i] = 0.f;
#pragma unroll
                for (int st = 0; st < 8; ++st) {
                  uint32_t a[4];
                  decode_step<BITS>(w, st, a);
#pragma unroll
                  for (int c = 0; c < MCH; ++c) {
                    const uint2 x = __ldg(reinterpret_cast<const uint2*>(arow[c] + koff + 16 * st));
                    mma_bf16_16816(pr[c], a, x.x, x.y);
                    if constexpr (!GE::FP) mma_bf16_16816(sm[c], ones, x.x, x.y);
                  }
                }
#pragma unroll
                for (int c = 0; c < MCH; ++c)
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    acc[c][i] = fmaf(i < 2 ? s_lo : s_hi, fmaf(i < 2 ? -b_lo : -b_hi, sm[c][i], pr[c][i]),
                                     acc[c][i]);
              } else {
                static_assert(!ZP, "the asymmetric format runs with at most 16 token rows");
                const uint32_t bias2 = 0x43004300u + 0x10001u * (1u << (BITS - 1));  // BF16 pair of BIAS
                float part[MCH][4];
#pragma unroll
                for (int c = 0; c < MCH; ++c)
#pragma unroll
                  for (int i = 0; i < 4; ++i) part[c][i] = 0.f;
#pragma unroll
                for (int st = 0; st < 8; ++st) {
                  uint32_t a[4];
                  decode_step<BITS>(w, st, a);
                  if constexpr (!GE::FP) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) a[r] = bf16x2_sub(a[r], bias2);  // exact
                  }
#pragma unroll
                  for (int c = 0; c < MCH; ++c) {
                    const uint2 x = __ldg(reinterpret_cast<const uint2*>(arow[c] + koff + 16 * st));
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
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);  // this warp is done with the stage
        }
        if (++stage == R::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }

      // ---------------------------------------------------------- reduce and store
#pragma unroll
      for (int c = 0; c < MCH; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[((cw * MCH + c) * 4 + i) * 32 + lane] = acc[c][i];
      asm volatile("bar.sync 1, %0;" ::"r"(R::CONS * 32) : "memory");  // consumers only
      if (threadIdx.x == 32) flags[1] = *abort_flag;
      for (int o = threadIdx.x - 32; o < MCH * 128; o += R::CONS * 32) {
        float v = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < R::CONS; ++w2) v += red[w2 * MCH * 128 + o];
        // fragment (lane l, register i) -> weight row gq + 8 (i >> 1), token 2 tt + (i & 1)
        const int c = o >> 7, i = (o >> 5) & 3, l = o & 31;
        const int gq = l >> 2, tt = l & 3;
        const int n = nb * 16 + gq + 8 * (i >> 1);
        const int64_t r = rb + 8 * c + 2 * tt + (i & 1);
        if (n < p.N && r < re) {
          if (p.scale2) v *= __ldg(p.scale2 + (int64_t)e * p.N_pad + n);
          if (p.bias) v += __uint_as_float((uint32_t)__ldg(p.bias + (int64_t)e * p.N + n) << 16);
          __nv_bfloat16 h = __float2bfloat16_rn(v);
          p.C[r * p.N + n] = *reinterpret_cast<uint16_t*>(&h);
        }
      }
      asm volatile("bar.sync 1, %0;" ::"r"(R::CONS * 32) : "memory");
      if (flags[1]) break;  // one snapshot for all consumers: they stop together
    }
  }
  __syncthreads();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

template <int BITS, int MCH, class R, bool ZP>
qw_status launch_tma_variant(const CUtensorMap& tmW, const CUtensorMap& tmS, const CUtensorMap& tmZ,
                             const TmaParams& p, int64_t size_items, cudaStream_t st) {
  auto kern = gemv_tma_kernel<BITS, MCH, R, ZP>;
  const size_t smem = tma_smem_bytes<BITS, MCH, R, ZP>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, R::THREADS, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  if (grid > size_items) grid = size_items;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, (unsigned)grid, R::THREADS, smem, st, tmW, tmS, tmZ, p);
}

// Token rows per item / 8: the dispatcher sends dense calls of at most 16 rows and grouped
// calls averaging fewer than 16 rows per expert here (busier experts get more tiles).
int mch_for_rows(int64_t rows) { return rows <= 8 ? 1 : 2; }

int mch_for(const qw_packed_desc& d, int64_t rows, bool grouped) {
  if (!grouped) return mch_for_rows(rows);
  return mch_for_rows((rows + d.E - 1) / d.E);  // average rows per expert
}

// Dense calls of at most 8 token rows whose activations fit the staging buffer.
qw_status launch_dense_m8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                          const void* A, const void* bias, const float* scale2, void* C, int M,
                          cudaStream_t st) {
  const int G = d.K / kIntGroup;
  M8Params p{};
  p.wp = static_cast<const uint8_t*>(w_packed);
  p.sp = static_cast<const uint16_t*>(s_packed);
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.M = M;
  p.gpw = (G + kM8Warps - 1) / kM8Warps;
  p.scale2 = scale2;
  if (d.wfmt == QW_W_UINT4ZP_G128_BF16) {
    p.zplane = (int64_t)(d.s_expert_stride / 4);  // the second BF16 plane
    return launch_m8_variant<4, true>(p, st);
  }
  if (d.wfmt == QW_W_INT2_G128_BF16) return launch_m8_variant<2, false>(p, st);
  if (d.wfmt == QW_W_FP8E4M3_G128_BF16) return launch_m8_variant<8, false>(p, st);
  if (d.wfmt == QW_W_INT1_G128_BF16) return launch_m8_variant<1, false>(p, st);
  if (d.wfmt == QW_W_FP4E2M1_G128_BF16) return launch_m8_variant<kBitsFp4, false>(p, st);
  return d.wfmt == QW_W_INT4_G128_BF16 ? launch_m8_variant<4, false>(p, st)
                                       : launch_m8_variant<3, false>(p, st);
}

// Other dense calls with up to 16 token rows: the register-ring kernel.
qw_status launch_dense_reg(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* bias, const float* scale2, void* C,
                           int64_t M, int mch, cudaStream_t st) {
  const int G = d.K / kIntGroup;
  Params p{};
  p.wp = static_cast<const uint8_t*>(w_packed);
  p.sp = static_cast<const uint16_t*>(s_packed);
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.M = M;
  p.w_estride = (int64_t)d.w_expert_stride;
  p.s_estride = (int64_t)(d.s_expert_stride / 2);
  p.gpw = (G + kWarps - 1) / kWarps;
  p.scale2 = scale2;
  const int64_t items = (d.N_pad / 16) * ((M + 8 * mch - 1) / (8 * mch));
  if (items > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  if (d.wfmt == QW_W_UINT4ZP_G128_BF16) {
    p.zplane = (int64_t)(d.s_expert_stride / 4);  // the second BF16 plane
    return mch == 1 ? launch_reg_variant<4, 1, true>(p, items, st)
                    : launch_reg_variant<4, 2, true>(p, items, st);
  }
  if (d.wfmt == QW_W_INT2_G128_BF16)
    return mch == 1 ? launch_reg_variant<2, 1, false>(p, items, st)
                    : launch_reg_variant<2, 2, false>(p, items, st);
  if (d.wfmt == QW_W_FP8E4M3_G128_BF16)
    return mch == 1 ? launch_reg_variant<8, 1, false>(p, items, st)
                    : launch_reg_variant<8, 2, false>(p, items, st);
  if (d.wfmt == QW_W_INT1_G128_BF16)
    return mch == 1 ? launch_reg_variant<1, 1, false>(p, items, st)
                    : launch_reg_variant<1, 2, false>(p, items, st);
  if (d.wfmt == QW_W_FP4E2M1_G128_BF16)
    return mch == 1 ? launch_reg_variant<kBitsFp4, 1, false>(p, items, st)
                    : launch_reg_variant<kBitsFp4, 2, false>(p, items, st);
  const bool int4 = d.wfmt == QW_W_INT4_G128_BF16;
  if (mch == 1)
    return int4 ? launch_reg_variant<4, 1, false>(p, items, st)
                : launch_reg_variant<3, 1, false>(p, items, st);
  return int4 ? launch_reg_variant<4, 2, false>(p, items, st)
              : launch_reg_variant<3, 2, false>(p, items, st);
}

}  // namespace

uint64_t gemv_w4a16_workspace(const qw_packed_desc& d, int64_t max_rows) {
  // only grouped calls need device memory of their own: the tile queue
  if (d.E <= 1) return 0;
  // the tile rows shrink with the rows of a call: size the queue for the smallest tile, so
  // that it holds every call of at most max_rows rows
  return tile_queue_bytes(d.E, max_rows, 8);
}

qw_status launch_gemv_w4a16(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                            const void* A, const void* bias, void* C, const RowSet& rs,
                            void* ws, uint64_t ws_bytes, int32_t* err, cudaStream_t st) {
  const bool grouped = rs.offsets != nullptr;
  const int mch = mch_for(d, rs.rows, grouped);
  // single-token decode, symmetric INT4 / INT3 / INT2: the decode kernel
  if (!grouped && rs.rows == 1 && decode_eligible(d, A))
    return launch_decode(d, w_packed, s_packed, A, bias, rs.scale2, C, st);
  // single-token decode over a large matrix: the staged kernel (its staging pays off once a
  // warp streams many groups; measured slower on matrices of 16 M weights and below)
  if (!grouped && rs.rows == 1 && (int64_t)d.N * d.K >= kM8MinWeights &&
      (reinterpret_cast<uintptr_t>(A) & 15) == 0 && m8_smem_bytes(d.K, 1) <= kM8MaxSmem)
    return launch_dense_m8(d, w_packed, s_packed, A, bias, rs.scale2, C, 1, st);
  if (!grouped)
    return launch_dense_reg(d, w_packed, s_packed, A, bias, rs.scale2, C, rs.rows, mch, st);
  // Grouped calls (over the device tile queue), and dense calls the dispatcher sends here
  // with more rows: the TMA ring.
  const bool zp = d.wfmt == QW_W_UINT4ZP_G128_BF16;
  const bool int4 = d.wfmt == QW_W_INT4_G128_BF16 || zp;
  const bool int2 = d.wfmt == QW_W_INT2_G128_BF16;
  const bool fp8 = d.wfmt == QW_W_FP8E4M3_G128_BF16;
  const bool int1 = d.wfmt == QW_W_INT1_G128_BF16;
  const bool fp4 = d.wfmt == QW_W_FP4E2M1_G128_BF16;
  const int blk = int4 ? kInt4BlockBytes
                  : int2 ? kInt2BlockBytes
                  : fp8  ? kFp8BlockBytes
                  : int1 ? kInt1BlockBytes
                  : fp4  ? kFp4BlockBytes
                         : kInt3BlockBytes;
  const int G = d.K / kIntGroup;
  const int64_t nblocks = d.N_pad / 16;
  auto enc = encode_fn();
  if (!enc) return QW_ERR_CUDA;
  // weights: [E][G][N_pad/16][block] as 8-byte elements; one copy = 8 groups of a block
  CUtensorMap tmW, tmS, tmZ;
  {
    cuuint64_t dim[4] = {(cuuint64_t)(blk / 8), (cuuint64_t)nblocks, (cuuint64_t)G,
                         (cuuint64_t)d.E};
    cuuint64_t str[3] = {(cuuint64_t)blk, (cuuint64_t)(nblocks * blk),
                         (cuuint64_t)d.w_expert_stride};
    cuuint32_t box[4] = {(cuuint32_t)(blk / 8), 1, (cuuint32_t)kStageGroups, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<void*>(w_packed), dim, str, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QW_ERR_ALIGNMENT;
  }
  // scales: BF16 [E][G][N_pad]; one copy = the 16 rows of a block x 8 groups
  {
    cuuint64_t dim[3] = {(cuuint64_t)d.N_pad, (cuuint64_t)G, (cuuint64_t)d.E};
    cuuint64_t str[2] = {(cuuint64_t)d.N_pad * 2, (cuuint64_t)d.s_expert_stride};
    cuuint32_t box[3] = {16, (cuuint32_t)kStageGroups, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(s_packed), dim, str, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QW_ERR_ALIGNMENT;
    // asymmetric INT4: the plane of 128 + z, half an expert's scale stride further on
    tmZ = tmS;
    if (zp) {
      void* zbase = static_cast<uint8_t*>(const_cast<void*>(s_packed)) + d.s_expert_stride / 2;
      if (enc(&tmZ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, zbase, dim, str, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QW_ERR_ALIGNMENT;
    }
  }
  TmaParams p{};
  p.A = static_cast<const uint16_t*>(A);
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.M = rs.rows;
  p.err = err;
  p.scale2 = rs.scale2;
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
  if (mch == 1)
    return zp     ? launch_tma_variant<4, 1, GroupedRing, true>(tmW, tmS, tmZ, p, size_items, st)
           : int4 ? launch_tma_variant<4, 1, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
           : int2 ? launch_tma_variant<2, 1, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
           : fp8  ? launch_tma_variant<8, 1, GroupedRing8, false>(tmW, tmS, tmZ, p, size_items, st)
           : int1 ? launch_tma_variant<1, 1, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
           : fp4  ? launch_tma_variant<kBitsFp4, 1, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
                  : launch_tma_variant<3, 1, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st);
  return zp     ? launch_tma_variant<4, 2, GroupedRing, true>(tmW, tmS, tmZ, p, size_items, st)
         : int4 ? launch_tma_variant<4, 2, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
         : int2 ? launch_tma_variant<2, 2, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
         : fp8  ? launch_tma_variant<8, 2, GroupedRing8, false>(tmW, tmS, tmZ, p, size_items, st)
         : int1 ? launch_tma_variant<1, 2, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
         : fp4  ? launch_tma_variant<kBitsFp4, 2, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st)
                : launch_tma_variant<3, 2, GroupedRing, false>(tmW, tmS, tmZ, p, size_items, st);
}

}  // namespace qw
