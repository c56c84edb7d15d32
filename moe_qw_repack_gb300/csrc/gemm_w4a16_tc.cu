// gemm_w4a16_tc.cu - large-M W4A16 path: INT4/INT3 weights dequantized inside the SM and
// multiplied on the sm_103a tensor cores (tcgen05, BF16 operands, FP32 accumulation).
//
// What it computes (spke.com Humming announcement, "WnA16"; "フォーマットとアーキテクチャ
// を横断して共有されるCUDAコンポーネント": dequantization and scaling inside the kernel,
// bias in the output stage):
//     C[m][n] = bf16( sum_g s[n][g] * sum_{k in g} a[m][k] * q[n][k] + bias[n] )
// The integer weights go to the tensor core exactly (|q| <= 7 is exact in BF16); each
// scale group's sum is accumulated on its own and multiplied by the group scale in FP32,
// so no weight is ever rounded (rounding q * s to BF16 alone would cost ~2^-9 relative
// per weight).
//
// Structure (persistent, one CTA per SM; a tile is 128 weight rows x 128 tokens; one
// pipeline stage is one scale group of 128 k):
//   warp 0      producer: TMA loads of the activation tile (two 128 x 64 BF16 boxes,
//               128-byte swizzle) and a bulk copy of the 8 packed 16 x 128 weight blocks
//               into a 4-stage ring;
//   warp 1      TMEM owner and MMA issuer: per group, eight 128x128x16 MMAs with the
//               weights as the A operand read from tensor memory and the tokens as the B
//               operand, into one of two per-group accumulators;
//   warps 2-5   dequantizers: warp q covers TMEM lanes 32q .. 32q + 31, i.e. two packed
//               16 x 128 blocks; each lane decodes its own eight fragment words into BF16
//               integers (code | 0x4300 = 128 + code, minus the excess) and one
//               tcgen05.st.16x256b.x8 per block puts them at the rows and k columns of the
//               stage's A operand - the packed layout is the register layout of that store,
//               so the dequantized operand never touches shared memory and no lane moves data
//               for another;
//   warps 6-13  promotion and epilogue: read each group's accumulator (tcgen05.ld), add
//               scale x it to FP32 registers, release it; at the end of the tile add bias,
//               round to BF16 and write the tile into a shared-memory staging tile
//               [token][row] (lanes = consecutive rows: conflict-free 2-byte stores), which
//               one thread hands to a TMA store - the warps go straight back to promoting
//               the next tile instead of issuing 64 narrow global stores each.  MoE tiles
//               that end inside a tile of 128 tokens (the next rows belong to another
//               expert) and outputs whose row pitch is not a multiple of 16 bytes are stored
//               directly instead.
// Every wait is bounded; on expiry the kernel reports QW_ERR_TIMEOUT and shuts down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int BW = 128;  // weight rows per tile (MMA M)
constexpr int BT = 128;  // tokens per tile (MMA N)
constexpr int STAGES = 4;
constexpr int ACT_BOX = BT * 64 * 2;  // 128 tokens x 64 k of BF16
constexpr int ACT_BYTES = 2 * ACT_BOX;
constexpr int NUM_DQ_WARPS = 4, NUM_EPI_WARPS = 8;
constexpr int DQ_WARP0 = 2, EPI_WARP0 = DQ_WARP0 + NUM_DQ_WARPS;
constexpr int NUM_THREADS = (EPI_WARP0 + NUM_EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = 2 * BT;  // the two per-group accumulators use columns [0, 256)

// kind::f16 instruction descriptor: FP32 accumulator (bit 4), A = B = BF16 (bits 7, 10),
// both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BT >> 3) << 17) |
                           ((uint32_t)(BW >> 4) << 24);

template <int BITS, bool ZP>
struct Geo {
  static constexpr int BLK = wna16_block_bytes(BITS);  // one packed 16 x 128 block
  static constexpr int WBYTES = 8 * BLK;
  // asymmetric INT4: the tile's 128 rows of BF16 128 + zero point for the stage's group
  static constexpr int ZBYTES = ZP ? BW * 2 : 0;
  // stages start on 1 KiB boundaries: the 128-byte-swizzled activation boxes need it
  static constexpr int STAGE = (ACT_BYTES + WBYTES + ZBYTES + 1023) / 1024 * 1024;
};

struct Params {
  int64_t rows;  // tokens (M, or total grouped rows)
  int32_t N, N_pad, K;
  int32_t num_m_tiles;  // dense only
  int32_t num_n_tiles;
  const uint8_t* wp;
  const uint16_t* sp16;          // BF16 scales [E][K/128][N_pad]
  const uint16_t* zp16;          // asymmetric INT4: BF16 128 + z, same layout (else null)
  int64_t w_estride;             // bytes
  int64_t s_estride_elems;
  const uint16_t* bias;
  uint16_t* C;
  const int32_t* queue;
  int32_t* err;
  int32_t tma_store;  // C's tensor map is valid (row pitch a multiple of 16 bytes)
  const float* scale2;  // second-level scales [E][N_pad] or null
};

struct Tile {
  int e, nt;
  int64_t rb, re;
};

__device__ __forceinline__ Tile tile_at(const Params& p, int64_t t) {
  Tile x;
  x.nt = (int)(t % p.num_n_tiles);
  const int64_t mt = t / p.num_n_tiles;
  if (p.queue) {
    x.e = __ldg(p.queue + 1 + 3 * mt);
    x.rb = __ldg(p.queue + 2 + 3 * mt);
    x.re = __ldg(p.queue + 3 + 3 * mt);
  } else {
    x.e = 0;
    x.rb = mt * BT;
    x.re = min64(p.rows, x.rb + BT);
  }
  return x;
}

// 16 TMEM lanes x 64 columns: thread 4g + t, repetition j puts registers 4j .. 4j + 3 at
// (lane g, column 8j + 2t), (g, 8j + 2t + 1), (g + 8, 8j + 2t), (g + 8, 8j + 2t + 1).
__device__ __forceinline__ void tc_st_16x256b_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t bf16x2_sub_u32(uint32_t x, uint32_t y) {
  // x - y for a pair of BF16 values; here the difference is an exact small integer
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&y);
  __nv_bfloat162 r = __hsub2(a, b);
  return *reinterpret_cast<uint32_t*>(&r);
}

// acc (an FP32 pair, low = first) += s2 * (x0, x1): one packed two-wide FMA
__device__ __forceinline__ void fma2_acc(uint64_t& acc, uint64_t s2, uint32_t x0, uint32_t x1) {
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%2, %3};\n\tfma.rn.f32x2 %0, %1, t, %0;\n\t}"
      : "+l"(acc)
      : "l"(s2), "r"(x0), "r"(x1));
}

// (a & b) | c in one logic instruction (written out so the compiler cannot split it)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
}

__device__ __forceinline__ void tma_store_2d(const void* map, uint32_t smem_src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   map),
               "r"(x), "r"(y), "r"(smem_src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
constexpr int STAGING_BYTES = BT * BW * 2;  // one BF16 output tile [token][row]

template <int BITS, bool ZP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmC, const Params p) {
  using GE = Geo<BITS, ZP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* staging = smem + STAGES * GE::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* aready = full + STAGES;
  uint64_t* empty = aready + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2] per-group accumulators
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* final_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel may start its own set-up on SMs this grid has left
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&aready[s], NUM_DQ_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], NUM_EPI_WARPS);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmA);
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Launched as a programmatic dependent: the set-up above overlaps the previous kernel's
  // tail; every global access (tile queue, operands, scales, bias, output) comes after this.
  pdl_wait();

  const int64_t num_m = p.queue ? (int64_t)__ldg(p.queue) : (int64_t)p.num_m_tiles;
  const int64_t num_tiles = num_m * p.num_n_tiles;
  const int G = p.K / 128;
  const int nblocks = p.N_pad / 16;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        const Tile x = tile_at(p, t);
        const int nbs = min(8, nblocks - x.nt * 8);
        const uint8_t* wsrc = p.wp + x.e * p.w_estride + (int64_t)x.nt * 8 * GE::BLK;
        for (int g = 0; g < G; ++g) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * GE::STAGE;
          mbar_arrive_expect_tx(&full[stage], ACT_BYTES + nbs * GE::BLK + (ZP ? nbs * 32 : 0));
          tma_load_2d(st, &tmA, &full[stage], g * 128, (int32_t)x.rb);
          tma_load_2d(st + ACT_BOX, &tmA, &full[stage], g * 128 + 64, (int32_t)x.rb);
          bulk_load(st + ACT_BYTES, wsrc + (int64_t)g * nblocks * GE::BLK, nbs * GE::BLK,
                    &full[stage]);
          if constexpr (ZP)
            bulk_load(st + ACT_BYTES + GE::WBYTES,
                      p.zp16 + x.e * p.s_estride_elems + (int64_t)g * p.N_pad + x.nt * BW,
                      nbs * 32, &full[stage]);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) drain_wait(&full[s], (issued_phase >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint64_t gi = 0;  // groups issued so far: accumulator gi & 1
      for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int g = 0; g < G; ++g, ++gi) {
          const int ab = (int)(gi & 1);
          const uint32_t use = (uint32_t)(gi >> 1) & 1u;
          if (!mbar_wait(&acc_empty[ab], use ^ 1u, abort_flag, p.err) ||
              !mbar_wait(&aready[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t act = smem_u32(smem + stage * GE::STAGE);
          const uint32_t d = tbase + ab * BT;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint64_t bd = smem_desc(act + (s / 4) * ACT_BOX + (s % 4) * 32, 16, 1024, 2);
            tc_mma_f16_tmem_a(d, tbase + A_COL0 + 64 * stage + 8 * s, bd, IDESC, s != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          tc_commit(&acc_full[ab]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      tc_commit(final_bar);
      drain_wait(final_bar, 0);
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ dequantizers
    // Lane 4g + t holds, in word s of a packed block, rows g and g + 8 at k = 16s + 4t ..
    // 16s + 4t + 3: decoded to four BF16 pairs (a0..a3 = row g k+0/1, row g+8 k+0/1, row g
    // k+2/3, row g+8 k+2/3) they are exactly repetition s of a 16x256b TMEM store.
    const int q = warp & 3;  // TMEM lane quadrant: blocks 2q and 2q + 1 of the tile
    const uint32_t magic = 0x43004300u;
    const uint32_t excess = 0x43004300u + 0x10001u * (1u << (BITS - 1));  // BF16 pair 128 + excess
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const Tile x = tile_at(p, t);
      const int nbs = min(8, nblocks - x.nt * 8);
      for (int g = 0; g < G; ++g) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int b = 2 * q + hb;
          const uint32_t blk = smem_u32(smem + stage * GE::STAGE) + ACT_BYTES + b * GE::BLK;
          uint32_t v[32];
          if (b < nbs) {
            if constexpr (BITS == 4) {
              const uint4 w0 = lds128(blk + lane * 32), w1 = lds128(blk + lane * 32 + 16);
              const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
              // the excess of rows g and g + 8: the constant, or (asymmetric) 128 + z
              uint32_t ex_lo = excess, ex_hi = excess;
              if constexpr (ZP) {
                const uint32_t zrow = smem_u32(smem + stage * GE::STAGE) + ACT_BYTES + GE::WBYTES +
                                      (uint32_t)(16 * b + (lane >> 2)) * 2;
                ex_lo = lds16(zrow) * 0x10001u;
                ex_hi = lds16(zrow + 16) * 0x10001u;
              }
#pragma unroll
              for (int st = 0; st < 8; ++st) {
                // registers 4st, 4st + 1 hold row g; 4st + 2, 4st + 3 row g + 8
                v[4 * st + 0] = bf16x2_sub_u32(and_or(w[st], 0x000F000Fu, magic), ex_lo);
                v[4 * st + 2] = bf16x2_sub_u32(and_or(w[st] >> 4, 0x000F000Fu, magic), ex_hi);
                v[4 * st + 1] = bf16x2_sub_u32(and_or(w[st] >> 8, 0x000F000Fu, magic), ex_lo);
                v[4 * st + 3] = bf16x2_sub_u32(and_or(w[st] >> 12, 0x000F000Fu, magic), ex_hi);
              }
            } else if constexpr (BITS == 8) {
              // E4M3 codes: words 2st (rows g, g + 8 at k + 0/1) and 2st + 1 (k + 2/3),
              // decoded exactly, no excess
              uint32_t w[16];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 x4 = lds128(blk + lane * 64 + 16 * i);
                w[4 * i] = x4.x; w[4 * i + 1] = x4.y; w[4 * i + 2] = x4.z; w[4 * i + 3] = x4.w;
              }
#pragma unroll
              for (int st = 0; st < 8; ++st) {
                v[4 * st + 0] = e4m3x2_to_bf16x2(w[2 * st]);
                v[4 * st + 2] = e4m3x2_to_bf16x2(w[2 * st] >> 16);
                v[4 * st + 1] = e4m3x2_to_bf16x2(w[2 * st + 1]);
                v[4 * st + 3] = e4m3x2_to_bf16x2(w[2 * st + 1] >> 16);
              }
            } else if constexpr (BITS == kBitsFp4) {
              // E2M1 codes: byte r of word st is register r (rows g + 8 (r & 1), k + 2 (r >> 1)),
              // one hardware conversion to FP16, then to BF16 (exact), no excess
              const uint4 w0 = lds128(blk + lane * 32), w1 = lds128(blk + lane * 32 + 16);
              const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
              for (int st = 0; st < 8; ++st) {
                uint32_t h[4];
                e2m1x8_to_f16x2(w[st], h);
#pragma unroll
                for (int r = 0; r < 4; ++r)
                  v[4 * st + ((r & 1) << 1) + (r >> 1)] = f16x2_to_bf16x2(h[r]);
              }
            } else if constexpr (BITS == 1) {
              // INT1 sign codes: register r of step st at bits 4 (st % 4) + r (+ 16) of word
              // st / 4, decoded to BF16 +-1 pairs
              const uint2 W = lds64(blk + lane * 8);
#pragma unroll
              for (int st = 0; st < 8; ++st)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                  v[4 * st + ((r & 1) << 1) + (r >> 1)] =
                      int1_pair(st < 4 ? W.x : W.y, 4 * (st & 3) + r, 0x3F803F80u);
            } else if constexpr (BITS == 2) {
              const uint4 lo = lds128(blk + lane * 16);
              const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
              for (int st = 0; st < 8; ++st)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                  const uint32_t biased =
                      and_or(L[st >> 1] >> (2 * (4 * (st & 1) + r)), 0x00030003u, magic);
                  // register r (row g + 8 (r & 1), k + 2 (r >> 1)) -> store slot
                  v[4 * st + ((r & 1) << 1) + (r >> 1)] = bf16x2_sub_u32(biased, excess);
                }
            } else {
              // INT3: register j = 4st + r is the 3-bit field j % 5 of word j / 5, except
              // j = 30, 31, gathered from the spare bit 15 + 16h of words 0..2 and 3..5
              const uint4 lo = lds128(blk + lane * 16);
              const uint2 hi = lds64(blk + 512 + lane * 8);
              const uint32_t W[6] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y};
#pragma unroll
              for (int st = 0; st < 8; ++st)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                  const int j = 4 * st + r;
                  uint32_t biased;
                  if (j < 30) {
                    biased = and_or(W[j / 5] >> (3 * (j % 5)), 0x00070007u, magic);
                  } else {
                    const int b = j == 30 ? 0 : 3;
                    biased = and_or(W[b + 2] >> 13, 0x00040004u,
                                    and_or(W[b + 1] >> 14, 0x00020002u,
                                           and_or(W[b] >> 15, 0x00010001u, magic)));
                  }
                  // register r (row g + 8 (r & 1), k + 2 (r >> 1)) -> store slot
                  v[4 * st + ((r & 1) << 1) + (r >> 1)] = bf16x2_sub_u32(biased, excess);
                }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          tc_st_16x256b_x8(tbase + ((uint32_t)(32 * q + 16 * hb) << 16) + A_COL0 + 64 * stage, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aready[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    const int q = warp & 3;                    // TMEM lane quadrant = 32 weight rows
    const int half = (warp - EPI_WARP0) >> 2;  // tokens [64 half, 64 half + 64) of the tile
    uint64_t gi = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const Tile x = tile_at(p, t);
      const int n = x.nt * BW + 32 * q + lane;
      const bool nvalid = n < p.N;
      const uint16_t* srow = p.sp16 + x.e * p.s_estride_elems + (nvalid ? n : 0);
      uint64_t acc2[32];  // FP32 pairs (tokens 2i, 2i + 1), promoted with packed FMAs
#pragma unroll
      for (int i = 0; i < 32; ++i) acc2[i] = 0ull;
      uint32_t s_next = __ldg(srow);
      for (int g = 0; g < G; ++g, ++gi) {
        const uint32_t scb = s_next << 16;  // the group scale as FP32 bits
        const uint64_t sc2 = ((uint64_t)scb << 32) | scb;
        if (g + 1 < G) s_next = __ldg(srow + (int64_t)(g + 1) * p.N_pad);
        const int ab = (int)(gi & 1);
        const uint32_t use = (uint32_t)(gi >> 1) & 1u;
        if (!mbar_wait(&acc_full[ab], use, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tbase + ((uint32_t)(32 * q) << 16) + ab * BT + 64 * half;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tc_ld_32x32b_x32(ta + 32 * hh, v);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) fma2_acc(acc2[16 * hh + i], sc2, v[2 * i], v[2 * i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
      }
      if (!ok) break;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        acc[2 * i] = __uint_as_float((uint32_t)acc2[i]);
        acc[2 * i + 1] = __uint_as_float((uint32_t)(acc2[i] >> 32));
      }
      const float bias =
          (p.bias && nvalid) ? __uint_as_float((uint32_t)__ldg(p.bias + (int64_t)x.e * p.N + n) << 16)
                             : 0.f;
      if (p.scale2) {  // second-level scale of this output channel, before the bias
        const float t2 = nvalid ? __ldg(p.scale2 + (int64_t)x.e * p.N_pad + n) : 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] *= t2;
      }
      // dense tiles may run past the last row (the store clips them); MoE tiles may not
      if (p.tma_store && (!p.queue || x.re - x.rb == BT)) {
        const bool issuer = warp == EPI_WARP0 && lane == 0;
        if (issuer) bulk_wait_read_all();  // the previous tile's store has read the staging
        asm volatile("bar.sync 1, %0;" ::"r"(NUM_EPI_WARPS * 32) : "memory");
        const uint32_t sbase = smem_u32(staging) + (uint32_t)(64 * half) * (BW * 2) +
                               (uint32_t)(32 * q + lane) * 2;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          __nv_bfloat16 h = __float2bfloat16_rn(acc[i] + bias);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(sbase + i * (BW * 2)),
                       "h"(*reinterpret_cast<uint16_t*>(&h))
                       : "memory");
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, %0;" ::"r"(NUM_EPI_WARPS * 32) : "memory");
        if (issuer) tma_store_2d(&tmC, smem_u32(staging), x.nt * BW, (int32_t)x.rb);
      } else if (nvalid) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int64_t tok = x.rb + 64 * half + i;
          if (tok < x.re) {
            __nv_bfloat16 h = __float2bfloat16_rn(acc[i] + bias);
            p.C[tok * p.N + n] = *reinterpret_cast<uint16_t*>(&h);
          }
        }
      }
    }
    if (warp == EPI_WARP0 && lane == 0) bulk_wait_all();  // stores done before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
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

template <int BITS, bool ZP>
qw_status launch_bits(const CUtensorMap& tmA, const CUtensorMap& tmC, const Params& p,
                      int64_t tiles_max, cudaStream_t st) {
  using GE = Geo<BITS, ZP>;
  // ring + output staging + barriers + alignment
  constexpr size_t kSmem = (size_t)STAGES * GE::STAGE + STAGING_BYTES + 256 + 1024;
  static_assert(kSmem <= 232448, "shared memory of one CTA");
  const size_t smem = kSmem;
  static const cudaError_t attr = cudaFuncSetAttribute(
      gemm_w4a16_tc_kernel<BITS, ZP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return QW_ERR_CUDA;
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(tiles_max < sms ? (tiles_max < 1 ? 1 : tiles_max) : sms);
  return launch_pdl(gemm_w4a16_tc_kernel<BITS, ZP>, dim3(grid), dim3(NUM_THREADS), smem, st, tmA,
                    tmC, p);
}

}  // namespace

uint64_t gemm_w4a16_tc_workspace(const qw_packed_desc& d, int64_t max_rows) {
  return d.E > 1 ? tile_queue_bytes(d.E, max_rows, BT) : 0;
}

qw_status launch_gemm_w4a16_tc(const qw_packed_desc& d, const void* w_packed,
                               const void* s_packed, const void* A, const void* bias, void* C,
                               const RowSet& rs, void* ws, uint64_t ws_bytes, int32_t* err,
                               cudaStream_t st) {
  if (rs.rows == 0) return QW_OK;
  auto enc = encode_fn();
  if (!enc) return QW_ERR_CUDA;
  if (rs.rows > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  CUtensorMap tmA;
  cuuint64_t gdim[2] = {(cuuint64_t)d.K, (cuuint64_t)rs.rows};
  cuuint64_t gstr[1] = {(cuuint64_t)d.K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)BT};
  cuuint32_t es[2] = {1, 1};
  if (enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), gdim, gstr, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QW_ERR_ALIGNMENT;
  // output map: BF16 [rows][N], box 128 rows of N x 128 tokens, no swizzle; only when the
  // row pitch is a multiple of 16 bytes (otherwise the kernel stores directly)
  CUtensorMap tmC;
  memset(&tmC, 0, sizeof(tmC));
  bool tma_store = (d.N % 8) == 0 && (reinterpret_cast<uintptr_t>(C) % 16) == 0;
  if (tma_store) {
    cuuint64_t cdim[2] = {(cuuint64_t)d.N, (cuuint64_t)rs.rows};
    cuuint64_t cstr[1] = {(cuuint64_t)d.N * 2};
    cuuint32_t cbox[2] = {(cuuint32_t)BW, (cuuint32_t)BT};
    tma_store = enc(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, cdim, cstr, cbox, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  Params p{};
  p.tma_store = tma_store ? 1 : 0;
  p.rows = rs.rows;
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.num_n_tiles = (d.N_pad + BW - 1) / BW;
  p.num_m_tiles = (int32_t)((rs.rows + BT - 1) / BT);
  p.wp = static_cast<const uint8_t*>(w_packed);
  p.sp16 = static_cast<const uint16_t*>(s_packed);
  p.w_estride = (int64_t)d.w_expert_stride;
  p.s_estride_elems = (int64_t)(d.s_expert_stride / 2);
  if (d.wfmt == QW_W_UINT4ZP_G128_BF16)  // the second plane: half an expert's scale stride
    p.zp16 = p.sp16 + d.s_expert_stride / 4;
  p.bias = static_cast<const uint16_t*>(bias);
  p.C = static_cast<uint16_t*>(C);
  p.err = err;
  p.scale2 = rs.scale2;
  int64_t max_m = p.num_m_tiles;
  if (rs.offsets) {
    const uint64_t need = tile_queue_bytes(rs.E, rs.rows, BT);
    if (ws == nullptr || ws_bytes < need) return QW_ERR_WORKSPACE;
    int32_t* queue = static_cast<int32_t*>(ws);
    max_m = (int64_t)(need / 4 - 1) / 3;
    const qw_status s =
        launch_build_tile_queue(rs.offsets, rs.E, BT, rs.rows, queue, max_m, err, st);
    if (s != QW_OK) return s;
    p.queue = queue;
  }
  const int64_t tiles_max = max_m * p.num_n_tiles;
  if (d.wfmt == QW_W_UINT4ZP_G128_BF16) return launch_bits<4, true>(tmA, tmC, p, tiles_max, st);
  if (d.wfmt == QW_W_INT2_G128_BF16) return launch_bits<2, false>(tmA, tmC, p, tiles_max, st);
  if (d.wfmt == QW_W_FP8E4M3_G128_BF16) return launch_bits<8, false>(tmA, tmC, p, tiles_max, st);
  if (d.wfmt == QW_W_INT1_G128_BF16) return launch_bits<1, false>(tmA, tmC, p, tiles_max, st);
  if (d.wfmt == QW_W_FP4E2M1_G128_BF16)
    return launch_bits<kBitsFp4, false>(tmA, tmC, p, tiles_max, st);
  return d.wfmt == QW_W_INT4_G128_BF16 ? launch_bits<4, false>(tmA, tmC, p, tiles_max, st)
                                       : launch_bits<3, false>(tmA, tmC, p, tiles_max, st);
}

}  // namespace qw
