// gemm_w4a8_tc.cu - large-M W4A8 path: MXFP4 weights x MXFP8 activations on the
// sm_103a block-scaled tensor cores, and on the same skeleton the W8A8 MX kind (MXFP8
// weights: E4M3 as the B type) and W4A4 (NVFP4 x NVFP4: tcgen05 kind::mxf4nvf4 with
// scale_vec::4X - both operands packed E2M1 in shared memory, 256 k per stage, an
// unsigned E4M3 scale per 16 k, four scale images per stage instead of one).
//
// What it computes (aireiter.com "vLLM Humming performance benchmark", section "H100
// group-32 W4A8": MXFP4 weights, MXFP8 activations, group-32 scales; spke.com Humming
// announcement, section "W8A8 / W4A8 / W4A4": Blackwell runs the MX formats natively):
//   C[m][n] = bf16( sum_k e4m3(a[m][k]) 2^(sa[m][k/32]-127) e2m1(w[n][k]) 2^(sw[n][k/32]-127)
//                   + bias[n] )
// The pages' Hopper design upcasts FP4 to FP8 inside the SM; on sm_103a the tensor core
// takes E4M3 x E2M1 with per-32 E8M0 scales directly (tcgen05.mma kind::mxf8f6f4
// block_scale), so the "dequantization" is the MMA itself.
//
// Structure (one persistent CTA per SM, 128 x 256 output tiles, K in steps of 128):
//   warp 0      TMA producer: A tile (E4M3, 128 x 128 B, 128-byte swizzle), B tile
//               (E2M1 codes unpacked by TMA to one byte per code, 256 x 128), and the
//               repacked B scale chunks (bulk copies) into a 4-stage ring;
//   warp 1      TMEM owner and single-thread MMA issuer: tcgen05.cp the stage's scale
//               factors into TMEM, four 128x256x32 block-scaled MMAs, commit -> frees
//               the stage; commit -> accumulator full at the end of a tile;
//   warp 2      A scale fetcher: reads the canonical [rows][K/32] E8M0 bytes three stages
//               ahead into registers and writes the 32 x 16-byte image tcgen05.cp
//               expects (row r -> lane r % 32, column r / 32, byte = group within the
//               128-wide K step) into an 8-slot staging ring;
//   warp 3      A scale writer: copies a staged image into the stage once the stage is
//               free, then the proxy fence that lets the tensor core read it.  (A
//               fence waits for the thread's outstanding memory operations; keeping the
//               global loads in another warp keeps them off the fence.)
//   Indexed MoE calls skip the separate permutation: problem row r is activation row
//   sorted_pairs[r] / topk, fetched by TMA gather4 copies (four 128-byte rows each, a
//   one-row tensor-map box) whose row indices warp 0 looks up a tile ahead; the scale
//   fetcher reads the same rows' scales.  The results are those of permute + grouped.
//   warps 4-11  epilogue: tcgen05.ld the FP32 accumulator (each warp one 32-lane
//               quadrant x 128 columns), add bias, round to BF16, release TMEM, store.
// Every mbarrier wait is bounded; on expiry the kernel raises QW_ERR_TIMEOUT, lets its
// copies in flight land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

// BK = bytes of a row per stage (128: one 128-byte swizzle atom)
constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int A_BYTES = BM * BK;
// B in shared memory: E4M3 codes as they are, E2M1 codes unpacked by TMA to one byte each
// (W4A8: 16 codes in 8 bytes + 8 gap bytes), or packed E2M1 (W4A4)
constexpr int B_BYTES = BN * BK;
constexpr int NUM_WARPS = 12, NUM_THREADS = NUM_WARPS * 32;
constexpr int EPI_WARP0 = 4, NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256;  // accumulator uses columns [0, 256)

enum Kind { kW4A8 = 0, kW8A8 = 1, kW4A4 = 2 };

// Per-kind constants.  A scale image is the 32 x 16-byte block tcgen05.cp.32x128b.warpx4
// copies for 128 rows (row r -> lane r % 32, column (r % 128) / 32, four scale bytes):
// one image covers a stage's four 32-k groups (1X, E8M0) or one 64-k MMA's four 16-k groups
// (4X, E4M3).
template <int KIND>
struct KT {
  static constexpr bool NV = KIND == kW4A4;
  static constexpr int IMG = NV ? 4 : 1;        // scale images per 128 rows and stage
  static constexpr int KSTEP = NV ? 256 : 128;  // K elements per stage
  static constexpr int GROUP = NV ? 16 : 32;    // K elements per scale
  // bytes a B load credits to its barrier: the global bytes
  static constexpr int B_TX = KIND == kW8A8 ? BN * BK : (KIND == kW4A8 ? BN * BK / 2 : BN * BK);
  static constexpr int SFA_BYTES = 512 * IMG;
  static constexpr int SFB_CHUNK = 512 * IMG;  // 128 B rows
  static constexpr int SFB_BYTES = 2 * SFB_CHUNK;
  static constexpr uint32_t SF_COLS_PER_STAGE = 12 * IMG;  // A: 4 per image, B: 8 per image
  static constexpr int SF_STAGING = NV ? 4 : 8;            // staged A scale slots
  static constexpr uint32_t SF_PAD = NV ? 0x38383838u : 0x7F7F7F7Fu;  // scale 1
  static constexpr size_t SMEM_BYTES =
      (size_t)STAGES * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) +
      (size_t)SF_STAGING * SFA_BYTES + BM * 4 + 512 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Instruction descriptor.  kind::mxf8f6f4: A = E4M3 (0), B = E2M1 (5) or E4M3 (0), scale
// type UE8M0 (bit 23 set); kind::mxf4nvf4: A = B = E2M1 (1), scale type UE4M3 (bit 23
// clear).  Both K-major, N >> 3 at bit 17, M >> 4 at bit 24; the B / A scale-factor byte
// selectors sit at bits 4 and 29 (1X only; 4X reads a whole 32-bit column per MMA).
template <int KIND>
__host__ __device__ constexpr uint32_t idesc() {
  return KIND == kW4A4
             ? ((1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                ((uint32_t)(BM >> 4) << 24))
             : ((0u << 7) | ((KIND == kW8A8 ? 0u : 5u) << 10) | ((uint32_t)(BN >> 3) << 17) |
                (1u << 23) | ((uint32_t)(BM >> 4) << 24));
}

struct Params {
  int64_t rows;           // activation rows (M, or total grouped rows)
  int32_t N, N_pad, K, K_pad;
  int32_t num_m_tiles;    // dense only
  int32_t num_n_tiles;
  const uint8_t* A_sf;    // [rows][K/32]
  const uint8_t* s_packed;
  int64_t s_estride;
  const uint16_t* bias;   // [E][N] or null
  uint16_t* C;            // [rows][N]
  const int32_t* queue;   // grouped tile queue (BM rows per entry) or null
  int32_t* err;
  // indexed grouped calls: problem row r reads activation row gather[r] / topk (of
  // a_rows); the activation tile is then fetched with TMA gather4, four rows per copy
  const int32_t* gather;
  int32_t topk;
  int64_t a_rows;
  const float* scale2;  // second-level scales [E][N_pad] or null
};

struct Tile {
  int e, n0;
  int64_t rb, re;
};

__device__ __forceinline__ Tile tile_at(const Params& p, int64_t t) {
  Tile x;
  const int nb = (int)(t % p.num_n_tiles);
  const int64_t mt = t / p.num_n_tiles;
  x.n0 = nb * BN;
  if (p.queue) {
    x.e = __ldg(p.queue + 1 + 3 * mt);
    x.rb = __ldg(p.queue + 2 + 3 * mt);
    x.re = __ldg(p.queue + 3 + 3 * mt);
  } else {
    x.e = 0;
    x.rb = mt * BM;
    x.re = min64(p.rows, x.rb + BM);
  }
  return x;
}

// Scale word i of activation row `ar` (an act_row result, or -1 past the problem) for K
// step kb: the four scale bytes of groups 4 (IMG kb + i) .. + 3, padded with scale 1.
template <int KIND>
__device__ __forceinline__ uint32_t load_sf_word(const Params& p, int64_t ar, int kb, int i) {
  using T = KT<KIND>;
  const int G = p.K / T::GROUP;  // canonical groups per row
  const int g0 = (kb * T::IMG + i) * 4;
  if (ar < 0) return T::SF_PAD;
  const uint8_t* row = p.A_sf + ar * (int64_t)G;
  if ((G & 3) == 0 && g0 + 3 < G) return __ldg(reinterpret_cast<const uint32_t*>(row + g0));
  uint32_t w = 0;
  for (int j = 0; j < 4; ++j)
    w |= (uint32_t)(g0 + j < G ? __ldg(row + g0 + j) : (T::SF_PAD & 0xFFu)) << (8 * j);
  return w;
}

// The 4X kind's four scale words of activation row `ar` for K step kb (16 bytes: groups
// 16 kb .. 16 kb + 15), one 16-byte load where the row allows it.  (Sixteen 4-byte loads
// per lane and stage held the W4A4 GEMM back: a timing-only copy whose scale fetcher made
// no loads ran 157 against 199 us on (4096, 14336, 4096).)
template <int KIND>
__device__ __forceinline__ uint4 load_sf_row(const Params& p, int64_t ar, int kb) {
  using T = KT<KIND>;
  static_assert(T::IMG == 4, "four images per stage");
  const int G = p.K / T::GROUP;
  const int g0 = kb * 16;
  if (ar < 0) return make_uint4(T::SF_PAD, T::SF_PAD, T::SF_PAD, T::SF_PAD);
  const uint8_t* row = p.A_sf + ar * (int64_t)G;
  if (g0 + 15 < G && (reinterpret_cast<uintptr_t>(row + g0) & 15) == 0)
    return __ldg(reinterpret_cast<const uint4*>(row + g0));
  return make_uint4(load_sf_word<KIND>(p, ar, kb, 0), load_sf_word<KIND>(p, ar, kb, 1),
                    load_sf_word<KIND>(p, ar, kb, 2), load_sf_word<KIND>(p, ar, kb, 3));
}

// Activation row of problem row r: itself, or (indexed calls) the token of pair gather[r].
// Rows past the problem (tile tails) read row `fallback`; a pair outside [0, a_rows * topk)
// raises QW_ERR_INVALID_ARG and reads row 0.
__device__ __forceinline__ int64_t act_row(const Params& p, int64_t r, int64_t fallback) {
  if (r >= p.rows) r = fallback;
  if (!p.gather) return r;
  const int32_t pair = __ldg(p.gather + r);
  const int64_t tok = pair >= 0 ? (int64_t)(pair / p.topk) : -1;
  if (tok < 0 || tok >= p.a_rows) {
    set_error(p.err, QW_ERR_INVALID_ARG);
    return 0;
  }
  return tok;
}

// Four 128-byte rows of a tensor map with a one-row box into consecutive 128-byte rows of
// shared memory (the swizzle follows the destination address, as for a tiled load).
__device__ __forceinline__ void tma_gather4(void* dst, const void* map, uint64_t* bar, int32_t col,
                                            int32_t r0, int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// Wait for a phase without the CTA-wide abort shortcut (used when draining copies).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_w4a8_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const Params p) {
  using T = KT<KIND>;
  constexpr int SFA_BYTES = T::SFA_BYTES, SFB_BYTES = T::SFB_BYTES, SFB_CHUNK = T::SFB_CHUNK;
  constexpr int SF_STAGING = T::SF_STAGING, IMG = T::IMG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint8_t* sSFA = sB + STAGES * B_BYTES;
  uint8_t* sSFB = sSFA + STAGES * SFA_BYTES;
  uint8_t* sStage = sSFB + STAGES * SFB_BYTES;  // staged A scale images
  int32_t* sIdx = reinterpret_cast<int32_t*>(sStage + SF_STAGING * SFA_BYTES);  // [BM] rows
  uint64_t* full = reinterpret_cast<uint64_t*>(sIdx + BM);
  uint64_t* empty = full + STAGES;
  uint64_t* sfull = empty + STAGES;   // staging slot written (32 fetcher lanes)
  uint64_t* sempty = sfull + SF_STAGING;  // staging slot read (writer)
  uint64_t* acc_full = sempty + SF_STAGING;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* final_bar = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel may start its own set-up on SMs this grid has left
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + 32);  // producer arrive.expect_tx + 32 scale-writer lanes
      mbar_init(&empty[s], 1);      // MMA commit
    }
    for (int s = 0; s < SF_STAGING; ++s) {
      mbar_init(&sfull[s], 32);
      mbar_init(&sempty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, NUM_EPI_WARPS);
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
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
  const int KB = p.K_pad / T::KSTEP;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 issues every copy.  Indexed calls: the whole warp looks up the next tile's 128
    // activation rows while lane 0 streams the current one, and hands them over through
    // shared memory at the tile boundary.
    int32_t nxt[4];
    auto rows_of = [&](int64_t t) {
      const Tile y = tile_at(p, t);
#pragma unroll
      for (int j = 0; j < 4; ++j) nxt[j] = (int32_t)act_row(p, y.rb + 32 * j + lane, y.rb);
    };
    if (p.gather && blockIdx.x < num_tiles) rows_of(blockIdx.x);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_phase = 0;  // per-stage bitmasks for the final drain
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const Tile x = tile_at(p, t);
      if (p.gather) {
        __syncwarp();  // lane 0 is done with the previous tile's rows
#pragma unroll
        for (int j = 0; j < 4; ++j) sIdx[32 * j + lane] = nxt[j];
        __syncwarp();
        if (t + gridDim.x < num_tiles) rows_of(t + gridDim.x);
      }
      if (lane == 0) {
        const int nchunks = (x.n0 + 128 < p.N_pad) ? 2 : 1;
        const uint8_t* sfb = p.s_packed + x.e * p.s_estride;
        // indexed calls gather only the tile's own rows (groups of four): the rows past
        // them keep stale shared memory and produce outputs that are never stored
        const int ngather = p.gather ? (int)((min64(x.re - x.rb, BM) + 3) / 4) : 0;
        const uint32_t a_tx = p.gather ? (uint32_t)ngather * 4 * BK : A_BYTES;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], a_tx + T::B_TX + nchunks * SFB_CHUNK);
          if (p.gather) {
            for (int i = 0; i < ngather; ++i)
              tma_gather4(sA + stage * A_BYTES + i * 4 * BK, &tmA, &full[stage], kb * BK,
                          sIdx[4 * i], sIdx[4 * i + 1], sIdx[4 * i + 2], sIdx[4 * i + 3]);
          } else {
            tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, (int32_t)x.rb);
          }
          tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK,
                      x.e * p.N_pad + x.n0);
          for (int c = 0; c < nchunks; ++c)
            bulk_load(sSFB + stage * SFB_BYTES + c * SFB_CHUNK,
                      sfb + ((int64_t)(x.n0 / 128 + c) * KB + kb) * SFB_CHUNK, SFB_CHUNK,
                      &full[stage]);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    }
    // let every copy lane 0 issued land before shared memory goes away
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) drain_wait(&full[s], (issued_phase >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // scale images into TMEM: image i of A at columns sfa + 4i, image i of B's two
          // 128-row chunks at sfb + 8i and sfb + 8i + 4 (1X: one image per stage, read by
          // byte selector; 4X: one image per MMA)
          const uint32_t sfa_col = tbase + SF_COL0 + stage * T::SF_COLS_PER_STAGE;
          const uint32_t sfb_col = sfa_col + 4 * IMG;
#pragma unroll
          for (int i = 0; i < IMG; ++i) {
            tc_cp_32x128b_warpx4(sfa_col + 4 * i,
                                 smem_desc(smem_u32(sSFA + stage * SFA_BYTES + i * 512), 0, 128, 0));
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tc_cp_32x128b_warpx4(
                  sfb_col + 8 * i + 4 * c,
                  smem_desc(smem_u32(sSFB + stage * SFB_BYTES + c * SFB_CHUNK + i * 512), 0, 128, 0));
          }
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {  // 32 bytes of each row per MMA
            const uint64_t ad = smem_desc(a0 + kk * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b0 + kk * 32, 16, 1024, 2);
            if constexpr (T::NV) {
              tc_mma_mxf4nvf4_4x(tbase, ad, bd, idesc<KIND>(), sfa_col + 4 * kk, sfb_col + 8 * kk,
                                 (kb | kk) != 0 ? 1u : 0u);
            } else {
              const uint32_t id = idesc<KIND>() | ((uint32_t)kk << 4) | ((uint32_t)kk << 29);
              tc_mma_mxf8f6f4(tbase, ad, bd, id, sfa_col, sfb_col, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1u;
      }
      // every MMA this thread issued has finished before TMEM is released
      tc_commit(final_bar);
      drain_wait(final_bar, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ A scale fetcher
    // Global loads run ahead of the staging writes; this warp never fences.  1X kinds: a
    // three-deep register ring shifted each stage.  4X: two register sets of four words per
    // lane used in turn, two stages ahead (no copies between them: a copy of a register
    // whose load is in flight waits for it; the shifted ring ran the W4A4 GEMM at 166
    // against 162 us on (4096, 14336, 4096), and cost the W4A8 headline nothing).
    constexpr int AHEAD = 3;
    int64_t lt = blockIdx.x;  // load cursor: tile and K step
    int lkb = 0;
    int64_t ar[4];            // activation rows of this lane's four tile rows (-1: none)
    auto rows_of = [&](int64_t t) {
      const Tile y = tile_at(p, t);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t r = y.rb + 32 * j + lane;
        ar[j] = r < p.rows ? act_row(p, r, y.rb) : -1;
      }
    };
    if (lt < num_tiles) rows_of(lt);
    // one ring entry: image i, word j = scales of row 32 j + lane for the stage
    struct Entry {
      uint4 v[IMG];
    };
    auto load_next = [&]() {
      Entry e;
#pragma unroll
      for (int i = 0; i < IMG; ++i) e.v[i] = make_uint4(T::SF_PAD, T::SF_PAD, T::SF_PAD, T::SF_PAD);
      if (lt < num_tiles) {
        if constexpr (IMG == 4) {
          // a row's 16 bytes hold word i of every image i
          uint4 r[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) r[j] = load_sf_row<KIND>(p, ar[j], lkb);
          e.v[0] = make_uint4(r[0].x, r[1].x, r[2].x, r[3].x);
          e.v[1] = make_uint4(r[0].y, r[1].y, r[2].y, r[3].y);
          e.v[2] = make_uint4(r[0].z, r[1].z, r[2].z, r[3].z);
          e.v[3] = make_uint4(r[0].w, r[1].w, r[2].w, r[3].w);
        } else {
#pragma unroll
          for (int i = 0; i < IMG; ++i) {
            e.v[i].x = load_sf_word<KIND>(p, ar[0], lkb, i);
            e.v[i].y = load_sf_word<KIND>(p, ar[1], lkb, i);
            e.v[i].z = load_sf_word<KIND>(p, ar[2], lkb, i);
            e.v[i].w = load_sf_word<KIND>(p, ar[3], lkb, i);
          }
        }
        if (++lkb == KB) {
          lkb = 0;
          lt += gridDim.x;
          if (lt < num_tiles) rows_of(lt);
        }
      }
      return e;
    };
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    auto write = [&](const Entry& e) {
#pragma unroll
      for (int i = 0; i < IMG; ++i)
        *reinterpret_cast<uint4*>(sStage + slot * SFA_BYTES + i * 512 + lane * 16) = e.v[i];
      mbar_arrive(&sfull[slot]);
    };
    if constexpr (IMG == 4) {
      Entry set_a = load_next(), set_b = load_next();
      uint32_t n = 0;  // staging writes so far (even: set_a's turn)
      for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++n) {
          if (!mbar_wait(&sempty[slot], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          if (n & 1u) {
            write(set_b);
            set_b = load_next();
          } else {
            write(set_a);
            set_a = load_next();
          }
          if (++slot == SF_STAGING) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    } else {
      Entry ring[AHEAD];
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) ring[i] = load_next();
      for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&sempty[slot], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          write(ring[0]);
#pragma unroll
          for (int i = 0; i + 1 < AHEAD; ++i) ring[i] = ring[i + 1];
          ring[AHEAD - 1] = load_next();
          if (++slot == SF_STAGING) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ A scale writer
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&sfull[slot], sphase, abort_flag, p.err) ||
            !mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int i = 0; i < IMG; ++i) {
          const uint4 v =
              *reinterpret_cast<const uint4*>(sStage + slot * SFA_BYTES + i * 512 + lane * 16);
          *reinterpret_cast<uint4*>(sSFA + stage * SFA_BYTES + i * 512 + lane * 16) = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[slot]);
        fence_proxy_async_smem();  // only shared-memory accesses are outstanding here
        mbar_arrive(&full[stage]);
        if (++slot == SF_STAGING) {
          slot = 0;
          sphase ^= 1u;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                        // TMEM lane quadrant of this warp
    const int half = (warp - EPI_WARP0) / 4;       // accumulator columns [128 half, +128)
    uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const Tile x = tile_at(p, t);
      if (!mbar_wait(acc_full, acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int64_t row = x.rb + 32 * q + lane;
      const int col0 = x.n0 + 128 * half;
      if (p.scale2) {
        // second-level scales: C = t[n] * acc + bias[n], one 32-column chunk at a time,
        // stored as it is done (the accumulator is released after the last chunk)
        const float* tp = p.scale2 + (int64_t)x.e * p.N_pad + col0;
        uint16_t* crow = p.C + row * (int64_t)p.N + col0;
        const bool vec = col0 + 128 <= p.N && (p.N & 7) == 0;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tc_ld_32x32b_x32(tbase + ((uint32_t)(32 * q) << 16) + 128 * half + 32 * j, r);
          tc_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = col0 + 32 * j + 2 * i;
            const float2 t2 = __ldg(reinterpret_cast<const float2*>(tp + 32 * j) + i);
            float b0 = 0.f, b1 = 0.f;
            if (p.bias) {
              const uint16_t* bp = p.bias + (int64_t)x.e * p.N + c;
              if (c < p.N) b0 = __uint_as_float((uint32_t)__ldg(bp) << 16);
              if (c + 1 < p.N) b1 = __uint_as_float((uint32_t)__ldg(bp + 1) << 16);
            }
            pk[i] = pack_bf16x2(fmaf(__uint_as_float(r[2 * i]), t2.x, b0),
                                fmaf(__uint_as_float(r[2 * i + 1]), t2.y, b1));
          }
          if (row < x.re) {
            if (vec) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                reinterpret_cast<uint4*>(crow + 32 * j)[v] =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = col0 + 32 * j + 2 * i;
                if (c < p.N) crow[32 * j + 2 * i] = (uint16_t)(pk[i] & 0xFFFFu);
                if (c + 1 < p.N) crow[32 * j + 2 * i + 1] = (uint16_t)(pk[i] >> 16);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        acc_phase ^= 1u;
        continue;
      }
      uint32_t packed[64];
      // two 32-column loads in flight per wait: the drain gates the next tile's first MMA
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t r[2][32];
        const uint32_t ta = tbase + ((uint32_t)(32 * q) << 16) + 128 * half + 64 * jj;
        tc_ld_32x32b_x32(ta, r[0]);
        tc_ld_32x32b_x32(ta + 32, r[1]);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 2 * jj + h;
          float b[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) b[i] = 0.f;
          if (p.bias) {
            const uint16_t* bp = p.bias + (int64_t)x.e * p.N + col0 + 32 * j;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + 32 * j + i < p.N) b[i] = __uint_as_float((uint32_t)__ldg(bp + i) << 16);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[16 * j + i] = pack_bf16x2(__uint_as_float(r[h][2 * i]) + b[2 * i],
                                             __uint_as_float(r[h][2 * i + 1]) + b[2 * i + 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      if (row < x.re) {
        uint16_t* crow = p.C + row * (int64_t)p.N + col0;
        if (col0 + 128 <= p.N && (p.N & 7) == 0) {
#pragma unroll
          for (int v = 0; v < 16; ++v)
            reinterpret_cast<uint4*>(crow)[v] =
                make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (col0 + 2 * i < p.N) crow[2 * i] = (uint16_t)(packed[i] & 0xFFFFu);
            if (col0 + 2 * i + 1 < p.N) crow[2 * i + 1] = (uint16_t)(packed[i] >> 16);
          }
        }
      }
      acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
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

}  // namespace

uint64_t gemm_w4a8_workspace(const qw_packed_desc& d, int64_t max_rows) {
  return d.E > 1 ? tile_queue_bytes(d.E, max_rows, BM) : 0;
}

qw_status launch_gemm_w4a8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* A_sf, const void* bias, void* C,
                           const RowSet& rs, void* ws, uint64_t ws_bytes, int32_t* err,
                           cudaStream_t st) {
  if (rs.rows == 0) return QW_OK;
  auto enc = encode_fn();
  if (!enc) return QW_ERR_CUDA;
  if (rs.rows > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  const bool w8 = d.wfmt == QW_W_MXFP8_G32;
  const bool nv = d.wfmt == QW_W_NVFP4_G16;  // packed E2M1 activations: K / 2 bytes per row
  const int64_t a_row_bytes = nv ? d.K / 2 : d.K;

  CUtensorMap tmA, tmB;
  {
    // indexed calls read the unpermuted activations one row per box (gather4 copies)
    const bool gather = rs.gather != nullptr;
    if (gather && (rs.a_rows < 1 || rs.a_rows > 0x7FFFFFFFLL)) return QW_ERR_UNSUPPORTED;
    cuuint64_t gdim[2] = {(cuuint64_t)a_row_bytes, (cuuint64_t)(gather ? rs.a_rows : rs.rows)};
    cuuint64_t gstr[1] = {(cuuint64_t)a_row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)BK, gather ? 1u : (cuuint32_t)BM};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(A), gdim, gstr, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QW_ERR_ALIGNMENT;
  }
  {
    // W4A8: E2M1 codes unpacked by TMA (K_pad elements per row); W8A8: E4M3 bytes;
    // W4A4: packed E2M1 bytes (K_pad / 2 per row)
    cuuint64_t gdim[2] = {(cuuint64_t)(nv ? d.K_pad / 2 : d.K_pad),
                          (cuuint64_t)d.E * (cuuint64_t)d.N_pad};
    cuuint64_t gstr[1] = {(cuuint64_t)(w8 ? d.K_pad : d.K_pad / 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmB,
            (w8 || nv) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2,
            const_cast<void*>(w_packed), gdim,
            gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QW_ERR_ALIGNMENT;
  }

  Params p{};
  p.rows = rs.rows;
  p.N = d.N;
  p.N_pad = d.N_pad;
  p.K = d.K;
  p.K_pad = d.K_pad;
  p.num_n_tiles = (d.N + BN - 1) / BN;
  p.num_m_tiles = (int32_t)((rs.rows + BM - 1) / BM);
  p.A_sf = static_cast<const uint8_t*>(A_sf);
  p.s_packed = static_cast<const uint8_t*>(s_packed);
  p.s_estride = (int64_t)d.s_expert_stride;
  p.bias = static_cast<const uint16_t*>(bias);
  p.scale2 = rs.scale2;
  p.C = static_cast<uint16_t*>(C);
  p.err = err;
  p.gather = rs.gather;
  p.topk = rs.topk;
  p.a_rows = rs.a_rows;
  int64_t max_m_tiles = p.num_m_tiles;
  if (rs.offsets) {
    const uint64_t need = tile_queue_bytes(rs.E, rs.rows, BM);
    if (ws == nullptr || ws_bytes < need) return QW_ERR_WORKSPACE;
    int32_t* queue = static_cast<int32_t*>(ws);
    max_m_tiles = (int64_t)(need / 4 - 1) / 3;
    qw_status s = launch_build_tile_queue(rs.offsets, rs.E, BM, rs.rows, queue, max_m_tiles, err,
                                           st);
    if (s != QW_OK) return s;
    p.queue = queue;
  }

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gemm_w4a8_kernel<kW4A8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)KT<kW4A8>::SMEM_BYTES);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gemm_w4a8_kernel<kW8A8>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)KT<kW8A8>::SMEM_BYTES);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gemm_w4a8_kernel<kW4A4>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)KT<kW4A4>::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return QW_ERR_CUDA;

  const int64_t tiles_max = max_m_tiles * p.num_n_tiles;
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(tiles_max < sms ? (tiles_max < 1 ? 1 : tiles_max) : sms);
  if (w8)
    return launch_pdl(gemm_w4a8_kernel<kW8A8>, dim3(grid), dim3(NUM_THREADS),
                      KT<kW8A8>::SMEM_BYTES, st, tmA, tmB, p);
  if (nv)
    return launch_pdl(gemm_w4a8_kernel<kW4A4>, dim3(grid), dim3(NUM_THREADS),
                      KT<kW4A4>::SMEM_BYTES, st, tmA, tmB, p);
  return launch_pdl(gemm_w4a8_kernel<kW4A8>, dim3(grid), dim3(NUM_THREADS),
                    KT<kW4A8>::SMEM_BYTES, st, tmA, tmB, p);
}

}  // namespace qw
