// qw_internal.h - host-side launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/qw.h"

namespace qw {

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Packed-layout geometry shared by repack and the GEMM kernels.
constexpr int kIntGroup = 128;       // K elements per BF16 scale (INT formats)
constexpr int kMxGroup = 32;         // K elements per E8M0 scale (MX formats)
constexpr int kInt4BlockBytes = 1024;  // 16 rows x 128 k of INT4, fragment order
constexpr int kInt2BlockBytes = 512;   // 16 rows x 128 k of INT2, fragment order
constexpr int kInt3BlockBytes = 768;   // 16 rows x 128 k of INT3 (two bit planes)
constexpr int kFp8BlockBytes = 2048;   // 16 rows x 128 k of E4M3 codes, fragment order
constexpr int kInt1BlockBytes = 256;   // 16 rows x 128 k of INT1 sign bits, fragment order
constexpr int kFp4BlockBytes = 1024;   // 16 rows x 128 k of E2M1 codes, fragment order
// Format codes of the WnA16 kernels' templates: the integer bit width (4, 3, 2, 1), 8 for
// E4M3 weights and kBitsFp4 for E2M1 weights (FP4 codes in the INT4 block geometry).
constexpr int kBitsFp4 = 5;
// Bytes of one packed 16 x 128 block of a WnA16 format code.
__host__ __device__ constexpr int wna16_block_bytes(int bits) {
  return bits == kBitsFp4 ? kFp4BlockBytes : bits * 256;
}
constexpr int kSfChunkBytes = 512;     // 128 rows x 4 groups of E8M0 scales
constexpr int kNvGroup = 16;           // K elements per E4M3 scale (NVFP4)
constexpr int kNvChunkBytes = 2048;    // 128 rows x 16 groups of E4M3 scales (NVFP4)

qw_status launch_repack(const qw_packed_desc& d, const void* w_canon, const void* s_canon,
                        void* w_packed, void* s_packed, int32_t* err, cudaStream_t st);
qw_status launch_unpack(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                        void* w_canon, void* s_canon, int32_t* err, cudaStream_t st);
// second-level scales: fill the packed plane with 1.0, copy [E][N] <-> [E][N_pad]
qw_status launch_scale2_fill(float* t_packed, int64_t n, cudaStream_t st);
qw_status launch_scale2_repack(const float* t_canon, float* t_packed, int32_t E, int32_t N,
                               int32_t N_pad, int32_t* err, cudaStream_t st);
qw_status launch_scale2_unpack(const float* t_packed, float* t_canon, int32_t E, int32_t N,
                               int32_t N_pad, cudaStream_t st);

// Rows of a GEMM call: dense (offsets == nullptr, rows [0, M)) or grouped by expert
// (device offsets [E+1]; the work list of (expert, row tile) is built on the device).
struct RowSet {
  int64_t rows;                // M (dense) or total rows (grouped)
  const int32_t* offsets;      // device [E+1] or nullptr
  int32_t E;
  // Indexed grouped calls: row r of the problem is activation row gather[r] / topk of an
  // unpermuted [a_rows][K] input (gather = the router's sorted pair ids); else nullptr.
  const int32_t* gather = nullptr;
  int32_t topk = 1;
  int64_t a_rows = 0;
  // second-level scales: device FP32 [E][N_pad] multiplying each output channel's sum
  // before the bias, or nullptr
  const float* scale2 = nullptr;
};

// Small-M W4A16: tensor-core GEMV over the fragment-ordered packed weights.
qw_status launch_gemv_w4a16(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                            const void* A, const void* bias, void* C, const RowSet& rs,
                            void* ws, uint64_t ws_bytes, int32_t* err, cudaStream_t st);
uint64_t gemv_w4a16_workspace(const qw_packed_desc& d, int64_t max_rows);

// Large-M W4A16: in-SM dequantization into tensor memory + tcgen05 BF16 GEMM.
qw_status launch_gemm_w4a16_tc(const qw_packed_desc& d, const void* w_packed,
                               const void* s_packed, const void* A, const void* bias, void* C,
                               const RowSet& rs, void* ws, uint64_t ws_bytes, int32_t* err,
                               cudaStream_t st);
uint64_t gemm_w4a16_tc_workspace(const qw_packed_desc& d, int64_t max_rows);

// Rows from which W4A16 runs on the tensor-core path (dense M above it, or a grouped call
// averaging at least this many rows per expert); below it the GEMV streams the weights.
// Measured on GB300 (14336 x 4096 INT4): the GEMV is faster at M <= 16, the tcgen05 path
// from M = 32 (23.8 vs 36.3 us); MoE up projection E=128: GEMV 214 us vs tcgen05 114 us
// at 16 rows per expert.
constexpr int64_t kW4A16TensorCoreRows = 16;

// Activation-side MoE steps (act.cu).
qw_status launch_quantize_mxfp8(const void* A, int64_t rows, int32_t K, void* Q, void* SF,
                                int32_t* err, cudaStream_t st);
qw_status launch_silu_mul(const void* GU, int64_t rows, int32_t I, void* Y, cudaStream_t st);
qw_status launch_moe_combine(const void* Y, const int32_t* sorted_pairs, const int32_t* topk_ids,
                             const float* logits, int32_t T, int32_t E, int32_t topk, int32_t N,
                             void* out, int32_t* inv, int32_t* err, cudaStream_t st);

// Large-M W4A8: TMA + tcgen05 block-scaled GEMM.
qw_status launch_gemm_w4a8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* A_sf, const void* bias, void* C,
                           const RowSet& rs, void* ws, uint64_t ws_bytes, int32_t* err,
                           cudaStream_t st);
uint64_t gemm_w4a8_workspace(const qw_packed_desc& d, int64_t max_rows);

// Dense W4A8 (MXFP4 weights) calls of at most this many rows whose staged activations
// (FP16 B fragments and FP32 scales of every group) fit kW4A8GemvMaxSmem run the
// streaming GEMV.
constexpr int kW4A8GemvRows = 8;
constexpr size_t kW4A8GemvMaxSmem = 96 * 1024;
constexpr size_t w4a8_gemv_smem_bytes(int K, int M) {
  return (size_t)(K / 32) * ((size_t)M * 64 + 32);
}
qw_status launch_gemv_w4a8(const qw_packed_desc& d, const void* w_packed, const void* s_packed,
                           const void* A, const void* A_sf, const void* bias, const float* scale2,
                           void* C, int M, int32_t* err, cudaStream_t st);

// MoE scheduling.
qw_status launch_moe_route(const float* logits, int32_t T, int32_t E, int32_t topk,
                           int32_t* topk_ids, int32_t* sorted_pairs, int32_t* offsets, void* ws,
                           uint64_t ws_bytes, int32_t* err, cudaStream_t st);
uint64_t moe_route_workspace(int32_t T, int32_t E, int32_t topk);
qw_status launch_moe_permute(int32_t afmt, const void* A, const void* A_sf, int32_t K,
                             const int32_t* sorted_pairs, int64_t P, int32_t topk,
                             void* A_sorted, void* A_sf_sorted, cudaStream_t st);

// Device tile queue for grouped GEMMs: entry = (expert, row_begin, row_end) for each
// tile of `tile_rows` rows of every expert; count at queue[0].
uint64_t tile_queue_bytes(int32_t E, int64_t rows, int32_t tile_rows);
// Offsets outside [0, total_rows] or decreasing are reported (QW_ERR_INVALID_ARG) and
// produce no tiles.
qw_status launch_build_tile_queue(const int32_t* offsets, int32_t E, int32_t tile_rows,
                                  int64_t total_rows, int32_t* queue, int64_t max_entries,
                                  int32_t* err, cudaStream_t st);

qw_status launch_wait_timeout_probe(int32_t* err, int64_t limit_ns, cudaStream_t st);
// Diagnostics: a plain streaming read of `bytes` at `src` (one fold word per CTA to `sink`).
qw_status launch_stream_read(const void* src, uint64_t bytes, uint32_t* sink, bool chained,
                             cudaStream_t st);
// Diagnostics: the tcgen05 MMA issue rate (qw_mma_rate_probe; arguments checked there).
qw_status launch_mma_probe(int mode, int n, int iters, uint64_t* out, int32_t* err,
                           cudaStream_t st);

}  // namespace qw
