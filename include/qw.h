/*
 * qw.h - C ABI of the GB300 (sm_103a) low-bit weight-quantized GEMM library.
 *
 * The operations follow the Humming kernel library as its announcement describes it
 * (spke.com, "quantized推論のための高速かつ柔軟なカーネル「Humming」を発表"):
 *   - preprocessing validates parameters, pads dimensions and repacks the weight and
 *     scale tensors into kernel-friendly layouts (section "ワークロードごとのチューニング
 *     とJITコンパイル");
 *   - dequantization and scaling run inside the kernel; scale and bias are fused into
 *     the output stage (section "フォーマットとアーキテクチャを横断して共有される
 *     CUDAコンポーネント");
 *   - dense and MoE GEMMs have their own scheduling; MoE has a Grouped path over
 *     expert-contiguous tokens (sections "WnA16" and "W8A8 / W4A8 / W4A4");
 *   - symmetric integer weights are converted at preprocessing into a zero-exponent
 *     code for fast dequantization (section "量子化サポート").
 * Formats: W4A16 = group-128 symmetric INT4 / INT3 weights with BF16 scales times BF16
 * activations; W4A8 = MXFP4 (E2M1 + group-32 E8M0) weights times MXFP8 (E4M3 + group-32
 * E8M0) activations (aireiter.com "vLLM Humming performance benchmark", section
 * "H100 group-32 W4A8").  Also on the same kernels (announcement sections "WnA16" and
 * "W8A8 / W4A8 / W4A4"): INT2, asymmetric INT4 and FP8 E4M3 weights times BF16; MXFP8
 * times MXFP8; NVFP4 times NVFP4; and an optional FP32 second-level scale per output
 * channel on any of them (QW_W_SCALE2).
 *
 * Conventions shared by every entry point
 *   - The caller owns every buffer.  Pointers are DEVICE pointers unless the comment
 *     says "host".  The library never allocates, never synchronises the stream (except
 *     qw_read_error, which exists to do so) and never exits or asserts.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  All
 *     device work of a call is enqueued on it, in order.  The W4A16 GEMV kernels (M <= 16,
 *     and grouped calls below the tensor-core switch) are launched as programmatic
 *     dependents of the previous kernel on the stream: they may start reading w_packed and
 *     s_packed while that kernel finishes, and wait for it before anything else.  So the
 *     weights of such a call must not be written by the kernel enqueued immediately before
 *     it (qw_repack followed at once by a GEMV is fine: qw_repack's kernels do not release
 *     their dependents early, so the GEMV starts after they complete).
 *   - Shape, pointer-alignment and size errors are detected on the host before any
 *     launch and returned as a qw_status; nothing is enqueued in that case.
 *   - Value errors found on the device (while repacking: an INT4 code -8, an INT3 code
 *     -4, an INT2 code -2, a zero point above 15, an E4M3 NaN code, an E8M0 scale 0xFF,
 *     a negative or NaN NVFP4 scale, a non-finite second-level scale; a NaN router
 *     logit; a non-finite input to the MXFP8 quantizer - the GEMMs take their operands
 *     as valid) and bounded waits that gave up are
 *     reported through `d_err` (int32 in device memory, may be NULL): the first error
 *     code written wins (atomic compare-and-swap from 0).  The caller zeroes it and
 *     reads it when convenient, e.g. with qw_read_error.
 *   - Weights are logically [N][K] (output x input), activations [M][K] row-major,
 *     results [M][N] row-major BF16 (round to nearest even of the FP32 accumulator).
 *   - Every kernel is deterministic: no floating-point atomics, fixed reduction order.
 */
#ifndef QW_H
#define QW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qw_status {
  QW_OK = 0,
  QW_ERR_INVALID_ARG = 1,  /* null pointer, non-positive or inconsistent size        */
  QW_ERR_UNSUPPORTED = 2,  /* format / shape combination this build does not run      */
  QW_ERR_ALIGNMENT = 3,    /* a pointer or pitch violates the stated alignment         */
  QW_ERR_VALUE = 4,        /* a code outside its format's valid set (device-detected)  */
  QW_ERR_WORKSPACE = 5,    /* workspace missing or smaller than the queried size       */
  QW_ERR_TIMEOUT = 6,      /* a bounded device wait gave up (device-detected)          */
  QW_ERR_CUDA = 7          /* a CUDA runtime / driver call failed                      */
} qw_status;

typedef enum qw_wfmt {
  QW_W_INT4_G128_BF16 = 0, /* symmetric INT4 in [-7,7], BF16 scale per 128 along K      */
  QW_W_INT3_G128_BF16 = 1, /* symmetric INT3 in [-3,3], BF16 scale per 128 along K      */
  QW_W_MXFP4_G32 = 2,      /* E2M1 codes, E8M0 scale per 32 along K                      */
  QW_W_MXFP8_G32 = 3,      /* E4M3 codes, E8M0 scale per 32 along K (the W8A8 MX kind)    */
  QW_W_NVFP4_G16 = 4,      /* E2M1 codes, unsigned E4M3 scale per 16 along K (W4A4)       */
  QW_W_UINT4ZP_G128_BF16 = 5, /* unsigned 4-bit codes, BF16 scale and zero point per 128:
                                 w = s * (q - z) (asymmetric INT4)                         */
  QW_W_INT2_G128_BF16 = 6, /* symmetric INT2 in {-1, 0, 1}, BF16 scale per 128 along K    */
  QW_W_FP8E4M3_G128_BF16 = 7, /* E4M3 codes, BF16 scale per 128 along K (FP8-weight WnA16) */
  QW_W_INT1_G128_BF16 = 8, /* INT1 sign codes: bit b is the weight 2b - 1 (-1 or +1), BF16
                              scale per 128 along K                                     */
  QW_W_FP4E2M1_G128_BF16 = 9 /* E2M1 codes, BF16 scale per 128 along K (FP4-weight WnA16) */
} qw_wfmt;

/* Second-level scales (the announcement, section "統一されたquantization表現": the
 * quantization description carries second-level scales as a parameter of its own).  OR'ed
 * into any qw_wfmt, it adds one FP32 scale t per output channel and expert on top of the
 * format's group scales:  C[m][n] = bf16( t[e][n] * sum_k a[m,k] * w[n,k] + bias[n] ).
 * The descriptor's s_bytes then also covers an FP32 plane [E][N_pad] at byte offset
 * E * s_expert_stride of s_packed; qw_repack sets it to 1.0 and qw_repack_scale2 writes it. */
#define QW_W_SCALE2 0x100

typedef enum qw_afmt {
  QW_A_BF16 = 0,           /* BF16 [rows][K]                                          */
  QW_A_MXFP8_G32 = 1,      /* E4M3 codes [rows][K] + E8M0 scales [rows][K/32]          */
  QW_A_NVFP4_G16 = 2       /* E2M1 codes [rows][K/2] (even k in the low nibble) +
                              unsigned E4M3 scales [rows][K/16]                            */
} qw_afmt;

/* Description of one repacked weight set (E experts; E = 1 for a dense layer).
 * Filled by qw_repack_query; treat as read-only. */
typedef struct qw_packed_desc {
  int32_t wfmt;            /* qw_wfmt, possibly | QW_W_SCALE2                          */
  int32_t E, N, K;         /* logical sizes                                            */
  int32_t N_pad, K_pad;    /* padded sizes of the packed layout                        */
  int32_t group;           /* 128 (INT, FP8E4M3, FP4E2M1), 32 (MXFP4 / MXFP8) or 16
                              (NVFP4)                                                  */
  int32_t reserved;
  uint64_t w_bytes;        /* size of w_packed in bytes (all experts)                  */
  uint64_t s_bytes;        /* size of s_packed in bytes (all experts)                  */
  uint64_t w_expert_stride;/* bytes between consecutive experts in w_packed            */
  uint64_t s_expert_stride;/* bytes between consecutive experts in s_packed            */
} qw_packed_desc;

/* Status text (static storage; never NULL). */
const char* qw_status_str(int32_t status);

/* ABI version of this library (major * 100 + minor). */
int32_t qw_version(void);

/* --------------------------------------------------------------------------------------
 * qw_repack_query - sizes of the packed layout for E experts of an N x K weight.
 * Requirements: E >= 1, N >= 1, K >= 1; K % 128 == 0 for the INT formats, K % 32 == 0
 * for MXFP4 / MXFP8 / NVFP4.  Padding: INT formats pad N to a multiple of 16; the MX
 * formats pad N to a multiple of 128 and K to a multiple of 128 (NVFP4: 256).  N and K
 * are at most 2^31 - 256 (so the padded sizes fit in int32) and N_pad * E < 2^31.  `out`
 * is a host pointer.
 * Returns QW_ERR_INVALID_ARG / QW_ERR_UNSUPPORTED on a bad request, else QW_OK.
 */
qw_status qw_repack_query(int32_t wfmt, int32_t E, int32_t N, int32_t K, qw_packed_desc* out);

/* --------------------------------------------------------------------------------------
 * qw_repack - validate, pad and repack canonical weights and scales (the preprocessing
 * step of the spke.com announcement, section "ワークロードごとのチューニングとJITコンパイル").
 *
 * Canonical inputs (device, contiguous, experts outermost):
 *   INT4:  w_canon uint32 [E][N][K/8]; element k = 8j+i at bits [4i,4i+4) of word j,
 *          two's complement.  s_canon BF16 [E][N][K/128].
 *   INT3:  w_canon uint32 [E][N][K/32][3]; a 96-bit little-endian stream per 32
 *          elements, element i at stream bits [3i,3i+3), two's complement.
 *          s_canon BF16 [E][N][K/128].
 *   MXFP4: w_canon uint8 [E][N][K/2], even k in the low nibble.  s_canon uint8 E8M0
 *          [E][N][K/32].
 *   MXFP8: w_canon uint8 [E][N][K] E4M3 codes.  s_canon uint8 E8M0 [E][N][K/32].
 *   NVFP4: w_canon uint8 [E][N][K/2] as MXFP4.  s_canon uint8 E4M3 [E][N][K/16] (unsigned).
 *   INT2:  w_canon uint32 [E][N][K/16]; element k = 16j+i at bits [2i,2i+2) of word j,
 *          two's complement (-2 rejected).  s_canon BF16 [E][N][K/128].
 *   FP8E4M3: w_canon uint8 [E][N][K] E4M3 codes.  s_canon BF16 [E][N][K/128].
 *   INT1:  w_canon uint32 [E][N][K/32]; element k = 32j+i is bit i of word j, bit b
 *          standing for the weight 2b - 1.  s_canon BF16 [E][N][K/128].
 *   FP4E2M1: w_canon uint8 [E][N][K/2] E2M1 codes, even k in the low nibble.  s_canon BF16
 *          [E][N][K/128].
 *   UINT4ZP: w_canon uint32 [E][N][K/8] packed as INT4 but read unsigned (q in [0, 15]).
 *          s_canon uint32 [E][N][K/128]: bits 0-15 the BF16 scale, bits 16-23 the zero
 *          point z in [0, 15], bits 24-31 zero (else a value error).
 * Packed outputs (device, sizes from `desc`, 256-byte aligned):
 *   INT4:  per expert [K/128][N_pad/16] blocks of 1 KiB: 32 lanes x 8 words; word s of
 *          lane l = 4g + t holds the eight weights lane l feeds to the s-th m16n8k16 MMA of
 *          the group, as excess-8 nibbles (q + 8): nibble i -> row g + 8 (i & 1),
 *          k = 16s + 4t + 2 ((i >> 1) & 1) + (i >> 2) - rows g and g + 8 at the four k's
 *          16s + 4t .. 16s + 4t + 3 (also the register layout of a 16-lane TMEM store).
 *          Scales BF16 [K/128][N_pad].
 *   INT3:  per expert [K/128][N_pad/16] blocks of 768 B: 32 lanes x 4 words, then 32
 *          lanes x 2 words; the lane's six words hold u = q + 4 for its 64 weights (the
 *          INT4 (row, k) assignment) as 32 pairs, pair j = 4s + r for rows g + 8 (r & 1)
 *          at k = 16s + 4t + 2 (r >> 1) + h: for j < 30, bits 3 (j % 5) + 16h of word
 *          j / 5; pairs 30 and 31 keep bit i of u at bit 15 + 16h of word i and 3 + i.
 *          Scales BF16 [K/128][N_pad].
 *   MXFP4: codes uint8 [N_pad][K_pad/2] (canonical order, zero-padded); scales E8M0 in
 *          512-byte chunks per 128 rows x 4 groups, chunk (r/128, g/4) at
 *          ((r/128) * (K_pad/128) + g/4) * 512, byte (r%32)*16 + ((r%128)/32)*4 + g%4;
 *          padding bytes are 127 (scale 1).
 *   MXFP8: codes uint8 [N_pad][K_pad] (canonical order, zero-padded); scales as MXFP4.
 *   INT2:  per expert [K/128][N_pad/16] blocks of 512 B: 32 lanes x 4 words holding q + 2
 *          for the lane's 64 weights (the INT4 (row, k) assignment): pair j = 4s + r at
 *          bits 2 (4 (s % 2) + r) + 16h of word s / 2.  Scales BF16 [K/128][N_pad].
 *   FP8E4M3: per expert [K/128][N_pad/16] blocks of 2 KiB: 32 lanes x 16 words; byte b of
 *          word 2s + j of lane l = 4g + t is the code of row g + 8 (b >> 1) at
 *          k = 16s + 4t + 2j + (b & 1) (the INT4 (row, k) assignment, one byte per weight:
 *          each 16-bit half is one BF16 pair of the MMA fragment once decoded).
 *          Scales BF16 [K/128][N_pad].
 *   INT1:  per expert [K/128][N_pad/16] blocks of 256 B: 32 lanes x 2 words holding the
 *          lane's 64 sign bits (the INT4 (row, k) assignment): register r of MMA step s
 *          (rows g + 8 (r & 1), k = 16s + 4t + 2 (r >> 1) + h) at bit 4 (s % 4) + r + 16h
 *          of word s / 4.  Padding rows hold bit 0.  Scales BF16 [K/128][N_pad].
 *   FP4E2M1: per expert [K/128][N_pad/16] blocks of 1 KiB: 32 lanes x 8 words, word s for
 *          MMA step s; byte r of it holds register r - the E2M1 codes of row g + 8 (r & 1)
 *          at k = 16s + 4t + 2 (r >> 1) (low nibble) and k + 1 (high nibble).  Scales BF16
 *          [K/128][N_pad].
 *   UINT4ZP: codes in the INT4 block layout with the nibble q itself (an excess code
 *          whose excess is the group's zero point); scales: BF16 [K/128][N_pad] as INT4,
 *          then (at s_expert_stride / 2) the BF16 numbers 128 + z in the same layout.
 *   NVFP4: codes as MXFP4 with K_pad a multiple of 256; scales E4M3 in 2048-byte chunks per
 *          128 rows x 16 groups (256 k), chunk (r/128, g/16) at
 *          ((r/128) * (K_pad/256) + g/16) * 2048, byte ((g%16)/4) * 512 + (r%32)*16 +
 *          ((r%128)/32)*4 + g%4 (four 512-byte images, one per 64-k MMA); padding bytes
 *          are 0x38 (scale 1).  A scale with its sign bit set or the NaN code is a
 *          value error (packed as 0x38).
 * The zero-exponent codes: the announcement's section "量子化サポート" states that a
 * symmetric INT without its minimum has the value set of a float with zero exponent
 * bits; the excess code used here is that value set shifted so that its bit pattern
 * drops straight into a BF16 mantissa (one logic op and one subtract per two weights).
 * Device-detected errors: INT4 -8, INT3 -4, INT2 -2, a zero point above 15, E4M3 NaN
 * (0x7F, 0xFF), E8M0 0xFF, an NVFP4 scale with its sign bit set or NaN -> QW_ERR_VALUE in
 * *d_err (an offending code is packed as 0, an offending E8M0 or NVFP4 scale as scale 1).  Alignment: w_canon / s_canon 4-byte aligned
 * (INT) or 1 (MXFP4); w_packed / s_packed 256-byte aligned.
 */
qw_status qw_repack(const qw_packed_desc* desc, const void* w_canon, const void* s_canon,
                    void* w_packed, void* s_packed, int32_t* d_err, void* stream);

/* qw_unpack - exact inverse of qw_repack (for round-trip checks): writes canonical
 * w_canon / s_canon from the packed buffers.  Padding is dropped. */
qw_status qw_unpack(const qw_packed_desc* desc, const void* w_packed, const void* s_packed,
                    void* w_canon, void* s_canon, int32_t* d_err, void* stream);

/* qw_repack_scale2 - write the second-level scales t_canon (device FP32 [E][N], 4-byte
 * aligned) into the packed scale buffer of a descriptor whose wfmt carries QW_W_SCALE2
 * (QW_ERR_INVALID_ARG otherwise).  A non-finite t is a value error in *d_err (packed as 0).
 * qw_unpack_scale2 - the inverse: t_canon from s_packed. */
qw_status qw_repack_scale2(const qw_packed_desc* desc, const float* t_canon, void* s_packed,
                           int32_t* d_err, void* stream);
qw_status qw_unpack_scale2(const qw_packed_desc* desc, const void* s_packed, float* t_canon,
                           void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_workspace_size - bytes of device workspace qgemm_dense / qgemm_moe_grouped need
 * for up to `max_rows` activation rows (host output `bytes`; 0 is a valid answer).
 * The workspace holds the grouped calls' device tile queue, which every call writes in
 * full before reading it (no initialisation needed); dense calls need none (0 bytes; the
 * single-token GEMV's split of K across the CTAs of a cluster keeps its partial sums in
 * shared memory).  Calls that share one workspace must not overlap on the GPU.
 */
qw_status qgemm_workspace_size(const qw_packed_desc* desc, int32_t afmt, int64_t max_rows,
                               uint64_t* bytes);

/* --------------------------------------------------------------------------------------
 * qgemm_dense - C[M][N] = bf16( sum_k a[m,k] * w[n,k] + bias[n] ) with the weight
 * dequantization (and, for W4A8, both block scales) applied inside the kernel.
 *   W4A16: desc->wfmt INT4/INT3/INT2/INT1/UINT4ZP/FP8E4M3/FP4E2M1, afmt QW_A_BF16,
 *          A BF16 [M][K],
 *          A_sf NULL.
 *   W4A8:  desc->wfmt MXFP4,     afmt QW_A_MXFP8_G32, A E4M3 [M][K], A_sf E8M0 [M][K/32].
 *   W8A8:  desc->wfmt MXFP8,     afmt QW_A_MXFP8_G32, as W4A8.
 *   W4A4:  desc->wfmt NVFP4,     afmt QW_A_NVFP4_G16, A E2M1 [M][K/2], A_sf E4M3 [M][K/16]
 *          (NVFP4 x NVFP4 on tcgen05 kind::mxf4nvf4; the weights' per-tensor FP32 factor
 *          of the format rides on QW_W_SCALE2, the activations' is the caller's to apply
 *          to C).
 *   bias:  BF16 [N] or NULL.  C: BF16 [M][N].  desc->E must be 1.  With QW_W_SCALE2 in
 *          desc->wfmt each channel's sum is multiplied by its second-level scale first.
 * Dispatch by M (the device heuristic of the announcement, section "デバイスパラメータに
 * 基づくパフォーマンスチューニング"): W4A16 with M <= 16 streams the weights through a
 * split-K tensor-core GEMV, larger M dequantizes into tensor memory and runs tcgen05 BF16
 * MMAs (grouped calls switch at 16 rows per expert on average); W4A8 runs the TMA +
 * tcgen05 block-scaled GEMM.  With M = 1, at most half as many 16-row blocks of N as SMs
 * and K of 16384 or more, the GEMV splits K across the CTAs of thread-block clusters of up
 * to 8 (rank 0 adds the slices in a fixed order: results do not depend on timing).
 * Alignment: A, C 16-byte aligned with K % 8 == 0 (BF16) or K % 16 == 0 (E4M3);
 * A_sf 4-byte aligned.  M >= 0 (M == 0 is a no-op).
 * Ordering: the small-M kernels (W4A16 M <= 16, W4A8 M <= 8) start as programmatic
 * dependents of the kernel before them on the stream and read w_packed and s_packed
 * before waiting for it, so that their weight stream overlaps that kernel's tail.  The
 * packed weights and scales must therefore not be written by the kernel enqueued directly
 * before the call on the same stream.  qw_repack ends with an ordering point, so calling
 * qgemm_dense right after it is safe; after a kernel of your own that writes the packed
 * buffers, put a stream-ordered operation between (an event record/wait, a memcpy, or any
 * other library call).  A, bias, C and the workspace are only touched after the wait.
 */
qw_status qgemm_dense(const qw_packed_desc* desc, const void* w_packed, const void* s_packed,
                      int32_t afmt, const void* A, const void* A_sf, const void* bias,
                      void* C, int64_t M, void* workspace, uint64_t ws_bytes,
                      int32_t* d_err, void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_moe_route - top-k routing and expert sort for the Grouped MoE layout.
 *   logits float32 [T][E] (device).  Outputs (device, int32):
 *     topk_ids      [T][topk]: the topk experts with the largest logit in descending
 *                   order, equal logits to the lower expert index;
 *     expert_offsets[E+1]: exclusive prefix sum of the per-expert pair counts;
 *     sorted_pairs  [T*topk]: pair ids p = t*topk + j ordered by (expert, p).
 *   Requires 1 <= topk <= 32, topk <= E <= 1024, T >= 0.  Workspace from
 *   qgemm_moe_route_workspace_size.  Bit-exact and deterministic.
 */
qw_status qgemm_moe_route_workspace_size(int32_t T, int32_t E, int32_t topk, uint64_t* bytes);
qw_status qgemm_moe_route(const float* logits, int32_t T, int32_t E, int32_t topk,
                          int32_t* topk_ids, int32_t* sorted_pairs, int32_t* expert_offsets,
                          void* workspace, uint64_t ws_bytes, int32_t* d_err, void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_moe_route_noalloc - qgemm_moe_route without a caller-provided workspace, for
 * callers that cannot allocate device memory (for example a plugin whose host framework
 * owns all device memory through its own pool, or a decode loop in which an allocation,
 * which may synchronise the device, is not allowed).  The pages have no counterpart:
 * this is an interface convenience of this library, not part of the method.
 *   Arguments and results are those of qgemm_moe_route.  The routing scratch lives in a
 *   static device array of QW_NOALLOC_ROUTE_SCRATCH_BYTES (1 MiB) that every GPU loading
 *   the library holds until the process exits; requests needing more scratch than that
 *   (ceil(T * topk / 256) * E * 4 bytes) are rejected with QW_ERR_WORKSPACE.  Nothing is
 *   allocated.  All calls share the array: calls that overlap on the GPU race and give
 *   undefined results.  `stream` must belong to the current device (a stream of another
 *   device is rejected with QW_ERR_INVALID_ARG before anything is enqueued).  The first
 *   call on each device looks up the array's device address (with that device current);
 *   make it before any stream capture.
 */
#define QW_NOALLOC_ROUTE_SCRATCH_BYTES (1u << 20)
qw_status qgemm_moe_route_noalloc(const float* logits, int32_t T, int32_t E, int32_t topk,
                                  int32_t* topk_ids, int32_t* sorted_pairs,
                                  int32_t* expert_offsets, int32_t* d_err, void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_moe_permute - gather activation rows into the expert-contiguous order:
 *   A_sorted[r] = A[sorted_pairs[r] / topk] for r < P (and the same for A_sf rows when
 *   afmt is QW_A_MXFP8_G32 or QW_A_NVFP4_G16; A_sf / A_sf_sorted are NULL for BF16).
 *   A: [T][K] in afmt; A_sorted: [P][K].  Rows are 16-byte multiples (2K, K or K/2 bytes).
 */
qw_status qgemm_moe_permute(int32_t afmt, const void* A, const void* A_sf, int32_t K,
                            const int32_t* sorted_pairs, int64_t P, int32_t topk,
                            void* A_sorted, void* A_sf_sorted, void* stream);

/* --------------------------------------------------------------------------------------
 * Activation-side steps around the GEMMs of a MoE layer (the pages time gate-up + down as
 * one unit, spke.com announcement "パフォーマンス"; MXFP8 activations: "W8A8 / W4A8 / W4A4").
 *
 * qw_quantize_mxfp8 - BF16 activations -> the W4A8 GEMM's MXFP8 input.  Per group of 32
 *   consecutive values of a row (OCP Microscaling v1.0 conversion): X = floor(log2(max|v|))
 *   - 8 clamped to [-127, 127], A_sf = X + 127 (E8M0); A_q = E4M3(v / 2^X) rounded to
 *   nearest even and saturated to +-448; an all-zero group gets A_sf = 0.
 *   A: BF16 [rows][K]; A_q: uint8 [rows][K]; A_sf: uint8 [rows][K/32] (device).
 *   K % 32 == 0; A 16-byte aligned, A_q 8-byte aligned.  A non-finite input sets
 *   QW_ERR_VALUE in d_err (its group's outputs are then unspecified).
 */
qw_status qw_quantize_mxfp8(const void* A, int64_t rows, int32_t K, void* A_q, void* A_sf,
                            int32_t* d_err, void* stream);

/* qw_silu_mul - Y[r][i] = bf16( silu(GU[r][i]) * GU[r][I + i] ), silu(g) = g / (1 + e^-g):
 *   the fused gate+up projection output (gate in the first half of each row) -> the down
 *   projection's input.  GU: BF16 [rows][2I]; Y: BF16 [rows][I] (device).  FP32 arithmetic,
 *   BF16 round-to-nearest-even.  I % 8 == 0; GU and Y 16-byte aligned.
 */
qw_status qw_silu_mul(const void* GU, int64_t rows, int32_t I, void* Y, void* stream);

/* qgemm_moe_combine - out[t][n] = bf16( sum_j w[t][j] * Y[row of pair t*topk + j][n] ):
 *   the down projection's rows (in the sorted-pair order of qgemm_moe_route, row r holding
 *   pair sorted_pairs[r]) weighted and summed back per token, w[t][.] = softmax of token
 *   t's topk selected logits (logits[t][topk_ids[t][j]]), FP32.
 *   Y: BF16 [T*topk][N]; sorted_pairs int32 [T*topk]; topk_ids int32 [T][topk]; logits
 *   float32 [T][E]; out: BF16 [T][N] (all device).  N % 8 == 0; Y, out 16-byte aligned;
 *   1 <= topk <= 32.  workspace: >= qgemm_moe_combine_workspace_size(T, topk) device
 *   bytes (scratch, any content).  Out-of-range ids or pairs set QW_ERR_INVALID_ARG in d_err.
 */
qw_status qgemm_moe_combine_workspace_size(int32_t T, int32_t topk, uint64_t* bytes);
qw_status qgemm_moe_combine(const void* Y, const int32_t* sorted_pairs, const int32_t* topk_ids,
                            const float* logits, int32_t T, int32_t E, int32_t topk, int32_t N,
                            void* out, void* workspace, uint64_t ws_bytes, int32_t* d_err,
                            void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_moe_grouped - Grouped MoE GEMM: for every expert e and every row r in
 * [expert_offsets[e], expert_offsets[e+1]):
 *   C[r][n] = bf16( sum_k A_sorted[r][k] * W_e[n][k] + bias[e][n] ).
 *   expert_offsets: device int32 [E+1], non-decreasing, offsets[0] == 0 and
 *   offsets[E] == total_rows (read on the device; no host round trip).
 *   A_sorted / A_sf_sorted as for qgemm_dense with total_rows rows; bias BF16 [E][N] or
 *   NULL; C BF16 [total_rows][N].  The per-expert tile queue is built on the device in
 *   the workspace (qgemm_workspace_size with max_rows = total_rows).  Dimensions need
 *   not be multiples of 256 (e.g. an intermediate size of 640).
 */
qw_status qgemm_moe_grouped(const qw_packed_desc* desc, const void* w_packed,
                            const void* s_packed, int32_t afmt, const void* A_sorted,
                            const void* A_sf_sorted, const int32_t* expert_offsets,
                            int64_t total_rows, const void* bias, void* C, void* workspace,
                            uint64_t ws_bytes, int32_t* d_err, void* stream);

/* --------------------------------------------------------------------------------------
 * qgemm_moe_grouped_indexed - the Indexed MoE path (spke.com announcement, "WnA16" /
 * "W8A8 / W4A8 / W4A4": Indexed and Grouped MoE layouts): qgemm_moe_grouped with the
 * permutation folded into the kernel.  Problem row r (in the expert-contiguous order of
 * qgemm_moe_route) reads activation row sorted_pairs[r] / topk of the UNPERMUTED input:
 *   C[r][n] = bf16( sum_k A[sorted_pairs[r] / topk][k] * W_e[n][k] + bias[e][n] )
 * for r in [expert_offsets[e], expert_offsets[e+1]); the result equals
 * qgemm_moe_permute followed by qgemm_moe_grouped, bit for bit.
 *   MX weight formats only (W4A8 / W8A8; other formats return QW_ERR_UNSUPPORTED).
 *   A: E4M3 [T][K]; A_sf: E8M0 [T][K/32]; sorted_pairs: device int32 [total_rows] with
 *   total_rows <= T * topk; the rest as for qgemm_moe_grouped (same workspace size).
 *   A pair outside [0, T*topk) sets QW_ERR_INVALID_ARG in d_err (its row reads token 0).
 */
qw_status qgemm_moe_grouped_indexed(const qw_packed_desc* desc, const void* w_packed,
                                    const void* s_packed, int32_t afmt, const void* A,
                                    const void* A_sf, int64_t T, const int32_t* sorted_pairs,
                                    int32_t topk, const int32_t* expert_offsets,
                                    int64_t total_rows, const void* bias, void* C,
                                    void* workspace, uint64_t ws_bytes, int32_t* d_err,
                                    void* stream);

/* --------------------------------------------------------------------------------------
 * qw_read_error - synchronise `stream`, copy *d_err to the host (`host_code`, host
 * pointer) and return it as a qw_status (QW_ERR_CUDA if the synchronisation fails).
 */
qw_status qw_read_error(const int32_t* d_err, void* stream, int32_t* host_code);

/* --------------------------------------------------------------------------------------
 * qw_test_wait_timeout - diagnostics for the bounded waits every kernel relies on: one
 * CTA waits on an mbarrier that nothing ever arrives on, through the same bounded-wait
 * routine the GEMM pipelines use, and must give up after `limit_ns` (0 .. 2e9) with
 * QW_ERR_TIMEOUT in *d_err.  It exercises failure handling without hanging or
 * faulting the GPU.  (Failure handling of this kind is the pages' own advice: keep a
 * fallback because shape routing and backend checks fail - aireiter.com, "Backend
 * routing can block a valid Humming configuration".)
 */
qw_status qw_test_wait_timeout(int32_t* d_err, int64_t limit_ns, void* stream);

/* --------------------------------------------------------------------------------------
 * qw_stream_read - diagnostics: the reference point of the HBM-bound kernels.  Reads
 * `bytes` of device memory at `src` once with 16-byte loads from a full grid (eight CTAs
 * of 256 threads per SM) and writes one fold word per CTA to `sink` (device uint32,
 * QW_STREAM_READ_SINK_WORDS of them).  `chained` = 1 launches it as a programmatic
 * dependent of the previous kernel with every load before its griddepcontrol.wait (only
 * the sink write waits), the overlap a kernel that needs nothing from its predecessor can
 * have; 0 launches it in plain stream order.  The pages measure decode kernels as a
 * fraction of memory bandwidth (aireiter.com, "SM80 single-request decode: do not infer
 * Ampere gains"); this is the read such a fraction is compared with on this GPU.
 * Requires src 16-byte aligned and bytes % 16 == 0 (QW_ERR_ALIGNMENT otherwise).
 */
#define QW_STREAM_READ_SINK_WORDS 4096
qw_status qw_stream_read(const void* src, uint64_t bytes, uint32_t* sink, int32_t chained,
                         void* stream);

/* --------------------------------------------------------------------------------------
 * qw_mma_rate_probe - diagnostics: the tcgen05 MMA issue rate the tensor-core GEMMs are
 * bounded by (the pages tune per instruction shape and kind: spke.com Humming announcement,
 * "フォーマットとアーキテクチャを横断して共有されるCUDAコンポーネント"; "W8A8 / W4A8 / W4A4").
 * One CTA per SM (at most QW_MMA_PROBE_MAX_CTAS, 120 KiB of shared memory each, 512 TMEM
 * columns), one thread issuing `iters` back-to-back M = 128 MMAs into one accumulator on
 * zero operands, after a 64-MMA warm-up; then a commit and a bounded wait.  Modes:
 *   QW_MMA_PROBE_F16_TMEM_A   kind::f16, A (BF16) in TMEM, B (BF16, 128-byte swizzle) in
 *                             shared memory, N = n: the W4A16 GEMM's form (accumulation
 *                             restarts every 8 MMAs, one 128-k group);
 *   QW_MMA_PROBE_F16_SMEM     the same with A in shared memory;
 *   QW_MMA_PROBE_MXF8F6F4     kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3 x E2M1 (one
 *                             byte per code), N = 256: the W4A8 GEMM's MMA;
 *   QW_MMA_PROBE_MXF8F6F4_CP  the same plus its three tcgen05.cp.32x128b.warpx4 scale
 *                             copies per four MMAs (one 128-k stage), into scale columns
 *                             that rotate over four stages as in the GEMM's ring;
 *   QW_MMA_PROBE_MXF8F6F4_CP_AHEAD  the same copies issued one stage ahead (into the next
 *                             stage's columns, so no MMA reads what was just copied);
 *   QW_MMA_PROBE_MXF8F6F4_CP_WIDE   two copies per stage instead of three: A's image as one
 *                             tcgen05.cp.128x128b, B's two as one 128x256b (sources with
 *                             each 32-row image repeated for the four lane quarters);
 *   QW_MMA_PROBE_MXF4NVF4     kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 x E2M1 packed,
 *                             UE4M3 scales, 128 x 256 x 64: the W4A4 GEMM's MMA;
 *   QW_MMA_PROBE_MXF4NVF4_CP  the same plus its twelve tcgen05.cp.32x128b.warpx4 scale
 *                             copies per four MMAs (one 256-k stage).
 * QW_MMA_PROBE_RANDOM or'ed into a mode fills the operands with hashed finite values
 * instead of zeros (the tensor core's rate may depend on the data it multiplies).
 * n: 64, 128 or 256 for the f16 modes, 256 for the block-scaled ones; iters in [64, 2^20].
 * Writes, per CTA c, out[2c] = SM clock cycles and out[2c + 1] = nanoseconds from the first
 * issue to the completion (device uint64, 2 x QW_MMA_PROBE_MAX_CTAS of them); a wait that
 * gave up writes zeros and raises QW_ERR_TIMEOUT in *d_err.  Invalid mode / n / iters:
 * QW_ERR_INVALID_ARG; out not 8-byte aligned: QW_ERR_ALIGNMENT.
 */
#define QW_MMA_PROBE_F16_TMEM_A 0
#define QW_MMA_PROBE_F16_SMEM 1
#define QW_MMA_PROBE_MXF8F6F4 2
#define QW_MMA_PROBE_MXF8F6F4_CP 3
#define QW_MMA_PROBE_MXF8F6F4_CP_AHEAD 4
#define QW_MMA_PROBE_MXF8F6F4_CP_WIDE 5
#define QW_MMA_PROBE_MXF4NVF4 6
#define QW_MMA_PROBE_MXF4NVF4_CP 7
#define QW_MMA_PROBE_RANDOM 8
#define QW_MMA_PROBE_MAX_CTAS 1024
qw_status qw_mma_rate_probe(int32_t mode, int32_t n, int32_t iters, uint64_t* out,
                            int32_t* d_err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QW_H */
