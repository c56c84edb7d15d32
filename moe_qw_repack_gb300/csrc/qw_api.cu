// qw_api.cu - the extern "C" entry points declared in include/qw.h: host-side
// validation of every argument (the library returns a status and never asserts; the
// pages' vLLM issue #60700 is the cautionary tale of a shape check that asserted) and
// dispatch to the kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/qw.h"
#include "qw_internal.h"

namespace qw {

// SM count of the current device, cached per device (152 on GB300, also the value taken if
// the query fails); it only sizes the grids of kernels that stride over their work.
int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
  if (dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// block-scaled MX weight formats (E8M0 scale per 32 along K, tcgen05 block-scaled MMA)
// block-scaled formats: the tcgen05 kind::mxf8f6f4 / kind::mxf4nvf4 GEMM
bool is_mx(int32_t wfmt) {
  return wfmt == QW_W_MXFP4_G32 || wfmt == QW_W_MXFP8_G32 || wfmt == QW_W_NVFP4_G16;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Bytes of the second-level scale plane (FP32 [E][N_pad]) at the end of s_packed.
uint64_t scale2_bytes(const qw_packed_desc& d) {
  return (d.wfmt & QW_W_SCALE2) ? (uint64_t)round_up((int64_t)d.E * d.N_pad * 4, 256) : 0;
}
// The descriptor of the base format (no second-level scales) the kernels are launched with.
qw_packed_desc base_desc(const qw_packed_desc& d) {
  qw_packed_desc b = d;
  b.s_bytes -= scale2_bytes(d);
  b.wfmt &= ~QW_W_SCALE2;
  return b;
}
// Device FP32 [E][N_pad] second-level scales of a packed scale buffer, or null.
const float* scale2_of(const qw_packed_desc& d, const void* s_packed) {
  if (!(d.wfmt & QW_W_SCALE2) || !s_packed) return nullptr;
  return reinterpret_cast<const float*>(static_cast<const uint8_t*>(s_packed) +
                                        d.s_expert_stride * (uint64_t)d.E);
}

qw_status check_desc(const qw_packed_desc* d) {
  if (!d) return QW_ERR_INVALID_ARG;
  qw_packed_desc ref;
  if (qw_repack_query(d->wfmt, d->E, d->N, d->K, &ref) != QW_OK) return QW_ERR_INVALID_ARG;
  if (ref.N_pad != d->N_pad || ref.K_pad != d->K_pad || ref.w_bytes != d->w_bytes ||
      ref.s_bytes != d->s_bytes || ref.group != d->group)
    return QW_ERR_INVALID_ARG;
  return QW_OK;
}

qw_status check_afmt(const qw_packed_desc* d, int32_t afmt, const void* A_sf) {
  const int32_t wfmt = d->wfmt & ~QW_W_SCALE2;
  if (is_mx(wfmt)) {
    if (afmt != (wfmt == QW_W_NVFP4_G16 ? QW_A_NVFP4_G16 : QW_A_MXFP8_G32))
      return QW_ERR_UNSUPPORTED;
    if (!A_sf) return QW_ERR_INVALID_ARG;
  } else {
    if (afmt != QW_A_BF16) return QW_ERR_UNSUPPORTED;
  }
  return QW_OK;
}

}  // namespace
}  // namespace qw

using namespace qw;

extern "C" {

const char* qw_status_str(int32_t s) {
  switch (s) {
    case QW_OK: return "ok";
    case QW_ERR_INVALID_ARG: return "invalid argument";
    case QW_ERR_UNSUPPORTED: return "unsupported format or shape";
    case QW_ERR_ALIGNMENT: return "misaligned pointer or pitch";
    case QW_ERR_VALUE: return "code outside its format's valid set";
    case QW_ERR_WORKSPACE: return "workspace missing or too small";
    case QW_ERR_TIMEOUT: return "bounded device wait gave up";
    case QW_ERR_CUDA: return "CUDA call failed";
    default: return "unknown status";
  }
}

int32_t qw_version(void) { return 210; }

qw_status qw_repack_query(int32_t wfmt_in, int32_t E, int32_t N, int32_t K, qw_packed_desc* out) {
  if (!out || E < 1 || N < 1 || K < 1) return QW_ERR_INVALID_ARG;
  if (wfmt_in & ~(QW_W_SCALE2 | 0xFF)) return QW_ERR_UNSUPPORTED;
  // every padded size (N to 128, K to 256 at most) must still fit in int32
  constexpr int32_t kMaxDim = 0x7FFFFF00;
  if (N > kMaxDim || K > kMaxDim) return QW_ERR_UNSUPPORTED;
  const int32_t wfmt = wfmt_in & ~QW_W_SCALE2;
  qw_packed_desc d{};
  d.wfmt = wfmt_in;
  d.E = E;
  d.N = N;
  d.K = K;
  switch (wfmt) {
    case QW_W_INT4_G128_BF16:
    case QW_W_INT3_G128_BF16:
    case QW_W_INT2_G128_BF16:
    case QW_W_FP8E4M3_G128_BF16:
    case QW_W_INT1_G128_BF16:
    case QW_W_FP4E2M1_G128_BF16:
    case QW_W_UINT4ZP_G128_BF16: {
      if (K % kIntGroup) return QW_ERR_UNSUPPORTED;
      d.group = kIntGroup;
      d.N_pad = (int32_t)round_up(N, 16);
      d.K_pad = K;
      const int64_t blocks = (int64_t)(K / kIntGroup) * (d.N_pad / 16);
      d.w_expert_stride =
          (uint64_t)blocks * (wfmt == QW_W_INT3_G128_BF16   ? kInt3BlockBytes
                              : wfmt == QW_W_INT2_G128_BF16   ? kInt2BlockBytes
                              : wfmt == QW_W_FP8E4M3_G128_BF16 ? kFp8BlockBytes
                              : wfmt == QW_W_INT1_G128_BF16    ? kInt1BlockBytes
                              : wfmt == QW_W_FP4E2M1_G128_BF16 ? kFp4BlockBytes
                                                               : kInt4BlockBytes);
      // one BF16 plane of scales (UINT4ZP: a second plane of 128 + zero point)
      d.s_expert_stride = (uint64_t)round_up((int64_t)(K / kIntGroup) * d.N_pad * 2, 256) *
                          (wfmt == QW_W_UINT4ZP_G128_BF16 ? 2 : 1);
      break;
    }
    case QW_W_MXFP4_G32:
    case QW_W_MXFP8_G32: {
      if (K % kMxGroup) return QW_ERR_UNSUPPORTED;
      d.group = kMxGroup;
      d.N_pad = (int32_t)round_up(N, 128);
      d.K_pad = (int32_t)round_up(K, 128);
      d.w_expert_stride =
          (uint64_t)d.N_pad * (wfmt == QW_W_MXFP4_G32 ? d.K_pad / 2 : d.K_pad);
      d.s_expert_stride = (uint64_t)(d.N_pad / 128) * (d.K_pad / 128) * kSfChunkBytes;
      break;
    }
    case QW_W_NVFP4_G16: {
      if (K % 32) return QW_ERR_UNSUPPORTED;  // packed rows of 16-byte multiples
      d.group = kNvGroup;
      d.N_pad = (int32_t)round_up(N, 128);
      d.K_pad = (int32_t)round_up(K, 256);
      d.w_expert_stride = (uint64_t)d.N_pad * (d.K_pad / 2);
      d.s_expert_stride = (uint64_t)(d.N_pad / 128) * (d.K_pad / 256) * kNvChunkBytes;
      break;
    }
    default:
      return QW_ERR_UNSUPPORTED;
  }
  if ((int64_t)d.N_pad * E > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  d.w_bytes = d.w_expert_stride * (uint64_t)E;
  d.s_bytes = d.s_expert_stride * (uint64_t)E + scale2_bytes(d);
  *out = d;
  return QW_OK;
}

qw_status qw_repack(const qw_packed_desc* desc, const void* w_canon, const void* s_canon,
                    void* w_packed, void* s_packed, int32_t* d_err, void* stream) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if (!w_canon || !s_canon || !w_packed || !s_packed) return QW_ERR_INVALID_ARG;
  const qw_packed_desc bd = base_desc(*desc);
  if (!is_mx(bd.wfmt) && (!aligned(w_canon, 4) || !aligned(s_canon, 2)))
    return QW_ERR_ALIGNMENT;
  if (bd.wfmt == QW_W_UINT4ZP_G128_BF16 && !aligned(s_canon, 4)) return QW_ERR_ALIGNMENT;
  if (!aligned(w_packed, 256) || !aligned(s_packed, 256)) return QW_ERR_ALIGNMENT;
  s = launch_repack(bd, w_canon, s_canon, w_packed, s_packed, d_err,
                    static_cast<cudaStream_t>(stream));
  if (s != QW_OK || !(desc->wfmt & QW_W_SCALE2)) return s;
  return launch_scale2_fill(const_cast<float*>(scale2_of(*desc, s_packed)),
                            (int64_t)desc->E * desc->N_pad, static_cast<cudaStream_t>(stream));
}

qw_status qw_unpack(const qw_packed_desc* desc, const void* w_packed, const void* s_packed,
                    void* w_canon, void* s_canon, int32_t* d_err, void* stream) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if (!w_canon || !s_canon || !w_packed || !s_packed) return QW_ERR_INVALID_ARG;
  const qw_packed_desc bd = base_desc(*desc);
  if (!is_mx(bd.wfmt) && (!aligned(w_canon, 4) || !aligned(s_canon, 2)))
    return QW_ERR_ALIGNMENT;
  if (bd.wfmt == QW_W_UINT4ZP_G128_BF16 && !aligned(s_canon, 4)) return QW_ERR_ALIGNMENT;
  if (!aligned(w_packed, 256) || !aligned(s_packed, 256)) return QW_ERR_ALIGNMENT;
  return launch_unpack(bd, w_packed, s_packed, w_canon, s_canon, d_err,
                       static_cast<cudaStream_t>(stream));
}

qw_status qw_repack_scale2(const qw_packed_desc* desc, const float* t_canon, void* s_packed,
                           int32_t* d_err, void* stream) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if (!(desc->wfmt & QW_W_SCALE2) || !t_canon || !s_packed) return QW_ERR_INVALID_ARG;
  if (!aligned(t_canon, 4) || !aligned(s_packed, 256)) return QW_ERR_ALIGNMENT;
  return launch_scale2_repack(t_canon, const_cast<float*>(scale2_of(*desc, s_packed)), desc->E,
                              desc->N, desc->N_pad, d_err, static_cast<cudaStream_t>(stream));
}

qw_status qw_unpack_scale2(const qw_packed_desc* desc, const void* s_packed, float* t_canon,
                           void* stream) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if (!(desc->wfmt & QW_W_SCALE2) || !t_canon || !s_packed) return QW_ERR_INVALID_ARG;
  if (!aligned(t_canon, 4) || !aligned(s_packed, 256)) return QW_ERR_ALIGNMENT;
  return launch_scale2_unpack(scale2_of(*desc, s_packed), t_canon, desc->E, desc->N, desc->N_pad,
                              static_cast<cudaStream_t>(stream));
}

qw_status qgemm_workspace_size(const qw_packed_desc* desc, int32_t afmt, int64_t max_rows,
                               uint64_t* bytes) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if (!bytes || max_rows < 0) return QW_ERR_INVALID_ARG;
  if ((s = check_afmt(desc, afmt, reinterpret_cast<const void*>(1))) != QW_OK) return s;
  const qw_packed_desc bd = base_desc(*desc);
  if (is_mx(bd.wfmt)) {
    *bytes = gemm_w4a8_workspace(bd, max_rows);
  } else {
    const uint64_t a = gemv_w4a16_workspace(bd, max_rows);
    const uint64_t b = gemm_w4a16_tc_workspace(bd, max_rows);
    *bytes = a > b ? a : b;
  }
  return QW_OK;
}

static qw_status check_gemm_args(const qw_packed_desc* desc, const void* w_packed,
                                 const void* s_packed, int32_t afmt, const void* A,
                                 const void* A_sf, void* C, int64_t rows) {
  qw_status s = check_desc(desc);
  if (s != QW_OK) return s;
  if ((s = check_afmt(desc, afmt, A_sf)) != QW_OK) return s;
  if (rows < 0) return QW_ERR_INVALID_ARG;
  if (rows > 0 && (!w_packed || !s_packed || !A || !C)) return QW_ERR_INVALID_ARG;
  if (!aligned(w_packed, 256) || !aligned(s_packed, 256)) return QW_ERR_ALIGNMENT;
  if (!aligned(A, 16) || !aligned(C, 4)) return QW_ERR_ALIGNMENT;
  const int32_t wfmt = desc->wfmt & ~QW_W_SCALE2;
  if (is_mx(wfmt)) {
    // TMA row pitch of the activations: K bytes (E4M3) or K/2 bytes (E2M1), 16-byte multiple
    if (desc->K % (wfmt == QW_W_NVFP4_G16 ? 32 : 16)) return QW_ERR_ALIGNMENT;
    if (!aligned(A_sf, 4)) return QW_ERR_ALIGNMENT;
  } else if (desc->K % 8) {
    return QW_ERR_ALIGNMENT;
  }
  return QW_OK;
}

qw_status qgemm_dense(const qw_packed_desc* desc, const void* w_packed, const void* s_packed,
                      int32_t afmt, const void* A, const void* A_sf, const void* bias, void* C,
                      int64_t M, void* workspace, uint64_t ws_bytes, int32_t* d_err,
                      void* stream) {
  qw_status s = check_gemm_args(desc, w_packed, s_packed, afmt, A, A_sf, C, M);
  if (s != QW_OK) return s;
  if (desc->E != 1) return QW_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 2)) return QW_ERR_ALIGNMENT;
  if (M == 0) return QW_OK;
  RowSet rs{M, nullptr, 1};
  rs.scale2 = scale2_of(*desc, s_packed);
  const qw_packed_desc bd = base_desc(*desc);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bd.wfmt == QW_W_MXFP4_G32 && M <= kW4A8GemvRows &&
      w4a8_gemv_smem_bytes(bd.K, (int)M) <= kW4A8GemvMaxSmem)
    return launch_gemv_w4a8(bd, w_packed, s_packed, A, A_sf, bias, rs.scale2, C, (int)M, d_err,
                            st);
  if (is_mx(bd.wfmt))
    return launch_gemm_w4a8(bd, w_packed, s_packed, A, A_sf, bias, C, rs, workspace, ws_bytes,
                            d_err, st);
  if (M > kW4A16TensorCoreRows)
    return launch_gemm_w4a16_tc(bd, w_packed, s_packed, A, bias, C, rs, workspace, ws_bytes,
                                d_err, st);
  return launch_gemv_w4a16(bd, w_packed, s_packed, A, bias, C, rs, workspace, ws_bytes, d_err,
                           st);
}

qw_status qgemm_moe_route_workspace_size(int32_t T, int32_t E, int32_t topk, uint64_t* bytes) {
  if (!bytes || T < 0 || topk < 1 || topk > 32 || E < topk || E > 1024) return QW_ERR_INVALID_ARG;
  *bytes = moe_route_workspace(T, E, topk);
  return QW_OK;
}

qw_status qgemm_moe_route(const float* logits, int32_t T, int32_t E, int32_t topk,
                          int32_t* topk_ids, int32_t* sorted_pairs, int32_t* expert_offsets,
                          void* workspace, uint64_t ws_bytes, int32_t* d_err, void* stream) {
  if (T < 0 || topk < 1 || topk > 32 || E < topk || E > 1024) return QW_ERR_INVALID_ARG;
  if (!expert_offsets) return QW_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_ids || !sorted_pairs)) return QW_ERR_INVALID_ARG;
  if ((int64_t)T * topk > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(sorted_pairs, 4) ||
      !aligned(expert_offsets, 4))
    return QW_ERR_ALIGNMENT;
  if (!workspace || ws_bytes < moe_route_workspace(T, E, topk)) return QW_ERR_WORKSPACE;
  return launch_moe_route(logits, T, E, topk, topk_ids, sorted_pairs, expert_offsets, workspace,
                          ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

qw_status qgemm_moe_permute(int32_t afmt, const void* A, const void* A_sf, int32_t K,
                            const int32_t* sorted_pairs, int64_t P, int32_t topk, void* A_sorted,
                            void* A_sf_sorted, void* stream) {
  if (afmt != QW_A_BF16 && afmt != QW_A_MXFP8_G32 && afmt != QW_A_NVFP4_G16)
    return QW_ERR_UNSUPPORTED;
  if (K < 1 || P < 0 || topk < 1) return QW_ERR_INVALID_ARG;
  if (P == 0) return QW_OK;
  if (!A || !sorted_pairs || !A_sorted) return QW_ERR_INVALID_ARG;
  if (afmt == QW_A_NVFP4_G16 && K % 2) return QW_ERR_UNSUPPORTED;
  const int64_t row_bytes =
      afmt == QW_A_BF16 ? 2 * (int64_t)K : (afmt == QW_A_NVFP4_G16 ? K / 2 : (int64_t)K);
  if (row_bytes % 16 || !aligned(A, 16) || !aligned(A_sorted, 16) || !aligned(sorted_pairs, 4))
    return QW_ERR_ALIGNMENT;
  if (afmt != QW_A_BF16) {
    if (K % (afmt == QW_A_NVFP4_G16 ? 16 : 32)) return QW_ERR_UNSUPPORTED;
    if (!A_sf || !A_sf_sorted) return QW_ERR_INVALID_ARG;
  }
  return launch_moe_permute(afmt, A, A_sf, K, sorted_pairs, P, topk, A_sorted, A_sf_sorted,
                            static_cast<cudaStream_t>(stream));
}

qw_status qw_quantize_mxfp8(const void* A, int64_t rows, int32_t K, void* A_q, void* A_sf,
                            int32_t* d_err, void* stream) {
  if (rows < 0 || K < 32) return QW_ERR_INVALID_ARG;
  if (K % 32) return QW_ERR_UNSUPPORTED;
  if (rows == 0) return QW_OK;
  if (!A || !A_q || !A_sf) return QW_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(A_q, 8)) return QW_ERR_ALIGNMENT;
  if (rows * (int64_t)(K / 8) > ((int64_t)1 << 40)) return QW_ERR_UNSUPPORTED;
  return launch_quantize_mxfp8(A, rows, K, A_q, A_sf, d_err, static_cast<cudaStream_t>(stream));
}

qw_status qw_silu_mul(const void* GU, int64_t rows, int32_t I, void* Y, void* stream) {
  if (rows < 0 || I < 1) return QW_ERR_INVALID_ARG;
  if (I % 8) return QW_ERR_UNSUPPORTED;
  if (rows == 0) return QW_OK;
  if (!GU || !Y) return QW_ERR_INVALID_ARG;
  if (!aligned(GU, 16) || !aligned(Y, 16)) return QW_ERR_ALIGNMENT;
  return launch_silu_mul(GU, rows, I, Y, static_cast<cudaStream_t>(stream));
}

qw_status qgemm_moe_combine_workspace_size(int32_t T, int32_t topk, uint64_t* bytes) {
  if (!bytes || T < 0 || topk < 1 || topk > 32) return QW_ERR_INVALID_ARG;
  *bytes = (uint64_t)T * (uint64_t)topk * 4 + 256;
  return QW_OK;
}

qw_status qgemm_moe_combine(const void* Y, const int32_t* sorted_pairs, const int32_t* topk_ids,
                            const float* logits, int32_t T, int32_t E, int32_t topk, int32_t N,
                            void* out, void* workspace, uint64_t ws_bytes, int32_t* d_err,
                            void* stream) {
  if (T < 0 || E < 1 || topk < 1 || topk > 32 || topk > E || N < 1) return QW_ERR_INVALID_ARG;
  if (N % 8) return QW_ERR_UNSUPPORTED;
  if (T == 0) return QW_OK;
  if (!Y || !sorted_pairs || !topk_ids || !logits || !out) return QW_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(out, 16) || !aligned(sorted_pairs, 4) || !aligned(topk_ids, 4) ||
      !aligned(logits, 4))
    return QW_ERR_ALIGNMENT;
  uint64_t need = 0;
  qgemm_moe_combine_workspace_size(T, topk, &need);
  if (!workspace || ws_bytes < need || !aligned(workspace, 4)) return QW_ERR_WORKSPACE;
  return launch_moe_combine(Y, sorted_pairs, topk_ids, logits, T, E, topk, N, out,
                            static_cast<int32_t*>(workspace), d_err,
                            static_cast<cudaStream_t>(stream));
}

qw_status qgemm_moe_grouped(const qw_packed_desc* desc, const void* w_packed,
                            const void* s_packed, int32_t afmt, const void* A_sorted,
                            const void* A_sf_sorted, const int32_t* expert_offsets,
                            int64_t total_rows, const void* bias, void* C, void* workspace,
                            uint64_t ws_bytes, int32_t* d_err, void* stream) {
  qw_status s = check_gemm_args(desc, w_packed, s_packed, afmt, A_sorted, A_sf_sorted, C,
                                total_rows);
  if (s != QW_OK) return s;
  if (!expert_offsets || !aligned(expert_offsets, 4)) return QW_ERR_INVALID_ARG;
  if (desc->E > 1024) return QW_ERR_UNSUPPORTED;
  if (bias && !aligned(bias, 2)) return QW_ERR_ALIGNMENT;
  if (total_rows == 0) return QW_OK;
  uint64_t need = 0;
  qgemm_workspace_size(desc, afmt, total_rows, &need);
  if (!workspace || ws_bytes < need) return QW_ERR_WORKSPACE;
  RowSet rs{total_rows, expert_offsets, desc->E};
  rs.scale2 = scale2_of(*desc, s_packed);
  const qw_packed_desc bd = base_desc(*desc);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (is_mx(bd.wfmt))
    return launch_gemm_w4a8(bd, w_packed, s_packed, A_sorted, A_sf_sorted, bias, C, rs,
                            workspace, ws_bytes, d_err, st);
  if (total_rows >= kW4A16TensorCoreRows * bd.E)
    return launch_gemm_w4a16_tc(bd, w_packed, s_packed, A_sorted, bias, C, rs, workspace,
                                ws_bytes, d_err, st);
  return launch_gemv_w4a16(bd, w_packed, s_packed, A_sorted, bias, C, rs, workspace, ws_bytes,
                           d_err, st);
}

qw_status qgemm_moe_grouped_indexed(const qw_packed_desc* desc, const void* w_packed,
                                    const void* s_packed, int32_t afmt, const void* A,
                                    const void* A_sf, int64_t T, const int32_t* sorted_pairs,
                                    int32_t topk, const int32_t* expert_offsets,
                                    int64_t total_rows, const void* bias, void* C,
                                    void* workspace, uint64_t ws_bytes, int32_t* d_err,
                                    void* stream) {
  qw_status s = check_gemm_args(desc, w_packed, s_packed, afmt, A, A_sf, C, total_rows);
  if (s != QW_OK) return s;
  if (!is_mx(desc->wfmt & ~QW_W_SCALE2)) return QW_ERR_UNSUPPORTED;
  if (!expert_offsets || !aligned(expert_offsets, 4)) return QW_ERR_INVALID_ARG;
  if (desc->E > 1024) return QW_ERR_UNSUPPORTED;
  if (topk < 1 || T < 0 || T > 0x7FFFFFFFLL || total_rows > T * (int64_t)topk)
    return QW_ERR_INVALID_ARG;
  if (total_rows > 0 && (!sorted_pairs || !aligned(sorted_pairs, 4))) return QW_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 2)) return QW_ERR_ALIGNMENT;
  if (total_rows == 0) return QW_OK;
  uint64_t need = 0;
  qgemm_workspace_size(desc, afmt, total_rows, &need);
  if (!workspace || ws_bytes < need) return QW_ERR_WORKSPACE;
  RowSet rs{total_rows, expert_offsets, desc->E, sorted_pairs, topk, T};
  rs.scale2 = scale2_of(*desc, s_packed);
  return launch_gemm_w4a8(base_desc(*desc), w_packed, s_packed, A, A_sf, bias, C, rs, workspace,
                          ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

qw_status qw_read_error(const int32_t* d_err, void* stream, int32_t* host_code) {
  if (!d_err || !host_code) return QW_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QW_ERR_CUDA;
  if (cudaMemcpy(host_code, d_err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QW_ERR_CUDA;
  return static_cast<qw_status>(*host_code);
}

qw_status qw_test_wait_timeout(int32_t* d_err, int64_t limit_ns, void* stream) {
  if (!d_err || limit_ns < 0 || limit_ns > 2000000000LL) return QW_ERR_INVALID_ARG;
  return launch_wait_timeout_probe(d_err, limit_ns, static_cast<cudaStream_t>(stream));
}

qw_status qw_stream_read(const void* src, uint64_t bytes, uint32_t* sink, int32_t chained,
                         void* stream) {
  if (!sink || (bytes > 0 && !src)) return QW_ERR_INVALID_ARG;
  if (!aligned(src, 16) || bytes % 16 || !aligned(sink, 4)) return QW_ERR_ALIGNMENT;
  return launch_stream_read(src, bytes, sink, chained != 0, static_cast<cudaStream_t>(stream));
}

qw_status qw_mma_rate_probe(int32_t mode, int32_t n, int32_t iters, uint64_t* out,
                            int32_t* d_err, void* stream) {
  const int32_t base = mode & ~QW_MMA_PROBE_RANDOM;
  const bool f16 = base == QW_MMA_PROBE_F16_TMEM_A || base == QW_MMA_PROBE_F16_SMEM;
  const bool mx = base == QW_MMA_PROBE_MXF8F6F4 || base == QW_MMA_PROBE_MXF8F6F4_CP ||
                  base == QW_MMA_PROBE_MXF8F6F4_CP_AHEAD || base == QW_MMA_PROBE_MXF8F6F4_CP_WIDE ||
                  base == QW_MMA_PROBE_MXF4NVF4 || base == QW_MMA_PROBE_MXF4NVF4_CP;
  if (!f16 && !mx) return QW_ERR_INVALID_ARG;
  // only the shapes the GEMMs issue (a shape outside the MMA's table would not assemble to
  // a valid instruction)
  if (f16 && n != 64 && n != 128 && n != 256) return QW_ERR_INVALID_ARG;
  if (mx && n != 256) return QW_ERR_INVALID_ARG;
  if (iters < 64 || iters > (1 << 20) || !out || !d_err) return QW_ERR_INVALID_ARG;
  if (!aligned(out, 8) || !aligned(d_err, 4)) return QW_ERR_ALIGNMENT;
  return launch_mma_probe(mode, n, iters, out, d_err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
