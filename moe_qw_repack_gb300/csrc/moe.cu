// moe.cu - MoE scheduling for the Grouped layout: top-k routing, the stable sort of
// routed (token, slot) pairs by expert, the row permutation, and the device-built
// per-expert tile queue the grouped GEMMs walk.
//
// The pages describe MoE workloads where tokens spread over experts and the work per
// expert varies with load, served by Indexed and Grouped paths (spke.com Humming
// announcement, "背景" and "WnA16"), with dense and MoE GEMMs using their own task
// scheduling (section "フォーマットとアーキテクチャを横断して共有されるCUDAコンポーネント").
// Router reading: top-k by float32 logit, ties to the lower expert index; pairs
// p = t * k + j ordered by (expert, p).  Everything here is integer work and bit-exact.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kChunk = 256;  // pairs per histogram / scatter CTA

// -------------------------------------------------------------------- top-k (warp per token)
// One warp selects token t's k experts: ids[t k + r] for r = 0 .. k - 1 (and, when `sh` is
// given, the same ids in shared memory).
template <int VPL>  // logits held per lane: E <= 32 * VPL
__device__ __forceinline__ void topk_token(const float* __restrict__ logits, int64_t t, int32_t E,
                                           int32_t k, int32_t* __restrict__ ids, int32_t* sh,
                                           int32_t* err) {
  const int lane = threadIdx.x & 31;
  float v[VPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    v[j] = (e < E) ? __ldg(logits + t * E + e) : 0.f;
    if (e >= E) taken |= 1u << j;
    else if (isnan(v[j])) {
      set_error(err, QW_ERR_VALUE);
      taken |= 1u << j;
    }
  }
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      if (!(taken & (1u << j)) && (v[j] > bv || (v[j] == bv && e < bi))) {
        bv = v[j];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi == 0x7FFFFFFF) {  // fewer than k comparable logits
      set_error(err, QW_ERR_VALUE);
      bi = 0;
    } else if ((bi & 31) == lane) {
      taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
      ids[t * k + r] = bi;
      if (sh) sh[t * k + r] = bi;
    }
  }
}

template <int VPL>
__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, int32_t T, int32_t E, int32_t k,
                int32_t* __restrict__ ids, int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_token<VPL>(logits, t, E, k, ids, nullptr, err);
}

// -------------------------------------------------------------------- small batches: one CTA
// For at most kSmallPairs pairs and kSmallExperts experts (decode-sized batches) the whole
// routing runs in one CTA of 32 warps, with the same results as the four kernels below:
// top-k (warp per token), per-expert counts, the offsets scan, then the stable scatter in
// pair order, 1024 pairs at a time (ranks within a warp by __match_any_sync, across warps by
// per-warp counts in shared memory).
constexpr int kSmallPairs = 1024, kSmallExperts = 256;

template <int VPL>
__global__ void __launch_bounds__(1024)
    route_small_kernel(const float* __restrict__ logits, int32_t T, int32_t E, int32_t k,
                       int32_t* __restrict__ ids, int32_t* __restrict__ sorted_pairs,
                       int32_t* __restrict__ offsets, int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  __shared__ int32_t sid[kSmallPairs];
  __shared__ int32_t base[kSmallExperts + 1];
  __shared__ int32_t wcnt[32][kSmallExperts];
  __shared__ int32_t warp_sums[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int P = T * k;
  for (int t = w; t < T; t += 32) topk_token<VPL>(logits, t, E, k, ids, sid, err);
  for (int e = threadIdx.x; e < E; e += 1024) base[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += 1024) atomicAdd(&base[sid[p]], 1);
  __syncthreads();
  // exclusive scan of the counts over experts (E <= 256: warps 0 .. 7)
  {
    const int e = threadIdx.x;
    const int32_t x = e < E ? base[e] : 0;
    int32_t incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int32_t s0 = warp_sums[lane];
      int32_t si = s0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, si, off);
        if (lane >= off) si += y;
      }
      warp_sums[lane] = si - s0;
    }
    __syncthreads();
    const int32_t excl = incl - x + warp_sums[w];
    if (e < E) {
      offsets[e] = excl;
      if (e == E - 1) offsets[E] = excl + x;
      base[e] = excl;
    }
    __syncthreads();
  }
  // stable scatter, pair order; P <= 1024: one pass of 32 warps
  for (int i = threadIdx.x; i < 32 * kSmallExperts; i += 1024) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const int p = threadIdx.x;
  const bool valid = p < P;
  const int e = valid ? sid[p] : -1 - lane;  // distinct dummies never match
  const uint32_t m = __match_any_sync(0xFFFFFFFFu, e);
  const int wrank = __popc(m & ((1u << lane) - 1u));
  if (valid && wrank == 0) wcnt[w][e] = __popc(m);
  __syncthreads();
  if (valid) {
    int32_t r = base[e] + wrank;
    for (int ww = 0; ww < w; ++ww) r += wcnt[ww][e];
    sorted_pairs[r] = p;
  }
}

// -------------------------------------------------------------------- per-chunk histogram
__global__ void __launch_bounds__(kChunk)
    chunk_hist_kernel(const int32_t* __restrict__ ids, int64_t P, int32_t E,
                      int32_t* __restrict__ hist) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  extern __shared__ int32_t sh[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * kChunk + threadIdx.x;
  if (p < P) atomicAdd(&sh[__ldg(ids + p)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// -------------------------------------------------------------------- offsets (one CTA)
// hist[c][e] -> base[c][e] = offsets[e] + sum_{c' < c} hist[c'][e]; offsets = exclusive
// prefix of the per-expert totals.
__global__ void __launch_bounds__(1024)
    offsets_kernel(int32_t* __restrict__ hist, int64_t nchunks, int32_t E,
                   int32_t* __restrict__ offsets) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  __shared__ int32_t warp_sums[32];
  const int e = threadIdx.x;
  int32_t run = 0;
  if (e < E)
    for (int64_t c = 0; c < nchunks; ++c) {
      const int32_t h = hist[c * E + e];
      hist[c * E + e] = run;
      run += h;
    }
  // block-wide exclusive scan of run over e
  const int lane = e & 31, w = e >> 5;
  int32_t x = (e < E) ? run : 0;
  int32_t incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    int32_t s = warp_sums[lane];
    int32_t si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, si, off);
      if (lane >= off) si += y;
    }
    warp_sums[lane] = si - s;  // exclusive over warps
  }
  __syncthreads();
  const int32_t excl = incl - x + warp_sums[w];
  if (e < E) {
    offsets[e] = excl;
    if (e == E - 1) offsets[E] = excl + x;
    for (int64_t c = 0; c < nchunks; ++c) hist[c * E + e] += excl;
  }
}

// -------------------------------------------------------------------- stable scatter
__global__ void __launch_bounds__(kChunk)
    scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int32_t E,
                   const int32_t* __restrict__ base, int32_t* __restrict__ sorted_pairs) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  extern __shared__ int32_t cnt[];  // [kChunk / 32][E]
  constexpr int W = kChunk / 32;
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t p = (int64_t)blockIdx.x * kChunk + threadIdx.x;
  const bool valid = p < P;
  const int e = valid ? __ldg(ids + p) : -1 - lane;  // distinct dummies never match
  const uint32_t m = __match_any_sync(0xFFFFFFFFu, e);
  const int wrank = __popc(m & ((1u << lane) - 1u));
  if (valid && wrank == 0) cnt[w * E + e] = __popc(m);
  __syncthreads();
  if (valid) {
    int32_t r = __ldg(base + (int64_t)blockIdx.x * E + e) + wrank;
    for (int ww = 0; ww < w; ++ww) r += cnt[ww * E + e];
    sorted_pairs[r] = (int32_t)p;
  }
}

// -------------------------------------------------------------------- tile queue (one CTA)
__global__ void __launch_bounds__(1024)
    tile_queue_kernel(const int32_t* __restrict__ offsets, int32_t E, int32_t TR,
                      int64_t total_rows, int32_t* __restrict__ queue, int64_t max_entries,
                      int32_t* err) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int32_t b = 0, n = 0, cntile = 0;
    if (e < E) {
      // the offsets come from the caller's device memory: a segment outside
      // [0, total_rows] or a decreasing pair is reported and contributes no tiles, so
      // that no kernel ever touches a row outside the buffers
      const int64_t lo = __ldg(offsets + e), hi = __ldg(offsets + e + 1);
      if (lo < 0 || hi < lo || hi > total_rows) {
        set_error(err, QW_ERR_INVALID_ARG);
      } else {
        b = (int32_t)lo;
        n = (int32_t)(hi - lo);
      }
      cntile = (n + TR - 1) / TR;
    }
    int32_t incl = cntile;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int32_t s = warp_sums[lane];
      int32_t si = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, si, off);
        if (lane >= off) si += y;
      }
      warp_sums[lane] = si - s;
    }
    __syncthreads();
    const int32_t start = carry + warp_sums[w] + incl - cntile;
    for (int j = 0; j < cntile; ++j) {
      const int64_t q = (int64_t)start + j;
      if (q < max_entries) {
        queue[1 + 3 * q] = e;
        queue[2 + 3 * q] = b + j * TR;
        queue[3 + 3 * q] = min(b + n, b + (j + 1) * TR);
      } else {
        set_error(err, QW_ERR_WORKSPACE);
      }
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = start + cntile;
    __syncthreads();
  }
  if (threadIdx.x == 0) queue[0] = (int32_t)min64(carry, max_entries);
}

// -------------------------------------------------------------------- permutation
__global__ void permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t row_vecs, const int32_t* __restrict__ sorted_pairs,
                                    int64_t P, int32_t topk) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int64_t total = P * row_vecs;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / row_vecs, v = i % row_vecs;
    const int64_t tok = __ldg(sorted_pairs + r) / topk;
    dst[i] = __ldg(src + tok * row_vecs + v);
  }
}
__global__ void permute_bytes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                     int64_t row_bytes, const int32_t* __restrict__ sorted_pairs,
                                     int64_t P, int32_t topk) {
  pdl_wait();  // the previous kernel's outputs (launched as its dependent)
  pdl_launch_dependents();
  const int64_t total = P * row_bytes;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / row_bytes, v = i % row_bytes;
    const int64_t tok = __ldg(sorted_pairs + r) / topk;
    dst[i] = src[tok * row_bytes + v];
  }
}

// -------------------------------------------------------------------- bounded-wait probe
__global__ void wait_timeout_probe_kernel(int32_t* err, int64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up and report QW_ERR_TIMEOUT
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, (uint64_t)limit_ns);
  __syncthreads();
}

int grid_cap(int64_t total, int threads) {
  int64_t b = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

uint64_t moe_route_workspace(int32_t T, int32_t E, int32_t topk) {
  const int64_t P = (int64_t)T * topk;
  const int64_t nchunks = (P + kChunk - 1) / kChunk;
  return (uint64_t)(nchunks > 0 ? nchunks : 1) * E * 4;
}

qw_status launch_moe_route(const float* logits, int32_t T, int32_t E, int32_t topk,
                           int32_t* topk_ids, int32_t* sorted_pairs, int32_t* offsets, void* ws,
                           uint64_t ws_bytes, int32_t* err, cudaStream_t st) {
  const int64_t P = (int64_t)T * topk;
  if (ws_bytes < moe_route_workspace(T, E, topk) || ws == nullptr) return QW_ERR_WORKSPACE;
  int32_t* hist = static_cast<int32_t*>(ws);
  const int64_t nchunks = (P + kChunk - 1) / kChunk;
  if (T > 0 && P <= kSmallPairs && E <= kSmallExperts) {
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) (void)launch_pdl(route_small_kernel<1>, dim3(1), dim3(1024), 0, st, logits, T, E, topk, topk_ids, sorted_pairs, offsets, err);
    else if (vpl <= 2) (void)launch_pdl(route_small_kernel<2>, dim3(1), dim3(1024), 0, st, logits, T, E, topk, topk_ids, sorted_pairs, offsets, err);
    else if (vpl <= 4) (void)launch_pdl(route_small_kernel<4>, dim3(1), dim3(1024), 0, st, logits, T, E, topk, topk_ids, sorted_pairs, offsets, err);
    else (void)launch_pdl(route_small_kernel<8>, dim3(1), dim3(1024), 0, st, logits, T, E, topk, topk_ids, sorted_pairs, offsets, err);
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
  }
  if (T > 0) {
    const unsigned gt = (unsigned)((T + 7) / 8);
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) (void)launch_pdl(topk_kernel<1>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    else if (vpl <= 2) (void)launch_pdl(topk_kernel<2>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    else if (vpl <= 4) (void)launch_pdl(topk_kernel<4>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    else if (vpl <= 8) (void)launch_pdl(topk_kernel<8>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    else if (vpl <= 16) (void)launch_pdl(topk_kernel<16>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    else (void)launch_pdl(topk_kernel<32>, dim3(gt), dim3(256), 0, st, logits, T, E, topk, topk_ids, err);
    (void)launch_pdl(chunk_hist_kernel, dim3((unsigned)nchunks), dim3(kChunk), E * 4, st, topk_ids, P, E, hist);
  }
  (void)launch_pdl(offsets_kernel, dim3(1), dim3(1024), 0, st, hist, nchunks, E, offsets);
  if (T > 0)
    (void)launch_pdl(scatter_kernel, dim3((unsigned)nchunks), dim3(kChunk), (kChunk / 32) * E * 4, st, topk_ids, P, E, hist,
                                                                             sorted_pairs);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_moe_permute(int32_t afmt, const void* A, const void* A_sf, int32_t K,
                             const int32_t* sorted_pairs, int64_t P, int32_t topk,
                             void* A_sorted, void* A_sf_sorted, cudaStream_t st) {
  if (P == 0) return QW_OK;
  const int64_t row_bytes =
      afmt == QW_A_BF16 ? 2 * (int64_t)K : (afmt == QW_A_NVFP4_G16 ? K / 2 : (int64_t)K);
  const int64_t vecs = row_bytes / 16;
  (void)launch_pdl(permute_rows_kernel, dim3(grid_cap(P * vecs, 256)), dim3(256), 0, st, (const uint4*)A, (uint4*)A_sorted, vecs, sorted_pairs, P, topk);
  if (afmt != QW_A_BF16) {
    const int64_t sb = K / (afmt == QW_A_NVFP4_G16 ? 16 : 32);  // scale bytes per row
    (void)launch_pdl(permute_bytes_kernel, dim3(grid_cap(P * sb, 256)), dim3(256), 0, st, (const uint8_t*)A_sf, (uint8_t*)A_sf_sorted, sb, sorted_pairs, P, topk);
  }
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

uint64_t tile_queue_bytes(int32_t E, int64_t rows, int32_t tile_rows) {
  const int64_t entries = (rows + tile_rows - 1) / tile_rows + E;
  return (uint64_t)(1 + 3 * entries) * 4;
}

qw_status launch_build_tile_queue(const int32_t* offsets, int32_t E, int32_t tile_rows,
                                  int64_t total_rows, int32_t* queue, int64_t max_entries,
                                  int32_t* err, cudaStream_t st) {
  (void)launch_pdl(tile_queue_kernel, dim3(1), dim3(1024), 0, st, offsets, E, tile_rows, total_rows, queue, max_entries,
                                        err);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

qw_status launch_wait_timeout_probe(int32_t* err, int64_t limit_ns, cudaStream_t st) {
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
