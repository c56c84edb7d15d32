// diag.cu - a plain streaming read, the reference point the HBM-bound kernels are measured
// against: the same bytes read with 16-byte loads by a full grid, folded into one word per
// CTA (written out so the loads cannot be dropped).  No method arithmetic.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kReadUnroll = 4;  // 16-byte loads in flight per thread

// `chained`: loads go before griddepcontrol.wait (only the one output word waits), as a
// programmatic dependent launch allows for a kernel that reads nothing its predecessor wrote.
template <bool CHAINED>
__global__ void __launch_bounds__(256) stream_read_kernel(const uint4* __restrict__ src, uint64_t n16,
                                                          uint32_t* __restrict__ sink) {
  if (CHAINED) pdl_launch_dependents();
  uint32_t acc = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
  for (; i + (kReadUnroll - 1) * stride < n16; i += kReadUnroll * stride) {
    uint4 v[kReadUnroll];
#pragma unroll
    for (int u = 0; u < kReadUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kReadUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  __shared__ uint32_t part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (CHAINED) pdl_wait();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a ^= part[w];
    sink[blockIdx.x] = a;
  }
}

}  // namespace

qw_status launch_stream_read(const void* src, uint64_t bytes, uint32_t* sink, bool chained,
                             cudaStream_t st) {
  // a full grid: every SM holds eight CTAs of 256 threads (the thread limit)
  int64_t grid = (int64_t)device_sm_count() * 8;
  if (grid > QW_STREAM_READ_SINK_WORDS) grid = QW_STREAM_READ_SINK_WORDS;
  const uint4* p = static_cast<const uint4*>(src);
  if (chained)
    return launch_pdl(stream_read_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, p,
                      bytes / 16, sink);
  stream_read_kernel<false><<<(unsigned)grid, 256, 0, st>>>(p, bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ERR_CUDA;
}

}  // namespace qw
