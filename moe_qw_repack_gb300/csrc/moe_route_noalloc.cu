// moe_route_noalloc.cu - qgemm_moe_route for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: a plugin whose host framework owns
// every byte of device memory through its own pool, or a latency-critical decode loop
// in which an allocation (which may synchronise the device) is not permitted.  For them
// this entry point runs the same routing kernels as qgemm_moe_route, with the scratch
// those kernels need (one int32 per (chunk of 256 routed pairs, expert)) held in a
// file-scope device array instead of a caller-provided workspace.
//
// Costs and rules:
//   - The array is QW_NOALLOC_ROUTE_SCRATCH_BYTES (1 MiB) of device memory that every
//     GPU loading this library holds until the process exits.
//   - Calls whose ceil(T * topk / 256) * E * 4 bytes exceed it are rejected on the host
//     with QW_ERR_WORKSPACE before anything is enqueued.
//   - Every call shares the one array and leaves its contents behind.  Nothing in it
//     needs to start at zero: each call overwrites every element it later reads.
//     Calls that overlap on the GPU (on different streams, or from several threads
//     without ordering) race on the array and give undefined results.
//   - The stream must belong to the current device: the device address looked up below
//     is that of the current device, so a stream of another device is rejected.
//   - The first call on a device looks the array's device address up (with that device
//     current) and caches it; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/qw.h"
#include "qw_internal.h"

namespace {

constexpr int64_t kScratchInts = QW_NOALLOC_ROUTE_SCRATCH_BYTES / 4;

// The scratch itself.  In host code this name is only a host-side stand-in: the device
// address comes from cudaGetSymbolAddress (looked up once per device below).
static __device__ __align__(256) int32_t g_route_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
std::atomic<int32_t*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_route_scratch on the current device, which must be the device of
// `stream` (QW_ERR_INVALID_ARG otherwise: the kernels would run on the stream's device with
// another device's address).
qw_status scratch_for_stream(cudaStream_t stream, int32_t** out) {
  int dev = -1, sdev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QW_ERR_CUDA;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return QW_ERR_INVALID_ARG;
  if (sdev != dev) return QW_ERR_INVALID_ARG;
  int32_t* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_route_scratch) != cudaSuccess || addr == nullptr)
        return QW_ERR_CUDA;
      p = static_cast<int32_t*>(addr);
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return QW_OK;
}

}  // namespace

extern "C" qw_status qgemm_moe_route_noalloc(const float* logits, int32_t T, int32_t E,
                                             int32_t topk, int32_t* topk_ids,
                                             int32_t* sorted_pairs, int32_t* expert_offsets,
                                             int32_t* d_err, void* stream) {
  if (T < 0 || topk < 1 || topk > 32 || E < topk || E > 1024) return QW_ERR_INVALID_ARG;
  if (!expert_offsets) return QW_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_ids || !sorted_pairs)) return QW_ERR_INVALID_ARG;
  if ((int64_t)T * topk > 0x7FFFFFFFLL) return QW_ERR_UNSUPPORTED;
  if (qw::moe_route_workspace(T, E, topk) > (uint64_t)QW_NOALLOC_ROUTE_SCRATCH_BYTES)
    return QW_ERR_WORKSPACE;
  int32_t* scratch = nullptr;
  const qw_status s = scratch_for_stream(static_cast<cudaStream_t>(stream), &scratch);
  if (s != QW_OK) return s;
  return qgemm_moe_route(logits, T, E, topk, topk_ids, sorted_pairs, expert_offsets, scratch,
                         (uint64_t)QW_NOALLOC_ROUTE_SCRATCH_BYTES, d_err, stream);
}
