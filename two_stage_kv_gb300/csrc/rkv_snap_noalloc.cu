// Stage-1 eviction without a caller-provided workspace.
//
// rkv_snap_evict needs device scratch (softmax statistics, score partials and
// pooled scores) that its caller allocates.  Some callers cannot allocate:
// serving engines whose memory pool already owns all device memory (a
// cudaMalloc beside the pool can fail or fragment it), and plugin or callback
// hooks that run inside another framework's step and must not call cudaMalloc
// (it can synchronise the device).  rkv_snap_evict_noalloc serves them from
// one fixed array of device memory that belongs to this library.
#include <cstdio>
#include <mutex>

#include "rkv.h"
#include "rkv_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB

// The scratch itself.  Every GPU on which the library's device code is loaded
// holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_snap_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" rkv_status rkv_snap_evict_noalloc(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v,
                                             int64_t cap, int64_t S, int32_t pool_kernel, int32_t n_sink, int64_t B1,
                                             float scale, int32_t* keep_idx, int64_t keep_ld, void* k_out,
                                             void* v_out, int64_t out_cap, float* pooled_out, void* stream) {
  char msg[256];
  const size_t need = rkv_snap_evict_workspace(d, S, W);
  if (need > kScratchBytes) {
    snprintf(msg, sizeof(msg),
             "snap_evict_noalloc: this shape needs %zu bytes of scratch; the fixed scratch holds %zu", need,
             kScratchBytes);
    rkv::set_last_error(msg);
    return RKV_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "snap_evict_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    rkv::set_last_error(msg);
    return RKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof(msg), "snap_evict_noalloc: device ordinal %d is past the %d devices this entry point serves",
             dev, kMaxDevices);
    rkv::set_last_error(msg);
    return RKV_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  {
    // the host-side name of the array is not a device address: look the
    // address up once per device, with that device current
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
      e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_snap_scratch);
      if (e != cudaSuccess) {
        g_scratch_addr[dev] = nullptr;
        snprintf(msg, sizeof(msg), "snap_evict_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        rkv::set_last_error(msg);
        return RKV_ERR_CUDA;
      }
    }
    scratch = g_scratch_addr[dev];
  }
  return rkv_snap_evict(d, q_obs, W, k, v, cap, S, pool_kernel, n_sink, B1, scale, keep_idx, keep_ld, k_out, v_out,
                        out_cap, pooled_out, scratch, kScratchBytes, stream);
}
