// dp_gemm_wgrad_noalloc: the weight gradient for callers that cannot allocate.
//
// Some callers cannot hand the library a workspace: a serving or real-time runtime
// that reserves all device memory at start-up, or a plugin whose host forbids
// cudaMalloc on its hot path because it can synchronise the device.  For them this entry point runs the same weight-gradient
// kernels as dp_gemm_wgrad_ex, with its split partials placed in a scratch array
// that is part of the library image itself.
//
// The scratch array is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads this part of the library holds it until the process exits.  In host
// code its name is only a stand-in for the device symbol, so its device address
// is looked up once per device, with that device current, via
// cudaGetSymbolAddress; the first call on each device does this set-up.  Every call
// shares the one array (the
// partials need no initial value), so calls that overlap on the GPU (two streams,
// two threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "dp_gemm.h"

namespace {

constexpr size_t kScratchBytes = size_t{64} << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_wgrad_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
dp_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DP_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || p == nullptr) return DP_ERR_LAUNCH;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DP_OK;
}

}  // namespace

extern "C" dp_status dp_gemm_wgrad_noalloc(const void* dY, int64_t ldg, const void* X, int64_t ldx, void* dW,
                                           int64_t ldw, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                                           int deterministic, dp_stream stream) {
  // the plan of this very call (its deterministic flag included) sizes the scratch
  dp_plan_info info;
  dp_status st = dp_plan_query_ex(DP_OP_WGRAD, T, N, K, out, deterministic, 0, &info);
  if (st != DP_OK) return st;
  if (info.workspace_bytes > kScratchBytes) return DP_ERR_WORKSPACE;  // beyond the built-in 64 MiB
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != DP_OK) return st;
  return dp_gemm_wgrad_ex(dY, ldg, X, ldx, dW, ldw, T, N, K, out, deterministic, scratch, kScratchBytes, stream);
}
