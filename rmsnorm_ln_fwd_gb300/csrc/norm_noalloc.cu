// ln_backward without a caller-supplied workspace.
//
// The LayerNorm backward needs device scratch for its fp32 dgamma/dbeta
// partial rows.  ln_backward takes that scratch from the caller, who must
// have allocated it.  Some callers cannot allocate device memory when they
// call us: a plugin running inside a host framework that owns all device
// memory and hands plugins no allocator, or latency-critical code that must
// not pay for cudaMalloc (and the device-wide synchronisation it can imply)
// in the middle of a step.  For them, ln_backward_static_workspace uses a
// scratch array that lives in this library's device image instead.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds its own copy, NORM_STATIC_WORKSPACE_BYTES (64 MiB), until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it.  Nothing
// here calls cudaMalloc, cudaFree or any allocating routine.

#include <cuda_runtime.h>

#include <mutex>

#include "norm.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = NORM_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// One copy per device; shared by every call on that device.
static __device__ __align__(256) float g_static_workspace[kStaticWorkspaceBytes / sizeof(float)];

std::mutex g_mu;
void* g_addr[kMaxDevices];

// This device's copy of the array (set-up on the first call per device).
norm_status static_workspace(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return NORM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return NORM_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NORM_OK;
}

}  // namespace

extern "C" norm_status ln_backward_static_workspace(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                                                    const float* mean, const float* rstd, const void* gamma,
                                                    void* dx, int64_t lddx, void* dgamma, void* dbeta,
                                                    int64_t N, int64_t H, norm_dtype x_dtype,
                                                    norm_dtype w_dtype, norm_stream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return NORM_ERR_CUDA;
  if (dgamma != nullptr || dbeta != nullptr) {
    // A width whose partial rows do not fit the array is refused up front.
    const size_t need = norm_bwd_workspace_bytes(H, dev);
    if (need > kStaticWorkspaceBytes) return NORM_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const norm_status st = static_workspace(dev, &ws);
  if (st != NORM_OK) return st;
  return ln_backward(dy, lddy, x, ldx, mean, rstd, gamma, dx, lddx, dgamma, dbeta, ws, kStaticWorkspaceBytes, N,
                     H, x_dtype, w_dtype, stream);
}
