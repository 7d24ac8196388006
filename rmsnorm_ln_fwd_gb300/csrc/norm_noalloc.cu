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
// process exits.  With lazy module loading (CUDA's default) the driver
// reserves that memory when the module is first used on a device, which can
// be this entry point's first call there; a caller whose framework later
// takes all device memory should make one set-up call first (N == 0 does).
// Host code cannot use the array's name as a device address, so every call
// looks the current device's copy up with cudaGetSymbolAddress (a host-side
// lookup once the module is loaded; looking it up each time stays right after
// a device reset reloads the module).  Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.

#include <cuda_runtime.h>

#include "norm.h"

namespace normk {
void note_cuda_error(const char* where, cudaError_t e);
void note_error_text(const char* text);
}  // namespace normk

namespace {

constexpr size_t kStaticWorkspaceBytes = NORM_STATIC_WORKSPACE_BYTES;

// One copy per device; shared by every call on that device.
static __device__ __align__(256) float g_static_workspace[kStaticWorkspaceBytes / sizeof(float)];

}  // namespace

extern "C" norm_status ln_backward_static_workspace(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                                                    const float* mean, const float* rstd, const void* gamma,
                                                    void* dx, int64_t lddx, void* dgamma, void* dbeta,
                                                    int64_t N, int64_t H, norm_dtype x_dtype,
                                                    norm_dtype w_dtype, norm_stream_t stream) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    normk::note_cuda_error("cudaGetDevice", e);
    return NORM_ERR_CUDA;
  }
  if ((dgamma != nullptr || dbeta != nullptr) && N > 0) {
    // A width whose partial rows do not fit the array is refused up front; so
    // is a width the device cannot be asked to size (0: H out of range or no
    // device attributes).
    const size_t need = norm_bwd_workspace_bytes(H, dev);
    if (need == 0) {
      if (H < 1) return NORM_ERR_INVALID_VALUE;
      normk::note_error_text("ln_backward_static_workspace: could not size the partial rows on this device");
      return NORM_ERR_WORKSPACE;
    }
    if (need > kStaticWorkspaceBytes) return NORM_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  e = cudaGetSymbolAddress(&ws, g_static_workspace);  // this device's copy
  if (e != cudaSuccess || ws == nullptr) {
    normk::note_cuda_error("cudaGetSymbolAddress (static workspace)", e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    return NORM_ERR_CUDA;
  }
  return ln_backward(dy, lddy, x, ldx, mean, rstd, gamma, dx, lddx, dgamma, dbeta, ws, kStaticWorkspaceBytes, N,
                     H, x_dtype, w_dtype, stream);
}
