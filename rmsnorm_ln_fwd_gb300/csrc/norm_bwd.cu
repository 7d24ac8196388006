// Backward entry: the partial-count policy and the dtype/kind dispatch.  The
// kernels and their launch logic live in bwd_kernels.cuh, compiled once per
// row dtype (norm_bwd_<dtype>.cu) so the translation units build in parallel.

#include "common.cuh"
#include "launch.h"

namespace normk {

int bwd_max_partials(const DeviceInfo& dev) { return 2 * dev.sm_count; }

cudaError_t launch_backward(int kind, Dtype dt, BwdArgs a, void* dgamma, void* dbeta,
                            const DeviceInfo& dev, cudaStream_t s) {
  (void)cudaGetLastError();  // drop a stale, non-sticky error left by an earlier call
  if (dt == DT_BF16) {
    switch (kind) {
      case KIND_LN: return launch_bwd_typed<KIND_LN, BF16>(a, dgamma, dbeta, dev, s);
      case KIND_RMS: return launch_bwd_typed<KIND_RMS, BF16>(a, dgamma, nullptr, dev, s);
      case KIND_LN_Y: return launch_bwd_typed<KIND_LN_Y, BF16>(a, dgamma, dbeta, dev, s);
      case KIND_RMS_Y: return launch_bwd_typed<KIND_RMS_Y, BF16>(a, dgamma, nullptr, dev, s);
      default: return launch_bwd_typed<KIND_FUSED, BF16>(a, dgamma, nullptr, dev, s);
    }
  }
  if (dt == DT_F16) {
    switch (kind) {
      case KIND_LN: return launch_bwd_typed<KIND_LN, F16>(a, dgamma, dbeta, dev, s);
      case KIND_RMS: return launch_bwd_typed<KIND_RMS, F16>(a, dgamma, nullptr, dev, s);
      case KIND_LN_Y: return launch_bwd_typed<KIND_LN_Y, F16>(a, dgamma, dbeta, dev, s);
      case KIND_RMS_Y: return launch_bwd_typed<KIND_RMS_Y, F16>(a, dgamma, nullptr, dev, s);
      default: return launch_bwd_typed<KIND_FUSED, F16>(a, dgamma, nullptr, dev, s);
    }
  }
  switch (kind) {
    case KIND_LN: return launch_bwd_typed<KIND_LN, F32>(a, dgamma, dbeta, dev, s);
    case KIND_RMS: return launch_bwd_typed<KIND_RMS, F32>(a, dgamma, nullptr, dev, s);
    case KIND_LN_Y: return launch_bwd_typed<KIND_LN_Y, F32>(a, dgamma, dbeta, dev, s);
    case KIND_RMS_Y: return launch_bwd_typed<KIND_RMS_Y, F32>(a, dgamma, nullptr, dev, s);
    default: return launch_bwd_typed<KIND_FUSED, F32>(a, dgamma, nullptr, dev, s);
  }
}

}  // namespace normk
