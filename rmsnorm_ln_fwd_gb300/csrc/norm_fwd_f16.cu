// Forward kernels instantiated for f16 rows.

#include "fwd_kernels.cuh"

namespace normk {

template cudaError_t launch_fwd_typed<KIND_LN, F16>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_RMS, F16>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_FUSED, F16>(FwdArgs, const DeviceInfo&, cudaStream_t);

}  // namespace normk
