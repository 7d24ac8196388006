// Forward kernels instantiated for f32 rows.

#include "fwd_kernels.cuh"

namespace normk {

template cudaError_t launch_fwd_typed<KIND_LN, F32>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_RMS, F32>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_FUSED, F32>(FwdArgs, const DeviceInfo&, cudaStream_t);

}  // namespace normk
