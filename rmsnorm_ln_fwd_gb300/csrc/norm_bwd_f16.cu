// Backward kernels instantiated for f16 rows.

#include "bwd_kernels.cuh"

namespace normk {

template cudaError_t launch_bwd_typed<KIND_LN, F16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS, F16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_FUSED, F16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_LN_Y, F16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS_Y, F16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);

}  // namespace normk
