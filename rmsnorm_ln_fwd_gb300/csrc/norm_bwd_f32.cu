// Backward kernels instantiated for f32 rows.

#include "bwd_kernels.cuh"

namespace normk {

template cudaError_t launch_bwd_typed<KIND_LN, F32>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS, F32>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_FUSED, F32>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_LN_Y, F32>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS_Y, F32>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);

}  // namespace normk
