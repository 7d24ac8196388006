// Backward kernels instantiated for bf16 rows.

#include "bwd_kernels.cuh"

namespace normk {

template cudaError_t launch_bwd_typed<KIND_LN, BF16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS, BF16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_FUSED, BF16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_LN_Y, BF16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_bwd_typed<KIND_RMS_Y, BF16>(BwdArgs, void*, void*, const DeviceInfo&, cudaStream_t);

}  // namespace normk
