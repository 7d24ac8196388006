// Forward kernels instantiated for bf16 rows.

#include "fwd_kernels.cuh"

namespace normk {

template cudaError_t launch_fwd_typed<KIND_LN, BF16>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_RMS, BF16>(FwdArgs, const DeviceInfo&, cudaStream_t);
template cudaError_t launch_fwd_typed<KIND_FUSED, BF16>(FwdArgs, const DeviceInfo&, cudaStream_t);

}  // namespace normk
