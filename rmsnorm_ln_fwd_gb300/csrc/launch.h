// Internal interface between the C ABI (norm_api.cu) and the kernel
// translation units (norm_fwd.cu, norm_bwd.cu).  Arguments arrive here already
// validated; these functions only pick a kernel configuration and launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace normk {

enum Dtype : int { DT_F32 = 0, DT_BF16 = 1 };
enum Kind : int { KIND_LN = 0, KIND_RMS = 1, KIND_FUSED = 2 };

struct DeviceInfo {
  int sm_count;
  int max_smem_optin;  // bytes of shared memory one CTA may opt into
};

// Forward: LayerNorm (KIND_LN), RMSNorm (KIND_RMS), fused add + RMSNorm (KIND_FUSED).
struct FwdArgs {
  const void* x;
  int64_t ldx;
  const void* res;  // fused only
  int64_t ldr;
  const void* gamma;  // may be null (ones)
  const void* beta;   // LN only; may be null (zeros)
  void* y;
  int64_t ldy;
  void* h;  // fused only: the summed residual stream
  int64_t ldh;
  float* mean;  // LN only; may be null
  float* rstd;  // may be null
  int64_t N;
  int H;
  float eps;
  int w_f32;    // parameters are fp32 (else the row dtype)
  int h_alias;  // fused: h_out is exactly x or residual
  int tpr;      // threads per row (filled in by the launcher)
};

// Backward: LayerNorm (KIND_LN) or RMSNorm (KIND_RMS).
struct BwdArgs {
  const void* dy;
  int64_t lddy;
  const void* x;
  int64_t ldx;
  const float* mean;  // LN only
  const float* rstd;
  const void* gamma;  // may be null (ones)
  void* dx;
  int64_t lddx;
  float* ws;  // [2][P][Hp] fp32 partial rows (dgamma, dbeta), or null
  int Hp;     // partial row stride in floats (H rounded up to 4)
  int64_t N;
  int H;
  int w_f32;
  int tpr;  // threads per row (filled in by the launcher)
};

// Partial rows the backward may use on a device: a fixed multiple of the SM
// count, independent of the number of input rows.
int bwd_max_partials(const DeviceInfo& dev);
inline int bwd_partial_stride(int H) { return (H + 3) & ~3; }

cudaError_t launch_forward(int kind, Dtype dt, FwdArgs a, const DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_backward(int kind, Dtype dt, BwdArgs a, void* dgamma, void* dbeta,
                            const DeviceInfo& dev, cudaStream_t s);

}  // namespace normk
