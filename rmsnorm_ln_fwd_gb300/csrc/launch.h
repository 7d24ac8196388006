// Internal interface between the C ABI (norm_api.cu) and the kernel
// translation units (norm_fwd.cu, norm_bwd.cu).  Arguments arrive here already
// validated; these functions only pick a kernel configuration and launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace normk {

enum Dtype : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum Kind : int { KIND_LN = 0, KIND_RMS = 1, KIND_FUSED = 2, KIND_LN_Y = 3, KIND_RMS_Y = 4 };

// Backward kinds that recover x_hat from the forward's saved output y
// (x_hat = (y - beta)/gamma, RMSNorm y/gamma) instead of from x and mean.
__host__ __device__ constexpr bool kind_from_y(int k) { return k == KIND_LN_Y || k == KIND_RMS_Y; }
__host__ __device__ constexpr bool kind_is_ln(int k) { return k == KIND_LN || k == KIND_LN_Y; }

// Kernel-family policy (norm_set_kernel_path).  AUTO: register rows when a
// row needs at most kRowsAutoMaxThreads threads, else the bulk-copy pipeline,
// else register rows, else the loop.  ROWS: register rows, else loop.  LOOP:
// loop only.  STAGED: bulk-copy pipeline, else register rows, else loop.
enum Path : int { PATH_AUTO = 0, PATH_ROWS = 1, PATH_LOOP = 2, PATH_STAGED = 3 };
constexpr int kRowsAutoMaxThreads = 640;

struct DeviceInfo {
  int sm_count;
  int max_smem_optin;  // bytes of shared memory one CTA may opt into
  unsigned* err;       // this device's error-flag word (see norm_device_errors)
  int path;            // first kernel family to try (norm_set_kernel_path)
  void* split_event;   // cudaEvent_t recorded between the backward's two kernels, or null
                       // (norm_set_bwd_split_event; the reduction then runs without PDL)
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
  int tpr;      // threads per row (filled in by the launcher)
  unsigned* err;  // device error flags (bounded waits of cluster rows; filled in by the launcher)
};

// Backward: LayerNorm (KIND_LN) or RMSNorm (KIND_RMS) from x and the saved
// statistics, the same from the saved output (KIND_LN_Y, KIND_RMS_Y), or the
// fused add + RMSNorm from the stored sum (KIND_FUSED).
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
  // Backward from the saved output (KIND_LN_Y, KIND_RMS_Y; x is y):
  const void* beta;  // LN_Y: the forward's beta, or null (zeros)
  // Fused add + RMSNorm backward only (KIND_FUSED; x is the stored h):
  const void* dh_in;  // gradient arriving through h (the residual stream), or null
  int64_t lddh;
  void* dres;  // second copy of dL/dh for the residual input, or null
  int64_t lddres;
  int dx_twice;  // dres is dx itself (x and residual were one tensor): dx = 2 dL/dh
  int64_t N;
  int H;
  int w_f32;
  int tpr;        // threads per row (filled in by the launcher)
  unsigned* err;  // device error flags (bounded waits of cluster rows; filled in by the launcher)
};

// Shape of a staged (bulk-copy pipelined) launch, chosen on the host.  The CTA
// has W consumer warps plus one producer warp; each stage of the shared-memory
// ring holds G rows (one per consumer row group of W/G warps) of every staged
// tensor, tensor-major: [tensor][row][H elements].
struct StageCfg {
  int G;             // rows per stage = consumer row groups
  int S;             // stages in the ring
  int W;             // consumer warps
  int row_bytes;     // H * element size (a multiple of 16)
  int red_off;       // byte offset of the cross-warp reduction scratch
  int par_off;       // byte offset of the fp32 parameter copies (thread-interleaved)
  int data_off;      // byte offset of stage 0
  int contiguous;    // rows of every staged tensor are back to back (ld == H)
  unsigned* err;     // device error flags (bounded waits that ran out)
};

constexpr int kStagedConsumerWarps = 16;
constexpr int kStagedThreads = (kStagedConsumerWarps + 1) * 32;

// Partial rows the backward may use on a device: a fixed multiple of the SM
// count, independent of the number of input rows.
int bwd_max_partials(const DeviceInfo& dev);
inline int bwd_partial_stride(int H) { return (H + 3) & ~3; }

// Per-dtype launch logic, defined in fwd_kernels.cuh / bwd_kernels.cuh and
// instantiated in norm_fwd_<dtype>.cu / norm_bwd_<dtype>.cu.
template <int KIND, typename D>
cudaError_t launch_fwd_typed(FwdArgs a, const DeviceInfo& dev, cudaStream_t s);
template <int KIND, typename D>
cudaError_t launch_bwd_typed(BwdArgs a, void* dg, void* db, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_forward(int kind, Dtype dt, FwdArgs a, const DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_backward(int kind, Dtype dt, BwdArgs a, void* dgamma, void* dbeta,
                            const DeviceInfo& dev, cudaStream_t s);

}  // namespace normk
