// Forward entry: the bulk-copy stage planner (shared with the backward) and
// the dtype/kind dispatch.  The kernels and their launch logic live in
// fwd_kernels.cuh, compiled once per row dtype (norm_fwd_<dtype>.cu).

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "staged.cuh"

namespace normk {

#ifndef NORM_STAGED_MAX_STAGES
#define NORM_STAGED_MAX_STAGES 6
#endif

bool staged_config(int H, int es, int NT, int max_smem, int max_cols, StageCfg* c, int n_par) {
  const int row_bytes = H * es;
  if (H <= 0 || row_bytes % 16 != 0) return false;
  const int vec = 16 / es;
  const int hv = H / vec;
  c->W = kStagedConsumerWarps;
  c->row_bytes = row_bytes;
  c->red_off = 256;                           // barriers + abort flag
  c->par_off = c->red_off + 2 * c->W * 3 * 4;  // after the reduction scratch
  c->par_off = (c->par_off + 127) & ~127;
  for (int G = c->W; G >= 1; G /= 2) {
    const int tpr = 32 * (c->W / G);
    const int vpt = (hv + tpr - 1) / tpr;
    const int cols = vpt * vec;
    if (max_cols > 0 && cols > max_cols) continue;
    const int data_off = (c->par_off + n_par * vpt * vec * tpr * 4 + 127) & ~127;
    const size_t stage = (size_t)NT * G * row_bytes;
    const long S = (long)(max_smem - data_off) / (long)stage;
    if (S < 3) continue;
    c->G = G;
    c->S = (int)std::min<long>(S, NORM_STAGED_MAX_STAGES);
    c->data_off = data_off;
    return true;
  }
  return false;
}

size_t staged_smem_bytes(const StageCfg& c, int NT) { return c.data_off + (size_t)c.S * NT * c.G * c.row_bytes; }

cudaError_t launch_forward(int kind, Dtype dt, FwdArgs a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  (void)cudaGetLastError();  // drop a stale, non-sticky error left by an earlier call
  if (dt == DT_BF16) {
    switch (kind) {
      case KIND_LN: return launch_fwd_typed<KIND_LN, BF16>(a, dev, s);
      case KIND_RMS: return launch_fwd_typed<KIND_RMS, BF16>(a, dev, s);
      default: return launch_fwd_typed<KIND_FUSED, BF16>(a, dev, s);
    }
  }
  if (dt == DT_F16) {
    switch (kind) {
      case KIND_LN: return launch_fwd_typed<KIND_LN, F16>(a, dev, s);
      case KIND_RMS: return launch_fwd_typed<KIND_RMS, F16>(a, dev, s);
      default: return launch_fwd_typed<KIND_FUSED, F16>(a, dev, s);
    }
  }
  switch (kind) {
    case KIND_LN: return launch_fwd_typed<KIND_LN, F32>(a, dev, s);
    case KIND_RMS: return launch_fwd_typed<KIND_RMS, F32>(a, dev, s);
    default: return launch_fwd_typed<KIND_FUSED, F32>(a, dev, s);
  }
}

}  // namespace normk
