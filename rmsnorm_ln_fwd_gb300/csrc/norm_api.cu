// The C ABI declared in include/norm.h: host-side argument validation, the
// per-device attribute cache, and dispatch to the kernel launchers.
//
// Validation happens entirely on the host and before anything is enqueued, so
// an invalid call has no effect on the GPU.  No entry point throws, aborts or
// allocates.

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "norm.h"
#include <nvtx3/nvToolsExt.h>

using normk::BwdArgs;
using normk::DeviceInfo;
using normk::FwdArgs;

namespace {

constexpr int64_t kMaxH = int64_t(1) << 24;  // counts stay exact in fp32
constexpr int kMaxDevices = 64;

std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
std::atomic<int> g_path{normk::PATH_AUTO};
std::atomic<void*> g_split_event{nullptr};

}  // namespace

// One error word per device: kernels OR error bits into it (a bounded wait
// that ran out) instead of trapping; norm_device_errors reads it.
__device__ unsigned g_norm_device_errors;

// Self-test of the bounded wait: an mbarrier nothing ever arrives on, waited
// on by one warp with a short limit.  The wait must give up, record
// kErrWaitTimeout and let the kernel return; no copy is in flight.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    normk::mbar_init(&bar, 1);
    abort_flag = 0;
    normk::fence_barrier_init();
  }
  __syncwarp();
  normk::mbar_wait(&bar, 0, err, &abort_flag, limit_ns);
}

namespace {

thread_local char t_last_error[256] = "";

void note_error(const char* where, cudaError_t e) {
  snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

}  // namespace

namespace normk {
// For the other translation units of the library (not part of the C ABI).
void note_cuda_error(const char* where, cudaError_t e) { note_error(where, e); }
void note_error_text(const char* text) { snprintf(t_last_error, sizeof(t_last_error), "%s", text); }
}  // namespace normk

namespace {

bool device_info(int dev, DeviceInfo* out) {
  if (dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_have[dev]) {
    DeviceInfo d{};
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    if (d.sm_count < 1) return false;
    g_info[dev] = d;
    g_have[dev] = true;
  }
  *out = g_info[dev];
  return true;
}

bool current_device_info(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    note_error("cudaGetDevice", e);
    return false;
  }
  if (!device_info(dev, out)) {
    snprintf(t_last_error, sizeof(t_last_error), "device %d: attribute query failed", dev);
    return false;
  }
  if (out->err == nullptr) {
    // The symbol's address on the current device (this device).
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_device_errors);
    if (e != cudaSuccess) {
      note_error("cudaGetSymbolAddress", e);
      return false;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    g_info[dev].err = static_cast<unsigned*>(p);
    out->err = g_info[dev].err;
  }
  out->path = g_path.load(std::memory_order_relaxed);
  out->split_event = g_split_event.load(std::memory_order_relaxed);
  return true;
}

size_t elem_size(norm_dtype d) { return d == NORM_F32 ? 4 : 2; }

norm_status check_dtypes(norm_dtype x, norm_dtype w) {
  const bool xv = x == NORM_F32 || x == NORM_BF16 || x == NORM_F16;
  const bool wv = w == NORM_F32 || w == NORM_BF16 || w == NORM_F16;
  if (!xv || !wv) return NORM_ERR_UNSUPPORTED;
  if (w != x && w != NORM_F32) return NORM_ERR_UNSUPPORTED;
  return NORM_OK;
}

bool shape_ok(int64_t N, int64_t H) { return N >= 0 && H >= 1 && H <= kMaxH; }

bool eps_ok(float eps) { return std::isfinite(eps) && eps > 0.f; }

// The byte range [lo, hi) touched by N rows of H elements, `ld` apart.
struct Span {
  uintptr_t lo, hi;
};

// ld >= H and the extent (N-1)*ld + H elements fits comfortably in 63 bits.
bool ld_ok(int64_t ld, int64_t N, int64_t H, size_t es) {
  if (ld < H) return false;
  if (N <= 1) return true;
  const int64_t limit = (INT64_MAX / 8) / (int64_t)es;
  return (N - 1) <= (limit - H) / ld;
}

Span rows_span(const void* p, int64_t N, int64_t ld, int64_t H, size_t es) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  const uint64_t n = N == 0 ? 0 : (uint64_t)((N - 1) * ld + H) * es;
  return Span{lo, lo + n};
}

Span vec_span(const void* p, int64_t n, size_t es) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + (uint64_t)n * es};
}

bool overlap(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

// Whether any span of `a` overlaps any span of `b` (empty spans never do).
template <size_t NA, size_t NB>
bool any_overlap(const Span (&a)[NA], const Span (&b)[NB]) {
  for (const Span& p : a)
    for (const Span& q : b)
      if (overlap(p, q)) return true;
  return false;
}

constexpr Span kNoSpan{0, 0};

// Two row tensors may be the same buffer (same pointer and stride) or
// disjoint; anything in between is a partial overlap.
bool same_or_disjoint(const void* p, int64_t ldp, const void* q, int64_t ldq, int64_t N, int64_t H, size_t es) {
  if (p == q && ldp == ldq) return true;
  return !overlap(rows_span(p, N, ldp, H, es), rows_span(q, N, ldq, H, es));
}

bool disjoint_rows(const void* p, int64_t ldp, const void* q, int64_t ldq, int64_t N, int64_t H, size_t es) {
  return !overlap(rows_span(p, N, ldp, H, es), rows_span(q, N, ldq, H, es));
}

norm_status launch_result(const char* where, cudaError_t e) {
  if (e == cudaSuccess) return NORM_OK;
  note_error(where, e);
  return NORM_ERR_CUDA;
}

normk::Dtype to_dt(norm_dtype d) {
  return d == NORM_BF16 ? normk::DT_BF16 : (d == NORM_F16 ? normk::DT_F16 : normk::DT_F32);
}

norm_status forward_common(int kind, const void* x, int64_t ldx, const void* res, int64_t ldr,
                           const void* gamma, const void* beta, void* y, int64_t ldy, void* h,
                           int64_t ldh, float* mean, float* rstd, int64_t N, int64_t H, float eps,
                           norm_dtype xd, norm_dtype wd, norm_stream_t stream) {
  norm_status st = check_dtypes(xd, wd);
  if (st != NORM_OK) return st;
  if (!shape_ok(N, H) || !eps_ok(eps)) return NORM_ERR_INVALID_VALUE;
  if (N == 0) return NORM_OK;  // nothing to read or write; pointers may be NULL
  if (x == nullptr || y == nullptr) return NORM_ERR_INVALID_VALUE;
  const size_t es = elem_size(xd);
  if (!ld_ok(ldx, N, H, es) || !ld_ok(ldy, N, H, es)) return NORM_ERR_INVALID_VALUE;
  const bool fused = kind == normk::KIND_FUSED;
  if (fused) {
    if (res == nullptr || h == nullptr) return NORM_ERR_INVALID_VALUE;
    if (!ld_ok(ldr, N, H, es) || !ld_ok(ldh, N, H, es)) return NORM_ERR_INVALID_VALUE;
    // y is a fresh output: disjoint from every other row tensor.
    if (!disjoint_rows(y, ldy, x, ldx, N, H, es) || !disjoint_rows(y, ldy, res, ldr, N, H, es) ||
        !disjoint_rows(y, ldy, h, ldh, N, H, es))
      return NORM_ERR_INVALID_VALUE;
    // h may replace x or residual in place; then the other input must be that
    // same buffer too or stay clear of it.
    if (!same_or_disjoint(h, ldh, x, ldx, N, H, es) || !same_or_disjoint(h, ldh, res, ldr, N, H, es))
      return NORM_ERR_INVALID_VALUE;
  } else {
    if (!same_or_disjoint(y, ldy, x, ldx, N, H, es)) return NORM_ERR_INVALID_VALUE;
  }
  if (mean && rstd && overlap(vec_span(mean, N, 4), vec_span(rstd, N, 4))) return NORM_ERR_INVALID_VALUE;
  {
    // The statistics and parameters stay clear of every output, and the saved
    // statistics clear of the input rows.
    const size_t wes = elem_size(wd);
    const Span stats[] = {mean ? vec_span(mean, N, 4) : kNoSpan, rstd ? vec_span(rstd, N, 4) : kNoSpan};
    const Span params[] = {gamma ? vec_span(gamma, H, wes) : kNoSpan, beta ? vec_span(beta, H, wes) : kNoSpan};
    const Span out_rows[] = {rows_span(y, N, ldy, H, es), fused ? rows_span(h, N, ldh, H, es) : kNoSpan};
    const Span in_rows[] = {rows_span(x, N, ldx, H, es), fused ? rows_span(res, N, ldr, H, es) : kNoSpan};
    if (any_overlap(params, out_rows) || any_overlap(params, stats) || any_overlap(stats, out_rows) ||
        any_overlap(stats, in_rows))
      return NORM_ERR_INVALID_VALUE;
  }
  DeviceInfo dev;
  if (!current_device_info(&dev)) return NORM_ERR_CUDA;
  FwdArgs a{};
  a.x = x;
  a.ldx = ldx;
  a.res = res;
  a.ldr = ldr;
  a.gamma = gamma;
  a.beta = beta;
  a.y = y;
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.mean = mean;
  a.rstd = rstd;
  a.N = N;
  a.H = (int)H;
  a.eps = eps;
  a.w_f32 = wd == NORM_F32;
  return launch_result("forward launch", normk::launch_forward(kind, to_dt(xd), a, dev,
                                                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t workspace_bytes_for(int64_t H, const DeviceInfo& dev) {
  return 2 * (size_t)normk::bwd_max_partials(dev) * (size_t)normk::bwd_partial_stride((int)H) * sizeof(float);
}

norm_status backward_common(int kind, const void* dy, int64_t lddy, const void* x, int64_t ldx,
                            const float* mean, const float* rstd, const void* gamma, void* dx,
                            int64_t lddx, void* dgamma, void* dbeta, void* ws, size_t ws_bytes,
                            int64_t N, int64_t H, norm_dtype xd, norm_dtype wd, norm_stream_t stream,
                            const void* dh_in = nullptr, int64_t lddh = 0, void* dres = nullptr,
                            int64_t lddres = 0, const void* beta = nullptr) {
  norm_status st = check_dtypes(xd, wd);
  if (st != NORM_OK) return st;
  if (!shape_ok(N, H)) return NORM_ERR_INVALID_VALUE;
  const size_t es = elem_size(xd);
  const size_t wes = elem_size(wd);
  if (dgamma && dbeta && overlap(vec_span(dgamma, H, wes), vec_span(dbeta, H, wes))) return NORM_ERR_INVALID_VALUE;
  if (N == 0) {
    // A sum over no rows: the parameter gradients are zero.  No workspace.
    DeviceInfo dev;
    if (!current_device_info(&dev)) return NORM_ERR_CUDA;
    BwdArgs a{};
    a.N = 0;
    a.H = (int)H;
    a.w_f32 = wd == NORM_F32;
    return launch_result("backward (N = 0) launch", normk::launch_backward(kind, to_dt(xd), a, dgamma, dbeta, dev,
                                                                     reinterpret_cast<cudaStream_t>(stream)));
  }
  if (dy == nullptr || x == nullptr || dx == nullptr || rstd == nullptr) return NORM_ERR_INVALID_VALUE;
  if (kind == normk::KIND_LN && mean == nullptr) return NORM_ERR_INVALID_VALUE;
  if (!ld_ok(lddy, N, H, es) || !ld_ok(ldx, N, H, es) || !ld_ok(lddx, N, H, es)) return NORM_ERR_INVALID_VALUE;
  if (!disjoint_rows(dx, lddx, x, ldx, N, H, es) || !same_or_disjoint(dx, lddx, dy, lddy, N, H, es))
    return NORM_ERR_INVALID_VALUE;
  // Fused-add extras: the stream gradient may be dx itself (accumulate in
  // place); a second output is dx itself (one tensor fed both inputs) or a
  // separate buffer clear of everything but the inputs it may replace.
  const bool dx_twice = dres != nullptr && dres == dx && lddres == lddx;
  if (dh_in) {
    if (!ld_ok(lddh, N, H, es) || !same_or_disjoint(dx, lddx, dh_in, lddh, N, H, es)) return NORM_ERR_INVALID_VALUE;
  }
  if (dres && !dx_twice) {
    if (!ld_ok(lddres, N, H, es) || !disjoint_rows(dres, lddres, x, ldx, N, H, es) ||
        !disjoint_rows(dres, lddres, dx, lddx, N, H, es) || !same_or_disjoint(dres, lddres, dy, lddy, N, H, es))
      return NORM_ERR_INVALID_VALUE;
    if (dh_in && !same_or_disjoint(dres, lddres, dh_in, lddh, N, H, es)) return NORM_ERR_INVALID_VALUE;
  }
  const Span sdx = rows_span(dx, N, lddx, H, es);
  if (dgamma && overlap(vec_span(dgamma, H, wes), sdx)) return NORM_ERR_INVALID_VALUE;
  if (dbeta && overlap(vec_span(dbeta, H, wes), sdx)) return NORM_ERR_INVALID_VALUE;
  {
    // The saved statistics and parameters (inputs) stay clear of every
    // output, and the parameter gradients clear of every input.
    const Span small_in[] = {mean ? vec_span(mean, N, 4) : kNoSpan, vec_span(rstd, N, 4),
                             gamma ? vec_span(gamma, H, wes) : kNoSpan, beta ? vec_span(beta, H, wes) : kNoSpan};
    const Span pgrads[] = {dgamma ? vec_span(dgamma, H, wes) : kNoSpan, dbeta ? vec_span(dbeta, H, wes) : kNoSpan};
    const Span out_rows[] = {sdx, (dres && !dx_twice) ? rows_span(dres, N, lddres, H, es) : kNoSpan};
    const Span in_rows[] = {rows_span(dy, N, lddy, H, es), rows_span(x, N, ldx, H, es),
                            dh_in ? rows_span(dh_in, N, lddh, H, es) : kNoSpan};
    if (any_overlap(small_in, out_rows) || any_overlap(small_in, pgrads) || any_overlap(pgrads, in_rows) ||
        any_overlap(pgrads, out_rows))
      return NORM_ERR_INVALID_VALUE;
  }
  const bool want = dgamma != nullptr || dbeta != nullptr;
  if (want) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return NORM_ERR_WORKSPACE;
    const Span sws[] = {Span{reinterpret_cast<uintptr_t>(ws), reinterpret_cast<uintptr_t>(ws) + ws_bytes}};
    // The workspace is scratch: clear of every input and output.
    const Span others[] = {sdx,
                           (dres && !dx_twice) ? rows_span(dres, N, lddres, H, es) : kNoSpan,
                           dgamma ? vec_span(dgamma, H, wes) : kNoSpan,
                           dbeta ? vec_span(dbeta, H, wes) : kNoSpan,
                           rows_span(dy, N, lddy, H, es),
                           rows_span(x, N, ldx, H, es),
                           dh_in ? rows_span(dh_in, N, lddh, H, es) : kNoSpan,
                           mean ? vec_span(mean, N, 4) : kNoSpan,
                           vec_span(rstd, N, 4),
                           gamma ? vec_span(gamma, H, wes) : kNoSpan,
                           beta ? vec_span(beta, H, wes) : kNoSpan};
    if (any_overlap(sws, others)) return NORM_ERR_WORKSPACE;
  }
  DeviceInfo dev;
  if (!current_device_info(&dev)) return NORM_ERR_CUDA;
  if (want && ws_bytes < workspace_bytes_for(H, dev)) return NORM_ERR_WORKSPACE;
  BwdArgs a{};
  a.dy = dy;
  a.lddy = lddy;
  a.x = x;
  a.ldx = ldx;
  a.mean = mean;
  a.rstd = rstd;
  a.gamma = gamma;
  a.dx = dx;
  a.lddx = lddx;
  a.ws = static_cast<float*>(ws);
  a.N = N;
  a.H = (int)H;
  a.w_f32 = wd == NORM_F32;
  a.beta = beta;
  a.dh_in = dh_in;
  a.lddh = lddh;
  a.dres = dx_twice ? nullptr : dres;
  a.lddres = lddres;
  a.dx_twice = dx_twice;
  return launch_result("backward launch", normk::launch_backward(kind, to_dt(xd), a, dgamma, dbeta, dev,
                                                                 reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

// Each compute entry point is an NVTX range named after it, so a profiler
// (ncu --nvtx, nsys) can attribute kernels to the call that launched them; with
// no tool attached a range costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

extern "C" {

norm_status ln_forward(const void* x, int64_t ldx, const void* gamma, const void* beta, void* y, int64_t ldy,
                       float* mean, float* rstd, int64_t N, int64_t H, float eps, norm_dtype x_dtype,
                       norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("ln_forward");
  return forward_common(normk::KIND_LN, x, ldx, nullptr, 0, gamma, beta, y, ldy, nullptr, 0, mean, rstd, N, H,
                        eps, x_dtype, w_dtype, stream);
}

norm_status rms_forward(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy, float* rstd,
                        int64_t N, int64_t H, float eps, norm_dtype x_dtype, norm_dtype w_dtype,
                        norm_stream_t stream) {
  NvtxRange range("rms_forward");
  return forward_common(normk::KIND_RMS, x, ldx, nullptr, 0, gamma, nullptr, y, ldy, nullptr, 0, nullptr, rstd,
                        N, H, eps, x_dtype, w_dtype, stream);
}

norm_status fused_add_rms_forward(const void* x, int64_t ldx, const void* residual, int64_t ldr,
                                  const void* gamma, void* y, int64_t ldy, void* h_out, int64_t ldh,
                                  float* rstd, int64_t N, int64_t H, float eps, norm_dtype x_dtype,
                                  norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("fused_add_rms_forward");
  return forward_common(normk::KIND_FUSED, x, ldx, residual, ldr, gamma, nullptr, y, ldy, h_out, ldh, nullptr,
                        rstd, N, H, eps, x_dtype, w_dtype, stream);
}

size_t norm_bwd_workspace_bytes(int64_t H, int device) {
  if (H < 1 || H > kMaxH) return 0;
  DeviceInfo dev;
  if (!device_info(device, &dev)) return 0;
  return workspace_bytes_for(H, dev);
}

norm_status ln_backward(const void* dy, int64_t lddy, const void* x, int64_t ldx, const float* mean,
                        const float* rstd, const void* gamma, void* dx, int64_t lddx, void* dgamma, void* dbeta,
                        void* workspace, size_t workspace_bytes, int64_t N, int64_t H, norm_dtype x_dtype,
                        norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("ln_backward");
  return backward_common(normk::KIND_LN, dy, lddy, x, ldx, mean, rstd, gamma, dx, lddx, dgamma, dbeta, workspace,
                         workspace_bytes, N, H, x_dtype, w_dtype, stream);
}

norm_status rms_backward(const void* dy, int64_t lddy, const void* x, int64_t ldx, const float* rstd,
                         const void* gamma, void* dx, int64_t lddx, void* dgamma, void* workspace,
                         size_t workspace_bytes, int64_t N, int64_t H, norm_dtype x_dtype, norm_dtype w_dtype,
                         norm_stream_t stream) {
  NvtxRange range("rms_backward");
  return backward_common(normk::KIND_RMS, dy, lddy, x, ldx, nullptr, rstd, gamma, dx, lddx, dgamma, nullptr,
                         workspace, workspace_bytes, N, H, x_dtype, w_dtype, stream);
}

norm_status ln_backward_from_output(const void* dy, int64_t lddy, const void* y, int64_t ldy, const float* rstd,
                                    const void* gamma, const void* beta, void* dx, int64_t lddx, void* dgamma,
                                    void* dbeta, void* workspace, size_t workspace_bytes, int64_t N, int64_t H,
                                    norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("ln_backward_from_output");
  return backward_common(normk::KIND_LN_Y, dy, lddy, y, ldy, nullptr, rstd, gamma, dx, lddx, dgamma, dbeta,
                         workspace, workspace_bytes, N, H, x_dtype, w_dtype, stream, nullptr, 0, nullptr, 0, beta);
}

norm_status rms_backward_from_output(const void* dy, int64_t lddy, const void* y, int64_t ldy, const float* rstd,
                                     const void* gamma, void* dx, int64_t lddx, void* dgamma, void* workspace,
                                     size_t workspace_bytes, int64_t N, int64_t H, norm_dtype x_dtype,
                                     norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("rms_backward_from_output");
  return backward_common(normk::KIND_RMS_Y, dy, lddy, y, ldy, nullptr, rstd, gamma, dx, lddx, dgamma, nullptr,
                         workspace, workspace_bytes, N, H, x_dtype, w_dtype, stream);
}

norm_status fused_add_rms_backward(const void* dy, int64_t lddy, const void* h, int64_t ldh, const float* rstd,
                                   const void* gamma, const void* dh_in, int64_t lddh_in, void* dx, int64_t lddx,
                                   void* dres, int64_t lddres, void* dgamma, void* workspace,
                                   size_t workspace_bytes, int64_t N, int64_t H, norm_dtype x_dtype,
                                   norm_dtype w_dtype, norm_stream_t stream) {
  NvtxRange range("fused_add_rms_backward");
  return backward_common(normk::KIND_FUSED, dy, lddy, h, ldh, nullptr, rstd, gamma, dx, lddx, dgamma, nullptr,
                         workspace, workspace_bytes, N, H, x_dtype, w_dtype, stream, dh_in, lddh_in, dres, lddres);
}

const char* norm_status_str(norm_status status) {
  switch (status) {
    case NORM_OK: return "NORM_OK";
    case NORM_ERR_INVALID_VALUE: return "NORM_ERR_INVALID_VALUE: bad size, stride, eps, null or overlapping pointer";
    case NORM_ERR_UNSUPPORTED: return "NORM_ERR_UNSUPPORTED: dtype combination not provided";
    case NORM_ERR_WORKSPACE: return "NORM_ERR_WORKSPACE: backward workspace missing, too small or misaligned";
    case NORM_ERR_CUDA: return "NORM_ERR_CUDA: a CUDA runtime call or kernel launch failed";
  }
  return "NORM_ERR_UNKNOWN";
}

int norm_abi_version(void) { return 10000; }

const char* norm_last_error(void) { return t_last_error; }

norm_status norm_set_kernel_path(int path) {
  if (path < normk::PATH_AUTO || path > normk::PATH_STAGED) return NORM_ERR_INVALID_VALUE;
  g_path.store(path, std::memory_order_relaxed);
  return NORM_OK;
}

norm_status norm_set_bwd_split_event(void* event) {
  g_split_event.store(event, std::memory_order_relaxed);
  return NORM_OK;
}

norm_status norm_selftest_bounded_wait(unsigned long long limit_ns, norm_stream_t stream) {
  if (limit_ns < 1000000ull || limit_ns > normk::kWaitLimitNs) return NORM_ERR_INVALID_VALUE;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return NORM_ERR_CUDA;
  (void)cudaGetLastError();
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev.err, limit_ns);
  return launch_result("self-test launch", cudaGetLastError());
}

norm_status norm_device_errors(int device, unsigned int* flags, int clear) {
  if (flags == nullptr) return NORM_ERR_INVALID_VALUE;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return NORM_ERR_CUDA;
  if (device != cur && cudaSetDevice(device) != cudaSuccess) return NORM_ERR_CUDA;
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_norm_device_errors, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_norm_device_errors, &zero, sizeof(zero));
  }
  if (device != cur) cudaSetDevice(cur);
  if (e != cudaSuccess) return NORM_ERR_CUDA;
  *flags = v;
  return NORM_OK;
}

}  // extern "C"
