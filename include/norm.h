/*
 * norm.h -- C ABI of libnorm: row-wise LayerNorm and RMSNorm on one GB300 GPU
 * (sm_103a): forward, fused residual-add + RMSNorm forward, and the training
 * backward with gamma/beta gradients.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  A "row tensor" is N rows of H elements, row-major, the last
 *   (normalised) dimension contiguous, consecutive rows `ld` ELEMENTS apart
 *   (ld >= H).  A (B, T, H) tensor is passed as N = B*T rows.  gamma, beta,
 *   dgamma and dbeta have shape (H,) and are indexed by column only.  mean and
 *   rstd have shape (N,), fp32.
 * Memory.  Every pointer is CUDA device memory owned by the caller (any
 *   allocator, e.g. PyTorch's).  The library never allocates, frees or keeps a
 *   pointer after the call returns.  Its only device memory is module-scope:
 *   one error word per device (norm_device_errors) and the fixed workspace of
 *   ln_backward_static_workspace.
 * Streams.  Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and runs asynchronously; the call returns once the work is
 *   enqueued.  Outputs are valid after the stream reaches that point.
 * Dtypes.  `x_dtype` types the row tensors (x, residual, y, h_out, dy, dx);
 *   `w_dtype` types gamma, beta, dgamma, dbeta and must equal x_dtype or be
 *   NORM_F32.  All statistics and arithmetic are fp32; stored values are
 *   rounded to nearest, ties to even (an fp16 value past 65504 rounds to
 *   infinity).
 * eps.  Added INSIDE the square root: rstd = 1/sqrt(var + eps).  eps must be
 *   finite and > 0.
 * Alignment.  Rows whose pointers and strides are 16-byte aligned take the
 *   128-bit vector path; half-precision rows that are 32-byte aligned with H
 *   a multiple of 16 take the faster 256-bit paths; anything else is still
 *   correct (scalar path).
 * Errors.  Arguments are validated on the host before anything is enqueued;
 *   an invalid call returns an error and enqueues nothing.  A failed launch
 *   returns NORM_ERR_CUDA.  No entry point aborts, throws or prints.
 * Threads.  Every entry point is thread-safe.  The host-side library state
 *   is a per-device cache of device attributes (filled once, under a lock),
 *   the kernel-family override of norm_set_kernel_path and the timing event
 *   of norm_set_bwd_split_event (one atomic value each for the whole
 *   process).
 *
 * Sources: "Skill: Write a Triton LayerNorm Kernel", "Skill: Write CUDA
 * LayerNorm Kernel", "Skill: Write a Triton Fused Add+RMSNorm Kernel" and the
 * Fast-LLM pull request "Rewrite Triton normalization backward kernel_1
 * (#499)".  Each declaration names the section it implements.
 */
#ifndef NORM_H_
#define NORM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* norm_stream_t; /* same type as cudaStream_t */

typedef enum {
  NORM_OK = 0,
  NORM_ERR_INVALID_VALUE = 1, /* bad size, stride, eps, null or overlapping pointer */
  NORM_ERR_UNSUPPORTED = 2,   /* dtype combination not provided */
  NORM_ERR_WORKSPACE = 3,     /* backward workspace missing, too small or misaligned */
  NORM_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} norm_status;

/* fp32, bfloat16 and IEEE binary16 ("Skill: Write a Triton LayerNorm Kernel",
 * Inputs the agent should gather first, item 3: fp16, bf16 or fp32 inputs,
 * statistics accumulated in fp32). */
typedef enum { NORM_F32 = 0, NORM_BF16 = 1, NORM_F16 = 2 } norm_dtype;

/*
 * LayerNorm forward.  "Skill: Write a Triton LayerNorm Kernel", Required
 * reasoning process steps 1-10; "Skill: Write CUDA LayerNorm Kernel", steps
 * 1-7 (Welford statistics with the parallel merge, eps inside rsqrt):
 *   mean = sum_j x_j / H,  var = sum_j (x_j - mean)^2 / H  (biased),
 *   rstd = 1/sqrt(var + eps),  y_j = (x_j - mean) * rstd * gamma_j + beta_j.
 * x     [N x ldx]  input rows.
 * gamma [H] or NULL (= all ones);  beta [H] or NULL (= all zeros).
 * y     [N x ldy]  output rows.  May be exactly x (same pointer and stride) for
 *                  an in-place call; any other overlap with x is rejected.
 * mean, rstd [N] fp32 or NULL: the statistics saved for the backward.
 * N >= 0, H >= 1.  N == 0 enqueues nothing, and then every row and statistics
 * pointer may be NULL.
 */
norm_status ln_forward(const void* x, int64_t ldx, const void* gamma, const void* beta,
                       void* y, int64_t ldy, float* mean, float* rstd,
                       int64_t N, int64_t H, float eps,
                       norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * RMSNorm forward.  "Skill: Write CUDA LayerNorm Kernel", Kernel design rules
 * (RMSNorm); "Skill: Write a Triton LayerNorm Kernel", step 5:
 *   rstd = 1/sqrt(sum_j x_j^2 / H + eps),  y_j = x_j * rstd * gamma_j.
 * No mean subtraction and no beta.  Arguments as in ln_forward; rstd may be
 * NULL.
 */
norm_status rms_forward(const void* x, int64_t ldx, const void* gamma,
                        void* y, int64_t ldy, float* rstd,
                        int64_t N, int64_t H, float eps,
                        norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * Fused residual add + RMSNorm forward.  "Skill: Write a Triton Fused
 * Add+RMSNorm Kernel", Required reasoning process steps 1-9:
 *   h = x + residual formed in fp32;  h_out = h rounded to x_dtype;
 *   rstd = 1/sqrt(sum_j h_j^2 / H + eps);  y_j = h_j * rstd * gamma_j, with y
 *   computed from the fp32 h, not from the rounded h_out.
 * x [N x ldx], residual [N x ldr]: inputs.
 * h_out [N x ldh]: the summed residual stream.  It may be exactly x or exactly
 *   residual (same pointer and stride: in-place update); any other overlap is
 *   rejected.
 * y [N x ldy]: must not overlap x, residual or h_out.
 * rstd [N] fp32 or NULL (saved for training).
 */
norm_status fused_add_rms_forward(const void* x, int64_t ldx, const void* residual, int64_t ldr,
                                  const void* gamma, void* y, int64_t ldy,
                                  void* h_out, int64_t ldh, float* rstd,
                                  int64_t N, int64_t H, float eps,
                                  norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * Bytes of device workspace the backward needs for a row width H on CUDA
 * device `device`: the bounded fp32 partial buffer for dgamma/dbeta of
 * "Rewrite Triton normalization backward kernel_1 (#499)", Summary item 2
 * (a fixed number of partial rows tied to the SM count, independent of N).
 * Returns 0 if H < 1 or the device cannot be queried.
 */
size_t norm_bwd_workspace_bytes(int64_t H, int device);

/*
 * LayerNorm backward.  "Skill: Write CUDA LayerNorm Kernel", step 8, with
 * g_j = dy_j * gamma_j and x_hat_j = (x_j - mean) * rstd:
 *   dx_j     = rstd/H * (H*g_j - sum(g) - x_hat_j * sum(g * x_hat)),
 *   dgamma_j = sum over all N rows of dy_j * x_hat_j,
 *   dbeta_j  = sum over all N rows of dy_j.
 * Rows are grid-strided over a CTA count tied to the SM count; each CTA folds
 * its rows into one fp32 partial row in `workspace`, and a second kernel sums
 * the partials and casts once to w_dtype ("Rewrite Triton normalization
 * backward kernel_1 (#499)", Summary items 1-2).
 * dy [N x lddy], x [N x ldx]: inputs.  mean, rstd [N] fp32: the forward's
 *   saved statistics (required).
 * gamma [H] or NULL (= ones).
 * dx [N x lddx]: output; may be exactly dy (in place); must not overlap x.
 * dgamma, dbeta [H] in w_dtype, or NULL to skip that gradient.  They are
 *   overwritten, not accumulated into.  With N == 0 they are set to zero, the
 *   row and statistics pointers may be NULL and no workspace is needed.
 * workspace: device memory of at least norm_bwd_workspace_bytes(H, device)
 *   bytes, 16-byte aligned; needed only when dgamma or dbeta is non-NULL.  Its
 *   contents need no initialisation and are undefined afterwards.  Calls that
 *   share one workspace must be ordered on the GPU (e.g. one stream).
 */
norm_status ln_backward(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                        const float* mean, const float* rstd, const void* gamma,
                        void* dx, int64_t lddx, void* dgamma, void* dbeta,
                        void* workspace, size_t workspace_bytes,
                        int64_t N, int64_t H,
                        norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * RMSNorm backward (derived from the RMSNorm forward; no page prints it):
 * with g_j = dy_j * gamma_j and x_hat_j = x_j * rstd,
 *   dx_j     = rstd * (g_j - x_hat_j * sum(g * x_hat) / H),
 *   dgamma_j = sum over all N rows of dy_j * x_hat_j.
 * Arguments as in ln_backward, without mean and dbeta.
 */
norm_status rms_backward(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                         const float* rstd, const void* gamma,
                         void* dx, int64_t lddx, void* dgamma,
                         void* workspace, size_t workspace_bytes,
                         int64_t N, int64_t H,
                         norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * ln_backward for callers that cannot allocate device memory when they call
 * it -- for example a plugin inside a framework that owns all device memory
 * and gives plugins no allocator, or latency-critical code that must not pay
 * for cudaMalloc mid-step.  (The pages have no counterpart: this is an
 * interface convenience, not part of the method.)
 *
 * Same arguments and results as ln_backward, without the workspace: the
 * dgamma/dbeta partial rows go to a scratch array of
 * NORM_STATIC_WORKSPACE_BYTES (64 MiB) compiled into the library, one copy per
 * GPU that loads it, held until the process exits.  Nothing is allocated.
 * - Widths whose partial rows need more than that (when dgamma or dbeta is
 *   requested: norm_bwd_workspace_bytes(H, device) > the limit; H up to about
 *   27000 on a 152-SM GPU), or that the device cannot be asked to size, are
 *   refused with NORM_ERR_WORKSPACE.
 * - Every call looks up the current device's copy of the array
 *   (cudaGetSymbolAddress, a host-side lookup).  Under lazy module loading
 *   (CUDA's default) the 64 MiB are reserved when the library's device code
 *   is first used on a device, which may be this call: make one set-up call
 *   (N == 0 is enough) before any stream capture and before a framework takes
 *   the device's memory.  If that reservation fails the call returns
 *   NORM_ERR_CUDA and norm_last_error() names the failed step.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents; no part of it needs clearing, as each call writes every partial
 *   value before reading it.  Calls whose GPU work overlaps (other streams,
 *   other host threads) race on the array and must be ordered, e.g. on one
 *   stream.
 */
#define NORM_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)
norm_status ln_backward_static_workspace(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                                         const float* mean, const float* rstd, const void* gamma,
                                         void* dx, int64_t lddx, void* dgamma, void* dbeta,
                                         int64_t N, int64_t H,
                                         norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * LayerNorm backward from the forward's saved output instead of x.
 * "Rewrite Triton normalization backward kernel_1 (#499)", Benchmark harness:
 * the backward reads the output the forward saved.  x_hat is recovered as
 * (y - beta) / gamma and the formulas of ln_backward run on it with the saved
 * rstd ("Skill: Write CUDA LayerNorm Kernel", Required reasoning process
 * step 8).  x and mean are not needed.
 * y [N x ldy]: the forward's output (ln_forward's y, same gamma and beta).
 * rstd [N] fp32: the forward's saved rstd.  gamma, beta [H] or NULL (ones,
 *   zeros).  A column whose gamma is 0 holds no trace of x_hat: its dx and
 *   dgamma come out non-finite (IEEE division by zero); nothing is checked.
 * dx, dgamma, dbeta, workspace: as ln_backward; dx may be exactly dy and must
 *   not overlap y.  x_hat recovered from a rounded y carries that rounding
 *   (2^-9 relative for bf16, 2^-11 for fp16) into dx and dgamma.
 */
norm_status ln_backward_from_output(const void* dy, int64_t lddy, const void* y, int64_t ldy, const float* rstd,
                                    const void* gamma, const void* beta, void* dx, int64_t lddx, void* dgamma,
                                    void* dbeta, void* workspace, size_t workspace_bytes, int64_t N, int64_t H,
                                    norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/*
 * RMSNorm backward from the saved output: x_hat = y / gamma, then the
 * formulas of rms_backward with the saved rstd.  Arguments as
 * ln_backward_from_output without beta/dbeta.
 */
norm_status rms_backward_from_output(const void* dy, int64_t lddy, const void* y, int64_t ldy, const float* rstd,
                                     const void* gamma, void* dx, int64_t lddx, void* dgamma, void* workspace,
                                     size_t workspace_bytes, int64_t N, int64_t H, norm_dtype x_dtype,
                                     norm_dtype w_dtype, norm_stream_t stream);

/*
 * Fused residual add + RMSNorm backward.  "Skill: Write a Triton Fused
 * Add+RMSNorm Kernel", Required reasoning process steps 9-10: the backward
 * reads the stored sum h and rstd; the RMSNorm gradient with respect to h,
 *   dL/dh_j = rstd * (g_j - h_hat_j * sum(g * h_hat) / H) + dh_in_j,
 *   with g = dy * gamma and h_hat = h * rstd,
 * is the gradient of both inputs (dh/dx = dh/dresidual = 1).  dh_in is the
 * gradient arriving through the stored h itself (the residual stream's later
 * consumers), added in the same pass, or NULL.  dgamma_j = sum over rows of
 * dy_j * h_hat_j.
 * dy [N x lddy], h [N x ldh] (the forward's h_out), rstd [N] fp32, gamma [H]
 *   or NULL.
 * dx [N x lddx]: dL/dh for x.  May be exactly dy or dh_in (in place); must
 *   not overlap h.
 * dres [N x lddres]: dL/dh again, for the residual input; NULL to write dx
 *   only; exactly dx when x and residual were one tensor, which then
 *   receives the sum 2 * dL/dh.
 * dgamma [H] or NULL; workspace as in rms_backward.
 */
norm_status fused_add_rms_backward(const void* dy, int64_t lddy, const void* h, int64_t ldh,
                                   const float* rstd, const void* gamma,
                                   const void* dh_in, int64_t lddh_in,
                                   void* dx, int64_t lddx, void* dres, int64_t lddres, void* dgamma,
                                   void* workspace, size_t workspace_bytes, int64_t N, int64_t H,
                                   norm_dtype x_dtype, norm_dtype w_dtype, norm_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char* norm_status_str(norm_status status);

/* Version of this ABI: major*10000 + minor*100 + patch. */
int norm_abi_version(void);

/* The CUDA call and error behind the calling thread's most recent
 * NORM_ERR_CUDA ("" if none yet).  Static per-thread storage, never NULL. */
const char* norm_last_error(void);

/*
 * Device-side error bits raised since the last clear, for CUDA device
 * `device`.  Kernels never trap: every wait inside them is bounded (2 s), and a
 * wait that runs out sets NORM_DEVICE_ERR_WAIT_TIMEOUT here and abandons the
 * call's remaining work.  The read is synchronous; call it after the streams
 * that ran the kernels have been synchronised.  clear != 0 resets the bits.
 */
#define NORM_DEVICE_ERR_WAIT_TIMEOUT 1u
#define NORM_DEVICE_ERR_BAD_COPY 2u /* a bulk copy failed its bounds check and was skipped */
norm_status norm_device_errors(int device, unsigned int* flags, int clear);

/*
 * Self-test of the failure path above: enqueue one small kernel that waits,
 * with the given limit, on a barrier nothing ever signals.  The wait gives up
 * after limit_ns (1 ms .. 2 s, else NORM_ERR_INVALID_VALUE), sets
 * NORM_DEVICE_ERR_WAIT_TIMEOUT on the current device and returns; the CUDA
 * context stays usable.  No data is touched.
 */
norm_status norm_selftest_bounded_wait(unsigned long long limit_ns, norm_stream_t stream);

/*
 * Testing and tuning: the kernel-family policy for every later call in the
 * process.  0 = automatic (the default), 1 = register rows (else the strided
 * loop), 2 = strided loop only, 3 = bulk-copy pipeline first.  A family is
 * used only where the call meets its requirements (alignment, row width);
 * every family computes the same results within rounding.
 */
norm_status norm_set_kernel_path(int path);

/*
 * Timing: split every later backward call in the process into its two
 * kernels.  The bounded partial reduction of "Rewrite Triton normalization
 * backward kernel_1 (#499)" runs the backward as a main kernel (dx and the
 * per-CTA dgamma/dbeta partial rows) and a second kernel that sums the
 * partials; its Benchmark harness asks for the device time of each.  When
 * `event` (a cudaEvent_t, or NULL to turn the split off) is set, each backward
 * records it on its stream after the main kernel and launches the reduction
 * as an ordinary dependent launch instead of a programmatic one, so events
 * recorded before and after the call bracket the two kernels.  Results are
 * unchanged.  One value for the whole process; for benchmarks, not for
 * concurrent production calls.
 */
norm_status norm_set_bwd_split_event(void* event);

#ifdef __cplusplus
}
#endif

#endif /* NORM_H_ */
