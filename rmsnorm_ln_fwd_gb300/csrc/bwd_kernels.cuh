// Backward kernel templates and their launch logic, instantiated per row
// dtype by norm_bwd_f32.cu, norm_bwd_bf16.cu and norm_bwd_f16.cu.
//
// Backward kernels: LayerNorm and RMSNorm grad_input plus the gamma/beta
// gradients through a bounded fp32 partial reduction; the same from the
// forward's saved output (x_hat = (y - beta)/gamma); and the fused add's
// backward from the stored sum h (KIND_FUSED: RMSNorm math on h, the gradient
// arriving through h added, written to both inputs' gradients).
//
// Math ("Skill: Write CUDA LayerNorm Kernel", Required reasoning process
// step 8; the RMSNorm form is derived from its forward):
//   g = dy * gamma,  x_hat = (x - mean) * rstd   (RMSNorm: x * rstd)
//   LayerNorm: dx = rstd * (g - sum(g)/H - x_hat * sum(g*x_hat)/H)
//   RMSNorm:   dx = rstd * (g - x_hat * sum(g*x_hat)/H)
//   dgamma = sum over rows of dy * x_hat,  dbeta = sum over rows of dy.
// The saved fp32 mean can sit half an fp32 ulp away from the true mean; for
// rows with a large common offset that is a visible constant shift of x_hat.
// Because mean(x_hat) = 0 exactly, the kernel also sums x_hat and subtracts
// its row mean, which removes that shift (one extra value in the same
// reduction).
//
// Structure ("Rewrite Triton normalization backward kernel_1 (#499)",
// Summary items 1-2): a fixed grid of at most P = 2 x SM-count CTAs
// grid-strides the rows.  Each thread owns fixed columns, so its dgamma/dbeta
// accumulators stay in fp32 (registers or shared memory) across all rows it
// visits; at the end each CTA folds its row groups into ONE partial row (a
// cluster of CTAs sharing wide rows writes one partial row between them).  The
// partial buffer is therefore at most P x H, independent of N, and a second
// small kernel sums it column-wise, casting to the parameter dtype once at the
// store.

#pragma once

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "staged.cuh"

namespace normk {

// Register-row backward.  Persistent row groups walk rows row, row + stride,
// ...; the next row's x, dy and saved statistics are loaded while the current
// row computes.  Each thread owns fixed column vectors, so its dgamma/dbeta
// accumulators stay in fp32 across all its rows: in registers (ACC_SMEM =
// false), or, when one CTA covers a whole row (so every column has exactly one
// owner thread), in shared memory, updated by plain read-modify-write, which
// frees the registers for wide rows.  Elementwise math uses f32x2.
//
// CL > 1: a thread-block cluster of CL CTAs shares each row, CTA rank r
// taking columns [r*H/CL, (r+1)*H/CL) with its accumulators in registers; the
// CTAs' row sums meet through distributed shared memory
// (cluster_group_sum_async, one exchange a row), and cluster c writes partial
// row c.  Used for rows too wide for one CTA's registers, and for fp32 rows
// whose one-CTA kernels spill (the host policy in launch_bwd_typed).
template <typename D>
__device__ __forceinline__ BwdArgs part_row_view(BwdArgs a, int rank, int parts) {
  using T = typename D::T;
  const int64_t c0 = (int64_t)rank * (a.H / parts);
  const size_t wes = a.w_f32 ? 4 : sizeof(T);
  a.x = reinterpret_cast<const T*>(a.x) + c0;
  a.dy = reinterpret_cast<const T*>(a.dy) + c0;
  a.dx = reinterpret_cast<T*>(a.dx) + c0;
  if (a.dh_in) a.dh_in = reinterpret_cast<const T*>(a.dh_in) + c0;
  if (a.dres) a.dres = reinterpret_cast<T*>(a.dres) + c0;
  if (a.gamma) a.gamma = reinterpret_cast<const unsigned char*>(a.gamma) + c0 * wes;
  if (a.beta) a.beta = reinterpret_cast<const unsigned char*>(a.beta) + c0 * wes;
  if (a.ws) a.ws += c0;
  a.H /= parts;
  return a;
}

// The body of bwd_rows_kernel: `a` describes this CTA's columns, `h_full`
// is the row length the statistics divide by, `crank` the CTA's rank in its
// cluster (0 without clusters).
template <int KIND, typename D, int VPT, int MAXT, bool ACC_SMEM, int CL>
__device__ __forceinline__ void bwd_rows_body(const BwdArgs& a, int h_full, int crank) {
  static_assert(!(CL > 1 && ACC_SMEM), "cluster rows keep their accumulators in registers");
  constexpr bool CLUSTER = CL > 1;
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr int VP = VEC / 2;
  constexpr bool LN = kind_is_ln(KIND);
  constexpr bool FROM_Y = kind_from_y(KIND);   // x is the forward's output y
  constexpr bool RECENTER = KIND == KIND_LN;   // see the recentring note above
  constexpr int NS = LN ? (RECENTER ? 3 : 2) : 1;  // values per row reduction
  extern __shared__ __align__(16) float sh_dyn[];
  const int tpr = a.tpr;
  const int rpc = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;  // this CTA's columns (H/CL of the row in a cluster)
  const int hv = H / VEC;
  const float inv_h = 1.f / (float)h_full;
  const bool w_f32 = a.w_f32 != 0;
  float* sh = sh_dyn + slot * (2 * nw * NS);
  const int bar_id = 1 + slot;
  // Partial rows: one a CTA, or one a cluster.
  const int prow = (int)blockIdx.x / CL;
  const int nprow = (int)gridDim.x / CL;
  const int64_t stride = (int64_t)nprow * rpc;
  __shared__ float xch[2][CL * 4];  // cluster exchange of the row sums ([rank][value]), by parity
  __shared__ uint64_t xbar[2];      // their mbarriers, by parity
  __shared__ int xabort;            // a bounded wait ran out: later waits give up at once
  int nvec = 0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) nvec += (t + v * tpr < hv) ? 1 : 0;

  constexpr int VA = ACC_SMEM ? 1 : VPT;  // register accumulator vectors
  float2 acc_g[VA][VP], acc_b[VA][VP];
#pragma unroll
  for (int v = 0; v < VA; ++v)
#pragma unroll
    for (int p = 0; p < VP; ++p) acc_g[v][p] = acc_b[v][p] = splat2(0.f);
  // Half-precision LayerNorm with shared-memory accumulators and up to 640
  // threads: dbeta stays in registers (they fit there without spilling;
  // measured, the shared-memory pipe is what bounds this kernel: 8192x5120
  // bf16 66.4 -> 60.1 us).
  constexpr bool DB_REG = ACC_SMEM && KIND == KIND_LN && MAXT == 640 && VEC == 8;
  float2 acc_db[DB_REG ? VPT : 1][VP];
#pragma unroll
  for (int v = 0; v < (DB_REG ? VPT : 1); ++v)
#pragma unroll
    for (int p = 0; p < VP; ++p) acc_db[v][p] = splat2(0.f);
  constexpr bool FUSED = KIND == KIND_FUSED;
  constexpr int VH = FUSED ? VPT : 1;  // stream-gradient vectors (fused only)
  uint4 nx[VPT], nd[VPT];
  float nrs = 0.f, nmu = 0.f;
  auto fetch = [&](int64_t r) {
    const T* xrow = reinterpret_cast<const T*>(a.x) + r * a.ldx;
    const T* dyrow = reinterpret_cast<const T*>(a.dy) + r * a.lddy;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (t + v * tpr) * VEC;
      nx[v] = load_vec_or_zero<D>(xrow, c, H);
      nd[v] = load_vec_or_zero<D>(dyrow, c, H);
    }
    nrs = a.rstd[r];
    if (LN && !FROM_Y) nmu = a.mean[r];
  };

  int parity = 0;
  int64_t row = (int64_t)prow * rpc + slot;
  if (row < a.N) fetch(row);  // first row in flight while gamma is staged

  const int Hp = a.Hp;
  // Shared memory: group scratch | fp32 gamma (thread-interleaved, shared by
  // the row slots) | from the output: 1/gamma and (LayerNorm) beta, likewise |
  // accumulators (ACC_SMEM, thread-interleaved: dgamma then dbeta) or the fold
  // buffer of the row slots.
  constexpr int NPY = FROM_Y ? (LN ? 2 : 1) : 0;
  const int off_g = ((rpc * 2 * nw * NS) + 3) & ~3;
  const int slots = VPT * VEC * tpr;  // floats of one thread-interleaved array
  float4* gs = reinterpret_cast<float4*>(sh_dyn + off_g);
  float4* gis = gs + slots / 4;
  float4* bes = gis + slots / 4;
  float* sh_acc = sh_dyn + off_g + (1 + NPY) * slots;
  float4* sacc_g = reinterpret_cast<float4*>(sh_acc);
  float4* sacc_b = sacc_g + slots / 4;
  if (slot == 0) {
    stage_params<D, VPT>(gs, a.gamma, w_f32, 1.f, t, tpr, hv);
    if constexpr (FROM_Y) {
      stage_inv_params<D, VPT>(gis, a.gamma, w_f32, t, tpr, hv);
      if (LN) stage_params<D, VPT>(bes, a.beta, w_f32, 0.f, t, tpr, hv);
    }
  }
  if constexpr (ACC_SMEM) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      float2 z[VP];
#pragma unroll
      for (int p = 0; p < VP; ++p) z[p] = splat2(0.f);
      write_pairs<VEC>(sacc_g, v, t, tpr, z);
      if (LN) write_pairs<VEC>(sacc_b, v, t, tpr, z);
    }
  }
  __syncthreads();
  unsigned it = 0;  // rows this CTA has exchanged (cluster rows)
  if constexpr (CLUSTER) {
    if (threadIdx.x == 0) {
      mbar_init(&xbar[0], 1);
      mbar_init(&xbar[1], 1);
      xabort = 0;
      fence_barrier_init();
    }
    cluster_sync_all();  // every CTA's mbarriers exist before any CTA sends to them
  }


  for (; row < a.N; row += stride) {
    const float r = nrs;
    const float2 r2 = splat2(r);
    float2 xh[VPT][VP];
    uint4 dcur[VPT], hcur[VH];
    if constexpr (FROM_Y) {
      // x_hat = (y - beta) / gamma, from the forward's output.
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        float2 yv[VP], gi[VP], be[VP];
        unpack2<D>(nx[v], yv);
        read_pairs<VEC>(gis, v, t, tpr, gi);
        if (LN) read_pairs<VEC>(bes, v, t, tpr, be);
#pragma unroll
        for (int p = 0; p < VP; ++p) xh[v][p] = mul2(LN ? sub2(yv[p], be[p]) : yv[p], gi[p]);
        dcur[v] = nd[v];
      }
    } else {
      // x_hat = x*rstd - mean*rstd: the rounding of mean*rstd shifts the whole
      // row by one constant, which the recentring below removes.
      const float2 b2 = splat2(LN ? -nmu * r : 0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        float2 xv[VP];
        unpack2<D>(nx[v], xv);
#pragma unroll
        for (int p = 0; p < VP; ++p) xh[v][p] = LN ? fma2(xv[p], r2, b2) : mul2(xv[p], r2);
        dcur[v] = nd[v];
      }
    }
    if (row + stride < a.N) fetch(row + stride);
    if constexpr (FUSED) {
      // The gradient through h is only added in pass 2: load it for this row
      // now, in flight over the row reduction, rather than a row ahead.
      if (a.dh_in) {
        const T* hrow = reinterpret_cast<const T*>(a.dh_in) + row * a.lddh;
#pragma unroll
        for (int v = 0; v < VH; ++v) hcur[v] = load_vec_or_zero<D>(hrow, (t + v * tpr) * VEC, H);
      }
    }

    // Pass 1: sum(g), sum(g*x_hat) and (LayerNorm) sum(x_hat), g = dy*gamma.
    float2 sg = splat2(0.f), sgx = splat2(0.f), sx = splat2(0.f);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (v < nvec) {
        float2 d[VP], gm[VP];
        unpack2<D>(dcur[v], d);
        read_pairs<VEC>(gs, v, t, tpr, gm);
#pragma unroll
        for (int p = 0; p < VP; ++p) {
          const float2 g = mul2(d[p], gm[p]);
          sgx = fma2(g, xh[v][p], sgx);
          if (LN) sg = add2(sg, g);
          if (RECENTER) sx = add2(sx, xh[v][p]);
        }
      }
    }
    float S[NS];
    if (LN) {
      S[0] = sg.x + sg.y;
      S[1] = sgx.x + sgx.y;
      if constexpr (RECENTER) S[NS - 1] = sx.x + sx.y;
    } else {
      S[0] = sgx.x + sgx.y;
    }
    // Cluster parts have at most 16 warps: a compile-time butterfly for the
    // one-value sums (measured RMSNorm 2048x16384 bf16 43.3 -> 42.1 us,
    // 1024x32768 47.1 -> 45.5; the LayerNorm sums gain nothing).
    group_sum<NS, (CL > 1 && NS == 1) ? 16 : 0>(S, sh, nw, wig, lane, bar_id, parity);
    if constexpr (CLUSTER) {  // identical sums in every part
      cluster_group_sum_async<NS, CL>(S, xch[parity], &xbar[parity], (it >> 1) & 1u, crank, a.err, &xabort);
      ++it;
    }
    // LayerNorm: mean(x_hat) is 0 exactly; its computed value s0 is the shift
    // left by the saved mean's rounding, removed from x_hat here.  (From the
    // output there is no saved mean: x_hat is taken as recovered.)
    const float s0 = RECENTER ? S[NS - 1] * inv_h : 0.f;
    const float c1 = LN ? S[0] * inv_h : 0.f;
    const float c2 = LN ? fmaf(-s0, S[0], S[1]) * inv_h : S[0] * inv_h;
    const float2 s02 = splat2(s0), nc22 = splat2(-c2);
    const float2 na2 = splat2(-c2 * r), nb2 = splat2(-c1 * r);

    // Pass 2: dx = rstd * (g - c1 - x_hat * c2) and the accumulators
    // (LayerNorm as (-c2*rstd)*x_hat + (g*rstd - c1*rstd): two f32x2
    // instructions a pair).
    T* dxrow = reinterpret_cast<T*>(a.dx) + row * a.lddx;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (v < nvec) {
        const int col = (t + v * tpr) * VEC;
        float2 d[VP], gm[VP], out[VP];
        unpack2<D>(dcur[v], d);
        read_pairs<VEC>(gs, v, t, tpr, gm);
        float2 ag[VP], ab[VP];
        if constexpr (ACC_SMEM) {
          read_pairs<VEC>(sacc_g, v, t, tpr, ag);
          if constexpr (DB_REG) {
#pragma unroll
            for (int p = 0; p < VP; ++p) ab[p] = acc_db[v][p];
          } else if (LN) {
            read_pairs<VEC>(sacc_b, v, t, tpr, ab);
          }
        } else {
#pragma unroll
          for (int p = 0; p < VP; ++p) {
            ag[p] = acc_g[ACC_SMEM ? 0 : v][p];
            ab[p] = acc_b[ACC_SMEM ? 0 : v][p];
          }
        }
#pragma unroll
        for (int p = 0; p < VP; ++p) {
          const float2 xc = RECENTER ? sub2(xh[v][p], s02) : xh[v][p];
          const float2 g = mul2(d[p], gm[p]);
          if constexpr (LN) out[p] = fma2(xc, na2, fma2(g, r2, nb2));
          else out[p] = mul2(fma2(xc, nc22, g), r2);
          ag[p] = fma2(d[p], xc, ag[p]);
          if (LN) ab[p] = add2(ab[p], d[p]);
        }
        if constexpr (ACC_SMEM) {
          write_pairs<VEC>(sacc_g, v, t, tpr, ag);
          if constexpr (DB_REG) {
#pragma unroll
            for (int p = 0; p < VP; ++p) acc_db[v][p] = ab[p];
          } else if (LN) {
            write_pairs<VEC>(sacc_b, v, t, tpr, ab);
          }
        } else {
#pragma unroll
          for (int p = 0; p < VP; ++p) {
            acc_g[ACC_SMEM ? 0 : v][p] = ag[p];
            acc_b[ACC_SMEM ? 0 : v][p] = ab[p];
          }
        }
        if constexpr (FUSED) {
          // dL/dh = RMSNorm gradient + the gradient through h, for x and residual
          if (a.dh_in) {
            float2 e[VP];
            unpack2<D>(hcur[v], e);
#pragma unroll
            for (int p = 0; p < VP; ++p) out[p] = add2(out[p], e[p]);
          }
          if (a.dx_twice) {
#pragma unroll
            for (int p = 0; p < VP; ++p) out[p] = add2(out[p], out[p]);
          }
        }
        const uint4 packed = pack2<D>(out);
        st_vec(dxrow + col, packed);
        if constexpr (FUSED) {
          if (a.dres) st_vec(reinterpret_cast<T*>(a.dres) + row * a.lddres + col, packed);
        }
      }
    }
    parity ^= 1;
  }

  if constexpr (CLUSTER) cluster_sync_all();  // no CTA leaves while its partner may still write to it
  if (a.ws == nullptr) return;
  // Fold the CTA's row groups into partial row prow.
  float* pg = a.ws + (size_t)prow * Hp;
  float* pb = a.ws + ((size_t)nprow + prow) * Hp;
  if constexpr (ACC_SMEM) {
    // Each thread owns its accumulator slots: copy them straight out.
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (v < nvec) {
        const int col = (t + v * tpr) * VEC;
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
          *reinterpret_cast<float4*>(pg + col + 4 * q) = sacc_g[(v * (VEC / 4) + q) * tpr + t];
          if constexpr (DB_REG) {
            *reinterpret_cast<float4*>(pb + col + 4 * q) =
                make_float4(acc_db[v][2 * q].x, acc_db[v][2 * q].y, acc_db[v][2 * q + 1].x, acc_db[v][2 * q + 1].y);
          } else if (LN) {
            *reinterpret_cast<float4*>(pb + col + 4 * q) = sacc_b[(v * (VEC / 4) + q) * tpr + t];
          }
        }
      }
    }
    return;
  }
  if (rpc == 1) {
#pragma unroll
    for (int v = 0; v < VA; ++v) {
      if (v < nvec) {
        const int col = (t + v * tpr) * VEC;
#pragma unroll
        for (int q = 0; q < VP / 2; ++q) {
          *reinterpret_cast<float4*>(pg + col + 4 * q) =
              make_float4(acc_g[v][2 * q].x, acc_g[v][2 * q].y, acc_g[v][2 * q + 1].x, acc_g[v][2 * q + 1].y);
          if (LN)
            *reinterpret_cast<float4*>(pb + col + 4 * q) =
                make_float4(acc_b[v][2 * q].x, acc_b[v][2 * q].y, acc_b[v][2 * q + 1].x, acc_b[v][2 * q + 1].y);
        }
      }
    }
    return;
  }
  float* red_g = sh_acc;  // fold buffer: [Hp] dgamma then [Hp] dbeta
  float* red_b = red_g + Hp;
  for (int s2 = 0; s2 < rpc; ++s2) {
    if (slot == s2) {
#pragma unroll
      for (int v = 0; v < VA; ++v) {
        if (v < nvec) {
          const int col = (t + v * tpr) * VEC;
#pragma unroll
          for (int p = 0; p < VP; ++p) {
            float2* dg2 = reinterpret_cast<float2*>(red_g + col) + p;
            float2* db2 = reinterpret_cast<float2*>(red_b + col) + p;
            *dg2 = s2 == 0 ? acc_g[v][p] : add2(*dg2, acc_g[v][p]);
            if (LN) *db2 = s2 == 0 ? acc_b[v][p] : add2(*db2, acc_b[v][p]);
          }
        }
      }
    }
    __syncthreads();
  }
  for (int k = threadIdx.x * 4; k < H; k += blockDim.x * 4) {
    *reinterpret_cast<float4*>(pg + k) = *reinterpret_cast<const float4*>(red_g + k);
    if (LN) *reinterpret_cast<float4*>(pb + k) = *reinterpret_cast<const float4*>(red_b + k);
  }
}

template <int KIND, typename D, int VPT, int MAXT, int MINB, bool ACC_SMEM, int CL = 1>
__global__ void __launch_bounds__(MAXT, MINB) bwd_rows_kernel(const BwdArgs a) {
  if constexpr (CL > 1) {
    const int crank = (int)cluster_ctarank();
    const BwdArgs part = part_row_view<D>(a, crank, CL);
    bwd_rows_body<KIND, D, VPT, MAXT, ACC_SMEM, CL>(part, a.H, crank);
  } else {
    bwd_rows_body<KIND, D, VPT, MAXT, ACC_SMEM, CL>(a, a.H, 0);
  }
}

// Span backward (LayerNorm from x, rows of at most 256 threads): thread t of
// a row group owns the contiguous columns [t*16, t*16 + 16) of every row it
// visits, so a row's x, dy and dx each move in one 32-byte access a thread
// (two in fp32), the next row's through incremented pointers, and every
// shared-memory access is a constant offset from the thread's own slot.
// gamma is staged as fp32 in shared memory, each thread's 16 values followed
// by 4 floats of padding, so the 16-byte accesses of any eight consecutive
// threads hit distinct banks; the dgamma/dbeta accumulators stay in registers.
// The arithmetic and its order are those of bwd_rows_body (x_hat recentred by
// its row mean).  It runs about a tenth fewer instructions an element than the
// interleaved register rows; measured faster for narrow LayerNorm rows only
// (8192x1024 bf16 main kernel 16.7 -> 14.3 us), so the launcher uses it there.
// Requires H % 16 == 0 and 32-byte aligned rows.
constexpr int kSpanCols = 16;
constexpr int kSpanSlot = kSpanCols + 4;  // floats a thread's slot occupies in the shared arrays

template <int KIND, typename D, int MAXT, int MINB, int PW = 0>
__global__ void __launch_bounds__(MAXT, MINB) bwd_span_kernel(const BwdArgs a) {
  using T = typename D::T;
  constexpr int E = kSpanCols;
  constexpr int NP = E / 2;                    // fp32 pairs of a span
  constexpr int NWD = E * (int)sizeof(T) / 4;  // 32-bit words of a span
  constexpr int NL = NWD / 8;                  // 32-byte accesses of a span
  constexpr int SW = kSpanSlot;
  constexpr bool LN = KIND == KIND_LN;
  constexpr int NS = LN ? 3 : 1;
  static_assert(KIND == KIND_LN || KIND == KIND_RMS, "from x only");
  extern __shared__ __align__(16) float sh_dyn[];
  const int tpr = a.tpr;
  const int rpc = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const bool active = t * E < H;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  float* red = sh_dyn + slot * (2 * nw * NS);
  float* gsh = sh_dyn + (((rpc * 2 * nw * NS) + 3) & ~3);  // [tpr][SW] fp32 gamma
  const float* my_g = gsh + t * SW;

  const int64_t stride = (int64_t)gridDim.x * rpc;
  int64_t row = (int64_t)blockIdx.x * rpc + slot;
  const size_t es = sizeof(T);
  // Byte pointers to this thread's span; the fetch pointers run a row ahead.
  const int64_t col0 = (int64_t)t * E;
  const char* fx = reinterpret_cast<const char*>(a.x) + (row * a.ldx + col0) * es;
  const char* fdy = reinterpret_cast<const char*>(a.dy) + (row * a.lddy + col0) * es;
  char* dxp = reinterpret_cast<char*>(a.dx) + (row * a.lddx + col0) * es;
  const int64_t sx_step = stride * a.ldx * (int64_t)es, sdy_step = stride * a.lddy * (int64_t)es,
                sdx_step = stride * a.lddx * (int64_t)es;
  uint32_t nx[NWD], nd[NWD];
  float nrs = 0.f, nmu = 0.f;
  auto fetch = [&](int64_t r) {
    if (active) {
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        ld_stream32(fx + 32 * l, *reinterpret_cast<uint32_t(*)[8]>(nx + 8 * l));
        ld_stream32(fdy + 32 * l, *reinterpret_cast<uint32_t(*)[8]>(nd + 8 * l));
      }
    }
    nrs = a.rstd[r];
    if (LN) nmu = a.mean[r];
    fx += sx_step;
    fdy += sdy_step;
  };
  if (row < a.N) fetch(row);  // first row in flight while gamma is staged

  if (slot == 0) {  // every row slot owns the same columns
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      float4 g4 = make_float4(1.f, 1.f, 1.f, 1.f);
      if (a.gamma != nullptr && active) {
        const int c = (int)col0 + 4 * q;
        if (w_f32) {
          g4 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.gamma) + c);
        } else {
          const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const T*>(a.gamma) + c);
          const uint32_t w[2] = {u.x, u.y};
          const float2 lo = word_pair<D>(w, 0), hi = word_pair<D>(w, 1);
          g4 = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
      }
      *reinterpret_cast<float4*>(gsh + t * SW + 4 * q) = g4;
    }
  }
  float2 accg[NP], accb[LN ? NP : 1];
#pragma unroll
  for (int p = 0; p < NP; ++p) accg[p] = splat2(0.f);
#pragma unroll
  for (int p = 0; p < (LN ? NP : 1); ++p) accb[p] = splat2(0.f);
  __syncthreads();

  int parity = 0;
  for (; row < a.N; row += stride) {
    const float r = nrs;
    const float2 r2 = splat2(r);
    const float2 b2 = splat2(LN ? -nmu * r : 0.f);
    float2 xh[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const float2 xv = word_pair<D>(nx, p);
      xh[p] = LN ? fma2(xv, r2, b2) : mul2(xv, r2);
    }
    uint32_t dcur[NWD];
#pragma unroll
    for (int w = 0; w < NWD; ++w) dcur[w] = nd[w];
    if (row + stride < a.N) fetch(row + stride);

    // Pass 1: sum(g), sum(g*x_hat) and (LayerNorm) sum(x_hat), g = dy*gamma.
    float2 sg = splat2(0.f), sgx = splat2(0.f), sxh = splat2(0.f);
    if (active) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 g4 = *reinterpret_cast<const float4*>(my_g + 4 * q);
        const float2 gm[2] = {make_float2(g4.x, g4.y), make_float2(g4.z, g4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int p = 2 * q + h;
          const float2 g = mul2(word_pair<D>(dcur, p), gm[h]);
          sgx = fma2(g, xh[p], sgx);
          if (LN) {
            sg = add2(sg, g);
            sxh = add2(sxh, xh[p]);
          }
        }
      }
    }
    float S[NS];
    if (LN) {
      S[0] = sg.x + sg.y;
      S[1] = sgx.x + sgx.y;
      S[NS - 1] = sxh.x + sxh.y;
    } else {
      S[0] = sgx.x + sgx.y;
    }
    group_sum<NS, PW>(S, red, nw, wig, lane, 1 + slot, parity);
    const float s0 = LN ? S[NS - 1] * inv_h : 0.f;
    const float c1 = LN ? S[0] * inv_h : 0.f;
    const float c2 = LN ? fmaf(-s0, S[0], S[1]) * inv_h : S[0] * inv_h;
    const float2 s02 = splat2(s0), c12 = splat2(c1), nc22 = splat2(-c2);

    // Pass 2: dx = rstd * (g - c1 - x_hat * c2) and the accumulators (in
    // this order: the shorter form of the wider kernels spills here).
    if (active) {
      uint32_t out[NWD];
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 g4 = *reinterpret_cast<const float4*>(my_g + 4 * q);
        const float2 gm[2] = {make_float2(g4.x, g4.y), make_float2(g4.z, g4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int p = 2 * q + h;
          const float2 d = word_pair<D>(dcur, p);
          const float2 g = mul2(d, gm[h]);
          const float2 xc = LN ? sub2(xh[p], s02) : xh[p];
          pair_word<D>(out, p, mul2(fma2(xc, nc22, LN ? sub2(g, c12) : g), r2));
          accg[p] = fma2(d, xc, accg[p]);
          if (LN) accb[p] = add2(accb[p], d);
        }
      }
#pragma unroll
      for (int l = 0; l < NL; ++l) st_vec32(dxp + 32 * l, *reinterpret_cast<const uint32_t(*)[8]>(out + 8 * l));
    }
    dxp += sdx_step;
    parity ^= 1;
  }

  if (a.ws == nullptr) return;
  const int Hp = a.Hp;
  float* pg = a.ws + (size_t)blockIdx.x * Hp;
  float* pb = a.ws + ((size_t)gridDim.x + blockIdx.x) * Hp;
  auto quad = [](const float2* v, int q) { return make_float4(v[2 * q].x, v[2 * q].y, v[2 * q + 1].x, v[2 * q + 1].y); };
  if (rpc == 1) {
    if (active) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        *reinterpret_cast<float4*>(pg + col0 + 4 * q) = quad(accg, q);
        if constexpr (LN) *reinterpret_cast<float4*>(pb + col0 + 4 * q) = quad(accb, q);
      }
    }
    return;
  }
  // Several row slots: fold them in slot order through a [2][tpr][SW] buffer
  // in the padded layout, then write the CTA's partial row.
  float* fg = gsh + tpr * SW + t * SW;
  float* fb = gsh + 2 * tpr * SW + t * SW;
  for (int s2 = 0; s2 < rpc; ++s2) {
    if (slot == s2 && active) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        float4 g4 = quad(accg, q);
        float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (LN) b4 = quad(accb, q);
        if (s2 > 0) {
          const float4 og = *reinterpret_cast<const float4*>(fg + 4 * q);
          g4 = make_float4(og.x + g4.x, og.y + g4.y, og.z + g4.z, og.w + g4.w);
          if constexpr (LN) {
            const float4 ob = *reinterpret_cast<const float4*>(fb + 4 * q);
            b4 = make_float4(ob.x + b4.x, ob.y + b4.y, ob.z + b4.z, ob.w + b4.w);
          }
        }
        *reinterpret_cast<float4*>(fg + 4 * q) = g4;
        if constexpr (LN) *reinterpret_cast<float4*>(fb + 4 * q) = b4;
      }
    }
    __syncthreads();
  }
  if (slot == 0 && active) {
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      *reinterpret_cast<float4*>(pg + col0 + 4 * q) = *reinterpret_cast<const float4*>(fg + 4 * q);
      if constexpr (LN) *reinterpret_cast<float4*>(pb + col0 + 4 * q) = *reinterpret_cast<const float4*>(fb + 4 * q);
    }
  }
}

// Span rows with the next rows in shared memory (half-precision LayerNorm
// and RMSNorm, from x or from the saved output, one row a CTA of 257..640
// threads): the column ownership and the arithmetic of bwd_span_kernel, but
// no registers hold a row in flight: one thread of the CTA bulk-copies the
// next rows of x (or y) and dy into row buffers in shared memory, completing
// on the buffer's mbarrier, and refills a buffer once the row reduction's
// barrier has passed (every thread has then read it).  That leaves room for
// both accumulators in registers at two CTAs an SM (at most 93 registers, no
// spills), where the span kernel with its register prefetch had to keep
// dgamma in shared memory.  From the output, x_hat = (y - beta)/gamma with
// 1/gamma and beta staged next to gamma in the thread's slot.  Measured:
// LayerNorm 8192x5120 bf16 59.5 -> 55.4 us (main kernel 56.6 -> 51.6), fp16
// 61.3 -> 55.7, 4096x10240 62.0 -> 60.3; RMSNorm 8192x5120 48.6 -> 47.3.
// Every wait is bounded; a wait that runs out sets the error word and stops
// new copies, and the issuing thread drains its copies before the CTA exits.

// Row buffers (rows in flight a CTA): RMSNorm, with less arithmetic a row,
// waits on memory more and gains from a third (measured 8192x5120 bf16 45.6 ->
// 43.0 us); LayerNorm does not (53.3 -> 54.5).
template <int KIND>
__host__ __device__ constexpr int spanb_bufs() { return KIND == KIND_RMS || KIND == KIND_RMS_Y ? 3 : 2; }

// Floats of a thread's parameter slot: gamma of its 16 columns, from the
// output also 1/gamma and (LayerNorm) beta, then 4 floats of padding (the
// 16-byte reads of eight consecutive threads then hit distinct banks: the slot
// stride is 4 mod 32 words for 20 and 36, 20 mod 32 for 52).
template <int KIND>
__host__ __device__ constexpr int spanb_slot() {
  return kind_from_y(KIND) ? (kind_is_ln(KIND) ? 3 : 2) * kSpanCols + 4 : kSpanSlot;
}

struct SpanBLayout {
  int bars, abort, red, gamma, bufs, buf_bytes, total;
};
__host__ __device__ inline SpanBLayout spanb_layout(int tpr, int H, int es, int NS, int NB, int slot) {
  SpanBLayout L;
  L.bars = 0;
  L.abort = 8 * NB;
  L.red = (L.abort + 4 + 15) & ~15;
  L.gamma = (L.red + 4 * 2 * (tpr / 32) * NS + 15) & ~15;
  L.bufs = (L.gamma + 4 * tpr * slot + 127) & ~127;
  L.buf_bytes = (H * es + 127) & ~127;
  L.total = L.bufs + 2 * NB * L.buf_bytes;  // [buffers][x, dy]
  return L;
}

template <int KIND, typename D, int MAXT, int MINB, int PW>
__global__ void __launch_bounds__(MAXT, MINB) bwd_spanb_kernel(const BwdArgs a) {
  using T = typename D::T;
  constexpr int E = kSpanCols;
  constexpr int NP = E / 2;
  constexpr int NWD = E * (int)sizeof(T) / 4;
  constexpr int NL = NWD / 8;
  constexpr int SW = spanb_slot<KIND>();
  constexpr bool LN = kind_is_ln(KIND);
  constexpr bool FROM_Y = kind_from_y(KIND);  // x is the forward's output y
  constexpr bool RECENTER = KIND == KIND_LN;
  constexpr int NS = LN ? (RECENTER ? 3 : 2) : 1;
  static_assert(KIND != KIND_FUSED, "LayerNorm/RMSNorm, from x or from the output");
  extern __shared__ __align__(128) unsigned char smem_sb[];
  const int tpr = blockDim.x;
  const int t = threadIdx.x;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = t & 31;
  const int H = a.H;
  const bool active = t * E < H;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  const size_t es = sizeof(T);
  constexpr int NB = spanb_bufs<KIND>();
  const SpanBLayout L = spanb_layout(tpr, H, (int)es, NS, NB, SW);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_sb + L.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_sb + L.abort);
  float* red = reinterpret_cast<float*>(smem_sb + L.red);
  float* gsh = reinterpret_cast<float*>(smem_sb + L.gamma);
  const float* my_g = gsh + t * SW;
  unsigned char* bufs = smem_sb + L.bufs;
  const uint32_t row_bytes = (uint32_t)H * (uint32_t)es;
  // The two 16-byte halves of a thread's span, in the order the thread holds
  // them: threads 4..7 of every eight take the second half first, so the eight
  // 16-byte shared-memory reads of a quarter warp cover all 32 banks once (in
  // span order every bank is hit twice).  gamma, the accumulators, the partial
  // row and the two 16-byte dx stores follow the same order.  Measured:
  // LayerNorm 8192x5120 main kernel 52.0 -> 51.1 us, RMSNorm 44.9 -> 43.3,
  // LayerNorm 4096x10240 55.7 -> 57.3.
  constexpr bool SWZ = true;
  const int half_a = SWZ ? 8 * ((t >> 2) & 1) : 0;  // columns of the first held half, from the span's start
  const int half_b = 8 - half_a;
  auto held_col = [&](int q) { return q < 2 ? half_a + 4 * q : half_b + 4 * (q - 2); };  // float4 quad q

  if (t == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b) mbar_init(&bar[b], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Four parameters of held quad q as fp32 (p == nullptr or an idle thread: fill).
  auto param4 = [&](const void* p, int q, float fill) {
    float4 v = make_float4(fill, fill, fill, fill);
    if (p != nullptr && active) {
      const int c = t * E + held_col(q);
      if (w_f32) {
        v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + c);
      } else {
        const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const T*>(p) + c);
        const uint32_t w[2] = {u.x, u.y};
        const float2 lo = word_pair<D>(w, 0), hi = word_pair<D>(w, 1);
        v = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }
    return v;
  };
#pragma unroll
  for (int q = 0; q < E / 4; ++q) {
    const float4 g4 = param4(a.gamma, q, 1.f);
    *reinterpret_cast<float4*>(gsh + t * SW + 4 * q) = g4;
    if constexpr (FROM_Y) {  // 1/gamma (IEEE division: gamma = 0 gives infinity) and beta
      *reinterpret_cast<float4*>(gsh + t * SW + E + 4 * q) = make_float4(1.f / g4.x, 1.f / g4.y, 1.f / g4.z, 1.f / g4.w);
      if (LN) *reinterpret_cast<float4*>(gsh + t * SW + 2 * E + 4 * q) = param4(a.beta, q, 0.f);
    }
  }
  __syncthreads();

  const int64_t stride = gridDim.x;
  int64_t row = blockIdx.x;
  unsigned used = 0u, fills = 0u;  // per buffer: ever filled; fills issued, mod 2
  auto issue = [&](int64_t r, int b) {
    unsigned char* dst = bufs + (size_t)b * 2 * L.buf_bytes;
    const void* sx = reinterpret_cast<const T*>(a.x) + r * a.ldx;
    const void* sd = reinterpret_cast<const T*>(a.dy) + r * a.lddy;
    if (((reinterpret_cast<uintptr_t>(sx) | reinterpret_cast<uintptr_t>(sd) | row_bytes) & 15u) != 0) {
      atomicOr(a.err, kErrBadCopy);  // never issued: the row's wait runs out and the call is abandoned
      return;
    }
    mbar_arrive_expect_tx(&bar[b], 2 * row_bytes);
    bulk_g2s(dst, sx, row_bytes, &bar[b]);
    bulk_g2s(dst + L.buf_bytes, sd, row_bytes, &bar[b]);
    used |= 1u << b;
    fills ^= 1u << b;
  };
  if (t == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (row + b * stride < a.N) issue(row + b * stride, b);
  }
  float nrs = 0.f, nmu = 0.f;
  if (row < a.N) {
    nrs = a.rstd[row];
    if (RECENTER) nmu = a.mean[row];
  }
  char* dxp = reinterpret_cast<char*>(a.dx) + (row * a.lddx + (int64_t)t * E) * es;
  const int64_t sdx_step = stride * a.lddx * (int64_t)es;
  float2 accg[NP], accb[LN ? NP : 1];
#pragma unroll
  for (int p = 0; p < NP; ++p) accg[p] = splat2(0.f);
#pragma unroll
  for (int p = 0; p < (LN ? NP : 1); ++p) accb[p] = splat2(0.f);

  int parity = 0;
  for (int k = 0; row < a.N; row += stride, ++k) {
    const int b = k % NB;  // this row's buffer; (k / NB) mod 2 is the parity of its fill
    const int ph = (k / NB) & 1;
    const float r = nrs;
    const float2 r2 = splat2(r);
    const float2 b2 = splat2(RECENTER ? -nmu * r : 0.f);
    if (row + stride < a.N) {
      nrs = a.rstd[row + stride];
      if (RECENTER) nmu = a.mean[row + stride];
    }
    const bool ok = mbar_wait(&bar[b], (uint32_t)ph, a.err, abort_flag);
    const unsigned char* bx = bufs + (size_t)b * 2 * L.buf_bytes + (size_t)t * E * es;
    uint32_t xw[NWD], dw[NWD];
    if (active) {
#pragma unroll
      for (int l = 0; l < 2 * NL; ++l) {
        const int off = (l == 0 ? half_a : half_b) * (int)es;
        const uint4 ux = lds16(bx + off);
        const uint4 ud = lds16(bx + L.buf_bytes + off);
        xw[4 * l] = ux.x; xw[4 * l + 1] = ux.y; xw[4 * l + 2] = ux.z; xw[4 * l + 3] = ux.w;
        dw[4 * l] = ud.x; dw[4 * l + 1] = ud.y; dw[4 * l + 2] = ud.z; dw[4 * l + 3] = ud.w;
      }
    }
    float2 xh[NP];
    if constexpr (FROM_Y) {
      // x_hat = (y - beta) / gamma, from the forward's output.
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 i4 = *reinterpret_cast<const float4*>(my_g + E + 4 * q);
        const float2 gi[2] = {make_float2(i4.x, i4.y), make_float2(i4.z, i4.w)};
        float2 be[2] = {splat2(0.f), splat2(0.f)};
        if constexpr (LN) {
          const float4 b4 = *reinterpret_cast<const float4*>(my_g + 2 * E + 4 * q);
          be[0] = make_float2(b4.x, b4.y);
          be[1] = make_float2(b4.z, b4.w);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 yv = word_pair<D>(xw, 2 * q + h);
          xh[2 * q + h] = mul2(LN ? sub2(yv, be[h]) : yv, gi[h]);
        }
      }
    } else {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const float2 xv = word_pair<D>(xw, p);
        xh[p] = LN ? fma2(xv, r2, b2) : mul2(xv, r2);
      }
    }
    float2 sg = splat2(0.f), sgx = splat2(0.f), sxh = splat2(0.f);
    if (active) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 g4 = *reinterpret_cast<const float4*>(my_g + 4 * q);
        const float2 gm[2] = {make_float2(g4.x, g4.y), make_float2(g4.z, g4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int p = 2 * q + h;
          const float2 g = mul2(word_pair<D>(dw, p), gm[h]);
          sgx = fma2(g, xh[p], sgx);
          if (LN) sg = add2(sg, g);
          if (RECENTER) sxh = add2(sxh, xh[p]);
        }
      }
    }
    float S[NS];
    if (LN) {
      S[0] = sg.x + sg.y;
      S[1] = sgx.x + sgx.y;
      if constexpr (RECENTER) S[NS - 1] = sxh.x + sxh.y;
    } else {
      S[0] = sgx.x + sgx.y;
    }
    group_sum<NS, PW>(S, red, nw, wig, lane, 1, parity);
    // Every thread has read buffer b: refill it with the row NB ahead.
    if (t == 0 && row + NB * stride < a.N && !*abort_flag) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(row + NB * stride, b);
    }
    const float s0 = RECENTER ? S[NS - 1] * inv_h : 0.f;
    const float c1 = LN ? S[0] * inv_h : 0.f;
    const float c2 = LN ? fmaf(-s0, S[0], S[1]) * inv_h : S[0] * inv_h;
    // LayerNorm: dx = r*(g - c1 - c2*xc) taken as (-c2*r)*xc + (g*r - c1*r),
    // two f32x2 instructions a pair after xc (measured 8192x5120 bf16 main
    // kernel 50.9 -> 49.0 us).
    const float2 s02 = splat2(s0), nc22 = splat2(-c2);
    const float2 na2 = splat2(-c2 * r), nb2 = splat2(-c1 * r);
    if (active) {
      uint32_t out[NWD];
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 g4 = *reinterpret_cast<const float4*>(my_g + 4 * q);
        const float2 gm[2] = {make_float2(g4.x, g4.y), make_float2(g4.z, g4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int p = 2 * q + h;
          const float2 d = word_pair<D>(dw, p);
          const float2 g = mul2(d, gm[h]);
          const float2 xc = RECENTER ? sub2(xh[p], s02) : xh[p];
          if constexpr (LN) pair_word<D>(out, p, fma2(xc, na2, fma2(g, r2, nb2)));
          else pair_word<D>(out, p, mul2(fma2(xc, nc22, g), r2));
          accg[p] = fma2(d, xc, accg[p]);
          if (LN) accb[p] = add2(accb[p], d);
        }
      }
      if (ok) {
        if constexpr (SWZ) {
          st_vec(dxp + half_a * (int)es, make_uint4(out[0], out[1], out[2], out[3]));
          st_vec(dxp + half_b * (int)es, make_uint4(out[4], out[5], out[6], out[7]));
        } else {
#pragma unroll
          for (int l = 0; l < NL; ++l) st_vec32(dxp + 32 * l, *reinterpret_cast<const uint32_t(*)[8]>(out + 8 * l));
        }
      }
    }
    dxp += sdx_step;
    parity ^= 1;
  }
  if (t == 0) {
    for (int q = 0; q < NB; ++q)  // the last fill of buffer q has parity (fills - 1) mod 2
      if ((used >> q) & 1u) mbar_wait(&bar[q], ((fills >> q) & 1u) ^ 1u, a.err, nullptr);
  }
  if (a.ws == nullptr || !active) return;
  float* pg = a.ws + (size_t)blockIdx.x * a.Hp + (size_t)t * E;
  float* pb = a.ws + ((size_t)gridDim.x + blockIdx.x) * a.Hp + (size_t)t * E;
#pragma unroll
  for (int q = 0; q < E / 4; ++q) {
    *reinterpret_cast<float4*>(pg + held_col(q)) =
        make_float4(accg[2 * q].x, accg[2 * q].y, accg[2 * q + 1].x, accg[2 * q + 1].y);
    if constexpr (LN)
      *reinterpret_cast<float4*>(pb + held_col(q)) =
          make_float4(accb[2 * q].x, accb[2 * q].y, accb[2 * q + 1].x, accb[2 * q + 1].y);
  }
}

// Staged backward: the bulk-copy pipeline of staged.cuh with x and dy staged
// per row.  Each consumer row group owns one row of every stage; each thread
// owns VPT 16-byte column vectors (the same ones for every row), so its
// dgamma/dbeta accumulators stay in registers for the whole row range.  The
// saved mean/rstd of the group's next row are loaded one stage ahead.  At the
// end the groups' accumulators are summed in shared memory (fixed order) into
// this CTA's partial row, and the dependent reduction kernel is released.
template <int KIND, typename D, int VPT>
__global__ void __launch_bounds__(kStagedThreads, 1) bwd_staged_kernel(const BwdArgs a, const StageCfg c) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr bool LN = KIND == KIND_LN;
  constexpr int NS = LN ? 3 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  const StagedSmem m = staged_smem(smem, c);
  staged_init(m, c);
  int64_t lo, hi;
  cta_rows(a.N, blockIdx.x, gridDim.x, lo, hi);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const int hv = H / VEC;
  const int nwg = c.W / c.G;
  const int g = warp / nwg;
  const int wig = warp - g * nwg;
  const int tpr = nwg * 32;
  const int t = wig * 32 + lane;

  float acc_g[VPT][VEC], acc_b[VPT][VEC];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc_g[v][i] = acc_b[v][i] = 0.f;

  if (warp == c.W) {
    if (lane == 0) {
      const void* const src[2] = {a.x, a.dy};
      const int64_t ld[2] = {a.ldx, a.lddy};
      staged_produce<2>(m, c, src, ld, lo, hi, sizeof(T));
    }
    __syncwarp();  // reconverge before the CTA-wide barrier below
  } else {
    const float inv_h = 1.f / (float)H;
    const bool w_f32 = a.w_f32 != 0;
    float* sh = m.red + g * (2 * nwg * NS);
    const int bar_id = 1 + g;
    int parity = 0;
    int k = 0;
    float r_next = 0.f, mu_next = 0.f;
    if (lo + g < hi) {
      r_next = a.rstd[lo + g];
      if (LN) mu_next = a.mean[lo + g];
    }
    for (int64_t row0 = lo; row0 < hi; row0 += c.G, ++k) {
      const int s = k % c.S;
      const int64_t row = row0 + g;
      const float r = r_next, mu = mu_next;
      if (row + c.G < hi) {  // statistics of this group's next row, one stage ahead
        r_next = a.rstd[row + c.G];
        if (LN) mu_next = a.mean[row + c.G];
      }
      const bool have = mbar_wait(&m.full[s], (k / c.S) & 1, c.err, m.abort);
      if (row < hi) {
        const T* xs = staged_row<T>(m, c, 2, s, 0, g);
        const T* ds = staged_row<T>(m, c, 2, s, 1, g);
        float S[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) S[q] = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int j = t + v * tpr;
          if (j < hv) {
            float xv[VEC], dv[VEC], gm[VEC];
            unpack<D>(lds16(xs + j * VEC), xv);
            unpack<D>(lds16(ds + j * VEC), dv);
            load_param_vec<D>(a.gamma, j * VEC, w_f32, 1.f, gm);
            // per-vector tree sums: short dependency chains
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
              const float xh = LN ? (xv[i] - mu) * r : xv[i] * r;
              const float gg = __fmul_rn(dv[i], gm[i]);
              gm[i] = gg * xh;
              dv[i] = gg;
              xv[i] = xh;
            }
            if (LN) {
              S[0] += tree_sum<VEC>(dv);
              S[1] += tree_sum<VEC>(gm);
              S[2] += tree_sum<VEC>(xv);
            } else {
              S[0] += tree_sum<VEC>(gm);
            }
          }
        }
        group_sum<NS>(S, sh, nwg, wig, lane, bar_id, parity);
        const float s0 = LN ? S[2] * inv_h : 0.f;  // row mean of x_hat: removes the mean's rounding shift
        const float c1 = LN ? S[0] * inv_h : 0.f;
        const float c2 = LN ? fmaf(-s0, S[0], S[1]) * inv_h : S[0] * inv_h;
        T* dxrow = reinterpret_cast<T*>(a.dx) + row * a.lddx;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int j = t + v * tpr;
          if (j < hv) {
            float xv[VEC], dv[VEC], gm[VEC], out[VEC];
            unpack<D>(lds16(xs + j * VEC), xv);
            unpack<D>(lds16(ds + j * VEC), dv);
            load_param_vec<D>(a.gamma, j * VEC, w_f32, 1.f, gm);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
              const float xc = LN ? (xv[i] - mu) * r - s0 : xv[i] * r;
              const float gg = __fmul_rn(dv[i], gm[i]);
              out[i] = r * (gg - c1 - xc * c2);
              acc_g[v][i] = fmaf(dv[i], xc, acc_g[v][i]);
              if (LN) acc_b[v][i] += dv[i];
            }
            if (have) store_vec<D>(dxrow, j * VEC, out);
          }
        }
      }
      parity ^= 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.empty[s]);
    }
  }
  pdl_launch_dependents();
  // Every copy has landed (consumers waited on all of them; the producer
  // drained), so the ring is free: fold the groups into one partial row.
  __syncthreads();
  if (a.ws == nullptr) return;
  const int Hp = a.Hp;
  float* pg = a.ws + (size_t)blockIdx.x * Hp;
  float* pb = a.ws + ((size_t)gridDim.x + blockIdx.x) * Hp;
  const bool consumer = warp < c.W;
  if (c.G == 1) {
    if (consumer) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int j = t + v * tpr;
        if (j < hv) {
#pragma unroll
          for (int q = 0; q < VEC / 4; ++q) {
            *reinterpret_cast<float4*>(pg + j * VEC + 4 * q) = make_float4(
                acc_g[v][4 * q], acc_g[v][4 * q + 1], acc_g[v][4 * q + 2], acc_g[v][4 * q + 3]);
            if (LN)
              *reinterpret_cast<float4*>(pb + j * VEC + 4 * q) = make_float4(
                  acc_b[v][4 * q], acc_b[v][4 * q + 1], acc_b[v][4 * q + 2], acc_b[v][4 * q + 3]);
          }
        }
      }
    }
    return;
  }
  float* red_g = reinterpret_cast<float*>(m.data);
  float* red_b = red_g + Hp;
  for (int g2 = 0; g2 < c.G; ++g2) {
    if (consumer && g == g2) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int j = t + v * tpr;
        if (j < hv) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            const int col = j * VEC + i;
            red_g[col] = g2 == 0 ? acc_g[v][i] : red_g[col] + acc_g[v][i];
            if (LN) red_b[col] = g2 == 0 ? acc_b[v][i] : red_b[col] + acc_b[v][i];
          }
        }
      }
    }
    __syncthreads();
  }
  for (int col = threadIdx.x * 4; col < H; col += blockDim.x * 4) {
    *reinterpret_cast<float4*>(pg + col) = *reinterpret_cast<const float4*>(red_g + col);
    if (LN) *reinterpret_cast<float4*>(pb + col) = *reinterpret_cast<const float4*>(red_b + col);
  }
}

constexpr int LOOP_THREADS = 256;

// Any H, any alignment: one row per CTA iteration, two passes over the row.
// The CTA's partial row lives in the workspace; column j is always handled by
// thread j % LOOP_THREADS, so its read-modify-writes never race.
template <int KIND, typename D>
__global__ void __launch_bounds__(LOOP_THREADS) bwd_loop_kernel(const BwdArgs a) {
  using T = typename D::T;
  constexpr bool LN = kind_is_ln(KIND);
  constexpr bool FROM_Y = kind_from_y(KIND);
  constexpr bool RECENTER = KIND == KIND_LN;
  constexpr int NS = LN ? (RECENTER ? 3 : 2) : 1;
  constexpr int NW = LOOP_THREADS / 32;
  __shared__ float sh[2 * NW * NS];
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int wig = t >> 5;
  const int H = a.H;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  float* pg = a.ws ? a.ws + (size_t)blockIdx.x * a.Hp : nullptr;
  float* pb = a.ws ? a.ws + ((size_t)gridDim.x + blockIdx.x) * a.Hp : nullptr;
  if (pg) {
    for (int j = t; j < a.Hp; j += LOOP_THREADS) {
      pg[j] = 0.f;
      if (LN) pb[j] = 0.f;
    }
  }
  int parity = 0;
  for (int64_t row = blockIdx.x; row < a.N; row += gridDim.x) {
    const T* xrow = reinterpret_cast<const T*>(a.x) + row * a.ldx;
    const T* dyrow = reinterpret_cast<const T*>(a.dy) + row * a.lddy;
    const float r = a.rstd[row];
    const float mu = (LN && !FROM_Y) ? a.mean[row] : 0.f;
    // x_hat of column j: from x and the saved statistics, or from the output
    auto x_hat = [&](float xv, int j) {
      if constexpr (FROM_Y) {
        const float gj = a.gamma ? load_param<D>(a.gamma, j, w_f32) : 1.f;
        const float bj = (LN && a.beta) ? load_param<D>(a.beta, j, w_f32) : 0.f;
        return (xv - bj) / gj;
      } else {
        return LN ? (xv - mu) * r : xv * r;
      }
    };
    float S[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) S[k] = 0.f;
    for (int j = t; j < H; j += LOOP_THREADS) {
      const float xh = x_hat(load_elem<D>(xrow, j), j);
      const float g = __fmul_rn(load_elem<D>(dyrow, j), a.gamma ? load_param<D>(a.gamma, j, w_f32) : 1.f);
      if (LN) {
        S[0] += g;
        S[1] = fmaf(g, xh, S[1]);
        if constexpr (RECENTER) S[NS - 1] += xh;
      } else {
        S[0] = fmaf(g, xh, S[0]);
      }
    }
    group_sum<NS>(S, sh, NW, wig, lane, 1, parity);
    const float s0 = RECENTER ? S[NS - 1] * inv_h : 0.f;
    const float c1 = LN ? S[0] * inv_h : 0.f;
    const float c2 = LN ? fmaf(-s0, S[0], S[1]) * inv_h : S[0] * inv_h;
    T* dxrow = reinterpret_cast<T*>(a.dx) + row * a.lddx;
    for (int j = t; j < H; j += LOOP_THREADS) {
      const float dyv = load_elem<D>(dyrow, j);
      const float xc = x_hat(load_elem<D>(xrow, j), j) - s0;
      const float g = __fmul_rn(dyv, a.gamma ? load_param<D>(a.gamma, j, w_f32) : 1.f);
      float dxv = r * (g - c1 - xc * c2);
      if constexpr (KIND == KIND_FUSED) {
        if (a.dh_in) dxv += load_elem<D>(reinterpret_cast<const T*>(a.dh_in) + row * a.lddh, j);
        if (a.dx_twice) dxv += dxv;
        if (a.dres) store_elem<D>(reinterpret_cast<T*>(a.dres) + row * a.lddres, j, dxv);
      }
      store_elem<D>(dxrow, j, dxv);
      if (pg) {
        pg[j] = fmaf(dyv, xc, pg[j]);
        if (LN) pb[j] += dyv;
      }
    }
    parity ^= 1;
  }
}

// dgamma[j] = sum_p partial[0][p][j], dbeta[j] = sum_p partial[1][p][j],
// blockIdx.y picking the parameter.  A CTA has RG row groups (a power of two,
// the fewest with at most kReduceRows partial rows each) of 256/RG column
// lanes, a lane taking four columns: thread (rg, lane) sums partial rows rg,
// rg + RG, ..., issuing all its loads before adding, so the kernel costs about
// one L2 round trip; then a fixed-order tree over the RG sums in shared
// memory.  Few partial rows (the cluster rows' 76 at 16384 columns) get fewer
// row groups and more columns a CTA: measured against a fixed 32 row groups
// with a serial final sum, LayerNorm 2048x16384 bf16 55.4 -> 53.2 us, 512x16384
// 26.6 -> 24.1, the narrower shapes unchanged.  Fixed summation order, one
// rounding to the output dtype.
constexpr int kReduceRows = 16;

template <typename D, int RG>
__global__ void __launch_bounds__(256) bwd_param_reduce_kernel(const float* ws, int P, int Hp, int H, void* dg,
                                                               void* db, int w_f32) {
  pdl_wait_primary();  // launched as a programmatic dependent of the main kernel
  const int which = blockIdx.y;
  void* out = which ? db : dg;
  if (out == nullptr) return;
  const float* src = ws + (size_t)which * P * Hp;
  constexpr int lanes = 256 / RG;
  const int cl = threadIdx.x % lanes;
  const int rg = threadIdx.x / lanes;
  const int col = (blockIdx.x * lanes + cl) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < Hp) {
    for (int p0 = rg; p0 < P; p0 += RG * kReduceRows) {
      float4 v[kReduceRows];
#pragma unroll
      for (int k = 0; k < kReduceRows; ++k) {
        const int p = p0 + RG * k;
        v[k] = p < P ? *reinterpret_cast<const float4*>(src + (size_t)p * Hp + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kReduceRows; ++k) {
        acc.x += v[k].x;
        acc.y += v[k].y;
        acc.z += v[k].z;
        acc.w += v[k].w;
      }
    }
  }
  __shared__ float4 sm[256];
  sm[threadIdx.x] = acc;
  __syncthreads();
#pragma unroll
  for (int h = RG >> 1; h > 0; h >>= 1) {
    if (rg < h) {
      const float4 o = sm[threadIdx.x + h * lanes];
      float4 m = sm[threadIdx.x];
      m.x += o.x;
      m.y += o.y;
      m.z += o.z;
      m.w += o.w;
      sm[threadIdx.x] = m;
    }
    __syncthreads();
  }
  if (rg == 0 && col < H) {
    const float4 s = sm[threadIdx.x];
    const float vals[4] = {s.x, s.y, s.z, s.w};
    for (int i = 0; i < 4 && col + i < H; ++i) {
      if (w_f32) {
        reinterpret_cast<float*>(out)[col + i] = vals[i];
      } else {
        store_elem<D>(out, col + i, vals[i]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host-side configuration.
// ---------------------------------------------------------------------------

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Clusters of CL CTAs a row: as many clusters as can be resident at once, at
// most p_cap (one partial row each).
template <int KIND, typename D, int VPT, int CL>
static cudaError_t run_rows_cluster(const BwdArgs& a, int threads, int* P, int p_cap, size_t smem,
                                    cudaStream_t s) {
  auto kern = bwd_rows_kernel<KIND, D, VPT, 512, 1, false, CL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * (unsigned)p_cap);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int resident = 0;
  if (cudaOccupancyMaxActiveClusters(&resident, kern, &cfg) != cudaSuccess || resident < 1) resident = 1;
  *P = std::max(1, std::min(p_cap, resident));
  cfg.gridDim = dim3(CL * (unsigned)*P);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KIND, typename D, int VPT, int MAXT, int MINB, bool ACC_SMEM = false>
static cudaError_t run_rows(const BwdArgs& a, int threads, int* P, int p_cap, size_t smem, const DeviceInfo& dev,
                            cudaStream_t s) {
  auto kern = bwd_rows_kernel<KIND, D, VPT, MAXT, MINB, ACC_SMEM>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  *P = std::max(1, std::min(p_cap, per_sm * dev.sm_count));
  kern<<<*P, threads, smem, s>>>(a);
  return cudaGetLastError();
}

constexpr int kStagedMaxCols = 32;  // columns per consumer thread (register accumulators)

template <int KIND, typename D, int VPT>
static cudaError_t run_staged(const BwdArgs& a, const StageCfg& c, int P, size_t smem, cudaStream_t s) {
  auto kern = bwd_staged_kernel<KIND, D, VPT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<P, kStagedThreads, smem, s>>>(a, c);
  return cudaGetLastError();
}

template <int KIND, typename D>
cudaError_t launch_bwd_typed(BwdArgs a, void* dg, void* db, const DeviceInfo& dev,
                                    cudaStream_t s) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr int VPT_MAX = 16 / VEC;  // 16 elements per thread
  constexpr bool LN = kind_is_ln(KIND);
  constexpr bool FROM_Y = kind_from_y(KIND);
  constexpr int NS = KIND == KIND_LN ? 3 : (LN ? 2 : 1);
  constexpr int NPY = FROM_Y ? (LN ? 2 : 1) : 0;  // staged 1/gamma, beta arrays
  const size_t es = sizeof(T);
  const size_t wes = a.w_f32 ? 4 : es;
  const bool want = dg != nullptr || db != nullptr;
  if (a.N == 0) {
    if (dg && cudaMemsetAsync(dg, 0, (size_t)a.H * wes, s) != cudaSuccess) return cudaGetLastError();
    if (db && cudaMemsetAsync(db, 0, (size_t)a.H * wes, s) != cudaSuccess) return cudaGetLastError();
    return cudaSuccess;
  }
  if (!want) a.ws = nullptr;
  a.err = dev.err;
  a.Hp = bwd_partial_stride(a.H);
  const int p_max = bwd_max_partials(dev);
  bool aligned = aligned16(a.x) && aligned16(a.dy) && aligned16(a.dx) && (a.ldx * es) % 16 == 0 &&
                 (a.lddy * es) % 16 == 0 && (a.lddx * es) % 16 == 0;
  if (a.dh_in) aligned = aligned && aligned16(a.dh_in) && (a.lddh * es) % 16 == 0;
  if (a.dres) aligned = aligned && aligned16(a.dres) && (a.lddres * es) % 16 == 0;
  if (a.gamma) aligned = aligned && aligned16(a.gamma);
  if (FROM_Y && LN && a.beta) aligned = aligned && aligned16(a.beta);
  int P = 0;
  cudaError_t err = cudaSuccess;
  bool done = false;
  // Register-row shape: narrow rows one warp each, wider rows 16 elements a
  // thread with more warps, the widest rows shared by a cluster (below).
  const bool vec_ok = aligned && a.H % VEC == 0;
  const int Hv = a.H / VEC;
  // fp32 rows take twice the registers an element: at 16 elements a thread
  // the 640-thread kernels spill (fused 128 bytes, LayerNorm from the output
  // 72).  Where the row fits 640 threads at 8 elements a thread (H <= 5120),
  // fp32 rows take 8, except the plain RMSNorm backward, which barely spills
  // and is faster at 16 (measured at 8192x5120: fused 188 -> 127 us, LN from
  // the output 135 -> 92, LN 104 -> 90; RMS 4096x4096 32.8 -> 36.9 at 8).
  constexpr int VPT_F32 = 2;
  const bool f32_narrow = VEC == 4 && KIND != KIND_RMS && (Hv + VPT_F32 - 1) / VPT_F32 <= 640;
  const int vmax = f32_narrow ? VPT_F32 : VPT_MAX;
  int vpt = vmax, tpr = 0;
  if (Hv <= 32 * vmax) {
    tpr = 32;
    vpt = 1;
    while (vpt * 32 < Hv) vpt *= 2;
  } else {
    tpr = ((Hv + vmax - 1) / vmax + 31) / 32 * 32;
  }
  // Half-precision rows needing more than 640 threads at 16 elements each
  // (10240 < H <= 16384) take 32 elements a thread instead: up to 512
  // threads and 128 registers rather than 1024 threads at 64, which spill
  // (measured: 2048x16384 bf16 LN 101.9 -> 89.1 us, RMS 62.4 -> 49.2 us).
  const int tpr4 = ((Hv + 3) / 4 + 31) / 32 * 32;
  // Rows past 640 threads at 16 elements a thread and up to 16384 wide: a
  // cluster of two CTAs a row, each with half the columns at 16 elements a
  // thread and its accumulators in registers, or, for half precision, one CTA
  // at 32 elements a thread.  Measured (µs) with the asynchronous row-sum
  // exchange: the cluster for every kind (bf16 LN 3413x12288 81.9 -> 69.6,
  // 2048x16384 RMS 47.1 -> 43.0, RMS from the output 53.3 -> 45.1; fp32 2048x16384
  // LN 167.9 -> 108.5 against a spilling single CTA; the LN backward from the
  // output has no single-CTA shape that fits), except the half-precision RMSNorm
  // backward up to 14336 columns (4096x10752 57.3 vs 63.5 with the cluster).
  // Past 1024 threads a row (H > 16384 in half precision and fp32) every kind
  // takes clusters of 4 or 8 CTAs, 512 threads a CTA at most: one CTA's
  // registers and shared memory cannot hold such rows (the staged ring's
  // stages no longer fit either, and the loop reads every row twice).
  auto part_tpr = [&](int parts) { return ((Hv / parts + VPT_MAX - 1) / VPT_MAX + 31) / 32 * 32; };
  const bool cluster_pref = !(KIND == KIND_RMS && VEC == 8 && a.H <= 14336);
  // fp32 rows of 5120 < H <= 10240 for the fused and from-the-output kinds,
  // whose single-CTA kernels spill there: clusters with parts of 256 threads or
  // fewer (measured, fp32 fused 2560x8192 109.6 -> 71.7 us, LN from the output
  // 2048x10240 84.0 -> 65.5; LN and RMS from x gain nothing).
  int cl = 1;
  if (VEC == 4 && (KIND == KIND_FUSED || FROM_Y) && part_tpr(1) > 320 && part_tpr(1) <= 640) {
    for (int parts = 2; parts <= 8 && cl == 1; parts *= 2)
      if (a.H % (parts * VEC) == 0 && part_tpr(parts) <= 256) cl = parts;
  } else if (tpr > 640 && tpr <= 1024) {
    if (cluster_pref && a.H % (2 * VEC) == 0 && part_tpr(2) <= 512) cl = 2;
  } else if (tpr > 1024) {
    for (int parts = 2; parts <= 8 && cl == 1; parts *= 2)
      if (a.H % (parts * VEC) == 0 && part_tpr(parts) <= 512) cl = parts;
  }
  const bool cluster = cl > 1;
  const int tprc = cluster ? part_tpr(cl) : 0;
  const bool wide4 = !cluster && VEC == 8 && tpr > 640 && tpr4 <= 512;
  if (cluster) {
    vpt = VPT_MAX;
    tpr = tprc;
  } else if (wide4) {
    vpt = 4;
    tpr = tpr4;
  }
  const int rpc_rows = tpr <= 256 && !cluster ? 256 / tpr : 1;  // a cluster part: one row at a time
  // group scratch | fp32 gamma (| 1/gamma | beta) | shared accumulators (one
  // row slot) or the fold buffer of several row slots
  const size_t rows_slots = (size_t)vpt * VEC * tpr;
  size_t rows_smem_f = (size_t)((rpc_rows * 2 * (tpr / 32) * NS + 3) & ~3) + (1 + NPY) * rows_slots;
  if (rpc_rows == 1) rows_smem_f += (LN ? 2 : 1) * rows_slots;
  else if (want) rows_smem_f += 2 * (size_t)a.Hp;
  const size_t rows_smem = rows_smem_f * sizeof(float);
  const bool rows_ok = vec_ok && tpr <= 1024 && rows_smem <= (size_t)dev.max_smem_optin;
  // Staged shape.  17 warps leave at most 96 registers a thread (a
  // sub-partition holds 5 warps).  LayerNorm keeps two accumulators per
  // column, so it first tries shapes with at most 24 columns per thread.
  StageCfg c{};
  const bool staged_ok =
      KIND != KIND_FUSED && !FROM_Y && vec_ok &&
      ((KIND == KIND_LN && staged_config(a.H, (int)es, 2, dev.max_smem_optin, 24, &c)) ||
       staged_config(a.H, (int)es, 2, dev.max_smem_optin, kStagedMaxCols, &c));
  bool use_rows = false, use_staged = false;
  switch (dev.path) {
    case PATH_AUTO:
      // LayerNorm keeps two accumulators a column, which the bulk-copy
      // consumers hold in registers: measured, the register rows win for it up
      // to 1024 threads a row (2048x16384 bf16: 98 vs 113 us); RMSNorm gained
      // from the pipeline past 640 before cluster rows.  Now every row the
      // pipeline could hold fits a one-CTA shape of at most 640 threads or a
      // cluster, so AUTO no longer reaches it; PATH_STAGED still forces it.
      use_rows = rows_ok && tpr <= (KIND == KIND_LN ? 1024 : kRowsAutoMaxThreads);
      use_staged = !use_rows && staged_ok;
      use_rows = use_rows || (!use_staged && rows_ok);
      break;
    case PATH_ROWS: use_rows = rows_ok; break;
    case PATH_STAGED:
      use_staged = staged_ok;
      use_rows = !use_staged && rows_ok;
      break;
    default: break;
  }
  if constexpr (KIND != KIND_FUSED && !FROM_Y) {
   if (use_staged) {
    c.err = dev.err;
    c.contiguous = a.ldx == a.H && a.lddy == a.H;
    const int stpr = 32 * (c.W / c.G);
    const int svpt = (Hv + stpr - 1) / stpr;
    P = (int)std::min<int64_t>((int64_t)dev.sm_count, (a.N + c.G - 1) / c.G);
    const size_t smem = staged_smem_bytes(c, 2);
    if (svpt <= 1) err = run_staged<KIND, D, 1>(a, c, P, smem, s);
    else if (svpt <= 2) err = run_staged<KIND, D, 2>(a, c, P, smem, s);
    else if (svpt <= 3) err = run_staged<KIND, D, 3>(a, c, P, smem, s);
    else if (svpt <= 4) err = run_staged<KIND, D, 4>(a, c, P, smem, s);
    else if constexpr (VEC == 4) {
      if (svpt <= 6) err = run_staged<KIND, D, 6>(a, c, P, smem, s);
      else err = run_staged<KIND, D, 8>(a, c, P, smem, s);
    }
    done = true;
   }
  }
  // Span rows: half-precision LayerNorm rows of at most 256 threads at 16
  // contiguous columns a thread (measured: LayerNorm 8192x1024 19.3 -> 17.2 us,
  // 32768x1024 42.1 -> 40.6; RMSNorm gains nothing, wider rows lose).
  if constexpr (KIND == KIND_LN && VEC == 8) {
    auto al32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    const bool aligned32 = al32(a.x) && al32(a.dy) && al32(a.dx) && (a.ldx * es) % 32 == 0 &&
                           (a.lddy * es) % 32 == 0 && (a.lddx * es) % 32 == 0;
    const int stpr = (a.H / kSpanCols + 31) / 32 * 32;
    if (!done && dev.path == PATH_AUTO && aligned32 && a.H % kSpanCols == 0 && stpr <= 256 &&
        (!a.gamma || (reinterpret_cast<uintptr_t>(a.gamma) & 15u) == 0)) {
      const int srpc = 256 / stpr;
      const int threads = srpc * stpr;
      // group scratch | gamma [tpr][slot] | fold buffer [2][tpr][slot] (several row slots)
      const size_t smem = ((size_t)((srpc * 2 * (stpr / 32) * NS + 3) & ~3) +
                           (size_t)stpr * kSpanSlot * (srpc > 1 ? 3 : 1)) * sizeof(float);
      a.tpr = stpr;
      const int p_cap = (int)std::min<int64_t>((a.N + srpc - 1) / srpc, p_max);
      // The row reduction's cross-warp butterfly over a compile-time lane count
      // where the row takes 2, 4 or 5..8 warps (measured LayerNorm bf16
      // 8192x1024 17.7 -> 17.1 us, 16384x2048 40.8 -> 40.1, 8192x4096 42.5 -> 41.6).
      auto kern = bwd_span_kernel<KIND, D, 256, 2>;
      if (stpr == 64) kern = bwd_span_kernel<KIND, D, 256, 2, 2>;
      else if (stpr == 128) kern = bwd_span_kernel<KIND, D, 256, 2, 4>;
      else if (stpr > 128) kern = bwd_span_kernel<KIND, D, 256, 2, 8>;
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
      P = std::max(1, std::min(p_cap, per_sm * dev.sm_count));
      kern<<<P, threads, smem, s>>>(a);
      err = cudaGetLastError();
      done = true;
    }
  }
  // Span rows from shared memory: half-precision LayerNorm and RMSNorm rows,
  // from x or from the saved output (measured from the output against the
  // interleaved register rows: LayerNorm 8192x5120 bf16 74.0 -> 54.4 us,
  // 4096x10240 87.5 -> 63.3, RMSNorm 8192x5120 52.1 -> 46.4).
  if constexpr (KIND != KIND_FUSED && VEC == 8) {
    auto al32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    const bool aligned32 = al32(a.x) && al32(a.dy) && al32(a.dx) && (a.ldx * es) % 32 == 0 &&
                           (a.lddy * es) % 32 == 0 && (a.lddx * es) % 32 == 0;
    const int stpr = (a.H / kSpanCols + 31) / 32 * 32;
    const SpanBLayout SL = spanb_layout(stpr, a.H, (int)es, NS, spanb_bufs<KIND>(), spanb_slot<KIND>());
    const bool beta_ok = !(FROM_Y && LN) || !a.beta || (reinterpret_cast<uintptr_t>(a.beta) & 15u) == 0;
    if (!done && dev.path == PATH_AUTO && aligned32 && a.H % kSpanCols == 0 && stpr > 256 && stpr <= 640 &&
        (size_t)SL.total <= (size_t)dev.max_smem_optin && beta_ok &&
        (!a.gamma || (reinterpret_cast<uintptr_t>(a.gamma) & 15u) == 0)) {
      // The row reduction's cross-warp butterfly over a compile-time lane count
      // (measured LayerNorm 8192x5120 bf16 53.2 -> 51.9 us, 4096x8192 49.4 ->
      // 48.2, 8192x6144 71.7 -> 69.7; the wide forward gains nothing from it).
      auto kern = stpr <= 512 ? bwd_spanb_kernel<KIND, D, 640, 1, 16> : bwd_spanb_kernel<KIND, D, 640, 1, 32>;
      if (SL.total > 48 * 1024) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SL.total);
      }
      if (err == cudaSuccess) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, stpr, SL.total) != cudaSuccess || per_sm < 1)
          per_sm = 1;
        P = std::max(1, (int)std::min<int64_t>(std::min<int64_t>(a.N, p_max), (int64_t)per_sm * dev.sm_count));
        kern<<<P, stpr, SL.total, s>>>(a);
        err = cudaGetLastError();
      }
      done = true;
    }
  }
  // Register rows; the grid is persistent: as many CTAs as fit, at most
  // 2 x SM count (the partial rows the workspace holds).
  if (!done && use_rows) {
    a.tpr = tpr;
    const int rpc = rpc_rows;
    const int threads = rpc * tpr;
    const int p_cap = (int)std::min<int64_t>((a.N + rpc - 1) / rpc, p_max);
    const size_t smem = rows_smem;
    if (cluster) {  // first: a cluster part may have 256 threads or fewer
      const int cl_cap = (int)std::min<int64_t>(a.N, p_max);
      if (cl == 2) err = run_rows_cluster<KIND, D, VPT_MAX, 2>(a, threads, &P, cl_cap, smem, s);
      else if (cl == 4) err = run_rows_cluster<KIND, D, VPT_MAX, 4>(a, threads, &P, cl_cap, smem, s);
      else err = run_rows_cluster<KIND, D, VPT_MAX, 8>(a, threads, &P, cl_cap, smem, s);
    } else if (threads <= 256) {
      switch (vpt) {
        case 1: err = run_rows<KIND, D, 1, 256, 2>(a, threads, &P, p_cap, smem, dev, s); break;
        case 2: err = run_rows<KIND, D, 2, 256, 2>(a, threads, &P, p_cap, smem, dev, s); break;
        default:
          if constexpr (VPT_MAX >= 4) err = run_rows<KIND, D, 4, 256, 2>(a, threads, &P, p_cap, smem, dev, s);
          break;
      }
    } else if (wide4) {
      if constexpr (VEC == 8) err = run_rows<KIND, D, 4, 512, 1, true>(a, threads, &P, p_cap, smem, dev, s);
    } else if (threads <= 640) {
      if (vpt == VPT_F32 && VPT_MAX != VPT_F32) {
        if constexpr (VEC == 4) err = run_rows<KIND, D, VPT_F32, 640, 1, true>(a, threads, &P, p_cap, smem, dev, s);
      } else {
        err = run_rows<KIND, D, VPT_MAX, 640, 1, true>(a, threads, &P, p_cap, smem, dev, s);
      }
    } else {
      err = run_rows<KIND, D, VPT_MAX, 1024, 1, true>(a, threads, &P, p_cap, smem, dev, s);
    }
    done = true;
  }
  if (!done) {
    P = (int)std::min<int64_t>(a.N, p_max);
    bwd_loop_kernel<KIND, D><<<P, LOOP_THREADS, 0, s>>>(a);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess || !want) return err;
  // The column reduction is a programmatic dependent of the main kernel: it
  // is scheduled while the main kernel drains and waits for it on the device.
  // With a split event set (timing the two kernels apart), the event is
  // recorded between them and the reduction is an ordinary launch.
  const bool split = dev.split_event != nullptr;
  if (split) {
    err = cudaEventRecord(static_cast<cudaEvent_t>(dev.split_event), s);
    if (err != cudaSuccess) return err;
  }
  int RG = 4;
  while (RG < 32 && RG * kReduceRows < P) RG *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.Hp / 4 + 256 / RG - 1) / (256 / RG), LN ? 2 : 1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split ? 0 : 1;
  const float* ws = a.ws;
  void* dbeta = LN ? db : nullptr;
  if (RG <= 4) err = cudaLaunchKernelEx(&cfg, bwd_param_reduce_kernel<D, 4>, ws, P, a.Hp, a.H, dg, dbeta, a.w_f32);
  else if (RG <= 8) err = cudaLaunchKernelEx(&cfg, bwd_param_reduce_kernel<D, 8>, ws, P, a.Hp, a.H, dg, dbeta, a.w_f32);
  else if (RG <= 16) err = cudaLaunchKernelEx(&cfg, bwd_param_reduce_kernel<D, 16>, ws, P, a.Hp, a.H, dg, dbeta, a.w_f32);
  else err = cudaLaunchKernelEx(&cfg, bwd_param_reduce_kernel<D, 32>, ws, P, a.Hp, a.H, dg, dbeta, a.w_f32);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace normk
