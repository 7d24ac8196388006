// Forward kernel templates and their launch logic, instantiated per row
// dtype by norm_fwd_f32.cu, norm_fwd_bf16.cu and norm_fwd_f16.cu.
//
// Forward kernels: LayerNorm, RMSNorm and fused residual-add + RMSNorm.
//
// Kernel families (launch_fwd_typed picks one per call: register rows --
// wide-chunk rows where half-precision rows are 32-byte aligned, else 16-byte
// vector rows -- while a row needs at most 640 threads, then the bulk-copy
// pipeline, then register rows shared by a cluster of 2, 4 or 8 CTAs, then
// register rows of up to 1024 threads for widths no cluster split divides,
// then the loop):
//
// * fwd_rows_kernel -- the row lives in registers.  A "row group" of `tpr`
//   threads (one warp for narrow rows, up to 1024 threads for wide rows) owns
//   one row at a time and prefetches its next; each thread holds VPT 16-byte
//   vectors of it, so HBM is read exactly once and written exactly once.
//   Vector v of thread t covers columns [(v*tpr + t)*VEC, +VEC): consecutive
//   threads touch consecutive 16-byte chunks, so every warp-wide access is
//   fully coalesced.  Needs 16-byte aligned rows and H a multiple of the
//   vector width.
// * fwd_wide_kernel -- the register rows of half-precision LayerNorm,
//   RMSNorm and the fused add whose rows are 32-byte aligned (H >= 512, a
//   multiple of 16): the same walk, with 32-byte chunks of 16 contiguous
//   columns as the unit and gamma/beta in a per-thread slot, for fewer
//   instructions an element.
// * fwd_staged_kernel -- persistent, one CTA per SM; a producer warp streams
//   rows through a shared-memory ring with bulk copies (see staged.cuh) and
//   consumer row groups compute from shared memory.  Same alignment needs,
//   and at least three stages of rows in shared memory.
// * fwd_loop_kernel -- any H and any alignment: one CTA per row, a strided
//   loop over the row, a statistics pass and an output pass (the second read
//   mostly hits L2).  Per-thread statistics use Welford's recurrence.  The
//   fused kernel stores h in the output pass, after re-forming the fp32 sum.
//
// Statistics ("Skill: Write CUDA LayerNorm Kernel", Required reasoning process
// steps 2-5; "Skill: Write a Triton LayerNorm Kernel" steps 3-7):
// LayerNorm: the register-row kernel holds the whole row and reduces the
// shifted sums sum(d), sum(d^2) together, taking the exact second pass over
// the registers only when the pivot sits far from the mean (see the kernel).
// The kernels that stream the row keep a Welford triple (count, mean, M2) per
// thread and merge triples across lanes and warps with the parallel merge.
// M2 is divided by the full row length H.  Values are shifted before
// accumulating (by the mean of the row's first 16-byte vector in the register
// kernel, by the first element in the others; x - s is exact when the two are
// close), so rows with a large common offset keep full precision.
// RMSNorm sums x^2.  rstd = rsqrt(var + eps): eps inside the square root.
//
// Fused add ("Skill: Write a Triton Fused Add+RMSNorm Kernel", steps 2-7):
// h = x + residual in fp32, h stored (rounded to the row dtype) before the
// reduction, y computed from the fp32 h.  Each element of h is written by the
// thread that read that element of x and residual, so h_out may alias either.

#pragma once

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "staged.cuh"

namespace normk {

// Register-row kernel.  Persistent row groups of `tpr` threads walk rows
// row, row + stride, ...; while a group computes one row, the 16-byte loads
// of its next row are already in flight (software pipelining), so each warp
// keeps two rows' worth of HBM reads outstanding.  Each row is unpacked once
// into fp32 pairs and every elementwise step uses packed f32x2 instructions.
//
// CL > 1: a thread-block cluster of CL CTAs shares each row, CTA rank r taking
// columns [r*H/CL, (r+1)*H/CL); the row sums meet through distributed shared
// memory (cluster_group_sum_async: one exchange a row, two when the exact
// second pass runs).
// Used only for rows that neither one CTA's registers nor the bulk-copy ring
// can hold (measured: where one CTA still fits, it is faster).
template <typename D>
__device__ __forceinline__ FwdArgs part_row_view(FwdArgs a, int rank, int parts) {
  using T = typename D::T;
  const int64_t c0 = (int64_t)rank * (a.H / parts);
  const size_t wes = a.w_f32 ? 4 : sizeof(T);
  a.x = reinterpret_cast<const T*>(a.x) + c0;
  a.y = reinterpret_cast<T*>(a.y) + c0;
  if (a.res) a.res = reinterpret_cast<const T*>(a.res) + c0;
  if (a.h) a.h = reinterpret_cast<T*>(a.h) + c0;
  if (a.gamma) a.gamma = reinterpret_cast<const unsigned char*>(a.gamma) + c0 * wes;
  if (a.beta) a.beta = reinterpret_cast<const unsigned char*>(a.beta) + c0 * wes;
  a.H /= parts;
  return a;
}

// The body of fwd_rows_kernel: `a` describes this CTA's columns, `af` the
// whole row (its first vector sets the LayerNorm shift; its length is what
// the statistics divide by), `crank` the CTA's rank in its cluster.
template <int KIND, typename D, int VPT, int CL>
__device__ __forceinline__ void fwd_rows_body(const FwdArgs& a, const FwdArgs& af, int crank) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr int VP = VEC / 2;
  constexpr bool CLUSTER = CL > 1;
  extern __shared__ __align__(16) float sh_dyn[];
  __shared__ float xch[2][CL * 4];   // cluster exchange of the row sums ([rank][value]), by parity
  __shared__ float xch2[2][CL * 4];  // the exact second pass's exchange, by its own parity
  __shared__ uint64_t xbar[2], xbar2[2];
  __shared__ int xabort;
  const int tpr = a.tpr;
  const int rpc = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;  // this CTA's columns (a part of the row in a cluster)
  const int hv = H / VEC;
  const float inv_h = 1.f / (float)af.H;
  const bool w_f32 = a.w_f32 != 0;
  float* sh = sh_dyn + slot * (2 * nw * 3);
  const int bar_id = 1 + slot;
  const int prow = (int)blockIdx.x / CL;
  const int64_t stride = (int64_t)(gridDim.x / CL) * rpc;
  int nvec = 0;  // vectors of each row this thread owns
#pragma unroll
  for (int v = 0; v < VPT; ++v) nvec += (t + v * tpr < hv) ? 1 : 0;
  uint4 nx[VPT], nr[VPT];
  uint4 npv = make_uint4(0u, 0u, 0u, 0u);  // LayerNorm: the next row's first 16-byte vector (its shift)
  auto fetch = [&](int64_t r) {
    const T* xrow = reinterpret_cast<const T*>(a.x) + r * a.ldx;
#pragma unroll
    for (int v = 0; v < VPT; ++v) nx[v] = load_vec_or_zero<D>(xrow, (t + v * tpr) * VEC, H);
    if constexpr (KIND == KIND_FUSED) {
      const T* rrow = reinterpret_cast<const T*>(a.res) + r * a.ldr;
#pragma unroll
      for (int v = 0; v < VPT; ++v) nr[v] = load_vec_or_zero<D>(rrow, (t + v * tpr) * VEC, H);
    }
    // LayerNorm's shift is the mean of the row's first 16-byte vector (one
    // broadcast load), so that one outlying first element does not set it.
    // Only the load is issued here; the mean is formed when the row is used,
    // so the load stays in flight over the current row like the row's own.
    if constexpr (KIND == KIND_LN) npv = ld_cached(reinterpret_cast<const T*>(af.x) + r * af.ldx);
  };
  auto vector_mean = [](const uint4& u) {
    float f0[VEC];
    unpack<D>(u, f0);
    float sum0 = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) sum0 += f0[i];
    return sum0 * (1.f / VEC);
  };

  int parity = 0;
  int64_t row = (int64_t)prow * rpc + slot;
  if (row < a.N) fetch(row);  // first row in flight while the parameters are staged
  constexpr bool PF = kL2PrefetchRows > 1 && KIND != KIND_FUSED;
  auto l2_prefetch_row = [&](int64_t pr) {
    l2_prefetch_bulk(reinterpret_cast<const T*>(a.x) + pr * a.ldx, (uint32_t)(H * sizeof(T)));
    if constexpr (KIND == KIND_FUSED)
      l2_prefetch_bulk(reinterpret_cast<const T*>(a.res) + pr * a.ldr, (uint32_t)(H * sizeof(T)));
  };
  if constexpr (PF) {
    // rows 2 .. depth-1 strides ahead now; the loop asks for `depth` ahead
    if (t == 0) {
#pragma unroll 1
      for (int k = 2; k < kL2PrefetchRows; ++k)
        if (row + k * stride < a.N) l2_prefetch_row(row + k * stride);
    }
  }

  // gamma (and beta) as fp32, thread-interleaved, shared by the row slots.
  float4* gs = reinterpret_cast<float4*>(sh_dyn + ((rpc * 2 * nw * 3 + 3) & ~3));
  float4* bs = gs + VPT * (VEC / 4) * tpr;
  if (slot == 0) {
    stage_params<D, VPT>(gs, a.gamma, w_f32, 1.f, t, tpr, hv);
    if constexpr (KIND == KIND_LN) stage_params<D, VPT>(bs, a.beta, w_f32, 0.f, t, tpr, hv);
  }
  __syncthreads();
  unsigned it = 0, it2 = 0;  // exchanges this CTA has made (cluster rows)
  if constexpr (CLUSTER) {
    if (threadIdx.x == 0) {
      mbar_init(&xbar[0], 1);
      mbar_init(&xbar[1], 1);
      mbar_init(&xbar2[0], 1);
      mbar_init(&xbar2[1], 1);
      xabort = 0;
      fence_barrier_init();
    }
    cluster_sync_all();  // every CTA's mbarriers exist before any CTA sends to them
  }

  for (; row < a.N; row += stride) {
    // Unpack the current row (it arrived while the previous row computed).
    float2 f[VPT][VP];
#pragma unroll
    for (int v = 0; v < VPT; ++v) unpack2<D>(nx[v], f[v]);
    const float pivot = KIND == KIND_LN ? vector_mean(npv) : 0.f;
    if constexpr (KIND == KIND_FUSED) {
      T* hrow = reinterpret_cast<T*>(a.h) + row * a.ldh;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        float2 r[VP];
        unpack2<D>(nr[v], r);
#pragma unroll
        for (int p = 0; p < VP; ++p) f[v][p] = add2(f[v][p], r[p]);
        if (v < nvec) st_vec(reinterpret_cast<T*>(hrow) + (t + v * tpr) * VEC, pack2<D>(f[v]));
      }
    }
    // Issue the next row's loads before computing this one.  LayerNorm and
    // RMSNorm also ask L2 for a row further ahead (measured: it shortens the
    // wide-row forward; the fused add, already near the HBM roof, and the
    // backward, bound by the shared-memory pipe, lose with it).
    if (row + stride < a.N) fetch(row + stride);
    if constexpr (PF) {
      const int64_t pr = row + kL2PrefetchRows * stride;
      if (t == 0 && pr < a.N) l2_prefetch_row(pr);
    }

    float rstd, mean_d = 0.f;
    if constexpr (KIND == KIND_LN) {
      // Shifted sums of the row held in registers: with d = x - x0,
      // M2 = sum(d^2) - mean(d)*sum(d) in one reduction.  Its rounding error is
      // about eps_f32 * (M2 + H*mean(d)^2); while mean(d)^2 <= 4*M2/H (the
      // pivot within two standard deviations of the mean) that stays at the
      // fp32 noise of M2 itself.  Otherwise the row takes the exact second
      // pass, sum((d - mean(d))^2), a second reduction.  Every thread holds
      // the same reduced values, so the branch is uniform.
      const float2 pv = splat2(pivot);
      float2 s2 = splat2(0.f), q2 = splat2(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (v < nvec) {
#pragma unroll
          for (int p = 0; p < VP; ++p) f[v][p] = sub2(f[v][p], pv);
          float2 vs = f[v][0];
          float2 vq = mul2(f[v][0], f[v][0]);
#pragma unroll
          for (int p = 1; p < VP; ++p) {
            vs = add2(vs, f[v][p]);
            vq = fma2(f[v][p], f[v][p], vq);
          }
          s2 = add2(s2, vs);
          q2 = add2(q2, vq);
        }
      }
      float sq[2] = {s2.x + s2.y, q2.x + q2.y};
      group_sum<2>(sq, sh, nw, wig, lane, bar_id, parity);
      if constexpr (CLUSTER) {
        cluster_group_sum_async<2, CL>(sq, xch[it & 1], &xbar[it & 1], (it >> 1) & 1u, crank, a.err, &xabort);
        ++it;
      }
      mean_d = sq[0] * inv_h;
      float m2 = fmaf(-mean_d, sq[0], sq[1]);
      if (mean_d * mean_d * (float)af.H > 4.f * m2) {
        const float2 ml = splat2(mean_d);
        float2 e2 = splat2(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          if (v < nvec) {
#pragma unroll
            for (int p = 0; p < VP; ++p) {
              const float2 e = sub2(f[v][p], ml);
              e2 = fma2(e, e, e2);
            }
          }
        }
        float mm[1] = {e2.x + e2.y};
        group_sum<1>(mm, sh + 4 * nw, nw, wig, lane, bar_id, parity);
        if constexpr (CLUSTER) {  // uniform across the cluster: every part holds the same sums
          cluster_group_sum_async<1, CL>(mm, xch2[it2 & 1], &xbar2[it2 & 1], (it2 >> 1) & 1u, crank, a.err,
                                         &xabort);
          ++it2;
        }
        m2 = mm[0];
      }
      rstd = rsqrtf(fmaxf(m2, 0.f) * inv_h + a.eps);
    } else {
      float2 s2 = splat2(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (v < nvec) {
          float2 vq = mul2(f[v][0], f[v][0]);
#pragma unroll
          for (int p = 1; p < VP; ++p) vq = fma2(f[v][p], f[v][p], vq);
          s2 = add2(s2, vq);
        }
      }
      float ss[1] = {s2.x + s2.y};
      group_sum<1>(ss, sh, nw, wig, lane, bar_id, parity);
      if constexpr (CLUSTER) {
        cluster_group_sum_async<1, CL>(ss, xch[it & 1], &xbar[it & 1], (it >> 1) & 1u, crank, a.err, &xabort);
        ++it;
      }
      rstd = rsqrtf(ss[0] * inv_h + a.eps);
    }
    if (t == 0 && crank == 0) {
      if constexpr (KIND == KIND_LN) {
        if (a.mean) a.mean[row] = pivot + mean_d;
      }
      if (a.rstd) a.rstd[row] = rstd;
    }

    T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy;
    const float2 r2 = splat2(rstd);
    const float2 b2 = splat2(-mean_d * rstd);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (v < nvec) {
        const int col = (t + v * tpr) * VEC;
        float2 gm[VP], out[VP];
        read_pairs<VEC>(gs, v, t, tpr, gm);
        if constexpr (KIND == KIND_LN) {
          float2 be[VP];
          read_pairs<VEC>(bs, v, t, tpr, be);
#pragma unroll
          for (int p = 0; p < VP; ++p) out[p] = fma2(fma2(f[v][p], r2, b2), gm[p], be[p]);
        } else {
#pragma unroll
          for (int p = 0; p < VP; ++p) out[p] = mul2(mul2(f[v][p], r2), gm[p]);
        }
        st_vec(yrow + col, pack2<D>(out));
      }
    }
    parity ^= 1;
  }
  if constexpr (CLUSTER) cluster_sync_all();  // no CTA leaves while a partner may still write to it
}

template <int KIND, typename D, int VPT, int MAXT, int MINB, int CL = 1>
__global__ void __launch_bounds__(MAXT, MINB) fwd_rows_kernel(const FwdArgs a) {
  if constexpr (CL > 1) {
    const int crank = (int)cluster_ctarank();
    const FwdArgs part = part_row_view<D>(a, crank, CL);
    fwd_rows_body<KIND, D, VPT, CL>(part, a, crank);
  } else {
    fwd_rows_body<KIND, D, VPT, CL>(a, a, 0);
  }
}


// Wide-chunk register rows (half-precision LayerNorm, RMSNorm and the fused
// add, rows 32-byte aligned, H a multiple of 16): the row walk, prefetch and arithmetic of
// fwd_rows_body, but a thread's unit is a 32-byte chunk of 16 contiguous
// columns -- chunk c of thread t covers columns [16*(t + c*tpr), +16) -- so
// one 256-bit load or store moves it, the thread reaches its chunks from one
// pointer a row, and gamma/beta sit in a per-thread shared-memory slot
// ([gamma of its columns | beta of its columns | 4 floats of padding], so the
// 16-byte reads of eight consecutive threads hit distinct banks) read at
// constant offsets.
constexpr int kWideCols = 16;
template <int NCH>
__host__ __device__ constexpr int wide_slot() { return 2 * NCH * kWideCols + 4; }

template <int KIND, typename D, int NCH, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) fwd_wide_kernel(const FwdArgs a) {
  using T = typename D::T;
  static_assert(sizeof(T) == 2, "half precision");
  constexpr bool FUSED = KIND == KIND_FUSED;
  constexpr int NT = FUSED ? NCH : 1;  // residual chunks held (fused add only)
  constexpr int CW = kWideCols;
  constexpr int NP = CW / 2;  // fp32 pairs (32-bit words) a chunk
  constexpr int SLOT = wide_slot<NCH>();
  constexpr int VEC = D::VEC;
  extern __shared__ __align__(16) float sh_dyn[];
  const int tpr = a.tpr;
  const int rpc = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const int hc = H / CW;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  float* sh = sh_dyn + slot * (2 * nw * 3);
  float* my_p = sh_dyn + ((rpc * 2 * nw * 3 + 3) & ~3) + t * SLOT;
  const int bar_id = 1 + slot;
  const int64_t stride = (int64_t)gridDim.x * rpc;
  int nch = 0;  // chunks of each row this thread owns
#pragma unroll
  for (int c = 0; c < NCH; ++c) nch += (t + c * tpr < hc) ? 1 : 0;
  const int64_t cs = (int64_t)tpr * CW;  // elements from one chunk of a thread to its next

  int64_t row = (int64_t)blockIdx.x * rpc + slot;
  const T* xnext = reinterpret_cast<const T*>(a.x) + row * a.ldx + t * CW;
  const int64_t xstep = stride * a.ldx;
  const T* rnext = FUSED ? reinterpret_cast<const T*>(a.res) + row * a.ldr + t * CW : nullptr;
  const int64_t rstep = FUSED ? stride * a.ldr : 0;
  uint32_t nx[NCH][NP], nr[NT][NP];
  uint4 npv = make_uint4(0u, 0u, 0u, 0u);
  auto fetch = [&](int64_t r) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      if (c < nch) {
        ld_stream32(xnext + c * cs, nx[c]);
        if constexpr (FUSED) ld_stream32(rnext + c * cs, nr[c]);
      } else {
#pragma unroll
        for (int k = 0; k < NP; ++k) nx[c][k] = 0u;
        if constexpr (FUSED) {
#pragma unroll
          for (int k = 0; k < NP; ++k) nr[c][k] = 0u;
        }
      }
    }
    if constexpr (KIND == KIND_LN) npv = ld_cached(reinterpret_cast<const T*>(a.x) + r * a.ldx);
    xnext += xstep;
    if constexpr (FUSED) rnext += rstep;
  };
  auto vector_mean = [](const uint4& u) {
    float f0[VEC];
    unpack<D>(u, f0);
    float sum0 = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) sum0 += f0[i];
    return sum0 * (1.f / VEC);
  };
  if (row < a.N) fetch(row);
  constexpr bool PF = kL2PrefetchRows > 1 && !FUSED;
  auto l2_prefetch_row = [&](int64_t pr) {
    l2_prefetch_bulk(reinterpret_cast<const T*>(a.x) + pr * a.ldx, (uint32_t)(H * sizeof(T)));
  };
  if constexpr (PF) {
    if (t == 0) {
#pragma unroll 1
      for (int k = 2; k < kL2PrefetchRows; ++k)
        if (row + k * stride < a.N) l2_prefetch_row(row + k * stride);
    }
  }
  if (slot == 0) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int col = (t + c * tpr) * CW;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2 g[VEC / 2], b[VEC / 2];
        if (c < nch) {
          load_param_pairs<D>(a.gamma, col + h * VEC, w_f32, 1.f, g);
          if constexpr (KIND == KIND_LN) load_param_pairs<D>(a.beta, col + h * VEC, w_f32, 0.f, b);
        } else {
#pragma unroll
          for (int i = 0; i < VEC / 2; ++i) g[i] = b[i] = splat2(0.f);
        }
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
          const int o = c * CW + h * VEC + 4 * q;
          *reinterpret_cast<float4*>(my_p + o) = make_float4(g[2 * q].x, g[2 * q].y, g[2 * q + 1].x, g[2 * q + 1].y);
          if constexpr (KIND == KIND_LN)
            *reinterpret_cast<float4*>(my_p + NCH * CW + o) =
                make_float4(b[2 * q].x, b[2 * q].y, b[2 * q + 1].x, b[2 * q + 1].y);
        }
      }
    }
  }
  __syncthreads();

  T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy + t * CW;
  const int64_t ystep = stride * a.ldy;
  T* hrow = FUSED ? reinterpret_cast<T*>(a.h) + row * a.ldh + t * CW : nullptr;
  const int64_t hstep = FUSED ? stride * a.ldh : 0;
  int parity = 0;
  for (; row < a.N; row += stride, yrow += ystep) {
    float2 f[NCH][NP];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
      for (int p = 0; p < NP; ++p) f[c][p] = word_pair<D>(nx[c], p);
    if constexpr (FUSED) {
      // h = x + residual in fp32, stored (rounded) by the thread that read
      // both, before the next row's loads are issued
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint32_t hw[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          f[c][p] = add2(f[c][p], word_pair<D>(nr[c], p));
          pair_word<D>(hw, p, f[c][p]);
        }
        if (c < nch) st_vec32(hrow + c * cs, hw);
      }
      hrow += hstep;
    }
    const float pivot = KIND == KIND_LN ? vector_mean(npv) : 0.f;
    if (row + stride < a.N) fetch(row + stride);
    if constexpr (PF) {
      const int64_t pr = row + kL2PrefetchRows * stride;
      if (t == 0 && pr < a.N) l2_prefetch_row(pr);
    }

    float rstd, mean_d = 0.f;
    if constexpr (KIND == KIND_LN) {
      // Shifted one-pass sums and the guard of fwd_rows_body.
      const float2 pv = splat2(pivot);
      float2 s2 = splat2(0.f), q2 = splat2(0.f);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        if (c < nch) {
#pragma unroll
          for (int p = 0; p < NP; ++p) f[c][p] = sub2(f[c][p], pv);
          float2 vs = f[c][0];
          float2 vq = mul2(f[c][0], f[c][0]);
#pragma unroll
          for (int p = 1; p < NP; ++p) {
            vs = add2(vs, f[c][p]);
            vq = fma2(f[c][p], f[c][p], vq);
          }
          s2 = add2(s2, vs);
          q2 = add2(q2, vq);
        }
      }
      float sq[2] = {s2.x + s2.y, q2.x + q2.y};
      group_sum<2>(sq, sh, nw, wig, lane, bar_id, parity);
      mean_d = sq[0] * inv_h;
      float m2 = fmaf(-mean_d, sq[0], sq[1]);
      if (mean_d * mean_d * (float)H > 4.f * m2) {
        const float2 ml = splat2(mean_d);
        float2 e2 = splat2(0.f);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (c < nch) {
#pragma unroll
            for (int p = 0; p < NP; ++p) {
              const float2 e = sub2(f[c][p], ml);
              e2 = fma2(e, e, e2);
            }
          }
        }
        float mm[1] = {e2.x + e2.y};
        group_sum<1>(mm, sh + 4 * nw, nw, wig, lane, bar_id, parity);
        m2 = mm[0];
      }
      rstd = rsqrtf(fmaxf(m2, 0.f) * inv_h + a.eps);
    } else {
      float2 s2 = splat2(0.f);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        if (c < nch) {
          float2 vq = mul2(f[c][0], f[c][0]);
#pragma unroll
          for (int p = 1; p < NP; ++p) vq = fma2(f[c][p], f[c][p], vq);
          s2 = add2(s2, vq);
        }
      }
      float ss[1] = {s2.x + s2.y};
      group_sum<1>(ss, sh, nw, wig, lane, bar_id, parity);
      rstd = rsqrtf(ss[0] * inv_h + a.eps);
    }
    if (t == 0) {
      if constexpr (KIND == KIND_LN) {
        if (a.mean) a.mean[row] = pivot + mean_d;
      }
      if (a.rstd) a.rstd[row] = rstd;
    }

    const float2 r2 = splat2(rstd);
    const float2 b2 = splat2(-mean_d * rstd);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      if (c < nch) {
        uint32_t ow[NP];
#pragma unroll
        for (int q = 0; q < CW / 4; ++q) {
          const float4 g4 = *reinterpret_cast<const float4*>(my_p + c * CW + 4 * q);
          const float2 gm[2] = {make_float2(g4.x, g4.y), make_float2(g4.z, g4.w)};
          if constexpr (KIND == KIND_LN) {
            const float4 b4 = *reinterpret_cast<const float4*>(my_p + NCH * CW + c * CW + 4 * q);
            const float2 be[2] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
#pragma unroll
            for (int h = 0; h < 2; ++h)
              pair_word<D>(ow, 2 * q + h, fma2(fma2(f[c][2 * q + h], r2, b2), gm[h], be[h]));
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) pair_word<D>(ow, 2 * q + h, mul2(mul2(f[c][2 * q + h], r2), gm[h]));
          }
        }
        st_vec32(yrow + c * cs, ow);
      }
    }
    parity ^= 1;
  }
}


// Consumers copy their VPT vectors of the row from shared memory into packed
// registers, release the stage at once (the producer can refill it while they
// compute), unpack it once into fp32 pairs and run every pass from registers
// with f32x2 math; gamma/beta are read from fp32 copies staged once per CTA in
// shared memory (thread-interleaved, conflict-free).
template <int KIND, typename D, int VPT>
__global__ void __launch_bounds__(kStagedThreads, 1) fwd_staged_kernel(const FwdArgs a, const StageCfg c) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr int VP = VEC / 2;
  constexpr int NT = KIND == KIND_FUSED ? 2 : 1;  // staged tensors: x (and residual)
  extern __shared__ __align__(128) unsigned char smem[];
  const StagedSmem m = staged_smem(smem, c);
  staged_init(m, c);
  int64_t lo, hi;
  cta_rows(a.N, blockIdx.x, gridDim.x, lo, hi);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == c.W) {
    if (lane == 0) {
      if constexpr (NT == 2) {
        const void* const src[2] = {a.x, a.res};
        const int64_t ld[2] = {a.ldx, a.ldr};
        staged_produce<2>(m, c, src, ld, lo, hi, sizeof(T));
      } else {
        const void* const src[1] = {a.x};
        const int64_t ld[1] = {a.ldx};
        staged_produce<1>(m, c, src, ld, lo, hi, sizeof(T));
      }
    }
    return;
  }

  const int H = a.H;
  const int hv = H / VEC;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  const int nwg = c.W / c.G;  // warps per row group
  const int g = warp / nwg;
  const int wig = warp - g * nwg;
  const int tpr = nwg * 32;
  const int t = wig * 32 + lane;
  float* sh = m.red + g * (2 * nwg * 3);
  const int bar_id = 1 + g;
  int nvec = 0;  // vectors of each row this thread owns
#pragma unroll
  for (int v = 0; v < VPT; ++v) nvec += (t + v * tpr < hv) ? 1 : 0;
  // fp32 gamma (and beta), staged by row group 0 while the first copies fly.
  float4* gs = m.par;
  float4* bs = gs + VPT * (VEC / 4) * tpr;
  if (g == 0) {
    stage_params<D, VPT>(gs, a.gamma, w_f32, 1.f, t, tpr, hv);
    if constexpr (KIND == KIND_LN) stage_params<D, VPT>(bs, a.beta, w_f32, 0.f, t, tpr, hv);
  }
  named_barrier(15, c.W * 32);  // consumers only (group barriers use ids 1..G, G <= 8 when used)

  int parity = 0;
  int k = 0;
  for (int64_t row0 = lo; row0 < hi; row0 += c.G, ++k) {
    const int s = k % c.S;
    const bool have = mbar_wait(&m.full[s], (k / c.S) & 1, c.err, m.abort);
    const int64_t row = row0 + g;
    const bool mine = row < hi;  // uniform across the row group
    uint4 xr[VPT], rr[VPT];
    float pivot = 0.f;
    if (mine) {
      const T* xs = staged_row<T>(m, c, NT, s, 0, g);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int j = t + v * tpr;
        xr[v] = j < hv ? lds16(xs + j * VEC) : make_uint4(0u, 0u, 0u, 0u);
      }
      if constexpr (NT == 2) {
        const T* rs = staged_row<T>(m, c, NT, s, 1, g);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int j = t + v * tpr;
          rr[v] = j < hv ? lds16(rs + j * VEC) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if constexpr (KIND == KIND_LN) pivot = load_elem<D>(xs, 0);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&m.empty[s]);  // the row is in registers: the stage may be refilled
    const int par = parity;
    parity ^= 1;
    if (!mine) continue;

    float2 f[VPT][VP];
#pragma unroll
    for (int v = 0; v < VPT; ++v) unpack2<D>(xr[v], f[v]);
    if constexpr (KIND == KIND_FUSED) {
      T* hrow = reinterpret_cast<T*>(a.h) + row * a.ldh;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        float2 r[VP];
        unpack2<D>(rr[v], r);
#pragma unroll
        for (int p = 0; p < VP; ++p) f[v][p] = add2(f[v][p], r[p]);
        if (v < nvec && have) st_vec(hrow + (t + v * tpr) * VEC, pack2<D>(f[v]));
      }
    }
    float rstd, mean_d = 0.f;
    if constexpr (KIND == KIND_LN) {
      const float2 pv = splat2(pivot);
      float2 s2 = splat2(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (v < nvec) {
#pragma unroll
          for (int p = 0; p < VP; ++p) f[v][p] = sub2(f[v][p], pv);
          float2 vs = f[v][0];
#pragma unroll
          for (int p = 1; p < VP; ++p) vs = add2(vs, f[v][p]);
          s2 = add2(s2, vs);
        }
      }
      const float cnt = (float)(nvec * VEC);
      const float mloc = nvec > 0 ? __fdividef(s2.x + s2.y, cnt) : 0.f;
      const float2 ml = splat2(mloc);
      float2 q2 = splat2(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (v < nvec) {
          float2 e = sub2(f[v][0], ml);
          float2 vq = mul2(e, e);
#pragma unroll
          for (int p = 1; p < VP; ++p) {
            e = sub2(f[v][p], ml);
            vq = fma2(e, e, vq);
          }
          q2 = add2(q2, vq);
        }
      }
      const Welford w = group_welford(Welford{cnt, mloc, q2.x + q2.y}, sh, nwg, wig, lane, bar_id, par);
      mean_d = w.m;
      rstd = rsqrtf(w.m2 * inv_h + a.eps);
    } else {
      float2 s2 = splat2(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (v < nvec) {
          float2 vq = mul2(f[v][0], f[v][0]);
#pragma unroll
          for (int p = 1; p < VP; ++p) vq = fma2(f[v][p], f[v][p], vq);
          s2 = add2(s2, vq);
        }
      }
      float ss[1] = {s2.x + s2.y};
      group_sum<1>(ss, sh, nwg, wig, lane, bar_id, par);
      rstd = rsqrtf(ss[0] * inv_h + a.eps);
    }
    if (t == 0 && have) {
      if constexpr (KIND == KIND_LN) {
        if (a.mean) a.mean[row] = pivot + mean_d;
      }
      if (a.rstd) a.rstd[row] = rstd;
    }
    T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy;
    const float2 r2 = splat2(rstd);
    const float2 b2 = splat2(-mean_d * rstd);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (v < nvec) {
        const int col = (t + v * tpr) * VEC;
        float2 gm[VP], out[VP];
        read_pairs<VEC>(gs, v, t, tpr, gm);
        if constexpr (KIND == KIND_LN) {
          float2 be[VP];
          read_pairs<VEC>(bs, v, t, tpr, be);
#pragma unroll
          for (int p = 0; p < VP; ++p) out[p] = fma2(fma2(f[v][p], r2, b2), gm[p], be[p]);
        } else {
#pragma unroll
          for (int p = 0; p < VP; ++p) out[p] = mul2(mul2(f[v][p], r2), gm[p]);
        }
        if (have) st_vec(yrow + col, pack2<D>(out));
      }
    }
  }
}

constexpr int LOOP_THREADS = 256;

template <int KIND, typename D>
__global__ void __launch_bounds__(LOOP_THREADS) fwd_loop_kernel(const FwdArgs a) {
  using T = typename D::T;
  __shared__ float sh[2 * (LOOP_THREADS / 32) * 3];
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int wig = t >> 5;
  constexpr int NW = LOOP_THREADS / 32;
  const int H = a.H;
  const bool w_f32 = a.w_f32 != 0;
  int parity = 0;

  for (int64_t row = blockIdx.x; row < a.N; row += gridDim.x) {
    const T* xrow = reinterpret_cast<const T*>(a.x) + row * a.ldx;
    float rstd, mean_d = 0.f, pivot = 0.f;
    if constexpr (KIND == KIND_LN) {
      pivot = load_elem<D>(xrow, 0);
      // Welford's online recurrence ("Skill: Write CUDA LayerNorm Kernel",
      // step 2) over this thread's strided elements.
      Welford w{0.f, 0.f, 0.f};
      for (int j = t; j < H; j += LOOP_THREADS) {
        const float d = load_elem<D>(xrow, j) - pivot;
        w.n += 1.f;
        const float old = w.m;
        w.m = old + (d - old) / w.n;
        w.m2 = fmaf(d - old, d - w.m, w.m2);
      }
      w = group_welford(w, sh, NW, wig, lane, 1, parity);
      mean_d = w.m;
      rstd = rsqrtf(w.m2 / (float)H + a.eps);
    } else {
      float ss[1] = {0.f};
      if constexpr (KIND == KIND_FUSED) {
        // h is only summed here; it is stored in the second pass, so that
        // pass can still re-form the fp32 sum when h_out aliases an input.
        const T* rrow = reinterpret_cast<const T*>(a.res) + row * a.ldr;
        for (int j = t; j < H; j += LOOP_THREADS) {
          const float h = load_elem<D>(xrow, j) + load_elem<D>(rrow, j);
          ss[0] = fmaf(h, h, ss[0]);
        }
      } else {
        for (int j = t; j < H; j += LOOP_THREADS) {
          const float v = load_elem<D>(xrow, j);
          ss[0] = fmaf(v, v, ss[0]);
        }
      }
      group_sum<1>(ss, sh, NW, wig, lane, 1, parity);
      rstd = rsqrtf(ss[0] / (float)H + a.eps);
    }
    if (t == 0) {
      if constexpr (KIND == KIND_LN) {
        if (a.mean) a.mean[row] = pivot + mean_d;
      }
      if (a.rstd) a.rstd[row] = rstd;
    }

    T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy;
    for (int j = t; j < H; j += LOOP_THREADS) {
      const float g = a.gamma ? load_param<D>(a.gamma, j, w_f32) : 1.f;
      float out;
      if constexpr (KIND == KIND_LN) {
        const float b = a.beta ? load_param<D>(a.beta, j, w_f32) : 0.f;
        out = fmaf((load_elem<D>(xrow, j) - pivot - mean_d) * rstd, g, b);
      } else if constexpr (KIND == KIND_FUSED) {
        // Element j of x and residual is read, and h_out[j] written, by this
        // thread only, so storing h here is safe when h_out aliases an input.
        const float h = load_elem<D>(xrow, j) + load_elem<D>(reinterpret_cast<const T*>(a.res) + row * a.ldr, j);
        store_elem<D>(reinterpret_cast<T*>(a.h) + row * a.ldh, j, h);
        out = (h * rstd) * g;
      } else {
        out = (load_elem<D>(xrow, j) * rstd) * g;
      }
      store_elem<D>(yrow, j, out);
    }
    parity ^= 1;
  }
}

// ---------------------------------------------------------------------------
// Host-side configuration.
// ---------------------------------------------------------------------------

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Persistent grid for the row kernels: as many CTAs as fit on the GPU at
// once (queried per kernel), or fewer when there are fewer row groups.
template <typename K>
static int64_t persistent_blocks(K kern, int threads, size_t smem, const DeviceInfo& dev, int64_t want) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)per_sm * dev.sm_count));
}

template <typename K>
static cudaError_t launch_rows(K kern, const FwdArgs& a, int threads, size_t smem, const DeviceInfo& dev,
                               int64_t groups, cudaStream_t s) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)persistent_blocks(kern, threads, smem, dev, groups), threads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int KIND, typename D, int VPT>
static cudaError_t run_rows(const FwdArgs& a, int threads, int rpc, size_t smem, const DeviceInfo& dev,
                            cudaStream_t s) {
  const int64_t groups = (a.N + rpc - 1) / rpc;
  // One warp a row at 32 elements a lane: three CTAs an SM (80 registers, no
  // spills) keep more rows in flight than two (measured 8192x1024 bf16 LN
  // 12.7 -> 12.3 us, RMS 10.9 -> 10.6); wider rows keep two.
  if (threads <= 256 && VPT * D::VEC > 16 && a.tpr == 32)
    return launch_rows(fwd_rows_kernel<KIND, D, VPT, 256, 3>, a, threads, smem, dev, groups, s);
  if (threads <= 256)
    return launch_rows(fwd_rows_kernel<KIND, D, VPT, 256, (VPT * D::VEC > 16 ? 2 : 3)>, a, threads, smem, dev,
                       groups, s);
  if (threads <= 640) return launch_rows(fwd_rows_kernel<KIND, D, VPT, 640, 1>, a, threads, smem, dev, groups, s);
  return launch_rows(fwd_rows_kernel<KIND, D, VPT, 1024, 1>, a, threads, smem, dev, groups, s);
}

// Clusters of CL CTAs a row: as many clusters as can be resident at once, at
// most one a row.
// Wide-chunk rows.  One warp a row: RMSNorm keeps three CTAs an SM (80
// registers); LayerNorm two, where its 126 registers do not spill (measured
// 8192x1024 bf16 12.4 -> 10.7 us, 32768x1024 24.7 -> 22.6 against three CTAs
// at 80 registers with spills).
template <int KIND, typename D, int NCH>
static cudaError_t run_wide(const FwdArgs& a, int threads, int rpc, size_t smem, const DeviceInfo& dev,
                            cudaStream_t s) {
  const int64_t groups = (a.N + rpc - 1) / rpc;
  constexpr int W1_MINB = KIND == KIND_LN ? 2 : 3;
  if constexpr (KIND == KIND_FUSED) {  // 16 columns a thread up to 640 threads, three CTAs an SM when they fit
    if (threads <= 256) return launch_rows(fwd_wide_kernel<KIND, D, NCH, 256, 3>, a, threads, smem, dev, groups, s);
    return launch_rows(fwd_wide_kernel<KIND, D, NCH, 640, 1>, a, threads, smem, dev, groups, s);
  } else if constexpr (NCH == 1) {  // one chunk a lane: one-warp rows only
    return launch_rows(fwd_wide_kernel<KIND, D, NCH, 256, W1_MINB>, a, threads, smem, dev, groups, s);
  } else {
    if (a.tpr == 32) return launch_rows(fwd_wide_kernel<KIND, D, NCH, 256, W1_MINB>, a, threads, smem, dev, groups, s);
    if (threads <= 256) return launch_rows(fwd_wide_kernel<KIND, D, NCH, 256, 2>, a, threads, smem, dev, groups, s);
    return launch_rows(fwd_wide_kernel<KIND, D, NCH, 640, 1>, a, threads, smem, dev, groups, s);
  }
}

template <int KIND, typename D, int VPT, int CL>
static cudaError_t run_rows_cluster(const FwdArgs& a, int threads, size_t smem, cudaStream_t s) {
  auto kern = fwd_rows_kernel<KIND, D, VPT, 512, 1, CL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t want = std::max<int64_t>(1, std::min<int64_t>(a.N, 1 << 20));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * (unsigned)want);
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
  cfg.gridDim = dim3(CL * (unsigned)std::min<int64_t>(want, resident));
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KIND, typename D, int VPT>
static cudaError_t run_staged(const FwdArgs& a, const StageCfg& c, int64_t blocks, size_t smem, cudaStream_t s) {
  auto kern = fwd_staged_kernel<KIND, D, VPT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)blocks, kStagedThreads, smem, s>>>(a, c);
  return cudaGetLastError();
}

template <int KIND, typename D>
cudaError_t launch_fwd_typed(FwdArgs a, const DeviceInfo& dev, cudaStream_t s) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  // Elements a thread: 32 for bf16 LayerNorm/RMSNorm (halves the per-row
  // reduction overhead per element), else 16 (fused keeps two rows' inputs in
  // flight; fp32 takes twice the registers per element).
  constexpr int VPT_MAX = (KIND != KIND_FUSED && VEC == 8) ? 4 : 16 / VEC;
  const size_t es = sizeof(T);
  a.err = dev.err;
  bool aligned = aligned16(a.x) && aligned16(a.y) && (a.ldx * es) % 16 == 0 && (a.ldy * es) % 16 == 0;
  if (a.gamma) aligned = aligned && aligned16(a.gamma);
  if (a.beta) aligned = aligned && aligned16(a.beta);
  if (KIND == KIND_FUSED) {
    aligned = aligned && aligned16(a.res) && aligned16(a.h) && (a.ldr * es) % 16 == 0 &&
              (a.ldh * es) % 16 == 0;
  }
  // Register-row shape: narrow rows one warp each (VPT = smallest power of
  // two covering H), wider rows 16 elements a thread with more warps.
  const bool vec_ok = aligned && a.H % VEC == 0;
  const int Hv = a.H / VEC;
  int vpt = VPT_MAX, tpr = 0;
  if (Hv <= 32 * VPT_MAX) {
    tpr = 32;
    vpt = 1;
    while (vpt * 32 < Hv) vpt *= 2;
  } else {
    tpr = ((Hv + VPT_MAX - 1) / VPT_MAX + 31) / 32 * 32;
  }
  const int rpc_rows = tpr <= 256 ? 256 / tpr : 1;
  // group scratch, then fp32 gamma (and beta) for vpt vectors of tpr threads
  const size_t rows_smem = (((size_t)rpc_rows * 2 * (tpr / 32) * 3 + 3) & ~(size_t)3) * sizeof(float) +
                           (KIND == KIND_LN ? 2 : 1) * (size_t)vpt * VEC * tpr * sizeof(float);
  const bool rows_ok = vec_ok && tpr <= 1024 && rows_smem <= (size_t)dev.max_smem_optin;
  StageCfg c{};
  constexpr int NT = KIND == KIND_FUSED ? 2 : 1;
  // Staged consumers keep at most 8 packed vectors of each tensor, and fp32
  // copies of gamma (and beta) in shared memory.
  const bool staged_ok = vec_ok && staged_config(a.H, (int)es, NT, dev.max_smem_optin, (8 / NT) * VEC, &c,
                                                 KIND == KIND_LN ? 2 : 1);
  bool use_rows = false, use_staged = false, wide_rows = false;
  switch (dev.path) {
    case PATH_AUTO:
      // Rows of more than 640 threads: the bulk-copy ring where it fits, then
      // cluster rows (below), and one CTA of up to 1024 threads only for widths
      // no cluster split divides (its 32-element threads spill; measured: LN
      // 2048x24576 bf16 62.5 -> 49.3 us with clusters, fp32 fused 2048x16384
      // 98.9 -> 85.2, RMS 2048x24576 43.4 -> 38.8).
      use_rows = rows_ok && tpr <= kRowsAutoMaxThreads;
      use_staged = !use_rows && staged_ok;
      wide_rows = !use_rows && !use_staged && rows_ok;
      break;
    case PATH_ROWS: use_rows = rows_ok; break;
    case PATH_STAGED:
      use_staged = staged_ok;
      use_rows = !use_staged && rows_ok;
      break;
    default: break;
  }
  if (use_staged) {
    c.err = dev.err;
    c.contiguous = a.ldx == a.H && (NT == 1 || a.ldr == a.H);
    const int stpr = 32 * (c.W / c.G);
    const int svpt = (Hv + stpr - 1) / stpr;
    const size_t smem = staged_smem_bytes(c, NT);
    const int64_t blocks = std::min<int64_t>((int64_t)dev.sm_count, (a.N + c.G - 1) / c.G);
    if (svpt <= 1) return run_staged<KIND, D, 1>(a, c, blocks, smem, s);
    if (svpt <= 2) return run_staged<KIND, D, 2>(a, c, blocks, smem, s);
    if (svpt <= 3) return run_staged<KIND, D, 3>(a, c, blocks, smem, s);
    if (svpt <= 4) return run_staged<KIND, D, 4>(a, c, blocks, smem, s);
    if constexpr (NT == 1) {
      if (svpt <= 5) return run_staged<KIND, D, 5>(a, c, blocks, smem, s);
      if (svpt <= 6) return run_staged<KIND, D, 6>(a, c, blocks, smem, s);
      return run_staged<KIND, D, 8>(a, c, blocks, smem, s);
    }
  }
  // Half-precision rows of at least 512 columns take the wide-chunk kernel
  // where rows are 32-byte aligned (measured against the 16-byte register
  // rows: LayerNorm 8192x5120 bf16 31.1 -> 29.4 us, 2048x16384 29.3 -> 28.7,
  // 4096x8192 26.6 -> 25.9; RMSNorm 8192x5120 26.4 -> 25.5; the fused add
  // 8192x1024 14.1 -> 13.6, 8192x5120 51.5 -> 49.7, 32768x1024 41.3 -> 39.7).
  if constexpr (VEC == 8) {
    auto al32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    bool aligned32 = al32(a.x) && al32(a.y) && (a.ldx * es) % 32 == 0 && (a.ldy * es) % 32 == 0;
    if (KIND == KIND_FUSED)
      aligned32 = aligned32 && al32(a.res) && al32(a.h) && (a.ldr * es) % 32 == 0 && (a.ldh * es) % 32 == 0;
    if (use_rows && aligned32 && a.H >= 2 * kWideCols * 16 && a.H % kWideCols == 0) {
      const int hc = a.H / kWideCols;
      // The fused add keeps two tensors' next chunks in registers: one chunk a
      // thread while the row fits 640 threads.
      const bool one = KIND == KIND_FUSED ? true : hc <= 32;
      const int nch = one ? 1 : 2;
      const int wtpr = one ? (hc + 31) / 32 * 32 : (hc <= 64 ? 32 : ((hc + 1) / 2 + 31) / 32 * 32);
      // (fused rows past 640 threads fall through to the kernels below)
      const int wrpc = wtpr <= 256 ? 256 / wtpr : 1;
      const size_t wsmem = (((size_t)wrpc * 2 * (wtpr / 32) * 3 + 3) & ~(size_t)3) * sizeof(float) +
                           (size_t)wtpr * (nch == 1 ? wide_slot<1>() : wide_slot<2>()) * sizeof(float);
      if (wtpr <= kRowsAutoMaxThreads && wsmem <= (size_t)dev.max_smem_optin) {
        a.tpr = wtpr;
        if (nch == 1) return run_wide<KIND, D, 1>(a, wrpc * wtpr, wrpc, wsmem, dev, s);
        if constexpr (KIND != KIND_FUSED) return run_wide<KIND, D, 2>(a, wrpc * wtpr, wrpc, wsmem, dev, s);
      }
    }
  }
  if (use_rows) {
    a.tpr = tpr;
    const int rpc = rpc_rows;
    const int threads = rpc * tpr;
    const size_t smem = rows_smem;
    switch (vpt) {
      case 1: return run_rows<KIND, D, 1>(a, threads, rpc, smem, dev, s);
      case 2: return run_rows<KIND, D, 2>(a, threads, rpc, smem, dev, s);
      default:
        if constexpr (VPT_MAX >= 4) return run_rows<KIND, D, 4>(a, threads, rpc, smem, dev, s);
        break;
    }
  }
  // Rows neither one CTA's registers and shared memory nor the bulk-copy ring
  // can hold (H past about 16384): clusters of 2, 4 or 8 CTAs a row, at most
  // 512 threads a part, before the loop, which reads each row twice.
  if (vec_ok && dev.path != PATH_LOOP) {
    for (int parts = 2; parts <= 8; parts *= 2) {
      if (a.H % (parts * VEC) != 0) continue;
      const int ptpr = ((Hv / parts + VPT_MAX - 1) / VPT_MAX + 31) / 32 * 32;
      const size_t psmem = (((size_t)2 * (ptpr / 32) * 3 + 3) & ~(size_t)3) * sizeof(float) +
                           (KIND == KIND_LN ? 2 : 1) * (size_t)VPT_MAX * VEC * ptpr * sizeof(float);
      if (ptpr > 512 || psmem > (size_t)dev.max_smem_optin) continue;
      a.tpr = ptpr;
      if (parts == 2) return run_rows_cluster<KIND, D, VPT_MAX, 2>(a, ptpr, psmem, s);
      if (parts == 4) return run_rows_cluster<KIND, D, VPT_MAX, 4>(a, ptpr, psmem, s);
      return run_rows_cluster<KIND, D, VPT_MAX, 8>(a, ptpr, psmem, s);
    }
  }
  if (wide_rows) {
    a.tpr = tpr;
    switch (vpt) {
      case 1: return run_rows<KIND, D, 1>(a, tpr, 1, rows_smem, dev, s);
      case 2: return run_rows<KIND, D, 2>(a, tpr, 1, rows_smem, dev, s);
      default:
        if constexpr (VPT_MAX >= 4) return run_rows<KIND, D, 4>(a, tpr, 1, rows_smem, dev, s);
        break;
    }
  }
  const int64_t blocks = std::min<int64_t>(a.N, (int64_t)dev.sm_count * 8);
  fwd_loop_kernel<KIND, D><<<(unsigned)blocks, LOOP_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace normk
