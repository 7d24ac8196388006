// Forward kernels: LayerNorm, RMSNorm and fused residual-add + RMSNorm.
//
// Three kernel families, tried in this order:
//
// * fwd_staged_kernel -- persistent, one CTA per SM; a producer warp streams
//   rows through a shared-memory ring with bulk copies (see staged.cuh) and
//   consumer row groups compute from shared memory.  Needs 16-byte aligned
//   rows, H a multiple of the vector width and at least three stages of rows
//   in shared memory.
// * fwd_reg_kernel -- the row lives in registers.  A "row group" of `tpr`
//   threads (one warp for narrow rows, up to 1024 threads for wide rows) owns
//   one row at a time; each thread holds VPT 16-byte vectors of it, so HBM is
//   read exactly once and written exactly once.  Vector v of thread t covers
//   columns [(v*tpr + t)*VEC, +VEC): consecutive threads touch consecutive
//   16-byte chunks, so every warp-wide access is fully coalesced.  Needs
//   16-byte aligned rows and H a multiple of the vector width.
// * fwd_loop_kernel -- any H and any alignment: one CTA per row, a strided
//   loop over the row, a statistics pass and an output pass (the second read
//   mostly hits L2).  Per-thread statistics use Welford's recurrence.  The
//   fused kernel stores h in the output pass, after re-forming the fp32 sum.
//
// Statistics ("Skill: Write CUDA LayerNorm Kernel", Required reasoning process
// steps 2-5; "Skill: Write a Triton LayerNorm Kernel" steps 3-7):
// LayerNorm keeps a Welford triple (count, mean, M2) per thread, merges it
// across lanes with shuffles and across warps through shared memory with the
// parallel merge, and divides M2 by the full row length H.  Values are shifted
// by the row's first element before accumulating (x - x0 is exact when the
// two are close), so rows with a large common offset keep full precision.
// RMSNorm sums x^2.  rstd = rsqrt(var + eps): eps inside the square root.
//
// Fused add ("Skill: Write a Triton Fused Add+RMSNorm Kernel", steps 2-7):
// h = x + residual in fp32, h stored (rounded to the row dtype) before the
// reduction, y computed from the fp32 h.  Each element of h is written by the
// thread that read that element of x and residual, so h_out may alias either.

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "staged.cuh"

namespace normk {

template <int KIND, typename D, int VPT, int MAXT>
__global__ void __launch_bounds__(MAXT) fwd_reg_kernel(const FwdArgs a) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  extern __shared__ float sh_dyn[];
  const int tpr = a.tpr;
  const int rpc = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const int nw = tpr >> 5;
  const int wig = t >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const float inv_h = 1.f / (float)H;
  const bool w_f32 = a.w_f32 != 0;
  float* sh = sh_dyn + slot * (2 * nw * 3);
  const int bar_id = 1 + slot;
  const int64_t stride = (int64_t)gridDim.x * rpc;
  int parity = 0;

  for (int64_t row = (int64_t)blockIdx.x * rpc + slot; row < a.N; row += stride) {
    const T* xrow = reinterpret_cast<const T*>(a.x) + row * a.ldx;
    // Issue every 16-byte load of the row before the first use.
    uint4 raw[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) raw[v] = load_vec_or_zero<D>(xrow, (v * tpr + t) * VEC, H);
    float f[VPT][VEC];
    if constexpr (KIND == KIND_FUSED) {
      const T* rrow = reinterpret_cast<const T*>(a.res) + row * a.ldr;
      uint4 rraw[VPT];
#pragma unroll
      for (int v = 0; v < VPT; ++v) rraw[v] = load_vec_or_zero<D>(rrow, (v * tpr + t) * VEC, H);
      T* hrow = reinterpret_cast<T*>(a.h) + row * a.ldh;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = (v * tpr + t) * VEC;
        float r[VEC];
        unpack<D>(raw[v], f[v]);
        unpack<D>(rraw[v], r);
#pragma unroll
        for (int i = 0; i < VEC; ++i) f[v][i] += r[i];
        if (c < H) store_vec<D>(hrow, c, f[v]);
      }
    } else {
#pragma unroll
      for (int v = 0; v < VPT; ++v) unpack<D>(raw[v], f[v]);
    }

    float rstd, mean_d = 0.f, pivot = 0.f;
    if constexpr (KIND == KIND_LN) {
      pivot = load_elem<D>(xrow, 0);
      // This thread's Welford triple by two passes over its own values, then
      // the parallel merge across the row group.
      int nvec = 0;
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if ((v * tpr + t) * VEC < H) {
          ++nvec;
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            f[v][i] -= pivot;
            s += f[v][i];
          }
        }
      }
      const float cnt = (float)(nvec * VEC);
      const float m = nvec > 0 ? s / cnt : 0.f;
      float m2 = 0.f;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if ((v * tpr + t) * VEC < H) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            const float e = f[v][i] - m;
            m2 = fmaf(e, e, m2);
          }
        }
      }
      const Welford w = group_welford(Welford{cnt, m, m2}, sh, nw, wig, lane, bar_id, parity);
      mean_d = w.m;
      rstd = rsqrtf(w.m2 * inv_h + a.eps);
    } else {
      float ss[1] = {0.f};
#pragma unroll
      for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) ss[0] = fmaf(f[v][i], f[v][i], ss[0]);
      group_sum<1>(ss, sh, nw, wig, lane, bar_id, parity);
      rstd = rsqrtf(ss[0] * inv_h + a.eps);
    }

    if (t == 0) {
      if constexpr (KIND == KIND_LN) {
        if (a.mean) a.mean[row] = pivot + mean_d;
      }
      if (a.rstd) a.rstd[row] = rstd;
    }

    T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * tpr + t) * VEC;
      if (c >= H) continue;
      float g[VEC], out[VEC];
      load_param_vec<D>(a.gamma, c, w_f32, 1.f, g);
      if constexpr (KIND == KIND_LN) {
        float b[VEC];
        load_param_vec<D>(a.beta, c, w_f32, 0.f, b);
#pragma unroll
        for (int i = 0; i < VEC; ++i) out[i] = fmaf((f[v][i] - mean_d) * rstd, g[i], b[i]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) out[i] = (f[v][i] * rstd) * g[i];
      }
      store_vec<D>(yrow, c, out);
    }
    parity ^= 1;
  }
}


#ifndef NORM_STAGED_MAX_STAGES
#define NORM_STAGED_MAX_STAGES 6
#endif

bool staged_config(int H, int es, int NT, int max_smem, int max_cols, StageCfg* c) {
  const int row_bytes = H * es;
  if (H <= 0 || row_bytes % 16 != 0) return false;
  const int vec = 16 / es;
  const int hv = H / vec;
  c->W = kStagedConsumerWarps;
  c->row_bytes = row_bytes;
  c->red_off = 256;                                   // barriers + abort flag
  c->data_off = c->red_off + 2 * c->W * 3 * 4 + 256;  // scratch, rounded up
  c->data_off = (c->data_off + 127) & ~127;
  for (int G = c->W; G >= 1; G /= 2) {
    const int tpr = 32 * (c->W / G);
    const int cols = ((hv + tpr - 1) / tpr) * vec;
    if (max_cols > 0 && cols > max_cols) continue;
    const size_t stage = (size_t)NT * G * row_bytes;
    const long S = (long)(max_smem - c->data_off) / (long)stage;
    if (S < 3) continue;
    c->G = G;
    c->S = (int)std::min<long>(S, NORM_STAGED_MAX_STAGES);
    return true;
  }
  return false;
}

size_t staged_smem_bytes(const StageCfg& c, int NT) { return c.data_off + (size_t)c.S * NT * c.G * c.row_bytes; }

template <int KIND, typename D>
__global__ void __launch_bounds__(kStagedThreads, 1) fwd_staged_kernel(const FwdArgs a, const StageCfg c) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
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
  int parity = 0;
  int k = 0;
  for (int64_t row0 = lo; row0 < hi; row0 += c.G, ++k) {
    const int s = k % c.S;
    const bool have = mbar_wait(&m.full[s], (k / c.S) & 1, c.err, m.abort);
    const int64_t row = row0 + g;
    if (row < hi) {  // uniform across the row group
      const T* xs = staged_row<T>(m, c, NT, s, 0, g);
      float rstd, mean_d = 0.f, pivot = 0.f;
      if constexpr (KIND == KIND_LN) {
        // This thread's Welford triple by two passes over its vectors, then
        // the parallel merge across the row group.
        pivot = load_elem<D>(xs, 0);
        float sum = 0.f;
        int nvec = 0;
#pragma unroll 4
        for (int j = t; j < hv; j += tpr) {
          float f[VEC];
          unpack<D>(lds16(xs + j * VEC), f);
#pragma unroll
          for (int i = 0; i < VEC; ++i) sum += f[i] - pivot;
          ++nvec;
        }
        const float cnt = (float)(nvec * VEC);
        const float mloc = nvec > 0 ? sum / cnt : 0.f;
        float m2 = 0.f;
#pragma unroll 4
        for (int j = t; j < hv; j += tpr) {
          float f[VEC];
          unpack<D>(lds16(xs + j * VEC), f);
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            const float e = (f[i] - pivot) - mloc;
            m2 = fmaf(e, e, m2);
          }
        }
        const Welford w = group_welford(Welford{cnt, mloc, m2}, sh, nwg, wig, lane, bar_id, parity);
        mean_d = w.m;
        rstd = rsqrtf(w.m2 * inv_h + a.eps);
      } else {
        float ss[1] = {0.f};
        if constexpr (KIND == KIND_FUSED) {
          const T* rs = staged_row<T>(m, c, NT, s, 1, g);
          T* hrow = reinterpret_cast<T*>(a.h) + row * a.ldh;
#pragma unroll 4
          for (int j = t; j < hv; j += tpr) {
            float f[VEC], r[VEC];
            unpack<D>(lds16(xs + j * VEC), f);
            unpack<D>(lds16(rs + j * VEC), r);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
              f[i] += r[i];
              ss[0] = fmaf(f[i], f[i], ss[0]);
            }
            if (have) store_vec<D>(hrow, j * VEC, f);
          }
        } else {
#pragma unroll 4
          for (int j = t; j < hv; j += tpr) {
            float f[VEC];
            unpack<D>(lds16(xs + j * VEC), f);
#pragma unroll
            for (int i = 0; i < VEC; ++i) ss[0] = fmaf(f[i], f[i], ss[0]);
          }
        }
        group_sum<1>(ss, sh, nwg, wig, lane, bar_id, parity);
        rstd = rsqrtf(ss[0] * inv_h + a.eps);
      }
      if (t == 0 && have) {
        if constexpr (KIND == KIND_LN) {
          if (a.mean) a.mean[row] = pivot + mean_d;
        }
        if (a.rstd) a.rstd[row] = rstd;
      }
      T* yrow = reinterpret_cast<T*>(a.y) + row * a.ldy;
      const T* rs = KIND == KIND_FUSED ? staged_row<T>(m, c, NT, s, 1, g) : nullptr;
#pragma unroll 4
      for (int j = t; j < hv; j += tpr) {
        float f[VEC], gm[VEC], out[VEC];
        unpack<D>(lds16(xs + j * VEC), f);
        load_param_vec<D>(a.gamma, j * VEC, w_f32, 1.f, gm);
        if constexpr (KIND == KIND_LN) {
          float b[VEC];
          load_param_vec<D>(a.beta, j * VEC, w_f32, 0.f, b);
#pragma unroll
          for (int i = 0; i < VEC; ++i) out[i] = fmaf(((f[i] - pivot) - mean_d) * rstd, gm[i], b[i]);
        } else {
          if constexpr (KIND == KIND_FUSED) {
            float r[VEC];
            unpack<D>(lds16(rs + j * VEC), r);
#pragma unroll
            for (int i = 0; i < VEC; ++i) f[i] += r[i];
          }
#pragma unroll
          for (int i = 0; i < VEC; ++i) out[i] = (f[i] * rstd) * gm[i];
        }
        if (have) store_vec<D>(yrow, j * VEC, out);
      }
    }
    parity ^= 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&m.empty[s]);
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

template <int KIND, typename D, int VPT>
static cudaError_t run_reg(const FwdArgs& a, int threads, int64_t blocks, size_t smem, cudaStream_t s) {
  if (threads <= 256) {
    fwd_reg_kernel<KIND, D, VPT, 256><<<(unsigned)blocks, threads, smem, s>>>(a);
  } else {
    fwd_reg_kernel<KIND, D, VPT, 1024><<<(unsigned)blocks, threads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

// Register path: rows 16-byte aligned and H a multiple of the vector width.
// Narrow rows get one warp each (VPT = smallest power of two covering H, up to
// 32 elements per thread, 8 rows per 256-thread CTA); wider rows keep 32
// elements per thread and add warps: tpr = ceil(H / 32) rounded up to a warp,
// up to 1024 threads (H <= 32768).  Everything else takes the loop path.
template <int KIND, typename D>
static cudaError_t launch_fwd_typed(FwdArgs a, const DeviceInfo& dev, cudaStream_t s) {
  using T = typename D::T;
  constexpr int VEC = D::VEC;
  constexpr int VPT_MAX = 32 / VEC;
  const size_t es = sizeof(T);
  bool aligned = aligned16(a.x) && aligned16(a.y) && (a.ldx * es) % 16 == 0 && (a.ldy * es) % 16 == 0;
  if (a.gamma) aligned = aligned && aligned16(a.gamma);
  if (a.beta) aligned = aligned && aligned16(a.beta);
  if (KIND == KIND_FUSED) {
    aligned = aligned && aligned16(a.res) && aligned16(a.h) && (a.ldr * es) % 16 == 0 &&
              (a.ldh * es) % 16 == 0;
  }
  if (dev.path <= PATH_STAGED && aligned && a.H % VEC == 0) {
    StageCfg c{};
    constexpr int NT = KIND == KIND_FUSED ? 2 : 1;
    if (staged_config(a.H, (int)es, NT, dev.max_smem_optin, 0, &c)) {
      c.err = dev.err;
      c.contiguous = a.ldx == a.H && (NT == 1 || a.ldr == a.H);
      const size_t smem = staged_smem_bytes(c, NT);
      auto kern = fwd_staged_kernel<KIND, D>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      const int64_t blocks = std::min<int64_t>((int64_t)dev.sm_count, (a.N + c.G - 1) / c.G);
      kern<<<(unsigned)blocks, kStagedThreads, smem, s>>>(a, c);
      return cudaGetLastError();
    }
  }
  if (dev.path <= PATH_REGISTER && aligned && a.H % VEC == 0) {
    const int Hv = a.H / VEC;
    int vpt, tpr;
    if (Hv <= 32 * VPT_MAX) {
      tpr = 32;
      vpt = 1;
      while (vpt * 32 < Hv) vpt *= 2;
    } else {
      vpt = VPT_MAX;
      tpr = ((Hv + vpt - 1) / vpt + 31) / 32 * 32;
    }
    if (tpr <= 1024) {
      a.tpr = tpr;
      const int rpc = tpr <= 256 ? 256 / tpr : 1;
      const int threads = rpc * tpr;
      const int64_t blocks = std::min<int64_t>((a.N + rpc - 1) / rpc, 0x7fffffff);
      const size_t smem = (size_t)rpc * 2 * (tpr / 32) * 3 * sizeof(float);
      switch (vpt) {
        case 1: return run_reg<KIND, D, 1>(a, threads, blocks, smem, s);
        case 2: return run_reg<KIND, D, 2>(a, threads, blocks, smem, s);
        case 4: return run_reg<KIND, D, 4>(a, threads, blocks, smem, s);
        default:
          if constexpr (VPT_MAX >= 8) return run_reg<KIND, D, 8>(a, threads, blocks, smem, s);
          break;
      }
    }
  }
  const int64_t blocks = std::min<int64_t>(a.N, (int64_t)dev.sm_count * 8);
  fwd_loop_kernel<KIND, D><<<(unsigned)blocks, LOOP_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_forward(int kind, Dtype dt, FwdArgs a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (dt == DT_BF16) {
    switch (kind) {
      case KIND_LN: return launch_fwd_typed<KIND_LN, BF16>(a, dev, s);
      case KIND_RMS: return launch_fwd_typed<KIND_RMS, BF16>(a, dev, s);
      default: return launch_fwd_typed<KIND_FUSED, BF16>(a, dev, s);
    }
  }
  switch (kind) {
    case KIND_LN: return launch_fwd_typed<KIND_LN, F32>(a, dev, s);
    case KIND_RMS: return launch_fwd_typed<KIND_RMS, F32>(a, dev, s);
    default: return launch_fwd_typed<KIND_FUSED, F32>(a, dev, s);
  }
}

}  // namespace normk
