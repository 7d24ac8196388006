// Device helpers shared by the forward and backward kernels of libnorm.
//
// Everything here is bandwidth plumbing: 128- and 256-bit global loads and
// stores, bf16 and fp16 packing, warp-shuffle reductions, the parallel Welford
// merge, mbarriers and bulk copies, and packed fp32 pairs.  The normalisation
// arithmetic itself lives in fwd_kernels.cuh and bwd_kernels.cuh.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>
#include <stdint.h>

namespace normk {

// Element types.  VEC = elements per 16-byte vector.
struct F32 {
  using T = float;
  static constexpr int VEC = 4;
};
struct BF16 {
  using T = __nv_bfloat16;
  static constexpr int VEC = 8;
};
struct F16 {
  using T = __half;
  static constexpr int VEC = 8;
};

// ---------------------------------------------------------------------------
// 16-byte global memory access.  Streamed row data is read with an L1
// no-allocate hint (each byte is used once per kernel) and a 256-byte L2
// prefetch hint; parameters (gamma, beta) use the default cached path because
// every row reuses them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_cached(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void st_vec(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// Packing: a 16-byte vector <-> VEC fp32 values (element 0 in the low bits).
// bf16/fp16 -> fp32 is exact; fp32 -> bf16/fp16 rounds to nearest even (fp16
// overflows to infinity past its largest finite value, as IEEE rounding does).
// ---------------------------------------------------------------------------
template <typename D>
__device__ __forceinline__ void unpack(const uint4& u, float* f);

template <>
__device__ __forceinline__ void unpack<F32>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

template <>
__device__ __forceinline__ void unpack<BF16>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16);
  f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16);
  f[7] = __uint_as_float(u.w & 0xffff0000u);
}

template <>
__device__ __forceinline__ void unpack<F16>(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 b = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

template <typename D>
__device__ __forceinline__ uint4 pack(const float* f);

template <>
__device__ __forceinline__ uint4 pack<F32>(const float* f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

template <>
__device__ __forceinline__ uint4 pack<BF16>(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

template <>
__device__ __forceinline__ uint4 pack<F16>(const float* f) {
  return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                    pack_f16x2(f[6], f[7]));
}

// Scalar element access (tails and the unaligned path).
template <typename D>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (sizeof(typename D::T) == 4) {
    return reinterpret_cast<const float*>(base)[i];
  } else if constexpr (std::is_same<typename D::T, __half>::value) {
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
  } else {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  }
}

template <typename D>
__device__ __forceinline__ void store_elem(void* base, int64_t i, float v) {
  if constexpr (sizeof(typename D::T) == 4) {
    reinterpret_cast<float*>(base)[i] = v;
  } else if constexpr (std::is_same<typename D::T, __half>::value) {
    reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
  } else {
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  }
}

// Parameter element (gamma/beta): fp32 or the row dtype, chosen at run time.
template <typename D>
__device__ __forceinline__ float load_param(const void* p, int i, bool w_f32) {
  return w_f32 ? reinterpret_cast<const float*>(p)[i] : load_elem<D>(p, i);
}

// Whole 16-byte vectors of a row (the register path requires H % VEC == 0,
// so a vector is either entirely inside the row or entirely past its end).
template <typename D>
__device__ __forceinline__ uint4 load_vec_or_zero(const void* row, int c, int H) {
  return c < H ? ld_stream(reinterpret_cast<const typename D::T*>(row) + c) : make_uint4(0u, 0u, 0u, 0u);
}

template <typename D>
__device__ __forceinline__ void store_vec(void* row, int c, const float* f) {
  st_vec(reinterpret_cast<typename D::T*>(row) + c, pack<D>(f));
}

// gamma/beta for the full vector at column c: p == nullptr gives `fill` (1 for
// gamma, 0 for beta).  Cached 16-byte loads: every row reuses them.
template <typename D>
__device__ __forceinline__ void load_param_vec(const void* p, int c, bool w_f32, float fill, float* f) {
  constexpr int VEC = D::VEC;
  if (p == nullptr) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) f[i] = fill;
  } else if (w_f32) {
    const float* q = reinterpret_cast<const float*>(p) + c;
#pragma unroll
    for (int k = 0; k < VEC / 4; ++k) unpack<F32>(ld_cached(q + 4 * k), f + 4 * k);
  } else {
    unpack<D>(ld_cached(reinterpret_cast<const typename D::T*>(p) + c), f);
  }
}

// ---------------------------------------------------------------------------
// Reductions.  Every lane of a warp (and every thread of a row group) ends
// with bit-identical results: the butterfly adds are commutative, the Welford
// merge is evaluated with the lower-indexed partner as its left operand, and
// cross-warp partials are folded in warp order.
// ---------------------------------------------------------------------------
template <int K>
__device__ __forceinline__ void warp_sum(float (&v)[K]) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
  }
}

// Butterfly over groups of `p` lanes (p a power of two, 2 <= p <= 32): every
// lane ends with the sum over its group, and lanes holding the same values in
// the same group positions end with identical bits.
template <int K>
__device__ __forceinline__ void warp_sum_pow2(float (&v)[K], int p) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    if (off < p) {
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
    }
  }
}

// Smallest power of two >= n, for 2 <= n <= 32.
__device__ __forceinline__ int pow2_ceil(int n) { return 1 << (32 - __clz(n - 1)); }

// Tree sum of a short array: depth log2(n) instead of an n-long add chain.
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    return tree_sum<N / 2>(v) + tree_sum<N - N / 2>(v + N / 2);
  }
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp stage of a 2- or 3-value sum as a reduce-scatter: at the first levels
// each lane keeps half of the values it carries and sends the other half, so
// the warp's totals end spread over lanes (value k in lane 8k for three
// values, 16k for two) after fewer shuffles than a butterfly per value.
template <int K>
__device__ __forceinline__ float warp_sum_scatter(const float (&v)[K], int lane) {
  static_assert(K == 2 || K == 3, "two or three values");
  if constexpr (K == 3) {
    const bool hi4 = (lane & 16) != 0;
    const float s0 = hi4 ? v[0] : v[2], s1 = hi4 ? v[1] : 0.f;
    float k0 = hi4 ? v[2] : v[0], k1 = hi4 ? 0.f : v[1];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    const bool hi3 = (lane & 8) != 0;
    float k = hi3 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, hi3 ? k0 : k1, 8);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) k += __shfl_xor_sync(0xffffffffu, k, off);
    return k;  // lanes 0-7: value 0, 8-15: value 1, 16-23: value 2 (24-31: nothing)
  } else {
    const bool hi4 = (lane & 16) != 0;
    float k = hi4 ? v[1] : v[0];
    k += __shfl_xor_sync(0xffffffffu, hi4 ? v[0] : v[1], 16);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) k += __shfl_xor_sync(0xffffffffu, k, off);
    return k;  // lanes 0-15: value 0, 16-31: value 1
  }
}

// Sum K values over the `nw` (<= 32) warps of one row group (two or three
// values: the warp stage is the reduce-scatter above, measured LayerNorm
// forward 2048x16384 30.5 -> 28.8 us, backward 8192x1024 17.2 -> 16.7).  `sh` holds
// 2*nw*K floats private to the group; `parity` alternates per row so one
// barrier per row is enough (a buffer is rewritten only after the next row's
// barrier).  After the barrier, lane k picks up warp (k mod P)'s partial, P
// the power of two >= nw (0 past nw), and a butterfly over groups of P lanes
// finishes the sum in log2(P) steps, in a fixed order, identical in every
// thread (each group of P lanes holds the same values).  PW > 0: a power of
// two >= nw known at compile time, taken as P (the butterfly unrolled with no
// per-step tests; lanes past nw add exact zeros, so the sums are those of the
// runtime P up to the sign of a zero total).
template <int K, int PW = 0>
__device__ __forceinline__ void group_sum(float (&v)[K], float* sh, int nw, int wig, int lane,
                                          int bar_id, int parity) {
  float* buf = sh + parity * nw * K;
  if constexpr (K == 2 || K == 3) {
    constexpr int SH = K == 3 ? 3 : 4;  // value k lives in lanes [k << SH, (k + 1) << SH)
    const float part = warp_sum_scatter<K>(v, lane);
    if (nw == 1) {
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] = __shfl_sync(0xffffffffu, part, k << SH);
      return;
    }
    if ((lane & ((1 << SH) - 1)) == 0 && (lane >> SH) < K) buf[wig * K + (lane >> SH)] = part;
  } else {
    warp_sum<K>(v);
    if (nw == 1) return;
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < K; ++k) buf[wig * K + k] = v[k];
    }
  }
  named_barrier(bar_id, nw * 32);
  if constexpr (PW > 0) {
    const int src = lane & (PW - 1);
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = src < nw ? buf[src * K + k] : 0.f;
#pragma unroll
    for (int off = PW >> 1; off > 0; off >>= 1) {
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
    }
  } else {
    const int P = pow2_ceil(nw);
    const int src = lane & (P - 1);
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = src < nw ? buf[src * K + k] : 0.f;
    warp_sum_pow2<K>(v, P);
  }
}

// Welford accumulator (count, mean, M2) and the parallel merge of
// "Skill: Write CUDA LayerNorm Kernel", Required reasoning process step 3
// (n = na + nb, delta = mb - ma, mean = ma + delta*nb/n,
// M2 = M2a + M2b + delta^2*na*nb/n; count 0 is the identity), used below in
// its closed form for K parts.
struct Welford {
  float n, m, m2;
};

// Parallel merge of the 32 lanes' triples in the closed form for K parts:
// N = sum n_k, M = sum n_k m_k / N, M2 = sum (M2_k + n_k (m_k - M)^2) -- the
// pairwise merge applied across all parts at once.  Three shuffle
// all-reductions, no branches; every lane gets the same bits.
// Over groups of `p` lanes (p = 32: the whole warp).
__device__ __forceinline__ Welford warp_welford(Welford w, int p = 32) {
  float v[2] = {w.n, w.n * w.m};
  warp_sum_pow2<2>(v, p);
  const float m = v[0] > 0.f ? __fdividef(v[1], v[0]) : 0.f;
  const float d = w.m - m;
  float q[1] = {fmaf(w.n * d, d, w.m2)};
  warp_sum_pow2<1>(q, p);
  return Welford{v[0], m, q[0]};
}

// The same over the `nw` warps of a row group (buffering as group_sum): lane
// k picks up warp (k mod P)'s triple (the identity, count 0, past nw) and the
// merge runs over groups of P lanes.
__device__ __forceinline__ Welford group_welford(Welford w, float* sh, int nw, int wig, int lane,
                                                 int bar_id, int parity) {
  w = warp_welford(w);
  if (nw == 1) return w;
  float* buf = sh + parity * nw * 3;
  if (lane == 0) {
    buf[wig * 3 + 0] = w.n;
    buf[wig * 3 + 1] = w.m;
    buf[wig * 3 + 2] = w.m2;
  }
  named_barrier(bar_id, nw * 32);
  const int P = pow2_ceil(nw);
  const int src = lane & (P - 1);
  Welford x{0.f, 0.f, 0.f};
  if (src < nw) x = Welford{buf[3 * src], buf[3 * src + 1], buf[3 * src + 2]};
  return warp_welford(x, P);
}

// ---------------------------------------------------------------------------
// Bulk-copy pipeline primitives (sm_90+ PTX, used on sm_103a): mbarriers in
// shared memory, 1-D bulk global->shared copies that complete a transaction
// count on an mbarrier, and programmatic dependent launch.  Every wait is
// bounded by the global nanosecond timer; a wait that runs out records an
// error bit for the host and returns false instead of spinning forever.
// ---------------------------------------------------------------------------
constexpr unsigned kErrWaitTimeout = 1u;
constexpr unsigned kErrBadCopy = 2u;  // a bulk copy failed its bounds check and was skipped
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// The register-row LayerNorm/RMSNorm forward keeps the next row's loads in
// registers; beyond that, the row this many strides ahead is requested into
// L2 by one bulk prefetch per row group (0: off).
#ifndef NORM_L2_PREFETCH_ROWS
#define NORM_L2_PREFETCH_ROWS 2
#endif
constexpr int kL2PrefetchRows = NORM_L2_PREFETCH_ROWS;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// kWaitLimitNs.  On timeout, set kErrWaitTimeout in *err, raise the CTA's
// abort flag and return false.  Once the abort flag is up (another thread's
// wait ran out), later waits give up at once; pass abort == nullptr for a wait
// that must run its full limit regardless (draining copies before exit).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          volatile int* abort,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (abort && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (err) atomicOr(err, kErrWaitTimeout);
      if (abort) *abort = 1;
      return false;
    }
  }
  return true;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is counted on `bar`.
// Ask L2 to start fetching `bytes` (a multiple of 16, 16-byte aligned source)
// of global memory that a later load will want; nothing to wait for.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Row range [lo, hi) of CTA c when N rows are split over `grid` CTAs as
// evenly as possible (range sizes differ by at most one row).
__device__ __forceinline__ void cta_rows(int64_t N, int c, int grid, int64_t& lo, int64_t& hi) {
  lo = N * c / grid;
  hi = N * (c + 1) / grid;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait here until the previous kernel has finished and its
// writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block clusters (sm_90+ PTX): this CTA's rank in its cluster, and the
// cluster-wide barrier (every thread of every CTA of the cluster arrives;
// release/acquire order memory operations before it with those after it).
__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Asynchronous 16-byte store into another CTA of the cluster: `local_dst` and
// `local_bar` are this CTA's addresses of a buffer and an mbarrier at the same
// offsets as the target's; the store counts 16 bytes on the target's
// mbarrier when it lands.  No fence: the target's mbarrier wait orders it.
__device__ __forceinline__ void st_async_cluster_v4(const float* local_dst, const uint64_t* local_bar,
                                                    unsigned rank, float4 v) {
  unsigned dst, bar;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(smem_u32(local_dst)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(smem_u32(local_bar)), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

// The row-sum exchange of cluster rows without a cluster barrier: thread 0
// arms this CTA's mbarrier for the other CL-1 CTAs' 16-byte messages and sends
// this CTA's totals (held by every thread) into row `crank` of `slots` in each
// of them; every thread then waits (bounded) on its own mbarrier and adds the
// CL rows in rank order, its own totals in place of row `crank`, so all CTAs
// end with bit-identical sums.  `slots` ([CL][4] floats) and `bar` alternate
// by row parity; `phase` is the use count of this `bar` modulo 2.  A CTA can
// send its next row's totals only after receiving every CTA's totals of this
// row, so a buffer is never rewritten before it has been read.
template <int K, int CL>
__device__ __forceinline__ bool cluster_group_sum_async(float (&v)[K], float* slots, uint64_t* bar, unsigned phase,
                                                        int crank, unsigned* err, volatile int* abort) {
  static_assert(K <= 4, "four values a rank at most");
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)((CL - 1) * 16));
    const float4 m = make_float4(v[0], K > 1 ? v[K > 1 ? 1 : 0] : 0.f, K > 2 ? v[K > 2 ? 2 : 0] : 0.f,
                                 K > 3 ? v[K > 3 ? 3 : 0] : 0.f);
#pragma unroll
    for (int r = 0; r < CL; ++r)
      if (r != crank) st_async_cluster_v4(slots + crank * 4, bar, (unsigned)r, m);
  }
  const bool ok = mbar_wait(bar, phase, err, abort);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float t = 0.f;
#pragma unroll
    for (int r = 0; r < CL; ++r) t += r == crank ? v[k] : slots[r * 4 + k];
    v[k] = t;
  }
  return ok;
}

// 16-byte shared memory access.
__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(p)));
  return r;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 instructions): two IEEE fp32 operations,
// each rounded exactly as its scalar form, per instruction.  Row data are
// handled as pairs: a 16-byte vector is VEC/2 pairs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long f2_bits(float2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 bits_f2(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// A 16-byte vector as VEC/2 fp32 pairs (pair p holds elements 2p, 2p+1).
template <typename D>
__device__ __forceinline__ void unpack2(const uint4& u, float2* p);

template <>
__device__ __forceinline__ void unpack2<F32>(const uint4& u, float2* p) {
  p[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
  p[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}

template <>
__device__ __forceinline__ void unpack2<BF16>(const uint4& u, float2* p) {
  p[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
  p[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  p[2] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
  p[3] = make_float2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
}

template <>
__device__ __forceinline__ void unpack2<F16>(const uint4& u, float2* p) {
  p[0] = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  p[1] = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  p[2] = __half22float2(*reinterpret_cast<const __half2*>(&u.z));
  p[3] = __half22float2(*reinterpret_cast<const __half2*>(&u.w));
}

template <typename D>
__device__ __forceinline__ uint4 pack2(const float2* p);

template <>
__device__ __forceinline__ uint4 pack2<F32>(const float2* p) {
  return make_uint4(__float_as_uint(p[0].x), __float_as_uint(p[0].y), __float_as_uint(p[1].x),
                    __float_as_uint(p[1].y));
}

template <>
__device__ __forceinline__ uint4 pack2<BF16>(const float2* p) {
  return make_uint4(pack_bf16x2(p[0].x, p[0].y), pack_bf16x2(p[1].x, p[1].y), pack_bf16x2(p[2].x, p[2].y),
                    pack_bf16x2(p[3].x, p[3].y));
}

template <>
__device__ __forceinline__ uint4 pack2<F16>(const float2* p) {
  return make_uint4(pack_f16x2(p[0].x, p[0].y), pack_f16x2(p[1].x, p[1].y), pack_f16x2(p[2].x, p[2].y),
                    pack_f16x2(p[3].x, p[3].y));
}

// ---------------------------------------------------------------------------
// 32-byte global memory access (sm_100+ 256-bit vector loads and stores): one
// instruction moves a thread's 16 half-precision (or 8 fp32) elements.  Loads
// of streamed rows carry the same L1 no-allocate and L2 256-byte hints as
// ld_stream.  Addresses must be 32-byte aligned.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_stream32(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.L1::no_allocate.L2::256B.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

__device__ __forceinline__ void st_vec32(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// 32-bit words <-> fp32 pairs.  A half-precision word holds one pair (element
// 2p in the low half); fp32 takes two words a pair.
template <typename D>
__device__ __forceinline__ float2 word_pair(const uint32_t* w, int p) {
  if constexpr (sizeof(typename D::T) == 4) {
    return make_float2(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
  } else if constexpr (std::is_same<typename D::T, __half>::value) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w[p]));
  } else {
    return make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
  }
}

template <typename D>
__device__ __forceinline__ void pair_word(uint32_t* w, int p, float2 v) {
  if constexpr (sizeof(typename D::T) == 4) {
    w[2 * p] = __float_as_uint(v.x);
    w[2 * p + 1] = __float_as_uint(v.y);
  } else if constexpr (std::is_same<typename D::T, __half>::value) {
    w[p] = pack_f16x2(v.x, v.y);
  } else {
    w[p] = pack_bf16x2(v.x, v.y);
  }
}

// gamma/beta for the full vector at column c as pairs (p == nullptr: fill).
template <typename D>
__device__ __forceinline__ void load_param_pairs(const void* p, int c, bool w_f32, float fill, float2* out) {
  constexpr int VP = D::VEC / 2;
  if (p == nullptr) {
#pragma unroll
    for (int i = 0; i < VP; ++i) out[i] = splat2(fill);
  } else if (w_f32) {
    const float* q = reinterpret_cast<const float*>(p) + c;
#pragma unroll
    for (int k = 0; k < VP / 2; ++k) unpack2<F32>(ld_cached(q + 4 * k), out + 2 * k);
  } else {
    unpack2<D>(ld_cached(reinterpret_cast<const typename D::T*>(p) + c), out);
  }
}

// ---------------------------------------------------------------------------
// Per-CTA fp32 copies of gamma/beta for persistent row kernels.  A thread's
// columns never change, so the parameters are converted once and laid out
// thread-interleaved: float4 slot (v * VEC/4 + q) of thread t sits at
// [slot * tpr + t] and holds columns (t + v*tpr)*VEC + 4q .. +3.  Each thread
// reads only its own slots, with conflict-free 16-byte shared loads.
// ---------------------------------------------------------------------------
template <typename D, int VPT>
__device__ __forceinline__ void stage_params(float4* dst, const void* p, bool w_f32, float fill, int t, int tpr,
                                             int hv) {
  constexpr int VEC = D::VEC;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int j = t + v * tpr;
    float2 pr[VEC / 2];
    if (j < hv) {
      load_param_pairs<D>(p, j * VEC, w_f32, fill, pr);
    } else {
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) pr[i] = splat2(0.f);
    }
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q)
      dst[(v * (VEC / 4) + q) * tpr + t] = make_float4(pr[2 * q].x, pr[2 * q].y, pr[2 * q + 1].x, pr[2 * q + 1].y);
  }
}

// Reciprocals 1/gamma in the same layout (1 where gamma is absent; columns
// past the row get 0).  IEEE division: gamma = 0 gives infinity.
template <typename D, int VPT>
__device__ __forceinline__ void stage_inv_params(float4* dst, const void* p, bool w_f32, int t, int tpr, int hv) {
  constexpr int VEC = D::VEC;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int j = t + v * tpr;
    float2 pr[VEC / 2];
    if (j < hv) {
      load_param_pairs<D>(p, j * VEC, w_f32, 1.f, pr);
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) pr[i] = make_float2(1.f / pr[i].x, 1.f / pr[i].y);
    } else {
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) pr[i] = splat2(0.f);
    }
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q)
      dst[(v * (VEC / 4) + q) * tpr + t] = make_float4(pr[2 * q].x, pr[2 * q].y, pr[2 * q + 1].x, pr[2 * q + 1].y);
  }
}

// The VEC/2 pairs of vector v of this thread from a thread-interleaved array.
template <int VEC>
__device__ __forceinline__ void read_pairs(const float4* src, int v, int t, int tpr, float2* out) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 u = src[(v * (VEC / 4) + q) * tpr + t];
    out[2 * q] = make_float2(u.x, u.y);
    out[2 * q + 1] = make_float2(u.z, u.w);
  }
}

template <int VEC>
__device__ __forceinline__ void write_pairs(float4* dst, int v, int t, int tpr, const float2* in) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q)
    dst[(v * (VEC / 4) + q) * tpr + t] = make_float4(in[2 * q].x, in[2 * q].y, in[2 * q + 1].x, in[2 * q + 1].y);
}

}  // namespace normk
