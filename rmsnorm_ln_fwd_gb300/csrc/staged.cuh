// The bulk-copy row pipeline shared by the staged forward and backward
// kernels.
//
// A persistent CTA owns a contiguous range of rows (ranges differ by at most
// one row across CTAs, so there is no tail wave).  Warp W (the last warp) is
// the producer: one lane streams the range, G rows per stage, into a ring of S
// shared-memory stages with 1-D bulk copies that complete on the stage's
// `full` mbarrier.  Warps 0..W-1 are consumers: they wait on `full`, compute
// from shared memory, write outputs straight to global memory, and arrive on
// the stage's `empty` mbarrier, which the producer waits on before refilling
// the stage.  HBM reads stay in flight independently of the consumers'
// registers or occupancy: up to S stages per SM.
//
// Shared memory: [full[S] | empty[S] | reduction scratch | S stages], each
// stage tensor-major: NT tensors x G rows x row_bytes.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace normk {

struct StagedSmem {
  uint64_t* full;
  uint64_t* empty;
  float* red;
  float4* par;
  unsigned char* data;
  volatile int* abort;
};

__device__ __forceinline__ StagedSmem staged_smem(unsigned char* smem, const StageCfg& c) {
  StagedSmem m;
  m.full = reinterpret_cast<uint64_t*>(smem);
  m.empty = m.full + c.S;
  m.abort = reinterpret_cast<volatile int*>(m.empty + c.S);
  m.red = reinterpret_cast<float*>(smem + c.red_off);
  m.par = reinterpret_cast<float4*>(smem + c.par_off);
  m.data = smem + c.data_off;
  return m;
}

// One thread initialises the barriers; everyone syncs afterwards.
__device__ __forceinline__ void staged_init(const StagedSmem& m, const StageCfg& c) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < c.S; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], c.W);
    }
    *m.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
}

__device__ __forceinline__ size_t staged_stage_bytes(const StageCfg& c, int NT) {
  return (size_t)NT * c.G * c.row_bytes;
}

// The producer lane: stream rows [lo, hi) of NT tensors into the ring, then
// wait (bounded) until every copy it issued has landed, so the CTA never
// exits with a copy still writing its shared memory.
// Every copy is checked against the ring's bounds and 16-byte alignment
// before it is issued; a copy that fails is skipped and kErrBadCopy raised
// (the stage's transaction count is then short, so its waits run out and the
// call is abandoned with kErrWaitTimeout as well).
__device__ __forceinline__ bool copy_ok(const unsigned char* dst, const void* src, size_t bytes,
                                        const unsigned char* ring_lo, const unsigned char* ring_hi) {
  return dst >= ring_lo && dst + bytes <= ring_hi && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                                                      bytes) & 15u) == 0;
}

template <int NT>
__device__ void staged_produce(const StagedSmem& m, const StageCfg& c, const void* const (&src)[NT],
                               const int64_t (&ld)[NT], int64_t lo, int64_t hi, size_t es) {
  const size_t stage_bytes = staged_stage_bytes(c, NT);
  const unsigned char* ring_hi = m.data + (size_t)c.S * stage_bytes;
  int k = 0;
  for (int64_t row0 = lo; row0 < hi; row0 += c.G, ++k) {
    const int s = k % c.S;
    if (k >= c.S && !mbar_wait(&m.empty[s], ((k / c.S) - 1) & 1, c.err, m.abort)) break;
    const int nr = (int)(hi - row0 < (int64_t)c.G ? hi - row0 : (int64_t)c.G);
    mbar_arrive_expect_tx(&m.full[s], (uint32_t)(NT * nr * c.row_bytes));
    unsigned char* st = m.data + (size_t)s * stage_bytes;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const unsigned char* g = reinterpret_cast<const unsigned char*>(src[q]) + (size_t)(row0 * ld[q]) * es;
      unsigned char* dst = st + (size_t)q * c.G * c.row_bytes;
      if (c.contiguous) {
        const size_t bytes = (size_t)nr * c.row_bytes;
        if (copy_ok(dst, g, bytes, m.data, ring_hi)) bulk_g2s(dst, g, (uint32_t)bytes, &m.full[s]);
        else atomicOr(c.err, kErrBadCopy);
      } else {
        for (int r = 0; r < nr; ++r) {
          unsigned char* d = dst + (size_t)r * c.row_bytes;
          const unsigned char* gr = g + (size_t)(r * ld[q]) * es;
          if (copy_ok(d, gr, c.row_bytes, m.data, ring_hi)) bulk_g2s(d, gr, (uint32_t)c.row_bytes, &m.full[s]);
          else atomicOr(c.err, kErrBadCopy);
        }
      }
    }
  }
  // Drain: the last phase armed on each stage must complete before exit.
  for (int s = 0; s < c.S && s < k; ++s) {
    const int last = s + ((k - 1 - s) / c.S) * c.S;
    mbar_wait(&m.full[s], (last / c.S) & 1, c.err, nullptr);
  }
}

// Consumer-side view of one stage: row `g` of tensor q.
template <typename T>
__device__ __forceinline__ const T* staged_row(const StagedSmem& m, const StageCfg& c, int NT, int s, int q, int g) {
  return reinterpret_cast<const T*>(m.data + staged_stage_bytes(c, NT) * s + ((size_t)q * c.G + g) * c.row_bytes);
}

// Host side: pick G (rows per stage) and S (stages) for NT staged tensors of
// row_bytes each, within `max_smem` bytes of shared memory, with at least
// three stages, at most `max_cols` columns per consumer thread (0 = no limit)
// and room for `n_par` fp32 parameter arrays (one value per column a consumer
// thread owns, thread-interleaved).  Returns false when no shape fits.
bool staged_config(int H, int es, int NT, int max_smem, int max_cols, StageCfg* c, int n_par = 0);
size_t staged_smem_bytes(const StageCfg& c, int NT);

}  // namespace normk
