// Per-chunk vectors and decays shared by the chunk kernels (CUDA-core and
// tensor-core variants).
#pragma once

#include "common.cuh"

namespace ssd {
struct ChunkIds {
  int c, h, g, bb, t0;
};

__device__ __forceinline__ ChunkIds chunk_ids(const Problem &pr) {
  ChunkIds id;
  id.c = blockIdx.x;
  id.h = blockIdx.y;
  id.bb = blockIdx.z;
  id.g = id.h / pr.hpg;
  id.t0 = id.c * pr.Q;
  return id;
}

// Shared per-chunk vectors: Acs, dt, seq ids, and three derived weights.
struct ChunkVecs {
  float acs[256], dt[256], em[256], wdt[256], w[256];
  int seq[256];
};

// em[i]  = exp(Acs_i) * [token i continues the state entering the chunk: the
//          sequence of the token before it, or the row's initial state]
// w[j]   = exp(Acs_last - Acs_j) * [token j is in the last token's sequence]
// wdt[j] = w[j] * dt_j
__device__ __forceinline__ void load_chunk_vecs(const Problem &pr, const ChunkIds &id, const float *dtv,
                                                const float *acs, ChunkVecs &v) {
  const float *acs_bh = acs + ((size_t)id.bb * pr.H + id.h) * pr.L + id.t0;
  const float *dt_bh = dtv + ((size_t)id.bb * pr.H + id.h) * pr.L + id.t0;
  const int Q = pr.Q;
  const bool inc = chunk_has_incoming(pr, id.c);
  const int seq_prev = inc ? seq_before_chunk(pr, id.bb, id.c) : 0;
  const int seq_last = seq_of(pr, id.bb, id.t0 + Q - 1);
  const float acs_last = acs_bh[Q - 1];
  for (int i = threadIdx.x; i < Q; i += blockDim.x) {
    const int sq = seq_of(pr, id.bb, id.t0 + i);
    const float a = acs_bh[i], d = dt_bh[i];
    v.acs[i] = a;
    v.dt[i] = d;
    v.seq[i] = sq;
    v.em[i] = (inc && sq == seq_prev) ? expf(a) : 0.f;
    const float w = (sq == seq_last) ? expf(acs_last - a) : 0.f;
    v.w[i] = w;
    v.wdt[i] = w * d;
  }
  __syncthreads();
}

// decay carrying the segment's initial state to the start of chunk c
__device__ __forceinline__ float decay_seg_to_chunk(const Problem &pr, int bb, int h, int c) {
  return __ldg(pr.dstart + dtab_index(pr, bb, h, c));
}

// decay carrying the state at the end of chunk c to the end of its segment
__device__ __forceinline__ float decay_chunk_to_seg_end(const Problem &pr, int bb, int h, int c) {
  return __ldg(pr.dend + dtab_index(pr, bb, h, c));
}

}  // namespace ssd
