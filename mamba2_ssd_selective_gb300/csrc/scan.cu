// Segment summaries and the segment scans (forward and reverse).
//
// Megatron-LM PR #6808 "Add state-passing context parallelism for Mamba2"
// (description): the SSD over one causal segment is affine in its initial
// state, S_out = a_block * S_in + S_ext.  Each segment runs its chunk state
// passing from a zero state, giving (S_ext, a_block); an exclusive causal scan
// over the summaries, in fixed segment order, recovers each segment's true
// initial state.  Backward mirrors it with a reverse boundary scan.
//
// On one GPU the summary exchange is a write to / read from device memory at a
// kernel boundary.  Every element of the P x N state is independent, so each
// thread owns a few elements and walks the chunks (or segments) in order: the
// result is bit-identical from run to run.
#include "kernels.h"
#include "simt_gemm.cuh"

namespace ssd {

constexpr int kScanBatch = 4;  // chunks whose loads are in flight together

// Decay tables of one (b, h): cdec[c] = product of the chunk's per-token decays
// (from Acs and seq_idx), then per segment the exclusive prefix and suffix
// products dstart[c] = prod_{c' in seg, c' < c} cdec[c'], dend[c] = prod_{c' > c}.
__global__ void __launch_bounds__(256) decay_tables_kernel(Problem pr, const float *__restrict__ acs, float *cdec,
                                                           float *dstart, float *dend) {
  const int h = blockIdx.x, bb = blockIdx.y;
  const float *acs_bh = acs + ((size_t)bb * pr.H + h) * pr.L;
  const size_t base = ((size_t)bb * pr.H + h) * pr.nc;
  for (int c = threadIdx.x; c < pr.nc; c += blockDim.x) cdec[base + c] = chunk_decay_raw(pr, acs_bh, bb, c);
  __syncthreads();
  for (int k = threadIdx.x; k < pr.S; k += blockDim.x) {
    const int c0 = k * pr.cps, c1 = c0 + pr.cps;
    float d = 1.f;
    for (int c = c0; c < c1; ++c) {
      dstart[base + c] = d;
      d *= cdec[base + c];
    }
    d = 1.f;
    for (int c = c1 - 1; c >= c0; --c) {
      dend[base + c] = d;
      d *= cdec[base + c];
    }
  }
}

void launch_decay_tables(const Problem &pr, const float *acs, float *cdec, float *dstart, float *dend, cudaStream_t s) {
  decay_tables_kernel<<<dim3(pr.H, pr.b), 256, 0, s>>>(pr, acs, cdec, dstart, dend);
}

// out[b, c, h] = bf16(a[b, c, h] + d * seg[b, k(c), h]) over the P x N state, with
// d = dstart (mode 0: the true state entering the chunk) or dend (mode 1: the
// true state gradient at the chunk end).  8 elements per thread.
__global__ void __launch_bounds__(256) combine_state_kernel(Problem pr, const float *__restrict__ a,
                                                            const float *__restrict__ seg,
                                                            __nv_bfloat16 *__restrict__ out, int mode) {
  const int PN = pr.P * pr.N;
  const int e = (blockIdx.x * 256 + threadIdx.x) * 8;
  const int h = blockIdx.y, bc = blockIdx.z, bb = bc / pr.nc, c = bc % pr.nc, k = c / pr.cps;
  if (e >= PN) return;
  const float d = mode == 0 ? __ldg(pr.dstart + dtab_index(pr, bb, h, c)) : __ldg(pr.dend + dtab_index(pr, bb, h, c));
  const size_t co = (((size_t)bb * pr.nc + c) * pr.H + h) * PN + e;
  const size_t so = (((size_t)bb * pr.S + k) * pr.H + h) * PN + e;
  const float4 a0 = *reinterpret_cast<const float4 *>(a + co), a1 = *reinterpret_cast<const float4 *>(a + co + 4);
  const float4 s0 = *reinterpret_cast<const float4 *>(seg + so), s1 = *reinterpret_cast<const float4 *>(seg + so + 4);
  const float v[8] = {a0.x + d * s0.x, a0.y + d * s0.y, a0.z + d * s0.z, a0.w + d * s0.w,
                      a1.x + d * s1.x, a1.y + d * s1.y, a1.z + d * s1.z, a1.w + d * s1.w};
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&b2);
  }
  *reinterpret_cast<uint4 *>(out + co) = make_uint4(w[0], w[1], w[2], w[3]);
}

void launch_combine_state(const Problem &pr, const float *a, const float *seg, __nv_bfloat16 *out, int mode,
                          cudaStream_t s) {
  dim3 grid((pr.P * pr.N / 8 + 255) / 256, pr.H, pr.b * pr.nc);
  combine_state_kernel<<<grid, 256, 0, s>>>(pr, a, seg, out, mode);
}

// Backward form of the combination, one block per (row, chunk, head): the true
// state entering the chunk S_in = S_loc + dstart * S_seg and the true state
// gradient at its end dS = dS_loc + dend * G_out, both written in bf16 (the
// tensor-core operands), and in fp32 the chunk's decay term of the dt adjoint
//   sdot[b, c, h] = a_c <dS, S_in>
// summed in a fixed order (per thread, then the block tree).
__global__ void __launch_bounds__(256) combine_bwd_kernel(Problem pr, const float *__restrict__ sst,
                                                          const float *__restrict__ segin,
                                                          const float *__restrict__ dsl,
                                                          const float *__restrict__ gout,
                                                          __nv_bfloat16 *__restrict__ sin16,
                                                          __nv_bfloat16 *__restrict__ dse16, float *__restrict__ sdot) {
  __shared__ float red[8];
  const int PN = pr.P * pr.N;
  const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z, k = c / pr.cps;
  const size_t ti = dtab_index(pr, bb, h, c);
  const float dc = __ldg(pr.dstart + ti), de = __ldg(pr.dend + ti), ac = __ldg(pr.cdec + ti);
  const size_t co = (((size_t)bb * pr.nc + c) * pr.H + h) * PN;
  const size_t so = (((size_t)bb * pr.S + k) * pr.H + h) * PN;
  float part = 0.f;
#pragma unroll 4
  for (int e = threadIdx.x * 4; e < PN; e += 256 * 4) {
    const float4 a = *reinterpret_cast<const float4 *>(sst + co + e), b = *reinterpret_cast<const float4 *>(segin + so + e);
    const float4 x = *reinterpret_cast<const float4 *>(dsl + co + e), y = *reinterpret_cast<const float4 *>(gout + so + e);
    const float sv[4] = {a.x + dc * b.x, a.y + dc * b.y, a.z + dc * b.z, a.w + dc * b.w};
    const float gv[4] = {x.x + de * y.x, x.y + de * y.y, x.z + de * y.z, x.w + de * y.w};
    part += gv[0] * sv[0] + gv[1] * sv[1] + gv[2] * sv[2] + gv[3] * sv[3];
    __nv_bfloat162 s01 = __floats2bfloat162_rn(sv[0], sv[1]), s23 = __floats2bfloat162_rn(sv[2], sv[3]);
    __nv_bfloat162 g01 = __floats2bfloat162_rn(gv[0], gv[1]), g23 = __floats2bfloat162_rn(gv[2], gv[3]);
    *reinterpret_cast<uint2 *>(sin16 + co + e) =
        make_uint2(*reinterpret_cast<uint32_t *>(&s01), *reinterpret_cast<uint32_t *>(&s23));
    *reinterpret_cast<uint2 *>(dse16 + co + e) =
        make_uint2(*reinterpret_cast<uint32_t *>(&g01), *reinterpret_cast<uint32_t *>(&g23));
  }
  const float tot = block_sum256(part, red);
  if (threadIdx.x == 0) sdot[((size_t)bb * pr.nc + c) * pr.H + h] = ac != 0.f ? ac * tot : 0.f;
}

void launch_combine_bwd(const Problem &pr, const float *sst, const float *segin, const float *dsl, const float *gout,
                        __nv_bfloat16 *sin16, __nv_bfloat16 *dse16, float *sdot, cudaStream_t s) {
  combine_bwd_kernel<<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, sst, segin, dsl, gout, sin16, dse16, sdot);
}

// Local pass of segment k: S <- a_c * S + Sc[c] over the segment's chunks from
// S = 0.  Overwrites sst[c] (the chunk's own state contribution Sc) with the
// local state entering the chunk, and writes S_ext[k] and a_block[k].  Each
// thread owns two 16-byte groups of state elements (kScanVec4 float4, one per
// 256-thread stride, so every warp access stays contiguous), reads the chunk
// decays itself (the same address for the whole block: one broadcast line) and
// keeps the loads of kScanBatch chunks in flight.  No barriers.
constexpr int kScanVec4 = 2;
constexpr int kScanElems4 = 256 * kScanVec4;  // float4 groups per block

__global__ void __launch_bounds__(256) local_pass_kernel(Problem pr, const float *__restrict__ acs,
                                                         float *__restrict__ sst, float *__restrict__ sext,
                                                         float *__restrict__ ablk) {
  const int PN = pr.P * pr.N, PN4 = PN / 4;
  const int h = blockIdx.y, k = blockIdx.z % pr.S, bb = blockIdx.z / pr.S;
  const size_t cstride4 = (size_t)pr.H * PN / 4;  // float4 between consecutive chunks
  float4 *base = reinterpret_cast<float4 *>(sst + (((size_t)bb * pr.nc + (size_t)k * pr.cps) * pr.H + h) * PN);
  int e4[kScanVec4];
  float4 S[kScanVec4];
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u) {
    e4[u] = blockIdx.x * kScanElems4 + u * 256 + threadIdx.x;
    S[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float prod = 1.f;
  for (int c0 = 0; c0 < pr.cps; c0 += kScanBatch) {
    const int nb = min(kScanBatch, pr.cps - c0);
    float dec[kScanBatch];
    float4 v[kScanBatch][kScanVec4];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        dec[q] = chunk_decay(pr, bb, h, k * pr.cps + c0 + q);
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u)
          if (e4[u] < PN4) v[q][u] = base[(size_t)(c0 + q) * cstride4 + e4[u]];
      }
    }
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        const float a = dec[q];
        prod *= a;
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u) {
          if (e4[u] < PN4) {
            base[(size_t)(c0 + q) * cstride4 + e4[u]] = S[u];
            S[u] = make_float4(fmaf(a, S[u].x, v[q][u].x), fmaf(a, S[u].y, v[q][u].y), fmaf(a, S[u].z, v[q][u].z),
                               fmaf(a, S[u].w, v[q][u].w));
          }
        }
      }
    }
  }
  const size_t so = (((size_t)bb * pr.S + k) * pr.H + h);
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u)
    if (e4[u] < PN4) reinterpret_cast<float4 *>(sext + so * PN)[e4[u]] = S[u];
  if (blockIdx.x == 0 && threadIdx.x == 0) ablk[so] = prod;
}

void launch_local_pass(const Problem &pr, const float *acs, float *sst, float *sext, float *ablk, cudaStream_t s) {
  dim3 grid((pr.P * pr.N / 4 + kScanElems4 - 1) / kScanElems4, pr.H, pr.b * pr.S);
  local_pass_kernel<<<grid, 256, 0, s>>>(pr, acs, sst, sext, ablk);
}

// Exclusive scan: S_in[0] = 0, S_in[k] = a_block[k-1] * S_in[k-1] + S_ext[k-1];
// final state = a_block[S-1] * S_in[S-1] + S_ext[S-1].
__global__ void __launch_bounds__(256) seg_scan_kernel(Problem pr, const float *__restrict__ sext,
                                                       const float *__restrict__ ablk, float *__restrict__ segin,
                                                       float *__restrict__ final_state) {
  const int PN = pr.P * pr.N;
  const int e = blockIdx.x * 256 + threadIdx.x;
  const int h = blockIdx.y, bb = blockIdx.z;
  if (e >= PN) return;
  float s = 0.f;
  for (int k = 0; k < pr.S; ++k) {
    const size_t so = ((size_t)bb * pr.S + k) * pr.H + h;
    segin[so * PN + e] = s;
    s = fmaf(ablk[so], s, sext[so * PN + e]);
  }
  if (final_state) final_state[((size_t)bb * pr.H + h) * PN + e] = s;
}

void launch_seg_scan(const Problem &pr, const float *sext, const float *ablk, float *segin, float *final_state,
                     cudaStream_t s) {
  dim3 grid((pr.P * pr.N + 255) / 256, pr.H, pr.b);
  seg_scan_kernel<<<grid, 256, 0, s>>>(pr, sext, ablk, segin, final_state);
}

// Local reverse pass of segment k from dS = 0 at the segment end:
//   dS_end[c] = dS;  dS <- Z[c] + a_c * dS   (c from the last chunk down)
// where Z[c] (held in dsl on entry) is the adjoint the chunk's own outputs send
// to the state entering it.  Overwrites dsl[c] with the local gradient at the
// chunk's end and writes g_ext[k] = gradient w.r.t. the segment's initial state.
// Same access pattern as local_pass_kernel, walking the chunks backwards.
__global__ void __launch_bounds__(256) local_rev_kernel(Problem pr, const float *__restrict__ acs,
                                                        float *__restrict__ dsl, float *__restrict__ gext) {
  const int PN = pr.P * pr.N, PN4 = PN / 4;
  const int h = blockIdx.y, k = blockIdx.z % pr.S, bb = blockIdx.z / pr.S;
  const size_t cstride4 = (size_t)pr.H * PN / 4;
  float4 *base = reinterpret_cast<float4 *>(dsl + (((size_t)bb * pr.nc + (size_t)k * pr.cps) * pr.H + h) * PN);
  int e4[kScanVec4];
  float4 dS[kScanVec4];
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u) {
    e4[u] = blockIdx.x * kScanElems4 + u * 256 + threadIdx.x;
    dS[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int c1 = pr.cps; c1 > 0; c1 -= kScanBatch) {
    const int nb = min(kScanBatch, c1);
    const int c0 = c1 - nb;  // this batch covers chunks [c0, c1) of the segment, walked downwards
    float dec[kScanBatch];
    float4 z[kScanBatch][kScanVec4];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        dec[q] = chunk_decay(pr, bb, h, k * pr.cps + c0 + q);
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u)
          if (e4[u] < PN4) z[q][u] = base[(size_t)(c0 + q) * cstride4 + e4[u]];
      }
    }
    // the recurrence runs down the chunks; results are kept and stored in
    // increasing address order afterwards
    float4 outv[kScanBatch][kScanVec4];
#pragma unroll
    for (int q = kScanBatch - 1; q >= 0; --q) {
      if (q < nb) {
        const float a = dec[q];
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u) {
          outv[q][u] = dS[u];
          dS[u] = make_float4(fmaf(a, dS[u].x, z[q][u].x), fmaf(a, dS[u].y, z[q][u].y), fmaf(a, dS[u].z, z[q][u].z),
                              fmaf(a, dS[u].w, z[q][u].w));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q)
      if (q < nb) {
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u)
          if (e4[u] < PN4) base[(size_t)(c0 + q) * cstride4 + e4[u]] = outv[q][u];
      }
  }
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u)
    if (e4[u] < PN4) reinterpret_cast<float4 *>(gext + (((size_t)bb * pr.S + k) * pr.H + h) * PN)[e4[u]] = dS[u];
}

void launch_local_rev(const Problem &pr, const float *acs, float *dsl, float *gext, cudaStream_t s) {
  dim3 grid((pr.P * pr.N / 4 + kScanElems4 - 1) / kScanElems4, pr.H, pr.b * pr.S);
  local_rev_kernel<<<grid, 256, 0, s>>>(pr, acs, dsl, gext);
}

// Reverse exclusive scan: G_out[S-1] = dfinal; G_out[k-1] = a_block[k]*G_out[k] + g_ext[k].
// G_out[k] is the gradient w.r.t. the state at the end of segment k.
__global__ void __launch_bounds__(256) seg_rscan_kernel(Problem pr, const float *__restrict__ gext,
                                                        const float *__restrict__ ablk,
                                                        const float *__restrict__ dfinal, float *__restrict__ gout) {
  const int PN = pr.P * pr.N;
  const int e = blockIdx.x * 256 + threadIdx.x;
  const int h = blockIdx.y, bb = blockIdx.z;
  if (e >= PN) return;
  float g = dfinal ? dfinal[((size_t)bb * pr.H + h) * PN + e] : 0.f;
  for (int k = pr.S - 1; k >= 0; --k) {
    const size_t so = ((size_t)bb * pr.S + k) * pr.H + h;
    gout[so * PN + e] = g;
    g = fmaf(ablk[so], g, gext[so * PN + e]);
  }
}

void launch_seg_rscan(const Problem &pr, const float *gext, const float *ablk, const float *dfinal, float *gout,
                      cudaStream_t s) {
  dim3 grid((pr.P * pr.N + 255) / 256, pr.H, pr.b);
  seg_rscan_kernel<<<grid, 256, 0, s>>>(pr, gext, ablk, dfinal, gout);
}

}  // namespace ssd
