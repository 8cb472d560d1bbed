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

// Decay tables (common.cuh: decay_tables_bh), one block of 256 threads per (b, h).
__global__ void __launch_bounds__(256) decay_tables_kernel(Problem pr, const float *__restrict__ acs, float *cdec,
                                                           float *dstart, float *dend, float *ablk) {
  decay_tables_bh(pr, acs, blockIdx.y, blockIdx.x, cdec, dstart, dend, ablk, threadIdx.x, blockDim.x,
                  [] { __syncthreads(); });
}

void launch_decay_tables(const Problem &pr, const float *acs, float *cdec, float *dstart, float *dend, float *ablk,
                         cudaStream_t s) {
  decay_tables_kernel<<<dim3(pr.H, pr.b), 256, 0, s>>>(pr, acs, cdec, dstart, dend, ablk);
}

// Local pass of segment k: S <- a_c * S + Sc[c] over the segment's chunks from
// S = 0, giving S_ext[k] (the segment's summary; a_block[k] comes with the
// decay tables).  WriteLocal: also overwrite sst[c] (the chunk's own state
// contribution Sc) with the local state entering the chunk, for the kernels
// that read it; the tensor-core path re-forms it in the combine passes instead.
// Each thread owns two 16-byte groups of state elements (kScanVec4 float4, one
// per 256-thread stride, so every warp access stays contiguous), reads the
// chunk decays itself (the same address for the whole block: one broadcast
// line) and keeps the loads of kScanBatch chunks in flight.  No barriers.
constexpr int kScanVec4 = 2;
constexpr int kScanElems4 = 256 * kScanVec4;  // float4 groups per block
static_assert(kScanElems4 * 4 == kScanGroupElems, "segment-walk block size");

template <bool WriteLocal>
__global__ void __launch_bounds__(256) local_pass_kernel(Problem pr, float *__restrict__ sst,
                                                         float *__restrict__ sext) {
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
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u) {
          if (e4[u] < PN4) {
            if (WriteLocal) base[(size_t)(c0 + q) * cstride4 + e4[u]] = S[u];
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
}

void launch_local_pass(const Problem &pr, float *sst, float *sext, bool write_local, cudaStream_t s) {
  dim3 grid(scan_groups(pr), pr.H, pr.b * pr.S);
  if (write_local)
    local_pass_kernel<true><<<grid, 256, 0, s>>>(pr, sst, sext);
  else
    local_pass_kernel<false><<<grid, 256, 0, s>>>(pr, sst, sext);
}

// Exclusive scan: S_in[0] = the row's initial state (zero without one),
// S_in[k] = a_block[k-1] * S_in[k-1] + S_ext[k-1];
// final state = a_block[S-1] * S_in[S-1] + S_ext[S-1].
__global__ void __launch_bounds__(256) seg_scan_kernel(Problem pr, const float *__restrict__ sext,
                                                       const float *__restrict__ ablk, float *__restrict__ segin,
                                                       float *__restrict__ final_state) {
  const int PN = pr.P * pr.N;
  const int e = blockIdx.x * 256 + threadIdx.x;
  const int h = blockIdx.y, bb = blockIdx.z;
  if (e >= PN) return;
  float s = pr.init ? pr.init[((size_t)bb * pr.H + h) * PN + e] : 0.f;
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
// to the state entering it.  Writes g_ext[k] = gradient w.r.t. the segment's
// initial state and (WriteLocal) overwrites dsl[c] with the local gradient at
// the chunk's end; without it dsl keeps Z and the backward combine re-forms the
// local gradients itself.  Same access pattern as local_pass_kernel, walking the
// chunks backwards.
template <bool WriteLocal>
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
    // increasing address order afterwards (when the per-chunk states are wanted)
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
    if (WriteLocal) {
#pragma unroll
      for (int q = 0; q < kScanBatch; ++q)
        if (q < nb) {
#pragma unroll
          for (int u = 0; u < kScanVec4; ++u)
            if (e4[u] < PN4) base[(size_t)(c0 + q) * cstride4 + e4[u]] = outv[q][u];
        }
    }
  }
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u)
    if (e4[u] < PN4) reinterpret_cast<float4 *>(gext + (((size_t)bb * pr.S + k) * pr.H + h) * PN)[e4[u]] = dS[u];
}

void launch_local_rev(const Problem &pr, const float *acs, float *dsl, float *gext, bool write_local,
                      cudaStream_t s) {
  dim3 grid((pr.P * pr.N / 4 + kScanElems4 - 1) / kScanElems4, pr.H, pr.b * pr.S);
  if (write_local)
    local_rev_kernel<true><<<grid, 256, 0, s>>>(pr, acs, dsl, gext);
  else
    local_rev_kernel<false><<<grid, 256, 0, s>>>(pr, acs, dsl, gext);
}

// 4 floats -> 4 bf16 (8 bytes)
__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  return make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
}

// Forward combination, walking the chunks of segment k like the local pass:
//   S_in[c] = S_loc[c] + dstart[c] * S_seg[k]   (the true state entering chunk c, bf16)
//   S_loc[c + 1] = a_c * S_loc[c] + Sc[c],  S_loc[first] = 0,
// so the local states are re-formed from the chunk states Sc instead of being
// read back.  S_seg[k] is read once per segment.
__global__ void __launch_bounds__(256) combine_fwd_kernel(Problem pr, const float *__restrict__ sc,
                                                          const float *__restrict__ segin,
                                                          __nv_bfloat16 *__restrict__ out) {
  const int PN = pr.P * pr.N, PN4 = PN / 4;
  const int h = blockIdx.y, k = blockIdx.z % pr.S, bb = blockIdx.z / pr.S;
  const size_t cstride4 = (size_t)pr.H * PN / 4;
  const size_t first = (((size_t)bb * pr.nc + (size_t)k * pr.cps) * pr.H + h) * PN / 4;  // float4 index
  const float4 *sc4 = reinterpret_cast<const float4 *>(sc) + first;
  uint2 *out4 = reinterpret_cast<uint2 *>(out) + first;
  const float4 *g4 = reinterpret_cast<const float4 *>(segin + (((size_t)bb * pr.S + k) * pr.H + h) * PN);
  int e4[kScanVec4];
  float4 S[kScanVec4], G[kScanVec4];
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u) {
    e4[u] = blockIdx.x * kScanElems4 + u * 256 + threadIdx.x;
    S[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    G[u] = e4[u] < PN4 ? g4[e4[u]] : S[u];
  }
  for (int c0 = 0; c0 < pr.cps; c0 += kScanBatch) {
    const int nb = min(kScanBatch, pr.cps - c0);
    float dec[kScanBatch], dst[kScanBatch];
    float4 v[kScanBatch][kScanVec4];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        dec[q] = chunk_decay(pr, bb, h, k * pr.cps + c0 + q);
        dst[q] = decay_start(pr, bb, h, k * pr.cps + c0 + q);
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u)
          if (e4[u] < PN4) v[q][u] = sc4[(size_t)(c0 + q) * cstride4 + e4[u]];
      }
    }
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        const float a = dec[q], d = dst[q];
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u) {
          if (e4[u] < PN4) {
            out4[(size_t)(c0 + q) * cstride4 + e4[u]] =
                pack4_bf16(S[u].x + d * G[u].x, S[u].y + d * G[u].y, S[u].z + d * G[u].z, S[u].w + d * G[u].w);
            S[u] = make_float4(fmaf(a, S[u].x, v[q][u].x), fmaf(a, S[u].y, v[q][u].y), fmaf(a, S[u].z, v[q][u].z),
                               fmaf(a, S[u].w, v[q][u].w));
          }
        }
      }
    }
  }
}

void launch_combine_state(const Problem &pr, const float *sc, const float *segin, __nv_bfloat16 *out,
                          cudaStream_t s) {
  combine_fwd_kernel<<<dim3(scan_groups(pr), pr.H, pr.b * pr.S), 256, 0, s>>>(pr, sc, segin, out);
}

// Backward combination, walking the chunks of segment k: the true state
// entering chunk c (re-formed from the chunk states Sc as in the forward
// combination) and the true state gradient at its end
//   S_in[c] = S_loc[c] + dstart[c] * S_seg[k],   dS[c] = dS_loc[c] + dend[c] * G_out[k],
// both written in bf16 (the tensor-core operands), and the block's partial of
// the chunk's decay term of the dt adjoint, sdp[g, b, c, h] = <dS[c], S_in[c]>
// over this block's elements (fp32; the consumer multiplies by a_c and sums
// the groups in order).  S_seg and G_out are read once per segment.
template <int MaxCps>
__global__ void __launch_bounds__(256) combine_bwd_kernel(Problem pr, const float *__restrict__ sc,
                                                          const float *__restrict__ segin,
                                                          const float *__restrict__ dsl,
                                                          const float *__restrict__ gout,
                                                          __nv_bfloat16 *__restrict__ sin16,
                                                          __nv_bfloat16 *__restrict__ dse16, float *__restrict__ sdp) {
  __shared__ float red[8];
  const int PN = pr.P * pr.N, PN4 = PN / 4;
  const int h = blockIdx.y, k = blockIdx.z % pr.S, bb = blockIdx.z / pr.S;
  const size_t cstride4 = (size_t)pr.H * PN / 4;
  const size_t first = (((size_t)bb * pr.nc + (size_t)k * pr.cps) * pr.H + h) * PN / 4;
  const float4 *sc4 = reinterpret_cast<const float4 *>(sc) + first, *z4 = reinterpret_cast<const float4 *>(dsl) + first;
  uint2 *s16 = reinterpret_cast<uint2 *>(sin16) + first, *d16 = reinterpret_cast<uint2 *>(dse16) + first;
  const size_t so = (((size_t)bb * pr.S + k) * pr.H + h) * PN;
  const float4 *gi4 = reinterpret_cast<const float4 *>(segin + so), *go4 = reinterpret_cast<const float4 *>(gout + so);
  int e4[kScanVec4];
  float4 S[kScanVec4], GI[kScanVec4], GO[kScanVec4];
#pragma unroll
  for (int u = 0; u < kScanVec4; ++u) {
    e4[u] = blockIdx.x * kScanElems4 + u * 256 + threadIdx.x;
    S[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    GI[u] = e4[u] < PN4 ? gi4[e4[u]] : S[u];
    GO[u] = e4[u] < PN4 ? go4[e4[u]] : S[u];
  }
  // MaxCps > 0: dsl still holds Z (the local pass kept only the segment
  // summaries); the local gradients dS[c] at the chunk ends are re-formed here
  // by the same downward recurrence, dS[c] = sum_{c' > c} (decays) Z[c'], into
  // this thread's own shared-memory slots (no barrier needed)
  extern __shared__ float4 zloc[];  // [MaxCps][kScanVec4][256]
  if constexpr (MaxCps > 0) {
    // all of the segment's Z loads first (in flight together), then the recurrence
    float4 zz[MaxCps][kScanVec4];
    float dec[MaxCps];
#pragma unroll
    for (int c = 0; c < MaxCps; ++c) {
      dec[c] = c < pr.cps ? chunk_decay(pr, bb, h, k * pr.cps + c) : 0.f;
#pragma unroll
      for (int u = 0; u < kScanVec4; ++u)
        zz[c][u] = (c < pr.cps && e4[u] < PN4) ? z4[(size_t)c * cstride4 + e4[u]] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 G[kScanVec4];
#pragma unroll
    for (int u = 0; u < kScanVec4; ++u) G[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = MaxCps - 1; c >= 0; --c) {
      if (c < pr.cps) {
        const float a = dec[c];
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u) {
          zloc[(c * kScanVec4 + u) * 256 + threadIdx.x] = G[u];
          G[u] = make_float4(fmaf(a, G[u].x, zz[c][u].x), fmaf(a, G[u].y, zz[c][u].y), fmaf(a, G[u].z, zz[c][u].z),
                             fmaf(a, G[u].w, zz[c][u].w));
        }
      }
    }
  }
  const size_t BNH = (size_t)pr.b * pr.nc * pr.H;
  for (int c0 = 0; c0 < pr.cps; c0 += kScanBatch) {
    const int nb = min(kScanBatch, pr.cps - c0);
    float dec[kScanBatch], dst[kScanBatch], den[kScanBatch];
    float4 v[kScanBatch][kScanVec4], z[kScanBatch][kScanVec4];
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q < nb) {
        const int c = k * pr.cps + c0 + q;
        dec[q] = chunk_decay(pr, bb, h, c);
        dst[q] = decay_start(pr, bb, h, c);
        den[q] = decay_end(pr, bb, h, c);
#pragma unroll
        for (int u = 0; u < kScanVec4; ++u)
          if (e4[u] < PN4) {
            v[q][u] = sc4[(size_t)(c0 + q) * cstride4 + e4[u]];
            z[q][u] = MaxCps > 0 ? zloc[((c0 + q) * kScanVec4 + u) * 256 + threadIdx.x]
                                 : z4[(size_t)(c0 + q) * cstride4 + e4[u]];
          }
      }
    }
#pragma unroll
    for (int q = 0; q < kScanBatch; ++q) {
      if (q >= nb) break;  // block-uniform
      const float a = dec[q], dc = dst[q], de = den[q];
      float part = 0.f;
#pragma unroll
      for (int u = 0; u < kScanVec4; ++u) {
        if (e4[u] < PN4) {
          const float sv[4] = {S[u].x + dc * GI[u].x, S[u].y + dc * GI[u].y, S[u].z + dc * GI[u].z,
                               S[u].w + dc * GI[u].w};
          const float gv[4] = {z[q][u].x + de * GO[u].x, z[q][u].y + de * GO[u].y, z[q][u].z + de * GO[u].z,
                               z[q][u].w + de * GO[u].w};
          part += gv[0] * sv[0] + gv[1] * sv[1] + gv[2] * sv[2] + gv[3] * sv[3];
          s16[(size_t)(c0 + q) * cstride4 + e4[u]] = pack4_bf16(sv[0], sv[1], sv[2], sv[3]);
          d16[(size_t)(c0 + q) * cstride4 + e4[u]] = pack4_bf16(gv[0], gv[1], gv[2], gv[3]);
          S[u] = make_float4(fmaf(a, S[u].x, v[q][u].x), fmaf(a, S[u].y, v[q][u].y), fmaf(a, S[u].z, v[q][u].z),
                             fmaf(a, S[u].w, v[q][u].w));
        }
      }
      const float tot = block_sum256(part, red);
      if (threadIdx.x == 0) sdp[blockIdx.x * BNH + ((size_t)bb * pr.nc + k * pr.cps + c0 + q) * pr.H + h] = tot;
    }
  }
}

int combine_bwd_local_cps(const Problem &pr) { return pr.cps <= 4 ? 4 : pr.cps <= 8 ? 8 : 0; }

void launch_combine_bwd(const Problem &pr, const float *sc, const float *segin, const float *dsl, const float *gout,
                        __nv_bfloat16 *sin16, __nv_bfloat16 *dse16, float *sdp, cudaStream_t s) {
  const dim3 grid(scan_groups(pr), pr.H, pr.b * pr.S);
  const int m = combine_bwd_local_cps(pr);
  const int smem = m * kScanVec4 * 256 * (int)sizeof(float4);
  if (m == 4) {
    combine_bwd_kernel<4><<<grid, 256, smem, s>>>(pr, sc, segin, dsl, gout, sin16, dse16, sdp);
  } else if (m == 8) {
    static bool once = (cudaFuncSetAttribute(combine_bwd_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             8 * kScanVec4 * 256 * (int)sizeof(float4)),
                        true);
    (void)once;
    combine_bwd_kernel<8><<<grid, 256, smem, s>>>(pr, sc, segin, dsl, gout, sin16, dse16, sdp);
  } else {
    combine_bwd_kernel<0><<<grid, 256, 0, s>>>(pr, sc, segin, dsl, gout, sin16, dse16, sdp);
  }
}

// Reverse exclusive scan: G_out[S-1] = dfinal; G_out[k-1] = a_block[k]*G_out[k] + g_ext[k].
// G_out[k] is the gradient w.r.t. the state at the end of segment k; one step
// past segment 0, a_block[0]*G_out[0] + g_ext[0], is the gradient w.r.t. the
// row's initial state (written to dinit when given).
__global__ void __launch_bounds__(256) seg_rscan_kernel(Problem pr, const float *__restrict__ gext,
                                                        const float *__restrict__ ablk,
                                                        const float *__restrict__ dfinal, float *__restrict__ gout,
                                                        float *__restrict__ dinit) {
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
  if (dinit) dinit[((size_t)bb * pr.H + h) * PN + e] = g;
}

void launch_seg_rscan(const Problem &pr, const float *gext, const float *ablk, const float *dfinal, float *gout,
                      float *dinit, cudaStream_t s) {
  dim3 grid((pr.P * pr.N + 255) / 256, pr.H, pr.b);
  seg_rscan_kernel<<<grid, 256, 0, s>>>(pr, gext, ablk, dfinal, gout, dinit);
}

}  // namespace ssd
