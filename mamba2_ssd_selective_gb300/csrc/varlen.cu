// Per-sequence final states of a packed row (varlen batches, cu_seqlens):
// the state after the last token t_e of every sequence, for chunked prefill
// and continuation.  The pages list packed sequences and initial states as not
// supported yet ("Add state-passing context parallelism for Mamba2", "Not
// supported yet"); sequences are delimited by cu_seqlens as in "feat:
// context-parallel with nemotron v3" (Key changes, THD format).
//
// With c the chunk holding t_e and t0 its first token, Acs the chunk-local
// inclusive cumsum of dt*A:
//   h(t_e) = [the sequence entered chunk c with a state] exp(Acs_te) S_in[c]
//          + sum_{j = max(start, t0)}^{t_e} exp(Acs_te - Acs_j) dt_j x_j (outer) B_j
// where S_in[c] is the true state entering chunk c in fp32,
//   S_in[c] = S_loc[c] + dstart[c] S_seg[k],
// S_loc[c] the local state from the segment's start (read as it is on the
// CUDA-core path, re-formed from the chunk states Sc on the tensor-core path,
// S_loc[c'+1] = cdec[c'] S_loc[c'] + Sc[c']), and S_seg[k] the segment's true
// initial state from the exclusive scan.  The sequence entered chunk c with a
// state if it started before t0, or if it is the row's first sequence, the
// chunk is the row's first and the row has an initial state.
//
// One block per (sequence, head), 256 threads; each thread owns up to 32
// elements of the P x N state per pass and walks the chunk's tokens from
// shared-memory tiles of 16 tokens (CUDA cores, fp32: a few MFLOP per block).
#include "kernels.h"

namespace ssd {

namespace {

constexpr int kFinThreads = 256, kFinPer = 32, kFinTok = 16;

template <typename T>
__global__ void __launch_bounds__(kFinThreads) seq_finals_kernel(Problem pr, const T *__restrict__ u,
                                                                  const float *__restrict__ dtv,
                                                                  const float *__restrict__ acs,
                                                                  const float *__restrict__ sst, bool sst_local,
                                                                  const float *__restrict__ segin,
                                                                  const int *__restrict__ cu, float *__restrict__ out) {
  __shared__ float xs[kFinTok][256], bs[kFinTok][256], ws[kFinTok];
  const int q = blockIdx.x, h = blockIdx.y, bb = 0;  // packed rows: batch 1
  const int P = pr.P, N = pr.N, PN = P * N, Q = pr.Q, g = h / pr.hpg, HP = pr.H * pr.P;
  const int start = cu[q], end = cu[q + 1];
  float *o = out + ((size_t)q * pr.H + h) * PN;
  if (end <= start || start < 0 || end > pr.L) {  // an empty or malformed sequence: zero state
    for (int e = threadIdx.x; e < PN; e += kFinThreads) o[e] = 0.f;
    return;
  }
  const int te = end - 1, c = te / Q, t0 = c * Q, k = c / pr.cps;
  const bool entered = start < t0 || (start == 0 && t0 == 0 && pr.init != nullptr);
  const float *acs_bh = acs + ((size_t)bb * pr.H + h) * pr.L;
  const float *dt_bh = dtv + ((size_t)bb * pr.H + h) * pr.L;
  const float acs_te = acs_bh[te];
  const float ein = entered ? expf(acs_te) : 0.f;
  const int j0 = start > t0 ? start : t0;
  const T *ub = u + (size_t)bb * pr.L * pr.Cd;
  for (int e0 = 0; e0 < PN; e0 += kFinThreads * kFinPer) {
    float acc[kFinPer];
#pragma unroll
    for (int r = 0; r < kFinPer; ++r) {
      const int e = e0 + r * kFinThreads + threadIdx.x;
      float s = 0.f;
      if (entered && e < PN) {
        float loc;
        if (sst_local) {
          loc = sst[(((size_t)bb * pr.nc + c) * pr.H + h) * PN + e];
        } else {  // re-form the local state from the segment's first chunk
          loc = 0.f;
          for (int cc = k * pr.cps; cc < c; ++cc)
            loc = fmaf(chunk_decay(pr, bb, h, cc), loc, sst[(((size_t)bb * pr.nc + cc) * pr.H + h) * PN + e]);
        }
        s = ein * fmaf(decay_start(pr, bb, h, c), segin[(((size_t)bb * pr.S + k) * pr.H + h) * PN + e], loc);
      }
      acc[r] = s;
    }
    for (int jt = j0; jt <= te; jt += kFinTok) {
      const int nt = min(kFinTok, te + 1 - jt);
      __syncthreads();
      for (int z = threadIdx.x; z < nt * (P + N); z += kFinThreads) {
        const int r = z / (P + N), col = z % (P + N), j = jt + r;
        const size_t row = (size_t)j * pr.Cd;
        if (col < P)
          xs[r][col] = to_f(ub[row + h * P + col]);
        else
          bs[r][col - P] = to_f(ub[row + HP + g * N + (col - P)]);
      }
      for (int r = threadIdx.x; r < nt; r += kFinThreads)
        ws[r] = expf(acs_te - acs_bh[jt + r]) * dt_bh[jt + r];
      __syncthreads();
      for (int r = 0; r < nt; ++r) {
        const float w = ws[r];
#pragma unroll
        for (int a = 0; a < kFinPer; ++a) {
          const int e = e0 + a * kFinThreads + threadIdx.x;
          if (e < PN) acc[a] = fmaf(w * xs[r][e / N], bs[r][e % N], acc[a]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kFinPer; ++r) {
      const int e = e0 + r * kFinThreads + threadIdx.x;
      if (e < PN) o[e] = acc[r];
    }
  }
}

}  // namespace

template <typename T>
void launch_seq_finals(const Problem &pr, const T *u, const float *dtv, const float *acs, const float *sst,
                       bool sst_local, const float *segin, const int *cu_seqlens, int nseq, float *out,
                       cudaStream_t s) {
  seq_finals_kernel<T><<<dim3(nseq, pr.H), kFinThreads, 0, s>>>(pr, u, dtv, acs, sst, sst_local, segin, cu_seqlens,
                                                                  out);
}

template void launch_seq_finals<float>(const Problem &, const float *, const float *, const float *, const float *,
                                       bool, const float *, const int *, int, float *, cudaStream_t);
template void launch_seq_finals<__nv_bfloat16>(const Problem &, const __nv_bfloat16 *, const float *, const float *,
                                               const float *, bool, const float *, const int *, int, float *,
                                               cudaStream_t);

}  // namespace ssd
