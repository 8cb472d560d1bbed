// Chunked SSD kernels on CUDA cores (fp32 FMA): the path for fp32 activations
// and for shapes outside the tensor-core kernels' envelope.
//
// Chunked form (the Mamba2 chunked algorithm that state-spaces/mamba issue #482
// "Sequence parallelism in the mixer" builds on).  For chunk c of Q tokens,
// local index i, head h with group g, Acs = chunk-local inclusive cumsum of
// dt*A, and masks for packed sequences:
//   CB[i,j]   = C_i . B_j                                      (per group)
//   Y_diag[i] = sum_{j<=i, same seq} CB[i,j] exp(Acs_i - Acs_j) dt_j x_j
//   Sc        = sum_j exp(Acs_Q-1 - Acs_j) dt_j x_j (outer) B_j   (j in the last token's sequence)
//   Y_off[i]  = exp(Acs_i) [seq_i = seq of the token before the chunk] C_i . S_in[c]
//   y         = Y_diag + Y_off + D x
// with S_in[c] = S_loc_in[c] + d_c * S_seg_in[k] (local state from the segment
// pass plus the segment's true initial state carried by the decay d_c from the
// segment start to the chunk start: the correction pass of Megatron-LM PR #6808
// "Add state-passing context parallelism for Mamba2").
//
// Backward: the adjoints of the same expressions, with the true state S_in and
// the true state gradient at each chunk end rebuilt from the local passes and
// the segment scans.  Nothing here uses atomics; every reduction has a fixed order.
#include <type_traits>

#include "chunk_common.cuh"
#include "kernels.h"
#include "simt_gemm.cuh"

namespace ssd {

namespace {

template <typename F>
__device__ __forceinline__ void for_tile(const float (&acc)[4][4], int m0, int M, int n0, int Nn, F f) {
  const int tm = threadIdx.x >> 4, tn = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + tm * 4 + i, n = n0 + tn * 4 + j;
      if (m < M && n < Nn) f(m, n, acc[i][j]);
    }
}

}  // namespace

// ---------------------------------------------------------------- forward

template <typename T>
__global__ void __launch_bounds__(256) cb_kernel(Problem pr, const T *__restrict__ u, float *__restrict__ cb) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  const int c = blockIdx.x, g = blockIdx.y, bb = blockIdx.z, Q = pr.Q, N = pr.N, Cd = pr.Cd;
  const T *ub = u + ((size_t)bb * pr.L + (size_t)c * Q) * Cd;
  const int offB = pr.H * pr.P + g * N, offC = pr.H * pr.P + pr.G * N + g * N;
  float *out = cb + (((size_t)bb * pr.nc + c) * pr.G + g) * Q * Q;
  auto fa = [&](int i, int n) { return to_f(ub[(size_t)i * Cd + offC + n]); };
  auto fb = [&](int n, int j) { return to_f(ub[(size_t)j * Cd + offB + n]); };
  for (int ti = 0; ti * kTile < Q; ++ti)
    for (int tj = 0; tj <= ti; ++tj) {
      float acc[4][4];
      zero_acc(acc);
      gemm_tile<true, false>(acc, ti * kTile, Q, tj * kTile, Q, 0, N, fa, fb, smem);
      for_tile(acc, ti * kTile, Q, tj * kTile, Q, [&](int i, int j, float v) { out[(size_t)i * Q + j] = v; });
    }
}

template <typename T> void launch_cb(const Problem &pr, const T *u, float *cb, cudaStream_t s) {
  cb_kernel<T><<<dim3(pr.nc, pr.G, pr.b), 256, 0, s>>>(pr, u, cb);
}

// Sc[p, n] = sum_j wdt_j x_j[p] B_j[n]
template <typename T>
__global__ void __launch_bounds__(256) state_kernel(Problem pr, const T *__restrict__ u, const float *__restrict__ dtv,
                                                    const float *__restrict__ acs, float *__restrict__ sst) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const int offX = id.h * P, offB = pr.H * P + id.g * N;
  float *out = sst + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * P * N;
  auto fa = [&](int p, int j) { return to_f(ub[(size_t)j * Cd + offX + p]) * v.wdt[j]; };
  auto fb = [&](int j, int n) { return to_f(ub[(size_t)j * Cd + offB + n]); };
  for (int tp = 0; tp * kTile < P; ++tp)
    for (int tn = 0; tn * kTile < N; ++tn) {
      float acc[4][4];
      zero_acc(acc);
      gemm_tile<false, true>(acc, tp * kTile, P, tn * kTile, N, 0, pr.Q, fa, fb, smem);
      for_tile(acc, tp * kTile, P, tn * kTile, N, [&](int p, int n, float x) { out[(size_t)p * N + n] = x; });
    }
}

template <typename T>
void launch_chunk_state(const Problem &pr, const T *u, const float *dtv, const float *acs, float *sst, cudaStream_t s) {
  state_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dtv, acs, sst);
}

// y = Y_diag + Y_off + D x
template <typename T>
__global__ void __launch_bounds__(256) out_kernel(Problem pr, const T *__restrict__ u, const float *__restrict__ dtv,
                                                  const float *__restrict__ acs, const float *__restrict__ cb,
                                                  const float *__restrict__ sst, const float *__restrict__ segin,
                                                  T *__restrict__ y) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const int offX = id.h * P, offC = HP + pr.G * N + id.g * N;
  const float *cbm = cb + (((size_t)id.bb * pr.nc + id.c) * pr.G + id.g) * Q * Q;
  const int k = id.c / pr.cps;
  const float dc = decay_seg_to_chunk(pr, id.bb, id.h, id.c);
  const float *sloc = sst + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * P * N;
  const float *sseg = segin + (((size_t)id.bb * pr.S + k) * pr.H + id.h) * P * N;
  const float Dh = pr.D[id.h];
  T *yb = y + ((size_t)id.bb * pr.L + id.t0) * HP + offX;
  auto fa1 = [&](int i, int j) {
    return (j <= i && v.seq[i] == v.seq[j]) ? cbm[(size_t)i * Q + j] * expf(v.acs[i] - v.acs[j]) * v.dt[j] : 0.f;
  };
  auto fb1 = [&](int j, int p) { return to_f(ub[(size_t)j * Cd + offX + p]); };
  auto fa2 = [&](int i, int n) { return to_f(ub[(size_t)i * Cd + offC + n]) * v.em[i]; };
  auto fb2 = [&](int n, int p) { return sloc[(size_t)p * N + n] + dc * sseg[(size_t)p * N + n]; };
  for (int ti = 0; ti * kTile < Q; ++ti)
    for (int tp = 0; tp * kTile < P; ++tp) {
      float acc[4][4];
      zero_acc(acc);
      gemm_tile<true, true>(acc, ti * kTile, Q, tp * kTile, P, 0, min(Q, (ti + 1) * kTile), fa1, fb1, smem);
      if (chunk_has_incoming(pr, id.c)) gemm_tile<true, false>(acc, ti * kTile, Q, tp * kTile, P, 0, N, fa2, fb2, smem);
      for_tile(acc, ti * kTile, Q, tp * kTile, P, [&](int i, int p, float x) {
        yb[(size_t)i * HP + p] = from_f<T>(x + Dh * to_f(ub[(size_t)i * Cd + offX + p]));
      });
    }
}

template <typename T>
void launch_chunk_out(const Problem &pr, const T *u, const float *dtv, const float *acs, const float *cb,
                      const float *sst, const float *segin, T *y, cudaStream_t s) {
  out_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dtv, acs, cb, sst, segin, y);
}

// ---------------------------------------------------------------- backward

// Z[c][p, n] = sum_i em_i dy_i[p] C_i[n]: what the chunk's off-diagonal outputs
// send back to the state entering the chunk.
template <typename T>
__global__ void __launch_bounds__(256) z_kernel(Problem pr, const T *__restrict__ u, const T *__restrict__ dy,
                                                const float *__restrict__ dtv, const float *__restrict__ acs,
                                                float *__restrict__ dsl) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, HP = pr.H * pr.P;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const T *dyb = dy + ((size_t)id.bb * pr.L + id.t0) * HP + id.h * P;
  const int offC = HP + pr.G * N + id.g * N;
  float *out = dsl + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * P * N;
  auto fa = [&](int p, int i) { return to_f(dyb[(size_t)i * HP + p]); };
  auto fb = [&](int i, int n) { return to_f(ub[(size_t)i * Cd + offC + n]) * v.em[i]; };
  for (int tp = 0; tp * kTile < P; ++tp)
    for (int tn = 0; tn * kTile < N; ++tn) {
      float acc[4][4];
      zero_acc(acc);
      gemm_tile<false, true>(acc, tp * kTile, P, tn * kTile, N, 0, pr.Q, fa, fb, smem);
      for_tile(acc, tp * kTile, P, tn * kTile, N, [&](int p, int n, float x) { out[(size_t)p * N + n] = x; });
    }
}

template <typename T>
void launch_chunk_z(const Problem &pr, const T *u, const T *dy, const float *acs, float *dsl, cudaStream_t s) {
  // dtv is not needed by Z but load_chunk_vecs reads it; acs doubles as a valid pointer
  z_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dy, acs, acs, dsl);
}

// With dM[i,j] = dy_i . x_j (over P) and L = exp(Acs_i - Acs_j) (causal, same seq):
//   W[i,j] = dM L dt_j       -- the adjoint of CB[i,j], stored for the dB / dC products
//   V[i,j] = dM CB L         -- reduced to per-token sums for the dt / Acs adjoints:
//   vrow_i = sum_{j<i} V dt_j,  vcol_j = sum_{i>j} V,  vdiag_j = V[j,j].
// The diagonal is kept apart: in the Acs adjoint vrow_i - dt_i vcol_i its two
// copies cancel exactly, and summing them separately would leave only rounding
// noise there (large for heads that forget within a token).
template <typename T>
__global__ void __launch_bounds__(256) w_kernel(Problem pr, const T *__restrict__ u, const T *__restrict__ dy,
                                                const float *__restrict__ dtv, const float *__restrict__ acs,
                                                const float *__restrict__ cb, float *__restrict__ wbuf,
                                                float *__restrict__ tok) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  __shared__ float rowacc[kTile], colacc[256], scratch[8 * kTile];
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, Q = pr.Q, HP = pr.H * pr.P;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const T *dyb = dy + ((size_t)id.bb * pr.L + id.t0) * HP + id.h * P;
  const int offX = id.h * P;
  const float *cbm = cb + (((size_t)id.bb * pr.nc + id.c) * pr.G + id.g) * Q * Q;
  float *wm = wbuf + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * Q * Q;
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  const size_t tb = ((size_t)id.bb * pr.H + id.h) * pr.L + id.t0;
  for (int i = threadIdx.x; i < 256; i += 256) colacc[i] = 0.f;
  __syncthreads();
  auto fa = [&](int i, int p) { return to_f(dyb[(size_t)i * HP + p]); };
  auto fb = [&](int p, int j) { return to_f(ub[(size_t)j * Cd + offX + p]); };
  const int tm = threadIdx.x >> 4, tn = threadIdx.x & 15;
  for (int ti = 0; ti * kTile < Q; ++ti) {
    if (threadIdx.x < kTile) rowacc[threadIdx.x] = 0.f;
    __syncthreads();
    for (int tj = 0; tj <= ti; ++tj) {
      float acc[4][4], wv[4][4], vv[4][4];
      zero_acc(acc);
      gemm_tile<true, false>(acc, ti * kTile, Q, tj * kTile, Q, 0, P, fa, fb, smem);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b2 = 0; b2 < 4; ++b2) {
          const int i = ti * kTile + tm * 4 + a, j = tj * kTile + tn * 4 + b2;
          float dML = 0.f, cbij = 0.f;  // dM o L (masked) and CB
          if (i < Q && j < Q && j <= i && v.seq[i] == v.seq[j]) {
            dML = acc[a][b2] * expf(v.acs[i] - v.acs[j]);
            cbij = cbm[(size_t)i * Q + j];
          }
          const float dtj = (j < Q) ? v.dt[j] : 0.f;
          const float vij = dML * cbij;  // V = dM o CB o L
          if (i < Q && j < Q) wm[(size_t)i * Q + j] = dML * dtj;  // adjoint of CB
          if (i == j && i < Q) tok[1 * BHL + tb + i] = vij;   // the diagonal, kept apart
          vv[a][b2] = i == j ? 0.f : vij;
          wv[a][b2] = vv[a][b2] * dtj;  // V o dt: the dt / Acs adjoint pieces
        }
      tile_rowsum_add(wv, rowacc);
      tile_colsum_add(vv, colacc + tj * kTile, scratch);
    }
    if (threadIdx.x < kTile && ti * kTile + threadIdx.x < Q) tok[0 * BHL + tb + ti * kTile + threadIdx.x] = rowacc[threadIdx.x];
    __syncthreads();
  }
  for (int j = threadIdx.x; j < Q; j += 256) tok[2 * BHL + tb + j] = colacc[j];
}

template <typename T>
void launch_chunk_w(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs, const float *cb,
                    float *wbuf, float *tok, cudaStream_t s) {
  w_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dy, dtv, acs, cb, wbuf, tok);
}

// du_x[j, p] = sum_{i>=j} M[i,j] dy_i[p] + wdt_j sum_n B_j[n] dS_end[p,n] + D dy_j[p]
template <typename T>
__global__ void __launch_bounds__(256) dx_kernel(Problem pr, const T *__restrict__ u, const T *__restrict__ dy,
                                                 const float *__restrict__ dtv, const float *__restrict__ acs,
                                                 const float *__restrict__ cb, const float *__restrict__ dsl,
                                                 const float *__restrict__ gout, float *__restrict__ du) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const T *dyb = dy + ((size_t)id.bb * pr.L + id.t0) * HP + id.h * P;
  const int offX = id.h * P, offB = HP + id.g * N;
  const float *cbm = cb + (((size_t)id.bb * pr.nc + id.c) * pr.G + id.g) * Q * Q;
  const int k = id.c / pr.cps;
  const float de = decay_chunk_to_seg_end(pr, id.bb, id.h, id.c);
  const float *dsc = dsl + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * P * N;
  const float *gk = gout + (((size_t)id.bb * pr.S + k) * pr.H + id.h) * P * N;
  const float Dh = pr.D[id.h];
  float *dub = du + ((size_t)id.bb * pr.L + id.t0) * Cd + offX;
  auto fa1 = [&](int j, int i) {
    return (i >= j && v.seq[i] == v.seq[j]) ? cbm[(size_t)i * Q + j] * expf(v.acs[i] - v.acs[j]) * v.dt[j] : 0.f;
  };
  auto fb1 = [&](int i, int p) { return to_f(dyb[(size_t)i * HP + p]); };
  auto fa2 = [&](int j, int n) { return to_f(ub[(size_t)j * Cd + offB + n]) * v.wdt[j]; };
  auto fb2 = [&](int n, int p) { return dsc[(size_t)p * N + n] + de * gk[(size_t)p * N + n]; };
  for (int tj = 0; tj * kTile < Q; ++tj)
    for (int tp = 0; tp * kTile < P; ++tp) {
      float acc[4][4];
      zero_acc(acc);
      gemm_tile<false, true>(acc, tj * kTile, Q, tp * kTile, P, tj * kTile, Q, fa1, fb1, smem);
      gemm_tile<true, false>(acc, tj * kTile, Q, tp * kTile, P, 0, N, fa2, fb2, smem);
      for_tile(acc, tj * kTile, Q, tp * kTile, P, [&](int j, int p, float x) {
        dub[(size_t)j * Cd + p] = x + Dh * to_f(dyb[(size_t)j * HP + p]);
      });
    }
}

template <typename T>
void launch_chunk_dx(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs, const float *cb,
                     const float *dsl, const float *gout, float *du, cudaStream_t s) {
  dx_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dy, dtv, acs, cb, dsl, gout, du);
}

// Per-head partials of the B and C gradients (W = dM o L o dt, the adjoint of CB):
//   dC_h[i] = sum_{j<=i} W[i,j] B_j + em_i S_in^T dy_i
//   dB_h[j] = sum_{i>=j} W[i,j] C_i + wdt_j dS_end^T x_j
// plus per-token dots r_i = C_i . (em_i S_in^T dy_i) and q_j = B_j . (dS_end^T x_j).
template <typename T>
__global__ void __launch_bounds__(256) dcdb_kernel(Problem pr, const T *__restrict__ u, const T *__restrict__ dy,
                                                   const float *__restrict__ dtv, const float *__restrict__ acs,
                                                   const float *__restrict__ wbuf, const float *__restrict__ sst,
                                                   const float *__restrict__ segin, const float *__restrict__ dsl,
                                                   const float *__restrict__ gout, float *__restrict__ dcp,
                                                   float *__restrict__ dbp, float *__restrict__ tok) {
  __shared__ __align__(16) float smem[kGemmSmemFloats];
  __shared__ ChunkVecs v;
  __shared__ float rowacc[kTile];
  const ChunkIds id = chunk_ids(pr);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P, H = pr.H;
  const T *ub = u + ((size_t)id.bb * pr.L + id.t0) * Cd;
  const T *dyb = dy + ((size_t)id.bb * pr.L + id.t0) * HP + id.h * P;
  const int offX = id.h * P, offB = HP + id.g * N, offC = HP + pr.G * N + id.g * N;
  const float *wm = wbuf + (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * Q * Q;
  const int k = id.c / pr.cps;
  const float dc = decay_seg_to_chunk(pr, id.bb, id.h, id.c);
  const float de = decay_chunk_to_seg_end(pr, id.bb, id.h, id.c);
  const size_t so = (((size_t)id.bb * pr.S + k) * pr.H + id.h) * P * N;
  const size_t co = (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * P * N;
  const float *sloc = sst + co, *sseg = segin + so, *dsc = dsl + co, *gk = gout + so;
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  const size_t tb = ((size_t)id.bb * pr.H + id.h) * pr.L + id.t0;
  const int tm = threadIdx.x >> 4, tn = threadIdx.x & 15;
  // ---- dC
  {
    auto fa2 = [&](int i, int p) { return to_f(dyb[(size_t)i * HP + p]) * v.em[i]; };
    auto fb2 = [&](int p, int n) { return sloc[(size_t)p * N + n] + dc * sseg[(size_t)p * N + n]; };
    auto fa1 = [&](int i, int j) { return wm[(size_t)i * Q + j]; };
    auto fb1 = [&](int j, int n) { return to_f(ub[(size_t)j * Cd + offB + n]); };
    for (int ti = 0; ti * kTile < Q; ++ti) {
      if (threadIdx.x < kTile) rowacc[threadIdx.x] = 0.f;
      __syncthreads();
      for (int tq = 0; tq * kTile < N; ++tq) {
        float acc[4][4], prod[4][4];
        zero_acc(acc);
        if (chunk_has_incoming(pr, id.c)) gemm_tile<true, true>(acc, ti * kTile, Q, tq * kTile, N, 0, P, fa2, fb2, smem);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b2 = 0; b2 < 4; ++b2) {
            const int i = ti * kTile + tm * 4 + a, n = tq * kTile + tn * 4 + b2;
            prod[a][b2] = (i < Q && n < N) ? acc[a][b2] * to_f(ub[(size_t)i * Cd + offC + n]) : 0.f;
          }
        tile_rowsum_add(prod, rowacc);
        gemm_tile<true, true>(acc, ti * kTile, Q, tq * kTile, N, 0, min(Q, (ti + 1) * kTile), fa1, fb1, smem);
        for_tile(acc, ti * kTile, Q, tq * kTile, N, [&](int i, int n, float x) {
          dcp[(((size_t)id.bb * pr.L + id.t0 + i) * H + id.h) * N + n] = x;
        });
      }
      if (threadIdx.x < kTile && ti * kTile + threadIdx.x < Q) tok[3 * BHL + tb + ti * kTile + threadIdx.x] = rowacc[threadIdx.x];
      __syncthreads();
    }
  }
  // ---- dB
  {
    auto fa2 = [&](int j, int p) { return to_f(ub[(size_t)j * Cd + offX + p]); };
    auto fb2 = [&](int p, int n) { return dsc[(size_t)p * N + n] + de * gk[(size_t)p * N + n]; };
    auto fa1 = [&](int j, int i) { return wm[(size_t)i * Q + j]; };
    auto fb1 = [&](int i, int n) { return to_f(ub[(size_t)i * Cd + offC + n]); };
    for (int tj = 0; tj * kTile < Q; ++tj) {
      if (threadIdx.x < kTile) rowacc[threadIdx.x] = 0.f;
      __syncthreads();
      for (int tq = 0; tq * kTile < N; ++tq) {
        float acc[4][4], prod[4][4];
        zero_acc(acc);
        gemm_tile<true, true>(acc, tj * kTile, Q, tq * kTile, N, 0, P, fa2, fb2, smem);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b2 = 0; b2 < 4; ++b2) {
            const int j = tj * kTile + tm * 4 + a, n = tq * kTile + tn * 4 + b2;
            prod[a][b2] = (j < Q && n < N) ? acc[a][b2] * to_f(ub[(size_t)j * Cd + offB + n]) : 0.f;
            acc[a][b2] *= (j < Q) ? v.wdt[j] : 0.f;
          }
        tile_rowsum_add(prod, rowacc);
        gemm_tile<false, true>(acc, tj * kTile, Q, tq * kTile, N, tj * kTile, Q, fa1, fb1, smem);
        for_tile(acc, tj * kTile, Q, tq * kTile, N, [&](int j, int n, float x) {
          dbp[(((size_t)id.bb * pr.L + id.t0 + j) * H + id.h) * N + n] = x;
        });
      }
      if (threadIdx.x < kTile && tj * kTile + threadIdx.x < Q) tok[4 * BHL + tb + tj * kTile + threadIdx.x] = rowacc[threadIdx.x];
      __syncthreads();
    }
  }
}

template <typename T>
void launch_chunk_dcdb(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs,
                       const float *wbuf, const float *sst, const float *segin, const float *dsl, const float *gout,
                       float *dcp, float *dbp, float *tok, cudaStream_t s) {
  dcdb_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dy, dtv, acs, wbuf, sst, segin, dsl, gout, dcp, dbp,
                                                          tok);
}

// dt / A / D gradients of one (chunk, head).  On the tensor-core path (sdp
// given) the chunk's decay term and the per-token dy . x come precomputed.
// With vrow, vcol the row and column sums of V without its diagonal (tok[0];
// tok[2] plus, for vcol_parts > 1, tok[5]), vdiag the diagonal (tok[1]) and
// dAcs_i the total adjoint of the chunk-local cumsum:
//   dAcs_i = vrow_i - dt_i vcol_i + r_i - wdt_i q_i  (+ sum_j wdt_j q_j + a_c <dS_end, S_in> at the last token)
//   d(dA_t) = sum_{i>=t} dAcs_i;   d dt_t = vcol_t + vdiag_t + w_t q_t + A d(dA_t);   dA += dt_t d(dA_t)
// (the diagonal's two contributions to dAcs cancel exactly, so it enters d dt only).
//   d dt_raw = d dt * sigmoid(dt_raw + dt_bias)
template <typename T>
__global__ void __launch_bounds__(256) dt_bwd_kernel(Problem pr, const T *__restrict__ u, const T *__restrict__ dy,
                                                     const float *__restrict__ dtv, const float *__restrict__ acs,
                                                     const float *__restrict__ sst, const float *__restrict__ segin,
                                                     const float *__restrict__ dsl, const float *__restrict__ gout,
                                                     const float *__restrict__ tok, int vcol_parts,
                                                     const float *__restrict__ sdp, int sdp_groups, GradOut go,
                                                     float *__restrict__ chs) {
  __shared__ ChunkVecs v;
  __shared__ float red[8], red3[24], dacs[256], dda[256];
  const ChunkIds id = chunk_ids(pr);
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  const size_t tb = ((size_t)id.bb * pr.H + id.h) * pr.L + id.t0;
  const int i = threadIdx.x;
  const bool valid = i < pr.Q;
  // this token's inputs, loaded before the chunk vectors so that the loads overlap
  float tk0 = 0.f, tk1 = 0.f, tk2 = 0.f, tk3 = 0.f, tk4 = 0.f, tk5 = 0.f, dt_raw = 0.f;
  if (valid) {
    tk0 = tok[0 * BHL + tb + i];
    tk1 = tok[1 * BHL + tb + i];
    tk2 = tok[2 * BHL + tb + i];
    tk3 = tok[3 * BHL + tb + i];
    tk4 = tok[4 * BHL + tb + i];
    if (vcol_parts > 1 || sdp) tk5 = tok[5 * BHL + tb + i];
    dt_raw = to_f(static_cast<const T *>(pr.dt)[((size_t)id.bb * pr.L + id.t0 + i) * pr.dts + id.h]);
  }
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P;
  const int PN = P * N;
  const int k = id.c / pr.cps;
  const float dc = decay_seg_to_chunk(pr, id.bb, id.h, id.c);
  const float de = decay_chunk_to_seg_end(pr, id.bb, id.h, id.c);
  const float ac = chunk_decay(pr, id.bb, id.h, id.c);
  const size_t so = (((size_t)id.bb * pr.S + k) * pr.H + id.h) * PN;
  const size_t co = (((size_t)id.bb * pr.nc + id.c) * pr.H + id.h) * PN;
  // a_c <dS_end, S_in>; on the tensor-core path the combine pass left one
  // partial sum per group of state elements (sdp), added here in order
  float part = 0.f;
  if (!sdp && ac != 0.f) {
    const float4 *a4 = reinterpret_cast<const float4 *>(dsl + co), *g4 = reinterpret_cast<const float4 *>(gout + so);
    const float4 *s4 = reinterpret_cast<const float4 *>(sst + co), *q4 = reinterpret_cast<const float4 *>(segin + so);
    for (int e = threadIdx.x; e < PN / 4; e += 256) {
      const float4 a = a4[e], g = g4[e], x = s4[e], y = q4[e];
      part += (a.x + de * g.x) * (x.x + dc * y.x) + (a.y + de * g.y) * (x.y + dc * y.y) +
              (a.z + de * g.z) * (x.z + dc * y.z) + (a.w + de * g.w) * (x.w + dc * y.w);
    }
  }
  float dec;
  if (sdp) {
    const size_t BNH = (size_t)pr.b * pr.nc * pr.H, ci = ((size_t)id.bb * pr.nc + id.c) * pr.H + id.h;
    float tot = 0.f;
    for (int g = 0; g < sdp_groups; ++g) tot += sdp[g * BNH + ci];
    dec = ac != 0.f ? ac * tot : 0.f;
  } else {
    dec = ac * block_sum256(part, red);
  }

  float q = 0.f, wq = 0.f, vcol = 0.f;
  if (valid) {
    q = tk4;
    wq = v.wdt[i] * q;
  }
  const float ssum = block_sum256(wq, red);
  if (valid) {
    vcol = tk2 + (vcol_parts > 1 ? tk5 : 0.f);
    float d = tk0 - v.dt[i] * vcol + tk3 - wq;
    if (i == Q - 1) d += ssum + dec;
    dacs[i] = d;
  }
  __syncthreads();
  {  // suffix sums dda[i] = sum_{j >= i} dacs[j]: warp suffix scans, then warp totals (fixed order)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float x = valid ? dacs[i] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (lane == 0) red[warp] = x;  // warp total
    __syncthreads();
    float later = 0.f;
    for (int w2 = 7; w2 > warp; --w2) later += red[w2];
    if (valid) dda[i] = x + later;
    __syncthreads();
  }
  const float A = -expf(pr.A_log[id.h]);
  float dA_part = 0.f, dz = 0.f, dD_part = 0.f;
  if (valid) {
    const int t = id.t0 + i;
    const float ddt = vcol + tk1 + v.w[i] * q + A * dda[i];
    dA_part = v.dt[i] * dda[i];
    const float z = dt_raw + pr.dt_bias[id.h];
    dz = ddt * sigmoid_f(z);
    T *dst = static_cast<T *>(go.ddt) + ((size_t)id.bb * pr.L + t) * go.ddts + id.h;
    *dst = from_f<T>(dz);
    const T *xr = u + ((size_t)id.bb * pr.L + t) * Cd + id.h * P;
    const T *dyr = dy + ((size_t)id.bb * pr.L + t) * HP + id.h * P;
    if (sdp) {  // tensor-core path: dy_t . x_t was written to tok[5] by the column kernel
      dD_part = tk5;
    } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
      for (int p = 0; p < P; p += 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(xr + p), b = *reinterpret_cast<const uint4 *>(dyr + p);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dD_part += __uint_as_float(wa[q] << 16) * __uint_as_float(wb[q] << 16) +
                     __uint_as_float(wa[q] & 0xffff0000u) * __uint_as_float(wb[q] & 0xffff0000u);
      }
    } else {
      for (int p = 0; p < P; ++p) dD_part += to_f(dyr[p]) * to_f(xr[p]);
    }
  }
  // the three block sums share one pair of barriers (same fixed order as block_sum256)
  float s_dA = dA_part, s_dz = dz, s_dD = dD_part;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    s_dA += __shfl_xor_sync(0xffffffffu, s_dA, o);
    s_dz += __shfl_xor_sync(0xffffffffu, s_dz, o);
    s_dD += __shfl_xor_sync(0xffffffffu, s_dD, o);
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    const int w = threadIdx.x >> 5;
    red3[w] = s_dA;
    red3[8 + w] = s_dz;
    red3[16 + w] = s_dD;
  }
  __syncthreads();
  s_dA = s_dz = s_dD = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    s_dA += red3[w];
    s_dz += red3[8 + w];
    s_dD += red3[16 + w];
  }
  if (threadIdx.x == 0) {
    const size_t nch = (size_t)pr.b * pr.nc * pr.H;
    const size_t o = ((size_t)id.bb * pr.nc + id.c) * pr.H + id.h;
    chs[o] = s_dz;
    chs[nch + o] = s_dA;
    chs[2 * nch + o] = s_dD;
  }
}

// The same dt / A / D gradients on the tensor-core path, where every per-token
// piece comes precomputed (vrow, vdiag, vcol, r, q, dy . x in tok; the chunk's
// decay term as sdp partials): one warp per (chunk, head), a lane per 8
// consecutive tokens, the suffix sums and totals by shuffles (no block-wide
// barrier until the gradients of dt_raw are written back through shared memory
// so that the 8 heads of a block store whole tokens).
constexpr int kDtTok = 8;  // tokens per lane (chunks of up to 256 tokens)
template <typename T>
__global__ void __launch_bounds__(256) dt_bwd_warp_kernel(Problem pr, const float *__restrict__ dtv,
                                                          const float *__restrict__ acs, const float *__restrict__ tok,
                                                          const float *__restrict__ sdp, int sdp_groups, GradOut go,
                                                          float *__restrict__ chs) {
  __shared__ float dzs[256][8];  // [token in chunk][head in block]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, h = blockIdx.y * 8 + warp, bb = blockIdx.z, Q = pr.Q, t0 = c * Q;
  const bool live = h < pr.H;  // warp-uniform
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  const int i0 = lane * kDtTok;  // this lane's first token in the chunk
  float dsum = 0.f, dAp = 0.f, dDp = 0.f, dzp = 0.f;
  if (live) {
    const size_t tb = ((size_t)bb * pr.H + h) * pr.L + t0;
    const float A = -expf(pr.A_log[h]), bias = pr.dt_bias[h];
    const float acs_last = acs[tb + Q - 1];
    const int seq_last = seq_of(pr, bb, t0 + Q - 1);
    const size_t BNH = (size_t)pr.b * pr.nc * pr.H, ci = ((size_t)bb * pr.nc + c) * pr.H + h;
    float dtot = 0.f;  // the chunk's decay term a_c <dS_end, S_in>, partials in order
    for (int g = 0; g < sdp_groups; ++g) dtot += sdp[g * BNH + ci];
    const float ac = chunk_decay(pr, bb, h, c);
    const float dec = ac != 0.f ? ac * dtot : 0.f;
    // per token only what the later passes need stays live: base (the suffix-sum
    // term), pre (vcol + vdiag + w q, the dt adjoint's own terms) and dt
    float base[kDtTok], pre[kDtTok], dtk[kDtTok];
    float zr[kDtTok];  // the raw dt inputs (one per token row), loaded with the rest
#pragma unroll
    for (int k = 0; k < kDtTok; ++k) zr[k] = 0.f;
    float wqsum = 0.f;
    const bool has = i0 < Q;  // Q is a multiple of kDtTok: a lane has all or none of its tokens
    {
      // the lane's kDtTok consecutive tokens of each per-token array: two 16-byte
      // loads per array, all issued before any use (L and Q are multiples of 8)
      float t0v[kDtTok], t3v[kDtTok], t5v[kDtTok], acv[kDtTok], qv[kDtTok], vc[kDtTok], vdg[kDtTok];
      auto ld8 = [&](const float *a, float (&v)[kDtTok]) {
        const float4 lo = __ldg(reinterpret_cast<const float4 *>(a)), hi = __ldg(reinterpret_cast<const float4 *>(a) + 1);
        v[0] = lo.x, v[1] = lo.y, v[2] = lo.z, v[3] = lo.w, v[4] = hi.x, v[5] = hi.y, v[6] = hi.z, v[7] = hi.w;
      };
      if (has) {
        const size_t o = tb + i0;
        const T *dtr = static_cast<const T *>(pr.dt) + ((size_t)bb * pr.L + t0) * pr.dts + h;
#pragma unroll
        for (int k = 0; k < kDtTok; ++k) zr[k] = to_f(dtr[(size_t)(i0 + k) * pr.dts]);
        ld8(dtv + o, dtk);
        ld8(acs + o, acv);
        ld8(tok + 4 * BHL + o, qv);
        ld8(tok + 2 * BHL + o, vc);
        ld8(tok + 1 * BHL + o, vdg);
        ld8(tok + 0 * BHL + o, t0v);
        ld8(tok + 3 * BHL + o, t3v);
        ld8(tok + 5 * BHL + o, t5v);
      }
#pragma unroll
      for (int k = 0; k < kDtTok; ++k) {
        base[k] = pre[k] = 0.f;
        if (has) {
          const float w = seq_of(pr, bb, t0 + i0 + k) == seq_last ? expf(acs_last - acv[k]) : 0.f;
          const float wq = w * dtk[k] * qv[k];
          base[k] = t0v[k] - dtk[k] * vc[k] + t3v[k] - wq;
          pre[k] = vc[k] + vdg[k] + w * qv[k];
          dDp += t5v[k];
          wqsum += wq;
        } else {
          dtk[k] = 0.f;
        }
      }
    }
    // dAcs at the chunk's last token also gets sum_j wdt_j q_j and the decay term,
    // which every suffix sum then contains: add them to all tokens' suffix sums
    float tail = 0.f;
    for (int o = 16; o >= 1; o >>= 1) wqsum += __shfl_xor_sync(0xffffffffu, wqsum, o);
    tail = wqsum + dec;
    // suffix sums over the chunk: within the lane, then the later lanes' totals
    float run = 0.f, suf[kDtTok];
#pragma unroll
    for (int k = kDtTok - 1; k >= 0; --k) {
      run += base[k];
      suf[k] = run;
    }
    float later = run;  // inclusive suffix over lanes >= this one
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, later, o);
      if (lane + o < 32) later += y;
    }
    later -= run;  // exclusive: the lanes after this one
#pragma unroll
    for (int k = 0; k < kDtTok; ++k) {
      const int i = i0 + k;
      if (i < Q) {
        const float dda = suf[k] + later + tail;
        const float ddt = pre[k] + A * dda;
        dAp = fmaf(dtk[k], dda, dAp);
        const float dz = ddt * sigmoid_f(zr[k] + bias);
        dzp += dz;
        dzs[i][warp] = dz;
      }
    }
    dsum = dzp;
  }
  // fixed-order warp totals of the parameter pieces
  for (int o = 16; o >= 1; o >>= 1) {
    dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    dAp += __shfl_xor_sync(0xffffffffu, dAp, o);
    dDp += __shfl_xor_sync(0xffffffffu, dDp, o);
  }
  if (live && lane == 0) {
    const size_t nch = (size_t)pr.b * pr.nc * pr.H, o = ((size_t)bb * pr.nc + c) * pr.H + h;
    chs[o] = dsum;
    chs[nch + o] = dAp;
    chs[2 * nch + o] = dDp;
  }
  __syncthreads();
  const int nh = min(8, pr.H - (int)blockIdx.y * 8);
  T *dst = static_cast<T *>(go.ddt) + ((size_t)bb * pr.L + t0) * go.ddts + blockIdx.y * 8;
  for (int e = threadIdx.x; e < Q * 8; e += 256) {
    const int i = e >> 3, hh = e & 7;
    if (hh < nh) dst[(size_t)i * go.ddts + hh] = from_f<T>(dzs[i][hh]);
  }
}

template <typename T>
void launch_chunk_dt(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs,
                     const float *sst, const float *segin, const float *dsl, const float *gout, const float *tok,
                     int vcol_parts, const float *sdp, int sdp_groups, const GradOut &go, float *chs,
                     cudaStream_t s) {
  if (sdp && vcol_parts == 1 && pr.Q <= 32 * kDtTok)  // tensor-core path: every piece precomputed
    dt_bwd_warp_kernel<T><<<dim3(pr.nc, (pr.H + 7) / 8, pr.b), 256, 0, s>>>(pr, dtv, acs, tok, sdp, sdp_groups, go,
                                                                            chs);
  else
    dt_bwd_kernel<T><<<dim3(pr.nc, pr.H, pr.b), 256, 0, s>>>(pr, u, dy, dtv, acs, sst, segin, dsl, gout, tok,
                                                              vcol_parts, sdp, sdp_groups, go, chs);
}

#define SSD_INST(T)                                                                                                  \
  template void launch_cb<T>(const Problem &, const T *, float *, cudaStream_t);                                     \
  template void launch_chunk_state<T>(const Problem &, const T *, const float *, const float *, float *,             \
                                      cudaStream_t);                                                                 \
  template void launch_chunk_out<T>(const Problem &, const T *, const float *, const float *, const float *,         \
                                    const float *, const float *, T *, cudaStream_t);                                \
  template void launch_chunk_z<T>(const Problem &, const T *, const T *, const float *, float *, cudaStream_t);      \
  template void launch_chunk_w<T>(const Problem &, const T *, const T *, const float *, const float *, const float *, \
                                  float *, float *, cudaStream_t);                                                   \
  template void launch_chunk_dx<T>(const Problem &, const T *, const T *, const float *, const float *,              \
                                   const float *, const float *, const float *, float *, cudaStream_t);              \
  template void launch_chunk_dcdb<T>(const Problem &, const T *, const T *, const float *, const float *,            \
                                     const float *, const float *, const float *, const float *, const float *,      \
                                     float *, float *, float *, cudaStream_t);                                       \
  template void launch_chunk_dt<T>(const Problem &, const T *, const T *, const float *, const float *,              \
                                   const float *, const float *, const float *, const float *, const float *, int,   \
                                   const float *, int, const GradOut &, float *, cudaStream_t);

SSD_INST(float)
SSD_INST(__nv_bfloat16)

}  // namespace ssd
