// Chunk kernels of the bf16 path on the 5th-generation tensor cores (tcgen05,
// accumulators in TMEM), built on tc_engine.cuh.  Same decomposition and the
// same formulas as the CUDA-core kernels in simt_chunk.cu (the chunked form of
// the Mamba2 SSD, with the state correction of Megatron-LM PR #6808 "Add
// state-passing context parallelism for Mamba2"); here every contraction runs
// as 128 x N x 16 bf16 MMAs with fp32 accumulation, and the masks, decays and
// dt scalings are applied while the operands are staged into shared memory.
//
// Envelope (checked on the host): bf16 activations, headdim 64, dstate 128,
// chunk 128 or 256, an even number of heads per group.  Row tiles are 128
// tokens; a chunk has Q/128 of them.
#include "chunk_common.cuh"
#include "kernels.h"
#include "tc_engine.cuh"

namespace ssd {

namespace {

using bf16 = __nv_bfloat16;
using tc::K_MAJOR;
using tc::MN_MAJOR;

template <class E>
constexpr int dyn_smem() {
  return 1024 + E::RING_BYTES + E::BAR_BYTES + 16;
}

template <class E>
struct Carve {
  uint8_t *ring;
  uint64_t *bars;
  uint32_t *tslot;
  __device__ Carve(uint8_t *raw) {
    ring = tc::aligned_smem(raw);
    bars = reinterpret_cast<uint64_t *>(ring + E::RING_BYTES);
    tslot = reinterpret_cast<uint32_t *>(ring + E::RING_BYTES + E::BAR_BYTES);
  }
};

template <class K>
void set_smem(K kernel, int bytes) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

__device__ __forceinline__ void store_row_f32(float *dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    reinterpret_cast<float4 *>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Column sums over a warp: lane l holds row l's 32 values v[0..31]; after the
// halving butterfly (offsets 16, 8, 4, 2, 1; 31 shuffles) lane l holds the sum
// of column l over the warp's 32 rows.  Fixed order, so bit-reproducible.
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int q = 0; q < o; ++q) {
      const float send = upper ? v[q] : v[q + o];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[q] = (upper ? v[q + o] : v[q]) + recv;
    }
  }
  return v[0];
}

}  // namespace

// ---------------------------------------------------------------- CB = C B^T
// CTA = (chunk, row tile I, group, batch); for each column tile J <= I the
// 128 x 128 block of C_i . B_j is written in fp32 (upper blocks never read).
using EngCB = tc::Engine<128, 2>;
__global__ void __launch_bounds__(tc::kThreads, 3) tc_cb_kernel(Problem pr, const bf16 *__restrict__ u, float *__restrict__ cb,
                                                    int *status) {
  extern __shared__ uint8_t smem_raw[];
  Carve<EngCB> sm(smem_raw);
  const int NTI = pr.Q / 128;
  const int c = blockIdx.x / NTI, I = blockIdx.x % NTI, g = blockIdx.y, bb = blockIdx.z;
  const int Cd = pr.Cd, Q = pr.Q, N = pr.N, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + (size_t)c * Q) * Cd;
  const int offB = HP + g * N, offC = HP + pr.G * N + g * N;
  EngCB eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 256);
  auto fa = [&](int m, int k) { return static_cast<const void *>(ub + (size_t)(128 * I + m) * Cd + offC + k); };
  for (int J = 0; J <= I; ++J) {
    auto fb = [&](int n, int k) { return static_cast<const void *>(ub + (size_t)(128 * J + n) * Cd + offB + k); };
    for (int k0 = 0; k0 < N; k0 += 64) eng.slice<K_MAJOR, K_MAJOR>(tmem + 128 * J, k0, fa, tc::Async{}, fb, tc::Async{}, k0 > 0);
  }
  eng.finish();
  if (tc::owns_row()) {
  const int i = 128 * I + threadIdx.x;
  float *out = cb + (((size_t)bb * pr.nc + c) * pr.G + g) * Q * Q + (size_t)i * Q;
  for (int J = 0; J <= I; ++J)
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      sm100::tmem_ld32(tc::tmem_lane_addr(tmem, 128 * J + 32 * cc), v);
      store_row_f32(out + 128 * J + 32 * cc, v);
    }
  }
  tc::tmem_free_cta(tmem, 256);
}

void launch_tc_cb(const Problem &pr, const bf16 *u, float *cb, int *status, cudaStream_t s) {
  static bool once = (set_smem(tc_cb_kernel, dyn_smem<EngCB>()), true);
  (void)once;
  tc_cb_kernel<<<dim3(pr.nc * (pr.Q / 128), pr.G, pr.b), tc::kThreads, dyn_smem<EngCB>(), s>>>(pr, u, cb, status);
}

// ---------------------------------------------------------------- chunk states
// Sc^T[n, (h, p)] = sum_j B_j[n] wdt_h,j x_j[h, p] for a pair of heads of one
// group: M = n (128), N = 2 x 64, K = the chunk's tokens.
using EngPair = tc::Engine<128, 2>;
__global__ void __launch_bounds__(tc::kThreads, 3) tc_state_kernel(Problem pr, const bf16 *__restrict__ u,
                                                       const float *__restrict__ dtv, const float *__restrict__ acs,
                                                       float *__restrict__ sst, int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ChunkVecs v0, v1;
  Carve<EngPair> sm(smem_raw);
  const int c = blockIdx.x, h0 = 2 * blockIdx.y, bb = blockIdx.z;
  const ChunkIds id0 = make_ids(pr, c, h0, bb), id1 = make_ids(pr, c, h0 + 1, bb);
  load_chunk_vecs(pr, id0, dtv, acs, v0);
  load_chunk_vecs(pr, id1, dtv, acs, v1);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id0.t0) * Cd;
  const int offB = HP + id0.g * N;
  EngPair eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 128);
  auto fa = [&](int m0, int k) { return static_cast<const void *>(ub + (size_t)k * Cd + offB + m0); };
  auto fbl = [&](int n0, int k) { return tc::ldg16(ub + (size_t)k * Cd + (h0 + (n0 >> 6)) * P + (n0 & 63)); };
  auto fbm = [&](uint4 raw, int n0, int k) {
    float x[8];
    tc::unpack8(raw, x);
    const float s = (n0 >> 6) ? v1.wdt[k] : v0.wdt[k];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] *= s;
    return tc::pack8(x);
  };
  for (int k0 = 0; k0 < pr.Q; k0 += 64) eng.slice<MN_MAJOR, MN_MAJOR>(tmem, k0, fa, tc::Async{}, fbl, fbm, k0 > 0);
  eng.finish();
  if (tc::owns_row()) {
  const int n = threadIdx.x;
  for (int cc = 0; cc < 4; ++cc) {
    float v[32];
    sm100::tmem_ld32(tc::tmem_lane_addr(tmem, 32 * cc), v);
    const int hl = cc >> 1;
    float *o = sst + (((size_t)bb * pr.nc + c) * pr.H + h0 + hl) * P * N + n;
#pragma unroll
    for (int q = 0; q < 32; ++q) o[(size_t)((cc & 1) * 32 + q) * N] = v[q];
  }
  }
  tc::tmem_free_cta(tmem, 128);
}

void launch_tc_state(const Problem &pr, const bf16 *u, const float *dtv, const float *acs, float *sst, int *status,
                     cudaStream_t s) {
  static bool once = (set_smem(tc_state_kernel, dyn_smem<EngPair>()), true);
  (void)once;
  tc_state_kernel<<<dim3(pr.nc, pr.H / 2, pr.b), tc::kThreads, dyn_smem<EngPair>(), s>>>(pr, u, dtv, acs, sst, status);
}

// ---------------------------------------------------------------- backward: Z
// Z^T[n, (h, p)] = sum_i C_i[n] em_h,i dy_i[h, p]  for a pair of heads.
__global__ void __launch_bounds__(tc::kThreads, 3) tc_z_kernel(Problem pr, const bf16 *__restrict__ u,
                                                   const bf16 *__restrict__ dy, const float *__restrict__ dtv,
                                                   const float *__restrict__ acs, float *__restrict__ dsl,
                                                   int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ChunkVecs v0, v1;
  Carve<EngPair> sm(smem_raw);
  const int c = blockIdx.x, h0 = 2 * blockIdx.y, bb = blockIdx.z;
  const ChunkIds id0 = make_ids(pr, c, h0, bb), id1 = make_ids(pr, c, h0 + 1, bb);
  load_chunk_vecs(pr, id0, dtv, acs, v0);
  load_chunk_vecs(pr, id1, dtv, acs, v1);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id0.t0) * Cd;
  const bf16 *dyb = dy + ((size_t)bb * pr.L + id0.t0) * HP;
  const int offC = HP + pr.G * N + id0.g * N;
  EngPair eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 128);
  auto fa = [&](int m0, int i) { return static_cast<const void *>(ub + (size_t)i * Cd + offC + m0); };
  auto fbl = [&](int n0, int i) { return tc::ldg16(dyb + (size_t)i * HP + (h0 + (n0 >> 6)) * P + (n0 & 63)); };
  auto fbm = [&](uint4 raw, int n0, int i) {
    float x[8];
    tc::unpack8(raw, x);
    const float s = (n0 >> 6) ? v1.em[i] : v0.em[i];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] *= s;
    return tc::pack8(x);
  };
  for (int k0 = 0; k0 < pr.Q; k0 += 64) eng.slice<MN_MAJOR, MN_MAJOR>(tmem, k0, fa, tc::Async{}, fbl, fbm, k0 > 0);
  eng.finish();
  if (tc::owns_row()) {
  const int n = threadIdx.x;
  for (int cc = 0; cc < 4; ++cc) {
    float vv[32];
    sm100::tmem_ld32(tc::tmem_lane_addr(tmem, 32 * cc), vv);
    const int hl = cc >> 1;
    float *o = dsl + (((size_t)bb * pr.nc + c) * pr.H + h0 + hl) * P * N + n;
#pragma unroll
    for (int q = 0; q < 32; ++q) o[(size_t)((cc & 1) * 32 + q) * N] = vv[q];
  }
  }
  tc::tmem_free_cta(tmem, 128);
}

void launch_tc_z(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs, float *dsl,
                 int *status, cudaStream_t s) {
  static bool once = (set_smem(tc_z_kernel, dyn_smem<EngPair>()), true);
  (void)once;
  tc_z_kernel<<<dim3(pr.nc, pr.H / 2, pr.b), tc::kThreads, dyn_smem<EngPair>(), s>>>(pr, u, dy, dtv, acs, dsl, status);
}

// ---------------------------------------------------------------- backward: W
// dM = dy_i . x_j (K = P) per 128 x 128 block (J <= I); then, per element,
//   W = dM L dt_j  (bf16, the adjoint of CB)   V = dM CB L
// with row sums vrow_i = sum_j V dt_j (tok[0]) and this row tile's partial
// column sums vcol_j = sum_i V (tok[2] for tile 0, tok[5] for tile 1).
using EngW = tc::Engine<128, 2>;
__global__ void __launch_bounds__(tc::kThreads, 3) tc_w_kernel(Problem pr, const bf16 *__restrict__ u,
                                                   const bf16 *__restrict__ dy, const float *__restrict__ dtv,
                                                   const float *__restrict__ acs, const float *__restrict__ cb,
                                                   bf16 *__restrict__ wbuf, float *__restrict__ tok, int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ChunkVecs v;
  Carve<EngW> sm(smem_raw);
  const int NTI = pr.Q / 128;
  const int c = blockIdx.x / NTI, I = blockIdx.x % NTI, h = blockIdx.y, bb = blockIdx.z;
  const ChunkIds id = make_ids(pr, c, h, bb);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, Q = pr.Q, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id.t0) * Cd;
  const bf16 *dyb = dy + ((size_t)bb * pr.L + id.t0) * HP + h * P;
  const float *cbm = cb + (((size_t)bb * pr.nc + c) * pr.G + id.g) * Q * Q;
  bf16 *wm = wbuf + (((size_t)bb * pr.nc + c) * pr.H + h) * Q * Q;
  EngW eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 256);
  auto fa = [&](int m, int k0) { return static_cast<const void *>(dyb + (size_t)(128 * I + m) * HP + k0); };
  for (int J = 0; J <= I; ++J) {
    auto fb = [&](int n, int k0) { return static_cast<const void *>(ub + (size_t)(128 * J + n) * Cd + h * P + k0); };
    for (int k0 = 0; k0 < P; k0 += 64)
      eng.slice<K_MAJOR, K_MAJOR>(tmem + 128 * J, k0, fa, tc::Async{}, fb, tc::Async{}, k0 > 0);
  }
  eng.finish();
  const bool ep = tc::owns_row();
  const int m = threadIdx.x & (tc::kRows - 1), i = 128 * I + m, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float ai = v.acs[i];
  const int si = v.seq[i];
  float rowsum = 0.f;
  float colpart[8];  // this warp's column sums of V, column (32 * slot + lane)
#pragma unroll
  for (int q = 0; q < 8; ++q) colpart[q] = 0.f;
  if (ep) {
#pragma unroll
    for (int J = 0; J < 2; ++J) {
      if (J > I) break;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int j0 = 128 * J + 32 * cc;
        float a[32], vv[32];
        sm100::tmem_ld32(tc::tmem_lane_addr(tmem, j0), a);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float cv[8], wv[8];
          tc::ld8f(cbm + (size_t)i * Q + j0 + 8 * q8, cv);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j = j0 + 8 * q8 + q;
            const float dml = (j <= i && v.seq[j] == si) ? a[8 * q8 + q] * expf(ai - v.acs[j]) : 0.f;
            vv[8 * q8 + q] = dml * cv[q];
            wv[q] = dml * v.dt[j];
            rowsum += vv[8 * q8 + q] * v.dt[j];
          }
          *reinterpret_cast<uint4 *>(wm + (size_t)i * Q + j0 + 8 * q8) = tc::pack8(wv);
        }
        colpart[4 * J + cc] = warp_colsum32(vv, lane);
      }
    }
  }
  __shared__ float wpart[4][256];
  if (ep) {
#pragma unroll
    for (int q = 0; q < 8; ++q) wpart[warp][32 * q + lane] = colpart[q];
  }
  __syncthreads();
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  const size_t tb = ((size_t)bb * pr.H + h) * pr.L + id.t0;
  if (ep) tok[tb + i] = rowsum;
  float *vcol = tok + (I == 0 ? 2 : 5) * BHL + tb;
  for (int j = threadIdx.x; j < Q; j += tc::kThreads)
    vcol[j] = (j < 128 * (I + 1)) ? (wpart[0][j] + wpart[1][j]) + (wpart[2][j] + wpart[3][j]) : 0.f;
  tc::tmem_free_cta(tmem, 256);
}

void launch_tc_w(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs,
                 const float *cb, bf16 *wbuf, float *tok, int *status, cudaStream_t s) {
  static bool once = (set_smem(tc_w_kernel, dyn_smem<EngW>()), true);
  (void)once;
  tc_w_kernel<<<dim3(pr.nc * (pr.Q / 128), pr.H, pr.b), tc::kThreads, dyn_smem<EngW>(), s>>>(pr, u, dy, dtv, acs, cb, wbuf,
                                                                                   tok, status);
}

// ---------------------------------------------------------------- backward: dX
// rows j of tile I, two accumulators of P columns:
//   T_j = sum_{i>=j} M[i,j] dy_i                    (K = the chunk's tokens)
//   U_j = dS_end B_j                                 (K = N)
// du_x[j] = T_j + wdt_j U_j + D dy_j, and q_j = x_j . U_j = B_j . (dS_end^T x_j),
// the per-token piece of the chunk-state term of the dt adjoint.
using EngDx = tc::Engine<64, 2>;
__global__ void __launch_bounds__(tc::kThreads, 3) tc_dx_kernel(Problem pr, const bf16 *__restrict__ u,
                                                    const bf16 *__restrict__ dy, const float *__restrict__ dtv,
                                                    const float *__restrict__ acs, const float *__restrict__ cb,
                                                    const bf16 *__restrict__ dse16, float *__restrict__ du,
                                                    float *__restrict__ tok, int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ChunkVecs v;
  Carve<EngDx> sm(smem_raw);
  const int NTI = pr.Q / 128;
  const int c = blockIdx.x / NTI, I = blockIdx.x % NTI, h = blockIdx.y, bb = blockIdx.z;
  const ChunkIds id = make_ids(pr, c, h, bb);
  load_chunk_vecs(pr, id, dtv, acs, v);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id.t0) * Cd;
  const bf16 *dyb = dy + ((size_t)bb * pr.L + id.t0) * HP + h * P;
  const int offB = HP + id.g * N;
  const float *cbm = cb + (((size_t)bb * pr.nc + c) * pr.G + id.g) * Q * Q;
  const int k = c / pr.cps;
  const bf16 *dse = dse16 + (((size_t)bb * pr.nc + c) * pr.H + h) * P * N;  // true dS at the chunk end, bf16
  EngDx eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 128);
  auto fa1l = [&](int m0, int i) { return tc::ldf8(cbm + (size_t)i * Q + 128 * I + m0); };
  auto fa1 = [&](const tc::F8 &raw, int m0, int i) {
    const int j0 = 128 * I + m0;
    float cv[8], r[8];
    tc::f8_to(raw, cv);
    const float ai = v.acs[i];
    const int si = v.seq[i];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      r[q] = (j <= i && v.seq[j] == si) ? cv[q] * expf(ai - v.acs[j]) * v.dt[j] : 0.f;
    }
    return tc::pack8(r);
  };
  auto fb1 = [&](int n0, int i) { return static_cast<const void *>(dyb + (size_t)i * HP + n0); };
  for (int k0 = 128 * I; k0 < Q; k0 += 64)
    eng.slice<MN_MAJOR, MN_MAJOR>(tmem, k0, fa1l, fa1, fb1, tc::Async{}, k0 > 128 * I);
  auto fa2l = [&](int m, int k0) { return static_cast<const void *>(ub + (size_t)(128 * I + m) * Cd + offB + k0); };
  auto fb2 = [&](int p, int k0) { return static_cast<const void *>(dse + (size_t)p * N + k0); };
  for (int k0 = 0; k0 < N; k0 += 64)
    eng.slice<K_MAJOR, K_MAJOR>(tmem + 64, k0, fa2l, tc::Async{}, fb2, tc::Async{}, k0 > 0);
  eng.finish();
  if (tc::owns_row()) {
  const int j = 128 * I + threadIdx.x;
  const float Dh = pr.D[h], wdt = v.wdt[j];
  float *dr = du + ((size_t)bb * pr.L + id.t0 + j) * Cd + h * P;
  float qsum = 0.f;
  for (int cc = 0; cc < 2; ++cc) {
    float a[32], uu[32];
    sm100::tmem_ld32(tc::tmem_lane_addr(tmem, 32 * cc), a);
    sm100::tmem_ld32(tc::tmem_lane_addr(tmem, 64 + 32 * cc), uu);
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      float d8[8], x8[8];
      tc::unpack8(tc::ldg16(dyb + (size_t)j * HP + 32 * cc + 8 * q8), d8);
      tc::unpack8(tc::ldg16(ub + (size_t)j * Cd + h * P + 32 * cc + 8 * q8), x8);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = 8 * q8 + q;
        qsum += x8[q] * uu[col];
        a[col] += wdt * uu[col] + Dh * d8[q];
      }
    }
    store_row_f32(dr + 32 * cc, a);
  }
  tok[4 * (size_t)pr.b * pr.H * pr.L + ((size_t)bb * pr.H + h) * pr.L + id.t0 + j] = qsum;
  }
  tc::tmem_free_cta(tmem, 128);
}

void launch_tc_dx(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs,
                  const float *cb, const bf16 *dse16, float *du, float *tok, int *status, cudaStream_t s) {
  static bool once = (set_smem(tc_dx_kernel, dyn_smem<EngDx>()), true);
  (void)once;
  tc_dx_kernel<<<dim3(pr.nc * (pr.Q / 128), pr.H, pr.b), tc::kThreads, dyn_smem<EngDx>(), s>>>(pr, u, dy, dtv, acs, cb, dse16,
                                                                                     du, tok, status);
}

// ---------------------------------------------------------------- backward: dC, dB
// CTA = (chunk, row tile I, subset of HS heads of one group, batch).  Over the
// subset's heads the CTA accumulates in TMEM
//   dC[i] += sum_{j<=i} W_h[i,j] B_j + em_h,i S_in,h^T dy_h,i       (rows i of tile I)
//   dB[j] += sum_{i>=j} W_h[i,j] C_i + wdt_h,j dS_end,h^T x_h,j      (rows j of tile I)
// and writes one partial per subset (summed over subsets in fixed order later).
// The off-diagonal dC term is also issued into a per-head accumulator for
//   r_i = C_i . (em_i S_in^T dy_i)   (per head, the Y_off piece of the dt adjoint).
using EngDcdb = tc::Engine<128, 2>;
__global__ void __launch_bounds__(tc::kThreads) tc_dcdb_kernel(Problem pr, const bf16 *__restrict__ u,
                                                      const bf16 *__restrict__ dy, const float *__restrict__ dtv,
                                                      const float *__restrict__ acs, const bf16 *__restrict__ wbuf,
                                                      const bf16 *__restrict__ sin16, const bf16 *__restrict__ dse16,
                                                      float *__restrict__ dcp, float *__restrict__ dbp,
                                                      float *__restrict__ tok, int hs_size, int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ChunkVecs v;
  Carve<EngDcdb> sm(smem_raw);
  const int NTI = pr.Q / 128;
  const int c = blockIdx.x / NTI, I = blockIdx.x % NTI, sub = blockIdx.y, bb = blockIdx.z;
  const int nsub = pr.H / hs_size;
  const int Cd = pr.Cd, P = pr.P, N = pr.N, Q = pr.Q, HP = pr.H * pr.P;
  const int h_first = sub * hs_size, g = h_first / pr.hpg;
  const bf16 *ub = u + ((size_t)bb * pr.L + (size_t)c * Q) * Cd;
  const int offB = HP + g * N, offC = HP + pr.G * N + g * N;
  const int k = c / pr.cps;
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;
  EngDcdb eng;
  eng.init(sm.ring, sm.bars, status);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 512);
  const uint32_t accC = tmem, accB = tmem + 128, accR = tmem + 256;
  const int r = 128 * I + (threadIdx.x & (tc::kRows - 1));  // this thread's row (i for dC, j for dB)
  const bool has_off = c > 0;
  bool firstC = true, firstB = true;
  auto scaled = [](uint4 raw, float s) {
    float x[8];
    tc::unpack8(raw, x);
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] *= s;
    return tc::pack8(x);
  };
  for (int hh = 0; hh < hs_size; ++hh) {
    const int h = h_first + hh;
    const ChunkIds id = make_ids(pr, c, h, bb);
    __syncthreads();  // the previous head's functors are done with v
    load_chunk_vecs(pr, id, dtv, acs, v);
    const bf16 *dyb = dy + ((size_t)bb * pr.L + id.t0) * HP + h * P;
    const bf16 *wm = wbuf + (((size_t)bb * pr.nc + c) * pr.H + h) * Q * Q;
    const size_t so = (((size_t)bb * pr.S + k) * pr.H + h) * P * N;
    const size_t co = (((size_t)bb * pr.nc + c) * pr.H + h) * P * N;
    const bf16 *sin = sin16 + co, *dse = dse16 + co;
    // ---- dC
    if (has_off) {
      auto fal = [&](int mm, int p0) { return tc::ldg16(dyb + (size_t)(128 * I + mm) * HP + p0); };
      auto fam = [&](uint4 raw, int mm, int) { return scaled(raw, v.em[128 * I + mm]); };
      auto fb = [&](int n0, int p) { return static_cast<const void *>(sin + (size_t)p * N + n0); };
      for (int k0 = 0; k0 < P; k0 += 64)
        eng.slice<K_MAJOR, MN_MAJOR>(accR, k0, fal, fam, fb, tc::Async{}, k0 > 0, accC, !firstC || k0 > 0);
      firstC = false;
    }
    {
      auto fa = [&](int mm, int j0) { return static_cast<const void *>(wm + (size_t)(128 * I + mm) * Q + j0); };
      auto fb = [&](int n0, int j) { return static_cast<const void *>(ub + (size_t)j * Cd + offB + n0); };
      for (int k0 = 0; k0 < 128 * (I + 1); k0 += 64)
        eng.slice<K_MAJOR, MN_MAJOR>(accC, k0, fa, tc::Async{}, fb, tc::Async{}, !firstC || k0 > 0);
      firstC = false;
    }
    // ---- dB
    {
      auto fal = [&](int mm, int p0) { return tc::ldg16(ub + (size_t)(128 * I + mm) * Cd + h * P + p0); };
      auto fam = [&](uint4 raw, int mm, int) { return scaled(raw, v.wdt[128 * I + mm]); };
      auto fb = [&](int n0, int p) { return static_cast<const void *>(dse + (size_t)p * N + n0); };
      for (int k0 = 0; k0 < P; k0 += 64)
        eng.slice<K_MAJOR, MN_MAJOR>(accB, k0, fal, fam, fb, tc::Async{}, !firstB || k0 > 0);
      firstB = false;
    }
    {
      auto fa = [&](int m0, int i) { return static_cast<const void *>(wm + (size_t)i * Q + 128 * I + m0); };
      auto fb = [&](int n0, int i) { return static_cast<const void *>(ub + (size_t)i * Cd + offC + n0); };
      for (int k0 = 128 * I; k0 < Q; k0 += 64)
        eng.slice<MN_MAJOR, MN_MAJOR>(accB, k0, fa, tc::Async{}, fb, tc::Async{}, true);
    }
    // ---- r for this head
    float rsum = 0.f;
    if (has_off) eng.finish();
    if (has_off && tc::owns_row()) {
      for (int cc = 0; cc < 4; ++cc) {
        float b[32];
        sm100::tmem_ld32(tc::tmem_lane_addr(accR, 32 * cc), b);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float c8[8];
          tc::unpack8(tc::ldg16(ub + (size_t)r * Cd + offC + 32 * cc + 8 * q8), c8);
#pragma unroll
          for (int q = 0; q < 8; ++q) rsum += c8[q] * b[8 * q8 + q];
        }
      }
    }
    if (tc::owns_row()) tok[3 * BHL + ((size_t)bb * pr.H + h) * pr.L + (size_t)c * Q + r] = rsum;
  }
  eng.finish();
  if (tc::owns_row()) {
    float *oc = dcp + (((size_t)bb * pr.L + (size_t)c * Q + r) * nsub + sub) * N;
    float *ob = dbp + (((size_t)bb * pr.L + (size_t)c * Q + r) * nsub + sub) * N;
    for (int cc = 0; cc < 4; ++cc) {
      float a[32];
      sm100::tmem_ld32(tc::tmem_lane_addr(accC, 32 * cc), a);
      store_row_f32(oc + 32 * cc, a);
      sm100::tmem_ld32(tc::tmem_lane_addr(accB, 32 * cc), a);
      store_row_f32(ob + 32 * cc, a);
    }
  }
  tc::tmem_free_cta(tmem, 512);
}

int tc_head_subset(const Problem &pr) {
  for (int hs : {16, 8, 4, 2})
    if (pr.hpg % hs == 0) return hs;
  return 1;
}

void launch_tc_dcdb(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs,
                    const bf16 *wbuf, const bf16 *sin16, const bf16 *dse16, float *dcp, float *dbp, float *tok,
                    int *status, cudaStream_t s) {
  static bool once = (set_smem(tc_dcdb_kernel, dyn_smem<EngDcdb>()), true);
  (void)once;
  const int hs = tc_head_subset(pr);
  tc_dcdb_kernel<<<dim3(pr.nc * (pr.Q / 128), pr.H / hs, pr.b), tc::kThreads, dyn_smem<EngDcdb>(), s>>>(
      pr, u, dy, dtv, acs, wbuf, sin16, dse16, dcp, dbp, tok, hs, status);
}

}  // namespace ssd
