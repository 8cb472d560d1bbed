// Chunk-state and Z kernels of the bf16 path on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM), built on tc_engine.cuh: the
// per-chunk states S_c = sum_j w_j dt_j x_j B_j^T for a pair of heads, and the
// adjoint Z = sum_i C_i em_i dy_i feeding the reverse boundary scan.  Same
// formulas as the CUDA-core kernels in simt_chunk.cu (the chunked form of the
// Mamba2 SSD).  The output and the chunk gradients run in the persistent
// kernels of tc_out.cu, tc_bwd_row.cu and tc_bwd_col.cu.
//
// Envelope (checked on the host): bf16 activations, headdim 64, dstate 128,
// chunk 128 or 256, an even number of heads per group.
#include "chunk_common.cuh"
#include "kernels.h"
#include "tc_engine.cuh"

namespace ssd {

namespace {

using bf16 = __nv_bfloat16;

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

}  // namespace

// ---------------------------------------------------------------- chunk states
// Sc^T[n, (h, p)] = sum_j B_j[n] wdt_h,j x_j[h, p] for a pair of heads of one
// group: M = n (128), N = 2 x 64, K = the chunk's tokens.
using EngPair = tc::Engine<128, 2>;
__global__ void __launch_bounds__(tc::kThreads, 3) tc_state_kernel(Problem pr, const bf16 *__restrict__ u,
                                                       const float *__restrict__ dtv, const float *__restrict__ acs,
                                                       float *__restrict__ sst, int *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float wdt0[256], wdt1[256];
  Carve<EngPair> sm(smem_raw);
  const int c = blockIdx.x, h0 = 2 * blockIdx.y, bb = blockIdx.z;
  const ChunkIds id0 = make_ids(pr, c, h0, bb);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id0.t0) * Cd;
  const int offB = HP + id0.g * N;
  EngPair eng;
  eng.init(sm.ring, sm.bars, status);
  auto fa = [&](int m0, int k) { return static_cast<const void *>(ub + (size_t)k * Cd + offB + m0); };
  auto fbl = [&](int n0, int k) { return tc::ldg16(ub + (size_t)k * Cd + (h0 + (n0 >> 6)) * P + (n0 & 63)); };
  auto fbm = [&](uint4 raw, int n0, int k) {
    float x[8];
    tc::unpack8(raw, x);
    const float s = (n0 >> 6) ? wdt1[k] : wdt0[k];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] *= s;
    return tc::pack8(x);
  };
  // the first slice's loads fly while the weights are formed and TMEM is allocated
  uint4 cur[EngPair::PER_B];
  eng.prefetch0(fa, fbl, cur);
  // the rest of the chunk's rows hinted into L2 at once: per token the B row and
  // the pair's x row (two 128-byte lines each), one line per thread and pass
  for (int k0 = 64; k0 < pr.Q; k0 += 64) {
    const int r = threadIdx.x >> 2, q = threadIdx.x & 3;
    const bf16 *row = ub + (size_t)(k0 + r) * Cd + (q < 2 ? offB + 64 * q : h0 * P + 64 * (q - 2));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
  }
  load_wdt_pair(pr, c, h0, bb, dtv, acs, wdt0, wdt1);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 128);
  eng.contract(tmem, pr.Q, fa, fbl, fbm, cur);
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
  __shared__ float em0[256], em1[256];
  Carve<EngPair> sm(smem_raw);
  const int c = blockIdx.x, h0 = 2 * blockIdx.y, bb = blockIdx.z;
  const ChunkIds id0 = make_ids(pr, c, h0, bb);
  const int Cd = pr.Cd, P = pr.P, N = pr.N, HP = pr.H * pr.P;
  const bf16 *ub = u + ((size_t)bb * pr.L + id0.t0) * Cd;
  const bf16 *dyb = dy + ((size_t)bb * pr.L + id0.t0) * HP;
  const int offC = HP + pr.G * N + id0.g * N;
  EngPair eng;
  eng.init(sm.ring, sm.bars, status);
  auto fa = [&](int m0, int i) { return static_cast<const void *>(ub + (size_t)i * Cd + offC + m0); };
  auto fbl = [&](int n0, int i) { return tc::ldg16(dyb + (size_t)i * HP + (h0 + (n0 >> 6)) * P + (n0 & 63)); };
  auto fbm = [&](uint4 raw, int n0, int i) {
    float x[8];
    tc::unpack8(raw, x);
    const float s = (n0 >> 6) ? em1[i] : em0[i];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] *= s;
    return tc::pack8(x);
  };
  // the first slice's loads fly while the weights are formed and TMEM is allocated
  uint4 cur[EngPair::PER_B];
  eng.prefetch0(fa, fbl, cur);
  // the rest of the chunk's rows hinted into L2 at once: per token the C row and
  // the pair's dy row (two 128-byte lines each), one line per thread and pass
  for (int k0 = 64; k0 < pr.Q; k0 += 64) {
    const int r = threadIdx.x >> 2, q = threadIdx.x & 3;
    const bf16 *row =
        q < 2 ? ub + (size_t)(k0 + r) * Cd + offC + 64 * q : dyb + (size_t)(k0 + r) * HP + h0 * P + 64 * (q - 2);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
  }
  load_em_pair(pr, c, h0, bb, acs, em0, em1);
  const uint32_t tmem = tc::tmem_alloc_cta(sm.tslot, 128);
  eng.contract(tmem, pr.Q, fa, fbl, fbm, cur);
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

int tc_head_subset(const Problem &pr) {
  for (int hs : {16, 8, 4, 2})
    if (pr.hpg % hs == 0) return hs;
  return 1;
}

}  // namespace ssd
