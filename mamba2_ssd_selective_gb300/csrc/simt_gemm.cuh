// A 64x64 fp32 SIMT tile product used by the fp32 path's chunk kernels.
// 256 threads; thread (tm, tn) = (tid / 16, tid % 16) owns rows tm*4..+3 and
// columns tn*4..+3 of the tile.  Operands come from functors so that masks,
// decays and scalings are applied while staging (nothing is materialised).
#pragma once

namespace ssd {

constexpr int kTile = 64;
constexpr int kBK = 16;
constexpr int kLd = kTile + 4;  // padded smem row (floats); 272 B keeps float4 alignment
constexpr int kGemmSmemFloats = 2 * kBK * kLd;

// acc[i][j] += sum_{k in [kbeg,kend)} A(m0+tm*4+i, k) * B(k, n0+tn*4+j)
// A_K_FAST / B_N_FAST pick the staging loop order so that global reads are
// coalesced along whichever index is contiguous in memory.
template <bool A_K_FAST, bool B_N_FAST, class FA, class FB>
__device__ __forceinline__ void gemm_tile(float (&acc)[4][4], int m0, int M, int n0, int Nn, int kbeg, int kend,
                                          const FA &fa, const FB &fb, float *smem) {
  float *sA = smem;              // [kBK][kLd], element (k, m)
  float *sB = smem + kBK * kLd;  // [kBK][kLd], element (k, n)
  const int tid = threadIdx.x, tm = tid >> 4, tn = tid & 15;
  for (int k0 = kbeg; k0 < kend; k0 += kBK) {
    for (int e = tid; e < kTile * kBK; e += 256) {
      int m, k;
      if (A_K_FAST) { m = e / kBK; k = e % kBK; } else { m = e % kTile; k = e / kTile; }
      int gm = m0 + m, gk = k0 + k;
      sA[k * kLd + m] = (gm < M && gk < kend) ? fa(gm, gk) : 0.f;
    }
    for (int e = tid; e < kTile * kBK; e += 256) {
      int n, k;
      if (B_N_FAST) { n = e % kTile; k = e / kTile; } else { n = e / kBK; k = e % kBK; }
      int gn = n0 + n, gk = k0 + k;
      sB[k * kLd + n] = (gn < Nn && gk < kend) ? fb(gk, gn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float4 a = *reinterpret_cast<const float4 *>(sA + k * kLd + tm * 4);
      float4 bv = *reinterpret_cast<const float4 *>(sB + k * kLd + tn * 4);
      float av[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bw[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// Row sums of a tile (sum over its 64 columns), added into rowacc[0..63]
// (shared memory) in a fixed order.  vals[i][j] is the thread's contribution.
__device__ __forceinline__ void tile_rowsum_add(const float (&vals)[4][4], float *rowacc) {
  const int tid = threadIdx.x, tm = tid >> 4, tn = tid & 15;
  float r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[i] = (vals[i][0] + vals[i][1]) + (vals[i][2] + vals[i][3]);
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) r[i] += __shfl_xor_sync(0xffffffffu, r[i], o);
  }
  if (tn == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) rowacc[tm * 4 + i] += r[i];
  }
  __syncthreads();
}

// Column sums of a tile (sum over its 64 rows), added into colacc[0..63].
// scratch: 8 * 64 floats of shared memory.
__device__ __forceinline__ void tile_colsum_add(const float (&vals)[4][4], float *colacc, float *scratch) {
  const int tid = threadIdx.x, tn = tid & 15, warp = tid >> 5, lane = tid & 31;
  float cs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cs[j] = (vals[0][j] + vals[1][j]) + (vals[2][j] + vals[3][j]);
    cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], 16);
  }
  if (lane < 16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) scratch[warp * 64 + tn * 4 + j] = cs[j];
  }
  __syncthreads();
  if (tid < 64) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += scratch[w * 64 + tid];
    colacc[tid] += s;
  }
  __syncthreads();
}

// Deterministic block-wide sum (256 threads); every thread gets the result.
__device__ __forceinline__ float block_sum256(float v, float *scratch /* 8 floats */) {
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) s += scratch[w];
  return s;
}

}  // namespace ssd
