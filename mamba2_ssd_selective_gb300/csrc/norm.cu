// Gated RMSNorm after the mixer core (Mamba2's gated norm; the Megatron-LM PR
// keeps it outside its fused function: "Add state-passing context parallelism
// for Mamba2", description).  One norm group per B/C group of heads
// (gs = H*P/G channels), per token:
//   g_c = y_c silu(z_c),  r = 1/sqrt(mean_{c in group} g_c^2 + eps),  out_c = g_c r w_c
// and its backward, given dout:
//   dg_c = r w_c dout_c - g_c r^3 mean_k(w_k dout_k g_k)
//   dy_c = dg_c silu(z_c),  dz_c = dg_c y_c silu'(z_c),  dw_c = sum_t dout_c g_c r.
// One block of 256 threads per (token, group) in the forward, per (tile of
// tokens, group) in the backward; a thread owns groups of 8 consecutive
// channels (16-byte accesses for bf16).  Sums are block reductions in a fixed
// order; the weight gradient is a fixed-order sum of per-tile partials.
#include "kernels.h"
#include "simt_gemm.cuh"

namespace ssd {

namespace {

constexpr int kNormThreads = 256, kNormMaxV = 4;  // up to 4 x 8 channels per thread held in registers

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8]) {
  uint4 u;
  uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// two block sums at once (fixed order), scratch: 16 floats
__device__ __forceinline__ float2 block_sum2(float a, float b, float *scratch) {
  for (int o = 16; o >= 1; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    scratch[warp] = a;
    scratch[8 + warp] = b;
  }
  __syncthreads();
  float sa = 0.f, sb = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    sa += scratch[w];
    sb += scratch[8 + w];
  }
  return make_float2(sa, sb);
}

template <typename T>
__global__ void __launch_bounds__(kNormThreads) gated_norm_fwd_kernel(Problem pr, const T *__restrict__ ypre,
                                                                      T *__restrict__ y) {
  __shared__ float red[8];
  const size_t tok = blockIdx.x;  // flat (b, t)
  const int grp = blockIdx.y, HP = pr.H * pr.P, gs = HP / pr.G, nv = gs / 8;
  const T *yp = ypre + tok * HP + (size_t)grp * gs;
  const T *zp = static_cast<const T *>(pr.z) + tok * pr.zs + (size_t)grp * gs;
  const float *w = pr.norm_w + (size_t)grp * gs;
  T *out = y + tok * HP + (size_t)grp * gs;
  float gv[kNormMaxV][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormMaxV; ++k) {
    const int v = threadIdx.x + k * kNormThreads;
    if (v < nv) {
      float a[8], z[8];
      load8(yp + 8 * v, a);
      load8(zp + 8 * v, z);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        gv[k][e] = a[e] * z[e] * sigmoid_f(z[e]);
        ss = fmaf(gv[k][e], gv[k][e], ss);
      }
    }
  }
  for (int v = threadIdx.x + kNormMaxV * kNormThreads; v < nv; v += kNormThreads) {  // groups wider than 8192
    float a[8], z[8];
    load8(yp + 8 * v, a);
    load8(zp + 8 * v, z);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float g = a[e] * z[e] * sigmoid_f(z[e]);
      ss = fmaf(g, g, ss);
    }
  }
  const float r = rsqrtf(block_sum256(ss, red) / gs + pr.norm_eps);
#pragma unroll
  for (int k = 0; k < kNormMaxV; ++k) {
    const int v = threadIdx.x + k * kNormThreads;
    if (v < nv) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = gv[k][e] * r * w[8 * v + e];
      store8(out + 8 * v, o);
    }
  }
  for (int v = threadIdx.x + kNormMaxV * kNormThreads; v < nv; v += kNormThreads) {
    float a[8], z[8], o[8];
    load8(yp + 8 * v, a);
    load8(zp + 8 * v, z);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = a[e] * z[e] * sigmoid_f(z[e]) * r * w[8 * v + e];
    store8(out + 8 * v, o);
  }
}

// Backward over a tile of kNormBwdTok consecutive flat tokens for one group;
// dw partial row per tile.  Groups up to kNormMaxV * 8 * 256 channels.
constexpr int kNormBwdTok = 32;

template <typename T>
__global__ void __launch_bounds__(kNormThreads) gated_norm_bwd_kernel(Problem pr, const T *__restrict__ ypre,
                                                                      const T *__restrict__ dout, T *__restrict__ dy,
                                                                      GradOut go, float *__restrict__ dwp) {
  __shared__ float red[16];
  const int tile = blockIdx.x, grp = blockIdx.y, HP = pr.H * pr.P, gs = HP / pr.G, nv = gs / 8;
  const size_t ntok = (size_t)pr.b * pr.L;
  const float *w = pr.norm_w + (size_t)grp * gs;
  float dwacc[kNormMaxV][8];
#pragma unroll
  for (int k = 0; k < kNormMaxV; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) dwacc[k][e] = 0.f;
  for (int q = 0; q < kNormBwdTok; ++q) {
    const size_t tok = (size_t)tile * kNormBwdTok + q;
    if (tok >= ntok) break;  // block-uniform
    const T *yp = ypre + tok * HP + (size_t)grp * gs;
    const T *zp = static_cast<const T *>(pr.z) + tok * pr.zs + (size_t)grp * gs;
    const T *dp = dout + tok * HP + (size_t)grp * gs;
    float yv[kNormMaxV][8], zv[kNormMaxV][8], dv[kNormMaxV][8];
    float ss = 0.f, wdg = 0.f;
#pragma unroll
    for (int k = 0; k < kNormMaxV; ++k) {
      const int v = threadIdx.x + k * kNormThreads;
      if (v < nv) {
        load8(yp + 8 * v, yv[k]);
        load8(zp + 8 * v, zv[k]);
        load8(dp + 8 * v, dv[k]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float g = yv[k][e] * zv[k][e] * sigmoid_f(zv[k][e]);
          ss = fmaf(g, g, ss);
          wdg = fmaf(w[8 * v + e] * dv[k][e], g, wdg);
        }
      }
    }
    const float2 s2 = block_sum2(ss, wdg, red);
    const float r = rsqrtf(s2.x / gs + pr.norm_eps), m = s2.y / gs, r3m = r * r * r * m;
    T *dyp = dy + tok * HP + (size_t)grp * gs;
    T *dzp = static_cast<T *>(go.dz) + tok * go.dzs + (size_t)grp * gs;
#pragma unroll
    for (int k = 0; k < kNormMaxV; ++k) {
      const int v = threadIdx.x + k * kNormThreads;
      if (v < nv) {
        float oy[8], oz[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float zc = zv[k][e], sg = sigmoid_f(zc), s = zc * sg, g = yv[k][e] * s;
          const float dg = r * w[8 * v + e] * dv[k][e] - g * r3m;
          oy[e] = dg * s;
          oz[e] = dg * yv[k][e] * sg * (1.f + zc * (1.f - sg));
          dwacc[k][e] = fmaf(dv[k][e] * g, r, dwacc[k][e]);
        }
        store8(dyp + 8 * v, oy);
        store8(dzp + 8 * v, oz);
      }
    }
  }
  float *pp = dwp + (size_t)tile * HP + (size_t)grp * gs;
#pragma unroll
  for (int k = 0; k < kNormMaxV; ++k) {
    const int v = threadIdx.x + k * kNormThreads;
    if (v < nv) store8(pp + 8 * v, dwacc[k]);
  }
}

// dnorm_weight[c] = sum over tiles (in order) of the per-tile partials
__global__ void __launch_bounds__(256) norm_weight_reduce_kernel(int HP, int ntiles, const float *__restrict__ dwp,
                                                                 float *__restrict__ dw) {
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= HP) return;
  float s = 0.f;
  for (int k = 0; k < ntiles; ++k) s += dwp[(size_t)k * HP + c];
  dw[c] = s;
}

}  // namespace

int norm_bwd_tiles(const Problem &pr) { return (int)(((size_t)pr.b * pr.L + kNormBwdTok - 1) / kNormBwdTok); }

template <typename T>
void launch_gated_norm_fwd(const Problem &pr, const T *ypre, T *y, cudaStream_t s) {
  gated_norm_fwd_kernel<T><<<dim3((unsigned)((size_t)pr.b * pr.L), pr.G), kNormThreads, 0, s>>>(pr, ypre, y);
}

template <typename T>
void launch_gated_norm_bwd(const Problem &pr, const T *ypre, const T *dout, T *dy, const GradOut &go, float *dwp,
                           float *dnorm_w, cudaStream_t s) {
  const int HP = pr.H * pr.P, ntiles = norm_bwd_tiles(pr);
  gated_norm_bwd_kernel<T><<<dim3(ntiles, pr.G), kNormThreads, 0, s>>>(pr, ypre, dout, dy, go, dwp);
  norm_weight_reduce_kernel<<<(HP + 255) / 256, 256, 0, s>>>(HP, ntiles, dwp, dnorm_w);
}

template void launch_gated_norm_fwd<float>(const Problem &, const float *, float *, cudaStream_t);
template void launch_gated_norm_fwd<__nv_bfloat16>(const Problem &, const __nv_bfloat16 *, __nv_bfloat16 *,
                                                   cudaStream_t);
template void launch_gated_norm_bwd<float>(const Problem &, const float *, const float *, float *, const GradOut &,
                                           float *, float *, cudaStream_t);
template void launch_gated_norm_bwd<__nv_bfloat16>(const Problem &, const __nv_bfloat16 *, const __nv_bfloat16 *,
                                                   __nv_bfloat16 *, const GradOut &, float *, float *,
                                                   cudaStream_t);

}  // namespace ssd
