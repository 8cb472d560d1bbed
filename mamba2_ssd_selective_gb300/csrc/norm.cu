// Gated RMSNorm after the mixer core (Mamba2's gated norm; the Megatron-LM PR
// keeps it outside its fused function: "Add state-passing context parallelism
// for Mamba2", description).  One norm group per B/C group of heads
// (gs = H*P/G channels), per token:
//   g_c = y_c silu(z_c),  r = 1/sqrt(mean_{c in group} g_c^2 + eps),  out_c = g_c r w_c
// and its backward, given dout:
//   dg_c = r w_c dout_c - g_c r^3 mean_k(w_k dout_k g_k)
//   dy_c = dg_c silu(z_c),  dz_c = dg_c y_c silu'(z_c),  dw_c = sum_t dout_c g_c r.
// A (token, group) pair is handled by one warp when the group has at most 512
// channels, else by a block of 256 threads; a thread owns groups of 8
// consecutive channels (16-byte accesses for bf16) and keeps them in
// registers.  Sums are fixed-order warp or block reductions; the weight
// gradient is a fixed-order sum of per-tile partials.  These passes stream
// y, z (and dout) once and write their outputs once.
#include "kernels.h"
#include "simt_gemm.cuh"

namespace ssd {

namespace {

constexpr int kNormThreads = 256;
constexpr int kWarpModeMax = 512;  // channels per group handled by one warp (2 x 8 per lane)
constexpr int kNormBwdTok = 32;    // tokens per backward tile (one weight partial each)

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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums over the threads that share a (token, group): the warp (NT = 32) or the
// block (NT = 256, scratch of 16 floats), two values at once, fixed order.
template <int NT>
__device__ __forceinline__ float2 group_sum2(float a, float b, float *scratch) {
  a = warp_sum(a);
  b = warp_sum(b);
  if (NT == 32) return make_float2(a, b);
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

// NT threads per (token, group) and V vector groups of 8 channels per thread:
// NT = 32, V = 2 covers groups up to 512 channels, NT = 256, V = 2 up to 4096.
template <typename T, int NT, int V>
__global__ void __launch_bounds__(kNormThreads) gated_norm_fwd_kernel(Problem pr, const T *__restrict__ ypre,
                                                                      T *__restrict__ y) {
  __shared__ float red[16];
  constexpr int kPairs = kNormThreads / NT;
  const int HP = pr.H * pr.P, gs = HP / pr.G, nv = gs / 8, tid = threadIdx.x % NT;
  const size_t pair = (size_t)blockIdx.x * kPairs + threadIdx.x / NT, npair = (size_t)pr.b * pr.L * pr.G;
  const bool live = pair < npair;  // warp-uniform (and block-uniform for NT = 256)
  const size_t tok = live ? pair / pr.G : 0;
  const int grp = live ? (int)(pair % pr.G) : 0;
  const T *yp = ypre + tok * HP + (size_t)grp * gs;
  const T *zp = static_cast<const T *>(pr.z) + tok * pr.zs + (size_t)grp * gs;
  const float *w = pr.norm_w + (size_t)grp * gs;
  float gv[V][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int v = tid + k * NT;
    if (live && v < nv) {
      float a[8], z[8];
      load8(yp + 8 * v, a);
      load8(zp + 8 * v, z);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        gv[k][e] = a[e] * z[e] * sigmoid_fast(z[e]);
        ss = fmaf(gv[k][e], gv[k][e], ss);
      }
    }
  }
  const float r = rsqrtf(group_sum2<NT>(ss, 0.f, red).x / gs + pr.norm_eps);
  T *out = y + tok * HP + (size_t)grp * gs;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int v = tid + k * NT;
    if (live && v < nv) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = gv[k][e] * r * __ldg(w + 8 * v + e);
      store8(out + 8 * v, o);
    }
  }
}

// Backward over a tile of kNormBwdTok consecutive flat tokens for one group: the
// pairs (token, group) of the tile are taken by kNormThreads / NT thread sets
// in turn; the weight partial of the tile is summed over the sets in a fixed
// order.
template <typename T, int NT, int V>
__global__ void __launch_bounds__(kNormThreads, 2) gated_norm_bwd_kernel(Problem pr, const T *__restrict__ ypre,
                                                                         const T *__restrict__ dout,
                                                                         T *__restrict__ dy, GradOut go,
                                                                         float *__restrict__ dwp) {
  __shared__ float red[16];
  __shared__ float dwsum[kNormThreads / NT][V * NT * 8];
  constexpr int kSets = kNormThreads / NT;
  const int tile = blockIdx.x, grp = blockIdx.y, HP = pr.H * pr.P, gs = HP / pr.G, nv = gs / 8;
  const int set = threadIdx.x / NT, tid = threadIdx.x % NT;
  const size_t ntok = (size_t)pr.b * pr.L, t0 = (size_t)tile * kNormBwdTok;
  const size_t tend = t0 + kNormBwdTok < ntok ? t0 + kNormBwdTok : ntok;
  const float *w = pr.norm_w + (size_t)grp * gs;
  float dwacc[V][8];
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) dwacc[k][e] = 0.f;
  // for NT = 256 every set is the whole block and the loop is block-uniform
  for (size_t tok = t0 + set; tok < tend; tok += kSets) {
    const T *yp = ypre + tok * HP + (size_t)grp * gs;
    const T *zp = static_cast<const T *>(pr.z) + tok * pr.zs + (size_t)grp * gs;
    const T *dp = dout + tok * HP + (size_t)grp * gs;
    float yv[V][8], zv[V][8], dv[V][8];
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int v = tid + k * NT;
      if (v < nv) {
        load8(yp + 8 * v, yv[k]);
        load8(zp + 8 * v, zv[k]);
        load8(dp + 8 * v, dv[k]);
      } else {  // past the group: zeros, which add nothing to the sums
#pragma unroll
        for (int e = 0; e < 8; ++e) yv[k][e] = zv[k][e] = dv[k][e] = 0.f;
      }
    }
    float ss = 0.f, wdg = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int v = tid + k * NT;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = yv[k][e] * zv[k][e] * sigmoid_fast(zv[k][e]);
        ss = fmaf(g, g, ss);
        wdg = fmaf((v < nv ? __ldg(w + 8 * v + e) : 0.f) * dv[k][e], g, wdg);
      }
    }
    const float2 s2 = group_sum2<NT>(ss, wdg, red);
    const float r = rsqrtf(s2.x / gs + pr.norm_eps), r3m = r * r * r * (s2.y / gs);
    T *dyp = dy + tok * HP + (size_t)grp * gs;
    T *dzp = static_cast<T *>(go.dz) + tok * go.dzs + (size_t)grp * gs;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int v = tid + k * NT;
      if (v < nv) {
        float oy[8], oz[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float sg = sigmoid_fast(zv[k][e]), sz = zv[k][e] * sg, g = yv[k][e] * sz;
          const float dg = r * __ldg(w + 8 * v + e) * dv[k][e] - g * r3m;
          oy[e] = dg * sz;
          oz[e] = dg * yv[k][e] * sg * (1.f + zv[k][e] * (1.f - sg));
          dwacc[k][e] = fmaf(dv[k][e] * g, r, dwacc[k][e]);
        }
        store8(dyp + 8 * v, oy);
        store8(dzp + 8 * v, oz);
      }
    }
  }
  // the tile's weight partial: the sets' sums added in set order
  float *pp = dwp + (size_t)tile * HP + (size_t)grp * gs;
  if (kSets == 1) {
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int v = tid + k * NT;
      if (v < nv) store8(pp + 8 * v, dwacc[k]);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) dwsum[set][(k * NT + tid) * 8 + e] = dwacc[k][e];
  __syncthreads();
  for (int c = threadIdx.x; c < gs; c += kNormThreads) {
    const int v = c / 8, e = c % 8, k = v / NT, lt = v % NT;
    float sum = 0.f;
    for (int q = 0; q < kSets; ++q) sum += dwsum[q][(k * NT + lt) * 8 + e];
    pp[c] = sum;
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
  const size_t npair = (size_t)pr.b * pr.L * pr.G;
  if (pr.H * pr.P / pr.G <= kWarpModeMax)
    gated_norm_fwd_kernel<T, 32, 2><<<(unsigned)((npair + 7) / 8), kNormThreads, 0, s>>>(pr, ypre, y);
  else
    gated_norm_fwd_kernel<T, 256, 2><<<(unsigned)npair, kNormThreads, 0, s>>>(pr, ypre, y);
}

template <typename T>
void launch_gated_norm_bwd(const Problem &pr, const T *ypre, const T *dout, T *dy, const GradOut &go, float *dwp,
                           float *dnorm_w, cudaStream_t s) {
  const int HP = pr.H * pr.P, ntiles = norm_bwd_tiles(pr);
  if (HP / pr.G <= kWarpModeMax)
    gated_norm_bwd_kernel<T, 32, 2><<<dim3(ntiles, pr.G), kNormThreads, 0, s>>>(pr, ypre, dout, dy, go, dwp);
  else
    gated_norm_bwd_kernel<T, 256, 2><<<dim3(ntiles, pr.G), kNormThreads, 0, s>>>(pr, ypre, dout, dy, go, dwp);
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
