// Internal definitions shared by the libssd CUDA sources (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// Problem description handed to every kernel by value.
struct Problem {
  int b, L, H, P, N, G, Q, S;
  int Cd;   // H*P + 2*G*N conv channels, order [x | B | C]
  int nc;   // chunks per row, L / Q
  int cps;  // chunks per segment
  int hpg;  // heads per group
  const void *x, *B, *C, *dt;
  long long xs, Bs, Cs, dts;  // token strides (elements)
  const float *dt_bias, *A_log, *D, *conv_w, *conv_b;
  const int *seq_idx;  // (b, L) or nullptr
  const float *init;   // (b, H, P, N): each row's initial state (the state before token 0), or nullptr
  // gated RMSNorm after the mixer (z == nullptr: none): z (b, L, H*P) token stride zs
  const void *z;
  long long zs;
  const float *norm_w;  // (H*P)
  float norm_eps;
  // per (b, h, chunk) decay tables, (b, H, nc) fp32, filled by decay_tables_kernel:
  const float *cdec;    // product of the chunk's per-token decays (0 at row start / sequence start inside)
  const float *dstart;  // product of cdec over the segment's chunks before this one
  const float *dend;    // product of cdec over the segment's chunks after this one
  unsigned long long wait_ns;  // limit of the kernels' bounded hand-off waits (ssd_set_wait_limit_ns)
};

// ---------------------------------------------------------------- dtypes
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---------------------------------------------------------------- math
__device__ __forceinline__ float softplus_f(float z) { return z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z)); }
__device__ __forceinline__ float sigmoid_f(float v) { return 1.f / (1.f + expf(-v)); }
// sigmoid on the fast intrinsics (relative error ~1e-6; -v clamped so 1 + e^-v
// stays finite), for the conv activation where it is applied per element
__device__ __forceinline__ float sigmoid_fast(float v) { return __fdividef(1.f, 1.f + __expf(fminf(-v, 80.f))); }
// sigmoid as 1/2 + tanh(v/2)/2 on the special-function unit's tanh (PTX
// tanh.approx.f32, error about 2^-11): three instructions instead of five, for
// bf16 activations, whose own rounding (2^-9 relative) is coarser
__device__ __forceinline__ float sigmoid_tanh(float v) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * v));
  return fmaf(0.5f, t, 0.5f);
}
// the conv activation's sigmoid for activation type T
template <typename T> __device__ __forceinline__ float act_sigmoid(float v) { return sigmoid_tanh(v); }
template <> __device__ __forceinline__ float act_sigmoid<float>(float v) { return sigmoid_fast(v); }

// seq id of token t of row b (0 when there is no seq_idx)
__device__ __forceinline__ int seq_of(const Problem &pr, int b, int t) {
  return pr.seq_idx ? __ldg(pr.seq_idx + (size_t)b * pr.L + t) : 0;
}

// Whether the first tokens of chunk c receive a state from before the chunk:
// every chunk but a row's first, and the first one too when the row has an
// initial state (the state before token 0, which its decay then applies to).
__host__ __device__ __forceinline__ bool chunk_has_incoming(const Problem &pr, int c) {
  return c > 0 || pr.init != nullptr;
}
// The sequence that state belongs to: that of the token before the chunk, or
// for a row's first chunk the row's first sequence (only it starts from the
// initial state; later packed sequences start from zero).
__device__ __forceinline__ int seq_before_chunk(const Problem &pr, int b, int c) {
  return seq_of(pr, b, c > 0 ? c * pr.Q - 1 : 0);
}

// Product of the per-token decays over chunk c of row b, head h: the factor that
// carries the state entering the chunk to its end (computed from Acs; kernels
// read it from the decay tables through chunk_decay()).  Zero when no state
// enters the chunk (a row start without an initial state) and when a packed
// sequence starts inside it.  acs_bh: chunk-local inclusive cumsum of dt*A for
// (b, h), length L.
__device__ __forceinline__ float chunk_decay_raw(const Problem &pr, const float *acs_bh, int b, int c) {
  if (!chunk_has_incoming(pr, c)) return 0.f;
  int t0 = c * pr.Q, t1 = t0 + pr.Q - 1;
  if (pr.seq_idx && seq_before_chunk(pr, b, c) != seq_of(pr, b, t1)) return 0.f;
  return expf(acs_bh[t1]);
}

__device__ __forceinline__ size_t dtab_index(const Problem &pr, int b, int h, int c) {
  return ((size_t)b * pr.H + h) * pr.nc + c;
}
__device__ __forceinline__ float chunk_decay(const Problem &pr, int b, int h, int c) {
  return __ldg(pr.cdec + dtab_index(pr, b, h, c));
}
// decay from the start of chunk c's segment to the start of c, and from the end
// of c to the end of its segment
__device__ __forceinline__ float decay_start(const Problem &pr, int b, int h, int c) {
  return __ldg(pr.dstart + dtab_index(pr, b, h, c));
}
__device__ __forceinline__ float decay_end(const Problem &pr, int b, int h, int c) {
  return __ldg(pr.dend + dtab_index(pr, b, h, c));
}

// Decay tables of one (b, h), by `nthr` cooperating threads (this one `tid`):
// cdec[c] = product of the chunk's per-token decays (from Acs and seq_idx),
// then per segment the exclusive prefix and suffix products
// dstart[c] = prod_{c' in seg, c' < c} cdec[c'], dend[c] = prod_{c' > c}, and the
// segment's whole product a_block[k] (the factor of the affine summary).  `sync`
// makes the cdec writes visible to the cooperating threads before they are read.
template <class Sync>
__device__ __forceinline__ void decay_tables_bh(const Problem &pr, const float *acs, int bb, int h, float *cdec,
                                                float *dstart, float *dend, float *ablk, int tid, int nthr,
                                                Sync sync) {
  const float *acs_bh = acs + ((size_t)bb * pr.H + h) * pr.L;
  const size_t base = ((size_t)bb * pr.H + h) * pr.nc;
  for (int c = tid; c < pr.nc; c += nthr) cdec[base + c] = chunk_decay_raw(pr, acs_bh, bb, c);
  sync();
  for (int k = tid; k < pr.S; k += nthr) {
    const int c0 = k * pr.cps, c1 = c0 + pr.cps;
    float d = 1.f;
    for (int c = c0; c < c1; ++c) {
      dstart[base + c] = d;
      d *= cdec[base + c];
    }
    ablk[((size_t)bb * pr.S + k) * pr.H + h] = d;
    d = 1.f;
    for (int c = c1 - 1; c >= c0; --c) {
      dend[base + c] = d;
      d *= cdec[base + c];
    }
  }
}

__host__ __device__ __forceinline__ size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kConvBwdTok = 128;  // tokens per conv-backward block (one set of parameter partials each)

// Elements of the P x N state handled by one block of the segment-walk kernels
// (local pass, reverse pass, combines): 256 threads x two float4 groups.
constexpr int kScanGroupElems = 2048;
inline int scan_groups(const Problem &pr) { return (pr.P * pr.N + kScanGroupElems - 1) / kScanGroupElems; }

// The workspace starts with the device status word followed by one work
// counter per persistent kernel (zeroed with the status at every pass).
constexpr int kStatusBytes = 64;
enum CounterSlot : int { kCounterOut = 1, kCounterRow = 2, kCounterCol = 3, kCounterState = 4, kCounterZ = 5 };

// ---------------------------------------------------------------- workspace
// Offsets (bytes) of every scratch buffer; computed identically on host and
// used to carve one caller-provided workspace.
struct Workspace {
  size_t status;                               // int32 device status word, then the work counters
  size_t u;                                    // (b, L, Cd) act dtype: post-conv activations
  size_t dtv, acs;                             // (b, H, L) f32: dt, chunk-local cumsum of dt*A
  size_t cb;                                   // (b, nc, G, Q, Q) f32: C_i . B_j per chunk (CUDA-core path)
  size_t sst;                                  // (b, nc, H, P, N) f32: chunk states, then local S_in
  size_t sin16;                                // (b, nc, H, P, N) bf16: true S_in (tensor-core path)
  size_t dtab;                                 // 3 x (b, H, nc) f32: cdec, dstart, dend
  size_t sext, segin;                          // (b, S, H, P, N) f32
  size_t ablk;                                 // (b, S, H) f32
  // backward only
  size_t dsl;                                  // (b, nc, H, P, N) f32: Y_off adjoint, then local dS at chunk ends
  size_t dse16;                                // (b, nc, H, P, N) bf16: true dS at chunk ends (tensor-core path)
  size_t gext, gout;                           // (b, S, H, P, N) f32
  size_t du;                                   // (b, L, Cd) f32: grad of post-conv activations
  size_t w;                                    // (b, nc, H, Q, Q) f32: dM o L o dt (CUDA-core path)
  size_t tok;                                  // 6 x (b, H, L) f32 per-token adjoint pieces
  size_t dcp, dbp;                             // (b, L, H, N) f32 per-head dC / dB partials
  size_t chs;                                  // 4 x (b, nc, H) f32 per-chunk scalars
  size_t sdp;                                  // (scan groups, b, nc, H) f32: partial <dS, S_in> (tensor-core path)
  size_t convp;                                // (b, ntb, Cd, 5) f32 conv parameter partials
  // gated RMSNorm
  size_t ypre;                                 // (b, L, H*P) act dtype: the mixer output before the norm
  size_t dyn;                                  // backward: (b, L, H*P) act dtype, the mixer output's gradient
  size_t normp;                                // backward: (norm tiles, H*P) f32 norm-weight partials
  size_t total;
  int ntb;                                     // conv backward token blocks per row
};

// tc: the tensor-core path, which forms CB inside its kernels and keeps W on
// chip, so it needs neither the CB nor the W buffer.
int norm_bwd_tiles(const Problem &pr);  // norm.cu

inline Workspace plan_workspace(const Problem &pr, int elem_bytes, bool backward, bool tc, bool norm) {
  Workspace w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t b = pr.b, L = pr.L, H = pr.H, P = pr.P, N = pr.N, G = pr.G, Q = pr.Q, S = pr.S, nc = pr.nc,
               Cd = pr.Cd;
  w.status = take(256);
  w.u = take(b * L * Cd * elem_bytes);
  w.dtv = take(b * H * L * 4);
  w.acs = take(b * H * L * 4);
  w.cb = take(tc ? 0 : b * nc * G * Q * Q * 4);
  w.sst = take(b * nc * H * P * N * 4);
  w.sext = take(b * S * H * P * N * 4);
  w.segin = take(b * S * H * P * N * 4);
  w.ablk = take(b * S * H * 4);
  w.sin16 = take(b * nc * H * P * N * 2);
  w.dtab = take(3 * b * H * nc * 4);
  w.ntb = (int)((L + kConvBwdTok - 1) / kConvBwdTok);
  if (backward) {
    w.dsl = take(b * nc * H * P * N * 4);
    w.dse16 = take(b * nc * H * P * N * 2);
    w.gext = take(b * S * H * P * N * 4);
    w.gout = take(b * S * H * P * N * 4);
    w.du = take(b * L * Cd * 4);
    w.w = take(tc ? 0 : b * nc * H * Q * Q * 4);
    w.tok = take(6 * b * H * L * 4);
    w.dcp = take(b * L * H * N * 4);
    w.dbp = take(b * L * H * N * 4);
    w.chs = take(4 * b * nc * H * 4);
    w.sdp = take(tc ? (size_t)scan_groups(pr) * b * nc * H * 4 : 0);
    w.convp = take(b * (size_t)w.ntb * Cd * 5 * 4);
  }
  if (norm) {
    w.ypre = take(b * L * H * P * elem_bytes);
    if (backward) {
      w.dyn = take(b * L * H * P * elem_bytes);
      w.normp = take((size_t)norm_bwd_tiles(pr) * H * P * 4);
    }
  }
  w.total = off;
  return w;
}

}  // namespace ssd
