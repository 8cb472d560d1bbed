// Depthwise causal conv1d (width 4) + SiLU over the xBC channels, its backward,
// the dt preprocessing with the chunk-local cumsum of dt*A, the parameter-grad
// reductions, and cu_seqlens -> seq_idx.
//
// The conv halo: a chunk/segment starting at token t0 reads the raw inputs of
// tokens t0-3..t0-1, i.e. the previous segment's last d_conv-1 tokens (Megatron-LM
// PR #6808 "Add state-passing context parallelism for Mamba2", description; the
// conv must be adapted across shards: state-spaces/mamba issue #482 "Sequence
// parallelism in the mixer").  Taps that cross a packed-sequence boundary are
// zero (seq_idx, NeMo Automodel PR #1441 "feat: context-parallel with nemotron v3").
#include "kernels.h"

namespace ssd {

// Two consecutive channels as one packed fp32 pair (sm100.cuh: pk2 / mul2 /
// fma2; one 32-bit load for bf16), so that the arithmetic of a thread's two
// channels takes one instruction for both (IEEE rounding per lane).
using sm100::fma2;
using sm100::mul2;
using sm100::pk2;
using sm100::upk2;
__device__ __forceinline__ uint64_t loadp(const __nv_bfloat16 *p) {
  const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint64_t loadp(const float *p) { return *reinterpret_cast<const uint64_t *>(p); }
__device__ __forceinline__ void storep(__nv_bfloat16 *p, uint64_t v) {
  float lo, hi;
  upk2(v, lo, hi);
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(lo, hi);
}
__device__ __forceinline__ void storep(float *p, uint64_t v) { *reinterpret_cast<uint64_t *>(p) = v; }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the conv activation's sigmoid of both lanes
template <typename T> __device__ __forceinline__ uint64_t act_sigmoid2(uint64_t v) {
  float lo, hi;
  upk2(v, lo, hi);
  return pk2(act_sigmoid<T>(lo), act_sigmoid<T>(hi));
}
template <> __device__ __forceinline__ uint64_t act_sigmoid2<__nv_bfloat16>(uint64_t v) {
  // 1/2 + tanh(v/2)/2 (sigmoid_tanh) with the two multiply-adds packed
  const uint64_t half = pk2(0.5f, 0.5f);
  float lo, hi;
  upk2(mul2(v, half), lo, hi);
  float tl, th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(tl) : "f"(lo));
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hi));
  return fma2(half, pk2(tl, th), half);
}

// A tile of kCh channels that lies inside one of the x, B, C regions of xBC
// (tiles are numbered region by region, the last tile of a region may be
// partial): its raw-input and gradient bases for batch row bb, token strides,
// first channel (global and within the region) and width.
template <typename T> struct ChanTile {
  const T *src;
  T *grad;
  long long st, gst;
  int c0, nch;
};
template <typename T>
__device__ __forceinline__ ChanTile<T> chan_tile(const Problem &pr, const GradOut *go, int bb, int tile, int kCh) {
  const int HP = pr.H * pr.P, GN = pr.G * pr.N;
  const int ntx = (HP + kCh - 1) / kCh, ntg = (GN + kCh - 1) / kCh;
  ChanTile<T> ct;
  int rc0, width;
  const void *base;
  void *gbase = nullptr;
  long long st, gst = 0;
  if (tile < ntx) {
    rc0 = tile * kCh, width = HP, ct.c0 = rc0, base = pr.x, st = pr.xs;
    if (go) gbase = go->dx, gst = go->dxs;
  } else if (tile < ntx + ntg) {
    rc0 = (tile - ntx) * kCh, width = GN, ct.c0 = HP + rc0, base = pr.B, st = pr.Bs;
    if (go) gbase = go->dB, gst = go->dBs;
  } else {
    rc0 = (tile - ntx - ntg) * kCh, width = GN, ct.c0 = HP + GN + rc0, base = pr.C, st = pr.Cs;
    if (go) gbase = go->dC, gst = go->dCs;
  }
  ct.nch = min(kCh, width - rc0);
  ct.src = static_cast<const T *>(base) + (size_t)bb * pr.L * st + rc0;
  ct.grad = go ? static_cast<T *>(gbase) + (size_t)bb * pr.L * gst + rc0 : nullptr;
  ct.st = st;
  ct.gst = gst;
  return ct;
}
__host__ __device__ inline int chan_tiles(const Problem &pr, int kCh) {
  const int HP = pr.H * pr.P, GN = pr.G * pr.N;
  return (HP + kCh - 1) / kCh + 2 * ((GN + kCh - 1) / kCh);
}

// u[b, t, c] = silu(conv_b[c] + sum_k w[c,k] * xr[t-3+k, c]), taps masked at row
// start and at seq_idx changes.  A block owns a tile of kFwdTok tokens x
// kFwdCh channels: all of its raw inputs (plus the 3-token halo) are brought
// into shared memory with 16-byte cp.async copies at once (zero-filled before
// token 0), then each thread walks kFwdTok/4 tokens of 2 channels from shared
// memory; a warp's stores cover 64 consecutive channels of one token.
constexpr int kFwdTok = 128, kFwdCh = 128;

// One thread's run of n output rows (2 channels) from the shared tile, the
// last three raw inputs kept in registers.  HasSeq: taps masked at sequence
// changes.  With n a compile-time constant the loop unrolls completely.
template <typename T, bool HasSeq>
__device__ __forceinline__ void conv_fwd_rows(const T (*tile)[kFwdCh], const int *seqs, const float (&w)[2][4],
                                              const float (&bias)[2], int r0, int cp, int n, T *dst, int Cd) {
  const uint64_t w0 = pk2(w[0][0], w[1][0]), w1 = pk2(w[0][1], w[1][1]), w2 = pk2(w[0][2], w[1][2]),
                 w3 = pk2(w[0][3], w[1][3]), bp = pk2(bias[0], bias[1]);
  uint64_t x0 = loadp(&tile[r0][2 * cp]), x1 = loadp(&tile[r0 + 1][2 * cp]), x2 = loadp(&tile[r0 + 2][2 * cp]);
  int s0 = 0, s1 = 0, s2 = 0;
  if (HasSeq) {
    s0 = seqs[r0];
    s1 = seqs[r0 + 1];
    s2 = seqs[r0 + 2];
  }
#pragma unroll
  for (int k = 0; k < kFwdTok / 4; ++k) {
    if (k >= n) break;
    const uint64_t x3 = loadp(&tile[r0 + 3 + k][2 * cp]);
    const int sq = HasSeq ? seqs[r0 + 3 + k] : 0;
    const bool m2 = !HasSeq || s2 == sq, m1 = !HasSeq || s1 == sq, m0 = !HasSeq || s0 == sq;
    uint64_t v = fma2(w3, x3, bp);
    v = fma2(m2 ? w2 : 0ull, x2, v);
    v = fma2(m1 ? w1 : 0ull, x1, v);
    v = fma2(m0 ? w0 : 0ull, x0, v);
    storep(dst + (size_t)k * Cd, mul2(v, act_sigmoid2<T>(v)));
    x0 = x1;
    x1 = x2;
    x2 = x3;
    s0 = s1; s1 = s2; s2 = sq;
  }
}

// dt = softplus(dt_raw + dt_bias); acs = inclusive cumsum of dt*A within each
// chunk (A = -exp(A_log)); layouts (b, H, L).  A block takes one chunk of one
// row and 8 heads: the chunk's dt_raw for those heads (16 contiguous bytes per
// token in bf16) is staged in shared memory, then each warp takes a head, a
// lane 8 consecutive tokens: softplus, the lane's running sum, and the lanes'
// exclusive prefix by shuffles.  These blocks run inside the conv forward's
// launch (its last grid columns), in the conv tile's shared memory.
constexpr int kMaxChunk = 256, kDtHeads = 8, kDtPer = kMaxChunk / 32;
template <typename T>
__device__ __forceinline__ void dt_prep_block(const Problem &pr, float *__restrict__ dtv, float *__restrict__ acs,
                                              int c, int hgrp, int bb, float (*tile)[kDtHeads + 1]) {
  const int h0 = hgrp * kDtHeads;
  const int nh = min(kDtHeads, pr.H - h0), t0 = c * pr.Q;
  const T *src = static_cast<const T *>(pr.dt) + ((size_t)bb * pr.L + t0) * pr.dts + h0;
  // the block's heads of one token are contiguous: one 16-byte load per token
  // (two for fp32) when the rows allow it, else one load per element
  constexpr int kVec = 16 / (int)sizeof(T);
  const bool vec = nh == kDtHeads && pr.dts % kVec == 0 && ((uintptr_t)pr.dt % 16) == 0;
  if (vec) {
    for (int t = threadIdx.x; t < pr.Q; t += 256) {
      const uint4 *p = reinterpret_cast<const uint4 *>(src + (size_t)t * pr.dts);
#pragma unroll
      for (int v = 0; v < kDtHeads / kVec; ++v) {
        const uint4 u = __ldg(p + v);
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int k = 0; k < kVec; ++k) tile[t][v * kVec + k] = to_f(e[k]);
      }
    }
  } else {
    for (int e = threadIdx.x; e < pr.Q * kDtHeads; e += 256) {
      const int t = e / kDtHeads, hh = e % kDtHeads;
      if (hh < nh) tile[t][hh] = to_f(src[(size_t)t * pr.dts + hh]);
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, i0 = lane * kDtPer;
  for (int hh = warp; hh < nh; hh += 8) {
    const int h = h0 + hh;
    const float A = -expf(pr.A_log[h]), bias = pr.dt_bias[h];
    float d[kDtPer], a[kDtPer], run = 0.f;
#pragma unroll
    for (int k = 0; k < kDtPer; ++k) {
      const int i = i0 + k;
      d[k] = i < pr.Q ? softplus_f(tile[i][hh] + bias) : 0.f;
      run += d[k] * A;
      a[k] = run;
    }
    float pre = run;  // inclusive prefix of the lanes' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += y;
    }
    pre -= run;  // the lanes before this one
    const size_t ob = ((size_t)bb * pr.H + h) * pr.L + t0;
    if (i0 + kDtPer <= pr.Q) {  // the lane's 8 tokens: two 16-byte stores per array
      float4 *dv4 = reinterpret_cast<float4 *>(dtv + ob + i0), *av4 = reinterpret_cast<float4 *>(acs + ob + i0);
      dv4[0] = make_float4(d[0], d[1], d[2], d[3]);
      dv4[1] = make_float4(d[4], d[5], d[6], d[7]);
      av4[0] = make_float4(a[0] + pre, a[1] + pre, a[2] + pre, a[3] + pre);
      av4[1] = make_float4(a[4] + pre, a[5] + pre, a[6] + pre, a[7] + pre);
    } else {
#pragma unroll
      for (int k = 0; k < kDtPer; ++k)
        if (i0 + k < pr.Q) {
          dtv[ob + i0 + k] = d[k];
          acs[ob + i0 + k] = a[k] + pre;
        }
    }
  }
}

// Grid columns [0, conv_x) are conv tiles; the columns after them take the dt
// preparation of (chunk, group of kDtHeads heads) pairs, numbered column-major
// over (column, token tile) within a batch row.
template <typename T>
__global__ void __launch_bounds__(256) conv_fwd_kernel(Problem pr, T *__restrict__ u, float *__restrict__ dtv,
                                                       float *__restrict__ acs, int conv_x, int dt_hg) {
  constexpr int kRows = kFwdTok + 3;
  constexpr int kChunk = 16 / (int)sizeof(T);  // channels per 16-byte copy
  constexpr int kCpr = kFwdCh / kChunk;          // copies per row
  // dynamic shared memory (conv_fwd_smem bytes): tile | seqs
  extern __shared__ __align__(16) uint8_t conv_smem[];
  T(*tile)[kFwdCh] = reinterpret_cast<T(*)[kFwdCh]>(conv_smem);
  int *seqs = reinterpret_cast<int *>(conv_smem + sizeof(T) * kRows * kFwdCh);
  static_assert(sizeof(T) * kRows * kFwdCh >= sizeof(float) * kMaxChunk * (kDtHeads + 1), "dt tile inside the conv tile");
  if ((int)blockIdx.x >= conv_x) {
    const int id = ((int)blockIdx.x - conv_x) * (int)gridDim.y + (int)blockIdx.y, c = id / dt_hg;
    if (c < pr.nc)
      dt_prep_block<T>(pr, dtv, acs, c, id % dt_hg, blockIdx.z, reinterpret_cast<float(*)[kDtHeads + 1]>(&tile[0][0]));
    return;
  }
  const int t0 = blockIdx.y * kFwdTok, bb = blockIdx.z;
  const ChanTile<T> ct = chan_tile<T>(pr, nullptr, bb, blockIdx.x, kFwdCh);
  const int c0 = ct.c0, nch = ct.nch;
  for (int q = threadIdx.x; q < kRows * kCpr; q += 256) {
    const int r = q / kCpr, cc = (q % kCpr) * kChunk, t = t0 - 3 + r;
    if (cc >= nch) continue;
    const bool ok = t >= 0 && t < pr.L;
    const T *g = ct.src + (ok ? (size_t)t * ct.st : 0) + cc;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
                     &tile[r][cc]))),
                 "l"(g), "r"(ok ? 16 : 0)
                 : "memory");
  }
  for (int r = threadIdx.x; r < kRows; r += 256) {
    const int t = t0 - 3 + r;
    seqs[r] = (t >= 0 && t < pr.L) ? seq_of(pr, bb, t) : -1;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int cp = threadIdx.x % (kFwdCh / 2), tq = threadIdx.x / (kFwdCh / 2);
  const int c = c0 + 2 * cp;
  if (2 * cp >= nch) return;
  float w[2][4], bias[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 wq = reinterpret_cast<const float4 *>(pr.conv_w)[c + q];
    w[q][0] = wq.x; w[q][1] = wq.y; w[q][2] = wq.z; w[q][3] = wq.w;
    bias[q] = pr.conv_b[c + q];
  }
  constexpr int kPer = kFwdTok / 4;
  const int r0 = tq * kPer;  // first output row (token t0 + r0), inputs at rows r0 .. r0 + 3
  T *dst = u + ((size_t)bb * pr.L + t0 + r0) * pr.Cd + c;
  const int tend = min(kPer, pr.L - (t0 + r0));
  if (tend <= 0) return;
  if (pr.seq_idx) {
    conv_fwd_rows<T, true>(tile, seqs, w, bias, r0, cp, tend, dst, pr.Cd);
  } else if (tend == kPer) {  // full run: constant trip count, unrolled
    conv_fwd_rows<T, false>(tile, seqs, w, bias, r0, cp, kPer, dst, pr.Cd);
  } else {
    conv_fwd_rows<T, false>(tile, seqs, w, bias, r0, cp, tend, dst, pr.Cd);
  }
}

template <typename T> constexpr int conv_fwd_smem() {
  return (int)(sizeof(T) * (kFwdTok + 3) * kFwdCh + sizeof(int) * (kFwdTok + 3));
}

template <typename T> void launch_conv_fwd(const Problem &pr, T *u, float *dtv, float *acs, cudaStream_t s) {
  constexpr int smem = conv_fwd_smem<T>();
  static bool once = (cudaFuncSetAttribute(conv_fwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem), true);
  (void)once;
  const int conv_x = chan_tiles(pr, kFwdCh), ny = (pr.L + kFwdTok - 1) / kFwdTok;
  const int dt_hg = (pr.H + kDtHeads - 1) / kDtHeads, dt_x = (pr.nc * dt_hg + ny - 1) / ny;
  conv_fwd_kernel<T><<<dim3(conv_x + dt_x, ny, pr.b), 256, smem, s>>>(pr, u, dtv, acs, conv_x, dt_hg);
}


// Conv + SiLU backward over a tile of kConvBwdTok tokens x kBwdCh channels (one
// region of xBC):
//   dv = du * silu'(v);  dxr[s] = sum_k w[k] dv[s+3-k] (same sequence);
//   per-tile partials of dconv_w[c,k] = sum dv[t] xr[t-3+k] and dconv_b[c] = sum dv.
// The raw inputs of tokens t0-3 .. t0+kConvBwdTok+2 and du of t0 .. t0+kConvBwdTok+2
// are brought into shared memory with 16-byte cp.async copies at once (zero
// outside the row, so tokens past the end give dv = 0).  Each thread owns 2
// channels; in phase 1 it walks a run of consecutive rows with the last three
// raw inputs in registers and overwrites du with dv in place (v recomputed from
// the raw inputs), in phase 2 a run of output rows with the last three dv in
// registers.  The parameter partials are summed over the row groups in fixed
// order.  HasSeq: taps masked at sequence changes (without seq_idx every tap
// counts; the halo before token 0 is zero).
constexpr int kBwdCh = 64;

template <typename T, bool HasSeq>
__global__ void __launch_bounds__(256) conv_bwd_kernel(Problem pr, const float *__restrict__ du, BcParts bc,
                                                       GradOut go, float *__restrict__ convp, int ntb) {
  constexpr int kTok = kConvBwdTok;
  constexpr int kXRows = kTok + 6;  // raw inputs, tokens t0-3 .. t0+kTok+2
  constexpr int kDRows = kTok + 3;  // du / dv, tokens t0 .. t0+kTok+2
  constexpr int kChunk = 16 / (int)sizeof(T);
  // dynamic shared memory (conv_bwd_smem bytes): dv | xr | seqs | red
  extern __shared__ __align__(16) uint8_t conv_smem[];
  float(*dv)[kBwdCh] = reinterpret_cast<float(*)[kBwdCh]>(conv_smem);
  T(*xr)[kBwdCh] = reinterpret_cast<T(*)[kBwdCh]>(conv_smem + sizeof(float) * kDRows * kBwdCh);
  int *seqs = reinterpret_cast<int *>(conv_smem + sizeof(float) * kDRows * kBwdCh + sizeof(T) * kXRows * kBwdCh);
  float(*red)[kBwdCh][5] = reinterpret_cast<float(*)[kBwdCh][5]>(seqs + ((kXRows + 3) & ~3));
  const int blk = blockIdx.y, bb = blockIdx.z, t0 = blk * kTok;
  const ChanTile<T> ct = chan_tile<T>(pr, &go, bb, blockIdx.x, kBwdCh);
  const int nch = ct.nch;
  for (int q = threadIdx.x; q < kXRows * (kBwdCh / kChunk); q += 256) {
    const int r = q / (kBwdCh / kChunk), cc = (q % (kBwdCh / kChunk)) * kChunk, t = t0 - 3 + r;
    if (cc >= nch) continue;
    const bool ok = t >= 0 && t < pr.L;
    const T *g = ct.src + (ok ? (size_t)t * ct.st : 0) + cc;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(&xr[r][cc]))),
                 "l"(g), "r"(ok ? 16 : 0)
                 : "memory");
  }
  const int HP = pr.H * pr.P, GN = pr.G * pr.N;
  if (ct.c0 < HP) {  // x channels: du as the chunk kernels wrote it
    const float *dub = du + (size_t)bb * pr.L * pr.Cd + ct.c0;
    for (int q = threadIdx.x; q < kDRows * (kBwdCh / 4); q += 256) {
      const int r = q / (kBwdCh / 4), cc = (q % (kBwdCh / 4)) * 4, t = t0 + r;
      if (cc >= nch) continue;
      const bool ok = t < pr.L;
      const float *g = dub + (ok ? (size_t)t * pr.Cd : 0) + cc;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       static_cast<uint32_t>(__cvta_generic_to_shared(&dv[r][cc]))),
                   "l"(g), "r"(ok ? 16 : 0)
                   : "memory");
    }
  } else {  // B / C channels: the sum of the group's head-block partials, in block order
    const bool isB = ct.c0 < HP + GN;
    const float *parts = isB ? bc.dbp : bc.dcp;
    const int idx0 = ct.c0 - HP - (isB ? 0 : GN);  // channel within the region: g * N + n
    for (int q = threadIdx.x; q < kDRows * (kBwdCh / 4); q += 256) {
      const int r = q / (kBwdCh / 4), cc = (q % (kBwdCh / 4)) * 4, t = t0 + r;
      if (cc >= nch) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < pr.L) {
        const int idx = idx0 + cc, g = idx / pr.N, n = idx % pr.N;  // 4 channels of one group (N % 4 == 0)
        const float4 *pp = reinterpret_cast<const float4 *>(parts + ((size_t)bb * pr.L + t) * bc.nsub * pr.N + n);
        const int k0 = g * bc.spg, kN4 = pr.N / 4;
        int k = 0;
        for (; k + 4 <= bc.spg; k += 4) {  // four partials' loads in flight, added in order
          const float4 v0 = pp[(size_t)(k0 + k) * kN4], v1 = pp[(size_t)(k0 + k + 1) * kN4];
          const float4 v2 = pp[(size_t)(k0 + k + 2) * kN4], v3 = pp[(size_t)(k0 + k + 3) * kN4];
          acc.x += v0.x; acc.y += v0.y; acc.z += v0.z; acc.w += v0.w;
          acc.x += v1.x; acc.y += v1.y; acc.z += v1.z; acc.w += v1.w;
          acc.x += v2.x; acc.y += v2.y; acc.z += v2.z; acc.w += v2.w;
          acc.x += v3.x; acc.y += v3.y; acc.z += v3.z; acc.w += v3.w;
        }
        for (; k < bc.spg; ++k) {
          const float4 v = pp[(size_t)(k0 + k) * kN4];
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
      *reinterpret_cast<float4 *>(&dv[r][cc]) = acc;
    }
  }
  if (HasSeq)
    for (int r = threadIdx.x; r < kXRows; r += 256) {
      const int t = t0 - 3 + r;
      seqs[r] = (t >= 0 && t < pr.L) ? seq_of(pr, bb, t) : -1;
    }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int cp = threadIdx.x % (kBwdCh / 2), tq = threadIdx.x / (kBwdCh / 2);
  const int c = ct.c0 + 2 * cp;
  const bool live = 2 * cp < nch;  // nch is a multiple of 8
  float w[2][4] = {}, bias[2] = {}, dw[2][4] = {}, db[2] = {};
  if (live) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float4 wq = reinterpret_cast<const float4 *>(pr.conv_w)[c + q];
      w[q][0] = wq.x; w[q][1] = wq.y; w[q][2] = wq.z; w[q][3] = wq.w;
      bias[q] = pr.conv_b[c + q];
    }
    // phase 1: dv rows r0 .. r0 + n1 - 1 (kTok + 3 rows over 8 row groups: the
    // first 3 groups take kRun + 1 rows, the others kRun); both channels of the
    // thread as one packed pair
    constexpr int kRun = kTok / 8;
    const int r0 = tq * kRun + min(tq, 3), n1 = tq < 3 ? kRun + 1 : kRun;
    const uint64_t w0 = pk2(w[0][0], w[1][0]), w1 = pk2(w[0][1], w[1][1]), w2 = pk2(w[0][2], w[1][2]),
                   w3 = pk2(w[0][3], w[1][3]), bp = pk2(bias[0], bias[1]), one = pk2(1.f, 1.f);
    uint64_t x0 = loadp(&xr[r0][2 * cp]), x1 = loadp(&xr[r0 + 1][2 * cp]), x2 = loadp(&xr[r0 + 2][2 * cp]);
    uint64_t dw0 = 0ull, dw1 = 0ull, dw2 = 0ull, dw3 = 0ull, dbp = 0ull;
    int s0 = 0, s1 = 0, s2 = 0;
    if (HasSeq) {
      s0 = seqs[r0];
      s1 = seqs[r0 + 1];
      s2 = seqs[r0 + 2];
    }
#pragma unroll
    for (int k = 0; k < kRun + 1; ++k) {
      if (k < n1) {
        const int r = r0 + k;  // token t0 + r, inputs at raw rows r .. r + 3
        const uint64_t x3 = loadp(&xr[r + 3][2 * cp]);
        const int sq = HasSeq ? seqs[r + 3] : 0;
        const bool m2 = !HasSeq || s2 == sq, m1 = !HasSeq || s1 == sq, m0 = !HasSeq || s0 == sq;
        const uint64_t g = *reinterpret_cast<const uint64_t *>(&dv[r][2 * cp]);
        uint64_t v = fma2(w3, x3, bp);
        v = fma2(m2 ? w2 : 0ull, x2, v);
        v = fma2(m1 ? w1 : 0ull, x1, v);
        v = fma2(m0 ? w0 : 0ull, x0, v);
        const uint64_t sg = act_sigmoid2<T>(v);
        // d = (g sg) (1 + v (1 - sg))
        const uint64_t d = mul2(mul2(g, sg), fma2(v, sub2(one, sg), one));
        if (r < kTok) {  // the tile's own tokens
          dbp = add2(dbp, d);
          dw3 = fma2(d, x3, dw3);
          dw2 = fma2(m2 ? d : 0ull, x2, dw2);
          dw1 = fma2(m1 ? d : 0ull, x1, dw1);
          dw0 = fma2(m0 ? d : 0ull, x0, dw0);
        }
        x0 = x1;
        x1 = x2;
        x2 = x3;
        s0 = s1; s1 = s2; s2 = sq;
        *reinterpret_cast<uint64_t *>(&dv[r][2 * cp]) = d;  // own elements only
      }
    }
    upk2(dw0, dw[0][0], dw[1][0]);
    upk2(dw1, dw[0][1], dw[1][1]);
    upk2(dw2, dw[0][2], dw[1][2]);
    upk2(dw3, dw[0][3], dw[1][3]);
    upk2(dbp, db[0], db[1]);
  }
  __syncthreads();
  // phase 2: dxr for rows s in [kRun tq, kRun tq + kRun) (token t0 + s) from dv rows s .. s + 3
  if (live) {
    constexpr int kRun = kTok / 8;
    const int sr0 = tq * kRun;
    const uint64_t w0 = pk2(w[0][0], w[1][0]), w1 = pk2(w[0][1], w[1][1]), w2 = pk2(w[0][2], w[1][2]),
                   w3 = pk2(w[0][3], w[1][3]);
    uint64_t d0 = *reinterpret_cast<const uint64_t *>(&dv[sr0][2 * cp]),
             d1 = *reinterpret_cast<const uint64_t *>(&dv[sr0 + 1][2 * cp]),
             d2 = *reinterpret_cast<const uint64_t *>(&dv[sr0 + 2][2 * cp]);
    T *dst = ct.grad + 2 * cp;
#pragma unroll
    for (int k = 0; k < kRun; ++k) {
      const int sr = sr0 + k, t = t0 + sr;
      const uint64_t d3 = *reinterpret_cast<const uint64_t *>(&dv[sr + 3][2 * cp]);
      bool m1 = true, m2 = true, m3 = true;
      if (HasSeq) {
        const int q0 = seqs[sr + 3];  // token t
        m1 = seqs[sr + 4] == q0;
        m2 = seqs[sr + 5] == q0;
        m3 = seqs[sr + 6] == q0;
      }
      uint64_t a = mul2(w3, d0);
      a = fma2(m1 ? w2 : 0ull, d1, a);
      a = fma2(m2 ? w1 : 0ull, d2, a);
      a = fma2(m3 ? w0 : 0ull, d3, a);
      d0 = d1;
      d1 = d2;
      d2 = d3;
      if (t < pr.L) storep(dst + (size_t)t * ct.gst, a);
    }
  }
  // parameter partials: fixed-order sum over the row groups (0..3 and 4..7 folded pairwise first)
  if (tq < 4) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) red[tq][2 * cp + q][kk] = dw[q][kk];
      red[tq][2 * cp + q][4] = db[q];
    }
  }
  __syncthreads();
  if (tq >= 4) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) red[tq & 3][2 * cp + q][kk] += dw[q][kk];
      red[tq & 3][2 * cp + q][4] += db[q];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nch * 5; e += 256) {
    const int ch = e / 5, k5 = e % 5;
    const float v = (red[0][ch][k5] + red[1][ch][k5]) + (red[2][ch][k5] + red[3][ch][k5]);
    convp[(((size_t)bb * ntb + blk) * pr.Cd + ct.c0 + ch) * 5 + k5] = v;
  }
}

template <typename T> constexpr int conv_bwd_smem() {
  return (int)(sizeof(float) * (kConvBwdTok + 3) * kBwdCh + sizeof(T) * (kConvBwdTok + 6) * kBwdCh +
               sizeof(int) * ((kConvBwdTok + 6 + 3) & ~3) + sizeof(float) * 4 * kBwdCh * 5);
}

template <typename T>
void launch_conv_bwd(const Problem &pr, const float *du, const BcParts &bc, const GradOut &go, float *convp, int ntb,
                     cudaStream_t s) {
  constexpr int smem = conv_bwd_smem<T>();
  static bool once = (cudaFuncSetAttribute(conv_bwd_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                      cudaFuncSetAttribute(conv_bwd_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                      true);
  (void)once;
  dim3 grid(chan_tiles(pr, kBwdCh), ntb, pr.b);
  if (pr.seq_idx)
    conv_bwd_kernel<T, true><<<grid, 256, smem, s>>>(pr, du, bc, go, convp, ntb);
  else
    conv_bwd_kernel<T, false><<<grid, 256, smem, s>>>(pr, du, bc, go, convp, ntb);
}

// Parameter gradients: fixed-order sums of per-chunk / per-block partials.
// Fixed xor-shuffle tree over a warp's lanes.
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Parameter gradients from the per-block partials, each sum in a fixed order.
// Conv: a block takes 32 consecutive elements of a partial row (Cd x 5 floats:
// dconv_w[c, 0..3], dconv_b[c]) and 8 interleaved slices of the b * ntb rows, so
// every warp load is one contiguous 128-byte line; the slices are added in
// order at the end.  Per head (one warp each, after the conv blocks): ddt_bias,
// dA_log and dD from the per-chunk scalars.
constexpr int kParamSlices = 8;
__global__ void __launch_bounds__(256) param_reduce_kernel(Problem pr, const float *__restrict__ chs,
                                                           const float *__restrict__ convp, int ntb,
                                                           float *ddt_bias, float *dA_log, float *dD,
                                                           float *dconv_w, float *dconv_b, int conv_blocks) {
  __shared__ float part[kParamSlices][32];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  if ((int)blockIdx.x < conv_blocks) {
    const int row = pr.Cd * 5, nparts = pr.b * ntb;
    const int e = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (e < row) {
      const float *pp = convp + e;
#pragma unroll 8
      for (int k = slice; k < nparts; k += kParamSlices) acc += pp[(size_t)k * row];
    }
    part[slice][lane] = acc;
    __syncthreads();
    if (slice == 0 && e < row) {
      float t = 0.f;
#pragma unroll
      for (int q = 0; q < kParamSlices; ++q) t += part[q][lane];
      const int c = e / 5, q = e % 5;
      if (q < 4)
        dconv_w[c * 4 + q] = t;
      else
        dconv_b[c] = t;
    }
    return;
  }
  const int h = (blockIdx.x - conv_blocks) * (blockDim.x >> 5) + slice;
  if (h >= pr.H) return;
  const size_t nch = (size_t)pr.b * pr.nc * pr.H;
  const int nparts = pr.b * pr.nc;
  float sb = 0.f, sa = 0.f, sd = 0.f;
  for (int k = lane; k < nparts; k += 32) {  // k = bb * nc + c
    const size_t o = (size_t)k * pr.H + h;
    sb += chs[o];
    sa += chs[nch + o];
    sd += chs[2 * nch + o];
  }
  sb = warp_tree_sum(sb);
  sa = warp_tree_sum(sa);
  sd = warp_tree_sum(sd);
  if (lane == 0) {
    ddt_bias[h] = sb;
    dA_log[h] = sa * (-expf(pr.A_log[h]));  // dA/dA_log = A
    dD[h] = sd;
  }
}

void launch_param_reduce(const Problem &pr, const float *chs, const float *convp, int ntb, float *ddt_bias,
                         float *dA_log, float *dD, float *dconv_w, float *dconv_b, cudaStream_t s) {
  const int conv_blocks = (pr.Cd * 5 + 31) / 32, head_blocks = (pr.H + 7) / 8;
  param_reduce_kernel<<<conv_blocks + head_blocks, 256, 0, s>>>(pr, chs, convp, ntb, ddt_bias, dA_log, dD, dconv_w,
                                                                dconv_b, conv_blocks);
}

__global__ void cu_seqlens_kernel(const int *__restrict__ cu, int nseq, int *__restrict__ seq_idx, int total) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  int lo = 0, hi = nseq;  // find i with cu[i] <= t < cu[i+1]
  if (t < cu[0] || t >= cu[nseq]) {
    seq_idx[t] = -1;
    return;
  }
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  seq_idx[t] = lo;
}

void launch_cu_seqlens(const int *cu, int nseq, int *seq_idx, int total, cudaStream_t s) {
  cu_seqlens_kernel<<<(total + 255) / 256, 256, 0, s>>>(cu, nseq, seq_idx, total);
}

template void launch_conv_fwd<float>(const Problem &, float *, float *, float *, cudaStream_t);
template void launch_conv_fwd<__nv_bfloat16>(const Problem &, __nv_bfloat16 *, float *, float *, cudaStream_t);
template void launch_conv_bwd<float>(const Problem &, const float *, const BcParts &, const GradOut &, float *, int,
                                     cudaStream_t);
template void launch_conv_bwd<__nv_bfloat16>(const Problem &, const float *, const BcParts &, const GradOut &, float *,
                                             int,
                                             cudaStream_t);

}  // namespace ssd
