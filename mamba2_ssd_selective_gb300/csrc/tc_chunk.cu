// Chunk-state and Z kernels of the bf16 path on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM): the per-chunk states
//   S_c,h = sum_j wdt_h,j x_j,h B_j^T      (wdt_h,j = exp(Acs_last - Acs_j) dt_j,
//                                           0 outside the chunk's last sequence)
// and the adjoint feeding the reverse boundary scan
//   Z_c,h = sum_i em_h,i dy_i,h C_i^T      (em_h,i = exp(Acs_i), 0 for tokens that
//                                           do not continue the incoming state),
// the chunked form of the Mamba2 SSD.  Same formulas as the CUDA-core kernels
// in simt_chunk.cu.  The output and the chunk gradients run in the persistent
// kernels of tc_out.cu, tc_bwd_row.cu and tc_bwd_col.cu.
//
// One persistent, warp-specialised kernel serves both (one CTA per SM, 15
// warps).  Work unit = (batch row, chunk, block of HB heads of one group):
//   warp 0      TMA producer: the unit's A tile (B or C of the group, all Q
//               tokens, double-buffered across units), per head the chunk
//               vectors (Acs, dt, seq) and the Q/64 operand slices
//               [64 tokens x 64] of x_h or dy_h into an 11-slice ring;
//   warp 1      TMEM owner and MMA issuer: per head D^T[n, p] = sum_t A[t, n] X'[t, p]
//               (M = dstate 128, N = headdim 64, both operands MN-major) into
//               one of four 64-column accumulators;
//   warps 2-9   transform: scale each landed slice in place by the per-token
//               weight (wdt or em), rounded to bf16 as the MMA's operand;
//   warps 10-13 epilogue: drain an accumulator (TMEM lane = n) into the
//               (P, N) state, 128 consecutive n per store instruction;
//   warp 14     the chunk-state instance only: the decay tables of a share of
//               the (row, head) pairs (cdec, dstart, dend, a_block), which no
//               other part of this kernel reads, instead of a launch of their own.
// The slice ring keeps about 88 KB of loads in flight per SM, and the next
// unit's A tile loads while the current one is still in use.
//
// Envelope (checked on the host): bf16 activations, headdim 64, dstate 128,
// chunk 128 or 256, an even number of heads per group.
#include "kernels.h"
#include "tc_util.cuh"
#include "tc_pipe.cuh"

namespace ssd {

namespace {

using bf16 = __nv_bfloat16;
using namespace sm100;
using pipe::parity;

constexpr int kWarps = 15, kThreads = kWarps * 32;
constexpr int kTWarp0 = 2, kTWarps = 8;              // transform: warps 2-9
constexpr int kEWarp0 = kTWarp0 + kTWarps, kEWarps = 4;  // epilogue: warps 10-13
constexpr int kTabWarp = kEWarp0 + kEWarps;          // decay tables: warp 14
constexpr int kNX = 11;   // operand slice ring, [64 tokens x 64 columns] bf16 each
constexpr int kNAcc = 4;  // accumulators in tensor memory, 64 columns each

constexpr uint32_t kSmA = 0;                      // 2 x A tile: Q/64 slices x 2 n halves x [64 tokens x 128 B]
constexpr uint32_t kSmX = kSmA + 2 * 65536;       // ring of operand slices
constexpr uint32_t kVecStride = 3200;             // acs[256] | dt[256] | seq[4 + 256]
constexpr uint32_t kSmV = kSmX + kNX * 8192;      // 2 vector buffers
constexpr uint32_t kSmBar = kSmV + 2 * kVecStride;
constexpr int kNumBars = 4 + 3 * kNX + 2 * kNAcc + 4 + 4 + 1;
constexpr uint32_t kSmEnd = kSmBar + kNumBars * 8 + 16;
constexpr int kSmemBytes = (int)kSmEnd + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Unit {
  int bb, c, h0;
};

struct DecayTabs {
  float *cdec, *dstart, *dend, *ablk;
};

// Unit u: the head blocks of one (row, chunk) adjacent, so that the CTAs
// working on them at about the same time share the A tile in L2.
__device__ __forceinline__ Unit unit_of(const Problem &pr, int nhb, int HB, int u) {
  Unit o;
  const int hb = u % nhb, bc = u / nhb;
  o.c = bc % pr.nc;
  o.bb = bc / pr.nc;
  o.h0 = hb * HB;
  return o;
}

struct Bars {
  uint64_t *a_full, *a_free;                // [2]
  uint64_t *x_full, *x_ready, *x_free;      // [kNX]: landed, scaled, read by the MMAs
  uint64_t *acc_full, *acc_free;            // [kNAcc]
  uint64_t *vec_full, *vec_free;            // [2]
  uint64_t *drain;                          // the MMA issuer's final commit
  pipe::UnitRing units;
  __device__ Bars(uint64_t *b, int *slot) {
    a_full = b;
    a_free = b + 2;
    x_full = b + 4;
    x_ready = x_full + kNX;
    x_free = x_ready + kNX;
    acc_full = x_free + kNX;
    acc_free = acc_full + kNAcc;
    vec_full = acc_free + kNAcc;
    vec_free = vec_full + 2;
    units.full = vec_free + 2;
    units.free = units.full + 2;
    drain = units.free + 2;
    units.slot = slot;
  }
};

}  // namespace

// kZ = false: S_c (A = B, operand x, weight wdt, out = sst), and the decay
//             tables into tab = {cdec, dstart, dend, ablk};
// kZ = true:  Z_c (A = C, operand dy, weight em, out = dsl); tab unused.
// Both outputs are (b, nc, H, P, N) fp32.
template <bool kZ>
__global__ void __launch_bounds__(kThreads, 1)
    tc_sz_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_x, Problem pr,
                 const float *__restrict__ dtv, const float *__restrict__ acs, float *__restrict__ out,
                 DecayTabs tab, int HB, int nunits, int *counter, int *status_word) {
  extern __shared__ uint8_t smem_raw[];
  const WaitCtl status{status_word, pr.wait_ns};
  uint8_t *sm = tc::aligned_smem(smem_raw);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + kSmBar + kNumBars * 8);
  Bars bar(reinterpret_cast<uint64_t *>(sm + kSmBar), reinterpret_cast<int *>(tslot + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nhb = pr.H / HB, HP = pr.H * pr.P, nsl = pr.Q / 64;
  const bool has_seq = pr.seq_idx != nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.a_full[i], 1);
      mbar_init(&bar.a_free[i], 1);
      mbar_init(&bar.vec_full[i], 1);
      mbar_init(&bar.vec_free[i], kTWarps);
      mbar_init(&bar.units.full[i], 1);
      mbar_init(&bar.units.free[i], 1 + kTWarps + kEWarps);
    }
    for (int i = 0; i < kNX; ++i) {
      mbar_init(&bar.x_full[i], 1);
      mbar_init(&bar.x_ready[i], kTWarps);
      mbar_init(&bar.x_free[i], 1);
    }
    for (int i = 0; i < kNAcc; ++i) {
      mbar_init(&bar.acc_full[i], 1);
      mbar_init(&bar.acc_free[i], kEWarps);
    }
    mbar_init(bar.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_u);
      prefetch_tmap(&tm_x);
      // counts of armed loads per barrier; once a wait has failed (ok = false)
      // no further load is issued, stop is published, and the loads in flight
      // are drained before the CTA ends
      uint32_t nu = 0, nua = 0, nh = 0, k = 0;
      bool ok = true;
      int next = atomicAdd(counter, 1);
      for (;; ++nu) {
        const int ui = pipe::publish_unit(bar.units, nu, ok ? next : nunits, nunits);
        if (ui >= nunits) break;
        next = atomicAdd(counter, 1);
        const Unit o = unit_of(pr, nhb, HB, ui);
        const int g = o.h0 / pr.hpg, t0 = o.c * pr.Q, row0 = o.bb * pr.L + t0;
        const int offA = kZ ? HP + pr.G * pr.N + g * pr.N : HP + g * pr.N;
        const int ab = nu & 1;
        if (nu >= 2) ok = mbar_wait(&bar.a_free[ab], parity(nu / 2 - 1), status);
        if (!ok) continue;
        mbar_expect_tx(&bar.a_full[ab], nsl * 16384);
        for (int s = 0; s < nsl; ++s)
          for (int mh = 0; mh < 2; ++mh)
            tma_load_2d(sm + kSmA + ab * 65536 + s * 16384 + mh * 8192, &tm_u, &bar.a_full[ab], offA + 64 * mh,
                        row0 + 64 * s);
        ++nua;
        for (int hh = 0; hh < HB && ok; ++hh) {
          const int h = o.h0 + hh, vb = nh & 1;
          if (nh >= 2 && !mbar_wait(&bar.vec_free[vb], parity(nh / 2 - 1), status)) {
            ok = false;
            break;
          }
          uint8_t *vec = sm + kSmV + vb * kVecStride;
          const size_t bh = ((size_t)o.bb * pr.H + h) * pr.L + t0;
          // Z also needs the seq id of the token before the chunk (at vec + 2048 + 12)
          const bool seq_prev = kZ && o.c > 0;
          const uint32_t seq_bytes = !has_seq ? 0u : (uint32_t)(seq_prev ? (pr.Q + 4) * 4 : pr.Q * 4);
          mbar_expect_tx(&bar.vec_full[vb], (kZ ? 1 : 2) * pr.Q * 4 + seq_bytes);
          pipe::bulk_load(vec, acs + bh, pr.Q * 4, &bar.vec_full[vb]);
          if (!kZ) pipe::bulk_load(vec + 1024, dtv + bh, pr.Q * 4, &bar.vec_full[vb]);
          if (has_seq) {
            const int *sq = pr.seq_idx + (size_t)o.bb * pr.L + t0;
            if (seq_prev)
              pipe::bulk_load(vec + 2048, sq - 4, seq_bytes, &bar.vec_full[vb]);
            else
              pipe::bulk_load(vec + 2048 + 16, sq, seq_bytes, &bar.vec_full[vb]);
          }
          ++nh;
          for (int s = 0; s < nsl; ++s) {
            const int slot = k % kNX;
            if (k >= kNX && !mbar_wait(&bar.x_free[slot], parity(k / kNX - 1), status)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&bar.x_full[slot], 8192);
            tma_load_2d(sm + kSmX + slot * 8192, &tm_x, &bar.x_full[slot], h * pr.P, row0 + 64 * s);
            ++k;
          }
        }
      }
      // every load issued has landed before the CTA releases its shared memory
      for (uint32_t m = nua > 2u ? nua - 2u : 0u; m < nua; ++m) mbar_wait_drain(&bar.a_full[m & 1], parity(m / 2));
      for (uint32_t m = nh > 2u ? nh - 2u : 0u; m < nh; ++m) mbar_wait_drain(&bar.vec_full[m & 1], parity(m / 2));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_full[m % kNX], parity(m / kNX));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t dA = desc_sw128(smem_u32(sm + kSmA), 8192, 1024), dX = desc_sw128(smem_u32(sm + kSmX), 8192, 1024);
      constexpr uint32_t idesc = idesc_bf16(128, 64, true, true);
      uint32_t nu = 0, nh = 0, k = 0;
      for (;; ++nu) {
        const int ui = pipe::next_unit(bar.units, nu, nunits, false);
        if (ui >= nunits) break;
        const int ab = nu & 1;
        mbar_wait(&bar.a_full[ab], parity(nu / 2), status);
        for (int hh = 0; hh < HB; ++hh, ++nh) {
          const int as = nh % kNAcc;
          const uint32_t tacc = tmem + 64 * as;
          if (nh >= (uint32_t)kNAcc) mbar_wait(&bar.acc_free[as], parity(nh / kNAcc - 1), status);
          for (int s = 0; s < nsl; ++s, ++k) {
            const int slot = k % kNX;
            mbar_wait(&bar.x_ready[slot], parity(k / kNX), status);
            tc_fence_after();
            pipe::umma_k<4>(tacc, dA + (ab * 65536 + s * 16384) / 16, dX + slot * (8192 / 16), pipe::kStepMN,
                            pipe::kStepMN, idesc, s > 0);
            umma_commit(&bar.x_free[slot]);
          }
          umma_commit(&bar.acc_full[as]);
        }
        umma_commit(&bar.a_free[ab]);
      }
      // drain: every MMA issued here has completed and every commit arrival
      // has landed before the CTA releases its shared and tensor memory
      umma_commit(bar.drain);
      mbar_wait_drain(bar.drain, 0);
      for (uint32_t m = nu > 2u ? nu - 2u : 0u; m < nu; ++m) mbar_wait_drain(&bar.a_free[m & 1], parity(m / 2));
      for (uint32_t m = nh > (uint32_t)kNAcc ? nh - kNAcc : 0u; m < nh; ++m)
        mbar_wait_drain(&bar.acc_full[m % kNAcc], parity(m / kNAcc));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_free[m % kNX], parity(m / kNX));
    }
  } else if (warp < kEWarp0) {
    // ------------------------------------------------------------ transform
    // thread tt scales 16-byte chunks tt and tt + 256 of each 8 KB slice: token
    // row r = chunk / 8 of the slice, 8 columns (chunk % 8)
    const int tt = threadIdx.x - 32 * kTWarp0;
    const uint32_t sX = smem_u32(sm + kSmX), sV = smem_u32(sm + kSmV);
    uint32_t nu = 0, nh = 0, k = 0;
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, nhb, HB, ui);
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int vb = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vdt = vacs + 1024, vseq = vacs + 2048 + 16;
        // the weights of this thread's two token rows in every slice
        int ref_seq = 0;
        bool use_ref = false;
        float acs_last = 0.f;
        if constexpr (kZ) {
          use_ref = chunk_has_incoming(pr, o.c);
          if (use_ref && has_seq) ref_seq = pipe::lds_i(o.c > 0 ? vseq - 4 : vseq);
        } else {
          acs_last = pipe::lds_f(vacs + 4 * (pr.Q - 1));
          if (has_seq) ref_seq = pipe::lds_i(vseq + 4 * (pr.Q - 1));
        }
        float wt[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = e >> 1, r = (tt >> 3) + 32 * (e & 1), t = 64 * s + r;
          float w = 0.f;
          if (s < nsl) {
            const float a = pipe::lds_f(vacs + 4 * t);
            const bool same = !has_seq || pipe::lds_i(vseq + 4 * t) == ref_seq;
            if constexpr (kZ)
              w = (use_ref && same) ? expf(a) : 0.f;
            else
              w = same ? expf(acs_last - a) * pipe::lds_f(vdt + 4 * t) : 0.f;
          }
          wt[e] = w;
        }
        pipe::warp_arrive(&bar.vec_free[vb]);
#pragma unroll
        for (int s = 0; s < 4; ++s, ++k) {  // Q / 64 = nsl <= 4 slices
          if (s >= nsl) break;
          const int slot = k % kNX;
          mbar_wait(&bar.x_full[slot], parity(k / kNX), status);
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int ch = tt + 256 * e2, r = ch >> 3, cc = ch & 7;
            const uint32_t a = sX + slot * 8192 + sw128_offset(r, 8 * cc);
            float v[8];
            uint4 raw;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                         : "r"(a));
            tc::unpack8(raw, v);
            const float w = wt[2 * s + e2];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] *= w;
            pipe::sts_u4(a, tc::pack8(v));
          }
          fence_async_smem();
          pipe::warp_arrive(&bar.x_ready[slot]);
        }
      }
    }
  } else if (warp < kTabWarp) {
    // ------------------------------------------------------------ epilogue
    // thread = state column n (TMEM lane); out[(b, c, h), p, n]
    const int n = 32 * (warp & 3) + lane;
    uint32_t nu = 0, nh = 0;
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, nhb, HB, ui);
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, as = nh % kNAcc;
        mbar_wait(&bar.acc_full[as], parity(nh / kNAcc), status);
        tc_fence_after();
        float *dst = out + (((size_t)o.bb * pr.nc + o.c) * pr.H + h) * pr.P * pr.N + n;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          float v[32];
          tmem_ld32(pipe::tmem_quad(tmem + 64 * as, 32 * cc), v);
#pragma unroll
          for (int p = 0; p < 32; ++p) dst[(size_t)(32 * cc + p) * pr.N] = v[p];
        }
        tc_fence_before();
        pipe::warp_arrive(&bar.acc_free[as]);
      }
    }
  } else if constexpr (!kZ) {
    // ------------------------------------------------------------ decay tables
    // (row, head) pairs blockIdx.x, blockIdx.x + gridDim.x, ..., a lane per chunk
    for (int p = blockIdx.x; p < pr.b * pr.H; p += gridDim.x)
      decay_tables_bh(pr, acs, p / pr.H, p % pr.H, tab.cdec, tab.dstart, tab.dend, tab.ablk, lane, 32,
                      [] { __syncwarp(); });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

namespace {

// heads per unit: 8 (or the largest power of two dividing the group's heads)
int sz_head_block(const Problem &pr) {
  for (int hs : {8, 4, 2})
    if (pr.hpg % hs == 0) return hs;
  return 1;
}

template <bool kZ>
void launch_sz(const Problem &pr, const bf16 *u, const bf16 *xsrc, const float *dtv, const float *acs, float *out,
               DecayTabs tab, int *status, cudaStream_t s) {
  static bool once = (cudaFuncSetAttribute(tc_sz_kernel<kZ>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes),
                      true);
  (void)once;
  CUtensorMap tm_u, tm_x;
  const uint64_t HP = (uint64_t)pr.H * pr.P;
  const uint64_t xcols = kZ ? HP : (uint64_t)pr.Cd;
  if (!encode_tmap_bf16_2d(&tm_u, u, pr.Cd, (uint64_t)pr.b * pr.L, (uint64_t)pr.Cd * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_x, xsrc, xcols, (uint64_t)pr.b * pr.L, xcols * 2, 64, 64)) {
    note_host_error();
    return;
  }
  const int HB = sz_head_block(pr);
  const int nunits = pr.b * pr.nc * (pr.H / HB);
  const int grid = nunits < device_sm_count() ? nunits : device_sm_count();
  int *counter = status + (kZ ? kCounterZ : kCounterState);  // zeroed with the status word
  tc_sz_kernel<kZ><<<grid, kThreads, kSmemBytes, s>>>(tm_u, tm_x, pr, dtv, acs, out, tab, HB, nunits, counter,
                                                      status);
}

}  // namespace

void launch_tc_state(const Problem &pr, const bf16 *u, const float *dtv, const float *acs, float *sst, float *cdec,
                     float *dstart, float *dend, float *ablk, int *status, cudaStream_t s) {
  launch_sz<false>(pr, u, u, dtv, acs, sst, DecayTabs{cdec, dstart, dend, ablk}, status, s);
}

void launch_tc_z(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs, float *dsl,
                 int *status, cudaStream_t s) {
  launch_sz<true>(pr, u, dy, dtv, acs, dsl, DecayTabs{}, status, s);
}

int tc_head_subset(const Problem &pr) {
  for (int hs : {16, 8, 4, 2})
    if (pr.hpg % hs == 0) return hs;
  return 1;
}

}  // namespace ssd
