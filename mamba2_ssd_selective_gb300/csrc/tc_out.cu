// Chunk output of the bf16 path (Mamba2 SSD, chunked form: the diagonal block
// Y_diag = (C B^T o L o dt) X plus the off-diagonal term em o (C S_in^T)), as a
// persistent, warp-specialised tcgen05 kernel.
//
// Work unit = (batch row, chunk, 128-token row tile I, block of HB heads of one
// group).  Per unit the tensor cores first form CB = C_I B^T (K = dstate) into
// tensor memory, once for all HB heads; then per head
//   Yd  = A_h X_h,   A_h[i, j] = CB[i, j] exp(Acs_i - Acs_j) dt_j [j <= i, same sequence]
//   Yo  = C_I S_in,h^T       (every chunk that receives a state: all but a row's
//                            first, and that one too when the row has an initial state)
//   y_i = Yd_i + em_i Yo_i + D_h x_i.
// Roles (22 warps, one CTA per SM):
//   warp 0      TMA producer: C/B tiles per unit, per head the chunk vectors
//               (Acs, dt, seq), 64-token X slices and the bf16 S_in tile;
//   warp 1      TMEM owner and MMA issuer (one thread);
//   warps 2-17  transform: read CB rows from TMEM, apply mask, decay and dt,
//               write the bf16 A slice back into tensor memory, where the MMA
//               takes it as its A operand (four warps per lane quadrant, one per
//               16-column group of the 64-wide slice = one K step of 8 columns);
//   warps 18-21 epilogue: drain the two per-head accumulators and write y.
// Decays without an exponential per element: Acs does not increase along the
// chunk, so for a 16-column group ending at column m and rows i >= m
//   exp(Acs_i - Acs_j) dt_j = exp(Acs_i - Acs_m) * [exp(Acs_m - Acs_j) dt_j],
// both factors <= 1 (dt_j aside): the bracket is tabulated per head and
// column, the first factor costs one 2^x per row and group.  Groups that
// straddle the diagonal use 2^(a_i + b_j) per element, a_i = Acs_i log2(e),
// b_j = log2(dt_j) - Acs_j log2(e).  The mask is the row's interval
// [start_i, i], start_i the first token of i's sequence inside the chunk.
// The Yd accumulator is double-buffered, so the epilogue of head n overlaps the
// transform and MMAs of head n+1; Yo, formed at the end of a head, has one
// buffer (the epilogue has read the previous head's long before).  The X
// slices have their own ring, deep enough to cover the TMA latency; the A
// slices never leave tensor memory.
#include "chunk_common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tc_pipe.cuh"

namespace ssd {

namespace {

using bf16 = __nv_bfloat16;
using namespace sm100;
using pipe::parity;

constexpr int kWarps = 22;
constexpr int kEpiWarp0 = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kNA = 2;   // A slice slots in tensor memory (transform -> MMA)
constexpr int kNX = 4;   // X slice ring (TMA -> MMA; a head of a 256-token tile; deeper rings measured slower)
constexpr int kNSB = 2;  // S_in buffers (loaded a head ahead of use)

// shared memory map, offsets from the 1024-aligned base
constexpr uint32_t kSmC = 0;                     // C_I: 2 K halves x [128 rows x 128 B]
constexpr uint32_t kSmB = kSmC + 2 * 16384;      // B rows: 2 K halves x [256 rows x 128 B]
constexpr uint32_t kSmX = kSmB + 2 * 32768;      // ring of X slices [64 tokens x 64] bf16, MN-major
constexpr uint32_t kSmS = kSmX + kNX * 8192;     // kNSB x S_in,h: 2 K halves x [64 x 128 B]
constexpr uint32_t kVecStride = 3200;            // acs[256] f32 | dt[256] f32 | seq[4 + 256] i32
constexpr uint32_t kSmV = kSmS + kNSB * 16384;   // 2 vector buffers
constexpr uint32_t kSmD = kSmV + 2 * kVecStride;   // 2 x {a[256], b[256], f[256]} f32 (decay tables per head)
constexpr uint32_t kSmBar = kSmD + 2 * 3072;
constexpr int kNumBars = 9 + 2 * kNA + 2 * kNX + 2 * kNSB + 4 + 4 + 1;
constexpr uint32_t kSmEnd = kSmBar + kNumBars * 8 + 16;
constexpr int kSmemBytes = (int)kSmEnd + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// tensor memory: [0, 256) CB | [256, 384) Yd[2] | [384, 448) Yo | [448, 512) A[2]
// (a slot: 4 K steps x 8 columns of bf16 pairs, element 2c in the low half of column c)
constexpr uint32_t kTmYd = 256, kTmYo = 384, kTmA = 448;

struct Unit {
  int bb, c, I, h0;
};

// Unit u of the launch, claimed dynamically in this order: the tiles with more
// work first (every CTA then ends on light ones), and within a tile class the
// head blocks of one (row, chunk) adjacent, sharing C and B in L2.
__device__ __forceinline__ Unit unit_of(const Problem &pr, int NTI, int nhb, int HB, int u) {
  const int per = pr.b * pr.nc * nhb;
  const int cls = u / per, r = u % per;
  Unit o;
  o.I = NTI - 1 - cls;
  const int hb = r % nhb, bc = r / nhb;
  o.c = bc % pr.nc;
  o.bb = bc / pr.nc;
  o.h0 = hb * HB;
  return o;
}

struct Bars {
  uint64_t *unit_full, *b_free, *c_free, *cb_full, *cb_used;
  uint64_t *vec_full, *vec_free;             // [2]
  uint64_t *a_full, *a_free;                 // [kNA]
  uint64_t *x_full, *x_free;                 // [kNX]
  uint64_t *s_full, *s_free;                 // [kNSB]
  uint64_t *acc_full, *acc_free;             // [2]
  uint64_t *drain;                           // the MMA issuer's final commit
  pipe::UnitRing units;
  __device__ Bars(uint64_t *b, int *slot) {
    unit_full = b;
    b_free = b + 1;
    c_free = b + 2;
    cb_full = b + 3;
    cb_used = b + 4;
    vec_full = b + 5;
    vec_free = b + 7;
    a_full = b + 9;
    a_free = a_full + kNA;
    x_full = a_free + kNA;
    x_free = x_full + kNX;
    s_full = x_free + kNX;
    s_free = s_full + kNSB;
    acc_full = s_free + kNSB;
    acc_free = acc_full + 2;
    units.full = acc_free + 2;
    units.free = units.full + 2;
    drain = units.free + 2;
    units.slot = slot;
  }
};

constexpr int kTransformThreads = 16 * 32;
constexpr int kTransformWarps = 16, kEpilogueWarps = 4;


}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    tc_out_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_s, Problem pr,
                  const bf16 *__restrict__ u, const float *__restrict__ dtv, const float *__restrict__ acs,
                  bf16 *__restrict__ y, int HB, int nunits, int *counter, int *status_word) {
  extern __shared__ uint8_t smem_raw[];
  const WaitCtl status{status_word, pr.wait_ns};
  uint8_t *sm = tc::aligned_smem(smem_raw);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + kSmBar + kNumBars * 8);
  Bars bar(reinterpret_cast<uint64_t *>(sm + kSmBar), reinterpret_cast<int *>(tslot + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NTI = pr.Q / 128, nhb = pr.H / HB, HP = pr.H * pr.P, Cd = pr.Cd;
  const bool has_seq = pr.seq_idx != nullptr;

  if (threadIdx.x == 0) {
    mbar_init(bar.unit_full, 1);
    mbar_init(bar.b_free, 1);
    mbar_init(bar.c_free, 1);
    mbar_init(bar.cb_full, 1);
    mbar_init(bar.cb_used, kTransformWarps);
    mbar_init(bar.drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.vec_full[i], 1);
      mbar_init(&bar.vec_free[i], kTransformWarps + kEpilogueWarps);
      mbar_init(&bar.acc_full[i], 1);
      mbar_init(&bar.acc_free[i], kEpilogueWarps);
    }
    for (int i = 0; i < kNSB; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.units.full[i], 1);
      mbar_init(&bar.units.free[i], 1 + kTransformWarps + kEpilogueWarps);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&bar.a_full[i], kTransformWarps);
      mbar_init(&bar.a_free[i], 1);
    }
    for (int i = 0; i < kNX; ++i) {
      mbar_init(&bar.x_full[i], 1);
      mbar_init(&bar.x_free[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
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
      prefetch_tmap(&tm_s);
      // counts of armed loads per barrier (nua: unit operand sets); once a
      // wait has failed (ok = false) no further load is issued, stop is
      // published, and the loads in flight are drained before the CTA ends
      uint32_t nu = 0, nua = 0, nh = 0, ns = 0, k = 0;
      bool ok = true;
      int next = atomicAdd(counter, 1);
      for (;; ++nu) {
        const int ui = pipe::publish_unit(bar.units, nu, ok ? next : nunits, nunits);
        if (ui >= nunits) break;
        next = atomicAdd(counter, 1);
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int g = o.h0 / pr.hpg, t0 = o.c * pr.Q, row0 = o.bb * pr.L + t0, NB = 128 * (o.I + 1);
        const int offB = HP + g * pr.N, offC = HP + pr.G * pr.N + g * pr.N;
        if (nu > 0) ok = mbar_wait(bar.b_free, parity(nu - 1), status) && mbar_wait(bar.c_free, parity(nu - 1), status);
        if (!ok) continue;
        mbar_expect_tx(bar.unit_full, 2 * 16384 + 2 * NB * 128);
        for (int kh = 0; kh < 2; ++kh) {
          for (int r = 0; r < 2; ++r)
            tma_load_2d(sm + kSmC + kh * 16384 + r * 8192, &tm_u, bar.unit_full, offC + 64 * kh, row0 + 128 * o.I + 64 * r);
          for (int r = 0; r < NB / 64; ++r)
            tma_load_2d(sm + kSmB + kh * 32768 + r * 8192, &tm_u, bar.unit_full, offB + 64 * kh, row0 + 64 * r);
        }
        ++nua;
        for (int hh = 0; hh < HB && ok; ++hh) {
          const int h = o.h0 + hh, vb = nh & 1;
          if (nh >= 2 && !mbar_wait(&bar.vec_free[vb], parity(nh / 2 - 1), status)) {
            ok = false;
            break;
          }
          uint8_t *vec = sm + kSmV + vb * kVecStride;
          const size_t bh = ((size_t)o.bb * pr.H + h) * pr.L + t0;
          const uint32_t seq_bytes = !has_seq ? 0u : (uint32_t)(o.c > 0 ? (pr.Q + 4) * 4 : pr.Q * 4);
          mbar_expect_tx(&bar.vec_full[vb], 2 * pr.Q * 4 + seq_bytes);
          pipe::bulk_load(vec, acs + bh, pr.Q * 4, &bar.vec_full[vb]);
          pipe::bulk_load(vec + 1024, dtv + bh, pr.Q * 4, &bar.vec_full[vb]);
          if (has_seq) {
            if (o.c > 0)
              pipe::bulk_load(vec + 2048, pr.seq_idx + (size_t)o.bb * pr.L + t0 - 4, seq_bytes, &bar.vec_full[vb]);
            else
              pipe::bulk_load(vec + 2048 + 16, pr.seq_idx + (size_t)o.bb * pr.L + t0, seq_bytes, &bar.vec_full[vb]);
          }
          ++nh;
          if (chunk_has_incoming(pr, o.c)) {
            const int sb = ns % kNSB;
            if (ns >= kNSB && !mbar_wait(&bar.s_free[sb], parity(ns / kNSB - 1), status)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&bar.s_full[sb], 16384);
            const int srow = (int)((((size_t)o.bb * pr.nc + o.c) * pr.H + h) * pr.P);
            tma_load_2d(sm + kSmS + sb * 16384, &tm_s, &bar.s_full[sb], 0, srow);
            tma_load_2d(sm + kSmS + sb * 16384 + 8192, &tm_s, &bar.s_full[sb], 64, srow);
            ++ns;
          }
          for (int s = 0; s < 2 * (o.I + 1); ++s) {
            const int slot = k % kNX;
            if (k >= kNX && !mbar_wait(&bar.x_free[slot], parity(k / kNX - 1), status)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&bar.x_full[slot], 8192);
            tma_load_2d(sm + kSmX + slot * 8192, &tm_u, &bar.x_full[slot], h * pr.P, row0 + 64 * s);
            ++k;
          }
        }
      }
      // every load issued has landed before the CTA releases its shared memory
      if (nua > 0) mbar_wait_drain(bar.unit_full, parity(nua - 1));
      for (uint32_t m = nh > 2u ? nh - 2u : 0u; m < nh; ++m) mbar_wait_drain(&bar.vec_full[m & 1], parity(m / 2));
      for (uint32_t m = ns > (uint32_t)kNSB ? ns - kNSB : 0u; m < ns; ++m)
        mbar_wait_drain(&bar.s_full[m % kNSB], parity(m / kNSB));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_full[m % kNX], parity(m / kNX));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // operand descriptors, built once; ring slots and K steps are additions
      const uint64_t dC = desc_sw128(smem_u32(sm + kSmC), 16, 1024), dB = desc_sw128(smem_u32(sm + kSmB), 16, 1024),
                     dX = desc_sw128(smem_u32(sm + kSmX), 8192, 1024),
                     dS = desc_sw128(smem_u32(sm + kSmS), 16, 1024);
      constexpr uint32_t id_acc = idesc_bf16(128, 64, false, true);
      constexpr uint32_t id_off = idesc_bf16(128, 64, false, false);
      uint32_t nu = 0, nh = 0, ns = 0, k = 0;
      for (;; ++nu) {
        const int ui = pipe::next_unit(bar.units, nu, nunits, false);
        if (ui >= nunits) break;
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int NB = 128 * (o.I + 1);
        mbar_wait(bar.unit_full, parity(nu), status);
        if (nu > 0) mbar_wait(bar.cb_used, parity(nu - 1), status);
        tc_fence_after();
        const uint32_t id_cb = idesc_bf16(128, NB, false, false);
        pipe::umma_k<4>(tmem, dC, dB, pipe::kStepK, pipe::kStepK, id_cb, false);
        pipe::umma_k<4>(tmem, dC + 16384 / 16, dB + 32768 / 16, pipe::kStepK, pipe::kStepK, id_cb, true);
        umma_commit(bar.cb_full);
        umma_commit(bar.b_free);
        for (int hh = 0; hh < HB; ++hh, ++nh) {
          const int ab = nh & 1;
          const uint32_t tyd = tmem + kTmYd + 64 * ab;
          if (nh >= 2) mbar_wait(&bar.acc_free[ab], parity(nh / 2 - 1), status);
          tc_fence_after();
          for (int s = 0; s < 2 * (o.I + 1); ++s, ++k) {
            const int as = k % kNA, xs = k % kNX;
            mbar_wait(&bar.a_full[as], parity(k / kNA), status);
            mbar_wait(&bar.x_full[xs], parity(k / kNX), status);
            tc_fence_after();
            pipe::umma_ts_k<4>(tyd, tmem + kTmA + 32 * as, dX + xs * (8192 / 16), 8, pipe::kStepMN, id_acc, s > 0);
            umma_commit(&bar.a_free[as]);
            umma_commit(&bar.x_free[xs]);
          }
          if (chunk_has_incoming(pr, o.c)) {
            const int sb = ns % kNSB;
            mbar_wait(&bar.s_full[sb], parity(ns / kNSB), status);
            // one Yo buffer: the previous head's epilogue has read it
            if (nh >= 1) mbar_wait(&bar.acc_free[(nh - 1) & 1], parity((nh - 1) / 2), status);
            tc_fence_after();
            const uint64_t dSb = dS + sb * (16384 / 16);
            pipe::umma_k<4>(tmem + kTmYo, dC, dSb, pipe::kStepK, pipe::kStepK, id_off, false);
            pipe::umma_k<4>(tmem + kTmYo, dC + 16384 / 16, dSb + 8192 / 16, pipe::kStepK, pipe::kStepK, id_off, true);
            umma_commit(&bar.s_free[sb]);
            ++ns;
          }
          umma_commit(&bar.acc_full[ab]);
        }
        umma_commit(bar.c_free);
      }
      // drain: every MMA issued here has completed and every commit arrival
      // has landed before the CTA releases its shared and tensor memory
      umma_commit(bar.drain);
      mbar_wait_drain(bar.drain, 0);
      if (nu > 0) {
        mbar_wait_drain(bar.cb_full, parity(nu - 1));
        mbar_wait_drain(bar.b_free, parity(nu - 1));
        mbar_wait_drain(bar.c_free, parity(nu - 1));
      }
      for (uint32_t m = nh > 2u ? nh - 2u : 0u; m < nh; ++m) mbar_wait_drain(&bar.acc_full[m & 1], parity(m / 2));
      for (uint32_t m = k > (uint32_t)kNA ? k - kNA : 0u; m < k; ++m)
        mbar_wait_drain(&bar.a_free[m % kNA], parity(m / kNA));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_free[m % kNX], parity(m / kNX));
      for (uint32_t m = ns > (uint32_t)kNSB ? ns - kNSB : 0u; m < ns; ++m)
        mbar_wait_drain(&bar.s_free[m % kNSB], parity(m / kNSB));
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ transform
    const int q = warp & 3, cg = (warp - 2) >> 2, il = 32 * q + lane, tt = threadIdx.x - 64;
    const uint32_t sV = smem_u32(sm + kSmV), sD = smem_u32(sm + kSmD);
    const float kLog2e = 1.4426950408889634f;
    uint32_t nu = 0, nh = 0, k = 0;
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int i = 128 * o.I + il, row_lo = 128 * o.I + 32 * q, row_hi = row_lo + 31;
      int start_i = 0;
      mbar_wait(bar.cb_full, parity(nu), status);
      tc_fence_after();
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int vb = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vdt = vacs + 1024, vseq = vacs + 2048 + 16;
        const uint32_t da = sD + vb * 3072, db = da + 1024, df = da + 2048;
        if (hh == 0 && has_seq) {  // first token of row i's sequence inside the chunk
          const int si = pipe::lds_i(vseq + 4 * i);
          start_i = i;
          while (start_i > 0 && pipe::lds_i(vseq + 4 * (start_i - 1)) == si) --start_i;
        }
        if (tt < pr.Q) {
          const float acs_j = pipe::lds_f(vacs + 4 * tt), dt_j = pipe::lds_f(vdt + 4 * tt);
          const float a = acs_j * kLog2e;
          const float f = ex2_approx((pipe::lds_f(vacs + 4 * (tt | 15)) - acs_j) * kLog2e) * dt_j;
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(da + 4 * tt), "f"(a) : "memory");
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(db + 4 * tt), "f"(__log2f(dt_j) - a) : "memory");
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(df + 4 * tt), "f"(f) : "memory");
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kTransformThreads) : "memory");
        const float ai = pipe::lds_f(da + 4 * i);
        // two 64-column slices per pass (a head has 2 or 4): both TMEM loads in
        // flight at once, one proxy fence and two arrivals; the ring slots are
        // waited for only when the values are ready to be stored
        for (int s = 0; s < 2 * (o.I + 1); s += 2, k += 2) {
          uint32_t raw[2][16];
          bool live[2];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const int j0 = 64 * (s + p) + 16 * cg;
            live[p] = j0 <= row_hi;  // warp-uniform
            if (live[p]) {
              tmem_ld16_async(pipe::tmem_quad(tmem, j0), raw[p]);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) raw[p][e] = 0u;
            }
          }
          tmem_wait_ld(raw[0], raw[1]);
          uint4 pk[2][2];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const int j0 = 64 * (s + p) + 16 * cg;
            float r[16];
            if (!live[p]) {
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = 0.f;
            } else if (row_lo >= j0 + 15) {  // whole group below the diagonal: factorised decay
              const float ei = ex2_approx(ai - pipe::lds_f(da + 4 * (j0 + 15)));
              const bool nomask = __all_sync(0xffffffffu, start_i <= j0);
              const uint64_t ei2 = pk2(ei, ei);
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 f4 = pipe::lds_f4(df + 4 * (j0 + e));
                // two columns per packed fp32 instruction
                const uint64_t v01 = mul2(pk2(__uint_as_float(raw[p][e]), __uint_as_float(raw[p][e + 1])),
                                          mul2(pk2(f4.x, f4.y), ei2));
                const uint64_t v23 = mul2(pk2(__uint_as_float(raw[p][e + 2]), __uint_as_float(raw[p][e + 3])),
                                          mul2(pk2(f4.z, f4.w), ei2));
                upk2(v01, r[e], r[e + 1]);
                upk2(v23, r[e + 2], r[e + 3]);
                if (!nomask) {
#pragma unroll
                  for (int m = 0; m < 4; ++m) r[e + m] = j0 + e + m >= start_i ? r[e + m] : 0.f;
                }
              }
            } else {  // group on the diagonal: one 2^x per element
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 b4 = pipe::lds_f4(db + 4 * (j0 + e));
                const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const int j = j0 + e + m;
                  r[e + m] = (unsigned)(j - start_i) <= (unsigned)(i - start_i)
                                 ? __uint_as_float(raw[p][e + m]) * ex2_approx(ai + bv[m])
                                 : 0.f;
                }
              }
            }
            float r0[8], r1[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              r0[m] = r[m];
              r1[m] = r[8 + m];
            }
            pk[p][0] = tc::pack8(r0);
            pk[p][1] = tc::pack8(r1);
          }
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const uint32_t kp = k + p, slot = kp % kNA;
            if (kp >= (uint32_t)kNA) mbar_wait(&bar.a_free[slot], parity(kp / kNA - 1), status);
            // this warp's K step (8 columns) of the slot, in its lane quadrant
            const uint32_t tdst = pipe::tmem_quad(tmem + kTmA + 32 * slot, 8 * cg);
            tmem_st4_async(tdst, pk[p][0].x, pk[p][0].y, pk[p][0].z, pk[p][0].w);
            tmem_st4_async(tdst + 4, pk[p][1].x, pk[p][1].y, pk[p][1].z, pk[p][1].w);
          }
          tmem_wait_st();
          tc_fence_before();
#pragma unroll
          for (int p = 0; p < 2; ++p) pipe::warp_arrive(&bar.a_full[(k + p) % kNA]);
        }
        pipe::warp_arrive(&bar.vec_free[vb]);
      }
      tc_fence_before();
      pipe::warp_arrive(bar.cb_used);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, il = 32 * q + lane;
    const uint32_t sV = smem_u32(sm + kSmV);
    uint32_t nh = 0;
    for (uint32_t nu = 0;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int i = 128 * o.I + il, t = o.c * pr.Q + i;
      const bool has_off = chunk_has_incoming(pr, o.c);
      const bf16 *xrow = u + ((size_t)o.bb * pr.L + t) * Cd;
      bf16 *yrow = y + ((size_t)o.bb * pr.L + t) * HP;
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, vb = nh & 1, ab = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vseq = vacs + 2048 + 16;
        // row i continues the state entering the chunk (the sequence before it,
        // or in a row's first chunk the first sequence, which takes the initial state)
        const bool cont = !has_seq || pipe::lds_i(vseq + 4 * i) == pipe::lds_i(o.c > 0 ? vseq - 4 : vseq);
        const float em = (has_off && cont) ? expf(pipe::lds_f(vacs + 4 * i)) : 0.f;
        pipe::warp_arrive(&bar.vec_free[vb]);
        const float Dh = __ldg(pr.D + h);
        // the x row's first 16 columns are loaded first, in flight while the
        // accumulators finish, and each next 16 one step ahead
        const bf16 *xh = xrow + h * pr.P;
        uint4 xr0 = tc::ldg16(xh), xr1 = tc::ldg16(xh + 8);
        mbar_wait(&bar.acc_full[ab], parity(nh / 2), status);
        tc_fence_after();
        const uint32_t tyd = tmem + kTmYd + 64 * ab;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 xr[2] = {xr0, xr1};
          const int cn = cc < 3 ? 16 * cc + 16 : 48;  // the last step reloads its own columns
          xr0 = tc::ldg16(xh + cn);
          xr1 = tc::ldg16(xh + cn + 8);
          float yd[16], yo[16];
          tmem_ld16(pipe::tmem_quad(tyd, 16 * cc), yd);
          if (has_off) tmem_ld16(pipe::tmem_quad(tmem + kTmYo, 16 * cc), yo);
#pragma unroll
          for (int q8 = 0; q8 < 2; ++q8) {
            float x[8], o8[8];
            tc::unpack8(xr[q8], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int col = 8 * q8 + e;
              o8[e] = yd[col] + (has_off ? em * yo[col] : 0.f) + Dh * x[e];
            }
            *reinterpret_cast<uint4 *>(yrow + h * pr.P + 16 * cc + 8 * q8) = tc::pack8(o8);
          }
        }
        tc_fence_before();
        pipe::warp_arrive(&bar.acc_free[ab]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

void launch_tc_out(const Problem &pr, const bf16 *u, const float *dtv, const float *acs, const bf16 *sin16, bf16 *y,
                   int *status, cudaStream_t s) {
  int *counter = status + kCounterOut;  // zeroed with the status word
  static bool once = (cudaFuncSetAttribute(tc_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes),
                      true);
  (void)once;
  CUtensorMap tm_u, tm_s;
  if (!encode_tmap_bf16_2d(&tm_u, u, pr.Cd, (uint64_t)pr.b * pr.L, (uint64_t)pr.Cd * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_s, sin16, pr.N, (uint64_t)pr.b * pr.nc * pr.H * pr.P, (uint64_t)pr.N * 2, 64, 64)) {
    note_host_error();
    return;
  }
  const int HB = tc_head_subset(pr);
  const int nunits = (pr.Q / 128) * pr.b * pr.nc * (pr.H / HB);
  const int grid = nunits < device_sm_count() ? nunits : device_sm_count();
  tc_out_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_u, tm_s, pr, u, dtv, acs, y, HB, nunits, counter, status);
}

}  // namespace ssd
