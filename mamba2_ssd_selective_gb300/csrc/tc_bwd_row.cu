// Backward of the chunked Mamba2 SSD, row side, on the tensor cores: for the
// rows i of one 128-token tile I of a chunk it forms, per head h,
//   dM = dy_h x_h^T                         (only the blocks j <= i)
//   W  = dM o L_h o dt,   L_h[i, j] = exp(Acs_i - Acs_j) [j <= i, same sequence]
//   vrow_i = sum_{j<i} V[i, j] dt_j = sum_{j<i} W[i, j] CB[i, j]   (V = dM o CB o L;
//            the diagonal cancels in the Acs adjoint and is left out)
//   r_i    = em_i dy_i . (C_i S_in,h^T)     (the Y_off piece of the dt adjoint)
// and accumulates over the heads of a block (in tensor memory)
//   dC_i  += sum_j W[i, j] B_j + em_i dy_i S_in,h,
// written as one fp32 partial per (token, head block).
//
// Persistent, warp-specialised (22 warps, one CTA per SM), same layout of roles
// as the output kernel: warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 2-17 transform (four per TMEM lane quadrant, 16 columns each), warps
// 18-21 epilogue.  Work unit = (row, chunk, tile I, block of HB heads of one
// group); CB = C_I B^T stays in tensor memory for the unit.
//
// Tensor memory: [0, 256) CB | [256, 320) dM (one 64-column slice) |
//                [320, 384) Y_off = C_I S_in^T | [384, 512) dC.
#include "chunk_common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tc_pipe.cuh"

namespace ssd {

namespace {

using bf16 = __nv_bfloat16;
using namespace sm100;
using pipe::parity;

constexpr int kWarps = 22, kThreads = kWarps * 32, kEpiWarp0 = 18;
constexpr int kTWarps = 16, kEWarps = 4, kTThreads = kTWarps * 32;
constexpr int kNX = 2;  // x slice ring
constexpr int kNA = 2;  // transformed operand ring (W slices, em dy)

constexpr uint32_t kSmC = 0;                    // C_I: 2 K halves x [128 x 128 B]
constexpr uint32_t kSmB = kSmC + 32768;         // B rows j < 128(I+1): 2 K halves x [256 x 128 B]
constexpr uint32_t kSmDY = kSmB + 65536;        // 2 x dy_h tile [128 x 64] bf16
constexpr uint32_t kSmX = kSmDY + 2 * 16384;    // ring of x slices [64 x 64] bf16
constexpr uint32_t kSmA = kSmX + kNX * 8192;    // ring of [128 x 64] bf16 operands
constexpr uint32_t kSmS = kSmA + kNA * 16384;   // 2 x S_in,h: 2 K halves x [64 x 128 B]
constexpr uint32_t kVecStride = 3200;           // acs[256] | dt[256] | seq[4 + 256]
constexpr uint32_t kSmV = kSmS + 2 * 16384;     // 2 vector buffers
constexpr uint32_t kSmD = kSmV + 2 * kVecStride;  // 2 x {a[256], b[256], f[256]}
constexpr uint32_t kSmVR = kSmD + 2 * 3072;     // 2 x vrow partials [4][128] f32
constexpr uint32_t kSmBar = kSmVR + 2 * 2048;
constexpr int kNumBars = 22 + 2 * kNX + 2 * kNA + 4 + 1;
constexpr uint32_t kSmEnd = kSmBar + kNumBars * 8 + 16;
constexpr int kSmemBytes = (int)kSmEnd + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmDM = 256, kTmYo = 320, kTmDC = 384;

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
  uint64_t *unit_full, *unit_free, *cb_full, *cb_used, *dm_full, *dm_free, *yo_full, *yo_free, *dc_full, *dc_free;
  uint64_t *vec_full, *vec_free, *dy_full, *dy_free, *s_full, *s_free;  // [2]
  uint64_t *x_full, *x_free;                          // [kNX]
  uint64_t *a_full, *a_free;                          // [kNA]
  uint64_t *drain;                                    // the MMA issuer's final commit
  pipe::UnitRing units;
  __device__ Bars(uint64_t *b, int *slot) {
    unit_full = b;
    unit_free = b + 1;
    cb_full = b + 2;
    cb_used = b + 3;
    dm_full = b + 4;
    dm_free = b + 5;
    yo_full = b + 6;
    yo_free = b + 7;
    dc_full = b + 8;
    dc_free = b + 9;
    vec_full = b + 10;
    vec_free = b + 12;
    dy_full = b + 14;
    dy_free = b + 16;
    s_full = b + 18;
    s_free = b + 20;
    x_full = b + 22;
    x_free = x_full + kNX;
    a_full = x_free + kNX;
    a_free = a_full + kNA;
    units.full = a_free + kNA;
    units.free = units.full + 2;
    drain = units.free + 2;
    units.slot = slot;
  }
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_row_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dy,
                      const __grid_constant__ CUtensorMap tm_s, Problem pr, const bf16 *__restrict__ dy,
                      const float *__restrict__ dtv, const float *__restrict__ acs, float *__restrict__ dcp,
                      float *__restrict__ tok, int HB, int nunits, int *counter, int *status_word) {
  extern __shared__ uint8_t smem_raw[];
  const WaitCtl status{status_word, pr.wait_ns};
  uint8_t *sm = tc::aligned_smem(smem_raw);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + kSmBar + kNumBars * 8);
  Bars bar(reinterpret_cast<uint64_t *>(sm + kSmBar), reinterpret_cast<int *>(tslot + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NTI = pr.Q / 128, nhb = pr.H / HB, HP = pr.H * pr.P;
  const bool has_seq = pr.seq_idx != nullptr;
  const size_t BHL = (size_t)pr.b * pr.H * pr.L;

  if (threadIdx.x == 0) {
    uint64_t *ones[] = {bar.unit_full, bar.unit_free, bar.cb_full, bar.dm_full,  bar.yo_full, bar.dc_full,
                        bar.s_full,    bar.s_full + 1, bar.s_free, bar.s_free + 1, bar.drain};
    for (uint64_t *b : ones) mbar_init(b, 1);
    mbar_init(bar.cb_used, kTWarps);
    mbar_init(bar.dm_free, kTWarps);
    mbar_init(bar.yo_free, kEWarps);
    mbar_init(bar.dc_free, kEWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.vec_full[i], 1);
      mbar_init(&bar.vec_free[i], kTWarps + kEWarps);
      mbar_init(&bar.dy_full[i], 1);
      mbar_init(&bar.dy_free[i], 1 + kTWarps + kEWarps);
    }
    for (int i = 0; i < kNX; ++i) {
      mbar_init(&bar.x_full[i], 1);
      mbar_init(&bar.x_free[i], 1);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&bar.a_full[i], kTWarps);
      mbar_init(&bar.a_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.units.full[i], 1);
      mbar_init(&bar.units.free[i], 1 + kTWarps + kEWarps);
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
      prefetch_tmap(&tm_dy);
      prefetch_tmap(&tm_s);
      // counts of armed loads per barrier (nua: unit operand sets); once a
      // wait has failed (ok = false) no further load is issued, stop is
      // published, and the loads in flight are drained before the CTA ends
      uint32_t nu = 0, nua = 0, nh = 0, ndy = 0, k = 0, ns = 0;
      bool ok = true;
      int next = atomicAdd(counter, 1);
      for (;; ++nu) {
        const int ui = pipe::publish_unit(bar.units, nu, ok ? next : nunits, nunits);
        if (ui >= nunits) break;
        next = atomicAdd(counter, 1);
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int g = o.h0 / pr.hpg, t0 = o.c * pr.Q, row0 = o.bb * pr.L + t0, NB = 128 * (o.I + 1);
        const int offB = HP + g * pr.N, offC = HP + pr.G * pr.N + g * pr.N;
        if (nu > 0) ok = mbar_wait(bar.unit_free, parity(nu - 1), status);
        if (!ok) continue;
        mbar_expect_tx(bar.unit_full, 32768 + 2 * NB * 128);
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
          if (ndy >= 2 && !mbar_wait(&bar.dy_free[vb], parity(ndy / 2 - 1), status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bar.dy_full[vb], 16384);
          for (int r = 0; r < 2; ++r)
            tma_load_2d(sm + kSmDY + vb * 16384 + r * 8192, &tm_dy, &bar.dy_full[vb], h * pr.P,
                        row0 + 128 * o.I + 64 * r);
          ++ndy;
          if (chunk_has_incoming(pr, o.c)) {  // S_in first: a whole head of slack before its use
            const int sb = ns & 1;
            if (ns >= 2 && !mbar_wait(&bar.s_free[sb], parity(ns / 2 - 1), status)) {
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
      for (uint32_t m = ndy > 2u ? ndy - 2u : 0u; m < ndy; ++m) mbar_wait_drain(&bar.dy_full[m & 1], parity(m / 2));
      for (uint32_t m = ns > 2u ? ns - 2u : 0u; m < ns; ++m) mbar_wait_drain(&bar.s_full[m & 1], parity(m / 2));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_full[m % kNX], parity(m / kNX));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // operand descriptors, built once; ring slots and K steps are additions
      const uint64_t dC = desc_sw128(smem_u32(sm + kSmC), 16, 1024), dB = desc_sw128(smem_u32(sm + kSmB), 16, 1024),
                     dBmn = desc_sw128(smem_u32(sm + kSmB), 32768, 1024),
                     dDY = desc_sw128(smem_u32(sm + kSmDY), 16, 1024), dX = desc_sw128(smem_u32(sm + kSmX), 16, 1024),
                     dA = desc_sw128(smem_u32(sm + kSmA), 16, 1024), dS = desc_sw128(smem_u32(sm + kSmS), 16, 1024),
                     dSmn = desc_sw128(smem_u32(sm + kSmS), 8192, 1024);
      constexpr uint32_t id_dm = idesc_bf16(128, 64, false, false);   // dy_I x_s^T
      constexpr uint32_t id_yo = idesc_bf16(128, 64, false, false);   // C_I S^T
      constexpr uint32_t id_dc = idesc_bf16(128, 128, false, true);   // W B_s, (em dy) S
      uint32_t nu = 0, nh = 0, k = 0, na = 0, ns = 0;
      for (;; ++nu) {
        const int ui = pipe::next_unit(bar.units, nu, nunits, false);
        if (ui >= nunits) break;
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int NB = 128 * (o.I + 1), nsl = 2 * (o.I + 1);
        mbar_wait(bar.unit_full, parity(nu), status);
        if (nu > 0) mbar_wait(bar.cb_used, parity(nu - 1), status);
        tc_fence_after();
        const uint32_t id_cb = idesc_bf16(128, NB, false, false);
        pipe::umma_k<4>(tmem, dC, dB, pipe::kStepK, pipe::kStepK, id_cb, false);
        pipe::umma_k<4>(tmem, dC + 16384 / 16, dB + 32768 / 16, pipe::kStepK, pipe::kStepK, id_cb, true);
        umma_commit(bar.cb_full);
        bool first_dc = true;
        // dM slice m (of the head numbered hn) into the single dM slot (after the
        // transform has read the previous one)
        auto issue_dm = [&](uint32_t m, uint32_t hn) {
          const int slot = m % kNX;
          const uint64_t ddy = dDY + (hn & 1) * (16384 / 16);
          mbar_wait(&bar.x_full[slot], parity(m / kNX), status);
          if (m > 0) mbar_wait(bar.dm_free, parity(m - 1), status);
          tc_fence_after();
          pipe::umma_k<4>(tmem + kTmDM, ddy, dX + slot * (8192 / 16), pipe::kStepK, pipe::kStepK, id_dm, false);
          umma_commit(&bar.x_free[slot]);
          umma_commit(bar.dm_full);
        };
        mbar_wait(&bar.dy_full[nh & 1], parity(nh / 2), status);
        issue_dm(k, nh);
        for (int hh = 0; hh < HB; ++hh, ++nh) {
          const int vb = nh & 1;
          for (int s = 0; s < nsl; ++s) {
            if (s + 1 < nsl) {
              issue_dm(k + s + 1, nh);
            } else if (hh + 1 < HB) {  // the next head's first slice, ahead of this head's closing products
              mbar_wait(&bar.dy_full[(nh + 1) & 1], parity((nh + 1) / 2), status);
              issue_dm(k + s + 1, nh + 1);
            }
            const int as = na % kNA;
            mbar_wait(&bar.a_full[as], parity(na / kNA), status);
            if (first_dc && nu > 0) mbar_wait(bar.dc_free, parity(nu - 1), status);
            tc_fence_after();
            pipe::umma_k<4>(tmem + kTmDC, dA + as * (16384 / 16), dBmn + s * (8192 / 16), pipe::kStepK, pipe::kStepMN,
                            id_dc, !first_dc);
            first_dc = false;
            umma_commit(&bar.a_free[as]);
            ++na;
          }
          k += nsl;
          if (chunk_has_incoming(pr, o.c)) {
            const int sb = ns & 1;
            const uint64_t dSb = dS + sb * (16384 / 16);
            mbar_wait(&bar.s_full[sb], parity(ns / 2), status);
            if (ns > 0) mbar_wait(bar.yo_free, parity(ns - 1), status);
            tc_fence_after();
            pipe::umma_k<4>(tmem + kTmYo, dC, dSb, pipe::kStepK, pipe::kStepK, id_yo, false);
            pipe::umma_k<4>(tmem + kTmYo, dC + 16384 / 16, dSb + 8192 / 16, pipe::kStepK, pipe::kStepK, id_yo, true);
            umma_commit(bar.yo_full);
            const int as = na % kNA;
            mbar_wait(&bar.a_full[as], parity(na / kNA), status);
            tc_fence_after();
            pipe::umma_k<4>(tmem + kTmDC, dA + as * (16384 / 16), dSmn + sb * (16384 / 16), pipe::kStepK, pipe::kStepMN,
                            id_dc, true);
            umma_commit(&bar.a_free[as]);
            ++na;
            umma_commit(&bar.s_free[sb]);
            ++ns;
          }
          umma_commit(&bar.dy_free[vb]);
        }
        umma_commit(bar.dc_full);
        umma_commit(bar.unit_free);
      }
      // drain: every MMA issued here has completed and every commit arrival
      // has landed before the CTA releases its shared and tensor memory
      umma_commit(bar.drain);
      mbar_wait_drain(bar.drain, 0);
      if (nu > 0) {
        mbar_wait_drain(bar.cb_full, parity(nu - 1));
        mbar_wait_drain(bar.dc_full, parity(nu - 1));
        mbar_wait_drain(bar.unit_free, parity(nu - 1));
      }
      if (k > 0) mbar_wait_drain(bar.dm_full, parity(k - 1));
      if (ns > 0) mbar_wait_drain(bar.yo_full, parity(ns - 1));
      for (uint32_t m = k > (uint32_t)kNX ? k - kNX : 0u; m < k; ++m)
        mbar_wait_drain(&bar.x_free[m % kNX], parity(m / kNX));
      for (uint32_t m = na > (uint32_t)kNA ? na - kNA : 0u; m < na; ++m)
        mbar_wait_drain(&bar.a_free[m % kNA], parity(m / kNA));
      for (uint32_t m = ns > 2u ? ns - 2u : 0u; m < ns; ++m) mbar_wait_drain(&bar.s_free[m & 1], parity(m / 2));
      for (uint32_t m = nh > 2u ? nh - 2u : 0u; m < nh; ++m) mbar_wait_drain(&bar.dy_free[m & 1], parity(m / 2));
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ transform
    const int q = warp & 3, cg = (warp - 2) >> 2, il = 32 * q + lane, tt = threadIdx.x - 64;
    const uint32_t sA = smem_u32(sm + kSmA), sV = smem_u32(sm + kSmV), sD = smem_u32(sm + kSmD),
                   sVR = smem_u32(sm + kSmVR), sDY = smem_u32(sm + kSmDY);
    const float kLog2e = 1.4426950408889634f;
    uint32_t nu = 0, nh = 0, k = 0, na = 0;
    size_t prev_tok = 0;  // tok offset of the previous head's row il (vrow flush)
    int prev_vb = -1;
    auto flush_vrow = [&]() {  // sum of the four column-group partials, fixed order
      if (prev_vb >= 0 && cg == 0) {
        const uint32_t base = sVR + prev_vb * 2048 + 4 * il;
        tok[prev_tok] = (pipe::lds_f(base) + pipe::lds_f(base + 512)) + (pipe::lds_f(base + 1024) + pipe::lds_f(base + 1536));
      }
    };
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int i = 128 * o.I + il, row_lo = 128 * o.I + 32 * q, row_hi = row_lo + 31, nsl = 2 * (o.I + 1);
      int start_i = 0;
      mbar_wait(bar.cb_full, parity(nu), status);
      tc_fence_after();
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, vb = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vdt = vacs + 1024, vseq = vacs + 2048 + 16;
        const uint32_t da = sD + vb * 3072, db = da + 1024, df = da + 2048;
        if (hh == 0 && has_seq) {  // first token of row i's sequence inside the chunk
          const int si = pipe::lds_i(vseq + 4 * i);
          start_i = i;
          while (start_i > 0 && pipe::lds_i(vseq + 4 * (start_i - 1)) == si) --start_i;
        }
        const bool inc = chunk_has_incoming(pr, o.c);
        const bool cont = !has_seq || pipe::lds_i(vseq + 4 * i) == pipe::lds_i(o.c > 0 ? vseq - 4 : vseq);
        const float em = (inc && cont) ? expf(pipe::lds_f(vacs + 4 * i)) : 0.f;
        if (tt < pr.Q) {
          const float acs_j = pipe::lds_f(vacs + 4 * tt), dt_j = pipe::lds_f(vdt + 4 * tt);
          const float a = acs_j * kLog2e;
          pipe::sts_f(da + 4 * tt, a);
          pipe::sts_f(db + 4 * tt, __log2f(dt_j) - a);
          pipe::sts_f(df + 4 * tt, ex2_approx((pipe::lds_f(vacs + 4 * (tt | 15)) - acs_j) * kLog2e) * dt_j);
        }
        pipe::transform_sync<kTThreads>();
        flush_vrow();
        const float ai = pipe::lds_f(da + 4 * i);
        float vrow = 0.f;
        for (int s = 0; s < nsl; ++s, ++k) {
          const int j0 = 64 * s + 16 * cg;
          float w[16];
          mbar_wait(bar.dm_full, parity(k), status);
          tc_fence_after();
          if (j0 > row_hi) {
            pipe::warp_arrive(bar.dm_free);
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = 0.f;
          } else {
            float dm[16], cbv[16];
            tmem_ld16(pipe::tmem_quad(tmem + kTmDM, 16 * cg), dm);
            tmem_ld16(pipe::tmem_quad(tmem, j0), cbv);
            tc_fence_before();
            pipe::warp_arrive(bar.dm_free);
            if (row_lo >= j0 + 15) {  // below the diagonal: factorised decay
              const float ei = ex2_approx(ai - pipe::lds_f(da + 4 * (j0 + 15)));
              const bool nomask = __all_sync(0xffffffffu, start_i <= j0);
              const uint64_t ei2 = pk2(ei, ei);
              uint64_t vr2 = pk2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 f4 = pipe::lds_f4(df + 4 * (j0 + e));
                // two columns per packed fp32 instruction
                upk2(mul2(pk2(dm[e], dm[e + 1]), mul2(pk2(f4.x, f4.y), ei2)), w[e], w[e + 1]);
                upk2(mul2(pk2(dm[e + 2], dm[e + 3]), mul2(pk2(f4.z, f4.w), ei2)), w[e + 2], w[e + 3]);
                if (!nomask) {
#pragma unroll
                  for (int m = 0; m < 4; ++m) w[e + m] = j0 + e + m >= start_i ? w[e + m] : 0.f;
                }
                vr2 = fma2(pk2(w[e], w[e + 1]), pk2(cbv[e], cbv[e + 1]), vr2);
                vr2 = fma2(pk2(w[e + 2], w[e + 3]), pk2(cbv[e + 2], cbv[e + 3]), vr2);
              }
              float vr_lo, vr_hi;
              upk2(vr2, vr_lo, vr_hi);
              vrow += vr_lo + vr_hi;
            } else {  // on the diagonal
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 b4 = pipe::lds_f4(db + 4 * (j0 + e));
                const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const int j = j0 + e + m;
                  w[e + m] = (unsigned)(j - start_i) <= (unsigned)(i - start_i) ? dm[e + m] * ex2_approx(ai + bv[m]) : 0.f;
                }
              }
              // the row sum leaves out j = i: that term cancels exactly against the
              // column sum's in the Acs adjoint (the column kernel keeps it apart)
#pragma unroll
              for (int e = 0; e < 16; ++e) vrow = fmaf(j0 + e == i ? 0.f : w[e], cbv[e], vrow);
            }
          }
          const int as = na % kNA;
          if (na >= (uint32_t)kNA) mbar_wait(&bar.a_free[as], parity(na / kNA - 1), status);
          float w0[8], w1[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            w0[e] = w[e];
            w1[e] = w[8 + e];
          }
          const uint32_t A = sA + as * 16384;
          pipe::sts_u4(A + sw128_offset(il, 16 * cg), tc::pack8(w0));
          pipe::sts_u4(A + sw128_offset(il, 16 * cg + 8), tc::pack8(w1));
          fence_async_smem();
          pipe::warp_arrive(&bar.a_full[as]);
          ++na;
        }
        if (inc) {  // em_i dy_i, the A operand of the S_in term of dC
          mbar_wait(&bar.dy_full[vb], parity(nh / 2), status);
          const int as = na % kNA;
          if (na >= (uint32_t)kNA) mbar_wait(&bar.a_free[as], parity(na / kNA - 1), status);
          const uint32_t A = sA + as * 16384, T = sDY + vb * 16384;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            float x[8];
            tc::unpack8(pipe::lds_sw128(T, il, 2 * cg + t), x);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= em;
            pipe::sts_u4(A + sw128_offset(il, 16 * cg + 8 * t), tc::pack8(x));
          }
          fence_async_smem();
          pipe::warp_arrive(&bar.a_full[as]);
          ++na;
        }
        pipe::sts_f(sVR + vb * 2048 + cg * 512 + 4 * il, vrow);
        prev_tok = ((size_t)o.bb * pr.H + h) * pr.L + (size_t)o.c * pr.Q + i;
        prev_vb = vb;
        pipe::warp_arrive(&bar.dy_free[vb]);
        pipe::warp_arrive(&bar.vec_free[vb]);
      }
      tc_fence_before();
      pipe::warp_arrive(bar.cb_used);
    }
    pipe::transform_sync<kTThreads>();
    flush_vrow();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, il = 32 * q + lane;
    const uint32_t sV = smem_u32(sm + kSmV), sDY = smem_u32(sm + kSmDY);
    uint32_t nu = 0, nh = 0, ny = 0;
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int i = 128 * o.I + il, t = o.c * pr.Q + i;
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, vb = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vseq = vacs + 2048 + 16;
        const bool inc = chunk_has_incoming(pr, o.c);
        const bool cont = !has_seq || pipe::lds_i(vseq + 4 * i) == pipe::lds_i(o.c > 0 ? vseq - 4 : vseq);
        const float em = (inc && cont) ? expf(pipe::lds_f(vacs + 4 * i)) : 0.f;
        pipe::warp_arrive(&bar.vec_free[vb]);
        float r = 0.f;
        mbar_wait(&bar.dy_full[vb], parity(nh / 2), status);  // dy row i from the head's tile
        if (inc) {
          const uint32_t T = sDY + vb * 16384;
          mbar_wait(bar.yo_full, parity(ny), status);
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float yo[16];
            tmem_ld16(pipe::tmem_quad(tmem + kTmYo, 16 * cc), yo);
#pragma unroll
            for (int t8 = 0; t8 < 2; ++t8) {
              float d8[8];
              tc::unpack8(pipe::lds_sw128(T, il, 2 * cc + t8), d8);
#pragma unroll
              for (int e = 0; e < 8; ++e) r = fmaf(d8[e], yo[8 * t8 + e], r);
            }
          }
          tc_fence_before();
          pipe::warp_arrive(bar.yo_free);
          ++ny;
          r *= em;
        }
        pipe::warp_arrive(&bar.dy_free[vb]);
        tok[3 * BHL + ((size_t)o.bb * pr.H + h) * pr.L + t] = r;
      }
      mbar_wait(bar.dc_full, parity(nu), status);
      tc_fence_after();
      float *out = dcp + (((size_t)o.bb * pr.L + t) * nhb + o.h0 / HB) * pr.N;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        float a[16];
        tmem_ld16(pipe::tmem_quad(tmem + kTmDC, 16 * cc), a);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          reinterpret_cast<float4 *>(out + 16 * cc)[e] = make_float4(a[4 * e], a[4 * e + 1], a[4 * e + 2], a[4 * e + 3]);
      }
      tc_fence_before();
      pipe::warp_arrive(bar.dc_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

void launch_tc_bwd_row(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs,
                       const bf16 *sin16, float *dcp, float *tok, int *status, cudaStream_t s) {
  static bool once = (cudaFuncSetAttribute(tc_bwd_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes),
                      true);
  (void)once;
  CUtensorMap tm_u, tm_dy, tm_s;
  const uint64_t HP = (uint64_t)pr.H * pr.P;
  if (!encode_tmap_bf16_2d(&tm_u, u, pr.Cd, (uint64_t)pr.b * pr.L, (uint64_t)pr.Cd * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_dy, dy, HP, (uint64_t)pr.b * pr.L, HP * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_s, sin16, pr.N, (uint64_t)pr.b * pr.nc * pr.H * pr.P, (uint64_t)pr.N * 2, 64, 64)) {
    note_host_error();
    return;
  }
  const int HB = tc_head_subset(pr);
  const int nunits = (pr.Q / 128) * pr.b * pr.nc * (pr.H / HB);
  const int grid = nunits < device_sm_count() ? nunits : device_sm_count();
  int *counter = status + kCounterRow;  // zeroed with the status word
  tc_bwd_row_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_u, tm_dy, tm_s, pr, dy, dtv, acs, dcp, tok, HB, nunits, counter, status);
}

}  // namespace ssd
