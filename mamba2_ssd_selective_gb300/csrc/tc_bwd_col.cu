// Backward of the chunked Mamba2 SSD, column side, on the tensor cores: for the
// rows j of one 128-token tile J of a chunk (columns i >= 128 J), per head h,
//   dM^T = x_h dy_h^T,   CB^T = B_J C^T            (64-column slices, recomputed)
//   M^T  = CB^T o L^T o dt_j,   W^T = dM^T o L^T o dt_j,  L^T[j, i] = exp(Acs_i - Acs_j)
//   T_j  = sum_i M^T[j, i] dy_i,   U_j = dS_end,h B_j,     (tensor memory)
//   du_x[j] = T_j + wdt_j U_j + D_h dy_j,   q_j = x_j . U_j,   dy_j . x_j (for dD),
//   vcol_j = sum_{i>j} V[i, j] = sum_{i>j} dM^T CB^T L^T,  vdiag_j = V[j, j]
//            (kept apart: the diagonal cancels in the Acs adjoint, not in dt's)
// and accumulates over the heads of a block
//   dB_j += sum_i W^T[j, i] C_i + wdt_j dS_end,h^T x_j,
// written as one fp32 partial per (token, head block).
//
// Roles as in the row kernel (22 warps, one CTA per SM).  Tensor memory:
//   [0, 256) two slice slots {dM^T 64 | CB^T 64} | [256, 320) T | [320, 384) U |
//   [384, 512) dB.
// The transform warps write M^T and W^T, rounded to bf16, back into the slot's
// CB^T columns they have just read (each warp its own 16 columns: M^T in the
// first 8, W^T in the last 8, two values per column); the T and dB products
// take their A operand from there, so the slice's operands never pass through
// shared memory.  A slot's dM^T columns are refilled as soon as the transform
// has read them; its CB^T columns once the T and dB products have read M^T and
// W^T (slot_free).
// The epilogue takes the tile's dy rows from a 16 KB tile the producer loads
// per head, and writes du_x back through the same buffer: each epilogue warp
// stages its 32 rows x 32 columns of fp32 there and stores them with one TMA
// store, so the rows leave as whole lines rather than as one line per thread.
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
constexpr int kNY = 3;  // dy slice ring
constexpr int kNA = 1;  // transformed operand in shared memory (wdt x, once per head)

constexpr uint32_t kSmBJ = 0;                   // B_J: 2 K halves x [128 x 128 B]
constexpr uint32_t kSmCR = kSmBJ + 32768;       // C rows i >= 128 J: 2 K halves x [256 x 128 B]
constexpr uint32_t kSmXT = kSmCR + 65536;       // 2 x x_h tile [128 x 64] bf16
constexpr uint32_t kSmDY = kSmXT + 2 * 16384;   // ring of dy slices [64 x 64] bf16
constexpr uint32_t kSmA = kSmDY + kNY * 8192;   // ring of [128 x 64] bf16 operands
constexpr uint32_t kSmDS = kSmA + kNA * 16384;  // dS_end,h: 2 K halves x [64 x 128 B]
constexpr uint32_t kSmE = kSmDS + 16384;        // epilogue: dy rows [128 x 64] bf16, then du_x staging
constexpr uint32_t kVecStride = 3200;           // acs[256] | dt[256] | seq[4 + 256]
constexpr uint32_t kSmV = kSmE + 16384;
constexpr uint32_t kSmD = kSmV + 2 * kVecStride;  // 2 x {a[256], g[256]}
constexpr uint32_t kSmVC = kSmD + 2 * 2048;     // 2 x vcol partials [4][128] f32
constexpr uint32_t kSmBar = kSmVC + 2 * 2048;
constexpr int kNumBars = 20 + 2 * kNY + 2 * kNA + 4 + 1 + 2 + 2;
constexpr uint32_t kSmEnd = kSmBar + kNumBars * 8 + 16;
constexpr int kSmemBytes = (int)kSmEnd + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmT = 256, kTmU = 320, kTmDB = 384;

struct Unit {
  int bb, c, J, h0;
};

// NP transformed 16-column groups of TMEM lane row `row` into the next NP
// slots of the shared-memory operand ring (bf16, 128-byte swizzle): each slot
// waited for only when its values are ready, one proxy fence, then one arrival
// per slot.
template <int NP>
__device__ __forceinline__ void put_operands(const float (&v)[NP][16], uint32_t &na, uint32_t sA, int row, int cg,
                                             uint64_t *a_full, uint64_t *a_free, const WaitCtl &status) {
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const uint32_t n = na + p, as = n % kNA;
    float v0[8], v1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v0[e] = v[p][e];
      v1[e] = v[p][8 + e];
    }
    const uint4 lo = tc::pack8(v0), hi = tc::pack8(v1);
    if (n >= (uint32_t)kNA) mbar_wait(&a_free[as], pipe::parity(n / kNA - 1), status);
    const uint32_t A = sA + as * 16384;
    pipe::sts_u4(A + sw128_offset(row, 16 * cg), lo);
    pipe::sts_u4(A + sw128_offset(row, 16 * cg + 8), hi);
  }
  fence_async_smem();
#pragma unroll
  for (int p = 0; p < NP; ++p) pipe::warp_arrive(&a_full[(na + p) % kNA]);
  na += NP;
}

// Unit u of the launch, claimed dynamically in this order: the tiles with more
// work first (every CTA then ends on light ones), and within a tile class the
// head blocks of one (row, chunk) adjacent, sharing C and B in L2.
__device__ __forceinline__ Unit unit_of(const Problem &pr, int NTI, int nhb, int HB, int u) {
  const int per = pr.b * pr.nc * nhb;
  const int cls = u / per, r = u % per;
  (void)NTI;
  Unit o;
  o.J = cls;
  const int hb = r % nhb, bc = r / nhb;
  o.c = bc % pr.nc;
  o.bb = bc / pr.nc;
  o.h0 = hb * HB;
  return o;
}

struct Bars {
  uint64_t *unit_full, *unit_free, *tu_full, *tu_free, *ds_full, *ds_free, *db_full, *db_free;
  uint64_t *ring_full, *slot_free, *vec_full, *vec_free, *xt_full, *xt_free;  // [2]
  uint64_t *op_full;                                                          // [2]
  uint64_t *ey_full, *ey_free;                                                // the epilogue's dy tile
  uint64_t *dy_full, *dy_free;                                                // [kNY]
  uint64_t *a_full, *a_free;                                                  // [kNA]
  uint64_t *drain;                                                            // the MMA issuer's final commit
  pipe::UnitRing units;
  __device__ Bars(uint64_t *b, int *slot) {
    unit_full = b;
    unit_free = b + 1;
    tu_full = b + 2;
    tu_free = b + 3;
    ds_full = b + 4;
    ds_free = b + 5;
    db_full = b + 6;
    db_free = b + 7;
    ring_full = b + 8;
    slot_free = b + 10;
    vec_full = b + 12;
    vec_free = b + 14;
    xt_full = b + 16;
    xt_free = b + 18;
    dy_full = b + 20;
    dy_free = dy_full + kNY;
    a_full = dy_free + kNY;
    a_free = a_full + kNA;
    units.full = a_free + kNA;
    units.free = units.full + 2;
    drain = units.free + 2;
    op_full = drain + 1;
    ey_full = op_full + 2;
    ey_free = ey_full + 1;
    units.slot = slot;
  }
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_col_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dy,
                      const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_du,
                      const __grid_constant__ CUtensorMap tm_db, Problem pr, const float *__restrict__ dtv,
                      const float *__restrict__ acs, float *__restrict__ tok, int HB, int nunits, int *counter,
                      int *status_word) {
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
    uint64_t *ones[] = {bar.unit_full, bar.unit_free, bar.tu_full, bar.ds_full,
                        bar.ds_free,   bar.db_full,   bar.drain,   bar.ey_full};
    for (uint64_t *b : ones) mbar_init(b, 1);
    mbar_init(bar.tu_free, kEWarps);
    mbar_init(bar.db_free, kEWarps);
    mbar_init(bar.ey_free, kEWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.ring_full[i], 1);
      mbar_init(&bar.slot_free[i], 1);
      mbar_init(&bar.op_full[i], kTWarps);
      mbar_init(&bar.vec_full[i], 1);
      mbar_init(&bar.vec_free[i], kTWarps + kEWarps);
      mbar_init(&bar.xt_full[i], 1);
      mbar_init(&bar.xt_free[i], 1 + kTWarps + kEWarps);
    }
    for (int i = 0; i < kNY; ++i) {
      mbar_init(&bar.dy_full[i], 1);
      mbar_init(&bar.dy_free[i], 1);
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
      prefetch_tmap(&tm_ds);
      // counts of armed loads per barrier (nua: unit operand sets); once a
      // wait has failed (ok = false) no further load is issued, stop is
      // published, and the loads in flight are drained before the CTA ends
      uint32_t nu = 0, nua = 0, nh = 0, nxt = 0, m = 0, nd = 0, ne = 0;
      bool ok = true;
      int next = atomicAdd(counter, 1);
      for (;; ++nu) {
        const int ui = pipe::publish_unit(bar.units, nu, ok ? next : nunits, nunits);
        if (ui >= nunits) break;
        next = atomicAdd(counter, 1);
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int g = o.h0 / pr.hpg, t0 = o.c * pr.Q, row0 = o.bb * pr.L + t0, nsl = (pr.Q - 128 * o.J) / 64;
        const int offB = HP + g * pr.N, offC = HP + pr.G * pr.N + g * pr.N, rJ = row0 + 128 * o.J;
        if (nu > 0) ok = mbar_wait(bar.unit_free, parity(nu - 1), status);
        if (!ok) continue;
        mbar_expect_tx(bar.unit_full, 32768 + 2 * nsl * 8192);
        for (int kh = 0; kh < 2; ++kh) {
          for (int r = 0; r < 2; ++r)
            tma_load_2d(sm + kSmBJ + kh * 16384 + r * 8192, &tm_u, bar.unit_full, offB + 64 * kh, rJ + 64 * r);
          for (int r = 0; r < nsl; ++r)
            tma_load_2d(sm + kSmCR + kh * 32768 + r * 8192, &tm_u, bar.unit_full, offC + 64 * kh, rJ + 64 * r);
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
          const uint32_t seq_bytes = !has_seq ? 0u : (uint32_t)(pr.Q * 4);
          mbar_expect_tx(&bar.vec_full[vb], 2 * pr.Q * 4 + seq_bytes);
          pipe::bulk_load(vec, acs + bh, pr.Q * 4, &bar.vec_full[vb]);
          pipe::bulk_load(vec + 1024, dtv + bh, pr.Q * 4, &bar.vec_full[vb]);
          if (has_seq)
            pipe::bulk_load(vec + 2048 + 16, pr.seq_idx + (size_t)o.bb * pr.L + t0, seq_bytes, &bar.vec_full[vb]);
          ++nh;
          if (nxt >= 2 && !mbar_wait(&bar.xt_free[vb], parity(nxt / 2 - 1), status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bar.xt_full[vb], 16384);
          for (int r = 0; r < 2; ++r)
            tma_load_2d(sm + kSmXT + vb * 16384 + r * 8192, &tm_u, &bar.xt_full[vb], h * pr.P, rJ + 64 * r);
          ++nxt;
          for (int s = 0; s < nsl; ++s) {
            const int ys = m % kNY;
            if (m >= kNY && !mbar_wait(&bar.dy_free[ys], parity(m / kNY - 1), status)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&bar.dy_full[ys], 8192);
            tma_load_2d(sm + kSmDY + ys * 8192, &tm_dy, &bar.dy_full[ys], h * pr.P, rJ + 64 * s);
            ++m;
          }
          if (!ok) break;
          if (nd >= 1 && !mbar_wait(bar.ds_free, parity(nd - 1), status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar.ds_full, 16384);
          const int srow = (int)((((size_t)o.bb * pr.nc + o.c) * pr.H + h) * pr.P);
          tma_load_2d(sm + kSmDS, &tm_ds, bar.ds_full, 0, srow);
          tma_load_2d(sm + kSmDS + 8192, &tm_ds, bar.ds_full, 64, srow);
          ++nd;
          // the epilogue's dy rows, once it has stored the previous head's du_x
          if (ne >= 1 && !mbar_wait(bar.ey_free, parity(ne - 1), status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar.ey_full, 16384);
          for (int r = 0; r < 2; ++r) tma_load_2d(sm + kSmE + r * 8192, &tm_dy, bar.ey_full, h * pr.P, rJ + 64 * r);
          ++ne;
        }
      }
      // every load issued has landed before the CTA releases its shared memory
      if (nua > 0) mbar_wait_drain(bar.unit_full, parity(nua - 1));
      for (uint32_t n = nh > 2u ? nh - 2u : 0u; n < nh; ++n) mbar_wait_drain(&bar.vec_full[n & 1], parity(n / 2));
      for (uint32_t n = nxt > 2u ? nxt - 2u : 0u; n < nxt; ++n) mbar_wait_drain(&bar.xt_full[n & 1], parity(n / 2));
      for (uint32_t n = m > (uint32_t)kNY ? m - kNY : 0u; n < m; ++n)
        mbar_wait_drain(&bar.dy_full[n % kNY], parity(n / kNY));
      if (nd > 0) mbar_wait_drain(bar.ds_full, parity(nd - 1));
      if (ne > 0) mbar_wait_drain(bar.ey_full, parity(ne - 1));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // operand descriptors, built once; ring slots and K steps are additions
      const uint64_t dBJ = desc_sw128(smem_u32(sm + kSmBJ), 16, 1024), dCR = desc_sw128(smem_u32(sm + kSmCR), 16, 1024),
                     dCRmn = desc_sw128(smem_u32(sm + kSmCR), 32768, 1024),
                     dXT = desc_sw128(smem_u32(sm + kSmXT), 16, 1024), dDY = desc_sw128(smem_u32(sm + kSmDY), 16, 1024),
                     dDYmn = desc_sw128(smem_u32(sm + kSmDY), 8192, 1024), dA = desc_sw128(smem_u32(sm + kSmA), 16, 1024),
                     dDS = desc_sw128(smem_u32(sm + kSmDS), 16, 1024), dDSmn = desc_sw128(smem_u32(sm + kSmDS), 8192, 1024);
      constexpr uint32_t id_64 = idesc_bf16(128, 64, false, false);    // x dy^T, B_J C^T, B_J dS^T
      constexpr uint32_t id_t = idesc_bf16(128, 64, false, true);      // M^T dy
      constexpr uint32_t id_db = idesc_bf16(128, 128, false, true);    // W^T C, (wdt x) dS
      uint32_t nu = 0, nh = 0, m = 0, na = 0, nd = 0;
      for (;; ++nu) {
        const int ui = pipe::next_unit(bar.units, nu, nunits, false);
        if (ui >= nunits) break;
        const Unit o = unit_of(pr, NTI, nhb, HB, ui);
        const int nsl = (pr.Q - 128 * o.J) / 64;
        mbar_wait(bar.unit_full, parity(nu), status);
        bool first_db = true;
        for (int hh = 0; hh < HB; ++hh, ++nh) {
          const int vb = nh & 1;
          const uint64_t dxt = dXT + vb * (16384 / 16);
          mbar_wait(&bar.xt_full[vb], parity(nh / 2), status);
          // slice item n: dM^T and CB^T of columns [64 s, 64 s + 64) into slot n % 2.
          // The transform of item n - 2 has read the slot (its op_full was waited
          // for before item n - 1's products); CB^T waits for those products too.
          auto issue_item = [&](uint32_t n, int s) {
            const int rs = n & 1, ys = n % kNY;
            mbar_wait(&bar.dy_full[ys], parity(n / kNY), status);
            tc_fence_after();
            const uint32_t td = tmem + 128 * rs;
            pipe::umma_k<4>(td, dxt, dDY + ys * (8192 / 16), pipe::kStepK, pipe::kStepK, id_64, false);
            if (n >= 2) mbar_wait(&bar.slot_free[rs], parity(n / 2 - 1), status);
            tc_fence_after();
            const uint64_t dcs = dCR + s * (8192 / 16);
            pipe::umma_k<4>(td + 64, dBJ, dcs, pipe::kStepK, pipe::kStepK, id_64, false);
            pipe::umma_k<4>(td + 64, dBJ + 16384 / 16, dcs + 32768 / 16, pipe::kStepK, pipe::kStepK, id_64, true);
            umma_commit(&bar.ring_full[rs]);
          };
          issue_item(m, 0);
          for (int s = 0; s < nsl; ++s) {
            if (s + 1 < nsl) issue_item(m + s + 1, s + 1);
            const uint32_t n = m + s;
            const int rs = n & 1, ys = n % kNY;
            // M^T and W^T of item n in its slot (tensor memory): K step kk is the
            // 16 columns of transform warp group kk
            mbar_wait(&bar.op_full[rs], parity(n / 2), status);
            if (s == 0 && nh > 0) mbar_wait(bar.tu_free, parity(nh - 1), status);
            tc_fence_after();
            const uint32_t top = tmem + 128 * rs + 64;
            // T += M^T_s dy_s
            pipe::umma_ts_k<4>(tmem + kTmT, top, dDYmn + ys * (8192 / 16), 16, pipe::kStepMN, id_t, s > 0);
            umma_commit(&bar.dy_free[ys]);
            // dB += W^T_s C_s
            if (first_db && nu > 0) mbar_wait(bar.db_free, parity(nu - 1), status);
            tc_fence_after();
            pipe::umma_ts_k<4>(tmem + kTmDB, top + 8, dCRmn + s * (8192 / 16), 16, pipe::kStepMN, id_db, !first_db);
            first_db = false;
            umma_commit(&bar.slot_free[rs]);
          }
          m += nsl;
          // U = B_J dS^T, and dB += (wdt x) dS
          mbar_wait(bar.ds_full, parity(nd), status);
          tc_fence_after();
          pipe::umma_k<4>(tmem + kTmU, dBJ, dDS, pipe::kStepK, pipe::kStepK, id_64, false);
          pipe::umma_k<4>(tmem + kTmU, dBJ + 16384 / 16, dDS + 8192 / 16, pipe::kStepK, pipe::kStepK, id_64, true);
          umma_commit(bar.tu_full);
          const int as = na % kNA;
          mbar_wait(&bar.a_full[as], parity(na / kNA), status);
          tc_fence_after();
          pipe::umma_k<4>(tmem + kTmDB, dA + as * (16384 / 16), dDSmn, pipe::kStepK, pipe::kStepMN, id_db, true);
          umma_commit(&bar.a_free[as]);
          ++na;
          umma_commit(bar.ds_free);
          ++nd;
          umma_commit(&bar.xt_free[vb]);
        }
        umma_commit(bar.db_full);
        umma_commit(bar.unit_free);
      }
      // drain: every MMA issued here has completed and every commit arrival
      // has landed before the CTA releases its shared and tensor memory
      umma_commit(bar.drain);
      mbar_wait_drain(bar.drain, 0);
      if (nu > 0) {
        mbar_wait_drain(bar.unit_free, parity(nu - 1));
        mbar_wait_drain(bar.db_full, parity(nu - 1));
      }
      if (nh > 0) mbar_wait_drain(bar.tu_full, parity(nh - 1));
      for (uint32_t n = m > 2u ? m - 2u : 0u; n < m; ++n) {
        mbar_wait_drain(&bar.ring_full[n & 1], parity(n / 2));
        mbar_wait_drain(&bar.slot_free[n & 1], parity(n / 2));
      }
      for (uint32_t n = m > (uint32_t)kNY ? m - kNY : 0u; n < m; ++n)
        mbar_wait_drain(&bar.dy_free[n % kNY], parity(n / kNY));
      for (uint32_t n = na > (uint32_t)kNA ? na - kNA : 0u; n < na; ++n)
        mbar_wait_drain(&bar.a_free[n % kNA], parity(n / kNA));
      if (nd > 0) mbar_wait_drain(bar.ds_free, parity(nd - 1));
      for (uint32_t n = nh > 2u ? nh - 2u : 0u; n < nh; ++n) mbar_wait_drain(&bar.xt_free[n & 1], parity(n / 2));
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ transform
    // thread = row j of the tile (TMEM lane), 16 columns i per slice
    const int q = warp & 3, cg = (warp - 2) >> 2, jl = 32 * q + lane, tt = threadIdx.x - 64;
    const uint32_t sA = smem_u32(sm + kSmA), sV = smem_u32(sm + kSmV), sD = smem_u32(sm + kSmD),
                   sVC = smem_u32(sm + kSmVC), sXT = smem_u32(sm + kSmXT);
    const float kLog2e = 1.4426950408889634f;
    uint32_t nu = 0, nh = 0, m = 0, na = 0;
    size_t prev_tok = 0;
    int prev_vb = -1;
    auto flush_vcol = [&]() {
      if (prev_vb >= 0 && cg == 0) {
        const uint32_t base = sVC + prev_vb * 2048 + 4 * jl;
        tok[prev_tok] = (pipe::lds_f(base) + pipe::lds_f(base + 512)) + (pipe::lds_f(base + 1024) + pipe::lds_f(base + 1536));
      }
    };
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int j = 128 * o.J + jl, row_lo = 128 * o.J + 32 * q, row_hi = row_lo + 31;
      const int nsl = (pr.Q - 128 * o.J) / 64;
      int end_j = pr.Q - 1;
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, vb = nh & 1;
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vdt = vacs + 1024, vseq = vacs + 2048 + 16;
        const uint32_t ta = sD + vb * 2048, tg = ta + 1024;
        if (hh == 0 && has_seq) {  // last token of row j's sequence inside the chunk
          const int sj = pipe::lds_i(vseq + 4 * j);
          end_j = j;
          while (end_j < pr.Q - 1 && pipe::lds_i(vseq + 4 * (end_j + 1)) == sj) ++end_j;
        }
        const float acs_j = pipe::lds_f(vacs + 4 * j), dt_j = pipe::lds_f(vdt + 4 * j);
        const bool in_last = !has_seq || pipe::lds_i(vseq + 4 * j) == pipe::lds_i(vseq + 4 * (pr.Q - 1));
        const float wdt = in_last ? expf(pipe::lds_f(vacs + 4 * (pr.Q - 1)) - acs_j) * dt_j : 0.f;
        if (tt < pr.Q) {
          const float a = pipe::lds_f(vacs + 4 * tt) * kLog2e;
          pipe::sts_f(ta + 4 * tt, a);
          pipe::sts_f(tg + 4 * tt, ex2_approx(a - pipe::lds_f(vacs + 4 * (tt & ~15)) * kLog2e));
        }
        pipe::transform_sync<kTThreads>();
        flush_vcol();
        const float aj = acs_j * kLog2e;
        float vcol = 0.f;
        for (int s = 0; s < nsl; ++s, ++m) {
          const int rs = m & 1, i0 = 128 * o.J + 64 * s + 16 * cg;
          // M^T and W^T of this slice go, as bf16 pairs, over the CB^T columns this
          // warp has just read (no other warp reads them): M^T in the first 8,
          // W^T in the last 8, each half stored as soon as it is packed
          const uint32_t tdst = pipe::tmem_quad(tmem + 128 * rs + 64, 16 * cg);
          uint32_t mw[4], ww[4];
          auto put_half = [tdst](int e, const uint32_t(&a)[4], const uint32_t(&b)[4]) {
            const int off = e < 8 ? 0 : 4;  // columns 0-7 (e = 4) or 8-15 (e = 12) are packed
            tmem_st4_async(tdst + off, a[0], a[1], a[2], a[3]);
            tmem_st4_async(tdst + 8 + off, b[0], b[1], b[2], b[3]);
          };
          mbar_wait(&bar.ring_full[rs], parity(m / 2), status);
          tc_fence_after();
          if (i0 + 15 < row_lo) {  // every column before every row: zero
#pragma unroll
            for (int e = 0; e < 4; ++e) mw[e] = ww[e] = 0u;
            put_half(4, mw, ww);
            put_half(12, mw, ww);
          } else {
            float dm[16], cbv[16];
            tmem_ld16(pipe::tmem_quad(tmem + 128 * rs, 16 * cg), dm);
            tmem_ld16(pipe::tmem_quad(tmem + 128 * rs + 64, 16 * cg), cbv);
            if (i0 >= row_hi) {  // every column at or after every row: factorised decay
              const float e0 = ex2_approx(pipe::lds_f(ta + 4 * i0) - aj), ed = e0 * dt_j;
              const bool nomask = __all_sync(0xffffffffu, end_j >= i0 + 15);
              // two columns per packed fp32 instruction
              const uint64_t ed2 = pk2(ed, ed);
              uint64_t vs2 = pk2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 g4 = pipe::lds_f4(tg + 4 * (i0 + e));
                float gv[4] = {g4.x, g4.y, g4.z, g4.w};
                if (!nomask) {
#pragma unroll
                  for (int k4 = 0; k4 < 4; ++k4) gv[k4] = i0 + e + k4 <= end_j ? gv[k4] : 0.f;
                }
#pragma unroll
                for (int k4 = 0; k4 < 4; k4 += 2) {
                  const uint64_t g2 = pk2(gv[k4], gv[k4 + 1]), t2 = mul2(g2, ed2);
                  const uint64_t dm2 = pk2(dm[e + k4], dm[e + k4 + 1]), cb2 = pk2(cbv[e + k4], cbv[e + k4 + 1]);
                  vs2 = fma2(mul2(dm2, cb2), g2, vs2);
                  float m0, m1, w0, w1;
                  upk2(mul2(cb2, t2), m0, m1);
                  upk2(mul2(dm2, t2), w0, w1);
                  mw[((e + k4) / 2) & 3] = tc::pack_bf16x2(m0, m1);
                  ww[((e + k4) / 2) & 3] = tc::pack_bf16x2(w0, w1);
                }
                if (e == 4 || e == 12) put_half(e, mw, ww);
              }
              float vs_lo, vs_hi;
              upk2(vs2, vs_lo, vs_hi);
              vcol = fmaf(vs_lo + vs_hi, e0, vcol);
            } else {  // on the diagonal: one 2^x per element, the products two columns at a time
              float vdiag = 0.f;
              const uint64_t dt2 = pk2(dt_j, dt_j);
              uint64_t vc2 = pk2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 a4 = pipe::lds_f4(ta + 4 * (i0 + e));
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
                float ee[4], vx[4];
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                  const int i = i0 + e + k4;
                  const bool ok = (unsigned)(i - j) <= (unsigned)(end_j - j);
                  ee[k4] = ok ? ex2_approx(av[k4] - aj) : 0.f;
                  // the column sum leaves out i = j (it cancels exactly against the row
                  // sum's in the Acs adjoint); that term V_jj goes to its own slot
                  const float vij = dm[e + k4] * cbv[e + k4];
                  vdiag = i == j ? vij : vdiag;
                  vx[k4] = i == j ? 0.f : vij;
                }
#pragma unroll
                for (int k4 = 0; k4 < 4; k4 += 2) {
                  const uint64_t e2 = pk2(ee[k4], ee[k4 + 1]), t2 = mul2(e2, dt2);
                  vc2 = fma2(pk2(vx[k4], vx[k4 + 1]), e2, vc2);
                  float m0, m1, w0, w1;
                  upk2(mul2(pk2(cbv[e + k4], cbv[e + k4 + 1]), t2), m0, m1);
                  upk2(mul2(pk2(dm[e + k4], dm[e + k4 + 1]), t2), w0, w1);
                  mw[((e + k4) / 2) & 3] = tc::pack_bf16x2(m0, m1);
                  ww[((e + k4) / 2) & 3] = tc::pack_bf16x2(w0, w1);
                }
                if (e == 4 || e == 12) put_half(e, mw, ww);
              }
              float vc_lo, vc_hi;
              upk2(vc2, vc_lo, vc_hi);
              vcol += vc_lo + vc_hi;
              if ((unsigned)(j - i0) < 16u) tok[1 * BHL + ((size_t)o.bb * pr.H + h) * pr.L + (size_t)o.c * pr.Q + j] = vdiag;
            }
          }
          tmem_wait_st();
          tc_fence_before();
          pipe::warp_arrive(&bar.op_full[rs]);
        }
        {  // wdt_j x_j, the A operand of the dS_end term of dB
          mbar_wait(&bar.xt_full[vb], parity(nh / 2), status);
          float xv[1][16];
          const uint32_t T = sXT + vb * 16384;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            float x8[8];
            tc::unpack8(pipe::lds_sw128(T, jl, 2 * cg + t), x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[0][8 * t + e] = x8[e] * wdt;
          }
          put_operands<1>(xv, na, sA, jl, cg, bar.a_full, bar.a_free, status);
        }
        pipe::sts_f(sVC + vb * 2048 + cg * 512 + 4 * jl, vcol);
        prev_tok = 2 * BHL + ((size_t)o.bb * pr.H + h) * pr.L + (size_t)o.c * pr.Q + j;
        prev_vb = vb;
        pipe::warp_arrive(&bar.xt_free[vb]);
        pipe::warp_arrive(&bar.vec_free[vb]);
      }
    }
    pipe::transform_sync<kTThreads>();
    flush_vcol();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, jl = 32 * q + lane;
    const uint32_t sV = smem_u32(sm + kSmV), sXT = smem_u32(sm + kSmXT), sE = smem_u32(sm + kSmE);
    // this warp's 32 rows of the dy tile, reused as its du_x staging: a box of
    // 32 rows x 32 fp32 columns, 128-byte rows in the 128-byte swizzle
    const uint32_t stage = sE + 4096 * q, srow = stage + 128 * lane;
    uint32_t nu = 0, nh = 0;
    for (;; ++nu) {
      const int ui = pipe::next_unit(bar.units, nu, nunits, true);
      if (ui >= nunits) break;
      const Unit o = unit_of(pr, NTI, nhb, HB, ui);
      const int j = 128 * o.J + jl, t = o.c * pr.Q + j;
      const int ybox = o.bb * pr.L + o.c * pr.Q + 128 * o.J + 32 * q;  // du row of the warp's first row
      for (int hh = 0; hh < HB; ++hh, ++nh) {
        const int h = o.h0 + hh, vb = nh & 1;
        // this thread's dy row from the head's dy tile; x from the x tile
        mbar_wait(bar.ey_full, parity(nh), status);
        uint4 dyr[8];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) dyr[q8] = pipe::lds_sw128(sE, jl, q8);
        mbar_wait(&bar.vec_full[vb], parity(nh / 2), status);
        const uint32_t vacs = sV + vb * kVecStride, vdt = vacs + 1024, vseq = vacs + 2048 + 16;
        const bool in_last = !has_seq || pipe::lds_i(vseq + 4 * j) == pipe::lds_i(vseq + 4 * (pr.Q - 1));
        const float wdt =
            in_last ? expf(pipe::lds_f(vacs + 4 * (pr.Q - 1)) - pipe::lds_f(vacs + 4 * j)) * pipe::lds_f(vdt + 4 * j)
                    : 0.f;
        pipe::warp_arrive(&bar.vec_free[vb]);
        const float Dh = __ldg(pr.D + h);
        mbar_wait(&bar.xt_full[vb], parity(nh / 2), status);
        const uint32_t xt = sXT + vb * 16384;
        mbar_wait(bar.tu_full, parity(nh), status);
        tc_fence_after();
        float qsum = 0.f, ddsum = 0.f;  // q_j and dy_j . x_j (the dD piece)
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          float tv[16], uv[16];
          tmem_ld16(pipe::tmem_quad(tmem + kTmT, 16 * cc), tv);
          tmem_ld16(pipe::tmem_quad(tmem + kTmU, 16 * cc), uv);
          if (cc == 3) {  // T and U read: the next head's products may start
            tc_fence_before();
            pipe::warp_arrive(bar.tu_free);
          }
#pragma unroll
          for (int t8 = 0; t8 < 2; ++t8) {
            float d8[8], x8[8];
            tc::unpack8(dyr[2 * cc + t8], d8);
            tc::unpack8(pipe::lds_sw128(xt, jl, 2 * cc + t8), x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int col = 8 * t8 + e;
              qsum = fmaf(x8[e], uv[col], qsum);
              ddsum = fmaf(d8[e], x8[e], ddsum);
              tv[col] += wdt * uv[col] + Dh * d8[e];
            }
          }
          // columns 16 cc.. of the row into the staging box of columns 32 (cc / 2)..;
          // the second box reuses the first's buffer once its store has read it
          if (cc == 2) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t k = 4 * (cc & 1) + e;  // 16-byte chunk of the 128-byte row
            pipe::sts_u4(srow + 16 * (k ^ (uint32_t)(lane & 7)),
                         make_uint4(__float_as_uint(tv[4 * e]), __float_as_uint(tv[4 * e + 1]),
                                    __float_as_uint(tv[4 * e + 2]), __float_as_uint(tv[4 * e + 3])));
          }
          if (cc & 1) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_du, stage, h * pr.P + 32 * (cc >> 1), ybox);
              bulk_commit();
            }
          }
        }
        pipe::warp_arrive(&bar.xt_free[vb]);
        tok[4 * BHL + ((size_t)o.bb * pr.H + h) * pr.L + t] = qsum;
        tok[5 * BHL + ((size_t)o.bb * pr.H + h) * pr.L + t] = ddsum;
        // the buffer takes the next head's dy rows once the stores have read it
        // (after the unit's last head, once the dB stores below have read it too)
        if (hh + 1 < HB) {
          if (lane == 0) bulk_wait_read0();
          pipe::warp_arrive(bar.ey_free);
        }
      }
      // the unit's dB partial (columns of its head block in the (b L, H/HB N)
      // partial rows) through the same staging box, 32 columns at a time
      mbar_wait(bar.db_full, parity(nu), status);
      tc_fence_after();
      const int xdb = (o.h0 / HB) * pr.N;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        float a[16];
        tmem_ld16(pipe::tmem_quad(tmem + kTmDB, 16 * cc), a);
        if (cc == 7) {
          tc_fence_before();
          pipe::warp_arrive(bar.db_free);
        }
        if ((cc & 1) == 0) {  // a new box: the buffer's previous store has read it
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t k = 4 * (cc & 1) + e;
          pipe::sts_u4(srow + 16 * (k ^ (uint32_t)(lane & 7)),
                       make_uint4(__float_as_uint(a[4 * e]), __float_as_uint(a[4 * e + 1]),
                                  __float_as_uint(a[4 * e + 2]), __float_as_uint(a[4 * e + 3])));
        }
        if (cc & 1) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm_db, stage, xdb + 32 * (cc >> 1), ybox);
            bulk_commit();
          }
        }
      }
      if (lane == 0) bulk_wait_read0();
      pipe::warp_arrive(bar.ey_free);
    }
    if (lane == 0) bulk_wait0();  // the du_x and dB stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

void launch_tc_bwd_col(const Problem &pr, const bf16 *u, const bf16 *dy, const float *dtv, const float *acs,
                       const bf16 *dse16, float *du, float *dbp, float *tok, int *status, cudaStream_t s) {
  static bool once = (cudaFuncSetAttribute(tc_bwd_col_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes),
                      true);
  (void)once;
  CUtensorMap tm_u, tm_dy, tm_ds, tm_du, tm_db;
  const uint64_t HP = (uint64_t)pr.H * pr.P;
  const int HB = tc_head_subset(pr);
  const uint64_t dbcols = (uint64_t)(pr.H / HB) * pr.N;  // the dB partial rows: (b L, H / HB, N)
  if (!encode_tmap_bf16_2d(&tm_u, u, pr.Cd, (uint64_t)pr.b * pr.L, (uint64_t)pr.Cd * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_dy, dy, HP, (uint64_t)pr.b * pr.L, HP * 2, 64, 64) ||
      !encode_tmap_bf16_2d(&tm_ds, dse16, pr.N, (uint64_t)pr.b * pr.nc * pr.H * pr.P, (uint64_t)pr.N * 2, 64, 64) ||
      !encode_tmap_f32_2d(&tm_du, du, pr.Cd, (uint64_t)pr.b * pr.L, (uint64_t)pr.Cd * 4, 32, 32) ||
      !encode_tmap_f32_2d(&tm_db, dbp, dbcols, (uint64_t)pr.b * pr.L, dbcols * 4, 32, 32)) {
    note_host_error();
    return;
  }
  const int nunits = (pr.Q / 128) * pr.b * pr.nc * (pr.H / HB);
  const int grid = nunits < device_sm_count() ? nunits : device_sm_count();
  int *counter = status + kCounterCol;  // zeroed with the status word
  tc_bwd_col_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_u, tm_dy, tm_ds, tm_du, tm_db, pr, dtv, acs, tok, HB, nunits,
                                                       counter, status);
}

}  // namespace ssd
