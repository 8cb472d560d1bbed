// A small tcgen05 contraction engine for the chunk kernels of the bf16 path.
//
// One CTA of 256 threads owns a 128-row accumulator block in tensor memory
// (TMEM lane = row, owned by threads 0..127; all 256 threads stage operands).  A contraction  D[128 x NT] (+)= sum_k A[m,k] B[n,k]  is
// fed 64 k at a time: every thread stages its share of the A and B tiles
// straight into shared memory in the 128-byte-swizzled UMMA layout (so masks,
// decays and scalings are applied while staging and nothing is materialised in
// HBM), then one thread issues four 128 x NT x 16 tcgen05.mma and commits them
// to the stage's mbarrier.  A ring of NSTAGE stages lets the staging of the
// next 64-k slice overlap the tensor-core work of the previous ones.
//
// Each operand is given as fetch(m, k) -> raw data and make(raw, m, k) -> 8 bf16
// packed in a uint4:
//   K-major operand:  elements (m, k .. k+7)
//   MN-major operand: elements (m .. m+7, k)
// (pick the one whose 8 elements are contiguous in the source).
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "sm100.cuh"

namespace ssd {
namespace tc {

using namespace sm100;

enum Major : int { K_MAJOR = 0, MN_MAJOR = 1 };
// Every engine CTA has kThreads threads: all of them stage operands; the first
// 128 (warps 0-3, one per TMEM lane quadrant) own the accumulator rows.
constexpr int kThreads = 256;
constexpr int kRows = 128;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 ldg16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void ld8f(const float *p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// make() marker for operands copied as they are: fetch(m, k) then returns the
// global address of the 16 bytes, and the engine copies them with cp.async
// straight into their swizzled slot (no registers, every copy in flight at once).
struct Async {};
template <class FM>
constexpr bool kIsAsync = std::is_same<FM, Async>::value;

template <int NT, int NSTAGE>
struct Engine {
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "UMMA N for M = 128");
  static constexpr uint32_t A_BYTES = 128 * 128;  // 128 rows x 64 k bf16
  static constexpr uint32_t B_BYTES = NT * 128;   // NT rows x 64 k bf16
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr uint32_t BAR_BYTES = (NSTAGE + 1) * 8;

  uint8_t *ring;   // 1024-aligned
  uint64_t *bars;  // [0, NSTAGE): stage free;  [NSTAGE]: all issued MMAs done
  int *status;
  uint32_t uses[NSTAGE];
  uint32_t done_uses;
  int stage;

  // call from all threads; thread 0 initialises the barriers (sync afterwards)
  __device__ void init(uint8_t *ring_, uint64_t *bars_, int *status_) {
    ring = ring_;
    bars = bars_;
    status = status_;
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) uses[s] = 0;
    done_uses = 0;
    stage = 0;
    if (threadIdx.x == 0) {
      for (int s = 0; s <= NSTAGE; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
    }
  }

  // Operands come as two callables: fetch(m, k) issues the global loads and
  // returns the raw data, make(raw, m, k) turns it into 8 packed bf16.  Every
  // thread first issues the loads of kBatch chunks back to back, then
  // transforms and stores them, so kBatch loads per thread are in flight.
  static constexpr int kBatchMax = 4;

  template <int MA, class FL, class FM>
  __device__ __forceinline__ void stage_A(uint8_t *A, int k0, const FL &fl, const FM &fm) {
    using Raw = decltype(fl(0, 0));
    constexpr int PER = (128 * 8) / kThreads;  // 16-byte chunks per thread
    constexpr int kBatch = PER < kBatchMax ? PER : kBatchMax;
    if constexpr (kIsAsync<FM>) {
      const uint32_t a0 = smem_u32(A);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int e = threadIdx.x + q * kThreads;
        if constexpr (MA == K_MAJOR) {
          const int m = e >> 3, c = e & 7;
          cp_async16(a0 + sw128_offset(m, c * 8), fl(m, k0 + c * 8));
        } else {
          const int r = e >> 4, c = e & 15;
          cp_async16(a0 + (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8), fl(c * 8, k0 + r));
        }
      }
      return;
    } else {
#pragma unroll
    for (int g = 0; g < PER; g += kBatch) {
      Raw raw[kBatch];
      int mm[kBatch], kk[kBatch];
      uint32_t off[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int e = threadIdx.x + (g + q) * kThreads;
        if constexpr (MA == K_MAJOR) {
          const int m = e >> 3, c = e & 7;
          mm[q] = m; kk[q] = k0 + c * 8; off[q] = sw128_offset(m, c * 8);
        } else {  // two 64-wide MN atoms, 64 k-rows each
          const int r = e >> 4, c = e & 15;
          mm[q] = c * 8; kk[q] = k0 + r; off[q] = (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8);
        }
        raw[q] = fl(mm[q], kk[q]);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) *reinterpret_cast<uint4 *>(A + off[q]) = fm(raw[q], mm[q], kk[q]);
    }
    }
  }

  template <int MB, class FL, class FM>
  __device__ __forceinline__ void stage_B(uint8_t *B, int k0, const FL &fl, const FM &fm) {
    using Raw = decltype(fl(0, 0));
    static_assert(MB == K_MAJOR || NT % 64 == 0, "MN-major B needs whole 64-wide atoms");
    constexpr int CPR = NT / 8;  // 16-byte chunks per k-row (MN-major)
    constexpr int PER = (NT * 8) / kThreads;
    constexpr int kBatch = PER < kBatchMax ? PER : kBatchMax;
    static_assert(PER >= 1 && PER % kBatch == 0, "B chunks per thread");
    if constexpr (kIsAsync<FM>) {
      const uint32_t b0 = smem_u32(B);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int e = threadIdx.x + q * kThreads;
        if constexpr (MB == K_MAJOR) {
          const int n = e >> 3, c = e & 7;
          cp_async16(b0 + sw128_offset(n, c * 8), fl(n, k0 + c * 8));
        } else {
          const int r = e / CPR, c = e % CPR;
          cp_async16(b0 + (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8), fl(c * 8, k0 + r));
        }
      }
      return;
    } else {
#pragma unroll
    for (int g = 0; g < PER; g += kBatch) {
      Raw raw[kBatch];
      int nn[kBatch], kk[kBatch];
      uint32_t off[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int e = threadIdx.x + (g + q) * kThreads;
        if constexpr (MB == K_MAJOR) {
          const int n = e >> 3, c = e & 7;
          nn[q] = n; kk[q] = k0 + c * 8; off[q] = sw128_offset(n, c * 8);
        } else {
          const int r = e / CPR, c = e % CPR;
          nn[q] = c * 8; kk[q] = k0 + r; off[q] = (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8);
        }
        raw[q] = fl(nn[q], kk[q]);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) *reinterpret_cast<uint4 *>(B + off[q]) = fm(raw[q], nn[q], kk[q]);
    }
    }
  }

  // Stage the 64-wide k slice [k0, k0+64) of A and B and issue its MMAs into the
  // accumulator at TMEM address tmem_d.  Must be called by all 128 threads.
  // With tmem_d2 != kNone the same staged operands are also issued into a
  // second accumulator (accumulate2 selects whether that one accumulates).
  static constexpr uint32_t kNone = 0xffffffffu;
  template <int MA, int MB, class FAL, class FAM, class FBL, class FBM>
  __device__ __forceinline__ void slice(uint32_t tmem_d, int k0, const FAL &fal, const FAM &fam, const FBL &fbl,
                                        const FBM &fbm, bool accumulate, uint32_t tmem_d2 = kNone,
                                        bool accumulate2 = false) {
    const int s = stage;
    if (uses[s] > 0) mbar_wait(&bars[s], (uses[s] - 1) & 1, status);
    uint8_t *A = ring + s * STAGE_BYTES;
    uint8_t *B = A + A_BYTES;
    stage_A<MA>(A, k0, fal, fam);
    stage_B<MB>(B, k0, fbl, fbm);
    if constexpr (kIsAsync<FAM> || kIsAsync<FBM>) cp_async_wait_all();
    fence_async_smem();
    tc_fence_before();  // order this thread's earlier TMEM reads before the MMAs below
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
      constexpr uint32_t idesc = idesc_bf16(128, NT, MA == MN_MAJOR, MB == MN_MAJOR);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = MA == K_MAJOR ? desc_sw128(a0 + kk * 32, 16, 1024) : desc_sw128(a0 + kk * 2048, 8192, 1024);
        const uint64_t bd = MB == K_MAJOR ? desc_sw128(b0 + kk * 32, 16, 1024) : desc_sw128(b0 + kk * 2048, 8192, 1024);
        umma_bf16(tmem_d, ad, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
        if (tmem_d2 != kNone) umma_bf16(tmem_d2, ad, bd, idesc, (accumulate2 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&bars[s]);
    }
    uses[s] += 1;
    stage = (s + 1 == NSTAGE) ? 0 : s + 1;
  }

  // Wait until every MMA issued so far has completed (all threads).
  __device__ __forceinline__ void finish() {
    if (threadIdx.x == 0) umma_commit(&bars[NSTAGE]);
    mbar_wait(&bars[NSTAGE], done_uses & 1, status);
    done_uses += 1;
    tc_fence_after();
  }
};

// make() for operands that are already 8 packed bf16
struct AsIs {
  __device__ __forceinline__ uint4 operator()(uint4 r, int, int) const { return r; }
};
// 8 fp32 values fetched as two float4
struct F8 {
  float4 a, b;
};
__device__ __forceinline__ F8 ldf8(const float *p) {
  return F8{__ldg(reinterpret_cast<const float4 *>(p)), __ldg(reinterpret_cast<const float4 *>(p) + 1)};
}
__device__ __forceinline__ void f8_to(const F8 &r, float (&v)[8]) {
  v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w; v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}
// two fp32 rows fetched together (state + segment state, combined in make())
struct F16 {
  F8 x, y;
};

// Shared-memory carve-up helper for kernels built on the engine: returns the
// 1024-aligned ring base inside the dynamic shared memory window.
__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw) {
  const uint32_t a = smem_u32(raw);
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

// TMEM allocation by warp 0 of the CTA; returns the base address to all threads.
__device__ __forceinline__ uint32_t tmem_alloc_cta(uint32_t *slot, uint32_t ncols) {
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *slot;
}
__device__ __forceinline__ void tmem_free_cta(uint32_t base, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(base, ncols);
}

// TMEM address of (this thread's lane, column col); threads 0..127 own lanes 0..127.
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int col) {
  return base + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}
// true for the threads that own an accumulator row
__device__ __forceinline__ bool owns_row() { return threadIdx.x < kRows; }

}  // namespace tc
}  // namespace ssd
