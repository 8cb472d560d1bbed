// A small tcgen05 contraction engine for the chunk-state and Z kernels of the
// bf16 path.
//
// One CTA of 256 threads owns a 128-row accumulator block in tensor memory
// (TMEM lane = row; all 256 threads stage operands, threads 0..127 drain it).
// A contraction  D[128 x NT] = sum_k A[m,k] B[n,k]  with both operands MN-major
// (8 consecutive m or n of one k contiguous in the source) is fed 64 k at a
// time: A is copied as it is with cp.async, B goes through registers as
// fetch(n, k) -> raw data and make(raw, n, k) -> 8 packed bf16 (so scalings are
// applied while staging and nothing is materialised in HBM), both straight into
// the 128-byte-swizzled UMMA layout; one thread then issues four 128 x NT x 16
// tcgen05.mma and commits them to the stage's mbarrier.  The loads of the next
// slice are in flight while the current one is staged and its MMAs run.
#pragma once

#include <cuda_bf16.h>

#include "sm100.cuh"

namespace ssd {
namespace tc {

using namespace sm100;

// Every engine CTA has kThreads threads: all of them stage operands; the first
// 128 (warps 0-3, one per TMEM lane quadrant) drain the accumulator rows.
constexpr int kThreads = 256;

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
  int *status;     // raised if an MMA completion ever fails to arrive in time
  uint32_t uses[NSTAGE];
  uint32_t done_uses;

  // call from all threads; thread 0 initialises the barriers (sync afterwards)
  __device__ void init(uint8_t *ring_, uint64_t *bars_, int *status_) {
    ring = ring_;
    bars = bars_;
    status = status_;
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) uses[s] = 0;
    done_uses = 0;
    if (threadIdx.x == 0) {
      for (int s = 0; s <= NSTAGE; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
    }
  }

  // The engine's only waits are for completions of MMAs this CTA issued, which
  // always arrive: they ignore the status word (so a failure elsewhere in the
  // pass does not corrupt this kernel's results) and are bounded all the same.
  __device__ __forceinline__ void wait_mma(uint64_t *bar, uint32_t parity) {
    if (!mbar_wait_drain(bar, parity)) atomicExch(status, 1);
  }

  // cp.async of the A tile of the 64-wide k slice [k0, k0+64) into its stage:
  // fl(m, k) is the global address of the 16 bytes holding A[m .. m+7, k].
  template <class FL>
  __device__ __forceinline__ void stage_A(uint8_t *A, int k0, const FL &fl) {
    constexpr int PER = (128 * 8) / kThreads;  // 16-byte chunks per thread
    const uint32_t a0 = smem_u32(A);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int e = threadIdx.x + q * kThreads;
      const int r = e >> 4, c = e & 15;  // two 64-wide MN atoms, 64 k-rows each
      cp_async16(a0 + (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8), fl(c * 8, k0 + r));
    }
  }

  // A whole contraction over k in [0, nk) (nk a multiple of 64) with both
  // operands MN-major, A copied as it is (cp.async) and B through fetch/make,
  // software-pipelined: the loads of slice s+1 (A's copies and B's registers)
  // are issued before slice s's B is transformed and stored and its MMAs
  // issued, so a slice of loads is always in flight behind the one being
  // staged.  Split in two so that the caller can issue slice 0's loads first
  // and overlap them with its own prologue (per-token weights, TMEM
  // allocation): prefetch0() issues them into `cur`, contract() runs the rest.
  // Both must be called by all threads.
  static constexpr int CPR = NT / 8, PER_B = (NT * 8) / kThreads;
  template <class FAL, class FBL, class Raw>
  __device__ __forceinline__ void issue(int s, const FAL &fal, const FBL &fbl, Raw (&raw)[PER_B]) {
    const int st = s % NSTAGE, k0 = 64 * s;
    if (uses[st] > 0) wait_mma(&bars[st], (uses[st] - 1) & 1);
    stage_A(ring + st * STAGE_BYTES, k0, fal);
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int q = 0; q < PER_B; ++q) {
      const int e = threadIdx.x + q * kThreads, r = e / CPR, c = e % CPR;
      raw[q] = fbl(c * 8, k0 + r);
    }
  }
  template <class FAL, class FBL, class Raw>
  __device__ __forceinline__ void prefetch0(const FAL &fal, const FBL &fbl, Raw (&cur)[PER_B]) {
    static_assert(NSTAGE >= 2 && NT % 64 == 0, "pipelined contraction: two stages, whole MN atoms");
    issue(0, fal, fbl, cur);
  }
  template <class FAL, class FBL, class FBM, class Raw>
  __device__ __forceinline__ void contract(uint32_t tmem_d, int nk, const FAL &fal, const FBL &fbl, const FBM &fbm,
                                           Raw (&cur)[PER_B]) {
    Raw nxt[PER_B];
    const int ns = nk / 64;
    for (int s = 0; s < ns; ++s) {
      const int st = s % NSTAGE, k0 = 64 * s;
      const bool more = s + 1 < ns;
      if (more) issue(s + 1, fal, fbl, nxt);
      uint8_t *A = ring + st * STAGE_BYTES, *B = A + A_BYTES;
#pragma unroll
      for (int q = 0; q < PER_B; ++q) {
        const int e = threadIdx.x + q * kThreads, r = e / CPR, c = e % CPR;
        *reinterpret_cast<uint4 *>(B + (c >> 3) * 8192 + sw128_offset(r, (c & 7) * 8)) = fbm(cur[q], c * 8, k0 + r);
      }
      if (more)
        asm volatile("cp.async.wait_group 1;" ::: "memory");  // this slice's copies; the next may fly
      else
        cp_async_wait_all();
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
        constexpr uint32_t idesc = idesc_bf16(128, NT, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem_d, desc_sw128(a0 + kk * 2048, 8192, 1024), desc_sw128(b0 + kk * 2048, 8192, 1024), idesc,
                    (s > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[st]);
      }
      uses[st] += 1;
      if (more) {
#pragma unroll
        for (int q = 0; q < PER_B; ++q) cur[q] = nxt[q];
      }
    }
  }

  // Wait until every MMA issued so far has completed (all threads).
  __device__ __forceinline__ void finish() {
    if (threadIdx.x == 0) umma_commit(&bars[NSTAGE]);
    wait_mma(&bars[NSTAGE], done_uses & 1);
    done_uses += 1;
    tc_fence_after();
  }
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
// true for the threads that drain an accumulator row
__device__ __forceinline__ bool owns_row() { return threadIdx.x < 128; }

}  // namespace tc
}  // namespace ssd
