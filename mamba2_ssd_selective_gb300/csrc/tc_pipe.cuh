// Pieces shared by the persistent, warp-specialised tensor-core kernels: 1-D
// bulk copies, phase bookkeeping for mbarrier rings, and the host-side TMA
// tensor-map encoder (fetched from the driver at run time, no libcuda link).
//
// Ring discipline used by every such kernel: the m-th completion of a barrier
// has phase parity m & 1; a waiter on the m-th completion passes
// mbar_wait(bar, m & 1).  Every barrier's (m+1)-th completion depends on an
// arrival from each of its waiters' m-th use, so no barrier ever runs two
// phases ahead of a waiter (which parity waits could not tell apart).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "sm100.cuh"

namespace ssd {
namespace pipe {

using namespace sm100;

// 1-D bulk copy global -> this CTA's shared memory; completion counted in bytes
// on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint32_t parity(uint32_t m) { return m & 1u; }

// explicit shared-memory accesses (32-bit shared addresses)
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ int4 lds_i4(uint32_t a) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_i(uint32_t a) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u4(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Consumer arrivals are made once per warp: every lane's earlier shared-memory
// writes (made visible to the async proxy by its own fence where needed) are
// ordered before lane 0's release by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void sts_f(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// barrier among the `n` threads of the transform warps (named barrier 1)
template <int n>
__device__ __forceinline__ void transform_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(n) : "memory");
}

// 8 bf16 from a 128-byte-swizzled [rows x 64] bf16 tile: row r, columns 8c..8c+7
__device__ __forceinline__ uint4 lds_sw128(uint32_t tile, int r, int c) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(tile + sw128_offset(r, 8 * c)));
  return v;
}

// Dynamic work distribution for the persistent kernels: the producer lane
// claims the next work unit from a global counter and hands it to the other
// roles through a two-entry ring in shared memory (full[b]: count 1; free[b]:
// one arrival per consumer warp or thread).
//
// Both sides wait on this ring with mbar_wait_drain, which does not give up
// when the status word is raised: every consumer reads every published value,
// in order, so all warps of a role work through the same units and reach
// their named barriers the same number of times, even on a failing pass.  The
// producer always publishes: after one of its own waits has failed it
// publishes `stop`, and the consumers end together.
struct UnitRing {
  uint64_t *full, *free;  // [2] each
  int *slot;              // [2]
};
// Producer lane: publish unit `u` (claimed earlier with atomicAdd, so the
// atomic's latency hides behind the previous unit's loads) as the n-th unit.
__device__ __forceinline__ int publish_unit(const UnitRing &r, uint32_t n, int u, int stop) {
  const int b = n & 1;
  if (n >= 2 && !mbar_wait_drain(&r.free[b], parity(n / 2 - 1))) u = stop;
  if (u > stop) u = stop;
  *reinterpret_cast<volatile int *>(&r.slot[b]) = u;
  mbar_arrive(&r.full[b]);
  return u;
}
// consumers: warp_level = one arrival per warp (all lanes call), else one per thread
__device__ __forceinline__ int next_unit(const UnitRing &r, uint32_t n, int stop, bool warp_level) {
  const int b = n & 1;
  const bool ok = mbar_wait_drain(&r.full[b], parity(n / 2));
  const int u = ok ? *reinterpret_cast<volatile int *>(&r.slot[b]) : stop;
  if (warp_level)
    warp_arrive(&r.free[b]);
  else
    mbar_arrive(&r.free[b]);
  return u;
}

// MMA issue with precomputed descriptors.  A 128-byte-swizzled descriptor's
// start address (16-byte units, bits 0-13) advances by a constant per K step
// of 16 elements: 2 for a K-major operand (32 bytes), 128 for an MN-major one
// (16 rows of 128 bytes).  Shared addresses stay below 2^18, so the field never
// carries.  D (+)= A B over K = 16 * NK, issued by the calling thread.
constexpr uint64_t kStepK = 2, kStepMN = 128;
template <int NK>
__device__ __forceinline__ void umma_k(uint32_t d, uint64_t a, uint64_t b, uint64_t sa, uint64_t sb, uint32_t idesc,
                                       bool accumulate) {
  umma_bf16(d, a, b, idesc, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < NK; ++kk) umma_bf16(d, a + kk * sa, b + kk * sb, idesc, 1u);
}

// The same with A in tensor memory: K step kk takes A from the 8 columns at
// a + kk * sa (sa >= 8 columns; the K steps need not be adjacent).
template <int NK>
__device__ __forceinline__ void umma_ts_k(uint32_t d, uint32_t a, uint64_t b, uint32_t sa, uint64_t sb, uint32_t idesc,
                                          bool accumulate) {
  umma_bf16_ts(d, a, b, idesc, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < NK; ++kk) umma_bf16_ts(d, a + kk * sa, b + kk * sb, idesc, 1u);
}

// TMEM address of (lane quadrant of this warp, column col)
__device__ __forceinline__ uint32_t tmem_quad(uint32_t base, int col) {
  return base + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}

}  // namespace pipe

// Host: 2-D bf16 tensor map over a row-major matrix (cols contiguous), box
// box_cols x box_rows, 128-byte swizzle (box_cols * 2 must be 128).  Returns
// false if the driver entry point is missing or the encoder rejects the map.
bool encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                         uint32_t box_cols, uint32_t box_rows);
// Host: the same for fp32 (box_cols * 4 must be 128).
bool encode_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_cols, uint32_t box_rows);
// Host: SM count of the current device (cached per device).
int device_sm_count();
// Host: record an error found while preparing a launch; the pass then returns
// SSD_ERR_CUDA (cleared when read).
void note_host_error();
bool take_host_error();

}  // namespace ssd
