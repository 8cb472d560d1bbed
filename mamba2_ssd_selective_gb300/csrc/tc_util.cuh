// Small helpers of the tensor-core kernels: bf16 packing and unpacking, a
// read-only 16-byte global load, and the 1024-byte alignment of the dynamic
// shared-memory window (128-byte-swizzled TMA tiles and UMMA operands need it).
#pragma once

#include <cuda_bf16.h>

#include "sm100.cuh"

namespace ssd {
namespace tc {

using namespace sm100;

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

// The 1024-aligned base inside the dynamic shared memory window.
__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw) {
  const uint32_t a = smem_u32(raw);
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace tc
}  // namespace ssd
