// Host helpers for the tensor-core launchers: TMA tensor-map encoding through
// the driver entry point (no link against libcuda), the SM count, and a
// per-thread flag for errors found while preparing a launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tc_pipe.cuh"

namespace ssd {

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiled>(nullptr);
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

thread_local bool t_host_error = false;

}  // namespace

namespace {

// 2-D map with 128-byte rows in the box and the 128-byte swizzle
bool encode_sw128_2d(CUtensorMap *map, CUtensorMapDataType type, uint32_t elem_bytes, const void *base, uint64_t cols,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiled fn = encoder();
  if (!fn || box_cols * elem_bytes != 128 || (reinterpret_cast<uintptr_t>(base) & 15) || (row_bytes & 15))
    return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                         uint32_t box_cols, uint32_t box_rows) {
  return encode_sw128_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, row_bytes, box_cols, box_rows);
}

bool encode_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_cols, uint32_t box_rows) {
  return encode_sw128_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, rows, row_bytes, box_cols, box_rows);
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

void note_host_error() { t_host_error = true; }
bool take_host_error() {
  const bool e = t_host_error;
  t_host_error = false;
  return e;
}

}  // namespace ssd
