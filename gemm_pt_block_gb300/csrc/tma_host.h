// tma_host.h -- host-side helpers for TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so no libcuda link is needed).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace mx {

inline PFN_cuTensorMapEncodeTiled_v12000 tma_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The tensor-map encoder is a driver-API call: it needs the device's context to
// be current in the calling thread, which a thread that has not yet made a
// runtime call that binds it (for example a framework's worker thread) may
// lack. Binds the current device's primary context once per thread.
inline void ensure_context() {
  thread_local bool bound = false;
  if (!bound) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaSetDevice(dev);
    bound = true;
  }
}

// 2-D row-major tensor [rows, cols] with leading dimension ld (elements), box
// [box_rows, box_cols], 128-byte swizzle (box_cols * elem_bytes must be <= 128),
// out-of-bounds elements read as zero.
inline bool make_tma_2d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t elem_bytes, const void* base,
                        int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
                        uint32_t box_cols) {
  auto fn = tma_encode_fn();
  if (!fn) return false;
  ensure_context();
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * elem_bytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte array [rows, row_bytes] (row_bytes % 16 == 0, base 16-byte aligned)
// written by tiled stores of box_rows x box_bytes boxes, unswizzled: the box's
// image in shared memory is row-major. Stores are clipped at the edges.
inline bool make_byte_store_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes,
                                uint32_t box_rows, uint32_t box_bytes) {
  auto fn = tma_encode_fn();
  if (!fn) return false;
  ensure_context();
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mx
