// Host helper: TMA tensor maps for [rows][heads][head_dim] bf16 tensors,
// tiled 64 elements (128 bytes, 128-byte swizzle) x 1 head x 128 rows, and for
// the backward's float32 dQ accumulator.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>

namespace cpattn {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};  // an idempotent first lookup
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// Map of a bf16 tensor viewed as [rows][heads][d] (d innermost), box
// {64, 1, box_rows}.  Returns false on failure.
inline bool make_tmap_rows(CUtensorMap* map, const void* base, int64_t rows, int heads, int d,
                           int box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, cuuint32_t(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map of a float32 tensor viewed as [planes][rows][128] (128 innermost), box
// {32, 128 rows, 1}: 128-byte rows, 128-byte swizzle (used to reduce 32-column
// chunks of a 128-row tile).  Returns false on failure.
inline bool make_tmap_f32_chunks(CUtensorMap* map, void* base, int64_t planes, int64_t rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, cuuint64_t(rows), cuuint64_t(planes)};
  cuuint64_t strides[2] = {128 * 4, cuuint64_t(rows) * 128 * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline int num_sms() {
  static std::atomic<int> n[64] = {};  // per device (an idempotent first lookup)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  int c = n[dev].load(std::memory_order_relaxed);
  if (!c) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    c = v > 0 ? v : 148;
    n[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace cpattn
