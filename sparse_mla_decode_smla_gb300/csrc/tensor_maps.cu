// Host-side TMA tensor maps of the decode inputs, encoded through the driver entry point
// (no link against the driver library). The last map of each kind is reused while its
// tensor and shape stay the same.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace smla {

cudaError_t tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  // looked up once; host threads that make their first call together look it up twice and
  // store the same value
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> encode{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = encode.load(std::memory_order_acquire);
  if (!f) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return cudaErrorNotSupported;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    encode.store(f, std::memory_order_release);
  }
  *out = f;
  return cudaSuccess;
}

int kv_row_bytes(int32_t kv_format) {
  return kv_format == SMLA_KV_FP8_TENSOR ? kFp8TensorRowBytes
                                         : (kv_format == SMLA_KV_FP8_DS ? kFp8RowBytes : kBf16RowBytes);
}

cudaError_t kv_gather_map(const DecodeArgs& a, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (tensor_map_encoder(&encode) != cudaSuccess) return cudaErrorNotSupported;
  thread_local const void* last_kv = nullptr;
  thread_local int64_t last_slots = -1;
  thread_local int32_t last_fmt = -1;
  thread_local CUtensorMap last_map;
  const int64_t slots = a.num_pages << a.log2_page;
  if (slots >= kMaxGatherSlots) return cudaErrorInvalidValue;
  if (last_kv == a.kv && last_slots == slots && last_fmt == a.kv_format) {
    *out = last_map;
    return cudaSuccess;
  }
  const cuuint64_t row = cuuint64_t(kv_row_bytes(a.kv_format));
  const cuuint64_t dims[2] = {row / 8, cuuint64_t(slots)};
  const cuuint64_t strides[1] = {row};
  const cuuint32_t box[2] = {cuuint32_t(row / 8), 1};
  const cuuint32_t estr[2] = {1, 1};
  // no L2 promotion: a row sits at an arbitrary offset, and promoting its fetches to 256-byte
  // lines would read about 3.5 lines (900 bytes) of HBM per 656-byte row
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(a.kv), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  last_kv = a.kv;
  last_slots = slots;
  last_fmt = a.kv_format;
  last_map = *out;
  return cudaSuccess;
}

cudaError_t q_tile_map(const DecodeArgs& a, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (tensor_map_encoder(&encode) != cudaSuccess) return cudaErrorNotSupported;
  thread_local const void* last_q = nullptr;
  thread_local int64_t last_rows = -1;
  thread_local CUtensorMap last_map;
  const int64_t rows = int64_t(a.T) * a.H;
  if (last_q == a.q && last_rows == rows) {
    *out = last_map;
    return cudaSuccess;
  }
  const cuuint64_t dims[2] = {cuuint64_t(kDim), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(2 * kDim)};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  last_q = a.q;
  last_rows = rows;
  last_map = *out;
  return cudaSuccess;
}

cudaError_t q_e4m3_maps(const DecodeArgs& a, CUtensorMap* map128, CUtensorMap* map32) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (tensor_map_encoder(&encode) != cudaSuccess) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(kDim), cuuint64_t(int64_t(a.T) * a.H)};
  const cuuint64_t strides[1] = {cuuint64_t(kDim)};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint32_t box128[2] = {128, 64};
  CUresult r = encode(map128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.q), dims, strides, box128, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const cuuint32_t box32[2] = {32, 64};
  r = encode(map32, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.q), dims, strides, box32, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace smla
