// tma.cu -- host-side encoding of the row-gather tensor maps.
#include <cudaTypedefs.h>

#include <mutex>

#include "attn_tile.cuh"
#include "tma.cuh"

namespace gattn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

bool encode_rows_map(CUtensorMap* map, const void* base, int elem_bytes, bool is_bf16,
                     int64_t rows, int64_t width) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                 : (is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_UINT16);
  const cuuint64_t dims[2] = {cuuint64_t(width), cuuint64_t(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {cuuint64_t(width) * elem_bytes};
  const cuuint32_t box[2] = {cuuint32_t(width < kGatherBoxMax ? width : kGatherBoxMax), 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %lld map", int(r),
              (long long)rows, (long long)width);
    return false;
  }
  return true;
}

bool encode_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t width) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const cuuint64_t dims[2] = {cuuint64_t(width), cuuint64_t(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {cuuint64_t(width) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %lld tile map", int(r),
              (long long)rows, (long long)width);
    return false;
  }
  return true;
}

}  // namespace gattn
