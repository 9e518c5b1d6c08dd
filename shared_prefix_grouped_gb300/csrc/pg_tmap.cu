// Host helper: TMA tensor maps, created through the driver entry point the runtime exposes (so the
// library does not link the driver library and loads on machines without one).
#include <cudaTypedefs.h>

#include <mutex>

#include "pg_internal.h"
#include "pg_tmap.h"

namespace pg {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

pg_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return PG_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_stride_bytes & 15u)) {
    set_error("TMA needs 16-byte aligned base and row stride");
    return PG_ERR_INVALID_ARG;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, stride %llu, box %u x %u",
              (int)r, (unsigned long long)inner, (unsigned long long)outer,
              (unsigned long long)row_stride_bytes, box_inner, box_outer);
    return PG_ERR_CUDA;
  }
  return PG_OK;
}

pg_status make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                            uint32_t box0, uint32_t box1, uint32_t box2) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return PG_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (stride1_bytes & 15u) || (stride2_bytes & 15u)) {
    set_error("TMA needs 16-byte aligned base and strides");
    return PG_ERR_INVALID_ARG;
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (3-D) failed (%d): dims %llu x %llu x %llu, box %u x %u x %u",
              (int)r, (unsigned long long)d0, (unsigned long long)d1, (unsigned long long)d2,
              box0, box1, box2);
    return PG_ERR_CUDA;
  }
  return PG_OK;
}

pg_status make_tmap_2d_b32(CUtensorMap* map, const void* base, bool is_float, uint64_t inner,
                           uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                           uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return PG_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_stride_bytes & 15u)) {
    set_error("TMA needs 16-byte aligned base and row stride");
    return PG_ERR_INVALID_ARG;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, is_float ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_INT32,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (32-bit) failed (%d)", (int)r);
    return PG_ERR_CUDA;
  }
  return PG_OK;
}

}  // namespace pg
