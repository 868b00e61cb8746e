// tma.cu -- host-side tensor-map encoding (see tma.h).
#include <cudaTypedefs.h>
#include <mutex>

#include "tma.h"

namespace mla {

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_stride, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_3d_colblocks(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t cols, uint64_t rows, uint64_t row_stride, uint32_t inner,
                              uint32_t box_rows, uint32_t box_blocks, uint32_t elem_bytes,
                              CUtensorMapSwizzle swizzle) {
  auto fn = get_encode();
  if (!fn || cols % inner != 0) return false;
  cuuint64_t dims[3] = {inner, rows, cols / inner};
  cuuint64_t strides[2] = {row_stride, (cuuint64_t)inner * elem_bytes};
  cuuint32_t box[3] = {inner, box_rows, box_blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mla
