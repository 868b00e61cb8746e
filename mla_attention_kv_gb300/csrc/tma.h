// tma.h -- Tensor Memory Accelerator helpers: host-side encoding of 2-D
// tiled tensor maps (through the runtime's driver entry point, so the
// library does not link libcuda directly) and the device-side tiled copy.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Encode a 2-D row-major tensor map: `inner` elements per row (contiguous),
// `outer` rows, `row_stride` bytes between rows (multiple of 16), box of
// box_inner x box_outer elements.  Returns false if the CUDA driver rejects it.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_stride, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Encode a 3-D view of a row-major matrix [rows, cols] (cols a multiple of
// `inner`): element (x, y, z) = M[y][z * inner + x], i.e. dims {inner, rows,
// cols / inner} with strides {row_stride, inner * element size}.  A box
// {inner, box_rows, box_blocks} lands in shared memory as box_blocks
// consecutive [box_rows x inner] blocks -- the MN-major layout of a tensor-core
// operand made of inner-wide column groups.
bool encode_tmap_3d_colblocks(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t cols, uint64_t rows, uint64_t row_stride, uint32_t inner,
                              uint32_t box_rows, uint32_t box_blocks, uint32_t elem_bytes,
                              CUtensorMapSwizzle swizzle);

#ifdef __CUDACC__
// Tiled 2-D load of one box into shared memory; completion is counted in
// bytes on `bar`.  c_inner * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c_inner,
                                            int c_outer, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(map), "r"(c_inner), "r"(c_outer), "r"(bar)
      : "memory");
}
// Tiled loads into this CTA's shared memory whose completion (bytes) is
// counted on an mbarrier of either CTA of a pair (`bar` is a cluster
// address): the 2-SM MMA's operands arrive on the issuing CTA's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c_inner,
                                                 int c_outer, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(map), "r"(c_inner), "r"(c_outer), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// L2 prefetch of one box (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c_inner, int c_outer) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(map),
               "r"(c_inner), "r"(c_outer)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
#endif

}  // namespace mla
