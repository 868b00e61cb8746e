// w8a8.cu -- W8A8 full MLA prolog (int8 weights, per-token int8 activations).
#include "common.cuh"
#include "internal.h"

namespace mla {

size_t w8_workspace_bytes(int, int, int, int) { return 0; }
void w8_workspace_carve(void*, int, int, int, int, W8Workspace* w) { *w = W8Workspace{}; }
cudaError_t w8a8_launch(const W8Params&, const W8Workspace&, int, cudaStream_t, int* launches) {
  *launches = 0;
  return cudaErrorNotSupported;
}
cudaError_t w8a8_quant_rows_launch(const void*, int, int, int8_t*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t w8a8_gemm_s32_launch(const int8_t*, const int8_t*, int, int, int, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t w8a8_copy_operands(const W8Workspace&, int, int, int8_t*, float*, int8_t*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
