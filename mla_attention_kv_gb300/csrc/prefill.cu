// prefill.cu -- tensor-core (tcgen05) MLA KV prolog for large token counts.
#include "common.cuh"
#include "internal.h"

namespace mla {

bool prefill_preferred(int, int, int, int) { return false; }

cudaError_t prefill_launch(bool, const PrefillParams&, int, cudaStream_t, int* launches) {
  *launches = 0;
  return cudaErrorNotSupported;
}

}  // namespace mla
