// Linformer-style low-rank branch (WorldAttention review page, HSA section,
// linear branch).  Placeholder until the projection kernel lands.
#include "wa_internal.cuh"

namespace wa {

wa_status launch_linear_branch(const void*, int, const void*, const void*, int, const void*,
                               const void*, int, const void*, const void*, int, int, float,
                               const float*, const float*, int, void*, int, cudaStream_t) {
  return WA_ERR_UNIMPLEMENTED;
}

}  // namespace wa
