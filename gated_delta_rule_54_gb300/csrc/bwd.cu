// Backward (identity STE) — placeholder until the kernels land.
#include "common.cuh"
#include "launch.h"

namespace gdn {
size_t bwd_workspace_bytes(const gdn_problem&, const Dims&) { return 0; }
gdn_status launch_bwd(const gdn_problem&, const Dims&, const void*, const void*, const void*,
                      const float*, const float*, const void*, const void*, const float*, float*,
                      float*, float*, float*, float*, float*, void*, cudaStream_t) {
  return GDN_ERR_UNSUPPORTED_MODE;
}
}  // namespace gdn
