// gdn_fused.cu -- single-launch fused path (tcgen05 / TMEM / TMA on sm_103a).
#include "gdn_internal.h"

namespace gdn {

bool fused_supported(const gdn_problem&) { return false; }
size_t fused_workspace_bytes(const gdn_problem&) { return 0; }
size_t fused_status_offset(const gdn_problem&) { return 0; }
gdn_status run_fused(const gdn_problem&, const void*, const void*, const void*, const float*, const float*, float,
                     const float*, const int32_t*, void*, float*, void*, cudaStream_t) {
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
