// Entry points whose kernels are not built yet: they validate nothing and report UNSUPPORTED.
#include "../../include/attnfuse.h"

extern "C" {
attnfuse_status attnfuse_bwd_workspace_size(int, int, int, int, int, attnfuse_rope_mode,
                                            size_t* bytes) {
  if (bytes) *bytes = 0;
  return ATTNFUSE_ERR_UNSUPPORTED;
}
attnfuse_status attnfuse_bwd(const void*, const int64_t*, const void*, const int64_t*,
                             const void*, const int64_t*, const void*, const int64_t*,
                             const float*, const void*, const int64_t*, void*, const int64_t*,
                             void*, const int64_t*, void*, const int64_t*, int, int, int, int,
                             int, float, float, attnfuse_rope_mode, const attnfuse_variant*,
                             void*, size_t, cudaStream_t) {
  return ATTNFUSE_ERR_UNSUPPORTED;
}
}
