// fm_bwd.cu — placeholder until the backward kernels land.
#include "fm_internal.h"
namespace fm {
size_t bwd_ws_bytes(const fm_problem& p) { return 256; }
cudaError_t launch_bwd(const fm_problem&, const void*, const void*, const void*, const void*, const float*,
                       const void*, const int32_t*, const int32_t*, const int32_t*, const int32_t*,
                       const int32_t*, const int32_t*, void*, void*, void*, void*, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}
}  // namespace fm
