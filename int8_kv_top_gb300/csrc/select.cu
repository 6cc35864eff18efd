// qsa_select (placeholder until the selection kernels land).
#include "common.cuh"
namespace qsa {
size_t select_workspace_bytes(int, int, int, Params) { return 0; }
cudaError_t launch_select(const __half*, const int8_t*, const __half*, int, int, int, int32_t*, void*, Params, int*,
                          cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace qsa
