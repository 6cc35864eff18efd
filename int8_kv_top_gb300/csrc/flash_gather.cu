// qsa_flash_prefill for selected tokens (placeholder until the gathered kernel lands).
#include "common.cuh"
namespace qsa {
cudaError_t launch_flash_gather(const FlashArgs&, int t_begin, int t_end, cudaStream_t) {
  return t_end > t_begin ? cudaErrorNotSupported : cudaSuccess;
}
}  // namespace qsa
