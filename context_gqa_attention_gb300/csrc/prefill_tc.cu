// Tensor-core (tcgen05) partial attention -- filled in by the sm_103a kernel.
#include "common.cuh"

bool cp_prefill_tc_supported(const cp_prefill_args&) { return false; }
cudaError_t cp_launch_prefill_tc(const cp_prefill_args&, float, cudaStream_t) {
  return cudaErrorNotSupported;
}
