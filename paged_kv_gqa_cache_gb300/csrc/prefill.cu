// Causal chunked-prefill attention on the tcgen05 tensor cores (sm_103a).
#include "pa_device.cuh"

namespace pa {

cudaError_t launch_prefill(const PrefillParams &, const CUtensorMap &, const CUtensorMap &,
                           const CUtensorMap &, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
