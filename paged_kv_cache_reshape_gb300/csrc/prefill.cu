// Varlen causal prefill on tcgen05 tensor cores (not built yet).
#include "step.h"

namespace pa {

cudaError_t prefill_configure(int, size_t* smem) {
  *smem = 0;
  return cudaErrorNotSupported;
}

cudaError_t launch_prefill(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const PrefillParams&,
                           int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
