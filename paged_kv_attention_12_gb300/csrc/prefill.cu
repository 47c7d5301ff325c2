// Paged prefill / mixed-batch attention (sm_103a).  Placeholder until the
// tcgen05 kernel lands: reports "not supported".
#include "common.cuh"
#include "kernels.h"

namespace pka {

cudaError_t launch_prefill(const PrefillArgs&, int, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pka
