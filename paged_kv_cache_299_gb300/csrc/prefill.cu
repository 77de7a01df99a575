// Causal chunked-prefill attention over a paged prefix (tcgen05 version in progress).
#include "common.cuh"
#include "internal.h"

namespace pkv {

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  (void)a;
  (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace pkv
