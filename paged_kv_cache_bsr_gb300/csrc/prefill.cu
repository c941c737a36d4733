// prefill.cu -- causal ragged batch prefill over a paged KV cache (tcgen05).
#include <cuda_runtime.h>

#include "pkv_bsr.h"
#include "pkv_launch.h"

namespace pkv {

bool prefill_supported(int, int, int, int) { return false; }

cudaError_t launch_prefill(const PrefillArgs&, int, int, int, bool, int, int64_t, int64_t, cudaStream_t) {
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_merge(const PrefillArgs&, int, int, int, int, cudaStream_t) {
  return cudaErrorInvalidValue;
}

}  // namespace pkv
