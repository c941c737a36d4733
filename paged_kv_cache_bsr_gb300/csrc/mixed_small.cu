// mixed_small.cu -- the mixed prefill + decode kernel instances for pages of 1, 2
// or 4 rows (the prefill half gathers them with cp.async); the kernel is in
// mixed_kernel.cuh.
#include "mixed_kernel.cuh"

namespace pkv {
namespace mixed_impl {

template cudaError_t launch_mixed_kernel<__nv_bfloat16, true>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                              const CUtensorMap&, const CUtensorMap&, cudaStream_t);
template cudaError_t launch_mixed_kernel<__half, true>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                       const CUtensorMap&, const CUtensorMap&, cudaStream_t);

}  // namespace mixed_impl
}  // namespace pkv
