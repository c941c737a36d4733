// prefill_masked.cu -- the prefill kernel instances that apply a caller's packed custom mask on
// top of the causal limit, for pages of 8 rows or more
// (the kernel is in prefill_kernel.cuh; each instance set is its own translation
// unit so they build in parallel).
#include "prefill_kernel.cuh"

namespace pkv {
namespace prefill_impl {

template cudaError_t launch_kernel<__nv_bfloat16, true, false>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                              const CUtensorMap&, cudaStream_t);
template cudaError_t launch_kernel<__half, true, false>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                       const CUtensorMap&, cudaStream_t);

}  // namespace prefill_impl
}  // namespace pkv
