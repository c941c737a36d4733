// prefill_small.cu -- the prefill kernel instances for pages of 1, 2 or 4 rows (column-vector
// BSR), whose K/V rows are gathered with cp.async
// (the kernel is in prefill_kernel.cuh; each instance set is its own translation
// unit so they build in parallel).
#include "prefill_kernel.cuh"

namespace pkv {
namespace prefill_impl {

template cudaError_t launch_kernel<__nv_bfloat16, false, true>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                              const CUtensorMap&, cudaStream_t);
template cudaError_t launch_kernel<__half, false, true>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                       const CUtensorMap&, cudaStream_t);

}  // namespace prefill_impl
}  // namespace pkv
