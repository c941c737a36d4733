// decode_gather.cu -- the decode kernel instances for one-row pages
// (column-vector BSR), whose tiles arrive as four-row tensor gathers (the kernel is in
// decode_kernel.cuh; each instance set is its own translation unit so they build
// in parallel).
#include "decode_kernel.cuh"

namespace pkv {
namespace decode_impl {

template cudaError_t launch_decode_kernel<__nv_bfloat16, true>(const DecodeArgs&, int, int, bool, int, cudaStream_t);
template cudaError_t launch_decode_kernel<__half, true>(const DecodeArgs&, int, int, bool, int, cudaStream_t);

}  // namespace decode_impl
}  // namespace pkv
