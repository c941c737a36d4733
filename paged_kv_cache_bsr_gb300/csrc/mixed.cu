// mixed.cu -- host launch of the one-launch mixed prefill + decode kernel
// (mixed_kernel.cuh) and its instances for pages of 8 rows or more.
#include "mixed_kernel.cuh"

namespace pkv {
namespace mixed_impl {

template cudaError_t launch_mixed_kernel<__nv_bfloat16, false>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                               const CUtensorMap&, const CUtensorMap&, cudaStream_t);
template cudaError_t launch_mixed_kernel<__half, false>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                        const CUtensorMap&, const CUtensorMap&, cudaStream_t);

}  // namespace mixed_impl

cudaError_t launch_mixed(const PrefillArgs& pa, const DecodeArgs& da, int head_dim, int group, int dtype, bool cap,
                         int grid, int64_t total_q, int64_t num_pages, cudaStream_t stream) {
  if (!prefill_supported(head_dim, group, dtype, pa.page_size) || !decode_supported(head_dim, group, dtype))
    return cudaErrorInvalidValue;
  CUtensorMap tq, tkv;
  cudaError_t e = prefill_impl::make_tensor_maps(pa, group, dtype, total_q, num_pages, tq, tkv);
  if (e != cudaSuccess) return e;
  const bool small = pa.page_size < 8;
  using L = cudaError_t (*)(const PrefillArgs&, const DecodeArgs&, int, bool, int, const CUtensorMap&,
                            const CUtensorMap&, cudaStream_t);
  L fn;
  if (dtype == PKV_BF16)
    fn = small ? mixed_impl::launch_mixed_kernel<__nv_bfloat16, true> : mixed_impl::launch_mixed_kernel<__nv_bfloat16, false>;
  else
    fn = small ? mixed_impl::launch_mixed_kernel<__half, true> : mixed_impl::launch_mixed_kernel<__half, false>;
  return fn(pa, da, group, cap, grid, tq, tkv, stream);
}

}  // namespace pkv
