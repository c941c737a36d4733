// mixed.cu -- host launch of the one-launch mixed prefill + decode kernel
// (mixed_kernel.cuh) and its instances for pages of 8 rows or more.
#include "mixed_kernel.cuh"

namespace pkv {
namespace mixed_impl {

template cudaError_t launch_mixed_kernel<__nv_bfloat16, false>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                               const CUtensorMap&, const CUtensorMap&, cudaStream_t);
template cudaError_t launch_mixed_kernel<__half, false>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                        const CUtensorMap&, const CUtensorMap&, cudaStream_t);

// Both halves' merges in one grid: warps take the decode pairs (item, head of
// the group) first, then the prefill rows (item, packed row).
template <int G, typename T>
__global__ void __launch_bounds__(kMergeThreads) mixed_merge_kernel(const __grid_constant__ PrefillArgs pa,
                                                                    const __grid_constant__ DecodeArgs da) {
  // A programmatic dependent of the mixed kernel: wait until that grid has
  // finished and its partial states are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int warp_id = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * (kMergeThreads / 32);
  const int dec_pairs = da.hdr->num_merge * G;
  const int pairs = dec_pairs + pa.hdr->num_merge * prefill_impl::kWR;
  for (int pair = warp_id; pair < pairs; pair += n_warps) {
    if (pair < dec_pairs)
      decode_impl::decode_merge_pair<128, G, T>(da, pair, lane);
    else
      prefill_impl::prefill_merge_row<T>(pa, pair - dec_pairs, lane, G);
  }
}

}  // namespace mixed_impl

cudaError_t launch_mixed_merge(const PrefillArgs& pa, const DecodeArgs& da, int group, int dtype, int grid,
                               cudaStream_t stream) {
  void (*kern)(PrefillArgs, DecodeArgs) = nullptr;
#define PKV_MM_CASE(GG)                                                                                   \
  if (group == GG)                                                                                        \
    kern = dtype == PKV_BF16 ? mixed_impl::mixed_merge_kernel<GG, __nv_bfloat16>                          \
                             : (dtype == PKV_F16 ? mixed_impl::mixed_merge_kernel<GG, __half> : nullptr);
  PKV_MM_CASE(1) PKV_MM_CASE(2) PKV_MM_CASE(4) PKV_MM_CASE(8)
#undef PKV_MM_CASE
  if (!kern) return cudaErrorInvalidValue;
  return launch_dependent(kern, grid, kMergeThreads, 0, stream, pa, da);
}

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
