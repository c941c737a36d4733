// decode.cu -- batch decode over a paged KV cache: the decode kernel instances
// that read pages with bulk copies (the kernel, one CTA of kDecodeWarps
// independent workers per SM, is in decode_kernel.cuh), the n-way merge of split
// sequences, and their launches.
#include <cuda_runtime.h>
#include <math.h>

#include "decode_kernel.cuh"

namespace pkv {
namespace decode_impl {

template cudaError_t launch_decode_kernel<__nv_bfloat16, false>(const DecodeArgs&, int, int, bool, int, cudaStream_t);
template cudaError_t launch_decode_kernel<__half, false>(const DecodeArgs&, int, int, bool, int, cudaStream_t);

}  // namespace decode_impl

namespace {

using namespace decode_impl;

// n-way merge of the partial states of split (request, kv head) sequences
// (decode_merge_pair in decode_kernel.cuh): one warp per (item, head of the group).
template <int D, int G, typename T>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const __grid_constant__ DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp_id = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * (kMergeThreads / 32);
  // Launched as a programmatic dependent of the decode kernel: wait until that
  // grid has finished and its partial states are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int pairs = a.hdr->num_merge * G;
  for (int pair = warp_id; pair < pairs; pair += n_warps) decode_merge_pair<D, G, T>(a, pair, lane);
}

template <typename T>
cudaError_t dispatch_merge(const DecodeArgs& a, int D, int G, int grid, cudaStream_t s) {
// The merge kernel is a programmatic dependent of the decode kernel just
// before it on the stream: it is launched as the decode CTAs exit (the decode
// kernel triggers no earlier, so waiting merge CTAs never hold SMs that work on
// another stream needs), and it waits (griddepcontrol.wait) for the whole
// grid before reading partial states.
#define PKV_MERGE_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_dependent(decode_merge_kernel<DD, GG, T>, grid, kMergeThreads, 0, s, a);
  PKV_MERGE_CASE(128, 1) PKV_MERGE_CASE(128, 2) PKV_MERGE_CASE(128, 4) PKV_MERGE_CASE(128, 8)
  PKV_MERGE_CASE(64, 1) PKV_MERGE_CASE(64, 2) PKV_MERGE_CASE(64, 4) PKV_MERGE_CASE(64, 8)
#undef PKV_MERGE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_supported(int head_dim, int group, int dtype) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == PKV_F16 || dtype == PKV_BF16);
}

cudaError_t launch_decode(const DecodeArgs& a0, int head_dim, int group, int dtype, bool cap, int grid,
                          int64_t num_pages, cudaStream_t stream) {
  if (!decode_supported(head_dim, group, dtype)) return cudaErrorInvalidValue;
  if (a0.page_size > kDecodeGatherMaxRows) {
    return dtype == PKV_BF16 ? launch_decode_kernel<__nv_bfloat16, false>(a0, head_dim, group, cap, grid, stream)
                             : launch_decode_kernel<__half, false>(a0, head_dim, group, cap, grid, stream);
  }
  DecodeArgs a = a0;
  cudaError_t e = set_kv_rows_map(a, head_dim, dtype, num_pages);
  if (e != cudaSuccess) return e;
  return dtype == PKV_BF16 ? launch_decode_kernel<__nv_bfloat16, true>(a, head_dim, group, cap, grid, stream)
                           : launch_decode_kernel<__half, true>(a, head_dim, group, cap, grid, stream);
}

cudaError_t launch_decode_merge(const DecodeArgs& a, int head_dim, int group, int dtype, int grid,
                                cudaStream_t stream) {
  if (dtype == PKV_BF16) return dispatch_merge<__nv_bfloat16>(a, head_dim, group, grid, stream);
  if (dtype == PKV_F16) return dispatch_merge<__half>(a, head_dim, group, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
