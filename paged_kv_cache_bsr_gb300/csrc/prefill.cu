// prefill.cu -- causal ragged batch prefill over a paged KV cache: host launch
// code, the merge of split key ranges, and the kernel instances for pages of 8
// rows or more without a custom mask (the kernel itself is in
// prefill_kernel.cuh).
#include "prefill_kernel.cuh"

namespace pkv {
namespace prefill_impl {

template cudaError_t launch_kernel<__nv_bfloat16, false, false>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                               const CUtensorMap&, cudaStream_t);
template cudaError_t launch_kernel<__half, false, false>(const PrefillArgs&, int, bool, int, const CUtensorMap&,
                                                        const CUtensorMap&, cudaStream_t);

}  // namespace prefill_impl

using namespace prefill_impl;

namespace {

// Rows of query tiles whose key range the plan split (prefill_merge_row in
// prefill_kernel.cuh): one warp per packed row.
template <typename T>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const __grid_constant__ PrefillArgs a) {
  // Launched as a programmatic dependent of the kernel before it: wait until that
  // grid has finished and its partial states are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int warp_id = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * 8;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int pairs = a.hdr->num_merge * kWR;
  for (int pair = warp_id; pair < pairs; pair += n_warps) prefill_merge_row<T>(a, pair, lane, G);
}

// Packed copy of small pages: one CTA of 256 threads per packed page at a time.
// Thread t owns row t / 16 of the page and its 16-byte piece t % 16 (16 pieces to
// a 256-byte row: head_dim 128, 16-bit values) in every (K|V, head) block hs, so
// it looks its source page up once and then issues the 2 Hkv loads of its piece
// back to back.  The copy's layout [2, Hkv, 16, D] puts piece t of block hs at
// hs * 256 + t; rows past the page's keys are zeros.
constexpr int kPackThreads = 256;
__global__ void __launch_bounds__(kPackThreads) pack_pages_kernel(const __grid_constant__ PackArgs a) {
  constexpr int kPieces = kD * 2 / 16;  // 16-byte pieces per row
  static_assert(kPackThreads == 16 * kPieces, "a thread per (row, piece) of a 16-row page");
  // Launched as a programmatic dependent of the kernel before it on the stream:
  // nothing global is touched before that grid has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nblk = 2 * a.num_kv_heads;   // (K|V, head) blocks of a page
  const int n_packed = a.hdr->num_packed;
  const int lp = __ffs(a.page_size) - 1;  // P is a power of two here
  const int64_t row_elems = static_cast<int64_t>(a.page_size) * kD;  // one (page, K|V, head)
  const int t = threadIdx.x, r = t / kPieces, piece = t % kPieces;
  const uint4* kv = static_cast<const uint4*>(a.kv);
  uint4* out = static_cast<uint4*>(a.packed);
  for (int p = blockIdx.x; p < n_packed; p += gridDim.x) {
    const PackedSrc sp = a.src[p];
    int64_t e0 = -1;  // element offset of this thread's piece in block 0 of its source page
    if (r < sp.ntok) {
      const int u = sp.tok0 + r;
      const int page = __ldg(a.kv_indices + (u >> lp));
      if (page >= 0 && page < a.num_pages)
        e0 = static_cast<int64_t>(page) * nblk * row_elems + static_cast<int64_t>(u & (a.page_size - 1)) * kD +
             piece * 8;
      else
        atomicOr(a.err, kErrPageIndex);
    }
    uint4* dst = out + static_cast<int64_t>(p) * nblk * kPackThreads + t;
#pragma unroll 16
    for (int hs = 0; hs < nblk; ++hs)
      dst[hs * kPackThreads] = e0 >= 0 ? ld_nc_v4(kv + (e0 + hs * row_elems) / 8) : make_uint4(0u, 0u, 0u, 0u);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool prefill_supported(int head_dim, int group, int dtype, int page_size) {
  return head_dim == kD && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == PKV_F16 || dtype == PKV_BF16) &&
         (page_size == 1 || page_size == 2 || page_size == 4 || page_size == 8 || page_size == 16 ||
          page_size == 32 || page_size == 64 || page_size == 128);
}

namespace prefill_impl {

cudaError_t make_tensor_maps(const PrefillArgs& a, int group, int dtype, int64_t total_q, int64_t num_pages,
                             CUtensorMap& tq, CUtensorMap& tkv) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t hq = a.num_qo_heads, hkv = a.num_kv_heads, P = a.page_size;
  {
    // q [total_q, Hq, D]: box = 64 columns x the G heads of a group x 128/G positions.
    cuuint64_t dims[3] = {kD, hq, static_cast<cuuint64_t>(total_q > 0 ? total_q : 1)};
    cuuint64_t strides[2] = {kD * 2, hq * kD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(kTM / group)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tq, dt, 3, const_cast<void*>(a.q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // kv_data [num_pages, 2, Hkv, P, D]: box = 64 columns x the P rows of one (page, K|V, head).
    cuuint64_t dims[5] = {kD, P, hkv, 2, static_cast<cuuint64_t>(num_pages > 0 ? num_pages : 1)};
    cuuint64_t strides[4] = {kD * 2, P * kD * 2, hkv * P * kD * 2, 2 * hkv * P * kD * 2};
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(P), 1, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (encode(&tkv, dt, 5, const_cast<void*>(a.kv), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace prefill_impl

cudaError_t set_kv_rows_map(DecodeArgs& a, int head_dim, int dtype, int64_t num_pages) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const int64_t rows = (num_pages > 0 ? num_pages : 1) * 2 * a.num_kv_heads * a.page_size;
  if (rows >= INT32_MAX) return cudaErrorInvalidValue;  // row coordinates are 32-bit
  const CUtensorMapDataType dt = dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(head_dim), 1};
  cuuint32_t es[2] = {1, 1};
  if (encode(&a.kv_rows, dt, 2, const_cast<void*>(a.kv), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  a.kv_rows_n = static_cast<int32_t>(rows);
  return cudaSuccess;
}

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, int group, int dtype, bool cap, int grid,
                           int64_t total_q, int64_t num_pages, cudaStream_t stream) {
  if (!prefill_supported(head_dim, group, dtype, a.page_size)) return cudaErrorInvalidValue;
  CUtensorMap tq, tkv;
  cudaError_t e = make_tensor_maps(a, group, dtype, total_q, num_pages, tq, tkv);
  if (e != cudaSuccess) return e;
  const bool masked = a.mask != nullptr, small = a.page_size < 8;
  using L = cudaError_t (*)(const PrefillArgs&, int, bool, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
  L fn;
  if (dtype == PKV_BF16)
    fn = masked ? (small ? launch_kernel<__nv_bfloat16, true, true> : launch_kernel<__nv_bfloat16, true, false>)
                : (small ? launch_kernel<__nv_bfloat16, false, true> : launch_kernel<__nv_bfloat16, false, false>);
  else
    fn = masked ? (small ? launch_kernel<__half, true, true> : launch_kernel<__half, true, false>)
                : (small ? launch_kernel<__half, false, true> : launch_kernel<__half, false, false>);
  // An ordinary launch: launched as a programmatic dependent (with a
  // griddepcontrol.wait at its top) the kernel ran 0.3-0.6 % slower on the ragged
  // causal batch, and in a prefill step the plan's table copy comes just before it.
  return fn(a, group, cap, grid, tq, tkv, stream);
}

cudaError_t launch_pack_pages(const PackArgs& a, int head_dim, int grid, cudaStream_t stream) {
  if (head_dim != kD || !(a.page_size == 1 || a.page_size == 2 || a.page_size == 4)) return cudaErrorInvalidValue;
  return launch_dependent(pack_pages_kernel, grid, kPackThreads, 0, stream, a);
}

cudaError_t launch_prefill_merge(const PrefillArgs& a, int head_dim, int group, int dtype, int grid,
                                 cudaStream_t stream) {
  if (head_dim != kD || group <= 0) return cudaErrorInvalidValue;
  // A programmatic dependent of the prefill (or mixed) kernel before it: its CTAs
  // start as that grid's CTAs leave, and wait for the whole grid before reading.
  if (dtype == PKV_BF16) return launch_dependent(prefill_merge_kernel<__nv_bfloat16>, grid, 256, 0, stream, a);
  if (dtype == PKV_F16) return launch_dependent(prefill_merge_kernel<__half>, grid, 256, 0, stream, a);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
