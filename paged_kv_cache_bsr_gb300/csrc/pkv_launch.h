// pkv_launch.h -- host-side launch interface between the C ABI layer and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Arguments of the decode and decode-merge kernels.
struct DecodeArgs {
  const void* q;               // [batch, Hq, D]
  const void* kv;              // [num_pages, 2, Hkv, P, D]
  const int32_t* kv_indices;   // page table (BSR column indices)
  const int32_t* kv_indptr;    // checked against the plan
  void* o;                     // [batch, Hq, D]
  float* lse;                  // [batch, Hq] or nullptr
  const PlanHeader* hdr;       // plan tables in the device workspace
  const int32_t* worker_ptr;
  const DecodeSeg* segs;
  const MergeItem* merge;
  float* part_o;               // [slots, G, D]
  float* part_lse;             // [slots, G]
  int32_t* err;                // &hdr->error
  int num_qo_heads;
  int num_kv_heads;
  int page_size;
  float q_scale;               // multiplies q: sm_scale * log2(e) without a cap, sm_scale with one
  float cap;                   // logits cap (> 0 only in the capped instantiation)
  // One-row pages (the gather instances): kv_data as a 2-D tensor of
  // head_dim-element rows, row ((page * 2 + K|V) * Hkv + kv head) * page_size +
  // slot, with kv_rows_n rows; set by the launch, unused otherwise.
  int32_t kv_rows_n;
  CUtensorMap kv_rows;
};

// Raise a kernel's dynamic shared-memory limit once per (kernel, device): the
// first launch on a device does it, so later launches (e.g. inside CUDA-graph
// capture) make no attribute call.
cudaError_t ensure_smem_limit_ptr(const void* kern, int bytes);
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, int bytes) {
  return ensure_smem_limit_ptr(reinterpret_cast<const void*>(kern), bytes);
}

// Launch a kernel as a programmatic dependent of the kernel before it on the
// stream.  No kernel of this library triggers its dependents early, so the new
// grid's CTAs are placed as the previous grid's CTAs exit, which hides the gap
// between the two launches.  The launched kernel executes griddepcontrol.wait
// before its first global-memory access; the wait returns once the previous
// grid has finished and its writes are visible.  Every thread waits before it
// can return, so no grid launched this way finishes before the grid it depends
// on, and a chain of such launches stays ordered after every earlier kernel on
// the stream.  After a copy, a memset or an event on the stream it is an
// ordinary launch.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(Params...), int grid, int block, int smem, cudaStream_t s,
                                   const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Warps per decode CTA; each warp streams its own pages (one CTA per SM).
constexpr int kDecodeWarps = 8;
// Shared memory each decode warp uses for its ring of page tiles.
constexpr int kDecodeWarpSmem = 24 * 1024;
constexpr int kDecodeTileRows = 16;
// Pages of one row (column-vector BSR) reach decode tiles as four-row tensor
// gathers; pages of two rows or more as one bulk copy per page (measured: one-row
// pages 4.31 vs 3.92 TB/s, two-row pages 4.47 vs 4.86 TB/s with gathers vs copies).
constexpr int kDecodeGatherMaxRows = 1;
constexpr int kMergeThreads = 256;

// Launch the decode kernel for (head_dim, group, dtype, cap) over a pool of
// num_pages pages; returns cudaErrorInvalidValue for a combination that was not
// built.
cudaError_t launch_decode(const DecodeArgs& a, int head_dim, int group, int dtype, bool cap,
                          int grid, int64_t num_pages, cudaStream_t stream);
// Fill a.kv_rows / a.kv_rows_n for the gather instances: kv_data as rows of
// head_dim elements, one-row boxes.
cudaError_t set_kv_rows_map(DecodeArgs& a, int head_dim, int dtype, int64_t num_pages);
// Launch the n-way merge of split decode sequences (fixed grid).
cudaError_t launch_decode_merge(const DecodeArgs& a, int head_dim, int group, int dtype, int grid,
                                cudaStream_t stream);
// Elementwise two-state merge_state.
cudaError_t launch_merge_state(const void* o_a, const float* lse_a, const void* o_b,
                               const float* lse_b, void* o_out, float* lse_out, int64_t rows,
                               int head_dim, int dtype, cudaStream_t stream);

// n-state merge_state: state k of flat row r at rows k * stride + r of o_in / lse_in.
cudaError_t launch_merge_states(const void* o_in, const float* lse_in, int n_states, int64_t stride, void* o_out,
                                float* lse_out, int64_t rows, int head_dim, int dtype, cudaStream_t stream);

bool decode_supported(int head_dim, int group, int dtype);

// Prefill work tile: kPrefillRows packed query rows (two 128-row UMMA tiles),
// visited kPrefillKeys keys at a time.
constexpr int kPrefillRows = 256;
constexpr int kPrefillKeys = 128;

bool prefill_supported(int head_dim, int group, int dtype, int page_size);

// Arguments of the prefill and prefill-merge kernels (tensor maps for q and
// kv_data are built at launch and passed separately).
struct PrefillArgs {
  const void* q;               // [total_q, Hq, D]
  const void* kv;              // [num_pages, 2, Hkv, P, D]
  const int32_t* kv_indices;
  void* o;                     // [total_q, Hq, D]
  float* lse;                  // [total_q, Hq] or nullptr
  const PlanHeader* hdr;
  const int32_t* worker_ptr;
  const PrefillTile* tiles;
  const PrefillMerge* merge;
  float* part_o;               // [slots, kPrefillRows, D]
  float* part_lse;             // [slots, kPrefillRows]
  int32_t* err;
  int num_qo_heads;
  int num_kv_heads;
  int page_size;
  int causal;
  float sm_scale;
  float cap;                   // > 0 only in the capped instantiation
  const uint32_t* mask;        // packed custom mask (bit k of word w = bit 32 w + k), or nullptr
  int64_t mask_words;          // 32-bit words of the mask buffer
};

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, int group, int dtype, bool cap, int grid,
                           int64_t total_q, int64_t num_pages, cudaStream_t stream);

// Packed prefill plans: copy the requests' K/V rows from pages of fewer than 8
// rows into 16-row pages of the workspace, page p from the keys src[p] names.
struct PackArgs {
  const void* kv;              // [num_pages, 2, Hkv, P, D], the caller's pool
  const int32_t* kv_indices;
  const PackedSrc* src;        // [num_packed]
  const PlanHeader* hdr;       // num_packed
  void* packed;                // [max_packed, 2, Hkv, 16, D]
  int32_t* err;
  int num_kv_heads;
  int page_size;               // 1, 2 or 4
  int64_t num_pages;
};
cudaError_t launch_pack_pages(const PackArgs& a, int head_dim, int grid, cudaStream_t stream);
cudaError_t launch_prefill_merge(const PrefillArgs& a, int head_dim, int group, int dtype, int grid,
                                 cudaStream_t stream);

// Launch the mixed prefill + decode kernel on `grid` CTAs: the CTAs below the
// decode tables' cta_offset run the prefill half, the rest the decode half
// (head_dim 128 only).  Both halves' merges follow in one launch (launch_mixed_merge).
cudaError_t launch_mixed(const PrefillArgs& pa, const DecodeArgs& da, int head_dim, int group, int dtype, bool cap,
                         int grid, int64_t total_q, int64_t num_pages, cudaStream_t stream);
// The merges of both halves of a mixed batch (split decode sequences and split
// prefill tiles) in one launch, a programmatic dependent of the mixed kernel.
cudaError_t launch_mixed_merge(const PrefillArgs& pa, const DecodeArgs& da, int group, int dtype, int grid,
                               cudaStream_t stream);

}  // namespace pkv
