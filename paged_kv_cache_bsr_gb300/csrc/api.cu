// api.cu -- the extern "C" run entry points declared in include/pkv_bsr.h.
//
// Each call checks its arguments on the host, fills the kernel argument block
// from the plan's fixed tables, and enqueues fixed-grid kernels on the
// caller's stream.  Nothing here allocates, synchronises (except
// pkv_get_device_error) or depends on the batch contents, which live in the
// device workspace; so a sequence of run calls can be captured in a CUDA graph
// and replayed after plan_run has written a new plan into the same workspace.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "pkv_bsr.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_plan.h"

namespace pkv {

cudaError_t ensure_smem_limit_ptr(const void* kern, int bytes) {
  struct Entry {
    const void* kern;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : done)
    if (x.kern == kern && x.dev == dev && x.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back({kern, dev, bytes});
  return e;
}

}  // namespace pkv

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_device(const pkv_plan* plan) {
  if (plan->device < 0) return PKV_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return cur == plan->device ? PKV_OK : PKV_ERR_INVALID_ARG;
}

// Offset of the table image the next run reads (pipelined plans alternate two).
size_t table_off(const pkv_plan* plan) { return (plan->pipelined && plan->cur) ? plan->L.alt : 0; }

template <typename Args>
void fill_tables(Args& a, const pkv_plan* plan, void* dev_ws) {
  auto* base = static_cast<uint8_t*>(dev_ws);
  auto* tb = base + table_off(plan);
  a.hdr = reinterpret_cast<const pkv::PlanHeader*>(tb + plan->L.header);
  a.worker_ptr = reinterpret_cast<const int32_t*>(tb + plan->L.worker_ptr);
  a.part_o = reinterpret_cast<float*>(base + plan->L.part_o);
  a.part_lse = reinterpret_cast<float*>(base + plan->L.part_lse);
  a.err = reinterpret_cast<int32_t*>(tb + plan->L.header + offsetof(pkv::PlanHeader, error));
}

// Pipelined plans: the run waits for its table image's copy, and marks the image
// free again once its kernels have finished.
cudaError_t wait_tables(const pkv_plan* plan, cudaStream_t s) {
  return plan->pipelined ? cudaStreamWaitEvent(s, plan->copy_ev[plan->cur], 0) : cudaSuccess;
}
cudaError_t release_tables(const pkv_plan* plan, cudaStream_t s) {
  if (!plan->pipelined) return cudaSuccess;
  const_cast<pkv_plan*>(plan)->used[plan->cur] = true;
  return cudaEventRecord(plan->free_ev[plan->cur], s);
}

pkv::DecodeArgs decode_args(const pkv_plan* plan, void* dev_ws, const void* q, const void* kv_data,
                            const int32_t* kv_indices_d, const int32_t* kv_indptr_d, void* o, float* lse) {
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  pkv::DecodeArgs a{};
  fill_tables(a, plan, dev_ws);
  auto* tb = static_cast<uint8_t*>(dev_ws) + table_off(plan);
  a.segs = reinterpret_cast<const pkv::DecodeSeg*>(tb + plan->L.segs);
  a.merge = reinterpret_cast<const pkv::MergeItem*>(tb + plan->L.merge);
  a.q = q;
  a.kv = kv_data;
  a.kv_indices = kv_indices_d;
  a.kv_indptr = kv_indptr_d;
  a.o = o;
  a.lse = lse;
  a.num_qo_heads = p.num_qo_heads;
  a.num_kv_heads = p.num_kv_heads;
  a.page_size = p.page_size;
  a.q_scale = cap ? p.sm_scale : p.sm_scale * pkv::kLog2e;
  a.cap = cap ? p.logits_cap : 0.f;
  return a;
}

pkv::PrefillArgs prefill_args(const pkv_plan* plan, void* dev_ws, const void* q, const void* kv_data,
                              const int32_t* kv_indices_d, const uint8_t* mask, size_t mask_bytes, void* o,
                              float* lse) {
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  pkv::PrefillArgs a{};
  fill_tables(a, plan, dev_ws);
  auto* tb = static_cast<uint8_t*>(dev_ws) + table_off(plan);
  a.tiles = reinterpret_cast<const pkv::PrefillTile*>(tb + plan->L.segs);
  a.merge = reinterpret_cast<const pkv::PrefillMerge*>(tb + plan->L.merge);
  a.q = q;
  a.kv = kv_data;
  a.kv_indices = kv_indices_d;
  a.o = o;
  a.lse = lse;
  a.num_qo_heads = p.num_qo_heads;
  a.num_kv_heads = p.num_kv_heads;
  a.page_size = p.page_size;
  a.causal = p.causal;
  a.sm_scale = p.sm_scale;
  a.cap = cap ? p.logits_cap : 0.f;
  a.mask = reinterpret_cast<const uint32_t*>(mask);
  a.mask_words = mask ? static_cast<int64_t>(mask_bytes / 4) : 0;
  return a;
}

pkv_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  cudaGetLastError();
  return e == cudaErrorInvalidValue ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
}

// The prefill kernel and its merge over a plan's prefill tables (a prefill plan,
// or a decode plan whose work runs on the tensor cores); a packed plan's copy of
// small pages (`pack`) is made first, inside the timed span.
cudaError_t launch_prefill_tables(const pkv_plan* plan, const pkv::PrefillArgs& a, cudaStream_t s,
                                  const pkv::PackArgs* pack = nullptr) {
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  cudaError_t e = wait_tables(plan, s);
  if (plan->time_start && e == cudaSuccess) cudaEventRecord(plan->time_start, s);
  if (pack && e == cudaSuccess) e = pkv::launch_pack_pages(*pack, p.head_dim, plan->num_sms * 8, s);
  if (e == cudaSuccess)
    e = pkv::launch_prefill(a, p.head_dim, plan->group, p.dtype, cap, plan->grid_ctas, plan->total_q,
                            plan->packed ? plan->max_packed : plan->num_pages, s);
  if (plan->time_stop && e == cudaSuccess) cudaEventRecord(plan->time_stop, s);
  if (e == cudaSuccess) e = pkv::launch_prefill_merge(a, p.head_dim, plan->group, p.dtype, plan->merge_grid, s);
  if (e == cudaSuccess) e = release_tables(plan, s);
  return e;
}

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_BAD_INDEX: return "bad index array";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace too small or limits exceeded";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

int pkv_version(void) { return 100; }

pkv_status pkv_batch_decode_paged(const pkv_plan* plan, const void* q, const void* kv_data,
                                  const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                  const int32_t* kv_last_page_len_d, void* o, float* lse, void* dev_ws,
                                  void* stream) {
  if (!plan || plan->kind != PKV_PLAN_DECODE || !plan->planned) return PKV_ERR_INVALID_ARG;
  if (!q || !kv_data || !kv_indices_d || !kv_indptr_d || !kv_last_page_len_d || !o || !dev_ws)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_data, 16) || !aligned(o, 16) || !aligned(dev_ws, 256) ||
      !aligned(kv_indices_d, 4) || !aligned(kv_indptr_d, 4) || (lse && !aligned(lse, 4)))
    return PKV_ERR_INVALID_ARG;
  pkv_status st = check_device(plan);
  if (st != PKV_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (plan->exec_prefill)  // one query row per request on the tensor cores
    return launch_status(launch_prefill_tables(
        plan, prefill_args(plan, dev_ws, q, kv_data, kv_indices_d, nullptr, 0, o, lse), s));
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  const pkv::DecodeArgs a = decode_args(plan, dev_ws, q, kv_data, kv_indices_d, kv_indptr_d, o, lse);
  cudaError_t e = wait_tables(plan, s);
  if (plan->time_start && e == cudaSuccess) cudaEventRecord(plan->time_start, s);
  if (e == cudaSuccess)
    e = pkv::launch_decode(a, p.head_dim, plan->group, p.dtype, cap, plan->grid_ctas, plan->num_pages, s);
  if (plan->time_stop && e == cudaSuccess) cudaEventRecord(plan->time_stop, s);
  if (e == cudaSuccess) e = pkv::launch_decode_merge(a, p.head_dim, plan->group, p.dtype, plan->merge_grid, s);
  if (e == cudaSuccess) e = release_tables(plan, s);
  return launch_status(e);
}

static pkv_status prefill_run(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d, const void* kv_data,
                              const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                              const int32_t* kv_last_page_len_d, const uint8_t* mask, size_t mask_bytes, void* o,
                              float* lse, void* dev_ws, void* stream) {
  if (!plan || plan->kind != PKV_PLAN_PREFILL || !plan->planned) return PKV_ERR_INVALID_ARG;
  if (mask) {
    // whole 32-bit words covering every request's [qo_len, kv_len] block
    if (!aligned(mask, 4) || mask_bytes / 4 < static_cast<size_t>((plan->mask_bits + 31) / 32))
      return PKV_ERR_INVALID_ARG;
  }
  if (!q || !qo_indptr_d || !kv_data || !kv_indices_d || !kv_indptr_d || !kv_last_page_len_d || !o || !dev_ws)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_data, 16) || !aligned(o, 16) || !aligned(dev_ws, 256) ||
      !aligned(kv_indices_d, 4) || (lse && !aligned(lse, 4)))
    return PKV_ERR_INVALID_ARG;
  pkv_status st = check_device(plan);
  if (st != PKV_OK) return st;
  pkv::PrefillArgs a = prefill_args(plan, dev_ws, q, kv_data, kv_indices_d, mask, mask_bytes, o, lse);
  if (!plan->packed) return launch_status(launch_prefill_tables(plan, a, static_cast<cudaStream_t>(stream)));
  // Pages of fewer than 8 rows: the kernel reads the packed copy, in 16-row pages
  // whose ids are the plan's own table.
  auto* base = static_cast<uint8_t*>(dev_ws);
  auto* tb = base + table_off(plan);
  pkv::PackArgs pk{};
  pk.kv = kv_data;
  pk.kv_indices = kv_indices_d;
  pk.src = reinterpret_cast<const pkv::PackedSrc*>(tb + plan->L.pk_src);
  pk.hdr = a.hdr;
  pk.packed = base + plan->L.pk_kv;
  pk.err = a.err;
  pk.num_kv_heads = plan->p.num_kv_heads;
  pk.page_size = plan->p.page_size;
  pk.num_pages = plan->num_pages;
  a.kv = pk.packed;
  a.kv_indices = reinterpret_cast<const int32_t*>(tb + plan->L.pk_ids);
  a.page_size = 16;
  return launch_status(launch_prefill_tables(plan, a, static_cast<cudaStream_t>(stream), &pk));
}

pkv_status pkv_batch_prefill_paged(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                   const void* kv_data, const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                   const int32_t* kv_last_page_len_d, void* o, float* lse, void* dev_ws,
                                   void* stream) {
  return prefill_run(plan, q, qo_indptr_d, kv_data, kv_indices_d, kv_indptr_d, kv_last_page_len_d, nullptr, 0, o, lse,
                     dev_ws, stream);
}

pkv_status pkv_batch_prefill_paged_masked(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                          const void* kv_data, const int32_t* kv_indices_d,
                                          const int32_t* kv_indptr_d, const int32_t* kv_last_page_len_d,
                                          const uint8_t* packed_mask_d, size_t mask_bytes, void* o, float* lse,
                                          void* dev_ws, void* stream) {
  if (!packed_mask_d) return PKV_ERR_INVALID_ARG;
  return prefill_run(plan, q, qo_indptr_d, kv_data, kv_indices_d, kv_indptr_d, kv_last_page_len_d, packed_mask_d,
                     mask_bytes, o, lse, dev_ws, stream);
}

pkv_status pkv_batch_mixed_paged(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                 const void* kv_data, const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                 const int32_t* kv_last_page_len_d, void* o, float* lse, void* dev_ws,
                                 void* stream) {
  if (!plan || plan->kind != PKV_PLAN_MIXED || !plan->planned) return PKV_ERR_INVALID_ARG;
  if (!q || !qo_indptr_d || !kv_data || !kv_indices_d || !kv_indptr_d || !kv_last_page_len_d || !o || !dev_ws)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_data, 16) || !aligned(o, 16) || !aligned(dev_ws, 256) ||
      !aligned(kv_indices_d, 4) || !aligned(kv_indptr_d, 4) || (lse && !aligned(lse, 4)))
    return PKV_ERR_INVALID_ARG;
  pkv_status st = check_device(plan);
  if (st != PKV_OK) return st;
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  auto* base = static_cast<uint8_t*>(dev_ws);
  const pkv_plan* dp = plan->sub_dec;
  const pkv_plan* pp = plan->sub_pre;
  // Decode segments carry their row of q / o / lse, so both halves read and
  // write the caller's tensors in place.
  const pkv::DecodeArgs da =
      decode_args(dp, base + plan->dec_dev_off, q, kv_data, kv_indices_d, kv_indptr_d, o, lse);
  const pkv::PrefillArgs pa = prefill_args(pp, base + plan->pre_dev_off, q, kv_data, kv_indices_d, nullptr, 0, o, lse);
  auto s = static_cast<cudaStream_t>(stream);
  // One persistent launch serves both halves (the CTA split is in the decode
  // tables); then one launch merges both halves' split sequences.
  cudaError_t e = cudaSuccess;
  if (plan->time_start) cudaEventRecord(plan->time_start, s);
  e = pkv::launch_mixed(pa, da, p.head_dim, plan->group, p.dtype, cap, plan->grid_ctas, pp->total_q, pp->num_pages, s);
  if (plan->time_stop && e == cudaSuccess) cudaEventRecord(plan->time_stop, s);
  if (e == cudaSuccess)
    e = pkv::launch_mixed_merge(pa, da, plan->group, p.dtype, std::max(pp->merge_grid, dp->merge_grid), s);
  return launch_status(e);
}

pkv_status pkv_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o_out,
                           float* lse_out, int64_t n_rows, int num_heads, int head_dim, int dtype, void* stream) {
  if (n_rows < 0 || num_heads <= 0 || head_dim <= 0) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
  if (n_rows == 0) return PKV_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out) return PKV_ERR_INVALID_ARG;
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o_out, 16) || !aligned(lse_a, 4) ||
      !aligned(lse_b, 4) || (lse_out && !aligned(lse_out, 4)))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e = pkv::launch_merge_state(o_a, lse_a, o_b, lse_b, o_out, lse_out, n_rows * num_heads, head_dim,
                                          dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status pkv_merge_states(const void* o_states, const float* lse_states, int num_states, int64_t state_stride_rows,
                            void* o_out, float* lse_out, int64_t n_rows, int num_heads, int head_dim, int dtype,
                            void* stream) {
  if (n_rows < 0 || num_heads <= 0 || head_dim <= 0 || num_states < 1 || state_stride_rows < n_rows)
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
  if (n_rows == 0) return PKV_OK;
  if (!o_states || !lse_states || !o_out) return PKV_ERR_INVALID_ARG;
  if (!aligned(o_states, 16) || !aligned(o_out, 16) || !aligned(lse_states, 4) || (lse_out && !aligned(lse_out, 4)))
    return PKV_ERR_INVALID_ARG;
  // Flat (row, head) indices and state offsets stay within int64.
  if (state_stride_rows > INT64_MAX / num_heads / num_states) return PKV_ERR_INVALID_ARG;
  cudaError_t e = pkv::launch_merge_states(o_states, lse_states, num_states, state_stride_rows * num_heads, o_out,
                                           lse_out, n_rows * num_heads, head_dim, dtype,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status pkv_plan_set_timing_events(pkv_plan* plan, void* start, void* stop) {
  if (!plan || (!start) != (!stop)) return PKV_ERR_INVALID_ARG;
  plan->time_start = static_cast<cudaEvent_t>(start);
  plan->time_stop = static_cast<cudaEvent_t>(stop);
  return PKV_OK;
}

pkv_status pkv_get_device_error(const pkv_plan* plan, void* dev_ws, int* code, int clear, void* stream) {
  if (!plan || !dev_ws || !code) return PKV_ERR_INVALID_ARG;
  if (plan->kind == PKV_PLAN_MIXED) {  // the OR of both halves' words
    int cd = 0, cp = 0;
    auto* base = static_cast<uint8_t*>(dev_ws);
    pkv_status st = pkv_get_device_error(plan->sub_dec, base + plan->dec_dev_off, &cd, clear, stream);
    if (st == PKV_OK) st = pkv_get_device_error(plan->sub_pre, base + plan->pre_dev_off, &cp, clear, stream);
    *code = cd | cp;
    return st;
  }
  auto s = static_cast<cudaStream_t>(stream);
  *code = 0;
  // Both table images of a pipelined plan carry an error word.
  for (int r = 0; r < (plan->pipelined ? 2 : 1); ++r) {
    auto* word = static_cast<uint8_t*>(dev_ws) + (r ? plan->L.alt : 0) + plan->L.header +
                 offsetof(pkv::PlanHeader, error);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    *code |= v;
    if (clear && v) {
      if (cudaMemsetAsync(word, 0, sizeof(int32_t), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
      }
    }
  }
  return PKV_OK;
}

}  // extern "C"
