// noalloc.cu -- batch decode whose scratch memory is a static device array.
//
// pkv_batch_decode_paged needs a device workspace from the caller: the plan
// tables and the fp32 partial states of split sequences live there.  Some
// callers cannot provide one: plug-ins whose host framework owns every byte
// of device memory through its own allocator, services that run under a
// fixed device-memory budget, and code paths that must not pay the implicit
// device synchronisation a cudaMalloc can cause.
// pkv_batch_decode_paged_noalloc serves them: its scratch is the file-scope
// array below, which exists on every device that loads this library until
// the process exits, so the call itself allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_bsr.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_plan.h"

namespace {

// Size of the static scratch: plan tables plus fp32 partial states.  The
// Llama-3-8B-shaped batch of 64 requests needs about 5 MB of it on a GB300.
constexpr size_t kScratchBytes = size_t{8} << 20;

// Shared by every call on a device; holds the last call's tables and partials.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the symbol names a host-side stand-in, so kernels must receive the
// address that cudaGetSymbolAddress returns with the device current.
cudaError_t scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[device] = p;
  }
  *out = addr[device];
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" pkv_status pkv_batch_decode_paged_noalloc(const pkv_plan* plan, const void* host_tables,
                                                     size_t host_tables_bytes, const void* q, const void* kv_data,
                                                     const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                                     const int32_t* kv_last_page_len_d, void* o, float* lse,
                                                     void* stream) {
  if (!plan || plan->kind != PKV_PLAN_DECODE || !plan->planned || plan->device < 0 || plan->pipelined)
    return PKV_ERR_INVALID_ARG;
  if (!host_tables || host_tables_bytes < plan->used_bytes) return PKV_ERR_INVALID_ARG;
  if (!q || !kv_data || !kv_indices_d || !kv_indptr_d || !kv_last_page_len_d || !o) return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_data, 16) || !aligned(o, 16) || !aligned(kv_indices_d, 4) ||
      !aligned(kv_indptr_d, 4) || (lse && !aligned(lse, 4)))
    return PKV_ERR_INVALID_ARG;
  if (plan->L.total > kScratchBytes) return PKV_ERR_WORKSPACE;  // the plan's limits need more scratch
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (cur != plan->device) return PKV_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (scratch_address(cur, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  auto s = static_cast<cudaStream_t>(stream);
  // The tables carry a zeroed error word, so nothing left by an earlier call survives.
  if (cudaMemcpyAsync(scratch, host_tables, plan->used_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  const pkv_params& p = plan->p;
  const bool cap = p.logits_cap > 0.f;
  auto* base = static_cast<uint8_t*>(scratch);
  pkv::DecodeArgs a{};
  a.hdr = reinterpret_cast<const pkv::PlanHeader*>(base + plan->L.header);
  a.worker_ptr = reinterpret_cast<const int32_t*>(base + plan->L.worker_ptr);
  a.segs = reinterpret_cast<const pkv::DecodeSeg*>(base + plan->L.segs);
  a.merge = reinterpret_cast<const pkv::MergeItem*>(base + plan->L.merge);
  a.part_o = reinterpret_cast<float*>(base + plan->L.part_o);
  a.part_lse = reinterpret_cast<float*>(base + plan->L.part_lse);
  a.err = reinterpret_cast<int32_t*>(base + plan->L.header + offsetof(pkv::PlanHeader, error));
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
  cudaError_t e = pkv::launch_decode(a, p.head_dim, plan->group, p.dtype, cap, plan->grid_ctas, plan->num_pages, s);
  if (e == cudaSuccess) e = pkv::launch_decode_merge(a, p.head_dim, plan->group, p.dtype, plan->merge_grid, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? PKV_ERR_UNSUPPORTED : PKV_ERR_CUDA;
  }
  return PKV_OK;
}
