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
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

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

// Driver calls that name the current context and its process-unique id.
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns* ctx_fns() {
  static std::once_flag once;
  static CtxFns f;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return (f.get_current && f.get_id) ? &f : nullptr;
}

// Device address of g_noalloc_scratch in the current context of `device`.
// In host code the symbol names a host-side stand-in, so kernels must receive
// the address that cudaGetSymbolAddress returns with the device current.  The
// lookup is the set-up step: done once per device, and again only when the
// device's context has changed (a context made after cudaDeviceReset holds a
// fresh copy of the array, possibly at another address), which the context's
// process-unique id tells.
cudaError_t scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  static unsigned long long ctx_of[kMaxDevices] = {0};
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  const CtxFns* f = ctx_fns();
  if (!f) return cudaErrorNotSupported;
  // The id of the current context; 0 while the runtime has made none current on
  // this thread yet (cudaGetSymbolAddress below makes the device's one current).
  auto current_id = [&](unsigned long long* id) {
    CUcontext ctx = nullptr;
    *id = 0;
    if (f->get_current(&ctx) != CUDA_SUCCESS) return false;
    return !ctx || f->get_id(ctx, id) == CUDA_SUCCESS;
  };
  unsigned long long id = 0;
  if (!current_id(&id)) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(mu);
  if (id == 0 || !addr[device] || ctx_of[device] != id) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!current_id(&id) || id == 0) return cudaErrorDeviceUninitialized;
    addr[device] = p;
    ctx_of[device] = id;
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
  // Tensor-core decode plans keep prefill tables and 128-row partial states, far
  // more than the static array holds.
  if (plan->exec_prefill) return PKV_ERR_UNSUPPORTED;
  if (!host_tables || host_tables_bytes < plan->host_bytes) return PKV_ERR_INVALID_ARG;
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
