/*
 * pkv_bsr.h -- C ABI of a GB300 (sm_103a) library for attention over a KV
 * cache stored as a block-sparse row (BSR) matrix of pages.
 *
 * The method is the one the FlashInfer pages describe:
 *  - "FlashInfer" guide (infra.bea.ai), section 2 "Page-Level Attention":
 *    each request owns a page table; token t of request b lives in page
 *    kv_indices[kv_indptr[b] + t / page_size] at slot t % page_size, and the
 *    last page holds kv_last_page_len[b] valid slots.
 *  - Same guide, "The Interface": batch_prefill (causal) and batch_decode
 *    take (q, kv_data, kv_indices, kv_indptr, kv_last_page_len).
 *  - Same guide, section 3 "FlashDecoding" and "Cascade Attention": split-KV
 *    partial states and their log-sum-exp merge (merge_state).
 *  - fdeinterviews summary, "Load balancing that survives CUDA graphs": a CPU
 *    plan splits long KV sequences into equal chunks across the SMs and
 *    records where partial results go; fixed-grid kernels then run (and can be
 *    captured in a CUDA graph) and merge the partials.
 *  - greptalks summary, "Runtime Scheduler": the plan / run split.
 *
 * Conventions for every entry point
 *  - All tensors are dense, row-major, caller-owned device memory unless a
 *    parameter says "host".  The library never allocates device memory and
 *    never frees caller memory.  Pointers must be 16-byte aligned.
 *  - Layouts:
 *      q, o        [total_q, num_qo_heads, head_dim]  fp16 or bf16 (same dtype)
 *      lse         [total_q, num_qo_heads]            fp32, natural log
 *      kv_data     [num_pages, 2, num_kv_heads, page_size, head_dim]
 *                  K at index 0, V at index 1 of the second axis.
 *      qo_indptr   [batch + 1] int32, rows of request b: qo_indptr[b] .. qo_indptr[b+1]-1
 *      kv_indptr   [batch + 1] int32, CSR row pointer over kv_indices
 *      kv_indices  [kv_indptr[batch]] int32, physical page ids in [0, num_pages)
 *      kv_last_page_len [batch] int32 in [1, page_size]; ignored for a request
 *                  without pages, whose output is o = 0, lse = -inf
 *  - Query head h reads kv head h / (num_qo_heads / num_kv_heads).
 *  - logits = sm_scale * q.k; when logits_cap > 0 they become
 *    logits_cap * tanh(logits / logits_cap) before the softmax; lse is the
 *    natural log-sum-exp of the final logits.
 *  - Causal prefill: row i of a request with qo_len rows and kv_len keys sees
 *    keys j <= i + kv_len - qo_len.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Run calls
 *    enqueue work and return; they never synchronise the host.  Their kernels
 *    (all but the standalone prefill kernel) are launched as programmatic
 *    dependents of the kernel before them on `stream`: their blocks may be
 *    placed as that kernel's blocks exit, but read and write nothing before
 *    it has completed and its writes are visible, so stream order holds.
 *  - Errors are returned as pkv_status; nothing is thrown and nothing is
 *    printed.  A failed call enqueues no kernel.
 */
#ifndef PKV_BSR_H
#define PKV_BSR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer, wrong plan kind */
    PKV_ERR_BAD_INDEX = -2,    /* malformed indptr, page id out of range, bad last_page_len */
    PKV_ERR_UNSUPPORTED = -3,  /* head_dim / group size / dtype / page size not built */
    PKV_ERR_WORKSPACE = -4,    /* a workspace is too small, or the batch exceeds the plan limits */
    PKV_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed */
    PKV_ERR_DEVICE_CHECK = -6  /* a kernel recorded an error word (see pkv_get_device_error) */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/* DECODE: one query row per request (CUDA cores, split-KV).  PREFILL: ragged
 * query rows (tcgen05 tensor cores).  MIXED: a batch holding both; requests with
 * one query row take the decode path, longer ones the prefill path, and one
 * persistent kernel serves both on disjoint SMs (see pkv_batch_mixed_paged). */
typedef enum { PKV_PLAN_DECODE = 0, PKV_PLAN_PREFILL = 1, PKV_PLAN_MIXED = 2 } pkv_plan_kind;

/* Problem description shared by plan and run calls. */
typedef struct {
    int num_qo_heads;   /* Hq, a multiple of num_kv_heads */
    int num_kv_heads;   /* Hkv */
    int head_dim;       /* d: 64 or 128 */
    int page_size;      /* P: 1..16, or a multiple of 16 */
    int dtype;          /* pkv_dtype of q, kv_data and o: PKV_F16 or PKV_BF16 */
    float sm_scale;     /* usually 1/sqrt(head_dim) */
    float logits_cap;   /* <= 0: off */
    int causal;         /* prefill: end-aligned causal mask; ignored by decode */
} pkv_params;

/* Upper bounds a plan is sized for (fixed for the plan's lifetime, so that a
 * captured CUDA graph can be replayed after re-planning a different batch). */
typedef struct {
    int max_batch;          /* requests per call */
    int64_t max_total_q;    /* query rows per call (decode: = max_batch) */
    int64_t max_kv_pages;   /* entries of kv_indices per call */
} pkv_limits;

/* Opaque host-side plan object (inspector of the inspector-executor pair). */
typedef struct pkv_plan pkv_plan;

/* Human-readable name of a status code (static storage). */
const char* pkv_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * Create a plan for `kind` on CUDA device `device`.  Validates params and
 * limits, queries the device's SM count, and fixes the worker grid.
 * Allocates only host memory (freed by pkv_plan_destroy).
 * Errors: PKV_ERR_INVALID_ARG (also limits whose tables would need more than
 * 2^31 - 1 work entries: decode max_batch * num_kv_heads, prefill about
 * (max_total_q * group / 256 + max_batch) * num_kv_heads), PKV_ERR_UNSUPPORTED,
 * PKV_ERR_CUDA.
 */
pkv_status pkv_plan_create(pkv_plan** out, int kind, const pkv_params* params,
                           const pkv_limits* limits, int device);

pkv_status pkv_plan_destroy(pkv_plan* plan);

/*
 * Create a plan for a device with `num_sms` SMs without any CUDA call, so that
 * the plan's decisions can be inspected on a machine without a GPU.  Such a
 * plan computes tables (pkv_plan_compute) but cannot run (PKV_ERR_INVALID_ARG).
 * Errors: as pkv_plan_create, less PKV_ERR_CUDA.
 */
pkv_status pkv_plan_create_host(pkv_plan** out, int kind, const pkv_params* params,
                                const pkv_limits* limits, int num_sms);

/*
 * Bytes of caller-provided memory the plan needs:
 *  - dev_bytes: device workspace (plan tables, fp32 partial states, error word;
 *    for a prefill plan on pages of fewer than 8 rows also the 16-row-page copy
 *    of up to limits->max_kv_pages pages' keys);
 *  - host_bytes: pinned host staging buffer for the plan tables.
 * Both depend only on params and limits.
 */
pkv_status pkv_plan_workspace_bytes(const pkv_plan* plan, size_t* dev_bytes, size_t* host_bytes);

/*
 * The plan step (fdeinterviews "Load balancing"; greptalks "Runtime
 * Scheduler").  Reads HOST copies of the index arrays, validates them
 * (monotone indptr, page ids in [0, num_pages), last_page_len in range,
 * sizes within the limits), splits the KV work into chunks of equal cost over
 * the fixed worker grid (pages, plus one page's worth for each piece of a
 * (request, kv head) page list), records where every partial state goes, and enqueues one
 * host-to-device copy of the tables (from `host_ws`, which must be pinned) into
 * `dev_ws` on `stream`.  Clears the device error word.
 *  - qo_indptr_h: host [batch+1]; NULL for decode (one row per request).
 *  - kv_indices_h: host, may be NULL to skip the page-id range check.
 *  - num_pages: rows of kv_data's first axis (the pool size).
 * A later plan_run on the same plan first waits for the previous copy out of
 * host_ws to finish.  Run calls must be enqueued after this call on the same
 * stream (or ordered after it).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_BAD_INDEX, PKV_ERR_WORKSPACE (also a
 * request of 2^31 keys or more), PKV_ERR_CUDA.
 */
pkv_status pkv_plan_run(pkv_plan* plan, int batch, const int32_t* qo_indptr_h,
                        const int32_t* kv_indptr_h, const int32_t* kv_indices_h,
                        const int32_t* kv_last_page_len_h, int64_t num_pages, void* dev_ws,
                        size_t dev_ws_bytes, void* host_ws, size_t host_ws_bytes, void* stream);

/*
 * The host half of pkv_plan_run: validate the host index arrays and write
 * the plan tables into `host_ws` (ordinary or pinned host memory), with no
 * CUDA call.  pkv_plan_run is this step followed by one asynchronous copy.
 * Prefill and mixed plans keep their working arrays in the plan object and
 * reuse them from call to call (they grow with the largest batch planned).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_BAD_INDEX, PKV_ERR_WORKSPACE.
 */
pkv_status pkv_plan_compute(pkv_plan* plan, int batch, const int32_t* qo_indptr_h,
                            const int32_t* kv_indptr_h, const int32_t* kv_indices_h,
                            const int32_t* kv_last_page_len_h, int64_t num_pages, void* host_ws,
                            size_t host_ws_bytes);

/* Summary of the fixed grid and of the last computed plan. */
typedef struct {
    int grid_ctas;       /* CTAs of the main kernel's fixed grid */
    int workers;         /* workers of the grid (decode: warps; prefill: CTAs) */
    int active_workers;  /* workers the last plan gave work to */
    int num_work;        /* work entries (decode segments / prefill tiles) */
    int num_merge;       /* split sequences whose partial states get merged */
    int num_slots;       /* partial-state slots used */
    int64_t max_cost;    /* largest per-worker cost (decode: pages; prefill: KV blocks) */
    int64_t total_cost;  /* sum of the per-worker costs */
    int prefill_ctas;    /* mixed plans: SMs the last plan gave the prefill half (0 otherwise) */
    int decode_ctas;     /* mixed plans: SMs the last plan gave the decode half (0 otherwise) */
} pkv_plan_info;

pkv_status pkv_plan_get_info(const pkv_plan* plan, pkv_plan_info* info);

/*
 * Copy the last computed work list, 8 int32 per entry, in worker order:
 *   decode:  {worker, b, kv_head, page_begin, n_pages, last_rows, slot, 0}
 *   prefill: {worker, b, kv_head, q_pos0, n_pos, kv_begin, kv_end, slot}
 * (slot = -1: the entry writes the final output itself).
 * *rows_written receives the number of entries (also when capacity is short,
 * in which case nothing is copied and PKV_ERR_WORKSPACE is returned).
 */
pkv_status pkv_plan_get_work(const pkv_plan* plan, int32_t* out, int64_t capacity,
                             int64_t* rows_written);

/*
 * Profiling hook.  While set, every run call on this plan records `start` on
 * its stream just before the main kernel (decode or prefill; for a prefill
 * plan on pages of fewer than 8 rows, before the copy into 16-row pages that
 * precedes it) and `stop` just after it, before the merge kernel, so the caller
 * can time the main kernel alone with cudaEventElapsedTime.  The events (cudaEvent_t) stay the
 * caller's; pass NULL for both to clear.
 * Errors: PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_plan_set_timing_events(pkv_plan* plan, void* start, void* stop);

/*
 * Pipelined planning, for a step loop that re-plans every call (a serving loop's
 * decode steps).  The plan keeps two images of its tables, in two halves of the
 * host workspace and in two regions of the device workspace (both sizes from
 * pkv_plan_workspace_bytes already include them).  With on != 0 each
 * pkv_plan_run fills the image the previous run is not reading and copies it on a
 * stream the plan owns, so that copy overlaps the previous call's kernels; the next
 * run call waits for it on its own stream.  Not for CUDA-graph capture of the run
 * calls (the image a run reads alternates).  Call before the first pkv_plan_run;
 * device plans of kind DECODE or PREFILL only.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.
 */
pkv_status pkv_plan_set_pipelined(pkv_plan* plan, int on);

/*
 * Split-KV on or off for a decode plan (default on).  On, the plan step cuts
 * the (request, kv head) page lists into runs of equal cost over the workers and merges
 * the partial states ("FlashInfer" guide, section 3 "FlashDecoding"; fdeinterviews
 * summary, "Load balancing that survives CUDA graphs").  Off, each page list goes
 * whole to one worker (one warp), longest first onto the least-loaded worker,
 * with no partial states and no merge: the baseline the split is measured
 * against, in which one long request rests on one warp per kv head.  Ties go to
 * the earlier list, then to the worker of lower rank, rank r being warp r / C of
 * CTA r % C over the plan's C CTAs (equal loads spread over the SMs first).
 * Takes effect at the next plan step; the run call is unchanged.  The switch is
 * the CUDA-core decode schedule's: a decode plan on the tensor-core path (see
 * pkv_batch_decode_paged) refuses on = 0.
 * Errors: PKV_ERR_INVALID_ARG (NULL, or not a plan of kind DECODE),
 * PKV_ERR_UNSUPPORTED (on = 0 for a tensor-core decode plan).
 */
pkv_status pkv_plan_set_split_kv(pkv_plan* plan, int on);

/*
 * Batch decode over the paged KV cache ("The Interface", step 3; guide
 * section 3 "FlashDecoding"): one query row per request, all query heads.
 * q and o: [batch, Hq, d]; lse: [batch, Hq] fp32 (may be NULL).
 * kv_indptr_d and kv_last_page_len_d must hold the values the plan saw; the
 * kernels read page ids from kv_indices_d and check kv_indptr_d against the
 * plan (a mismatch sets the device error word and skips the work).
 * Long sequences are split into chunks whose fp32 partial states go to dev_ws
 * and are merged by log-sum-exp in a second fixed-grid kernel.  Graph-capturable.
 * Pages of one row (column-vector BSR) reach the kernel through a TMA tensor
 * map over kv_data built at launch from kv_data and num_pages of the current
 * plan: with page_size 1 a captured graph can be replayed after re-planning a
 * batch over the same kv_data buffer and pool size (page_size 1 with more than
 * 2^31 (page, K|V, kv head) rows in the pool is refused with PKV_ERR_UNSUPPORTED).
 * Tensor-core path: with 8 query heads per kv head, head_dim 128 and pages of 8
 * rows or more, the plan makes prefill work tiles of one query row per request
 * (greptalks summary, "Head Group Packing": the 8 heads of a group form the
 * rows of one 128-row tile; fdeinterviews summary, "Customizable attention": a
 * query tile size matched to the batch) and this call runs the tcgen05 prefill
 * kernel and its merge on them, causal mask off.  There a group-8 decode worker
 * on the CUDA cores is compute-bound.  The device kv_indptr is not re-checked
 * on that path, and dev_ws is sized for prefill tables and 128-row partial
 * states (pkv_plan_workspace_bytes reports it).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_batch_decode_paged(const pkv_plan* plan, const void* q, const void* kv_data,
                                  const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                  const int32_t* kv_last_page_len_d, void* o, float* lse,
                                  void* dev_ws, void* stream);

/*
 * Batch prefill over the paged KV cache ("The Interface", step 2), ragged
 * query rows given by qo_indptr_d, causal per params->causal, computed with
 * tcgen05 tensor-core MMAs (bf16 and fp16) and fp32 TMEM accumulators.
 * Built for head_dim 128, groups 1/2/4/8 and page sizes 1, 2, 4, 8, 16, 32,
 * 64 and 128.  Pages of 1-4 rows (the column-vector BSR of sparse patterns)
 * are first copied, row by row, into 16-row pages of the device workspace (each
 * request's keys in order, ceil(kv_len / 16) pages), and the tensor-core kernel
 * runs over that copy; larger pages are read in place, one tensor copy per page.
 * q and o: [total_q, Hq, d]; lse: [total_q, Hq] fp32 (may be NULL).
 * With causal = 0 and one request whose rows are many requests' queries, this
 * is the shared-prefix half of cascade attention.  The kernel's TMA tensor maps
 * are built at launch from q, kv_data, the total query rows and num_pages of
 * the current plan, so a captured CUDA graph can be replayed after re-planning
 * a batch with the same q and kv_data buffers, total query rows and pool size.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_batch_prefill_paged(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                   const void* kv_data, const int32_t* kv_indices_d,
                                   const int32_t* kv_indptr_d, const int32_t* kv_last_page_len_d,
                                   void* o, float* lse, void* dev_ws, void* stream);

/*
 * Batch prefill with a custom attention mask, for tree attention (speculative
 * decoding verifies a tree of draft tokens: each draft sees the cached prefix
 * and its own ancestors) and any other block-sparse pattern finer than a
 * page.  The pages list masks among the pieces a variant supplies
 * (fdeinterviews summary, "Customizable attention, compiled just in time")
 * and the token trees of speculative decoding among the KV layouts the BSR
 * format covers (greptalks summary, "Radix Tree / Token Tree").
 * packed_mask_d: device bits, request b's boolean matrix [qo_len_b, kv_len_b]
 *   row-major, the requests back to back from bit 0 with no padding between
 *   them (request b starts at bit sum over b' < b of qo_len_b' * kv_len_b');
 *   bit k of 32-bit word w is bit 32 w + k (little-endian bytes, least
 *   significant bit first).  1 = the query row sees the key.
 * mask_bytes: size of that buffer; it must hold whole 32-bit words covering all
 *   bits (4 * ceil(total_bits / 32) bytes) and be 4-byte aligned.  The kernel
 *   never reads past mask_bytes.
 * The mask applies on top of params->causal (both must allow a key).  A row
 * that sees no key gets o = 0, lse = -inf.  Other arguments, layouts and graph
 * capture as for pkv_batch_prefill_paged.
 * Errors: PKV_ERR_INVALID_ARG (also for a short or misaligned mask),
 * PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_batch_prefill_paged_masked(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                          const void* kv_data, const int32_t* kv_indices_d,
                                          const int32_t* kv_indptr_d, const int32_t* kv_last_page_len_d,
                                          const uint8_t* packed_mask_d, size_t mask_bytes, void* o, float* lse,
                                          void* dev_ws, void* stream);

/*
 * Batch decode for callers that cannot allocate device memory: plug-ins whose
 * host framework owns all device memory through its own allocator, services
 * under a fixed device-memory budget, and code paths that must not pay the
 * implicit device synchronisation a cudaMalloc can cause.  The FlashInfer
 * pages have no counterpart of this call.
 * It computes exactly what pkv_batch_decode_paged computes, but the plan
 * tables and the fp32 partial states live in one static 8 MiB device array
 * inside this library (present on every device that loads it, until the
 * process exits) instead of a caller workspace, and the call allocates
 * nothing.
 *  - plan: a decode plan whose tables pkv_plan_compute wrote into
 *    host_tables (pageable or pinned host memory of host_tables_bytes, at
 *    least the plan's host_bytes).  The call copies them into the static array
 *    on `stream`; pinned host_tables must stay unchanged until that copy runs.
 *  - A plan whose device workspace (dev_bytes of pkv_plan_workspace_bytes)
 *    exceeds 8 MiB is rejected with PKV_ERR_WORKSPACE.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents (each call rewrites the tables, with a zeroed error word, before
 *    its kernels read them).  Calls whose work overlaps on the GPU (on other
 *    streams, or from several host threads) race on the array: serialise them.
 *  - The first call on each device looks up the array's device address with
 *    that device current, and so does the first call after the device's
 *    context was made anew (after cudaDeviceReset, say); make such a call
 *    before any stream capture.
 *  - The device error word lives in the static array and is not reported.
 *  - Decode plans on the tensor-core path (8 query heads per kv head at
 *    head_dim 128, see pkv_batch_decode_paged) are refused with
 *    PKV_ERR_UNSUPPORTED: their prefill-sized partial states do not fit.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_WORKSPACE, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_batch_decode_paged_noalloc(const pkv_plan* plan, const void* host_tables,
                                          size_t host_tables_bytes, const void* q, const void* kv_data,
                                          const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                          const int32_t* kv_last_page_len_d, void* o, float* lse,
                                          void* stream);

/*
 * Mixed batch: requests with one query row (decode) and requests with more
 * (prefill: chunked prompts, new requests) in one call, on a plan of kind
 * PKV_PLAN_MIXED.  The plan routes each request by its query-tile size: one
 * row to the CUDA-core decode path (split-KV over warp workers), several rows
 * to the tcgen05 prefill path (128-row tiles), and splits the SMs between the
 * two halves in proportion to their estimated times.  Where single rows run on
 * the tensor cores (8 query heads per kv head, head_dim 128, pages of 8 rows or
 * more; see pkv_batch_decode_paged) every request goes to the prefill half.  The run call makes one
 * persistent launch on every SM: the CTAs below the split run the prefill
 * half, the others the decode workers; then one merge launch folds both
 * halves' split sequences, on `stream` ("FlashInfer" guide, "Prefill-Decode Mixing";
 * fdeinterviews summary, "Customizable attention": a query tile size from 1 to
 * 128 picked per batch; greptalks, "Future Directions and Features": mixed
 * prefill and decode phases in one batch).  The split is read from the device
 * tables and the prefill half's tensor maps are built at launch as for
 * pkv_batch_prefill_paged, so a captured graph stays valid across re-planning
 * within the limits with the same q and kv_data buffers, total query rows and
 * pool size.
 * Arguments and layouts as for pkv_batch_prefill_paged (qo_indptr_d covers
 * every request; causal per params->causal applies to the prefill half, and a
 * single-row request sees all its keys either way).
 * Errors: PKV_ERR_INVALID_ARG (a null or misaligned pointer, a plan of another
 * kind or not planned), PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_batch_mixed_paged(const pkv_plan* plan, const void* q, const int32_t* qo_indptr_d,
                                 const void* kv_data, const int32_t* kv_indices_d, const int32_t* kv_indptr_d,
                                 const int32_t* kv_last_page_len_d, void* o, float* lse, void* dev_ws,
                                 void* stream);

/*
 * merge_state (guide section 3, "Cascade Attention": the two partial results
 * are combined with the online-softmax correction).  For each of n_rows *
 * num_heads rows with states (o_a, lse_a) and (o_b, lse_b) over disjoint key
 * sets:  m = max(lse_a, lse_b); w_x = exp(lse_x - m);
 *        o = (w_a o_a + w_b o_b) / (w_a + w_b); lse = m + ln(w_a + w_b).
 * Both lse = -inf gives o = 0, lse = -inf; a state with lse = -inf adds nothing.
 * o_* : [n_rows, num_heads, head_dim] of `dtype` (PKV_F16, PKV_BF16 or PKV_F32;
 * inputs and output share it); lse_*: [n_rows, num_heads] fp32.  o_out and
 * lse_out may alias o_a and lse_a.  lse_out may be NULL.  The kernel is
 * launched as a programmatic dependent of the work before it on `stream`: its
 * CTAs may start early but read nothing before that work has completed.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                           void* o_out, float* lse_out, int64_t n_rows, int num_heads, int head_dim,
                           int dtype, void* stream);

/*
 * merge_state over n states at once (the same composition as pkv_merge_state,
 * applied to any number of states over disjoint key sets: FlashDecoding's
 * partial outputs, or the levels of a shared-prefix tree, guide section 3):
 * for each of n_rows * num_heads rows, m = max_k lse_k, w_k = exp(lse_k - m),
 * o = sum_k w_k o_k / sum_k w_k, lse = m + ln(sum_k w_k); every lse_k = -inf
 * gives o = 0, lse = -inf, and a state with lse = -inf adds nothing.
 * State k of row r is row k * state_stride_rows + r of o_states ([rows,
 * num_heads, head_dim] of `dtype`) and lse_states ([rows, num_heads] fp32), so
 * n states of n_rows rows laid out one after another have state_stride_rows =
 * n_rows.  o_out / lse_out ([n_rows, num_heads, ...]) may be the rows of one of
 * the states (in place); lse_out may be NULL.  Launched as a programmatic
 * dependent of the work before it on `stream`, like pkv_merge_state.
 * Errors: PKV_ERR_INVALID_ARG (num_states < 1, state_stride_rows < n_rows, a
 * null or misaligned pointer), PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
pkv_status pkv_merge_states(const void* o_states, const float* lse_states, int num_states,
                            int64_t state_stride_rows, void* o_out, float* lse_out, int64_t n_rows,
                            int num_heads, int head_dim, int dtype, void* stream);

/*
 * Append new tokens' K and V into their pages, with the rotary position
 * embedding (RoPE) of the keys and of the queries fused into the same pass.
 * Serving appends each step's new tokens to the KV cache (greptalks MLSys
 * 2025 talk summary, Background, "Dynamic Problem Shapes": the prefill,
 * decode and append stages), and RoPE
 * is one of the query/key transforms an attention variant fuses
 * (fdeinterviews summary, "Customizable attention, compiled just in time").
 *
 * params       : num_qo_heads, num_kv_heads, head_dim (64 or 128), page_size
 *                and dtype (PKV_F16 / PKV_BF16) are used; the rest is ignored.
 * batch, nnz   : requests, and new tokens over all requests.
 * num_pages    : pool size; page ids outside [0, num_pages) are not written.
 * append_indptr_d  [batch + 1] int32 device: new rows of request b are
 *                append_indptr[b] .. append_indptr[b+1]-1 (append_indptr[0] = 0,
 *                append_indptr[batch] = nnz).
 * kv_indptr_d, kv_indices_d, kv_last_page_len_d: the page table as for the
 *                attention calls, already INCLUDING the new tokens: the n_b new
 *                tokens of request b are its last n_b tokens, so new token i sits
 *                at position kv_len_b - n_b + i, in page
 *                kv_indices[kv_indptr[b] + pos / page_size], slot pos % page_size.
 * k_new, v_new [nnz, num_kv_heads, head_dim] device, dtype.
 * kv_data      [num_pages, 2, num_kv_heads, page_size, head_dim] device: only the
 *                new tokens' slots are written.
 * q_in, q_out  [nnz, num_qo_heads, head_dim] device, dtype, or both NULL.  Row t
 *                of q is the query of new token t and turns by the same position.
 *                q_out may equal q_in (in place).
 * rope_theta   : > 0: keys and queries are rotated, "rotate half" pairing (element
 *                i < head_dim/2 with i + head_dim/2) by the angle
 *                pos * rope_theta^(-2i/head_dim); 0: copied unchanged.  Positions
 *                must be below 2^24.  V is never rotated.
 * error_d      : device int32 or NULL; OR-ed with 1 (a page id out of range) and
 *                16 (a row outside every request's new rows, more new tokens than
 *                kv_len, or a last-page length outside [1, page_size]).  Such
 *                tokens are skipped.  The caller clears it.
 * Errors: PKV_ERR_INVALID_ARG (null or misaligned pointer, bad size or theta),
 * PKV_ERR_UNSUPPORTED (head_dim, dtype), PKV_ERR_CUDA.  nnz = 0 is a no-op.
 */
pkv_status pkv_append_paged_kv(const pkv_params* params, int batch, int64_t nnz, int64_t num_pages,
                               const int32_t* append_indptr_d, const int32_t* kv_indptr_d,
                               const int32_t* kv_indices_d, const int32_t* kv_last_page_len_d,
                               const void* k_new, const void* v_new, void* kv_data, const void* q_in,
                               void* q_out, double rope_theta, int32_t* error_d, void* stream);

/*
 * Read (and, with clear != 0, reset) the device error word a plan's kernels
 * write when a check fails (page id out of range, indptr mismatch, a bounded
 * wait that ran out).  Synchronises `stream`.  *code = 0 means no error.
 */
pkv_status pkv_get_device_error(const pkv_plan* plan, void* dev_ws, int* code, int clear,
                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BSR_H */
