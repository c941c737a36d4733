// pkv_plan.h -- the host plan object behind the opaque pkv_plan handle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "pkv_bsr.h"
#include "pkv_internal.h"

namespace pkv {

// A prefill work item before it has its place: the query tile of request b, kv
// head kvh and positions from pos0, against keys [kv_begin, kv_end), with its
// partial slot or -1.
struct PlanItem {
  int32_t b, kvh, pos0, kv_begin, kv_end, slot;
};

// Working arrays of the prefill and mixed plan steps.  They live in the plan and
// keep their capacity from call to call, so re-planning a batch no larger than
// one planned before allocates nothing.
struct PlanScratch {
  std::vector<PlanItem> items;
  std::vector<PrefillMerge> merges;
  std::vector<int32_t> item_cost;
  std::vector<int64_t> mask_off, load, nb_tiles, by_cost, by_load;
  std::vector<int> start, order, cta_of, per_cta, by_cta, fill;
  std::vector<uint64_t> buckets;
  std::vector<DecodeSeg> dsegs;
  std::vector<int32_t> run_ptr;
  std::vector<int32_t> pk_indptr, pk_last;
  std::vector<std::pair<int, int32_t>> cuts;
};

}  // namespace pkv

struct pkv_plan {
  int kind = 0;
  pkv_params p{};
  pkv_limits lim{};
  int device = -1;          // -1: host-only plan (pkv_plan_create_host)
  int num_sms = 0;
  int group = 1;
  // Fixed grid and table capacities (depend on params and limits only).
  int grid_ctas = 0;
  int workers = 0;
  int max_work = 0;
  int max_merge = 0;
  int max_slots = 0;
  int rows_per_slot = 0;
  int merge_grid = 0;
  bool split_kv = true;     // decode: cut page lists into equal runs (pkv_plan_set_split_kv)
  // Decode plan whose batches run on the tcgen05 prefill kernel, one query row per
  // request (group 8 at head_dim 128, pages of 8 rows or more): its tables are
  // prefill tables, planned over row_indptr = 0, 1, ..., batch.
  bool exec_prefill = false;
  std::vector<int32_t> row_indptr;
  // Prefill plan on pages of fewer than 8 rows: each run first copies the
  // requests' K/V rows into 16-row pages of its workspace (pack_pages_kernel),
  // and the tables describe the prefill over that copy.
  bool packed = false;
  int64_t max_packed = 0;
  pkv::WorkspaceLayout L{};
  size_t host_bytes = 0;
  // Last computed plan.
  bool planned = false;
  int batch = 0;
  int64_t num_pages = 0;
  int64_t total_q = 0;
  int64_t mask_bits = 0;    // prefill: sum over requests of qo_len * kv_len (custom-mask size)
  int active_workers = 0;
  int num_work = 0;
  int num_merge = 0;
  int num_slots = 0;
  int64_t max_cost = 0;
  int64_t total_cost = 0;
  size_t used_bytes = 0;
  std::vector<int32_t> work_rows;  // 8 int32 per work entry, for pkv_plan_get_work
  pkv::PlanScratch scratch;
  // The copy of the tables out of the pinned buffer.
  cudaEvent_t copy_done = nullptr;
  bool copy_pending = false;
  // Pipelined plans (pkv_plan_set_pipelined): the tables alternate between two
  // images (host region r at r * tables_end, device region 0 at 0 and 1 at
  // L.alt); each plan_run copies the next image on copy_stream while the
  // previous run's kernels still read the other one.
  bool pipelined = false;
  int cur = 0;                       // image the next run reads
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t copy_ev[2] = {nullptr, nullptr};   // image r copied
  cudaEvent_t free_ev[2] = {nullptr, nullptr};   // the last run reading image r has finished
  bool copy_pend[2] = {false, false};
  bool used[2] = {false, false};
  // Caller events recorded around the main kernel (pkv_plan_set_timing_events).
  cudaEvent_t time_start = nullptr;
  cudaEvent_t time_stop = nullptr;
  // Mixed plans: the decode and prefill halves (each a plan of its own kind,
  // sharing this plan's device), where their tables and workspaces sit inside
  // this plan's workspaces, and the last SM split.
  pkv_plan* sub_dec = nullptr;
  pkv_plan* sub_pre = nullptr;
  size_t dec_dev_off = 0, pre_dev_off = 0, dec_host_off = 0, pre_host_off = 0;
  int prefill_ctas = 0;
  int decode_ctas = 0;
};
