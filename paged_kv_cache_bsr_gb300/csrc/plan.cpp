// plan.cpp -- the host-side plan (the "inspector" of an inspector-executor pair).
//
// fdeinterviews summary, "Load balancing that survives CUDA graphs": each
// step a CPU-side plan splits long KV sequences into equal chunks across the
// GPU's processors and records where partial results go; fixed-grid kernels
// then run.  greptalks summary, "Runtime Scheduler": a cost model decides the
// schedule deterministically from the sequence lengths alone.
//
// Decode: the work is the sequence of (request, kv head) page lists laid end
// to end.  With W workers (warps of the fixed grid) every worker takes one
// contiguous run of that sequence of the same cost: its pages plus a fixed
// cost for each piece of a list it holds (the piece's q load, first page-id
// window and epilogue), so all workers finish together whatever the length
// mix.  A page list cut by a run boundary becomes several partial states, each
// with its own slot, and one merge record.
//
// Prefill: the work is one tile per (request, kv head, block of query
// positions); its cost is the number of 128-key blocks it must visit (after
// the causal limit).  A tile costing more than total/CTAs is cut into key
// chunks with partial slots; tiles are then assigned longest-first to the
// least-loaded CTA.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <new>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "pkv_bsr.h"
#include "pkv_internal.h"
#include "pkv_launch.h"
#include "pkv_plan.h"

using pkv::DecodeSeg;
using pkv::MergeItem;
using pkv::PlanHeader;
using pkv::PlanScratch;
using pkv::PrefillMerge;
using pkv::PrefillTile;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_pow2_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// Single-row (decode) work that runs on the tcgen05 prefill kernel instead of the
// CUDA-core decode kernel.  With a group of 8 query heads per kv head the decode
// worker does 8 dot products and 8 P V accumulations per key on the CUDA cores
// and turns compute-bound (3.7 TB/s on the Llama-3-8B lengths, head_dim 128); the
// tensor cores take one request's 8 rows as a 128-row tile (4.95 TB/s).  Pages of
// fewer than 8 rows keep the decode kernel's tensor gathers.
bool decode_on_tensor_cores(const pkv_params* p) {
  const int g = p->num_qo_heads / p->num_kv_heads;
  return g == 8 && p->head_dim == 128 && p->page_size >= 8 &&
         pkv::prefill_supported(p->head_dim, g, p->dtype, p->page_size);
}

pkv_status check_params(int kind, const pkv_params* p, const pkv_limits* lim) {
  if (!p || !lim) return PKV_ERR_INVALID_ARG;
  if (kind != PKV_PLAN_DECODE && kind != PKV_PLAN_PREFILL && kind != PKV_PLAN_MIXED) return PKV_ERR_INVALID_ARG;
  if (p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_qo_heads % p->num_kv_heads)
    return PKV_ERR_INVALID_ARG;
  if (p->page_size <= 0 || (p->page_size > 16 && p->page_size % 16)) return PKV_ERR_UNSUPPORTED;
  if (!(p->sm_scale > 0.f)) return PKV_ERR_INVALID_ARG;
  if (lim->max_batch < 0 || lim->max_total_q < 0 || lim->max_kv_pages < 0) return PKV_ERR_INVALID_ARG;
  if (lim->max_kv_pages > INT32_MAX || lim->max_total_q > INT32_MAX) return PKV_ERR_INVALID_ARG;
  const int g = p->num_qo_heads / p->num_kv_heads;
  if (p->dtype != PKV_F16 && p->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (kind != PKV_PLAN_PREFILL && !pkv::decode_supported(p->head_dim, g, p->dtype)) return PKV_ERR_UNSUPPORTED;
  if (kind != PKV_PLAN_DECODE && !pkv::prefill_supported(p->head_dim, g, p->dtype, p->page_size))
    return PKV_ERR_UNSUPPORTED;
  if (!is_pow2_group(g)) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

void set_layout(pkv_plan* pl) {
  pkv::WorkspaceLayout& L = pl->L;
  const bool dec = pl->kind == PKV_PLAN_DECODE && !pl->exec_prefill;
  const size_t work_bytes = dec ? sizeof(DecodeSeg) : sizeof(PrefillTile);
  const size_t merge_bytes = dec ? sizeof(MergeItem) : sizeof(PrefillMerge);
  L.header = 0;
  L.worker_ptr = align_up(sizeof(PlanHeader), 256);
  L.merge = align_up(L.worker_ptr + sizeof(int32_t) * (pl->workers + 1), 256);
  // Packed prefill plans: the packed pages' ids and sources sit before the
  // tiles, so the table copy (up to the last tile in use) carries them.
  const size_t n_pk = pl->packed ? static_cast<size_t>(pl->max_packed) : 0;
  L.pk_ids = align_up(L.merge + merge_bytes * std::max(pl->max_merge, 1), 256);
  L.pk_src = align_up(L.pk_ids + sizeof(int32_t) * n_pk, 256);
  L.segs = align_up(L.pk_src + sizeof(pkv::PackedSrc) * n_pk, 256);
  L.tables_end = align_up(L.segs + work_bytes * std::max(pl->max_work, 1), 256);
  L.part_o = L.tables_end;
  L.part_lse = align_up(L.part_o + sizeof(float) * (size_t)pl->max_slots * pl->rows_per_slot * pl->p.head_dim, 256);
  L.pk_kv = align_up(L.part_lse + sizeof(float) * (size_t)pl->max_slots * pl->rows_per_slot, 256);
  // 2 bytes per element (fp16 / bf16), 16 rows per packed page.
  const size_t pk_bytes = n_pk * 2 * static_cast<size_t>(pl->p.num_kv_heads) * 16 * pl->p.head_dim * 2;
  L.alt = align_up(L.pk_kv + pk_bytes, 256);
  L.total = L.alt + L.tables_end;
}

// route_decode: a decode plan may run on the tensor cores (decode_on_tensor_cores);
// the decode half of a mixed plan never does (the mixed kernel's decode CTAs read
// decode tables).
pkv_status make_plan(pkv_plan** out, int kind, const pkv_params* params, const pkv_limits* limits,
                     int device, int num_sms, bool route_decode = true, bool allow_pack = true) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_status st = check_params(kind, params, limits);
  if (st != PKV_OK) return st;
  // Worker ids (num_sms x kDecodeWarps) fit the 24-bit field of the whole-list decode plan's heap keys.
  if (num_sms <= 0 || num_sms >= (1 << 20)) return PKV_ERR_INVALID_ARG;
  if (kind == PKV_PLAN_MIXED && num_sms < 2) return PKV_ERR_INVALID_ARG;  // one SM for each half at least
  pkv_plan* pl = new (std::nothrow) pkv_plan();
  if (!pl) return PKV_ERR_INVALID_ARG;
  pl->kind = kind;
  pl->p = *params;
  pl->lim = *limits;
  pl->device = device;
  pl->num_sms = num_sms;
  pl->group = params->num_qo_heads / params->num_kv_heads;
  const int64_t hkv = params->num_kv_heads;
  if (kind == PKV_PLAN_MIXED) {
    // Two plans of the same problem and limits; their workspaces are laid end to end.
    pkv_status s1 = make_plan(&pl->sub_dec, PKV_PLAN_DECODE, params, limits, device, num_sms, false);
    // The mixed kernel's prefill CTAs read the caller's pages (its own gather
    // instances for small pages): no packed copy.
    pkv_status s2 =
        s1 == PKV_OK ? make_plan(&pl->sub_pre, PKV_PLAN_PREFILL, params, limits, device, num_sms, true, false) : s1;
    if (s2 != PKV_OK) {
      delete pl->sub_dec;
      delete pl->sub_pre;
      delete pl;
      return s2;
    }
    pl->grid_ctas = num_sms;
    pl->workers = num_sms;
    pl->dec_dev_off = 0;
    pl->pre_dev_off = align_up(pl->sub_dec->L.total, 256);
    pl->L.total = pl->pre_dev_off + pl->sub_pre->L.total;
    pl->dec_host_off = 0;
    pl->pre_host_off = align_up(pl->sub_dec->host_bytes, 256);
    pl->host_bytes = pl->pre_host_off + pl->sub_pre->host_bytes;
    *out = pl;
    return PKV_OK;
  }
  pl->exec_prefill = kind == PKV_PLAN_DECODE && route_decode && decode_on_tensor_cores(params);
  if (kind == PKV_PLAN_DECODE && !pl->exec_prefill) {
    pl->grid_ctas = num_sms;
    pl->workers = num_sms * pkv::kDecodeWarps;
    // Each worker's run cuts at most two page lists, and every list adds at
    // most one uncut entry; see the decode branch of compute_decode.
    const int64_t max_work = pl->workers + static_cast<int64_t>(limits->max_batch) * hkv + 1;
    if (max_work > INT32_MAX) {  // table entries are counted in int32
      delete pl;
      return PKV_ERR_INVALID_ARG;
    }
    pl->max_work = static_cast<int>(max_work);
    pl->max_merge = static_cast<int>(std::min<int64_t>((int64_t)limits->max_batch * hkv, pl->workers) + 1);
    pl->max_slots = 2 * pl->workers;
    pl->rows_per_slot = pl->group;
    pl->merge_grid = num_sms * 4;
  } else {
    const int mp = pkv::kPrefillRows / pl->group;  // query positions per tile
    pl->grid_ctas = num_sms;
    pl->workers = num_sms;
    // A decode plan on the tensor cores has one query row per request.
    const int64_t max_rows = pl->exec_prefill ? limits->max_batch : limits->max_total_q;
    const int64_t tiles = (ceil_div(max_rows, mp) + limits->max_batch) * hkv;
    // Splitting only touches tiles costing more than total / CTAs (fewer than
    // CTAs of them), and adds at most CTAs chunks in total.
    const int64_t max_work = tiles + 2 * static_cast<int64_t>(num_sms) + 1;
    if (max_work > INT32_MAX) {  // table entries are counted in int32
      delete pl;
      return PKV_ERR_INVALID_ARG;
    }
    pl->max_work = static_cast<int>(max_work);
    pl->max_merge = num_sms + 1;
    pl->max_slots = 2 * num_sms + 2;
    pl->rows_per_slot = pkv::kPrefillRows;
    pl->merge_grid = num_sms * 4;
    // Pages of fewer than 8 rows: the tensor-core prefill runs over a packed copy
    // in 16-row pages (a request of L keys fills ceil(L / 16) of them).
    pl->packed = kind == PKV_PLAN_PREFILL && allow_pack && params->page_size < 8;
    if (pl->packed) {
      pl->max_packed = ceil_div(static_cast<int64_t>(limits->max_kv_pages) * params->page_size, 16) + limits->max_batch;
      // Packed page ids and the packed copy's row coordinates are 32-bit.
      if (pl->max_packed * 2 * hkv * 16 >= INT32_MAX) {
        delete pl;
        return PKV_ERR_INVALID_ARG;
      }
    }
  }
  set_layout(pl);
  pl->host_bytes = 2 * pl->L.tables_end;  // two table images: see pkv_plan_set_pipelined
  *out = pl;
  return PKV_OK;
}

// Common validation of the host index arrays.
pkv_status validate(const pkv_plan* pl, int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                    const int32_t* kv_indices, const int32_t* kv_last, int64_t num_pages) {
  if (batch < 0 || !kv_indptr || (batch > 0 && !kv_last)) return PKV_ERR_INVALID_ARG;
  if (batch > pl->lim.max_batch) return PKV_ERR_WORKSPACE;
  if (pl->kind != PKV_PLAN_DECODE && !qo_indptr) return PKV_ERR_INVALID_ARG;
  if (num_pages < 0 || num_pages > INT32_MAX) return PKV_ERR_INVALID_ARG;
  if (kv_indptr[0] != 0) return PKV_ERR_BAD_INDEX;
  for (int b = 0; b < batch; ++b) {
    // Compared before any subtraction: an int32 difference of a non-monotone
    // pair could wrap around to a positive page count.
    if (kv_indptr[b + 1] < kv_indptr[b]) return PKV_ERR_BAD_INDEX;
    const int64_t n = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
    if (n > 0 && (kv_last[b] < 1 || kv_last[b] > pl->p.page_size)) return PKV_ERR_BAD_INDEX;
    // Keys of one request are counted in int32 (a page id may be listed many times).
    if (n > 0 && (n - 1) * pl->p.page_size + kv_last[b] > INT32_MAX) return PKV_ERR_WORKSPACE;
  }
  const int64_t nnz = kv_indptr[batch];
  if (nnz > pl->lim.max_kv_pages) return PKV_ERR_WORKSPACE;
  if (nnz > 0 && num_pages == 0) return PKV_ERR_BAD_INDEX;
  if (kv_indices) {
    // One pass with no early exit, so that it vectorises: taken as unsigned, a
    // negative id wraps above every num_pages (at most INT32_MAX).
    const uint32_t np = static_cast<uint32_t>(num_pages);
    uint32_t bad = 0;
    for (int64_t j = 0; j < nnz; ++j) bad |= static_cast<uint32_t>(kv_indices[j]) >= np;
    if (bad) return PKV_ERR_BAD_INDEX;
  }
  if (qo_indptr) {
    if (qo_indptr[0] != 0) return PKV_ERR_BAD_INDEX;
    for (int b = 0; b < batch; ++b)
      if (qo_indptr[b + 1] < qo_indptr[b]) return PKV_ERR_BAD_INDEX;
    if (qo_indptr[batch] > pl->lim.max_total_q) return PKV_ERR_WORKSPACE;
  } else if (batch > pl->lim.max_total_q) {
    return PKV_ERR_WORKSPACE;
  }
  return PKV_OK;
}

int64_t kv_len_of(const int32_t* kv_indptr, const int32_t* kv_last, int b, int P) {
  const int64_t n = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
  return n > 0 ? (n - 1) * P + kv_last[b] : 0;
}

// Decode work with the split turned off (pkv_plan_set_split_kv): every
// (request, kv head) page list whole on one of `W` workers (warps of W / 8
// CTAs), longest first onto the least-loaded worker.  Ties go to the earlier
// list, and between workers to the lower rank, rank r being warp r / C of CTA
// r % C over C CTAs: so equal loads fill one warp on every SM before a second
// warp on any, and the longest lists land on different SMs.  No list is cut,
// so there are no partial slots and nothing to merge.
pkv_status compute_decode_whole(pkv_plan* pl, int batch, const int32_t* kv_indptr, const int32_t* kv_last,
                                uint8_t* host, int W) {
  const int hkv = pl->p.num_kv_heads;
  const int lists = batch * hkv;  // list i is request i / hkv, kv head i % hkv
  if (lists > pl->max_work) return PKV_ERR_WORKSPACE;
  const int ctas = std::max(1, W / pkv::kDecodeWarps);
  auto worker_of_rank = [&](int r) { return (r % ctas) * pkv::kDecodeWarps + r / ctas; };
  auto pages = [&](int i) { return kv_indptr[i / hkv + 1] - kv_indptr[i / hkv]; };
  PlanScratch& sc = pl->scratch;
  std::vector<int>& order = sc.order;
  order.resize(lists);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return pages(x) > pages(y); });
  const int ranks = std::min(W, lists);
  int n_workers = 0;  // highest worker used + 1
  for (int r = 0; r < ranks; ++r) n_workers = std::max(n_workers, worker_of_rank(r) + 1);
  std::vector<int64_t>& load = sc.load;  // by rank
  load.assign(ranks, 0);
  std::vector<int>& owner = sc.cta_of;   // worker of each list
  owner.resize(lists);
  std::vector<int>& per_worker = sc.per_cta;
  per_worker.assign(static_cast<size_t>(n_workers) + 1, 0);
  // Keys (load << 24) | rank order (load, rank) pairs by one integer comparison.
  constexpr int kRankBits = 24;
  std::priority_queue<uint64_t, std::vector<uint64_t>, std::greater<uint64_t>> heap;
  for (int r = 0; r < ranks; ++r) heap.push(static_cast<uint64_t>(r));
  for (int i : order) {
    const int r = static_cast<int>(heap.top() & ((uint64_t{1} << kRankBits) - 1));
    heap.pop();
    const int w = worker_of_rank(r);
    owner[i] = w;
    ++per_worker[static_cast<size_t>(w) + 1];
    load[r] += pages(i);
    heap.push((static_cast<uint64_t>(load[r]) << kRankBits) | static_cast<uint64_t>(r));
  }
  for (int w = 0; w < n_workers; ++w) per_worker[static_cast<size_t>(w) + 1] += per_worker[w];

  auto* hdr = reinterpret_cast<PlanHeader*>(host + pl->L.header);
  auto* wptr = reinterpret_cast<int32_t*>(host + pl->L.worker_ptr);
  auto* segs = reinterpret_cast<DecodeSeg*>(host + pl->L.segs);
  std::vector<int>& fill = sc.fill;  // each worker's lists in the order they were assigned
  fill.assign(per_worker.begin(), per_worker.end() - 1);
  for (int i : order) {
    const int b = i / hkv;
    const int32_t n = pages(i);
    DecodeSeg s{};
    s.b = b;
    s.kvh = i % hkv;
    s.q_row = b;
    s.idx_begin = kv_indptr[b];
    s.n_pages = n;
    s.last_rows = n > 0 ? kv_last[b] : 0;
    s.page_begin = 0;
    s.slot = -1;
    segs[fill[owner[i]]++] = s;
  }
  for (int w = 0; w <= n_workers; ++w) wptr[w] = per_worker[w];

  std::memset(hdr, 0, sizeof(PlanHeader));
  hdr->kind = PKV_PLAN_DECODE;
  hdr->batch = batch;
  hdr->num_workers = n_workers;  // workers below this with no list return at once
  hdr->num_segments = lists;

  pl->active_workers = ranks;
  pl->num_work = lists;
  pl->num_merge = 0;
  pl->num_slots = 0;
  int64_t total = 0, most = 0;
  for (int64_t v : load) {
    total += v;
    most = std::max(most, v);
  }
  pl->total_cost = total;
  pl->max_cost = most;
  pl->work_rows.assign(static_cast<size_t>(lists) * 8, 0);
  for (int w = 0; w < n_workers; ++w)
    for (int k = wptr[w]; k < wptr[w + 1]; ++k) {
      const DecodeSeg& s = segs[k];
      int32_t* r = &pl->work_rows[static_cast<size_t>(k) * 8];
      r[0] = w; r[1] = s.b; r[2] = s.kvh; r[3] = 0; r[4] = s.n_pages; r[5] = s.last_rows; r[6] = -1; r[7] = 0;
    }
  pl->used_bytes = pl->L.segs + sizeof(DecodeSeg) * static_cast<size_t>(lists);
  return PKV_OK;
}

// Decode work over `W` warp workers.  With qo_indptr (a mixed batch) only the
// requests holding exactly one query row take part, and each reads and writes
// its row qo_indptr[b]; without it every request is one row, row b.
// Decode run costs, in eighths of a page: a page, and the start of a piece of a
// page list (its q load, first page-id window and epilogue), which measured
// like one page.  Against runs of equal page counts (three A/B rounds on one
// box): the cascade as one mixed launch 27.6 -> 26.1 us, the mixed batch 169.0
// -> 167.7 us, the Llama-3-8B decode step 6160 -> 6178 GB/s.
constexpr int64_t kPageCost = 8;
constexpr int64_t kSegCost = 1 * kPageCost;
pkv_status compute_decode(pkv_plan* pl, int batch, const int32_t* kv_indptr, const int32_t* kv_last,
                          uint8_t* host, const int32_t* qo_indptr = nullptr, int W = 0) {
  const int P = pl->p.page_size;
  const int hkv = pl->p.num_kv_heads;
  if (W <= 0) W = pl->workers;
  if (!pl->split_kv && !qo_indptr) return compute_decode_whole(pl, batch, kv_indptr, kv_last, host, W);
  auto takes_part = [&](int b) { return !qo_indptr || qo_indptr[b + 1] - qo_indptr[b] == 1; };
  // Runs as short as one page: on the tiny fp16 batch (4 requests x 2 kv heads of
  // 5-13 pages) runs of one page took a run call from 10.1 us to 6.3 us against
  // a 4-tile minimum, and no batch measured slower (64 x 8 lists of 1-128 pages,
  // the Llama-3-8B lengths, the prefix tree, the mixed batch).
  int64_t total = 0;
  int parts = 0;
  for (int b = 0; b < batch; ++b)
    if (takes_part(b)) {
      total += (int64_t)(kv_indptr[b + 1] - kv_indptr[b]) * hkv;
      ++parts;
    }
  const int64_t run = total > 0 ? ceil_div(total, W) : 1;
  if (!qo_indptr && static_cast<int64_t>(batch) * hkv <= W) {
    // When no list is longer than a run there is nothing to split, and the run
    // sequence would only pack several short lists onto one warp while others
    // idle: each list then gets a worker of its own (measured, 64 x 8 lists of
    // one page: 8.2 us against 16.4 us).
    int32_t longest = 0;
    for (int b = 0; b < batch; ++b) longest = std::max(longest, kv_indptr[b + 1] - kv_indptr[b]);
    if (longest <= run) return compute_decode_whole(pl, batch, kv_indptr, kv_last, host, W);
  }

  auto* hdr = reinterpret_cast<PlanHeader*>(host + pl->L.header);
  auto* wptr = reinterpret_cast<int32_t*>(host + pl->L.worker_ptr);
  auto* merge = reinterpret_cast<MergeItem*>(host + pl->L.merge);
  auto* segs = reinterpret_cast<DecodeSeg*>(host + pl->L.segs);

  int n_seg = 0, n_merge = 0, n_slot = 0;
  int cur_worker = 0;
  wptr[0] = 0;
  auto emit = [&](int worker, const DecodeSeg& s) {
    while (cur_worker < worker) wptr[++cur_worker] = n_seg;
    segs[n_seg++] = s;
  };
  // Cost coordinate, in eighths of a page: the lists in order, each piece of a
  // list costing kSegCost (its q load, first page-id window and epilogue) before
  // its pages.  A page goes to the run r with r T <= its midpoint < (r + 1) T; a
  // piece ends where a list ends or its next page falls in the next run.  Every
  // list starts one piece and each of the W - 1 run boundaries at most one more,
  // so with T below the whole cost fits in W runs.  T holds at least a piece
  // start and a page, so a new piece's first page lands in the next run, never
  // past it.
  const int64_t lists = static_cast<int64_t>(parts) * hkv;
  const int64_t T = std::max<int64_t>(kSegCost + kPageCost,
                                      ceil_div(total * kPageCost + kSegCost * (lists + W - 1), W));
  int64_t X = 0;
  int used = 0;
  std::vector<std::pair<int, int32_t>>& cuts = pl->scratch.cuts;  // (run, first page) of each piece
  for (int b = 0; b < batch; ++b) {
    if (!takes_part(b)) continue;
    const int32_t n = kv_indptr[b + 1] - kv_indptr[b];
    const int32_t row = qo_indptr ? qo_indptr[b] : b;
    for (int h = 0; h < hkv; ++h) {
      DecodeSeg s{};
      s.b = b;
      s.kvh = h;
      s.q_row = row;
      if (n == 0) {
        const int w = static_cast<int>(std::min<int64_t>(X / T, W - 1));
        s.idx_begin = kv_indptr[b];
        s.n_pages = 0;
        s.last_rows = 0;
        s.page_begin = 0;
        s.slot = -1;
        emit(w, s);
        used = std::max(used, w + 1);
        continue;
      }
      cuts.clear();
      for (int32_t lo = 0; lo < n;) {
        X += kSegCost;
        const int64_t r = std::min<int64_t>((X + kPageCost / 2) / T, W - 1);
        const int64_t room = (r + 1) * T - X - kPageCost / 2;  // > 0: this page's midpoint is in run r
        const int32_t cnt =
            r == W - 1 ? n - lo : static_cast<int32_t>(std::min<int64_t>(n - lo, ceil_div(room, kPageCost)));
        cuts.push_back({static_cast<int>(r), lo});
        X += static_cast<int64_t>(cnt) * kPageCost;
        lo += cnt;
      }
      used = std::max(used, cuts.back().first + 1);
      if (cuts.size() == 1) {
        s.idx_begin = kv_indptr[b];
        s.n_pages = n;
        s.last_rows = kv_last[b];
        s.page_begin = 0;
        s.slot = -1;
        emit(cuts[0].first, s);
      } else {
        MergeItem m{row, h, n_slot, static_cast<int32_t>(cuts.size())};
        if (n_merge >= pl->max_merge || n_slot + m.n_slots > pl->max_slots) return PKV_ERR_WORKSPACE;
        merge[n_merge++] = m;
        for (size_t k = 0; k < cuts.size(); ++k) {
          const int32_t lo = cuts[k].second, hi = k + 1 < cuts.size() ? cuts[k + 1].second : n;
          s.idx_begin = kv_indptr[b] + lo;
          s.n_pages = hi - lo;
          s.last_rows = hi == n ? kv_last[b] : P;
          s.page_begin = lo;
          s.slot = n_slot++;
          emit(cuts[k].first, s);
        }
      }
    }
  }
  const int active = used;
  while (cur_worker < active) wptr[++cur_worker] = n_seg;
  if (n_seg > pl->max_work || n_slot > pl->max_slots || n_merge > pl->max_merge) return PKV_ERR_WORKSPACE;

  // The runs go to the warps CTA by CTA: run r to warp r / C of CTA r % C (C CTAs),
  // so a batch that fills only some of the workers still spreads them over every
  // SM instead of packing eight to an SM.  Segments are regrouped by worker.
  int n_workers = active;
  const int C = W / pkv::kDecodeWarps;
  if (C > 1 && active > 0) {
    PlanScratch& sc = pl->scratch;
    sc.dsegs.assign(segs, segs + n_seg);
    sc.run_ptr.assign(wptr, wptr + active + 1);
    n_workers = 0;
    int k = 0;
    wptr[0] = 0;
    for (int w = 0; w < W; ++w) {
      const int r = (w % pkv::kDecodeWarps) * C + w / pkv::kDecodeWarps;  // the run of worker w
      if (r < active) {
        for (int i = sc.run_ptr[r]; i < sc.run_ptr[r + 1]; ++i) segs[k++] = sc.dsegs[i];
        n_workers = w + 1;
      }
      wptr[w + 1] = k;
      if (w + 1 >= n_workers && k == n_seg) break;
    }
  }

  std::memset(hdr, 0, sizeof(PlanHeader));
  hdr->kind = PKV_PLAN_DECODE;
  hdr->batch = batch;
  hdr->num_workers = n_workers;  // workers below this with no run return at once
  hdr->num_segments = n_seg;
  hdr->num_merge = n_merge;
  hdr->num_slots = n_slot;

  pl->active_workers = active;
  pl->num_work = n_seg;
  pl->num_merge = n_merge;
  pl->num_slots = n_slot;
  pl->total_cost = total;
  pl->max_cost = 0;
  pl->work_rows.assign((size_t)n_seg * 8, 0);
  for (int w = 0; w < n_workers; ++w) {
    int64_t cost = 0;
    for (int i = wptr[w]; i < wptr[w + 1]; ++i) {
      const DecodeSeg& s = segs[i];
      int32_t* r = &pl->work_rows[(size_t)i * 8];
      r[0] = w; r[1] = s.b; r[2] = s.kvh; r[3] = s.page_begin; r[4] = s.n_pages;
      r[5] = s.last_rows; r[6] = s.slot; r[7] = 0;
      cost += s.n_pages;
    }
    pl->max_cost = std::max(pl->max_cost, cost);
  }
  pl->used_bytes = pl->L.segs + sizeof(DecodeSeg) * (size_t)n_seg;
  return PKV_OK;
}

// Key end of the query tile of positions [pos0, pos0 + npos) of a request with
// qo rows and kv keys: every key, or under the causal mask the limit of its last
// row, clipped to [0, kv].
int tile_kv_end(bool causal, int qo, int kv, int pos0, int npos) {
  return causal ? std::max(0, std::min(kv, pos0 + npos + kv - qo)) : kv;
}

// The prefill plan's query tiles are one per (request, kv head, block of
// kPrefillRows / group query positions), each against keys [0, kv_end).  Returns
// their key blocks in total, an empty tile counting one (independent of the CTA
// count); with nb_tiles, also the number of tiles of each count of key blocks.
// The kv heads of a request repeat its tiles, so they count once per block.
int64_t query_tile_blocks(const pkv_plan* pl, int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_last, bool skip_single, std::vector<int64_t>* nb_tiles,
                          int page_size = 0) {
  const int P = page_size > 0 ? page_size : pl->p.page_size;
  const int mp = pkv::kPrefillRows / pl->group;
  const int64_t hkv = pl->p.num_kv_heads;
  if (nb_tiles) nb_tiles->clear();
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) {
    const int qo = qo_indptr[b + 1] - qo_indptr[b];
    if (skip_single && qo == 1) continue;
    const int kv = static_cast<int>(kv_len_of(kv_indptr, kv_last, b, P));
    for (int pos0 = 0; pos0 < qo; pos0 += mp) {
      const int64_t nb = ceil_div(tile_kv_end(pl->p.causal, qo, kv, pos0, std::min(mp, qo - pos0)),
                                  pkv::kPrefillKeys);
      total += hkv * std::max<int64_t>(1, nb);
      if (nb_tiles) {
        if (nb >= static_cast<int64_t>(nb_tiles->size())) nb_tiles->resize(nb + 1, 0);
        (*nb_tiles)[nb] += hkv;
      }
    }
  }
  return total;
}

// Key blocks per work item when `total` blocks go to C CTAs: a tile longer than
// this is cut into that many near-equal chunks (each a partial state to merge),
// down to single blocks (against a 2-block minimum, single blocks took a 64-row
// prompt of 512 keys from 18.4 to 16.4 us and of 2048 keys from 20.4 to 18.5 us,
// with the ragged batch and the cascade unchanged).
int64_t key_chunk(int64_t total, int C) { return std::max<int64_t>(ceil_div(total, std::max(C, 1)), 1); }

// The busiest CTA's load (key blocks, plus kItemOverhead per item for its setup
// and epilogue) when compute_prefill chunks the tiles for C CTAs and assigns them
// longest first.  `nb_tiles[k]` counts the tiles of k key blocks: an item's cost
// depends on nothing else.  The costs are small integers and the least load of a
// longest-first schedule never decreases, so the schedule runs on counts (`by_cost`
// items per cost, `by_load` CTAs per load; both scratch), and a run of items of
// equal cost moves the least-loaded CTAs together, exactly as one at a time would.
// Ties change no load, so the result equals compute_prefill's assignment.
// A work item's setup and epilogue in key blocks' worth: a traced CTA spends about
// two block rounds at each change of work tile (Q load, first S, the last tile's
// epilogue).  With 2 instead of 1 the mixed batch's split moved from 68 to 72
// prefill CTAs and its launch from 170.3 to 168.3 us; prefill-only batches kept
// their times.
constexpr int64_t kItemOverhead = 2;
int64_t prefill_makespan(const std::vector<int64_t>& nb_tiles, int64_t total, int C, std::vector<int64_t>& by_cost,
                         std::vector<int64_t>& by_load) {
  if (C <= 0) return 0;
  const int64_t chunk = key_chunk(total, C);
  by_cost.assign(chunk + 1 + kItemOverhead, 0);
  int64_t items = 0;
  auto add = [&](int64_t c, int64_t m) {
    if (c >= static_cast<int64_t>(by_cost.size())) by_cost.resize(c + 1, 0);
    by_cost[c] += m;
    items += m;
  };
  for (int64_t nb = 0; nb < static_cast<int64_t>(nb_tiles.size()); ++nb) {
    const int64_t m = nb_tiles[nb];
    if (m == 0) continue;
    if (nb <= chunk) {
      add(std::max<int64_t>(nb, 1) + kItemOverhead, m);
    } else {
      const int64_t parts = ceil_div(nb, chunk);
      for (int64_t i = 0; i < parts; ++i) add((i + 1) * nb / parts - i * nb / parts + kItemOverhead, m);
    }
  }
  if (items == 0) return 0;
  const int64_t ctas = std::min<int64_t>(C, items);
  by_load.assign(1, ctas);
  int64_t least = 0, worst = 0;
  for (int64_t c = static_cast<int64_t>(by_cost.size()) - 1; c >= 1; --c) {
    int64_t k = by_cost[c];
    while (k > 0) {
      while (by_load[least] == 0) ++least;
      const int64_t take = std::min(k, by_load[least]);
      by_load[least] -= take;
      const int64_t l = least + c;
      if (l >= static_cast<int64_t>(by_load.size())) by_load.resize(l + 1, 0);
      by_load[l] += take;
      worst = std::max(worst, l);
      k -= take;
    }
  }
  return worst;
}

// Prefill work over `C` CTAs; with skip_single the requests holding one query
// row are left out (they are the decode half of a mixed batch).
pkv_status compute_prefill(pkv_plan* pl, int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                           const int32_t* kv_last, uint8_t* host, int C = 0, bool skip_single = false,
                           int page_size = 0) {
  const int P = page_size > 0 ? page_size : pl->p.page_size;
  const int BN = pkv::kPrefillKeys;
  if (C <= 0) C = pl->workers;

  PlanScratch& sc = pl->scratch;
  const int mp = pkv::kPrefillRows / pl->group;
  // Work items: one key chunk of one query tile each; the full table entry is
  // written only once the item has its place.
  std::vector<pkv::PlanItem>& items = sc.items;
  std::vector<int32_t>& item_cost = sc.item_cost;
  std::vector<PrefillMerge>& merges = sc.merges;
  items.clear();
  item_cost.clear();
  merges.clear();
  // Request b's custom-mask block starts at bit sum over b' < b of qo_len * kv_len.
  std::vector<int64_t>& mask_off = sc.mask_off;
  mask_off.assign(static_cast<size_t>(batch) + 1, 0);
  for (int b = 0; b < batch; ++b)
    mask_off[b + 1] = mask_off[b] + static_cast<int64_t>(qo_indptr[b + 1] - qo_indptr[b]) *
                                        kv_len_of(kv_indptr, kv_last, b, P);
  pl->mask_bits = mask_off[batch];
  const int64_t total = query_tile_blocks(pl, batch, qo_indptr, kv_indptr, kv_last, skip_single, nullptr, P);
  const int64_t chunk = key_chunk(total, C);
  // Each tile gives at most as many items as it counts blocks.
  items.reserve(static_cast<size_t>(std::min<int64_t>(total, pl->max_work) + 1));
  item_cost.reserve(items.capacity());
  int n_slot = 0;
  for (int b = 0; b < batch; ++b) {
    const int qo = qo_indptr[b + 1] - qo_indptr[b];
    if (skip_single && qo == 1) continue;
    const int kv = static_cast<int>(kv_len_of(kv_indptr, kv_last, b, P));
    for (int h = 0; h < pl->p.num_kv_heads; ++h)
      for (int pos0 = 0; pos0 < qo; pos0 += mp) {
        const int npos = std::min(mp, qo - pos0);
        const int kv_end = tile_kv_end(pl->p.causal, qo, kv, pos0, npos);
        const int64_t nb = ceil_div(kv_end, BN);
        if (nb <= chunk) {
          items.push_back({b, h, pos0, 0, kv_end, -1});
          item_cost.push_back(static_cast<int32_t>(std::max<int64_t>(nb, 1) + kItemOverhead));
          continue;
        }
        const int64_t parts = ceil_div(nb, chunk);
        PrefillMerge m{};
        m.b = b;
        m.kvh = h;
        m.q_row0 = qo_indptr[b] + pos0;
        m.n_pos = npos;
        m.slot_begin = n_slot;
        m.n_slots = static_cast<int32_t>(parts);
        merges.push_back(m);
        for (int64_t i = 0; i < parts; ++i) {
          const int64_t blo = i * nb / parts, bhi = (i + 1) * nb / parts;
          items.push_back({b, h, pos0, static_cast<int32_t>(blo * BN),
                           static_cast<int32_t>(std::min<int64_t>(bhi * BN, kv_end)), n_slot++});
          item_cost.push_back(static_cast<int32_t>(bhi - blo + kItemOverhead));
        }
      }
  }
  if ((int64_t)items.size() > pl->max_work || n_slot > pl->max_slots || (int)merges.size() > pl->max_merge)
    return PKV_ERR_WORKSPACE;

  // Longest processing time first onto the least-loaded CTA (ties: the lower
  // item, then the lower CTA).  Costs are small integers, so the items are
  // ordered by a stable counting sort on descending cost, and each CTA's list
  // is gathered afterwards by a stable counting pass over the assignment.
  const int n_items = static_cast<int>(items.size());
  int64_t max_c = 0;
  for (int32_t c : item_cost) max_c = std::max<int64_t>(max_c, c);
  std::vector<int>& start = sc.start;
  start.assign(static_cast<size_t>(max_c) + 2, 0);
  for (int32_t c : item_cost) ++start[static_cast<size_t>(max_c - c) + 1];
  for (size_t k = 1; k < start.size(); ++k) start[k] += start[k - 1];
  std::vector<int>& order = sc.order;
  order.resize(n_items);
  for (int i = 0; i < n_items; ++i) order[start[static_cast<size_t>(max_c - item_cost[i])]++] = i;
  const int ctas = static_cast<int>(std::min<int64_t>(C, (int64_t)n_items));
  std::vector<int64_t>& load = sc.load;
  load.assign(ctas, 0);
  std::vector<int>& cta_of = sc.cta_of;
  cta_of.resize(n_items);
  std::vector<int>& per_cta = sc.per_cta;
  per_cta.assign(static_cast<size_t>(ctas) + 1, 0);
  // The least-loaded CTA, ties to the lower index, without a heap: loads only
  // grow, the least load never falls, and every load lies within max_c of the
  // least one, so the CTAs sit in a ring of at least max_c + 1 buckets by load
  // (a power of two, indexed by the load's low bits), each a bitset over the
  // CTAs.  The lowest bit of the least non-empty bucket is the CTA a (load, cta)
  // min-heap would pop.
  const int words = (ctas + 63) / 64;
  int64_t ring = 1;
  while (ring < max_c + 1) ring <<= 1;
  std::vector<uint64_t>& buckets = sc.buckets;
  buckets.assign(static_cast<size_t>(ring * words), 0);
  for (int c = 0; c < ctas; ++c) buckets[c >> 6] |= uint64_t{1} << (c & 63);
  auto bucket = [&](int64_t l) { return &buckets[static_cast<size_t>((l & (ring - 1)) * words)]; };
  int64_t least = 0;
  for (int i : order) {
    uint64_t* bk = bucket(least);
    int w = 0;
    while (bk[w] == 0) ++w;
    const int c = w * 64 + __builtin_ctzll(bk[w]);
    bk[w] &= bk[w] - 1;
    cta_of[i] = c;
    ++per_cta[static_cast<size_t>(c) + 1];
    load[c] += item_cost[i];
    bucket(load[c])[c >> 6] |= uint64_t{1} << (c & 63);
    for (;;) {  // the next non-empty bucket (one exists: every CTA is in one)
      const uint64_t* b = bucket(least);
      bool any = false;
      for (int k = 0; k < words && !any; ++k) any = b[k] != 0;
      if (any) break;
      ++least;
    }
  }
  for (int c = 0; c < ctas; ++c) per_cta[static_cast<size_t>(c) + 1] += per_cta[c];
  std::vector<int>& by_cta = sc.by_cta;  // each CTA's items in the order they were assigned
  by_cta.resize(n_items);
  {
    std::vector<int>& fill = sc.fill;
    fill.assign(per_cta.begin(), per_cta.end() - 1);
    for (int i : order) by_cta[fill[cta_of[i]]++] = i;
  }

  auto* hdr = reinterpret_cast<PlanHeader*>(host + pl->L.header);
  auto* wptr = reinterpret_cast<int32_t*>(host + pl->L.worker_ptr);
  auto* mrec = reinterpret_cast<PrefillMerge*>(host + pl->L.merge);
  auto* work = reinterpret_cast<PrefillTile*>(host + pl->L.segs);
  int n = 0;
  pl->work_rows.assign(static_cast<size_t>(n_items) * 8, 0);
  pl->max_cost = 0;
  for (int c = 0; c < ctas; ++c) {
    wptr[c] = n;
    for (int k = per_cta[c]; k < per_cta[c + 1]; ++k) {
      const pkv::PlanItem& it = items[by_cta[k]];
      const int qo = qo_indptr[it.b + 1] - qo_indptr[it.b];
      PrefillTile t{};
      t.b = it.b;
      t.kvh = it.kvh;
      t.q_row0 = qo_indptr[it.b] + it.pos0;
      t.q_pos0 = it.pos0;
      t.n_pos = std::min(mp, qo - it.pos0);
      t.qo_len = qo;
      t.kv_len = static_cast<int32_t>(kv_len_of(kv_indptr, kv_last, it.b, P));
      t.kv_begin = it.kv_begin;
      t.kv_end = it.kv_end;
      t.idx_base = kv_indptr[it.b];
      t.last_rows = kv_last[it.b];
      t.slot = it.slot;
      t.mask_off = mask_off[it.b];
      work[n] = t;
      int32_t* r = &pl->work_rows[(size_t)n * 8];
      r[0] = c; r[1] = t.b; r[2] = t.kvh; r[3] = t.q_pos0; r[4] = t.n_pos;
      r[5] = t.kv_begin; r[6] = t.kv_end; r[7] = t.slot;
      ++n;
    }
    pl->max_cost = std::max(pl->max_cost, load[c]);
  }
  wptr[ctas] = n;
  for (size_t i = 0; i < merges.size(); ++i) mrec[i] = merges[i];

  std::memset(hdr, 0, sizeof(PlanHeader));
  hdr->kind = PKV_PLAN_PREFILL;
  hdr->batch = batch;
  hdr->num_workers = ctas;
  hdr->num_segments = n;
  hdr->num_merge = static_cast<int32_t>(merges.size());
  hdr->num_slots = n_slot;

  pl->active_workers = ctas;
  pl->num_work = n;
  pl->num_merge = static_cast<int>(merges.size());
  pl->num_slots = n_slot;
  int64_t tot = 0;
  for (int64_t v : load) tot += v;
  pl->total_cost = tot;
  pl->used_bytes = pl->L.segs + sizeof(PrefillTile) * (size_t)n;
  return PKV_OK;
}

// A prefill plan on pages of fewer than 8 rows: request b's L keys become
// ceil(L / 16) pages of 16 rows in the workspace's packed copy (page ids 0, 1, ...
// in request order), each with its source run of keys; the prefill tables are then
// planned over the packed page table as for 16-row pages.
pkv_status compute_packed(pkv_plan* pl, int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_last, uint8_t* host) {
  const int P = pl->p.page_size;
  PlanScratch& sc = pl->scratch;
  sc.pk_indptr.assign(static_cast<size_t>(batch) + 1, 0);
  sc.pk_last.assign(static_cast<size_t>(batch), 0);
  auto* ids = reinterpret_cast<int32_t*>(host + pl->L.pk_ids);
  auto* src = reinterpret_cast<pkv::PackedSrc*>(host + pl->L.pk_src);
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = kv_len_of(kv_indptr, kv_last, b, P);
    const int64_t np = ceil_div(L, 16);
    if (n + np > pl->max_packed) return PKV_ERR_WORKSPACE;
    sc.pk_indptr[b] = static_cast<int32_t>(n);
    sc.pk_last[b] = np > 0 ? static_cast<int32_t>(L - 16 * (np - 1)) : 0;
    // tok0 + L <= max_kv_pages * P (validate() bounds the listed pages), which the
    // size check at plan creation keeps far below 2^31.
    const int64_t tok0 = static_cast<int64_t>(kv_indptr[b]) * P;
    for (int64_t j = 0; j < np; ++j, ++n) {
      ids[n] = static_cast<int32_t>(n);
      src[n].tok0 = static_cast<int32_t>(tok0 + 16 * j);
      src[n].ntok = static_cast<int32_t>(std::min<int64_t>(16, L - 16 * j));
    }
  }
  sc.pk_indptr[batch] = static_cast<int32_t>(n);
  pkv_status st = compute_prefill(pl, batch, qo_indptr, sc.pk_indptr.data(), sc.pk_last.data(), host, 0, false, 16);
  if (st != PKV_OK) return st;
  reinterpret_cast<PlanHeader*>(host + pl->L.header)->num_packed = static_cast<int32_t>(n);
  return PKV_OK;
}

// Time of each half on n SMs, fitted to the two halves of a 60-decode +
// 4-prompt-chunk batch (32 q / 8 kv heads, head_dim 128, bf16) run alone on 20
// to 152 SMs: both follow a fixed part plus their plan's largest per-worker
// load to within 2 us.  Prefill: 13.8 us + 1.83 us per 128-key block of a
// 256-row tile on the busiest CTA (one extra block per work item).  Decode:
// 14.2 us + 1.38 us per 16-row page on the busiest warp.
constexpr double kPrefillFixedUs = 13.8;
constexpr double kPrefillBlockUs = 1.827;
constexpr double kDecodeFixedUs = 14.2;
constexpr double kDecodePage16Us = 1.384;

// Mixed batch: single-row requests to the decode half, the rest to the prefill
// half, and the SMs split so that both halves end together: the split that
// minimises the larger of the two estimated times (each half's time falls as
// it gains SMs, so the search brackets the crossing and then checks its
// neighbours, whose chunking can differ).
pkv_status compute_mixed(pkv_plan* pl, int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                         const int32_t* kv_last, int64_t num_pages, uint8_t* host) {
  const int P = pl->p.page_size;
  const int S = pl->num_sms;
  // Where single-row work runs on the tensor cores, every request goes to the
  // prefill half and the decode half is empty.
  const bool rows_to_prefill = decode_on_tensor_cores(&pl->p);
  int64_t dec_pages = 0;  // (request, kv head) pages of the decode half
  bool any_pre = false, any_dec = false;
  for (int b = 0; b < batch; ++b) {
    const int qo = qo_indptr[b + 1] - qo_indptr[b];
    const bool single = qo == 1 && !rows_to_prefill;
    any_dec |= single;
    any_pre |= qo >= 1 && !single;
    if (single) dec_pages += static_cast<int64_t>(kv_indptr[b + 1] - kv_indptr[b]) * pl->p.num_kv_heads;
  }
  int kp = 0;
  if (any_pre && !any_dec) {
    kp = S;
  } else if (any_pre && any_dec) {
    PlanScratch& sc = pl->scratch;
    std::vector<int64_t>& by_cost = sc.by_cost;
    std::vector<int64_t>& by_load = sc.by_load;
    std::vector<int64_t>& nb_tiles = sc.nb_tiles;  // tiles per count of key blocks
    const int64_t total = query_tile_blocks(pl, batch, qo_indptr, kv_indptr, kv_last, true, &nb_tiles);
    const double page_us = kDecodePage16Us * P / 16.0;
    auto t_pre = [&](int c) { return kPrefillFixedUs + kPrefillBlockUs * prefill_makespan(nb_tiles, total, c, by_cost, by_load); };
    auto t_dec = [&](int n) {
      const int64_t run = ceil_div(dec_pages, (int64_t)n * pkv::kDecodeWarps);
      return kDecodeFixedUs + page_us * run;
    };
    // Smallest prefill share whose prefill time no longer exceeds the decode time.
    int lo = 1, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi) / 2;
      if (t_pre(mid) <= t_dec(S - mid))
        hi = mid;
      else
        lo = mid + 1;
    }
    const int c0 = std::max(1, lo - 2), c1 = std::min(S - 1, lo + 2);
    double best = 0.0;
    kp = c0;
    for (int c = c0; c <= c1; ++c) {
      const double t = std::max(t_pre(c), t_dec(S - c));
      if (c == c0 || t < best) {
        best = t;
        kp = c;
      }
    }
    // The prefill load is a step function of the CTA count: take the fewest CTAs
    // that reach the same prefill time, leaving the decode half more SMs.
    const double target = t_pre(kp);
    int a = 1, z = kp;
    while (a < z) {
      const int mid = (a + z) / 2;
      if (t_pre(mid) <= target)
        z = mid;
      else
        a = mid + 1;
    }
    kp = a;
    // An even split: measured on a 60-decode + 4-chunk batch over splits 60 to
    // 81, odd splits ran up to 15% slower than their even neighbours, which fits
    // the SMs working in pairs (an odd number of prefill SMs must leave some
    // pair with one SM of each half).
    if ((kp & 1) && S >= 4) {
      const int lo_even = std::max(2, kp - 1), hi_even = std::min(S - 2, kp + 1);
      kp = std::max(t_pre(lo_even), t_dec(S - lo_even)) <= std::max(t_pre(hi_even), t_dec(S - hi_even)) ? lo_even
                                                                                                         : hi_even;
    }
  }
  pl->prefill_ctas = kp;
  pl->decode_ctas = any_dec ? S - kp : 0;
  pkv_plan* d = pl->sub_dec;
  pkv_plan* p = pl->sub_pre;
  pkv_status st = compute_decode(d, rows_to_prefill ? 0 : batch, kv_indptr, kv_last, host + pl->dec_host_off,
                                 qo_indptr, std::max(pl->decode_ctas, 1) * pkv::kDecodeWarps);
  if (st != PKV_OK) return st;
  st = compute_prefill(p, batch, qo_indptr, kv_indptr, kv_last, host + pl->pre_host_off, std::max(kp, 1),
                       !rows_to_prefill);
  if (st != PKV_OK) return st;
  // The mixed kernel's CTAs below this serve the prefill half, the rest the decode half.
  reinterpret_cast<PlanHeader*>(host + pl->dec_host_off + d->L.header)->cta_offset = any_dec ? kp : S;
  for (pkv_plan* q : {d, p}) {
    uint8_t* h = host + (q == d ? pl->dec_host_off : pl->pre_host_off);
    reinterpret_cast<PlanHeader*>(h + q->L.header)->num_pages = num_pages;
    q->batch = batch;
    q->num_pages = num_pages;
    q->total_q = batch > 0 ? qo_indptr[batch] : 0;
    q->planned = true;
  }
  pl->active_workers = p->active_workers + static_cast<int>(ceil_div(d->active_workers, pkv::kDecodeWarps));
  pl->num_work = d->num_work + p->num_work;
  pl->num_merge = d->num_merge + p->num_merge;
  pl->num_slots = d->num_slots + p->num_slots;
  pl->max_cost = 0;
  pl->total_cost = 0;
  pl->mask_bits = p->mask_bits;
  pl->work_rows = d->work_rows;
  pl->work_rows.insert(pl->work_rows.end(), p->work_rows.begin(), p->work_rows.end());
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_plan_create(pkv_plan** out, int kind, const pkv_params* params, const pkv_limits* limits,
                           int device) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  pkv_status st = make_plan(out, kind, params, limits, device, sms);
  if (st != PKV_OK) return st;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  cudaError_t e = cudaEventCreateWithFlags(&(*out)->copy_done, cudaEventDisableTiming);
  cudaSetDevice(prev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    pkv_plan_destroy(*out);
    *out = nullptr;
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status pkv_plan_create_host(pkv_plan** out, int kind, const pkv_params* params, const pkv_limits* limits,
                                int num_sms) {
  return make_plan(out, kind, params, limits, -1, num_sms);
}

pkv_status pkv_plan_destroy(pkv_plan* plan) {
  if (!plan) return PKV_ERR_INVALID_ARG;
  if (plan->copy_done) {
    if (plan->copy_pending) cudaEventSynchronize(plan->copy_done);
    cudaEventDestroy(plan->copy_done);
  }
  if (plan->copy_stream) {
    cudaStreamSynchronize(plan->copy_stream);
    cudaStreamDestroy(plan->copy_stream);
  }
  for (int r = 0; r < 2; ++r) {
    if (plan->copy_ev[r]) cudaEventDestroy(plan->copy_ev[r]);
    if (plan->free_ev[r]) cudaEventDestroy(plan->free_ev[r]);
  }
  delete plan->sub_dec;
  delete plan->sub_pre;
  delete plan;
  return PKV_OK;
}

pkv_status pkv_plan_workspace_bytes(const pkv_plan* plan, size_t* dev_bytes, size_t* host_bytes) {
  if (!plan) return PKV_ERR_INVALID_ARG;
  if (dev_bytes) *dev_bytes = plan->L.total;
  if (host_bytes) *host_bytes = plan->host_bytes;
  return PKV_OK;
}

pkv_status pkv_plan_compute(pkv_plan* plan, int batch, const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                            const int32_t* kv_indices_h, const int32_t* kv_last_page_len_h, int64_t num_pages,
                            void* host_ws, size_t host_ws_bytes) {
  if (!plan || !host_ws) return PKV_ERR_INVALID_ARG;
  if (host_ws_bytes < plan->host_bytes) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(host_ws) % 64) return PKV_ERR_INVALID_ARG;
  pkv_status st = validate(plan, batch, qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h, num_pages);
  if (st != PKV_OK) return st;
  if (plan->copy_pending) {
    cudaEventSynchronize(plan->copy_done);
    plan->copy_pending = false;
  }
  auto* host = static_cast<uint8_t*>(host_ws);
  if (plan->pipelined) {
    // Plan into the image the running kernels do not read; its last copy must be done.
    const int r = plan->cur ^ 1;
    if (plan->copy_pend[r]) {
      cudaEventSynchronize(plan->copy_ev[r]);
      plan->copy_pend[r] = false;
    }
    host += static_cast<size_t>(r) * plan->L.tables_end;
  }
  if (plan->kind == PKV_PLAN_MIXED) {
    st = compute_mixed(plan, batch, qo_indptr_h, kv_indptr_h, kv_last_page_len_h, num_pages, host);
  } else if (plan->kind == PKV_PLAN_DECODE && plan->exec_prefill) {
    // One query row per request: qo_indptr = 0, 1, ..., batch.
    std::vector<int32_t>& rows = plan->row_indptr;
    if (rows.size() < static_cast<size_t>(batch) + 1) {
      const size_t from = rows.size();
      rows.resize(static_cast<size_t>(batch) + 1);
      for (size_t i = from; i < rows.size(); ++i) rows[i] = static_cast<int32_t>(i);
    }
    st = compute_prefill(plan, batch, rows.data(), kv_indptr_h, kv_last_page_len_h, host);
  } else if (plan->kind == PKV_PLAN_DECODE) {
    st = compute_decode(plan, batch, kv_indptr_h, kv_last_page_len_h, host);
  } else if (plan->packed) {
    st = compute_packed(plan, batch, qo_indptr_h, kv_indptr_h, kv_last_page_len_h, host);
  } else {
    st = compute_prefill(plan, batch, qo_indptr_h, kv_indptr_h, kv_last_page_len_h, host);
  }
  if (st != PKV_OK) return st;
  // A packed plan's kernel reads the packed copy: its page-id check and its tensor
  // map span the copy's capacity (and an id of max_packed, past it, reads zeros).
  if (plan->kind != PKV_PLAN_MIXED)
    reinterpret_cast<PlanHeader*>(host + plan->L.header)->num_pages = plan->packed ? plan->max_packed : num_pages;
  plan->batch = batch;
  plan->num_pages = num_pages;
  plan->total_q = plan->kind == PKV_PLAN_DECODE ? batch : (batch > 0 ? qo_indptr_h[batch] : 0);
  plan->planned = true;
  return PKV_OK;
}

pkv_status pkv_plan_run(pkv_plan* plan, int batch, const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                        const int32_t* kv_indices_h, const int32_t* kv_last_page_len_h, int64_t num_pages,
                        void* dev_ws, size_t dev_ws_bytes, void* host_ws, size_t host_ws_bytes, void* stream) {
  if (!plan || !dev_ws) return PKV_ERR_INVALID_ARG;
  if (plan->device < 0) return PKV_ERR_INVALID_ARG;
  if (dev_ws_bytes < plan->L.total) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(dev_ws) % 256) return PKV_ERR_INVALID_ARG;
  pkv_status st = pkv_plan_compute(plan, batch, qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h,
                                   num_pages, host_ws, host_ws_bytes);
  if (st != PKV_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  bool ok = true;
  if (plan->pipelined) {
    const int r = plan->cur ^ 1;
    auto* dst = static_cast<uint8_t*>(dev_ws) + (r ? plan->L.alt : 0);
    auto* src = static_cast<uint8_t*>(host_ws) + static_cast<size_t>(r) * plan->L.tables_end;
    ok = (!plan->used[r] || cudaStreamWaitEvent(plan->copy_stream, plan->free_ev[r], 0) == cudaSuccess) &&
         cudaMemcpyAsync(dst, src, plan->used_bytes, cudaMemcpyHostToDevice, plan->copy_stream) == cudaSuccess &&
         cudaEventRecord(plan->copy_ev[r], plan->copy_stream) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      plan->planned = false;
      return PKV_ERR_CUDA;
    }
    plan->copy_pend[r] = true;
    plan->cur = r;
    return PKV_OK;
  }
  if (plan->kind == PKV_PLAN_MIXED) {
    auto* d = static_cast<uint8_t*>(dev_ws);
    auto* h = static_cast<uint8_t*>(host_ws);
    ok = cudaMemcpyAsync(d + plan->dec_dev_off, h + plan->dec_host_off, plan->sub_dec->used_bytes,
                         cudaMemcpyHostToDevice, s) == cudaSuccess &&
         cudaMemcpyAsync(d + plan->pre_dev_off, h + plan->pre_host_off, plan->sub_pre->used_bytes,
                         cudaMemcpyHostToDevice, s) == cudaSuccess;
  } else {
    ok = cudaMemcpyAsync(dev_ws, host_ws, plan->used_bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
  }
  if (!ok || cudaEventRecord(plan->copy_done, s) != cudaSuccess) {
    cudaGetLastError();
    plan->planned = false;
    return PKV_ERR_CUDA;
  }
  plan->copy_pending = true;
  return PKV_OK;
}

pkv_status pkv_plan_set_pipelined(pkv_plan* plan, int on) {
  if (!plan || plan->device < 0 || plan->kind == PKV_PLAN_MIXED || plan->planned) return PKV_ERR_INVALID_ARG;
  if (!on) {
    plan->pipelined = false;
    return PKV_OK;
  }
  if (!plan->copy_stream) {
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(plan->device);
    cudaError_t e = cudaStreamCreateWithFlags(&plan->copy_stream, cudaStreamNonBlocking);
    for (int r = 0; r < 2 && e == cudaSuccess; ++r) {
      e = cudaEventCreateWithFlags(&plan->copy_ev[r], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&plan->free_ev[r], cudaEventDisableTiming);
    }
    cudaSetDevice(prev);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
  }
  plan->pipelined = true;
  plan->cur = 1;  // the first plan_run fills image 0
  return PKV_OK;
}

pkv_status pkv_plan_set_split_kv(pkv_plan* plan, int on) {
  if (!plan || plan->kind != PKV_PLAN_DECODE) return PKV_ERR_INVALID_ARG;
  if (plan->exec_prefill && !on) return PKV_ERR_UNSUPPORTED;  // the switch is the CUDA-core decode schedule's
  plan->split_kv = on != 0;
  return PKV_OK;
}

pkv_status pkv_plan_get_info(const pkv_plan* plan, pkv_plan_info* info) {
  if (!plan || !info) return PKV_ERR_INVALID_ARG;
  info->grid_ctas = plan->grid_ctas;
  info->workers = plan->workers;
  info->active_workers = plan->active_workers;
  info->num_work = plan->num_work;
  info->num_merge = plan->num_merge;
  info->num_slots = plan->num_slots;
  info->max_cost = plan->max_cost;
  info->total_cost = plan->total_cost;
  info->prefill_ctas = plan->kind == PKV_PLAN_MIXED ? plan->prefill_ctas : 0;
  info->decode_ctas = plan->kind == PKV_PLAN_MIXED ? plan->decode_ctas : 0;
  return PKV_OK;
}

pkv_status pkv_plan_get_work(const pkv_plan* plan, int32_t* out, int64_t capacity, int64_t* rows_written) {
  if (!plan) return PKV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(plan->work_rows.size() / 8);
  if (rows_written) *rows_written = rows;
  if (!out) return rows == 0 ? PKV_OK : PKV_ERR_INVALID_ARG;
  if (capacity < rows) return PKV_ERR_WORKSPACE;
  std::memcpy(out, plan->work_rows.data(), plan->work_rows.size() * sizeof(int32_t));
  return PKV_OK;
}

}  // extern "C"
