// pkv_internal.h -- tables the host plan writes and the kernels read.
//
// The plan (fdeinterviews summary, "Load balancing that survives CUDA
// graphs") is computed on the host from the index arrays and copied once into
// the caller's device workspace.  Kernels read everything that depends on the
// batch from these tables, never from launch arguments, so a captured graph
// stays valid after re-planning a different batch within the same limits.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Device error word bits (OR-ed together; read with pkv_get_device_error).
enum : int {
  kErrPageIndex = 1,     // a page id outside [0, num_pages) reached a kernel
  kErrIndptrMismatch = 2,// kv_indptr on the device differs from the plan's host copy
  kErrWaitTimeout = 4,   // a bounded wait on an mbarrier ran out
  kErrTmemAlloc = 8,     // tensor-memory allocation failed
  kErrAppendLayout = 16, // append: a row outside every request's new rows, more new
                         // tokens than the request's kv_len, or a bad last-page length
};

struct alignas(64) PlanHeader {
  int32_t kind;          // pkv_plan_kind
  int32_t batch;
  int32_t num_workers;   // workers (decode: warps, prefill: CTAs) that have work
  int32_t num_segments;  // entries of the segment table
  int32_t num_merge;     // split items whose partial states need a merge
  int32_t num_slots;     // partial-state slots in use
  int64_t num_pages;     // pool size, for the device-side page-id check
  int32_t error;         // device error word; cleared by every plan_run
  int32_t cta_offset;    // mixed plans, decode half: the first CTA of the mixed launch
                         // that serves it (CTAs below it serve the prefill half); 0 otherwise
  int32_t num_packed;    // prefill plans on pages of fewer than 8 rows: 16-row pages in the
                         // packed copy of the requests' K/V (0 otherwise)
  int32_t pad[3];
};
static_assert(sizeof(PlanHeader) == 64, "PlanHeader layout");

// One contiguous run of one (request, kv head)'s pages, handled by one decode
// worker.  slot < 0: the run is the whole sequence and writes the output
// directly; otherwise it writes an fp32 partial state into that slot.
struct alignas(32) DecodeSeg {
  int32_t b;           // request
  int32_t kvh;         // kv head
  int32_t idx_begin;   // first entry of kv_indices (= kv_indptr[b] + page_begin)
  int32_t n_pages;     // pages in the run (0: empty request, write o = 0, lse = -inf)
  int32_t last_rows;   // valid slots of the run's final page
  int32_t page_begin;  // position of the run's first page in the request
  int32_t slot;        // partial slot, or -1
  int32_t q_row;       // row of q / o / lse (the request itself in a decode batch; its
                       // qo_indptr entry in a mixed prefill + decode batch)
};
static_assert(sizeof(DecodeSeg) == 32, "DecodeSeg layout");

// A (request, kv head) whose sequence was split into n_slots partial states.
struct alignas(16) MergeItem {
  int32_t row;         // row of o / lse
  int32_t kvh;
  int32_t slot_begin;
  int32_t n_slots;
};
static_assert(sizeof(MergeItem) == 16, "MergeItem layout");

// One prefill work tile: up to 128 packed query rows (query positions x the
// heads of one kv head's group) of one request, against the key range
// [kv_begin, kv_end) of that request.  slot >= 0 when the key range is one
// chunk of a split sequence.
struct alignas(64) PrefillTile {
  int32_t b;
  int32_t kvh;
  int32_t q_row0;      // first global query row (into q / qo_indptr numbering)
  int32_t q_pos0;      // position of that row within its request
  int32_t n_pos;       // query positions in the tile (rows = n_pos * group)
  int32_t qo_len;      // rows of the request
  int32_t kv_len;      // keys of the request
  int32_t kv_begin;    // key range of this tile (multiple of the KV tile size)
  int32_t kv_end;      //   (already clipped by the causal limit)
  int32_t idx_base;    // kv_indptr[b]
  int32_t last_rows;   // kv_last_page_len[b]
  int32_t slot;        // partial slot or -1
  int32_t pad[2];
  int64_t mask_off;    // bit offset of the request's [qo_len, kv_len] custom-mask block
};
static_assert(sizeof(PrefillTile) == 64, "PrefillTile layout");

// Prefill merge record: a query tile whose key range was split into n_slots
// chunks; its rows are combined from the partial slots.
struct alignas(32) PrefillMerge {
  int32_t b;
  int32_t kvh;
  int32_t q_row0;
  int32_t n_pos;
  int32_t slot_begin;
  int32_t n_slots;
  int32_t pad[2];
};
static_assert(sizeof(PrefillMerge) == 32, "PrefillMerge layout");

// Byte offsets of the regions inside the device workspace.
// Packed prefill plans: where the 16 rows of packed page p come from, the
// request's keys tok0 .. tok0 + ntok - 1 counted from its first kv_indices entry
// times the page size (so token u is row u % P of page kv_indices[u / P]).
struct PackedSrc {
  int32_t tok0;
  int32_t ntok;        // 1 .. 16
};
static_assert(sizeof(PackedSrc) == 8, "PackedSrc layout");

struct WorkspaceLayout {
  size_t header;       // PlanHeader
  size_t worker_ptr;   // int32 [max_workers + 1]
  size_t merge;        // MergeItem / PrefillMerge [max_merge]
  size_t pk_ids;       // packed prefill plans: int32 [max_packed], page p's id p
  size_t pk_src;       // packed prefill plans: PackedSrc [max_packed]
  size_t segs;         // DecodeSeg [max_segments]  or PrefillTile [max_tiles]
  size_t tables_end;   // everything above is copied from the pinned host buffer
  size_t part_o;       // fp32 [max_slots][rows_per_slot][head_dim]
  size_t part_lse;     // fp32 [max_slots][rows_per_slot]
  size_t pk_kv;        // packed prefill plans: [max_packed, 2, Hkv, 16, D] copy of the K/V rows
  size_t alt;          // a second copy of the tables [0, tables_end), for pipelined plans
  size_t total;
};

}  // namespace pkv
