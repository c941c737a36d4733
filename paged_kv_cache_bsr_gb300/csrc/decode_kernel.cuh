// decode_kernel.cuh -- the decode worker (one warp streaming its own pages),
// shared by the decode kernel (decode.cu) and the mixed prefill + decode kernel
// (mixed_kernel.cuh).
//
// Batch decode over a paged KV cache, split-KV capable.
//
// Method (FlashInfer pages): the kernel follows each request's page table to
// gather K/V from non-contiguous pages ("FlashInfer" guide, section 2
// "Page-Level Attention"), computes one query token's attention for all query
// heads of one kv head at once (greptalks summary, "Head Group Packing"), and,
// when the host plan split a long sequence into chunks, writes each chunk's
// partial output with its log-sum-exp so a merge can combine them (guide,
// section 3 "FlashDecoding"; fdeinterviews, "Load balancing").
//
// GB300 design.  Decode reads every K/V byte once, so it is HBM-bound
// (about half a flop per byte at a group of 4).  One CTA per SM holds
// kDecodeWarps independent workers (warps).  Each warp owns a ring of page
// tiles in shared memory (24 KB) that its lane 0 fills with TMA bulk copies
// (cp.async.bulk, completion on an mbarrier): one copy for the tile's K rows
// and one for its V rows, each a contiguous 16-row x head_dim block of a page.
// With one-row pages the tile's rows come instead as four-row tensor gathers
// (tile::gather4) over kv_data viewed as a 2-D tensor of rows.
// The copies run ahead of the compute by the depth of the ring, so every SM
// keeps up to 192 KB of reads in flight.  A warp works through the list of
// (request, kv head, page range) segments the plan gave it, back to back, so
// the ring never drains between segments.
//
// Inside a tile, LPT lanes share one token (each holding D/LPT dims as
// 16-byte chunks, interleaved so a quarter-warp reads 128 contiguous bytes),
// 32/LPT tokens go per step, scores are summed with xor-shuffles inside the
// token group, and the online softmax keeps (max, sum, o) per head in
// registers, with max and o rescaled only when a tile raises the max.
#pragma once
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_bsr.h"

namespace pkv {
namespace decode_impl {

constexpr unsigned kFull = 0xffffffffu;

template <int D, typename T>
struct DecodeShape {
  static constexpr int kTileBytes = kDecodeTileRows * D * 2;  // K (or V) rows of one tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = kDecodeWarpSmem / kStageBytes;
  static_assert(kStages >= 2, "ring too shallow");
};

struct SegInfo {
  int b, kvh, idx_begin, n_pages, last_rows, page_begin, slot, q_row;
};

__device__ __forceinline__ SegInfo load_seg(const DecodeSeg* segs, int i, int lane) {
  const int v = lane < 8 ? reinterpret_cast<const int32_t*>(segs + i)[lane] : 0;
  SegInfo s;
  s.b = __shfl_sync(kFull, v, 0);
  s.kvh = __shfl_sync(kFull, v, 1);
  s.idx_begin = __shfl_sync(kFull, v, 2);
  s.n_pages = __shfl_sync(kFull, v, 3);
  s.last_rows = __shfl_sync(kFull, v, 4);
  s.page_begin = __shfl_sync(kFull, v, 5);
  s.slot = __shfl_sync(kFull, v, 6);
  s.q_row = __shfl_sync(kFull, v, 7);
  return s;
}

// The copy side of a warp's ring: walks the same (segment, 16-token tile)
// sequence as the compute side, S tiles ahead of it.  A tile is 16 consecutive
// tokens of the segment; with pages of 16 rows or more it lies in one page (one
// bulk copy each for K and V), with smaller pages it spans several, one lane per
// page.  Page ids come from a 32-entry window of kv_indices held one per lane.
struct Producer {
  int seg, seg_end;
  int tok, n_tok;
  int idx_begin, kvh;
  int win_base, win;
  int win_next;  // one-row pages: the window after `win`, loaded a window ahead
  int issued;
};

__device__ __forceinline__ int seg_tokens(int n_pages, int last_rows, int P) {
  return n_pages > 0 ? (n_pages - 1) * P + last_rows : 0;
}

template <int D, typename T, bool GATHER>
__device__ __forceinline__ void producer_enter(Producer& p, const DecodeArgs& a, int lane) {
  const SegInfo s = load_seg(a.segs, p.seg, lane);
  p.idx_begin = s.idx_begin;
  p.n_tok = seg_tokens(s.n_pages, s.last_rows, a.page_size);
  p.kvh = s.kvh;
  p.tok = 0;
  p.win_base = 0;
  p.win = lane < s.n_pages ? __ldg(a.kv_indices + p.idx_begin + lane) : 0;
  // One-row pages also hold the next window, loaded a window ahead (the gather
  // path's tiles are 16 pages each, so a window lasts only two of them).
  if constexpr (GATHER) p.win_next = 32 + lane < s.n_pages ? __ldg(a.kv_indices + p.idx_begin + 32 + lane) : 0;
}

// Issue the next tile of the warp's stream into its stage; false when done.
// GATHER (one-row pages): the tile's rows come as four-row tensor gathers, four
// for K (lanes 0-3) and four for V (lanes 4-7), instead of one 256-byte bulk copy
// per page and K|V.
template <int D, typename T, bool GATHER>
__device__ __forceinline__ bool producer_issue(Producer& p, const DecodeArgs& a, uint8_t* ring,
                                               uint32_t bar0, int lane, int64_t num_pages,
                                               uint64_t policy) {
  using Shape = DecodeShape<D, T>;
  while (p.seg < p.seg_end) {
    if (p.tok < p.n_tok) {
      const int rows = min(kDecodeTileRows, p.n_tok - p.tok);
      const int stage = p.issued % Shape::kStages;
      const uint32_t dst = smem_addr(ring + stage * Shape::kStageBytes);
      const uint32_t bar = bar0 + 8 * stage;
      if constexpr (GATHER) {
        static_assert(kDecodeGatherMaxRows == 1, "the gather path takes one-row pages only");
        // One-row pages: token = page.  A tile of 16 tokens never straddles two
        // 32-id windows, and the next window was loaded one window earlier, so
        // the id load's latency hides behind two tiles of work.
        if (p.tok - p.win_base >= 32) {
          p.win_base += 32;
          p.win = p.win_next;
          const int k = p.win_base + 32 + lane;
          p.win_next = k < p.n_tok ? __ldg(a.kv_indices + p.idx_begin + k) : 0;
        }
        // Every gather writes four whole rows (rows past the segment, or of a bad
        // page id, as zeros from past the tensor), so the stage always gets a full tile.
        if (lane == 0) mbar_arrive_expect_tx(bar, 2u * kDecodeTileRows * D * sizeof(T));
        __syncwarp();
        const int q4 = lane & 3, sel = (lane >> 2) & 1;  // four tokens' rows of K (sel 0) or V (1)
        const int w0 = p.tok - p.win_base + 4 * q4;      // window slot of this lane's first token
        int rowi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int page_id = __shfl_sync(kFull, p.win, (w0 + i) & 31);
          rowi[i] = a.kv_rows_n;
          if (4 * q4 + i < rows) {
            if (page_id >= 0 && page_id < num_pages)
              rowi[i] = (page_id * 2 + sel) * a.num_kv_heads + p.kvh;
            else if (lane < 8)
              atomicOr(a.err, kErrPageIndex);
          }
        }
        if (lane < 8)
          tma_gather4(dst + sel * Shape::kTileBytes + q4 * 4 * D * static_cast<int>(sizeof(T)), &a.kv_rows, 0,
                      rowi[0], rowi[1], rowi[2], rowi[3], bar);
        ++p.issued;
        p.tok += rows;
        return true;
      }
      const int P = a.page_size;
      // Pages the tile overlaps: a shift for power-of-two page sizes (a division by a
      // run-time divisor costs the warp about twenty instructions per tile).
      int pa, pb;
      if ((P & (P - 1)) == 0) {
        const int lp = __ffs(P) - 1;
        pa = p.tok >> lp;
        pb = (p.tok + rows - 1) >> lp;
      } else {
        pa = p.tok / P;
        pb = (p.tok + rows - 1) / P;
      }
      if (pb - p.win_base >= 32) {
        p.win_base = pa;
        const int n_pages = (p.n_tok + P - 1) / P;
        p.win = (pa + lane < n_pages) ? __ldg(a.kv_indices + p.idx_begin + pa + lane) : 0;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar, 2u * rows * D * sizeof(T));
      __syncwarp();
      const int k = pa + lane;  // this lane's page
      int page_id = __shfl_sync(kFull, p.win, min(k - p.win_base, 31));
      if (k <= pb) {
        if (page_id < 0 || page_id >= num_pages) {
          atomicOr(a.err, kErrPageIndex);
          page_id = 0;
        }
        const int r_lo = max(p.tok, k * P) - k * P;           // rows of the page inside the tile
        const int r_hi = min(p.tok + rows, (k + 1) * P) - k * P;
        const uint32_t bytes = static_cast<uint32_t>(r_hi - r_lo) * D * sizeof(T);
        const uint32_t off = static_cast<uint32_t>(k * P + r_lo - p.tok) * D * sizeof(T);
        const T* kv = static_cast<const T*>(a.kv);
        const int64_t head_rows = static_cast<int64_t>(P) * D;  // elements of one (page, K|V, head)
        const T* k_src = kv + ((static_cast<int64_t>(page_id) * 2 + 0) * a.num_kv_heads + p.kvh) * head_rows +
                         static_cast<int64_t>(r_lo) * D;
        const T* v_src = k_src + static_cast<int64_t>(a.num_kv_heads) * head_rows;
        bulk_copy_g2s_hint(dst + off, k_src, bytes, bar, policy);
        bulk_copy_g2s_hint(dst + Shape::kTileBytes + off, v_src, bytes, bar, policy);
      }
      ++p.issued;
      p.tok += rows;
      return true;
    }
    ++p.seg;
    if (p.seg < p.seg_end) producer_enter<D, T, GATHER>(p, a, lane);
  }
  return false;
}

// Head owned by lane slice `sub` after reduce_scatter<G, LPT>.
template <int G, int LPT>
__device__ __forceinline__ int owned_head(int sub) {
  int h = 0, n = G;
#pragma unroll
  for (int o = LPT / 2; o >= 1; o >>= 1)
    if (n > 1) {
      if (sub & o) h += n / 2;
      n /= 2;
    }
  return h;
}

// Lane slice (within a token group) that owns head g.
template <int G, int LPT>
__device__ __forceinline__ int owner_of_head(int g) {
  int sub = 0, n = G;
#pragma unroll
  for (int o = LPT / 2; o >= 1; o >>= 1)
    if (n > 1) {
      if (g >= n / 2) {
        sub |= o;
        g -= n / 2;
      }
      n /= 2;
    }
  return sub;
}

// Sum G per-head partial dots over the LPT lanes of a token group.  Each
// xor-round halves the number of heads a lane carries (it keeps one half and
// sends the other), so G heads cost G-1 + log2(LPT/G) shuffles instead of
// G*log2(LPT); the lane ends with the full sum of head owned_head<G,LPT>(sub).
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter(const float (&v)[G], int sub) {
  float cur[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cur[g] = v[g];
  int n = G;
#pragma unroll
  for (int o = LPT / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (sub & o) != 0;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? cur[i] : cur[i + n / 2];
          const float keep = upper ? cur[i + n / 2] : cur[i];
          cur[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
      }
      n /= 2;
    } else {
      cur[0] += __shfl_xor_sync(kFull, cur[0], o);
    }
  }
  return cur[0];
}

// One 16-row tile of K and V in shared memory: scores of the owned head per
// step, the tile max, a rescale of O only when some head's max grows by more
// than 2^8 over its reference (so p stays <= 256 and most tiles skip it), then
// P V with packed FMAs.  FULL: all 16 rows valid, no per-token checks.
template <int D, int G, int LPT, typename T, bool CAP, bool FULL>
__device__ __forceinline__ void tile_step(const DecodeArgs& a, const T* ks, const T* vs, int rows, int sub, int grp,
                                          int my_head, const float2 (&qf)[G][D / LPT / 2], float (&m)[G],
                                          float& m_own, float& l_own, float2 (&acc)[G][D / LPT / 2]) {
  constexpr int VEC = D / LPT;
  constexpr int CH = VEC / 8;
  constexpr int TPS = 32 / LPT;
  constexpr int STEPS = kDecodeTileRows / TPS;
  float sc[STEPS];
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int tok = st * TPS + grp;
    // two partial sums per head: half-length FMA chains
    float2 pa[G], pb[G];
#pragma unroll
    for (int g = 0; g < G; ++g) pa[g] = pb[g] = make_float2(0.f, 0.f);
    if (FULL || tok < rows) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        float2 kf[4];
        to_float2x4<T>(*reinterpret_cast<const uint4*>(ks + tok * D + (sub + c * LPT) * 8), kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          pa[g] = ffma2(qf[g][c * 4 + 0], kf[0], pa[g]);
          pb[g] = ffma2(qf[g][c * 4 + 1], kf[1], pb[g]);
          pa[g] = ffma2(qf[g][c * 4 + 2], kf[2], pa[g]);
          pb[g] = ffma2(qf[g][c * 4 + 3], kf[3], pb[g]);
        }
      }
    }
    float part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 t = fadd2(pa[g], pb[g]);
      part[g] = t.x + t.y;
    }
    float x = reduce_scatter<G, LPT>(part, sub);
    if constexpr (CAP) x = a.cap * kLog2e * tanh_from_log2(x * (2.f * kLog2e / a.cap));
    sc[st] = (FULL || tok < rows) ? x : -INFINITY;
  }
  // Tile max of the owned head over the token groups.
  float mx = sc[0];
#pragma unroll
  for (int st = 1; st < STEPS; ++st) mx = fmaxf(mx, sc[st]);
  mx = warp_max(mx, 16, LPT);
  const bool grow = (m_own == -INFINITY) ? (mx != -INFINITY) : (mx > m_own + 8.f);
  if (__any_sync(kFull, grow)) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mg = __shfl_sync(kFull, mx, owner_of_head<G, LPT>(g));
      const bool up = (m[g] == -INFINITY) ? (mg != -INFINITY) : (mg > m[g] + 8.f);
      if (up) {
        const float alpha = fast_exp2(m[g] - mg);  // 0 while m[g] is -inf
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int v = 0; v < VEC / 2; ++v) acc[g][v] = fmul2(acc[g][v], a2);
        if (g == my_head) l_own *= alpha;
        m[g] = mg;
      }
      if (g == my_head) m_own = m[g];
    }
  }
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int tok = st * TPS + grp;
    const float p_own = fast_exp2(sc[st] - m_own);  // 0 for a masked token
    l_own += p_own;
    float2 p2[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float pg_ = __shfl_sync(kFull, p_own, grp * LPT + owner_of_head<G, LPT>(g));
      p2[g] = make_float2(pg_, pg_);
    }
    if (FULL || tok < rows) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        float2 vf[4];
        to_float2x4<T>(*reinterpret_cast<const uint4*>(vs + tok * D + (sub + c * LPT) * 8), vf);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[g][c * 4 + e] = ffma2(p2[g], vf[e], acc[g][c * 4 + e]);
      }
    }
  }
}


// One decode worker: the calling warp initialises the S barriers at bar0
// (shared-memory address) and streams the segments the plan gave `worker`
// through its ring of S stages of K and V tiles at `ring`.  Warps are
// independent: nothing here synchronises beyond the calling warp.
template <int D, int G, int LPT, typename T, bool CAP, bool GATHER>
__device__ __forceinline__ void decode_worker(const DecodeArgs& a, int worker, uint8_t* ring, uint32_t bar0) {
  using Shape = DecodeShape<D, T>;
  constexpr int S = Shape::kStages;
  constexpr int VEC = D / LPT;     // dims per lane
  constexpr int CH = VEC / 8;      // 16-byte chunks per lane per row
  constexpr int TPS = 32 / LPT;    // tokens per step
  static_assert(CH >= 1 && VEC % 8 == 0, "lane slice must be whole 16-byte chunks");
  static_assert(kDecodeTileRows % TPS == 0, "steps must tile the 16 rows");
  static_assert(G <= LPT, "every head needs an owning lane in the token group");

  const int lane = threadIdx.x & 31;
  const int sub = lane % LPT;   // dim slice of this lane
  const int grp = lane / LPT;   // token slot of this lane within a step
  const int my_head = owned_head<G, LPT>(sub);

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const PlanHeader* hdr = a.hdr;
  if (worker >= hdr->num_workers) return;
  const int64_t num_pages = hdr->num_pages;
  const int seg_begin = a.worker_ptr[worker];
  const int seg_end = a.worker_ptr[worker + 1];
  if (seg_begin >= seg_end) return;
  const uint64_t policy = l2_policy_evict_first();

  Producer prod;
  prod.seg = seg_begin;
  prod.seg_end = seg_end;
  prod.issued = 0;
  producer_enter<D, T, GATHER>(prod, a, lane);
  for (int s = 0; s < S; ++s)
    if (!producer_issue<D, T, GATHER>(prod, a, ring, bar0, lane, num_pages, policy)) break;

  int consumed = 0;
  bool ok = true;
  const T* q_all = static_cast<const T*>(a.q);

  for (int si = seg_begin; si < seg_end && ok; ++si) {
    const SegInfo sg = load_seg(a.segs, si, lane);
    const int hq0 = sg.kvh * G;
    int indptr_seen = 0;
    if (lane == 0) indptr_seen = __ldg(a.kv_indptr + sg.b);

    // Query rows of the head group as fp32 pairs, pre-scaled (log2 domain without a cap).
    float2 qf[G][VEC / 2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const T* qrow = q_all + (static_cast<int64_t>(sg.q_row) * a.num_qo_heads + hq0 + g) * D;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        float2 f[4];
        to_float2x4<T>(ld_nc_v4(qrow + (sub + c * LPT) * 8), f);
#pragma unroll
        for (int e = 0; e < 4; ++e) qf[g][c * 4 + e] = make_float2(f[e].x * a.q_scale, f[e].y * a.q_scale);
      }
    }
    float m[G];        // reference max per head (warp-uniform), log2 units
    float m_own = -INFINITY;  // m[] of the head this lane owns
    float l_own = 0.f; // running sum of the owned head over this lane's tokens
    float2 acc[G][VEC / 2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
#pragma unroll
      for (int v = 0; v < VEC / 2; ++v) acc[g][v] = make_float2(0.f, 0.f);
    }

    // 16-token tiles of the segment, in the producer's order.
    const int n_tok = seg_tokens(sg.n_pages, sg.last_rows, a.page_size);
    for (int tok0 = 0; tok0 < n_tok; tok0 += kDecodeTileRows) {
      const int rows = min(kDecodeTileRows, n_tok - tok0);
      const int stage = consumed % S;
      if (!mbar_wait(bar0 + 8 * stage, (consumed / S) & 1, a.err)) {
        ok = false;
        break;
      }
      const T* ks = reinterpret_cast<const T*>(ring + stage * Shape::kStageBytes);
      const T* vs = ks + kDecodeTileRows * D;
      // Full tiles (every tile but the last of a segment) skip the per-token checks.
      if (rows == kDecodeTileRows)
        tile_step<D, G, LPT, T, CAP, true>(a, ks, vs, rows, sub, grp, my_head, qf, m, m_own, l_own, acc);
      else
        tile_step<D, G, LPT, T, CAP, false>(a, ks, vs, rows, sub, grp, my_head, qf, m, m_own, l_own, acc);
      ++consumed;
      __syncwarp();
      producer_issue<D, T, GATHER>(prod, a, ring, bar0, lane, num_pages, policy);
    }
    if (!ok) break;

    // Combine the token groups: every lane ends with the full sums of its dims,
    // and the owner lanes with the full softmax denominator of their head.
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) {
      l_own += __shfl_xor_sync(kFull, l_own, o);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int v = 0; v < VEC / 2; ++v) {
          acc[g][v].x += __shfl_xor_sync(kFull, acc[g][v].x, o);
          acc[g][v].y += __shfl_xor_sync(kFull, acc[g][v].y, o);
        }
    }

    if (lane == 0 && indptr_seen != sg.idx_begin - sg.page_begin) atomicOr(a.err, kErrIndptrMismatch);

    const bool empty = sg.n_pages == 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float lg = __shfl_sync(kFull, l_own, owner_of_head<G, LPT>(g));
      if (g % TPS != grp) continue;
      const float inv = empty ? 0.f : 1.f / lg;
      const float lse_v = empty ? -INFINITY : (m[g] + log2f(lg)) * kLn2;
      if (sg.slot < 0) {
        T* orow = static_cast<T*>(a.o) + (static_cast<int64_t>(sg.q_row) * a.num_qo_heads + hq0 + g) * D;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            f[2 * e] = acc[g][c * 4 + e].x * inv;
            f[2 * e + 1] = acc[g][c * 4 + e].y * inv;
          }
          *reinterpret_cast<uint4*>(orow + (sub + c * LPT) * 8) = from_float8<T>(f);
        }
        if (sub == 0 && a.lse) a.lse[static_cast<int64_t>(sg.q_row) * a.num_qo_heads + hq0 + g] = lse_v;
      } else {
        float* prow = a.part_o + (static_cast<int64_t>(sg.slot) * G + g) * D;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          float4* dst = reinterpret_cast<float4*>(prow + (sub + c * LPT) * 8);
          dst[0] = make_float4(acc[g][c * 4 + 0].x * inv, acc[g][c * 4 + 0].y * inv,
                               acc[g][c * 4 + 1].x * inv, acc[g][c * 4 + 1].y * inv);
          dst[1] = make_float4(acc[g][c * 4 + 2].x * inv, acc[g][c * 4 + 2].y * inv,
                               acc[g][c * 4 + 3].x * inv, acc[g][c * 4 + 3].y * inv);
        }
        if (sub == 0) a.part_lse[static_cast<int64_t>(sg.slot) * G + g] = lse_v;
      }
    }
  }

  if (!ok) {
    // A wait ran out: let this warp's copies still in flight land before the
    // CTA's shared memory is released, each wait again bounded.
    for (int t = consumed + 1; t < prod.issued; ++t)
      if (!mbar_wait(bar0 + 8 * (t % S), (t / S) & 1, a.err)) break;
  }
}

template <int D, int G, int LPT, typename T, bool CAP, bool GATHER>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int S = DecodeShape<D, T>::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kDecodeWarps][S];
  // Launched as a programmatic dependent of the kernel before it on the stream:
  // nothing global is touched before that grid has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  decode_worker<D, G, LPT, T, CAP, GATHER>(a, blockIdx.x * kDecodeWarps + warp, smem + warp * kDecodeWarpSmem,
                                           smem_addr(&bars[warp][0]));
}

// n-way merge of the partial states of one split (request, kv head) sequence for
// one head of its group (pair = item * G + head), by the calling warp: lanes over
// head_dim, the slot loop unrolled so that several partial rows are in flight per
// lane.  Shared by the decode merge kernel and the mixed batch's merge kernel.
template <int D, int G, typename T>
__device__ __forceinline__ void decode_merge_pair(const DecodeArgs& a, int pair, int lane) {
  constexpr int PER = D / 32;  // dims per lane
  constexpr int U = 8;         // slots in flight per lane
  const MergeItem it = a.merge[pair / G];
  const int g = pair % G;
  const int n = it.n_slots;
  const float* lse_p = a.part_lse + static_cast<int64_t>(it.slot_begin) * G + g;
  const float* o_p = a.part_o + (static_cast<int64_t>(it.slot_begin) * G + g) * D + lane * PER;
  // Rows of slots i0 .. i0 + U - 1 (zeros past the last slot).
  auto load_rows = [&](int i0, float (&vals)[U][PER]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u < n) {
        const float* src = o_p + static_cast<int64_t>(i0 + u) * G * D;
        if constexpr (PER == 4) {
          const float4 t = *reinterpret_cast<const float4*>(src);
          vals[u][0] = t.x; vals[u][1] = t.y; vals[u][2] = t.z; vals[u][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(src);
          vals[u][0] = t.x; vals[u][1] = t.y;
        }
      } else {
#pragma unroll
        for (int v = 0; v < PER; ++v) vals[u][v] = 0.f;
      }
    }
  };
  // The first rows do not depend on the lse values: they load together with them,
  // so the merge waits for two dependent loads (item, then lse and rows), not three.
  float vals[U][PER];
  load_rows(0, vals);
  const float l0 = lane < n ? lse_p[static_cast<int64_t>(lane) * G] : -INFINITY;
  float mx = l0;
  for (int i = lane + 32; i < n; i += 32) mx = fmaxf(mx, lse_p[static_cast<int64_t>(i) * G]);
  mx = warp_max(mx);
  float acc[PER];
#pragma unroll
  for (int v = 0; v < PER; ++v) acc[v] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int i0 = 0; i0 < n; i0 += 32) {
      // lane j holds the weight of slot i0 + j
      const float l = i0 == 0 ? l0 : (i0 + lane < n ? lse_p[static_cast<int64_t>(i0 + lane) * G] : -INFINITY);
      const float w_lane = i0 + lane < n ? fast_exp2((l - mx) * kLog2e) : 0.f;
      const int cnt = min(32, n - i0);
      for (int j0 = 0; j0 < cnt; j0 += U) {
        if (i0 + j0 > 0) load_rows(i0 + j0, vals);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float w = __shfl_sync(kFull, w_lane, (j0 + u) & 31);
          if (j0 + u < cnt) {
#pragma unroll
            for (int v = 0; v < PER; ++v) acc[v] = fmaf(w, vals[u][v], acc[v]);
            wsum += w;
          }
        }
      }
    }
  }
  const int hq = it.kvh * G + g;
  T* orow = static_cast<T*>(a.o) + (static_cast<int64_t>(it.row) * a.num_qo_heads + hq) * D;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int v = 0; v < PER; ++v) orow[lane * PER + v] = from_float<T>(acc[v] * inv);
  if (lane == 0 && a.lse)
    a.lse[static_cast<int64_t>(it.row) * a.num_qo_heads + hq] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// Launch one decode instance (head_dim, group size and cap chosen at run time).
// Lanes per token: 8, or 16 for a group of 8 at head_dim 128.
template <typename T, bool GATHER>
cudaError_t launch_decode_kernel(const DecodeArgs& a, int D, int G, bool cap, int grid, cudaStream_t s) {
  void (*kern)(DecodeArgs) = nullptr;
#define PKV_DEC_CASE(DD, GG, LL)                                                                                 \
  if (D == DD && G == GG)                                                                                       \
    kern = cap ? decode_kernel<DD, GG, LL, T, true, GATHER> : decode_kernel<DD, GG, LL, T, false, GATHER>;
  PKV_DEC_CASE(128, 1, 8) PKV_DEC_CASE(128, 2, 8) PKV_DEC_CASE(128, 4, 8) PKV_DEC_CASE(128, 8, 16)
  PKV_DEC_CASE(64, 1, 8) PKV_DEC_CASE(64, 2, 8) PKV_DEC_CASE(64, 4, 8) PKV_DEC_CASE(64, 8, 8)
#undef PKV_DEC_CASE
  if (!kern) return cudaErrorInvalidValue;
  const int smem = kDecodeWarps * kDecodeWarpSmem;
  static_assert(kDecodeWarps * kDecodeWarpSmem <= 200 * 1024, "decode ring exceeds shared memory");
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, kDecodeWarps * 32, smem, s, a);
}

// Each instance set is compiled in its own translation unit (decode.cu: bulk
// copies; decode_gather.cu: tensor gathers for one-row pages).
extern template cudaError_t launch_decode_kernel<__nv_bfloat16, false>(const DecodeArgs&, int, int, bool, int,
                                                                       cudaStream_t);
extern template cudaError_t launch_decode_kernel<__half, false>(const DecodeArgs&, int, int, bool, int, cudaStream_t);
extern template cudaError_t launch_decode_kernel<__nv_bfloat16, true>(const DecodeArgs&, int, int, bool, int,
                                                                      cudaStream_t);
extern template cudaError_t launch_decode_kernel<__half, true>(const DecodeArgs&, int, int, bool, int, cudaStream_t);

}  // namespace decode_impl
}  // namespace pkv
