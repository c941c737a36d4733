// prefill_kernel.cuh -- the tcgen05 paged prefill kernel template, shared by the
// translation units that instantiate it (prefill.cu: without a custom mask,
// prefill_masked.cu: with one).
//
// Causal ragged batch prefill over a paged KV cache on tcgen05.
//
// Method (FlashInfer pages): batch_prefill with causal=True over the same
// page table as decode ("FlashInfer" guide, "The Interface"); the kernel
// gathers scattered pages into contiguous shared memory before using tensor
// cores (fdeinterviews, "One format for every KV layout"); query heads that
// share a kv head are packed into one row block (greptalks, "Head Group
// Packing"); with causal off and every request's query in one row block it is
// the shared-prefix half of cascade attention (guide section 3, "Cascade
// Attention"; fdeinterviews, composable formats with a large row block).
//
// GB300 design.  One CTA per SM walks the plan's list of work tiles.  A work
// tile is 256 packed query rows (256/G query positions x the G heads of one
// kv head) held as two 128-row UMMA tiles, A and B, against one key range
// visited 128 keys (128/P pages) at a time; every K/V block that lands in
// shared memory serves both tiles.
//   warps 0, 10 producers: TMA loads the two Q boxes once per tile and, per
//               key block, one 64-column box per (page, half) for K (warp 0,
//               two stages) and for V (warp 10, two stages), 128B-swizzled.
//               Pages past the request come from an out-of-range page
//               coordinate, which TMA fills with zeros; V rows past
//               kv_last_page_len of the last page are zeroed before the MMA
//               may read them.  Pages of 1, 2 or 4 rows (column-vector BSR)
//               are gathered instead with 16-byte cp.async, four lanes per
//               256-byte row, into the same swizzled layout, zero-filled past
//               the request; each lane waits for its own copies, fences them
//               for the tensor cores and arrives on the block's barrier, while
//               the next block's page ids load.
//   warp 1      one thread issues the tcgen05 MMAs, alternating the tiles:
//               P_A V -> O_A, S_A(next) = Q_A K^T, P_B V -> O_B, S_B(next)
//               (tile A only when the work tile's positions fit in it).
//               S, P and O stay in tensor memory: S_A, S_B, O_A, O_B take the
//               512 columns, and each P (bf16/fp16) overwrites the first 64
//               columns of its S, the A operand of its P V MMA.
//   warps 2-5   softmax of tile A, warps 6-9 of tile B (two warps per
//               scheduler, so one group's softmax overlaps the other group's
//               MMAs): thread = query row = TMEM lane.  Each reads its S row,
//               scales (and soft-caps), masks (causal limit and, in the MASK
//               instances, the caller's packed custom mask), keeps a running
//               max and sum,
//               writes P back to tensor memory and rescales O only when the
//               max grows by more than 2^8.  The epilogue divides O by the sum
//               and writes o and the natural-log lse (or an fp32 partial state
//               when the plan split the key range).
// Every wait is bounded; a wait that runs out records kErrWaitTimeout and
// makes all roles leave their loops, the MMA thread waits for its issued
// MMAs, and tensor memory is released.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <type_traits>

#include "pkv_bsr.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"


namespace pkv {
namespace prefill_impl {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kD = 128;                 // head_dim of the prefill kernel
constexpr int kTM = 128;                // rows of one UMMA tile
constexpr int kWR = kPrefillRows;       // rows of a work tile: two UMMA tiles
static_assert(kWR == 2 * kTM, "a work tile is two UMMA tiles");
constexpr int kBN = kPrefillKeys;       // keys per block
constexpr int kThreads = 352;           // K producer, MMA, 2 x 4 softmax warps, V producer
constexpr int kVWarp = 10;
constexpr uint32_t kTile = 32768;       // 128 rows x 128 16-bit values
constexpr uint32_t kHalf = 16384;       // one 64-column half of a tile
constexpr int kKStages = 2;             // K has its own producer: two blocks of lead cover the gather
constexpr int kVStages = 2;
// Shared-memory map; dynamic shared memory must start 1024-aligned (checked).
// The staging area gives each softmax warp 4 KB to turn its 32 rows into
// row-contiguous global stores in the epilogue.
// The two page-id arrays serve the cp.async gather of pages smaller than 8 rows
// (only those instances reserve them).
constexpr uint32_t kOffQ = 0, kOffK = 2 * kTile, kOffV = kOffK + kKStages * kTile,
                   kOffStage = kOffV + kVStages * kTile, kOffBar = kOffStage + 8 * 4096, kOffIds = kOffBar + 256;
constexpr int kSmemBytes = kOffBar + 256;
constexpr int kSmemBytesSmall = kOffIds + 2 * kBN * 4;
static_assert(kSmemBytesSmall <= 232448, "shared memory budget");
enum { Q_FULL = 0, Q_EMPTY = 1, K_FULL = 2, K_EMPTY = K_FULL + kKStages, V_FULL = K_EMPTY + kKStages,
       V_EMPTY = V_FULL + kVStages, S_FULL = V_EMPTY + kVStages, P_FULL = S_FULL + 2, O_DONE = P_FULL + 2,
       O_FREE = O_DONE + 2, V_LOAD = O_FREE + 2, DRAIN = V_LOAD + kVStages, NUM_BARS = DRAIN + 1 };
static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");
constexpr uint32_t kGroupThreads = 128;  // softmax threads of one tile
constexpr uint32_t kTmemCols = 512;      // S_A, S_B, O_A, O_B
constexpr uint32_t kColS = 0, kColO = 256;

struct Waiter {
  int32_t* err;
  volatile int* abort_flag;
  // Bounded wait; false when it ran out (recorded) or another role gave up.
  __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, kErrWaitTimeout);
        *abort_flag = 1;
        return false;
      }
    }
    return true;
  }
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return a <= 0 ? 0 : (a + b - 1) / b; }

// D[tmem] (+)= A * B with both shared-memory descriptors given as their low
// words and a common high word (every descriptor here has the same stride
// field, version and swizzle), so issuing an MMA costs two 32-bit adds in the
// caller.  In the TS form the A operand is read from tensor memory (K-major,
// 16-bit pairs per 32-bit column, even k in the low half).
template <bool ACC>
__device__ __forceinline__ void umma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .b64 da, db;\n\tmov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, %5;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "n"(ACC ? 1 : 0)
      : "memory");
}
template <bool ACC>
__device__ __forceinline__ void umma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .b64 db;\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, %5;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "n"(ACC ? 1 : 0)
      : "memory");
}

// SMALL: pages of fewer than 8 rows, gathered with cp.async (its own instance set,
// so the tensor-copy path of larger pages carries none of that code).
// STAGED: fp32 partial states of split tiles go out through the warp's staging
// slab, like the final output, so each store writes whole 128-byte segments
// (the masked and mixed-batch instances, where split tiles are common; compiled
// into the plain instances it cost the ragged causal batch 1.6 % through register
// allocation, and there no tile is split).
// One CTA's share of the work: `cta` indexes the plan's workers, `sm` is the
// CTA's dynamic shared memory (kSmemBytes, or kSmemBytesSmall for SMALL).  Warps
// 0-10 take the roles above; any further warp of the CTA only joins the two
// CTA-wide barriers.
template <int G, typename T, bool CAP, bool MASK, bool SMALL, bool STAGED>
__device__ __forceinline__ void prefill_cta(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tkv,
                                            int cta, uint8_t* sm) {
  constexpr uint32_t kFmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  constexpr int MP = kTM / G;  // query positions per UMMA tile
  const uint32_t base = smem_addr(sm);
  if (base & 1023u) {  // never expected; refuse rather than misread swizzled tiles
    if (threadIdx.x == 0) atomicOr(a.err, kErrTmemAlloc);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS + 1);
  auto bar = [&](int i) { return base + kOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  constexpr bool small = SMALL;  // cp.async gather: every producer lane arrives on the FULL barriers
  if (threadIdx.x == 0) {
    for (int i = 0; i < NUM_BARS; ++i) {
      uint32_t count = 1;
      if (i == P_FULL || i == P_FULL + 1 || i == O_FREE || i == O_FREE + 1) count = kGroupThreads;
      if (small && ((i >= K_FULL && i < K_FULL + kKStages) || (i >= V_FULL && i < V_FULL + kVStages))) count = 32;
      mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter wait{a.err, abort_flag};

  const PlanHeader* hdr = a.hdr;
  int t_begin = 0, t_end = 0;
  if (cta < hdr->num_workers) {
    t_begin = a.worker_ptr[cta];
    t_end = a.worker_ptr[cta + 1];
  }
  const int num_pages = static_cast<int>(hdr->num_pages);
  const int P = a.page_size;
  const int ppt = kBN / P;  // pages per key block

  auto page_of = [&](const PrefillTile& t, int j, int n_pages_req) {
    const int rel = (t.kv_begin + j * kBN) / P + lane;
    int id = num_pages;  // past the pool: TMA fills the box with zeros
    if (lane < ppt && rel < n_pages_req) {
      const int v = __ldg(a.kv_indices + t.idx_base + rel);
      if (v >= 0 && v < num_pages)
        id = v;
      else
        atomicOr(a.err, kErrPageIndex);
    }
    return id;
  };

  // Pages smaller than 8 rows.  gather_ids loads the page ids of block j of tile t
  // (up to 128, four per lane; -1 past the request); gather_block copies that
  // block's K (kv_sel 0) or V (1) rows into the swizzled stage at `dst` with
  // cp.async, 16 bytes a copy and four lanes per 256-byte row, zero-filling rows
  // past the request, waits for this lane's copies, fences them for the tensor
  // cores and arrives on `full_bar`.  The caller loads the next block's ids in
  // between (`next`), so their latency hides behind the copies.
  auto gather_ids = [&](const PrefillTile& t, int j, int (&idr)[4]) {
    const int rel0 = (t.kv_begin + j * kBN) / P;
    const int n_pages_req = ceil_div_i(t.kv_len, P);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int k = lane + 32 * m;
      idr[m] = -1;
      if (k < ppt && rel0 + k < n_pages_req) {
        const int v = __ldg(a.kv_indices + t.idx_base + rel0 + k);
        if (v >= 0 && v < num_pages)
          idr[m] = v;
        else
          atomicOr(a.err, kErrPageIndex);
      }
    }
  };
  auto gather_block = [&](const PrefillTile& t, int j, int kv_sel, uint32_t dst, int32_t* ids, const int (&idr)[4],
                          int full_bar, auto&& next) {
    const int key0 = t.kv_begin + j * kBN;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (lane + 32 * m < ppt) ids[lane + 32 * m] = idr[m];
    __syncwarp();
    const int lp = __ffs(P) - 1;     // P is a power of two (1, 2 or 4 here)
    // Four lanes per row: lane group g = lane / 4 takes rows 8q + g (q = 0 .. 15),
    // lane cl = lane % 4 the 16-byte chunks cl and cl + 4 of both 128-byte halves
    // of the row.  Every row's id lookup and address arithmetic then serve four
    // copies, and every copy instruction still reads whole 64-byte pieces of eight
    // rows.  (16 lanes per row issued four times the instructions: 31 % of peak on
    // 1-token pages against 42 %; 8 lanes per row gave 41 %.)
    const int g = lane >> 2, cl = lane & 3;
    const T* kvp = static_cast<const T*>(a.kv);
    // The chunk's address in page 0 of this (K|V, kv head) plus the row's slot in
    // its page (the same for every row of this lane: 8q is a multiple of P), and
    // the distance from one page to the next.
    const T* base_c =
        kvp + (static_cast<int64_t>(kv_sel) * a.num_kv_heads + t.kvh) * P * kD + (g & (P - 1)) * kD + cl * 8;
    const int page_stride = 2 * a.num_kv_heads * P * kD;
    // Swizzled shared-memory offsets of chunks cl and cl + 4 (first half): every row
    // of this lane has row % 8 = g.
    const uint32_t d0 = dst + g * 128 + ((cl ^ g) << 4), d1 = dst + g * 128 + (((cl + 4) ^ g) << 4);
    const int rows_left = t.kv_len - key0 - g;  // row 8q + g exists while 8q < rows_left
    // Eight rows at a time: their page ids first (independent shared loads), then
    // their copies; a copy is ordered after everything before it, so one id load
    // between two copies would expose its whole latency.
    constexpr int kBatch = 8;
#pragma unroll 1
    for (int q0 = 0; q0 < kBN / 8; q0 += kBatch) {
      int idb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) idb[u] = ids[(8 * (q0 + u) + g) >> lp];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const bool valid = idb[u] >= 0 && 8 * (q0 + u) < rows_left;
        const T* src = base_c + static_cast<int64_t>(valid ? idb[u] : 0) * page_stride;
        const uint32_t ro = (q0 + u) * 1024;  // row 8q + g is 1024 q bytes past row g
        const uint32_t nb = valid ? 16u : 0u;
        cp_async_16(d0 + ro, src, nb);
        cp_async_16(d1 + ro, src + 32, nb);
        cp_async_16(d0 + ro + kHalf, src + 64, nb);
        cp_async_16(d1 + ro + kHalf, src + 96, nb);
      }
    }
    cp_async_commit();
    next();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    mbar_arrive(bar(full_bar));
    __syncwarp();  // every lane has read ids before the next block rewrites them
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    int kvc = 0;
    bool ok = true;
    for (int ti = t_begin, tn = 0; ti < t_end && ok; ++ti, ++tn) {
      const PrefillTile t = a.tiles[ti];
      if (tn > 0) {
        ok = __all_sync(kFull, wait(bar(Q_EMPTY), (tn - 1) & 1));
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Q_FULL), 2 * kTile);
        for (int x = 0; x < 2; ++x)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(base + kOffQ + x * kTile + h * kHalf, &tq, h * 64, t.kvh * G, t.q_row0 + x * MP,
                        bar(Q_FULL));
      }
      const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
      const int n_pages_req = ceil_div_i(t.kv_len, P);
      int id_next = (n > 0 && !small) ? page_of(t, 0, n_pages_req) : num_pages;
      int idr[4] = {-1, -1, -1, -1};  // cp.async gather: page ids of the block being issued
      if (small && n > 0) gather_ids(t, 0, idr);
      for (int j = 0; j < n; ++j) {
        const int id = id_next;
        if (j + 1 < n && !small) id_next = page_of(t, j + 1, n_pages_req);  // next block's page ids load meanwhile
        const int s = kvc % kKStages;
        if (kvc >= kKStages) {
          ok = __all_sync(kFull, wait(bar(K_EMPTY + s), ((kvc / kKStages) - 1) & 1));
          if (!ok) break;
        }
        if constexpr (SMALL) {
          int idn[4];
          gather_block(t, j, 0, base + kOffK + s * kTile, reinterpret_cast<int32_t*>(sm + kOffIds), idr, K_FULL + s,
                       [&] {
                         if (j + 1 < n) gather_ids(t, j + 1, idn);
                       });
#pragma unroll
          for (int m = 0; m < 4; ++m) idr[m] = idn[m];
          ++kvc;
          continue;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(K_FULL + s), kTile);
        __syncwarp();
        const uint32_t sK = base + kOffK + s * kTile;
        if (lane < ppt)
          for (int h = 0; h < 2; ++h)
            tma_load_5d(sK + h * kHalf + lane * P * 128, &tkv, h * 64, 0, t.kvh, 0, id, bar(K_FULL + s));
        ++kvc;
      }
    }
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ V producer
    int kvc = 0;
    uint32_t vload_bits = 0;  // phase parity of each V_LOAD barrier
    bool ok = true;
    for (int ti = t_begin; ti < t_end && ok; ++ti) {
      const PrefillTile t = a.tiles[ti];
      const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
      const int n_pages_req = ceil_div_i(t.kv_len, P);
      int id_next = (n > 0 && !small) ? page_of(t, 0, n_pages_req) : num_pages;
      int idr[4] = {-1, -1, -1, -1};  // cp.async gather: page ids of the block being issued
      if (small && n > 0) gather_ids(t, 0, idr);
      for (int j = 0; j < n; ++j) {
        const int id = id_next;
        if (j + 1 < n && !small) id_next = page_of(t, j + 1, n_pages_req);
        const int s = kvc % kVStages;
        if (kvc >= kVStages) {
          ok = __all_sync(kFull, wait(bar(V_EMPTY + s), ((kvc / kVStages) - 1) & 1));
          if (!ok) break;
        }
        const uint32_t sV = base + kOffV + s * kTile;
        if constexpr (SMALL) {
          int idn[4];
          gather_block(t, j, 1, sV, reinterpret_cast<int32_t*>(sm + kOffIds) + kBN, idr, V_FULL + s, [&] {
            if (j + 1 < n) gather_ids(t, j + 1, idn);
          });
#pragma unroll
          for (int m = 0; m < 4; ++m) idr[m] = idn[m];
          ++kvc;
          continue;
        }
        const int rel0 = (t.kv_begin + j * kBN) / P;
        const int last_rel = n_pages_req - 1 - rel0;
        const bool partial = t.last_rows < P && last_rel >= 0 && last_rel < ppt;
        const uint32_t vbar = partial ? bar(V_LOAD + s) : bar(V_FULL + s);
        if (lane == 0) mbar_arrive_expect_tx(vbar, kTile);
        __syncwarp();
        if (lane < ppt)
          for (int h = 0; h < 2; ++h) tma_load_5d(sV + h * kHalf + lane * P * 128, &tkv, h * 64, 0, t.kvh, 1, id, vbar);
        if (partial) {
          // The last page's slots past kv_last_page_len may hold anything; the
          // P V product must see zeros there (0 * NaN would poison O).
          ok = __all_sync(kFull, wait(bar(V_LOAD + s), (vload_bits >> s) & 1));
          if (!ok) break;
          vload_bits ^= 1u << s;
          const int chunks = (P - t.last_rows) * 8;  // 16-byte chunks per half
          uint8_t* vgen = sm + kOffV + s * kTile;
          for (int i = lane; i < 2 * chunks; i += 32) {
            const int h = i / chunks, c = i % chunks;
            *reinterpret_cast<uint4*>(vgen + h * kHalf + (last_rel * P + t.last_rows) * 128 + c * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(V_FULL + s));
        }
        ++kvc;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = umma_idesc_f16(kFmt, kTM, kBN, 0);
      const uint32_t id_o = umma_idesc_f16(kFmt, kTM, kD, 1);
      int kvc = 0;
      int pc[2] = {0, 0}, ofree[2] = {0, 0};
      bool o_used[2] = {false, false};  // an earlier tile accumulated into O_x
      bool ok = true;
      // Descriptors are built once; a K step or a stage only adds to the start
      // address field of the low word (addresses stay below 2^18, so no carry
      // leaves it), and all of them share one high word.  Issuing an MMA then
      // takes a few instructions, well under the 64 cycles an M=128, N=128, K=16
      // MMA runs, even while this warp shares its scheduler with softmax warps.
      const uint64_t dq = sw128_desc(base + kOffQ, 16, 1024);
      const uint64_t dk = sw128_desc(base + kOffK, 16, 1024);
      const uint64_t dv = sw128_desc(base + kOffV, kHalf, 1024);
      const uint32_t hi = static_cast<uint32_t>(dq >> 32);
      const uint32_t q_lo = static_cast<uint32_t>(dq), k_lo = static_cast<uint32_t>(dk),
                     v_lo = static_cast<uint32_t>(dv);
      constexpr uint32_t kTile16 = kTile >> 4, kHalf16 = kHalf >> 4;
      // S_x = Q_x K_c^T into tensor memory.
      auto mma_s = [&](int x, int c) {
        const uint32_t a0 = q_lo + x * kTile16;
        const uint32_t b0 = k_lo + (c % kKStages) * kTile16;
        const uint32_t d = tmem + kColS + x * kTM;
        umma_ss_lo<false>(d, a0, b0, hi, id_s);
#pragma unroll
        for (int kk = 1; kk < kD / 16; ++kk) {
          const uint32_t koff = (kk / 4) * kHalf16 + (kk % 4) * 2;
          umma_ss_lo<true>(d, a0 + koff, b0 + koff, hi, id_s);
        }
        umma_commit(bar(S_FULL + x));
      };
      // O_x += P_x V_c, P_x from tensor memory; the tile's last one signals the epilogue.
      auto mma_pv = [&](int x, int c, bool acc, bool last) {
        const uint32_t b0 = v_lo + (c % kVStages) * kTile16;
        const uint32_t d = tmem + kColO + x * kTM, p = tmem + kColS + x * kTM;
        if (acc)
          umma_ts_lo<true>(d, p, b0, hi, id_o);
        else
          umma_ts_lo<false>(d, p, b0, hi, id_o);
#pragma unroll
        for (int kk = 1; kk < kBN / 16; ++kk) umma_ts_lo<true>(d, p + kk * 8, b0 + kk * (2048 >> 4), hi, id_o);
        if (last) umma_commit(bar(O_DONE + x));
      };
      for (int ti = t_begin, tn = 0; ti < t_end && ok; ++ti, ++tn) {
        const PrefillTile t = a.tiles[ti];
        const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
        // Tile B holds positions MP .. 2 MP - 1; a work tile of at most MP
        // positions (a request's short last tile, a decode row) runs tile A only.
        const int nx = t.n_pos > MP ? 2 : 1;
        if (!(ok = wait(bar(Q_FULL), tn & 1))) break;
        tc_fence_after();
        if (n == 0) {
          umma_commit(bar(Q_EMPTY));
          continue;
        }
        if (!(ok = wait(bar(K_FULL + kvc % kKStages), (kvc / kKStages) & 1))) break;
        tc_fence_after();
        mma_s(0, kvc);
        if (nx == 2) mma_s(1, kvc);
        umma_commit(bar(K_EMPTY + kvc % kKStages));
        if (n == 1) umma_commit(bar(Q_EMPTY));
        // The key blocks of the tile, compiled once for each number of UMMA tiles
        // (NX = 2 is the loop of a full work tile, with nothing tested per tile).
        auto blocks = [&](auto nx_c) {
          constexpr int NX = decltype(nx_c)::value;
          for (int j = 0; j < n && ok; ++j) {
            const int c = kvc + j;
            for (int x = 0; x < NX && ok; ++x) {
              if (!(ok = wait(bar(P_FULL + x), pc[x] & 1))) break;
              ++pc[x];
              if (j == 0 && o_used[x]) {  // the previous tile's epilogue has read O_x
                if (!(ok = wait(bar(O_FREE + x), ofree[x] & 1))) break;
                ++ofree[x];
              }
              if (x == 0 && !(ok = wait(bar(V_FULL + c % kVStages), (c / kVStages) & 1))) break;
              tc_fence_after();
              mma_pv(x, c, j > 0, j == n - 1);
              o_used[x] = true;
              if (x == NX - 1) umma_commit(bar(V_EMPTY + c % kVStages));  // every P V of block c issued
              if (j + 1 < n) {
                if (x == 0) {
                  if (!(ok = wait(bar(K_FULL + (c + 1) % kKStages), ((c + 1) / kKStages) & 1))) break;
                  tc_fence_after();
                }
                mma_s(x, c + 1);
                if (x == NX - 1) {
                  umma_commit(bar(K_EMPTY + (c + 1) % kKStages));  // every S of block c + 1 issued
                  if (j + 1 == n - 1) umma_commit(bar(Q_EMPTY));
                }
              }
            }
          }
        };
        if (nx == 2)
          blocks(std::integral_constant<int, 2>{});
        else
          blocks(std::integral_constant<int, 1>{});
        kvc += n;
      }
      // Every MMA issued so far must finish before tensor memory is released.
      umma_commit(bar(DRAIN));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(DRAIN), 0))
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
    }
    __syncwarp();
  } else if (warp < kVWarp) {
    // ------------------------------------------------------------ softmax + epilogue
    const int x = (warp - 2) >> 2;           // UMMA tile of this warp group
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;       // row within the UMMA tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col_s = tmem + lane_off + kColS + x * kTM;
    const uint32_t col_o = tmem + lane_off + kColO + x * kTM;
    const float scale = CAP ? a.sm_scale : a.sm_scale * kLog2e;
    int sc = 0, odc = 0;
    bool ok = true;
    for (int ti = t_begin; ti < t_end && ok; ++ti) {
      const PrefillTile t = a.tiles[ti];
      // A work tile of at most MP positions has no rows in tile B: the MMA thread
      // issues nothing for it, and its group skips the tile (its rows are past
      // n_pos, written nowhere and not read by the merge of a split key range).
      if (x == 1 && t.n_pos <= MP) continue;
      const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
      const int rpos = x * MP + r / G;     // position of this row within the work tile
      const bool row_valid = rpos < t.n_pos;
      const int pos = t.q_pos0 + rpos;
      int limit = t.kv_len, lim0 = t.kv_len;  // keys < limit are visible to this row / to every row of x
      if (a.causal) {
        limit = min(limit, pos + 1 + t.kv_len - t.qo_len);
        lim0 = min(lim0, t.q_pos0 + x * MP + 1 + t.kv_len - t.qo_len);
      }
      limit = min(limit, t.kv_end);
      lim0 = min(lim0, t.kv_end);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int key0 = t.kv_begin + j * kBN;
        // Custom mask: this row's bits for keys key0 .. key0 + 127, read (from L2)
        // before the wait for S so the loads overlap it.
        uint32_t mw[4] = {~0u, ~0u, ~0u, ~0u};
        if constexpr (MASK) {
          if (row_valid) {
            const int64_t bit = t.mask_off + static_cast<int64_t>(pos) * t.kv_len + key0;
            const int64_t w0 = bit >> 5;
            const uint32_t sh = static_cast<uint32_t>(bit & 31);
            uint32_t w[5];
#pragma unroll
            for (int k = 0; k < 5; ++k) w[k] = (w0 + k < a.mask_words) ? __ldg(a.mask + w0 + k) : 0u;
#pragma unroll
            for (int k = 0; k < 4; ++k) mw[k] = __funnelshift_r(w[k], w[k + 1], sh);
          }
        }
        if (!(ok = __all_sync(kFull, wait(bar(S_FULL + x), sc & 1)))) break;
        ++sc;
        tc_fence_after();
        const bool full = key0 + kBN <= lim0;
        uint32_t sr[kBN];
        tmem_ld128_sync(col_s, sr);
        // Logits in log2 units are v * mul (the cap, when on, is applied to v first).
        float mul = scale;
        if constexpr (CAP) {
          // cap * tanh(s * scale / cap), already in log2 units
          // in pairs: cap * tanh(y) = k_out - 2 k_out / (e^(2y) + 1), e^(2y) = 2^(s * k_in)
          const float k_in = scale * 2.f * kLog2e / a.cap, k_out = a.cap * kLog2e;
          const float2 kin2 = make_float2(k_in, k_in), one2 = make_float2(1.f, 1.f);
          const float2 m2k = make_float2(-2.f * k_out, -2.f * k_out), kout2 = make_float2(k_out, k_out);
#pragma unroll
          for (int i = 0; i < kBN; i += 2) {
            float2 e = fmul2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), kin2);
            e.x = fast_exp2(e.x);
            e.y = fast_exp2(e.y);
            float2 d = fadd2(e, one2);
            d.x = fast_rcp(d.x);
            d.y = fast_rcp(d.y);
            const float2 x = ffma2(d, m2k, kout2);
            sr[i] = __float_as_uint(x.x);
            sr[i + 1] = __float_as_uint(x.y);
          }
          mul = 1.f;
        }
        if (!full) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (key0 + i >= limit) sr[i] = 0xff800000u;  // -inf
        }
        if constexpr (MASK) {
          if ((mw[0] & mw[1] & mw[2] & mw[3]) != ~0u) {
#pragma unroll
            for (int i = 0; i < kBN; ++i)
              if (!((mw[i >> 5] >> (i & 31)) & 1u)) sr[i] = 0xff800000u;
          }
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int i = 8; i < kBN; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * mul;
        const float m_new = fmaxf(m_ref, mx);
        const bool resc = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_ref + 8.f);
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
        }
        const float sub = (m_ref == -INFINITY) ? 0.f : m_ref;
        // p = 2^(v * mul - sub): packed FMAs and the SFU exponential (the SFU has
        // room at this rate: two tiles' rows share it with the tensor pipe's time);
        // packed in place to 16-bit pairs.
        const float2 mul2 = make_float2(mul, mul), nsub2 = make_float2(-sub, -sub);
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kBN; i += 2) {
          float2 v = ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), mul2, nsub2);
          v.x = fast_exp2(v.x);
          v.y = fast_exp2(v.y);
          sum4[(i >> 1) & 3] = fadd2(sum4[(i >> 1) & 3], v);
          sr[i >> 1] = pack2<T>(v.x, v.y);
        }
        const float2 s4 = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
        l += s4.x + s4.y;
        // P over the first 64 columns of this tile's S (already read).
        tmem_st32(col_s, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_st32(col_s + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        if (j >= 1) {
          // P V of the previous block was issued before this S, so the S_FULL
          // wait above already covers it: O is complete and can be rescaled
          // before the next P V adds to it.
          if (__any_sync(kFull, resc)) {
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
              uint32_t rr[32];
              tmem_ld32_sync(col_o + c * 32, rr);
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st32(col_o + c * 32, rr);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(P_FULL + x));
      }
      if (!ok) break;
      if (n >= 1) {
        if (!(ok = __all_sync(kFull, wait(bar(O_DONE + x), odc & 1)))) break;
        ++odc;
        tc_fence_after();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      const int64_t orow = static_cast<int64_t>(t.q_row0 + rpos) * a.num_qo_heads + t.kvh * G + (r % G);
      const int srow = x * kTM + r;  // row of the work tile, for a partial-state slot
      if (t.slot < 0) {
        // Final output: through this warp's staging slab, half a row (64 values) per pass,
        // so each store instruction writes four whole 128-byte row segments.
        uint8_t* stg = sm + kOffStage + (warp - 2) * 4096;
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          uint32_t pk[32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t rr[32];
            if (n >= 1) {
              tmem_ld32_sync(col_o + (hp * 2 + cc) * 32, rr);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[cc * 16 + i] = pack2<T>(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr_ = it * 4 + (lane >> 3), piece = lane & 7;  // a row of this warp, a 16-byte piece
            const int r2 = quarter * 32 + rr_;
            const int rpos2 = x * MP + r2 / G;
            const uint4 v = *reinterpret_cast<const uint4*>(stg + rr_ * 128 + ((piece ^ (rr_ & 7)) << 4));
            if (rpos2 < t.n_pos) {
              const int64_t orow2 =
                  static_cast<int64_t>(t.q_row0 + rpos2) * a.num_qo_heads + t.kvh * G + (r2 % G);
              reinterpret_cast<uint4*>(static_cast<T*>(a.o) + orow2 * kD + hp * 64)[piece] = v;
            }
          }
          __syncwarp();
        }
      } else if constexpr (STAGED) {
        // Partial state: 32 columns of the warp's 32 rows per pass through the
        // slab, then four rows' 128-byte segments per store instruction.
        uint8_t* stg = sm + kOffStage + (warp - 2) * 4096;
        float* part0 = a.part_o + (static_cast<int64_t>(t.slot) * kWR + x * kTM + quarter * 32) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float ov[32];
          if (n >= 1) {
            uint32_t rr[32];
            tmem_ld32_sync(col_o + c * 32, rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(rr[i]) * inv;
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr_ = it * 4 + (lane >> 3), piece = lane & 7;  // a row of this warp, a 16-byte piece
            const float4 v = *reinterpret_cast<const float4*>(stg + rr_ * 128 + ((piece ^ (rr_ & 7)) << 4));
            reinterpret_cast<float4*>(part0 + rr_ * kD + c * 32)[piece] = v;
          }
          __syncwarp();
        }
      } else {
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float ov[32];
          if (n >= 1) {
            uint32_t rr[32];
            tmem_ld32_sync(col_o + c * 32, rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(rr[i]) * inv;
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0.f;
          }
          float4* dst =
              reinterpret_cast<float4*>(a.part_o + (static_cast<int64_t>(t.slot) * kWR + srow) * kD + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
      }
      if (t.slot < 0) {
        if (row_valid && a.lse) a.lse[orow] = lse_v;
      } else {
        a.part_lse[static_cast<int64_t>(t.slot) * kWR + srow] = lse_v;
      }
      if (n >= 1) {  // this tile's O is free for the next tile's P V
        tc_fence_before();
        mbar_arrive(bar(O_FREE + x));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Log-sum-exp merge of the chunks' fp32 partial states of one packed row of a
// query tile whose key range the plan split (pair = item * 256 + row), by the
// calling warp, lanes over head_dim.  Shared by the prefill merge kernel and the
// mixed batch's merge kernel.
template <typename T>
__device__ __forceinline__ void prefill_merge_row(const PrefillArgs& a, int pair, int lane, int G) {
  const PrefillMerge it = a.merge[pair / kWR];
  const int r = pair % kWR;
  if (r / G >= it.n_pos) return;
  float mx = -INFINITY;
  for (int i = lane; i < it.n_slots; i += 32)
    mx = fmaxf(mx, a.part_lse[static_cast<int64_t>(it.slot_begin + i) * kWR + r]);
  mx = warp_max(mx);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    // The row loads do not wait for the weights: a slot of weight 0 is dropped by
    // a select after its load, not by a branch before it.
#pragma unroll 4
    for (int i = 0; i < it.n_slots; ++i) {
      const int64_t row = static_cast<int64_t>(it.slot_begin + i) * kWR + r;
      const float4 v = reinterpret_cast<const float4*>(a.part_o + row * kD)[lane];
      const float w = fast_exp2((a.part_lse[row] - mx) * kLog2e);
      const bool use = w > 0.f;
      acc[0] = use ? fmaf(w, v.x, acc[0]) : acc[0];
      acc[1] = use ? fmaf(w, v.y, acc[1]) : acc[1];
      acc[2] = use ? fmaf(w, v.z, acc[2]) : acc[2];
      acc[3] = use ? fmaf(w, v.w, acc[3]) : acc[3];
      wsum += use ? w : 0.f;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t orow = static_cast<int64_t>(it.q_row0 + r / G) * a.num_qo_heads + it.kvh * G + (r % G);
  T* dst = static_cast<T*>(a.o) + orow * kD + lane * 4;
#pragma unroll
  for (int v = 0; v < 4; ++v) dst[v] = from_float<T>(acc[v] * inv);
  if (lane == 0 && a.lse) a.lse[orow] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <int G, typename T, bool CAP, bool MASK, bool SMALL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tkv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  prefill_cta<G, T, CAP, MASK, SMALL, MASK>(a, tq, tkv, blockIdx.x, smem_raw);
}


// Launch one instance of the kernel (group size and cap chosen at run time).
template <typename T, bool MASK, bool SMALL>
cudaError_t launch_kernel(const PrefillArgs& a, int G, bool cap, int grid, const CUtensorMap& tq,
                          const CUtensorMap& tkv, cudaStream_t s) {
  void (*kern)(PrefillArgs, CUtensorMap, CUtensorMap) = nullptr;
#define PKV_PF_CASE(GG)                                                                                \
  case GG:                                                                                             \
    kern = cap ? prefill_kernel<GG, T, true, MASK, SMALL> : prefill_kernel<GG, T, false, MASK, SMALL>; \
    break;
  switch (G) {
    PKV_PF_CASE(1) PKV_PF_CASE(2) PKV_PF_CASE(4) PKV_PF_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef PKV_PF_CASE
  constexpr int smem = SMALL ? kSmemBytesSmall : kSmemBytes;
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(a, tq, tkv);
  return cudaGetLastError();
}

// The tensor maps of q (3D boxes of 64 columns x G heads x 128/G positions) and
// kv_data (5D boxes of 64 columns x one page's rows) for the prefill tiles.
cudaError_t make_tensor_maps(const PrefillArgs& a, int group, int dtype, int64_t total_q, int64_t num_pages,
                             CUtensorMap& tq, CUtensorMap& tkv);

// Each instance set is compiled in its own translation unit.
extern template cudaError_t launch_kernel<__nv_bfloat16, false, false>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__half, false, false>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__nv_bfloat16, false, true>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__half, false, true>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__nv_bfloat16, true, false>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__half, true, false>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__nv_bfloat16, true, true>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_kernel<__half, true, true>(const PrefillArgs&, int, bool, int,
                                                     const CUtensorMap&, const CUtensorMap&, cudaStream_t);

}  // namespace prefill_impl
}  // namespace pkv
