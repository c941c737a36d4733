// prefill.cu -- causal ragged batch prefill over a paged KV cache on tcgen05.
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
// GB300 design.  One CTA per SM walks the plan's list of work tiles.  A tile
// is 128 packed query rows (128/G query positions x the G heads of one kv
// head) against a key range, visited 128 keys (128/P pages) at a time:
//   warps 0, 6  producers: TMA loads the Q box once per tile and, per key
//               block, one 64-column box per (page, half) for K (warp 0,
//               three stages) and for V (warp 6, two stages), 128B-swizzled
//               into shared memory.  K and V run independently, so the page
//               gather of K is never held back by the P V of older blocks.
//               Pages past the request come from an out-of-range page
//               coordinate, which TMA fills with zeros; V rows past
//               kv_last_page_len of the last page are zeroed before the MMA
//               may read them.
//   warp 1      one thread issues the tcgen05 MMAs: S_j = Q K_j^T into one of
//               two TMEM buffers (so S_{j+1} overlaps the softmax of S_j),
//               then O += P_j V_j into a third TMEM region.
//   warps 2-9   softmax: two warps per query row block quarter, each thread
//               one query row (= TMEM lane) and one half (64 keys) of it.  It
//               reads its half of S from TMEM, scales (and soft-caps), masks,
//               exchanges the half-row max with its partner warp through
//               shared memory, keeps a running max and sum, writes its half of
//               P as bf16/fp16 into shared memory (the A operand of the P V
//               MMA) and rescales its half of O in TMEM only when the max grows
//               by more than 2^8.  The epilogue divides O by the sum and writes
//               o and the natural-log lse (or an fp32 partial state when the
//               plan split the key range).
// Every wait is bounded; a wait that runs out records kErrWaitTimeout and
// makes all roles leave their loops, the MMA thread waits for its issued
// MMAs, and TMEM is released.
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
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kD = 128;                 // head_dim of the prefill kernel
constexpr int kBM = kPrefillRows;       // packed query rows per tile
constexpr int kBN = kPrefillKeys;       // keys per block
constexpr int kThreads = 352;           // K producer, MMA, 8 softmax warps, V producer
constexpr int kVWarp = 10;              // the V producer
constexpr uint32_t kTile = 32768;       // 128 rows x 128 16-bit values
constexpr uint32_t kHalf = 16384;       // one 64-column half of a tile
constexpr int kKStages = 3;             // K blocks in flight (gather latency is ~2 key blocks)
constexpr int kVStages = 2;
// Shared-memory map (offsets from a 1024-aligned base).
constexpr uint32_t kOffQ = 0, kOffK = kTile, kOffV = kOffK + kKStages * kTile, kOffP = kOffV + kVStages * kTile,
                   kOffBar = kOffP + kTile, kOffRed = kOffBar + 256;
// The tiles need 1024-byte alignment and the budget leaves no slack to align
// by hand: the kernel checks that dynamic shared memory starts aligned.
constexpr int kSmemBytes = kOffRed + 2 * 2 * kPrefillRows * 4;
static_assert(kSmemBytes <= 232448, "shared memory budget");
// Barrier slots.
enum { Q_FULL = 0, Q_EMPTY = 1, K_FULL = 2, K_EMPTY = K_FULL + kKStages, V_FULL = K_EMPTY + kKStages,
       V_EMPTY = V_FULL + kVStages, S_FULL = V_EMPTY + kVStages, P_FULL = S_FULL + 2, O_DONE = P_FULL + 1,
       O_FREE = O_DONE + 1, V_LOAD = O_FREE + 1, DRAIN = V_LOAD + kVStages, NUM_BARS = DRAIN + 1 };
static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");
constexpr uint32_t kSoftmaxThreads = 256;
constexpr uint32_t kTmemCols = 512;     // S0 [0,128), S1 [128,256), O [256,384)
constexpr uint32_t kColO = 256;

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

template <int G, typename T, bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tkv) {
  constexpr uint32_t kFmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t base = smem_addr(sm);
  if (base & 1023u) {  // never expected; refuse rather than misread swizzled tiles
    if (threadIdx.x == 0) atomicOr(a.err, kErrTmemAlloc);
    return;
  }
  const uint32_t sQ = base + kOffQ, sP = base + kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS + 1);
  auto bar = [&](int i) { return base + kOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NUM_BARS; ++i)
      mbar_init(bar(i), (i == P_FULL || i == O_FREE) ? kSoftmaxThreads : 1);
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
  if (static_cast<int>(blockIdx.x) < hdr->num_workers) {
    t_begin = a.worker_ptr[blockIdx.x];
    t_end = a.worker_ptr[blockIdx.x + 1];
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
        mbar_arrive_expect_tx(bar(Q_FULL), kTile);
        tma_load_3d(sQ, &tq, 0, t.kvh * G, t.q_row0, bar(Q_FULL));
        tma_load_3d(sQ + kHalf, &tq, 64, t.kvh * G, t.q_row0, bar(Q_FULL));
      }
      const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
      const int n_pages_req = ceil_div_i(t.kv_len, P);
      int id_next = n > 0 ? page_of(t, 0, n_pages_req) : num_pages;
      for (int j = 0; j < n; ++j) {
        const int id = id_next;
        if (j + 1 < n) id_next = page_of(t, j + 1, n_pages_req);  // next block's page ids load meanwhile
        const int s = kvc % kKStages;
        if (kvc >= kKStages) {
          ok = __all_sync(kFull, wait(bar(K_EMPTY + s), ((kvc / kKStages) - 1) & 1));
          if (!ok) break;
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
      int id_next = n > 0 ? page_of(t, 0, n_pages_req) : num_pages;
      for (int j = 0; j < n; ++j) {
        const int id = id_next;
        if (j + 1 < n) id_next = page_of(t, j + 1, n_pages_req);
        const int s = kvc % kVStages;
        if (kvc >= kVStages) {
          ok = __all_sync(kFull, wait(bar(V_EMPTY + s), ((kvc / kVStages) - 1) & 1));
          if (!ok) break;
        }
        const uint32_t sV = base + kOffV + s * kTile;
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
      const uint32_t id_s = umma_idesc_f16(kFmt, kBM, kBN, 0);
      const uint32_t id_o = umma_idesc_f16(kFmt, kBM, kD, 1);
      int kvc = 0, pc = 0, ofree = 0;
      bool o_used = false;  // an earlier tile accumulated into O: wait for its epilogue first
      bool ok = true;
      // O += P_c V_c for the key block with global count c (the i-th of its tile).
      auto pv = [&](int c, int i) -> bool {
        if (i == 0 && o_used) {
          if (!wait(bar(O_FREE), ofree & 1)) return false;
          ++ofree;
        }
        if (!wait(bar(P_FULL), pc & 1)) return false;
        ++pc;
        const int s = c % kVStages;
        if (!wait(bar(V_FULL + s), (c / kVStages) & 1)) return false;
        tc_fence_after();
        const uint32_t sV = base + kOffV + s * kTile;
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_f16(tmem + kColO, sw128_desc(sP + (kk / 4) * kHalf + (kk % 4) * 32, 16, 1024),
                   sw128_desc(sV + kk * 2048, kHalf, 1024), id_o, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(V_EMPTY + s));
        umma_commit(bar(O_DONE));
        o_used = true;
        return true;
      };
      for (int ti = t_begin, tn = 0; ti < t_end && ok; ++ti, ++tn) {
        const PrefillTile t = a.tiles[ti];
        const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
        if (!(ok = wait(bar(Q_FULL), tn & 1))) break;
        tc_fence_after();
        for (int j = 0; j < n; ++j) {
          const int s = kvc % kKStages;
          if (!(ok = wait(bar(K_FULL + s), (kvc / kKStages) & 1))) break;
          tc_fence_after();
          const uint32_t sK = base + kOffK + s * kTile;
          const uint32_t d_s = tmem + (kvc & 1) * kBN;
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t koff = (kk / 4) * kHalf + (kk % 4) * 32;
            umma_f16(d_s, sw128_desc(sQ + koff, 16, 1024), sw128_desc(sK + koff, 16, 1024), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(S_FULL + (kvc & 1)));
          umma_commit(bar(K_EMPTY + s));
          if (j == n - 1) umma_commit(bar(Q_EMPTY));  // Q is free once the tile's last S is done
          if (j >= 1 && !(ok = pv(kvc - 1, j - 1))) break;
          ++kvc;
        }
        if (!ok) break;
        if (n >= 1) {
          if (!(ok = pv(kvc - 1, n - 1))) break;
        } else {
          umma_commit(bar(Q_EMPTY));
        }
      }
      // Every MMA issued so far must finish before TMEM is released.
      umma_commit(bar(DRAIN));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar(DRAIN), 0))
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int hf = (warp - 2) >> 2;          // which 64 keys / O columns of the row
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t pair_bar = 1 + quarter;   // the two warps of this lane quarter
    float* red = reinterpret_cast<float*>(sm + kOffRed);  // [parity][half][row] half-row maxima / sums
    const float scale = CAP ? a.sm_scale : a.sm_scale * kLog2e;
    uint8_t* pgen = sm + kOffP;
    constexpr int kH = kBN / 2;
    int kvc = 0, odc = 0;
    bool ok = true;
    for (int ti = t_begin; ti < t_end && ok; ++ti) {
      const PrefillTile t = a.tiles[ti];
      const int n = ceil_div_i(t.kv_end - t.kv_begin, kBN);
      const int rpos = r / G;
      const bool row_valid = rpos < t.n_pos;
      const int pos = t.q_pos0 + rpos;
      int limit = t.kv_len, lim0 = t.kv_len;  // keys < limit are visible to this row / to every row
      if (a.causal) {
        limit = min(limit, pos + 1 + t.kv_len - t.qo_len);
        lim0 = min(lim0, t.q_pos0 + 1 + t.kv_len - t.qo_len);
      }
      limit = min(limit, t.kv_end);
      lim0 = min(lim0, t.kv_end);
      float m_ref = -INFINITY, l = 0.f;  // l: this half-row's share of the sum
      for (int j = 0; j < n; ++j) {
        const int b = kvc & 1;
        if (!(ok = __all_sync(kFull, wait(bar(S_FULL + b), (kvc >> 1) & 1)))) break;
        tc_fence_after();
        uint32_t sr[kH];
        tmem_ld64_sync(tmem + lane_off + b * kBN + hf * kH, sr);
        const int key0 = t.kv_begin + j * kBN + hf * kH;
        const bool full = key0 + kH <= lim0;
        // Logits in log2 units are x * mul; the max is taken on x (mul > 0).
        float mul = scale;
        if constexpr (CAP) {
#pragma unroll
          for (int i = 0; i < kH; ++i)
            sr[i] = __float_as_uint(a.cap * tanhf(__uint_as_float(sr[i]) * scale / a.cap) * kLog2e);
          mul = 1.f;
        }
        if (!full) {
#pragma unroll
          for (int i = 0; i < kH; ++i)
            if (key0 + i >= limit) sr[i] = 0xff800000u;  // -inf
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int i = 8; i < kH; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
        const float mx_half = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                    fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * mul;
        // Whole-row max from the partner warp (slots alternate by block parity).
        red[(b * 2 + hf) * kBM + r] = mx_half;
        named_bar_sync(pair_bar, 64);
        const float mx = fmaxf(mx_half, red[(b * 2 + (hf ^ 1)) * kBM + r]);
        const float m_new = fmaxf(m_ref, mx);
        const bool resc = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_ref + 8.f);
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
        }
        const float sub = (m_ref == -INFINITY) ? 0.f : m_ref;
        // p = 2^(x * mul - sub): packed FMAs, three of every four exponentials on the
        // SFU and one on the FMA pipe, sum in four packed partial sums.
        float x[kH];
        const float2 mul2 = make_float2(mul, mul), nsub2 = make_float2(-sub, -sub);
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kH; i += 2) {
          float2 v = ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), mul2, nsub2);
          v.x = fast_exp2(v.x);
          v.y = ((i >> 1) & 1) ? exp2_poly3(v.y) : fast_exp2(v.y);
          x[i] = v.x;
          x[i + 1] = v.y;
          sum4[(i >> 1) & 3] = fadd2(sum4[(i >> 1) & 3], v);
        }
        const float2 s4 = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
        l += s4.x + s4.y;
        if (j >= 1) {
          // P V of the previous block must be done before O is rescaled and P overwritten.
          if (!(ok = __all_sync(kFull, wait(bar(O_DONE), odc & 1)))) break;
          ++odc;
          tc_fence_after();
          if (__any_sync(kFull, resc)) {
#pragma unroll
            for (int c = 0; c < kH / 32; ++c) {
              uint32_t rr[32];
              const uint32_t addr = tmem + lane_off + kColO + hf * kH + c * 32;
              tmem_ld32_sync(addr, rr);
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st32(addr, rr);
            }
            tmem_wait_st();
          }
        }
        // This half of the P row -> shared memory, 128B-swizzled K-major: keys
        // 0-63 are the first 64-column half of the operand, keys 64-127 the second.
#pragma unroll
        for (int cc = 0; cc < kH / 8; ++cc) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = x[cc * 8 + e];
          *reinterpret_cast<uint4*>(pgen + hf * kHalf + r * 128 + ((cc ^ (r & 7)) << 4)) = from_float8<T>(f);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(P_FULL));
        ++kvc;
      }
      if (!ok) break;
      if (n >= 1) {
        if (!(ok = __all_sync(kFull, wait(bar(O_DONE), odc & 1)))) break;
        ++odc;
        tc_fence_after();
      }
      // Whole-row sum: the parity slot of the next block is free; a second barrier
      // keeps the partner from reusing it before both have read.
      const int pb = kvc & 1;
      red[(pb * 2 + hf) * kBM + r] = l;
      named_bar_sync(pair_bar, 64);
      const float l_row = l + red[(pb * 2 + (hf ^ 1)) * kBM + r];
      named_bar_sync(pair_bar, 64);
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
      const float lse_v = l_row > 0.f ? (m_ref + log2f(l_row)) * kLn2 : -INFINITY;
      const int64_t orow = static_cast<int64_t>(t.q_row0 + rpos) * a.num_qo_heads + t.kvh * G + (r % G);
#pragma unroll
      for (int c = 0; c < kH / 32; ++c) {
        const int col = hf * kH + c * 32;
        float ov[32];
        if (n >= 1) {
          uint32_t rr[32];
          tmem_ld32_sync(tmem + lane_off + kColO + col, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(rr[i]) * inv;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
        if (t.slot < 0) {
          if (row_valid) {
            T* dst = static_cast<T*>(a.o) + orow * kD + col;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = ov[q * 8 + e];
              reinterpret_cast<uint4*>(dst)[q] = from_float8<T>(f);
            }
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.part_o + (static_cast<int64_t>(t.slot) * kBM + r) * kD + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
      }
      if (hf == 0) {
        if (t.slot < 0) {
          if (row_valid && a.lse) a.lse[orow] = lse_v;
        } else {
          a.part_lse[static_cast<int64_t>(t.slot) * kBM + r] = lse_v;
        }
      }
      if (n >= 1) {  // this tile's O is free for the next tile's P V
        tc_fence_before();
        mbar_arrive(bar(O_FREE));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Rows of query tiles whose key range the plan split: one warp per packed row,
// lanes over head_dim, log-sum-exp merge of the chunks' fp32 partial states.
template <typename T>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const __grid_constant__ PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp_id = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * 8;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int pairs = a.hdr->num_merge * kBM;
  for (int pair = warp_id; pair < pairs; pair += n_warps) {
    const PrefillMerge it = a.merge[pair / kBM];
    const int r = pair % kBM;
    if (r / G >= it.n_pos) continue;
    float mx = -INFINITY;
    for (int i = lane; i < it.n_slots; i += 32)
      mx = fmaxf(mx, a.part_lse[static_cast<int64_t>(it.slot_begin + i) * kBM + r]);
    mx = warp_max(mx);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int i = 0; i < it.n_slots; ++i) {
        const int64_t row = static_cast<int64_t>(it.slot_begin + i) * kBM + r;
        const float w = fast_exp2((a.part_lse[row] - mx) * kLog2e);
        if (w > 0.f) {
          const float4 v = reinterpret_cast<const float4*>(a.part_o + row * kD)[lane];
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
          acc[2] = fmaf(w, v.z, acc[2]);
          acc[3] = fmaf(w, v.w, acc[3]);
          wsum += w;
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t orow = static_cast<int64_t>(it.q_row0 + r / G) * a.num_qo_heads + it.kvh * G + (r % G);
    T* dst = static_cast<T*>(a.o) + orow * kD + lane * 4;
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = from_float<T>(acc[v] * inv);
    if (lane == 0 && a.lse) a.lse[orow] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <typename T>
cudaError_t launch_t(const PrefillArgs& a, int G, bool cap, int grid, const CUtensorMap& tq, const CUtensorMap& tkv,
                     cudaStream_t s) {
  void (*kern)(PrefillArgs, CUtensorMap, CUtensorMap) = nullptr;
#define PKV_PF_CASE(GG)                                                                      \
  case GG:                                                                                   \
    kern = cap ? prefill_kernel<GG, T, true> : prefill_kernel<GG, T, false>;                 \
    break;
  switch (G) {
    PKV_PF_CASE(1) PKV_PF_CASE(2) PKV_PF_CASE(4) PKV_PF_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef PKV_PF_CASE
  cudaError_t e = ensure_smem_limit(kern, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, s>>>(a, tq, tkv);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int head_dim, int group, int dtype, int page_size) {
  return head_dim == kD && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == PKV_F16 || dtype == PKV_BF16) &&
         (page_size == 8 || page_size == 16 || page_size == 32 || page_size == 64 || page_size == 128);
}

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, int group, int dtype, bool cap, int grid,
                           int64_t total_q, int64_t num_pages, cudaStream_t stream) {
  if (!prefill_supported(head_dim, group, dtype, a.page_size)) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t hq = a.num_qo_heads, hkv = a.num_kv_heads, P = a.page_size;
  CUtensorMap tq, tkv;
  {
    // q [total_q, Hq, D]: box = 64 columns x the G heads of a group x 128/G positions.
    cuuint64_t dims[3] = {kD, hq, static_cast<cuuint64_t>(total_q > 0 ? total_q : 1)};
    cuuint64_t strides[2] = {kD * 2, hq * kD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(kBM / group)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tq, dt, 3, const_cast<void*>(a.q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // kv_data [num_pages, 2, Hkv, P, D]: box = 64 columns x the P rows of one (page, K|V, head).
    cuuint64_t dims[5] = {kD, P, hkv, 2, static_cast<cuuint64_t>(num_pages > 0 ? num_pages : 1)};
    cuuint64_t strides[4] = {kD * 2, P * kD * 2, hkv * P * kD * 2, 2 * hkv * P * kD * 2};
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(P), 1, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (encode(&tkv, dt, 5, const_cast<void*>(a.kv), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (dtype == PKV_BF16) return launch_t<__nv_bfloat16>(a, group, cap, grid, tq, tkv, stream);
  return launch_t<__half>(a, group, cap, grid, tq, tkv, stream);
}

cudaError_t launch_prefill_merge(const PrefillArgs& a, int head_dim, int group, int dtype, int grid,
                                 cudaStream_t stream) {
  if (head_dim != kD || group <= 0) return cudaErrorInvalidValue;
  if (dtype == PKV_BF16)
    prefill_merge_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
  else if (dtype == PKV_F16)
    prefill_merge_kernel<__half><<<grid, 256, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pkv
