// append.cu -- append new tokens' K/V into their pages, with the rotary
// position embedding (RoPE) of the new keys and of the queries fused into the
// same pass.
//
// The pages name both steps: serving has an "append" stage that adds the new
// tokens to the KV cache (greptalks MLSys 2025 talk summary, Background,
// "Dynamic Problem Shapes"), and the query/key transforms of an attention
// variant include RoPE, which FlashInfer fuses instead of running as a
// separate pass (fdeinterviews summary, "Customizable attention, compiled
// just in time").  Neither page fixes the
// rotation, so the embedding is the RoFormer one in its "rotate half" form:
// element i < D/2 of a head row pairs with element i + D/2, and the pair at
// position `pos` turns by the angle pos * theta^(-2i/D):
//     x'_i       = x_i cos a - x_{i+D/2} sin a
//     x'_{i+D/2} = x_{i+D/2} cos a + x_i sin a.
//
// Token t of request b's n_b new tokens (rows append_indptr[b] ..) sits at
// position kv_len_b - n_b + (t - append_indptr[b]), where kv_len_b comes from
// the page table that already includes the new tokens; its K and V go to page
// kv_indices[kv_indptr[b] + pos / P], slot pos % P.  The queries of those rows
// turn by the same positions.
//
// HBM-bound: one warp per token.  A head row of D elements is covered by D/16
// lanes, each holding 8 rotation pairs (16 bytes from each half), so a warp
// pass moves 32 / (D/16) head rows with 16-byte loads and stores and needs no
// shuffles.  Angles: theta^(-2i/D) comes from the host in double precision as
// an unevaluated float sum hi + lo; pos * (hi + lo) is reduced modulo 2 pi with
// an exact product error (fma) and a two-constant split of 2 pi (the
// Cody-Waite reduction), so |angle error| stays near 1e-6 rad even at
// positions of 10^5, before the fast hardware sine and cosine.
#include <cuda_runtime.h>
#include <math.h>

#include <cmath>

#include "pkv_bsr.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kAppendWarps = 8;
constexpr int kAppendThreads = kAppendWarps * 32;
constexpr int kMaxPairs = 64;          // D / 2 for the largest head_dim built (128)
constexpr int kIndptrSmem = 2048;      // append_indptr entries staged in shared memory

struct AppendArgs {
  const int32_t* append_indptr;  // [batch + 1] new-token rows per request
  const int32_t* kv_indptr;      // [batch + 1] pages per request (new tokens included)
  const int32_t* kv_indices;
  const int32_t* kv_last;        // [batch] valid slots of each last page
  const void* k_new;             // [nnz, Hkv, D]
  const void* v_new;             // [nnz, Hkv, D]
  void* kv;                      // [num_pages, 2, Hkv, P, D]
  const void* q_in;              // [nnz, Hq, D] or nullptr
  void* q_out;                   // [nnz, Hq, D]; may equal q_in
  int32_t* err;                  // device error word or nullptr
  int64_t num_pages;
  int64_t nnz;
  int batch;
  int num_qo_heads;
  int num_kv_heads;
  int page_size;
  int rope;                      // 0: keys and queries are copied unchanged
  float2 freq[kMaxPairs];        // theta^(-2i/D) = .x + .y
};

// 2 pi as a float plus the float nearest to the rest.
constexpr double k2Pi = 6.283185307179586476925286766559;
constexpr float k2PiHi = static_cast<float>(k2Pi);
constexpr float k2PiLo = static_cast<float>(k2Pi - static_cast<double>(k2PiHi));
constexpr float kInv2Pi = static_cast<float>(1.0 / k2Pi);

// Rotate (or copy) `passes` head rows of one token: lane (hsub, sub) handles
// head h0 + pass * HPP + hsub, pairs sub*8 .. sub*8+7.
template <int D, typename T, bool ROT, int CHUNK>
__device__ __forceinline__ void move_rows(const T* src, int64_t src_row0, T* dst_base,
                                          int64_t dst_head_stride, int heads, int sub, int hsub,
                                          const float (&c)[8], const float (&s)[8]) {
  constexpr int H2 = D / 2;
  constexpr int HPP = 32 / (D / 16);
  for (int h0 = 0; h0 < heads; h0 += CHUNK * HPP) {
    uint4 x1[CHUNK], x2[CHUNK];
#pragma unroll
    for (int k = 0; k < CHUNK; ++k) {
      const int h = h0 + k * HPP + hsub;
      if (h < heads) {
        const T* p = src + (src_row0 + h) * D + sub * 8;
        x1[k] = *reinterpret_cast<const uint4*>(p);
        x2[k] = *reinterpret_cast<const uint4*>(p + H2);
      }
    }
#pragma unroll
    for (int k = 0; k < CHUNK; ++k) {
      const int h = h0 + k * HPP + hsub;
      if (h < heads) {
        T* p = dst_base + h * dst_head_stride + sub * 8;
        if (ROT) {
          float a[8], b[8], ra[8], rb[8];
          to_float8<T>(x1[k], a);
          to_float8<T>(x2[k], b);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            ra[j] = fmaf(a[j], c[j], -b[j] * s[j]);
            rb[j] = fmaf(b[j], c[j], a[j] * s[j]);
          }
          *reinterpret_cast<uint4*>(p) = from_float8<T>(ra);
          *reinterpret_cast<uint4*>(p + H2) = from_float8<T>(rb);
        } else {
          *reinterpret_cast<uint4*>(p) = x1[k];
          *reinterpret_cast<uint4*>(p + H2) = x2[k];
        }
      }
    }
  }
}

template <int D, typename T, bool ROT>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int LPH = D / 16;  // lanes per head row
  __shared__ int32_t s_indptr[kIndptrSmem];
  // Launched as a programmatic dependent of the kernel before it on the stream:
  // nothing global is touched before that grid has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool staged = a.batch < kIndptrSmem;
  if (staged)
    for (int i = threadIdx.x; i <= a.batch; i += blockDim.x) s_indptr[i] = a.append_indptr[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane % LPH, hsub = lane / LPH;
  float fh[8], fl[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    fh[j] = ROT ? a.freq[sub * 8 + j].x : 0.f;
    fl[j] = ROT ? a.freq[sub * 8 + j].y : 0.f;
  }
  const int P = a.page_size;
  const int Hkv = a.num_kv_heads;
  const T* k_new = static_cast<const T*>(a.k_new);
  const T* v_new = static_cast<const T*>(a.v_new);
  T* kv = static_cast<T*>(a.kv);
  int32_t err = 0;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kAppendWarps + warp; t < a.nnz;
       t += static_cast<int64_t>(gridDim.x) * kAppendWarps) {
    // The request holding new row t: the last b with append_indptr[b] <= t.
    int lo = 0, hi = a.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      const int v = staged ? s_indptr[mid] : __ldg(a.append_indptr + mid);
      if (v <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int a0 = staged ? s_indptr[b] : __ldg(a.append_indptr + b);
    const int a1 = staged ? s_indptr[b + 1] : __ldg(a.append_indptr + b + 1);
    const int p0 = __ldg(a.kv_indptr + b);
    const int n_pages = __ldg(a.kv_indptr + b + 1) - p0;
    const int last = __ldg(a.kv_last + b);
    const int kv_len = n_pages > 0 ? (n_pages - 1) * P + last : 0;
    const int pos = kv_len - (a1 - a0) + static_cast<int>(t - a0);
    // A request claiming more new tokens than it holds is skipped whole.
    if (t < a0 || t >= a1 || a1 - a0 > kv_len || (n_pages > 0 && (last < 1 || last > P))) {
      err |= kErrAppendLayout;
      continue;
    }
    const int page = __ldg(a.kv_indices + p0 + pos / P);
    if (page < 0 || page >= a.num_pages) {
      err |= kErrPageIndex;
      continue;
    }
    float c[8], s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (ROT) {
        const float p = static_cast<float>(pos);
        const float ph = p * fh[j];
        const float pe = fmaf(p, fh[j], -ph);  // rounding error of p * fh, exactly
        const float k = rintf(ph * kInv2Pi);
        float r = fmaf(-k, k2PiHi, ph);
        r = fmaf(-k, k2PiLo, r);
        r += fmaf(p, fl[j], pe);
        __sincosf(r, &s[j], &c[j]);
      } else {
        c[j] = 1.f;
        s[j] = 0.f;
      }
    }
    const int slot = pos % P;
    // K of head h goes to ((page * 2 + 0) * Hkv + h) * P + slot, V to the same with 1.
    T* k_dst = kv + ((static_cast<int64_t>(page) * 2 * Hkv) * P + slot) * D;
    T* v_dst = k_dst + static_cast<int64_t>(Hkv) * P * D;
    const int64_t kv_row0 = t * Hkv;
    move_rows<D, T, ROT, 2>(k_new, kv_row0, k_dst, static_cast<int64_t>(P) * D, Hkv, sub, hsub, c, s);
    move_rows<D, T, false, 2>(v_new, kv_row0, v_dst, static_cast<int64_t>(P) * D, Hkv, sub, hsub, c, s);
    if (a.q_in) {
      const int Hq = a.num_qo_heads;
      move_rows<D, T, ROT, 4>(static_cast<const T*>(a.q_in), t * Hq, static_cast<T*>(a.q_out) + t * Hq * D,
                              D, Hq, sub, hsub, c, s);
    }
  }
  if (err && a.err) atomicOr(a.err, err);
}

template <int D, typename T>
cudaError_t launch_t(const AppendArgs& a, int grid, cudaStream_t s) {
  return a.rope ? launch_dependent(append_rope_kernel<D, T, true>, grid, kAppendThreads, 0, s, a)
                : launch_dependent(append_rope_kernel<D, T, false>, grid, kAppendThreads, 0, s, a);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_append_paged_kv(const pkv_params* p, int batch, int64_t nnz, int64_t num_pages,
                                          const int32_t* append_indptr_d, const int32_t* kv_indptr_d,
                                          const int32_t* kv_indices_d, const int32_t* kv_last_page_len_d,
                                          const void* k_new, const void* v_new, void* kv_data,
                                          const void* q_in, void* q_out, double rope_theta, int32_t* error_d,
                                          void* stream) {
  using namespace pkv;
  if (!p || batch < 0 || nnz < 0 || num_pages < 0) return PKV_ERR_INVALID_ARG;
  if (!(rope_theta >= 0.0) || !std::isfinite(rope_theta)) return PKV_ERR_INVALID_ARG;
  if (p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->page_size <= 0) return PKV_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (p->dtype != PKV_F16 && p->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (nnz == 0) return PKV_OK;
  if (batch == 0 || nnz > INT32_MAX) return PKV_ERR_INVALID_ARG;
  if (!append_indptr_d || !kv_indptr_d || !kv_indices_d || !kv_last_page_len_d || !k_new || !v_new || !kv_data)
    return PKV_ERR_INVALID_ARG;
  if (q_in && !q_out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_data) || (q_in && (!aligned16(q_in) || !aligned16(q_out))))
    return PKV_ERR_INVALID_ARG;
  AppendArgs a{};
  a.append_indptr = append_indptr_d;
  a.kv_indptr = kv_indptr_d;
  a.kv_indices = kv_indices_d;
  a.kv_last = kv_last_page_len_d;
  a.k_new = k_new;
  a.v_new = v_new;
  a.kv = kv_data;
  a.q_in = q_in;
  a.q_out = q_out;
  a.err = error_d;
  a.num_pages = num_pages;
  a.nnz = nnz;
  a.batch = batch;
  a.num_qo_heads = p->num_qo_heads;
  a.num_kv_heads = p->num_kv_heads;
  a.page_size = p->page_size;
  a.rope = rope_theta > 0.0 ? 1 : 0;
  const int pairs = p->head_dim / 2;
  if (a.rope) {
    const double l2 = std::log2(rope_theta);
    for (int i = 0; i < pairs; ++i) {
      const double f = std::exp2(-(2.0 * i / p->head_dim) * l2);
      const float hi = static_cast<float>(f);
      a.freq[i] = make_float2(hi, static_cast<float>(f - static_cast<double>(hi)));
    }
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  const int64_t want = (nnz + kAppendWarps - 1) / kAppendWarps;
  const int grid = static_cast<int>(want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8);
  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p->head_dim == 128)
    e = p->dtype == PKV_BF16 ? launch_t<128, __nv_bfloat16>(a, grid, s) : launch_t<128, __half>(a, grid, s);
  else
    e = p->dtype == PKV_BF16 ? launch_t<64, __nv_bfloat16>(a, grid, s) : launch_t<64, __half>(a, grid, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
