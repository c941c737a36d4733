// merge.cu -- merge_state: log-sum-exp composition of two attention states, and
// of n states laid out one after another (merge_states).
//
// Two states (o_a, lse_a), (o_b, lse_b) over disjoint key sets combine into
// the state over their union ("FlashInfer" guide, section 3: cascade
// attention merges the shared-prefix output with each request's suffix output
// "using online softmax correction"; FlashDecoding merges partial outputs the
// same way):  m = max(lse_a, lse_b),  w_x = exp(lse_x - m),
//             o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = m + ln(w_a + w_b).
//
// Elementwise and HBM-bound: one thread per 16-byte chunk of a row, the
// chunks of one (row, head) inside one warp so that lse can be read by all of
// them before any lane overwrites it (lse_out may alias lse_a).
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_bsr.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

template <typename T>
struct Chunk;  // 16 bytes of T as floats
template <>
struct Chunk<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float (&f)[N]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void store(void* p, const float (&f)[N]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <typename H>
struct Chunk16 {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float (&f)[N]) { to_float8<H>(*reinterpret_cast<const uint4*>(p), f); }
  __device__ static void store(void* p, const float (&f)[N]) { *reinterpret_cast<uint4*>(p) = from_float8<H>(f); }
};
template <>
struct Chunk<__nv_bfloat16> : Chunk16<__nv_bfloat16> {};
template <>
struct Chunk<__half> : Chunk16<__half> {};

template <typename T>
__global__ void __launch_bounds__(256) merge_state_kernel(const uint8_t* o_a, const float* lse_a,
                                                          const uint8_t* o_b, const float* lse_b,
                                                          uint8_t* o_out, float* lse_out, int64_t rows,
                                                          int chunks) {
  using C = Chunk<T>;
  // Launched as a programmatic dependent of whatever kernel precedes it on the
  // stream: wait until that grid has finished and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int per_warp = 32 / chunks;  // (row, head) pairs per warp
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int chunk = lane % chunks;
  for (int64_t base = warp_id * per_warp; base < rows; base += n_warps * per_warp) {
    const int64_t r = base + lane / chunks;
    const bool valid = r < rows;
    const float la = valid ? lse_a[r] : -INFINITY;
    const float lb = valid ? lse_b[r] : -INFINITY;
    __syncwarp();
    if (valid) {
      const float m = fmaxf(la, lb);
      const int64_t off = (r * chunks + chunk) * 16;
      float out[C::N];
      float lse;
      if (m == -INFINITY) {
#pragma unroll
        for (int i = 0; i < C::N; ++i) out[i] = 0.f;
        lse = -INFINITY;
      } else {
        const float wa = expf(la - m), wb = expf(lb - m);
        const float s = wa + wb, inv = 1.f / s;
        float fa[C::N], fb[C::N];
        C::load(o_a + off, fa);
        C::load(o_b + off, fb);
#pragma unroll
        for (int i = 0; i < C::N; ++i) {
          const float ta = wa > 0.f ? wa * fa[i] : 0.f;  // an empty state adds nothing
          const float tb = wb > 0.f ? wb * fb[i] : 0.f;
          out[i] = (ta + tb) * inv;
        }
        lse = m + logf(s);
      }
      C::store(o_out + off, out);
      if (chunk == 0 && lse_out) lse_out[r] = lse;
    }
  }
}

// n states of each (row, head), state k at rows k * stride + r: m = max_k lse_k,
// w_k = exp(lse_k - m), o = sum_k w_k o_k / sum_k w_k, lse = m + ln(sum_k w_k).
// Each lane reads its chunk of every state before writing it, and every lane of a
// (row, head) reads the lse values before any lane writes one, so the output may
// be one of the states (in place).
template <typename T>
__global__ void __launch_bounds__(256) merge_states_kernel(const uint8_t* o_in, const float* lse_in, int n_states,
                                                           int64_t stride, uint8_t* o_out, float* lse_out,
                                                           int64_t rows, int chunks) {
  using C = Chunk<T>;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int per_warp = 32 / chunks;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int chunk = lane % chunks;
  for (int64_t base = warp_id * per_warp; base < rows; base += n_warps * per_warp) {
    const int64_t r = base + lane / chunks;
    const bool valid = r < rows;
    float m = -INFINITY;
    if (valid)
      for (int k = 0; k < n_states; ++k) m = fmaxf(m, lse_in[k * stride + r]);
    float out[C::N];
#pragma unroll
    for (int i = 0; i < C::N; ++i) out[i] = 0.f;
    float s = 0.f;
    if (valid && m != -INFINITY) {
      for (int k = 0; k < n_states; ++k) {
        const float w = expf(lse_in[k * stride + r] - m);
        if (w > 0.f) {  // an empty state adds nothing (its o is not read)
          float f[C::N];
          C::load(o_in + ((k * stride + r) * chunks + chunk) * 16, f);
#pragma unroll
          for (int i = 0; i < C::N; ++i) out[i] = fmaf(w, f[i], out[i]);
          s += w;
        }
      }
    }
    __syncwarp();  // every lane has read the states' lse values
    if (valid) {
      const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
      for (int i = 0; i < C::N; ++i) out[i] *= inv;
      C::store(o_out + (r * chunks + chunk) * 16, out);
      if (chunk == 0 && lse_out) lse_out[r] = s > 0.f ? m + logf(s) : -INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                               void* o_out, float* lse_out, int64_t rows, int head_dim, int dtype,
                               cudaStream_t stream) {
  const int elem = dtype == PKV_F32 ? 4 : 2;
  const int bytes = head_dim * elem;
  if (bytes % 16) return cudaErrorInvalidValue;
  const int chunks = bytes / 16;
  if (chunks > 32 || (chunks & (chunks - 1))) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  const int per_warp = 32 / chunks;
  const int64_t warps = (rows + per_warp - 1) / per_warp;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (warps + 7) / 8;
  const int grid = static_cast<int>(want < sms * 8 ? want : sms * 8);
  auto a = static_cast<const uint8_t*>(o_a);
  auto b = static_cast<const uint8_t*>(o_b);
  auto o = static_cast<uint8_t*>(o_out);
  // A programmatic dependent of the kernel that produced the states: its CTAs
  // are placed as that grid's CTAs exit and wait for the whole grid before reading.
  switch (dtype) {
    case PKV_F32:
      return launch_dependent(merge_state_kernel<float>, grid, 256, 0, stream, a, lse_a, b, lse_b, o, lse_out, rows,
                              chunks);
    case PKV_BF16:
      return launch_dependent(merge_state_kernel<__nv_bfloat16>, grid, 256, 0, stream, a, lse_a, b, lse_b, o, lse_out,
                              rows, chunks);
    case PKV_F16:
      return launch_dependent(merge_state_kernel<__half>, grid, 256, 0, stream, a, lse_a, b, lse_b, o, lse_out, rows,
                              chunks);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge_states(const void* o_in, const float* lse_in, int n_states, int64_t stride, void* o_out,
                                float* lse_out, int64_t rows, int head_dim, int dtype, cudaStream_t stream) {
  const int elem = dtype == PKV_F32 ? 4 : 2;
  const int bytes = head_dim * elem;
  if (bytes % 16) return cudaErrorInvalidValue;
  const int chunks = bytes / 16;
  if (chunks > 32 || (chunks & (chunks - 1))) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  const int per_warp = 32 / chunks;
  const int64_t warps = (rows + per_warp - 1) / per_warp;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (warps + 7) / 8;
  const int grid = static_cast<int>(want < sms * 8 ? want : sms * 8);
  auto in = static_cast<const uint8_t*>(o_in);
  auto o = static_cast<uint8_t*>(o_out);
  switch (dtype) {
    case PKV_F32:
      return launch_dependent(merge_states_kernel<float>, grid, 256, 0, stream, in, lse_in, n_states, stride, o,
                              lse_out, rows, chunks);
    case PKV_BF16:
      return launch_dependent(merge_states_kernel<__nv_bfloat16>, grid, 256, 0, stream, in, lse_in, n_states, stride,
                              o, lse_out, rows, chunks);
    case PKV_F16:
      return launch_dependent(merge_states_kernel<__half>, grid, 256, 0, stream, in, lse_in, n_states, stride, o,
                              lse_out, rows, chunks);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
