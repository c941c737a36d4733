// mixed_kernel.cuh -- one persistent launch for a batch that mixes prompt chunks
// (many query rows) with decodes (one query row).
//
// Method (FlashInfer pages): a serving batch holds both kinds of request and
// each gets its own kernel ("FlashInfer" guide, "Prefill-Decode Mixing"), with
// the query tile size, from 1 to 128, matched to the requests
// (fdeinterviews summary, "Customizable attention, compiled just in time"),
// inside persistent kernels of a fixed grid that a captured graph can replay
// (same summary, "Load balancing that survives CUDA graphs").  Both kinds in
// one launch is the direction the greptalks summary names under "Future
// Directions and Features".
//
// GB300 design.  One CTA per SM, 384 threads.  The plan splits the SMs in
// proportion to the estimated time of each half; the split is read from the
// decode half's table header (cta_offset), so a graph captured once stays
// valid after re-planning.
//   CTAs [0, cta_offset)      the tcgen05 prefill CTA (prefill_kernel.cuh)
//                             over the prefill half's tiles; the twelfth warp
//                             only joins its CTA-wide barriers.
//   CTAs [cta_offset, grid)   kDecodeWarps decode workers (decode_kernel.cuh)
//                             over the decode half's segments.
// The register file decides the thread count: the prefill CTA's 11 warps put
// up to three on a scheduler, which caps them at 168 registers, a launch of 384
// threads gets the same 168, and a decode worker wants about 230.  So in a
// decode CTA the third warpgroup gives its registers back (setmaxnreg.dec to
// 24) and exits, and the two warpgroups of workers raise theirs to 232
// (setmaxnreg.inc): 2 x 128 x (232 - 168) <= 128 x (168 - 24).  The host
// refuses to launch an instance whose launch register count is not 168, since
// the increase would otherwise wait for registers that never come.
#pragma once

#include "decode_kernel.cuh"
#include "prefill_kernel.cuh"

namespace pkv {
namespace mixed_impl {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;   // registers per thread the instances must launch with
constexpr int kDecodeRegs = 232;   // per decode worker thread after setmaxnreg.inc
constexpr int kIdleRegs = 24;      // per thread of the warpgroup that leaves
static_assert(kThreads / 32 == 12 && kDecodeWarps == 8, "two warpgroups of decode workers and one that leaves");
static_assert(2 * 128 * (kDecodeRegs - kLaunchRegs) <= 128 * (kLaunchRegs - kIdleRegs),
              "the decode workers' increase must fit in what the third warpgroup releases");
static_assert(kLaunchRegs * kThreads <= 65536, "launch register budget");

// Decode lanes per token for a head group of G (as the decode kernel picks them at head_dim 128).
template <int G>
struct MixedLpt {
  static constexpr int value = G == 8 ? 16 : 8;
};

template <int G, typename T>
struct MixedSmem {
  static constexpr int kDecStages = decode_impl::DecodeShape<128, T>::kStages;
  static constexpr int kDecBarOff = kDecodeWarps * kDecodeWarpSmem;
  static constexpr int kDecBytes = kDecBarOff + kDecodeWarps * kDecStages * 8;
};

template <int G, typename T, bool CAP, bool SMALL>
__global__ void __launch_bounds__(kThreads, 1)
    mixed_kernel(const __grid_constant__ PrefillArgs pa, const __grid_constant__ DecodeArgs da,
                 const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkv) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // Launched as a programmatic dependent of the kernel before it on the stream:
  // nothing global is touched before that grid has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int split = da.hdr->cta_offset;
  const int cta = static_cast<int>(blockIdx.x);
  if (cta < split) {
    prefill_impl::prefill_cta<G, T, CAP, false, SMALL, true>(pa, tq, tkv, cta, smem);
    return;
  }
  const int warp = threadIdx.x >> 5;
  if (warp >= kDecodeWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kIdleRegs));
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kDecodeRegs));
  using M = MixedSmem<G, T>;
  decode_impl::decode_worker<128, G, MixedLpt<G>::value, T, CAP, false>(
      da, (cta - split) * kDecodeWarps + warp, smem + warp * kDecodeWarpSmem,
      smem_addr(smem + M::kDecBarOff) + 8u * M::kDecStages * warp);
}

// Launch register count of one instance, queried once (later launches, e.g.
// inside CUDA-graph capture, make no attribute call).
template <int G, typename T, bool CAP, bool SMALL>
int launch_regs() {
  static const int regs = [] {
    cudaFuncAttributes attr;
    return cudaFuncGetAttributes(&attr, mixed_kernel<G, T, CAP, SMALL>) == cudaSuccess ? attr.numRegs : -1;
  }();
  return regs;
}

// Launch one instance (group size and cap chosen at run time) on `grid` CTAs.
template <typename T, bool SMALL>
cudaError_t launch_mixed_kernel(const PrefillArgs& pa, const DecodeArgs& da, int G, bool cap, int grid,
                                const CUtensorMap& tq, const CUtensorMap& tkv, cudaStream_t s) {
  void (*kern)(PrefillArgs, DecodeArgs, CUtensorMap, CUtensorMap) = nullptr;
  int dec_bytes = 0, regs = -1;
#define PKV_MX_CASE(GG)                                                                                    \
  case GG:                                                                                                 \
    kern = cap ? mixed_kernel<GG, T, true, SMALL> : mixed_kernel<GG, T, false, SMALL>;                     \
    regs = cap ? launch_regs<GG, T, true, SMALL>() : launch_regs<GG, T, false, SMALL>();                   \
    dec_bytes = MixedSmem<GG, T>::kDecBytes;                                                               \
    break;
  switch (G) {
    PKV_MX_CASE(1) PKV_MX_CASE(2) PKV_MX_CASE(4) PKV_MX_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef PKV_MX_CASE
  // setmaxnreg.inc in the decode CTAs counts on exactly this many registers at launch.
  if (regs != kLaunchRegs) return cudaErrorInvalidValue;
  const int pre_bytes = SMALL ? prefill_impl::kSmemBytesSmall : prefill_impl::kSmemBytes;
  const int smem = pre_bytes > dec_bytes ? pre_bytes : dec_bytes;
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, kThreads, smem, s, pa, da, tq, tkv);
}

extern template cudaError_t launch_mixed_kernel<__nv_bfloat16, false>(const PrefillArgs&, const DecodeArgs&, int,
                                                                      bool, int, const CUtensorMap&,
                                                                      const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_mixed_kernel<__half, false>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                               const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_mixed_kernel<__nv_bfloat16, true>(const PrefillArgs&, const DecodeArgs&, int,
                                                                     bool, int, const CUtensorMap&,
                                                                     const CUtensorMap&, cudaStream_t);
extern template cudaError_t launch_mixed_kernel<__half, true>(const PrefillArgs&, const DecodeArgs&, int, bool, int,
                                                              const CUtensorMap&, const CUtensorMap&, cudaStream_t);

}  // namespace mixed_impl
}  // namespace pkv
