// fa4_launch.cuh -- host-side launch of one forward kernel instantiation.
// Included by the per-head-dimension translation units, which instantiate
// it for their head dimension with trace marks compiled in or out.
#pragma once
#include "fa4_internal.h"

namespace fa4 {
namespace detail {

template <int D, bool CAUSAL, int EMU, bool PERSIST, bool TRACE, bool FP8 = false>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, unsigned grid, cudaStream_t stream) {
  constexpr int kSmem = Smem<D, FP8>::kAlloc;
  constexpr auto kernel = fa4_fwd_kernel<D, CAUSAL, EMU, PERSIST, TRACE, FP8>;
  cudaError_t err = set_smem_once<kernel>(kSmem);
  if (err != cudaSuccess) return err;
  kernel<<<grid, kThreads, kSmem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// causal / non-causal x MUFU-only / one entry pair in 8 or in 4 through
// the software 2^x x one CTA per work tile / persistent grid.
template <int D, bool TRACE>
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, bool causal, int emu_period, bool persistent,
                       unsigned grid, cudaStream_t stream) {
#define FA4_LAUNCH(C, E) \
  (persistent ? launch_one<D, C, E, true, TRACE>(tq, tk, tv, p, grid, stream) \
              : launch_one<D, C, E, false, TRACE>(tq, tk, tv, p, grid, stream))
  if (causal) {
    if (emu_period == 8) return FA4_LAUNCH(true, 8);
    if (emu_period == 4) return FA4_LAUNCH(true, 4);
    return FA4_LAUNCH(true, 0);
  }
  if (emu_period == 8) return FA4_LAUNCH(false, 8);
  if (emu_period == 4) return FA4_LAUNCH(false, 4);
  return FA4_LAUNCH(false, 0);
#undef FA4_LAUNCH
}

}  // namespace detail
}  // namespace fa4
