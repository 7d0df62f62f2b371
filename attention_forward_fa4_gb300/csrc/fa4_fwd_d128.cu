// fa4_fwd_d128.cu -- instantiations of the forward kernel for head dim 128
// (causal / non-causal x MUFU-only / one entry pair in 8 through the
// software 2^x x one CTA per work tile / persistent grid).
#include "fa4_internal.h"

namespace fa4 {
namespace {

template <bool CAUSAL, int EMU, bool PERSIST>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, unsigned grid, cudaStream_t stream) {
  constexpr int kSmem = Smem<128>::kAlloc;
  auto kernel = fa4_fwd_kernel<128, CAUSAL, EMU, PERSIST>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  kernel<<<grid, kThreads, kSmem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <bool CAUSAL, int EMU>
cudaError_t launch_grid(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const FwdParams& p, bool persistent, unsigned grid, cudaStream_t stream) {
  return persistent ? launch_one<CAUSAL, EMU, true>(tq, tk, tv, p, grid, stream)
                    : launch_one<CAUSAL, EMU, false>(tq, tk, tv, p, grid, stream);
}

}  // namespace

cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, int emu_period, bool persistent,
                            unsigned grid, cudaStream_t stream) {
  if (causal)
    return emu_period ? launch_grid<true, 8>(tq, tk, tv, p, persistent, grid, stream)
                      : launch_grid<true, 0>(tq, tk, tv, p, persistent, grid, stream);
  return emu_period ? launch_grid<false, 8>(tq, tk, tv, p, persistent, grid, stream)
                    : launch_grid<false, 0>(tq, tk, tv, p, persistent, grid, stream);
}

}  // namespace fa4
