// fa4_fwd_d128.cu -- instantiations of the forward kernel for head dim 128
// (causal / non-causal x MUFU-only / one entry pair in 8 through the
// software 2^x).
#include "fa4_internal.h"

namespace fa4 {
namespace {

template <bool CAUSAL, int EMU>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, unsigned grid, cudaStream_t stream) {
  constexpr int kSmem = Smem<128>::kAlloc;
  auto kernel = fa4_fwd_kernel<128, CAUSAL, EMU>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  kernel<<<grid, kThreads, kSmem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, bool causal, int emu_period, unsigned grid,
                           cudaStream_t stream) {
  if (causal)
    return emu_period ? launch_one<true, 8>(tq, tk, tv, p, grid, stream)
                      : launch_one<true, 0>(tq, tk, tv, p, grid, stream);
  return emu_period ? launch_one<false, 8>(tq, tk, tv, p, grid, stream)
                    : launch_one<false, 0>(tq, tk, tv, p, grid, stream);
}

}  // namespace fa4
