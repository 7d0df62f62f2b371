// fa4_fwd_d128.cu -- forward kernel instantiations for head dim 128,
// without trace marks.
#include "fa4_launch.cuh"

namespace fa4 {

cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, bool causal, int emu_period, bool persistent,
                         unsigned grid, cudaStream_t stream) {
  return detail::launch_fwd<128, false>(tq, tk, tv, p, causal, emu_period, persistent, grid, stream);
}

}  // namespace fa4
