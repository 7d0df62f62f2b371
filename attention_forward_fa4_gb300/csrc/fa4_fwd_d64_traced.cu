// fa4_fwd_d64_traced.cu -- forward kernel instantiations for head dim 64,
// with the cycle-trace marks compiled in.
#include "fa4_launch.cuh"

namespace fa4 {

cudaError_t launch_fwd_d64_traced(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, bool causal, int emu_period, bool persistent,
                         unsigned grid, cudaStream_t stream) {
  return detail::launch_fwd<64, true>(tq, tk, tv, p, causal, emu_period, persistent, grid, stream);
}

}  // namespace fa4
