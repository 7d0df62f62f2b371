// fa4_fwd_fp8.cu -- forward kernel instantiations with e4m3 Q, K, V and P
// (head dim 128; causal / non-causal x one CTA per work tile / persistent
// grid; every exponential through MUFU.EX2).
#include "fa4_launch.cuh"

namespace fa4 {

cudaError_t launch_fwd_d128_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, bool causal, bool persistent, unsigned grid,
                                cudaStream_t stream) {
  using namespace detail;
  if (causal)
    return persistent ? launch_one<128, true, 0, true, false, true>(tq, tk, tv, p, grid, stream)
                      : launch_one<128, true, 0, false, false, true>(tq, tk, tv, p, grid, stream);
  return persistent ? launch_one<128, false, 0, true, false, true>(tq, tk, tv, p, grid, stream)
                    : launch_one<128, false, 0, false, false, true>(tq, tk, tv, p, grid, stream);
}

}  // namespace fa4
