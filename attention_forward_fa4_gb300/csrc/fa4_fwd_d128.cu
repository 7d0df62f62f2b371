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

#ifdef FA4_PROF
// Diagnostic builds: read and clear the phase profile of the head-dim-128
// kernels (32 uint64 sums).
extern "C" int fa4_prof_read_d128(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, fa4::g_prof, sizeof(unsigned long long) * 32) != cudaSuccess) return 1;
  const unsigned long long z[32] = {};
  return cudaMemcpyToSymbol(fa4::g_prof, z, sizeof z) != cudaSuccess;
}
#endif
