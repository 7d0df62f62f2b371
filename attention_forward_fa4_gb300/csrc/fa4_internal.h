// fa4_internal.h -- host-side declarations shared by the library's
// translation units (one per head dimension, plus the C-ABI layer).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fa4_fwd_kernel.cuh"

namespace fa4 {

// Raise KERNEL's dynamic shared-memory limit to `bytes` once per device (the
// attribute stays set in the device's context; later launches skip the
// call). One flag bit per device index below 64; others set it every time.
template <auto KERNEL>
cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0ull};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return cudaSuccess;
  e = cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Enqueue the forward kernel for head dim 64 / 128. `emu_period` is 0
// (MUFU.EX2 only), 8 or 4 (one entry pair in 8 / in 4 through the
// software 2^x).
// `persistent` picks the instantiation whose CTAs visit work tiles in turn
// (grid <= SM count); otherwise the grid has one CTA per work tile. The
// _traced forms record the cycle trace (FwdParams::trace).
#define FA4_DECLARE_LAUNCH(name)                                                              \
  cudaError_t name(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,         \
                   const FwdParams& p, bool causal, int emu_period, bool persistent, unsigned grid, \
                   cudaStream_t stream);
FA4_DECLARE_LAUNCH(launch_fwd_d64)
FA4_DECLARE_LAUNCH(launch_fwd_d128)
FA4_DECLARE_LAUNCH(launch_fwd_d64_traced)
FA4_DECLARE_LAUNCH(launch_fwd_d128_traced)
#undef FA4_DECLARE_LAUNCH

// Attention backward (fa4_bwd.cu): zero dq_acc, preprocess (lse2, delta),
// main kernel (dK, dV, dQ reduce-adds), dq_acc -> dq.
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const __nv_bfloat16* o,
                       const __nv_bfloat16* dout,
                       const float* lse, __nv_bfloat16* dq, __nv_bfloat16* dk, __nv_bfloat16* dv,
                       float* dq_acc, float* lse2, float* delta, int* dq_turn, int* cta_ticket,
                       int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale, bool causal,
                       long long test_stall_cycles, unsigned int* status, cudaStream_t s);

// FP8 forward (e4m3 Q, K, V; head dim 128).
cudaError_t launch_fwd_d128_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, bool causal, bool persistent, unsigned grid,
                                cudaStream_t stream);

// Largest number of key-range splits fa4_fwd_splitkv accepts.
constexpr int kMaxSplits = 128;

// Combine n_splits partial results (o_part [n][B][Sq][Hq][d] fp32 softmax-
// normalised outputs, lse_part [n][B][Hq][Sq] natural-log LSE, -inf for an
// empty split) into o (BF16) and lse.
cudaError_t launch_merge_splits(const float* o_part, const float* lse_part, __nv_bfloat16* o,
                                float* lse, int n_splits, int B, int Sq, int Hq, int d,
                                cudaStream_t stream);

}  // namespace fa4
