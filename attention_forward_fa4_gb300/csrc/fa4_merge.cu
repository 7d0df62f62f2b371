// fa4_merge.cu -- combines the per-split partial results of the key-range
// split forward into the final output.
//
// Each split s produced, for every query row, the softmax-normalised output
// O_s over its own keys and the logsumexp L_s of those keys' scaled scores
// (-inf when the split held no visible key). The exact result over all keys
// is the LSE-weighted combination
//   L = log sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s,
// which follows from softmax(x) over a union of disjoint key sets
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", Method: the output is recovered exactly by
// the final normalisation, here applied once more across key ranges).
//
// Bandwidth-bound: one warp per output row (b, i, h); each lane owns D/32
// consecutive elements, so a warp reads a split's whole row in one
// coalesced pass and neighbouring warps read neighbouring rows.
#include <cuda_bf16.h>

#include "fa4_internal.h"

namespace fa4 {
namespace {

constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_splits_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                        __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int n_splits, int B,
                        int Sq, int Hq) {
  constexpr int kPer = D / 32;                   // elements per lane: 4 (D = 128) or 2 (D = 64)
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(B) * Sq * Hq;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  // row = (b * Sq + i) * Hq + h  (the layout of o)
  const int h = static_cast<int>(row % Hq);
  const int64_t bi = row / Hq;
  const int i = static_cast<int>(bi % Sq);
  const int b = static_cast<int>(bi / Sq);
  const int64_t lse_idx = (static_cast<int64_t>(b) * Hq + h) * Sq + i;
  const int64_t split_rows = rows;               // rows per split in o_part / lse_part
  float m = -INFINITY;
  for (int s = 0; s < n_splits; ++s) m = fmaxf(m, lse_part[s * split_rows + lse_idx]);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
  float sum = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ls = lse_part[s * split_rows + lse_idx];
      if (ls == -INFINITY) continue;
      const float wgt = __expf(ls - m);
      sum += wgt;
      const float* src = o_part + (s * split_rows + row) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y;
      }
    }
  }
  const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
  __nv_bfloat16* dst = o + row * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) lse[lse_idx] = sum > 0.0f ? m + logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge_splits(const float* o_part, const float* lse_part, __nv_bfloat16* o,
                                float* lse, int n_splits, int B, int Sq, int Hq, int d,
                                cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * Sq * Hq;
  const int64_t blocks = (rows + kMergeWarps - 1) / kMergeWarps;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d == 64)
    merge_splits_kernel<64><<<static_cast<unsigned>(blocks), kMergeWarps * 32, 0, stream>>>(
        o_part, lse_part, o, lse, n_splits, B, Sq, Hq);
  else
    merge_splits_kernel<128><<<static_cast<unsigned>(blocks), kMergeWarps * 32, 0, stream>>>(
        o_part, lse_part, o, lse, n_splits, B, Sq, Hq);
  return cudaGetLastError();
}

}  // namespace fa4
