// fa4_bwd.cu -- host launch of the attention backward: a preprocessing
// kernel (Delta = rowsum(dO o O), LSE in log2 units, both padded to whole
// 128-row blocks), the tcgen05 main kernel (fa4_bwd_q64.cuh), and the
// conversion of the fp32 dQ accumulator to BF16.
#include <cuda_bf16.h>

#include "fa4_bwd_q64.cuh"
#include "fa4_internal.h"

namespace fa4 {
namespace {

// One warp per padded query row (b, h, i), i < Sq_pad: Delta = sum_e dO O in
// fp32 and LSE2 = LSE log2(e). Rows past Sq and rows without a visible key
// (LSE = -inf) get LSE2 = +inf, so every score of theirs exponentiates to 0.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ lse2,
                                                       float* __restrict__ delta, int B, int Hq,
                                                       int Sq, int Sq_pad) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(B) * Hq * Sq_pad;
  const int64_t id = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (id >= rows) return;
  const int i = static_cast<int>(id % Sq_pad);
  const int64_t bh = id / Sq_pad;
  const int h = static_cast<int>(bh % Hq);
  const int b = static_cast<int>(bh / Hq);
  float acc = 0.0f;
  float l2 = INFINITY;
  if (i < Sq) {
    const int64_t base = ((static_cast<int64_t>(b) * Sq + i) * Hq + h) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + base + e));
      const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + base + e));
      acc += a.x * g.x + a.y * g.y;
    }
    const float l = lse[(static_cast<int64_t>(b) * Hq + h) * Sq + i];
    l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    delta[id] = (i < Sq) ? acc : 0.0f;
    lse2[id] = l2;
  }
}

__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ src,
                                                             __nv_bfloat162* __restrict__ dst,
                                                             int64_t n4) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 x = src[i];
    dst[2 * i] = __floats2bfloat162_rn(x.x, x.y);
    dst[2 * i + 1] = __floats2bfloat162_rn(x.z, x.w);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_q64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                       unsigned grid, cudaStream_t s) {
  constexpr int kSmem = BwdQ64Smem<D>::kAlloc;
  constexpr auto kernel = fa4_bwd_q64_kernel<D, CAUSAL>;
  cudaError_t err = set_smem_once<kernel>(kSmem);
  if (err != cudaSuccess) return err;
  kernel<<<grid, kBwdQ64Threads, kSmem, s>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const __nv_bfloat16* o,
                       const __nv_bfloat16* dout,
                       const float* lse, __nv_bfloat16* dq, __nv_bfloat16* dk, __nv_bfloat16* dv,
                       float* dq_acc, float* lse2, float* delta, int* dq_turn, int* cta_ticket,
                       int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale, bool causal,
                       long long test_stall_cycles, unsigned int* status, cudaStream_t s) {
  const int Sq_pad = (Sq + 127) / 128 * 128;
  const int64_t dq_elems = static_cast<int64_t>(B) * Sq * Hq * d;
  cudaError_t err = cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(dq_elems) * 4, s);
  if (err != cudaSuccess) return err;
  if (dq_turn &&
      (err = cudaMemsetAsync(dq_turn, 0, static_cast<size_t>(B) * Hq * (Sq_pad / 64) * 4, s)) != cudaSuccess)
    return err;
  if (cta_ticket && (err = cudaMemsetAsync(cta_ticket, 0, sizeof(int), s)) != cudaSuccess) return err;
  const int64_t prep_rows = static_cast<int64_t>(B) * Hq * Sq_pad;
  const unsigned prep_blocks = static_cast<unsigned>((prep_rows + 7) / 8);
  if (d == 64)
    bwd_prep_kernel<64><<<prep_blocks, 256, 0, s>>>(o, dout, lse, lse2, delta, B, Hq, Sq, Sq_pad);
  else
    bwd_prep_kernel<128><<<prep_blocks, 256, 0, s>>>(o, dout, lse, lse2, delta, B, Hq, Sq, Sq_pad);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;

  BwdParams p;
  p.dk = dk;
  p.dv = dv;
  p.dq_acc = dq_acc;
  p.lse2 = lse2;
  p.delta = delta;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.Sq_pad = Sq_pad;
  p.n_kblk = (Sk + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.dq_turn = dq_turn;
  p.cta_ticket = cta_ticket;
  p.test_stall_cycles = test_stall_cycles;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(p.n_kblk) * B * Hkv);
  if (d == 64)
    err = causal ? launch_q64<64, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                 : launch_q64<64, false>(tq, tk, tv, tdo, tdq, p, grid, s);
  else
    err = causal ? launch_q64<128, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                 : launch_q64<128, false>(tq, tk, tv, tdo, tdq, p, grid, s);
  if (err != cudaSuccess) return err;

  const int64_t n4 = dq_elems / 4;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  bwd_dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<__nv_bfloat162*>(dq), n4);
  return cudaGetLastError();
}

}  // namespace fa4
