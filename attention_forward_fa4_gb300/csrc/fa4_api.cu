// fa4_api.cu -- the C ABI declared in include/fa4.h: argument validation,
// TMA tensor-map construction, kernel dispatch, the device status word and
// the diagnostic 2^x evaluator.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa4.h"
#include "fa4_internal.h"

static_assert(fa4::kTraceEvents == FA4_TRACE_EVENTS && fa4::kTraceSteps == FA4_TRACE_STEPS,
              "trace layout differs between the kernel and the C header");

namespace fa4 {
namespace {

// Kernel-side status: [0] code, [1] role, [2] barrier id, [3] block.
__device__ unsigned int g_status[4];

// Library-owned scratch of fa4_fwd_splitkv_static: one fixed device array
// per device, never allocated or freed at run time.
constexpr uint64_t kStaticScratchBytes = 32ull << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Device address of g_splitkv_scratch for the current device (looked up
// once each, on the first fa4_fwd_splitkv_static call there).
void* static_scratch_ptr(int dev) {
  static std::atomic<void*> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_splitkv_scratch) != cudaSuccess) return nullptr;
  cache[dev].store(addr, std::memory_order_release);
  return addr;
}

// Device address of g_status for the current device (looked up once each).
unsigned int* status_ptr(int dev) {
  static std::atomic<unsigned int*> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return nullptr;
  cache[dev].store(static_cast<unsigned int*>(addr), std::memory_order_release);
  return static_cast<unsigned int*>(addr);
}

// Automatic grid choice: the persistent grid pays off when work tiles are
// short (few key blocks each), where per-CTA start-up is a large share of a
// tile; long tiles keep one CTA per tile and the hardware's dynamic dispatch.
// Measured on GB300 over head dims 64 / 128, 512 to 32768 keys: persistent
// wins up to 8 key blocks at either head dim, and at head dim 64 (where its
// kernel keeps P in its own tensor-memory columns) up to 32 blocks;
// elsewhere one CTA per tile is as fast or faster.
bool use_persistent_grid(int64_t n_tiles, int sms, int nblk, int d, bool causal) {
  (void)causal;
  if (n_tiles <= sms) return false;
  if (nblk <= 8) return true;
  return d == 64 && nblk <= 32;
}

// Number of SMs of `dev` (looked up once each).
int sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev].store(n, std::memory_order_release);
  return n;
}

// [B, S, H, d] BF16 as a 4-D tensor (d, H, S, B); box = 64 columns x `rows`
// rows of one head, 128-byte swizzle (one swizzle row = 64 BF16).
bool make_map_rows(CUtensorMap* map, const void* ptr, int B, int S, int H, int d, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(S) * H * d * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_map(CUtensorMap* map, const void* ptr, int B, int S, int H, int d) {
  return make_map_rows(map, ptr, B, S, H, d, kBM);
}

// e4m3 [B, S, H, d] tensor as a 4-D map: a 128-column x 128-row box (128
// one-byte elements = one 128-byte swizzle row).
bool make_map_u8(CUtensorMap* map, const void* ptr, int B, int S, int H, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d,
                                 static_cast<cuuint64_t>(S) * H * d};
  const cuuint32_t box[4] = {128, 1, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [B, S, H, d] tensor (the backward's dQ accumulator) as a 4-D map with
// a 32-column x `rows`-row box and 128-byte swizzle (32 fp32 = 128 bytes).
bool make_map_f32(CUtensorMap* map, const void* ptr, int B, int S, int H, int d, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(H) * d * 4,
                                 static_cast<cuuint64_t>(S) * H * d * 4};
  const cuuint32_t box[4] = {32, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

fa4_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA4_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA4_ERR_CUDA;
  if (major != 10 || minor != 3) return FA4_ERR_UNSUPPORTED;
  return FA4_OK;
}

__global__ void no_keys_kernel(uint4* o, int64_t n_vec, float* lse, int64_t n_lse) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_vec; i += stride)
    o[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_lse; i += stride)
    lse[i] = -INFINITY;
}

// Evaluates the softmax's own paired emulation (ex2_emulated2) two inputs
// at a time, and MUFU.EX2 on each input.
__global__ void exp2_eval_kernel(const float* x, float* y_emu, float* y_mufu, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t pairs = (n + 1) / 2;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < pairs; i += stride) {
    const int64_t a = 2 * i, b = (2 * i + 1 < n) ? 2 * i + 1 : 2 * i;
    const float2 y = ex2_emulated2(make_float2(x[a], x[b]));
    y_emu[a] = y.x;
    y_mufu[a] = ex2_mufu(x[a]);
    if (b != a) {
      y_emu[b] = y.y;
      y_mufu[b] = ex2_mufu(x[b]);
    }
  }
}

}  // namespace
}  // namespace fa4

extern "C" {

void fa4_fwd_default_options(fa4_fwd_options* opt) {
  if (!opt) return;
  opt->tau = 8.0f;
  opt->exp2_emulation = 0;
  opt->rescale_stats = nullptr;
  opt->trace = nullptr;
  opt->trace_ctas = 0;
  opt->strict_mma_order = 0;
  opt->grid_mode = 0;
  opt->correction_warpgroup = 0;
  opt->test_stall_cycles = 0;
}

const char* fa4_status_string(fa4_status s) {
  switch (s) {
    case FA4_OK: return "FA4_OK";
    case FA4_ERR_INVALID_ARG: return "FA4_ERR_INVALID_ARG";
    case FA4_ERR_UNSUPPORTED: return "FA4_ERR_UNSUPPORTED";
    case FA4_ERR_MISALIGNED: return "FA4_ERR_MISALIGNED";
    case FA4_ERR_CUDA: return "FA4_ERR_CUDA";
    case FA4_ERR_TIMEOUT: return "FA4_ERR_TIMEOUT";
  }
  return "FA4_ERR_UNKNOWN";
}

int fa4_version(void) { return 100; }

namespace {

// Shared body of fa4_fwd_ex and fa4_fwd_splitkv. With num_splits > 0 the
// forward runs per key-range split into the workspace and a merge kernel
// writes o / lse; num_splits == 0 is the plain forward.
// Dequantisation scales of the FP8 forward (q, k, v hold e4m3 values whose
// true values are value * scale).
struct Fp8Scales {
  float q, k, v;
};

fa4_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                    int Hkv, int Sq, int Sk, int d, float scale, int causal,
                    const fa4_fwd_options* opt, int num_splits, void* workspace,
                    size_t workspace_bytes, fa4_stream_t stream, const Fp8Scales* fp8 = nullptr,
                    bool dry_run = false) {
  using namespace fa4;
  fa4_fwd_options o_def;
  fa4_fwd_default_options(&o_def);
  const fa4_fwd_options& op = opt ? *opt : o_def;

  // ---- arguments (nothing touches the GPU until they all pass)
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 1 || Hkv < 1) return FA4_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA4_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA4_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FA4_ERR_INVALID_ARG;
  if (!std::isfinite(op.tau) || op.tau < 0.0f || op.tau > 64.0f) return FA4_ERR_INVALID_ARG;
  if (op.exp2_emulation != 0 && op.exp2_emulation != 1 && op.exp2_emulation != 4 &&
      op.exp2_emulation != 8)
    return FA4_ERR_INVALID_ARG;
  if (op.strict_mma_order != 0 && op.strict_mma_order != 1) return FA4_ERR_INVALID_ARG;
  if (op.grid_mode < 0 || op.grid_mode > 2) return FA4_ERR_INVALID_ARG;
  if (op.test_stall_cycles < 0) return FA4_ERR_INVALID_ARG;
  if (op.correction_warpgroup != 0 && op.correction_warpgroup != 1) return FA4_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA4_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA4_ERR_INVALID_ARG;
  if (fp8) {
    auto bad = [](float x) { return !(x > 0.0f) || !std::isfinite(x); };
    if (bad(fp8->q) || bad(fp8->k) || bad(fp8->v)) return FA4_ERR_INVALID_ARG;
    // built for head dim 128, all exponentials on MUFU, no trace, no split
    if (d != 128 || op.exp2_emulation != 0 || op.trace || num_splits != 0) return FA4_ERR_UNSUPPORTED;
  }
  if (B == 0 || Sq == 0) return FA4_OK;  // empty output: nothing to do
  if (!q || !o || !lse || (Sk > 0 && (!k || !v))) return FA4_ERR_INVALID_ARG;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis16(q) || mis16(o) || (Sk > 0 && (mis16(k) || mis16(v))) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return FA4_ERR_MISALIGNED;
  if (op.rescale_stats && (reinterpret_cast<uintptr_t>(op.rescale_stats) & 7u) != 0)
    return FA4_ERR_MISALIGNED;
  if (op.trace && (reinterpret_cast<uintptr_t>(op.trace) & 7u) != 0) return FA4_ERR_MISALIGNED;
  if (op.trace && op.trace_ctas < 0) return FA4_ERR_INVALID_ARG;
  const uint64_t in_elem = fp8 ? 1 : 2;
  const uint64_t q_bytes = static_cast<uint64_t>(B) * Sq * Hq * d * in_elem;
  const uint64_t kv_bytes = static_cast<uint64_t>(B) * Sk * Hkv * d * in_elem;
  const uint64_t o_bytes = static_cast<uint64_t>(B) * Sq * Hq * d * 2;
  const uint64_t lse_bytes = static_cast<uint64_t>(B) * Hq * Sq * 4;
  if (overlaps(o, o_bytes, q, q_bytes) || overlaps(o, o_bytes, k, kv_bytes) ||
      overlaps(o, o_bytes, v, kv_bytes) || overlaps(o, o_bytes, lse, lse_bytes) ||
      overlaps(lse, lse_bytes, q, q_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
      overlaps(lse, lse_bytes, v, kv_bytes))
    return FA4_ERR_INVALID_ARG;
  // Key-range split: split_blocks key blocks per split; splits that would
  // start past the last key block are dropped.
  const int nblk_all = (Sk + kBN - 1) / kBN;
  int n_splits = 1, split_blocks = nblk_all > 0 ? nblk_all : 1;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (num_splits > 0 && Sk > 0) {
    const uint64_t need = fa4_fwd_splitkv_workspace_bytes(B, Hq, Sq, d, num_splits);
    if (!workspace || workspace_bytes < need) return FA4_ERR_INVALID_ARG;
    if (mis16(workspace)) return FA4_ERR_MISALIGNED;
    if (overlaps(workspace, need, q, q_bytes) || overlaps(workspace, need, k, kv_bytes) ||
        overlaps(workspace, need, v, kv_bytes) || overlaps(workspace, need, o, q_bytes) ||
        overlaps(workspace, need, lse, lse_bytes))
      return FA4_ERR_INVALID_ARG;
    split_blocks = (nblk_all + num_splits - 1) / num_splits;
    n_splits = (nblk_all + split_blocks - 1) / split_blocks;
    o_part = static_cast<float*>(workspace);
    lse_part = o_part + static_cast<uint64_t>(num_splits) * B * Sq * Hq * d;
  }
  const int64_t n_qblk = (static_cast<int64_t>(Sq) + 2 * kBM - 1) / (2 * kBM);
  const int64_t n_tiles = n_qblk * B * Hq * n_splits;
  if (n_tiles > 0x7fffffffLL) return FA4_ERR_UNSUPPORTED;
  // TMA limits: every global stride below 2^40 bytes.
  if (static_cast<uint64_t>(Sq) * Hq * d * 2 >= (1ull << 40) ||
      static_cast<uint64_t>(Sk) * Hkv * d * 2 >= (1ull << 40))
    return FA4_ERR_UNSUPPORTED;

  // ---- device
  fa4_status st = check_device();
  if (st != FA4_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA4_ERR_CUDA;
  unsigned int* status = status_ptr(dev);
  if (!status) return FA4_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms <= 0) return FA4_ERR_CUDA;
  if (dry_run) return FA4_OK;   // arguments checked, nothing enqueued
  // Grid: one CTA per work tile (the hardware hands the next tile to the
  // first free SM), or persistent (one CTA per SM -- the shared-memory
  // footprint allows no more -- walking its tiles in snake order).
  const int nblk = split_blocks;               // key blocks of the longest work tile
  bool persistent;
  if (op.grid_mode == 1) {
    persistent = false;
  } else if (op.grid_mode == 2) {
    persistent = true;
  } else {
    persistent = use_persistent_grid(n_tiles, sms, nblk, d, causal != 0);
  }
  const int64_t grid = persistent ? (n_tiles < sms ? n_tiles : sms) : n_tiles;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (Sk == 0) {  // no keys: O = 0, LSE = -inf
    no_keys_kernel<<<152, 256, 0, s>>>(static_cast<uint4*>(o), static_cast<int64_t>(o_bytes / 16),
                                       lse, static_cast<int64_t>(lse_bytes / 4));
    return cudaGetLastError() == cudaSuccess ? FA4_OK : FA4_ERR_CUDA;
  }

  CUtensorMap tq, tk, tv;
  auto map = fp8 ? make_map_u8 : make_map;
  if (!map(&tq, q, B, Sq, Hq, d) || !map(&tk, k, B, Sk, Hkv, d) || !map(&tv, v, B, Sk, Hkv, d))
    return FA4_ERR_CUDA;

  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.n_qblk = static_cast<int>(n_qblk);
  p.n_tiles = static_cast<int>(n_tiles);
  // Causal tiles are numbered heaviest first: over all heads for the
  // persistent grid (its snake assignment balances them), within chunks of 8
  // (batch, head) pairs whose K/V stay in L2 when the hardware schedules one
  // CTA per tile. Non-causal tiles of one head are numbered side by side so
  // their K/V reads meet in L2.
  p.head_chunk = causal ? (persistent ? B * Hq : (B * Hq < 8 ? B * Hq : 8)) : 1;
  p.scale_log2 = (fp8 ? scale * fp8->q * fp8->k : scale) * 1.4426950408889634f;
  p.out_scale = fp8 ? fp8->v : 1.0f;
  p.tau = op.tau;
  p.stats = op.rescale_stats;
  p.status = status;
  p.trace = op.trace;
  p.trace_ctas = op.trace ? op.trace_ctas : 0;
  p.strict_order = op.strict_mma_order ? 1 : 0;
  p.n_splits = n_splits;
  p.split_blocks = split_blocks;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.test_stall_cycles = op.test_stall_cycles;
  p.correction_wg = op.correction_warpgroup;

  const int emu = op.exp2_emulation == 1 ? 8 : op.exp2_emulation;   // pair period, 0 = off
  const bool traced = op.trace != nullptr;
  auto launch = (d == 64) ? (traced ? launch_fwd_d64_traced : launch_fwd_d64)
                          : (traced ? launch_fwd_d128_traced : launch_fwd_d128);
  cudaError_t err = fp8 ? launch_fwd_d128_fp8(tq, tk, tv, p, causal != 0, persistent,
                                              static_cast<unsigned>(grid), s)
                        : launch(tq, tk, tv, p, causal != 0, emu, persistent, static_cast<unsigned>(grid), s);
  if (err != cudaSuccess) return FA4_ERR_CUDA;
  if (o_part) {
    err = launch_merge_splits(o_part, lse_part, static_cast<__nv_bfloat16*>(o), lse, n_splits, B,
                              Sq, Hq, d, s);
    if (err != cudaSuccess) return FA4_ERR_CUDA;
  }
  return FA4_OK;
}

}  // namespace

fa4_status fa4_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                      const fa4_fwd_options* opt, fa4_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, 0, nullptr, 0, stream);
}

fa4_status fa4_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                       float q_scale, float k_scale, float v_scale, const fa4_fwd_options* opt,
                       fa4_stream_t stream) {
  const Fp8Scales sc{q_scale, k_scale, v_scale};
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, 0, nullptr, 0, stream,
                  &sc);
}

uint64_t fa4_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Sq < 0 || Sk < 0 || (d != 64 && d != 128)) return 0;
  auto up = [](uint64_t x) { return (x + 255u) & ~static_cast<uint64_t>(255u); };
  const uint64_t q = static_cast<uint64_t>(B) * Sq * Hq * d * 2;
  const uint64_t kv = static_cast<uint64_t>(B) * Sk * Hkv * d * 2;
  const uint64_t lse = static_cast<uint64_t>(B) * Hq * Sq * 4;
  return 2 * up(q) + 2 * up(kv) + up(lse);
}

fa4_status fa4_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                        void* workspace, uint64_t workspace_bytes, const fa4_fwd_options* opt,
                        fa4_stream_t stream) {
  using namespace fa4;
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 1 || Hkv < 1) return FA4_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA4_ERR_UNSUPPORTED;
  const uint64_t need = fa4_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d);
  if (B == 0 || Sq == 0) return FA4_OK;   // empty output: nothing to copy or compute
  if (!workspace || workspace_bytes < need) return FA4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA4_ERR_MISALIGNED;
  if (!q || !o || !lse || (Sk > 0 && (!k || !v))) return FA4_ERR_INVALID_ARG;
  auto up = [](uint64_t x) { return (x + 255u) & ~static_cast<uint64_t>(255u); };
  const uint64_t q_bytes = static_cast<uint64_t>(B) * Sq * Hq * d * 2;
  const uint64_t kv_bytes = static_cast<uint64_t>(B) * Sk * Hkv * d * 2;
  const uint64_t lse_bytes = static_cast<uint64_t>(B) * Hq * Sq * 4;
  // workspace: q | k | v | o | lse, each on a 256-byte boundary
  unsigned char* base = static_cast<unsigned char*>(workspace);
  unsigned char* dq = base;
  unsigned char* dk = dq + up(q_bytes);
  unsigned char* dv = dk + up(kv_bytes);
  unsigned char* dout = dv + up(kv_bytes);
  float* dlse = reinterpret_cast<float*>(dout + up(q_bytes));
  fa4_status st = fwd_impl(dq, dk, dv, dout, dlse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, 0,
                           nullptr, 0, stream, nullptr, /*dry_run=*/true);
  if (st != FA4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one copy per tensor, in, the forward, and out, all in stream order
  if (cudaMemcpyAsync(dq, q, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return FA4_ERR_CUDA;
  if (kv_bytes > 0 && (cudaMemcpyAsync(dk, k, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                       cudaMemcpyAsync(dv, v, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess))
    return FA4_ERR_CUDA;
  st = fwd_impl(dq, dk, dv, dout, dlse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, 0, nullptr, 0,
                stream);
  if (st != FA4_OK) return st;
  if (cudaMemcpyAsync(o, dout, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(lse, dlse, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FA4_ERR_CUDA;
  return FA4_OK;
}

uint64_t fa4_fwd_splitkv_workspace_bytes(int B, int Hq, int Sq, int d, int num_splits) {
  if (B < 0 || Hq < 0 || Sq < 0 || d < 0 || num_splits < 0) return 0;
  const uint64_t rows = static_cast<uint64_t>(num_splits) * B * Sq * Hq;
  return rows * static_cast<uint64_t>(d) * 4 + rows * 4;
}

uint64_t fa4_bwd_workspace_bytes(int B, int Hq, int Sq, int d) {
  if (B < 0 || Hq < 0 || Sq < 0 || d < 0) return 0;
  const uint64_t sq_pad = (static_cast<uint64_t>(Sq) + 127) / 128 * 128;
  // one int per (batch, query head, 64-query block)
  const uint64_t turns = (static_cast<uint64_t>(B) * Hq * (sq_pad / 64) * 4 + 15) / 16 * 16;
  // + 16 bytes: the deterministic mode's CTA ticket counter
  return static_cast<uint64_t>(B) * Sq * Hq * d * 4 + 2ull * B * Hq * sq_pad * 4 + turns + 16;
}

fa4_status fa4_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
                   int Sk, int d, float scale, int causal, void* workspace,
                   uint64_t workspace_bytes, fa4_stream_t stream) {
  return fa4_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, scale, causal, 0,
                    workspace, workspace_bytes, stream);
}

fa4_status fa4_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                      int Sq, int Sk, int d, float scale, int causal, int deterministic,
                      void* workspace, uint64_t workspace_bytes, fa4_stream_t stream) {
  fa4_bwd_options op;
  fa4_bwd_default_options(&op);
  op.deterministic = deterministic;
  return fa4_bwd_opt(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, scale, causal, &op,
                     workspace, workspace_bytes, stream);
}

void fa4_bwd_default_options(fa4_bwd_options* opt) {
  if (!opt) return;
  opt->deterministic = 0;
  opt->test_stall_cycles = 0;
}

fa4_status fa4_bwd_opt(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                       int Sq, int Sk, int d, float scale, int causal, const fa4_bwd_options* opt,
                       void* workspace, uint64_t workspace_bytes, fa4_stream_t stream) {
  using namespace fa4;
  fa4_bwd_options op;
  fa4_bwd_default_options(&op);
  if (opt) op = *opt;
  const int deterministic = op.deterministic;
  if (deterministic != 0 && deterministic != 1) return FA4_ERR_INVALID_ARG;
  if (op.test_stall_cycles < 0) return FA4_ERR_INVALID_ARG;
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 1 || Hkv < 1) return FA4_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA4_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA4_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FA4_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA4_ERR_UNSUPPORTED;
  if (B == 0 || (Sq == 0 && Sk == 0)) return FA4_OK;
  const uint64_t q_bytes = static_cast<uint64_t>(B) * Sq * Hq * d * 2;
  const uint64_t kv_bytes = static_cast<uint64_t>(B) * Sk * Hkv * d * 2;
  const uint64_t lse_bytes = static_cast<uint64_t>(B) * Hq * Sq * 4;
  const bool has_q = Sq > 0, has_k = Sk > 0;
  if ((has_q && (!q || !o || !dout || !lse || !dq)) || (has_k && (!k || !v || !dk || !dv)))
    return FA4_ERR_INVALID_ARG;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if ((has_q && (mis16(q) || mis16(o) || mis16(dout) || mis16(dq) ||
                 (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)) ||
      (has_k && (mis16(k) || mis16(v) || mis16(dk) || mis16(dv))))
    return FA4_ERR_MISALIGNED;
  const uint64_t need = fa4_bwd_workspace_bytes(B, Hq, Sq, d);
  if (has_q && has_k) {
    if (!workspace || workspace_bytes < need) return FA4_ERR_INVALID_ARG;
    if (mis16(workspace)) return FA4_ERR_MISALIGNED;
  }
  // Outputs overlap nothing: not the inputs, not each other, not the workspace.
  const void* ins[] = {q, k, v, o, dout, lse};
  const uint64_t in_n[] = {q_bytes, kv_bytes, kv_bytes, q_bytes, q_bytes, lse_bytes};
  const void* outs[] = {dq, dk, dv, (has_q && has_k) ? workspace : nullptr};
  const uint64_t out_n[] = {q_bytes, kv_bytes, kv_bytes, need};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_n[a], ins[b], in_n[b])) return FA4_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return FA4_ERR_INVALID_ARG;
  }
  const int64_t n_kblk = (static_cast<int64_t>(Sk) + 127) / 128;
  if (n_kblk * B * Hkv > 0x7fffffffLL) return FA4_ERR_UNSUPPORTED;
  if (static_cast<uint64_t>(Sq) * Hq * d * 2 >= (1ull << 40) ||
      static_cast<uint64_t>(Sk) * Hkv * d * 2 >= (1ull << 40))
    return FA4_ERR_UNSUPPORTED;

  fa4_status st = check_device();
  if (st != FA4_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA4_ERR_CUDA;
  unsigned int* status = status_ptr(dev);
  if (!status) return FA4_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!has_q || !has_k) {
    // no queries: dK = dV = 0; no keys: the output is constant 0, dQ = 0
    if (has_k && (cudaMemsetAsync(dk, 0, kv_bytes, s) != cudaSuccess ||
                  cudaMemsetAsync(dv, 0, kv_bytes, s) != cudaSuccess))
      return FA4_ERR_CUDA;
    if (has_q && cudaMemsetAsync(dq, 0, q_bytes, s) != cudaSuccess) return FA4_ERR_CUDA;
    return FA4_OK;
  }
  float* dq_acc = static_cast<float*>(workspace);
  // Q and dO move in blocks of 64 query rows, dQ reduce-adds in blocks of 32
  // rows at head dim 128 and 64 at 64; K and V in blocks of 128 key rows.
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_map_rows(&tq, q, B, Sq, Hq, d, 64) || !make_map(&tk, k, B, Sk, Hkv, d) ||
      !make_map(&tv, v, B, Sk, Hkv, d) || !make_map_rows(&tdo, dout, B, Sq, Hq, d, 64) ||
      !make_map_f32(&tdq, dq_acc, B, Sq, Hq, d, d == 128 ? 32 : 64))
    return FA4_ERR_CUDA;
  float* lse2 = dq_acc + static_cast<uint64_t>(B) * Sq * Hq * d;
  float* delta = lse2 + static_cast<uint64_t>(B) * Hq * ((Sq + 127) / 128 * 128);
  int* turns = reinterpret_cast<int*>(delta + static_cast<uint64_t>(B) * Hq * ((Sq + 127) / 128 * 128));
  const uint64_t turn_ints = (static_cast<uint64_t>(B) * Hq * ((Sq + 127) / 128 * 2) * 4 + 15) / 16 * 4;
  int* ticket = turns + turn_ints;
  cudaError_t err = launch_bwd(tq, tk, tv, tdo, tdq, static_cast<const __nv_bfloat16*>(o),
                               static_cast<const __nv_bfloat16*>(dout), lse,
                               static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
                               static_cast<__nv_bfloat16*>(dv), dq_acc, lse2, delta,
                               deterministic ? turns : nullptr, deterministic ? ticket : nullptr,
                               B, Hq, Hkv, Sq, Sk, d, scale, causal != 0, op.test_stall_cycles, status, s);
  return err == cudaSuccess ? FA4_OK : FA4_ERR_CUDA;
}

uint64_t fa4_fwd_splitkv_static_max_bytes(void) { return fa4::kStaticScratchBytes; }

fa4_status fa4_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                                  int causal, int num_splits, const fa4_fwd_options* opt,
                                  fa4_stream_t stream) {
  using namespace fa4;
  if (num_splits < 1 || num_splits > kMaxSplits) return FA4_ERR_INVALID_ARG;
  // Every argument check of the plain forward first (head dim, sizes,
  // pointers, alignment, device), so the codes match fa4_fwd_splitkv's; the
  // size cap then rejects only valid problems too large for the scratch.
  fa4_status st = fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, 0, nullptr,
                           0, stream, nullptr, /*dry_run=*/true);
  if (st != FA4_OK) return st;
  if (B == 0 || Sq == 0) return FA4_OK;   // empty output: nothing to do
  if (fa4_fwd_splitkv_workspace_bytes(B, Hq, Sq, d, num_splits) > kStaticScratchBytes)
    return FA4_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA4_ERR_CUDA;
  void* scratch = static_scratch_ptr(dev);
  if (!scratch) return FA4_ERR_CUDA;
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, num_splits, scratch,
                  static_cast<size_t>(kStaticScratchBytes), stream);
}

fa4_status fa4_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                           int num_splits, void* workspace, uint64_t workspace_bytes,
                           const fa4_fwd_options* opt, fa4_stream_t stream) {
  if (num_splits < 1) return FA4_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, opt, num_splits, workspace,
                  static_cast<size_t>(workspace_bytes), stream);
}

fa4_status fa4_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int d, float scale, int causal, fa4_stream_t stream) {
  return fa4_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale, causal, nullptr, stream);
}

fa4_status fa4_device_status(int clear, unsigned int* detail) {
  using namespace fa4;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA4_ERR_CUDA;
  unsigned int h[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(h, g_status, sizeof h) != cudaSuccess) return FA4_ERR_CUDA;
  if (detail) std::memcpy(detail, h, sizeof h);
  if (clear) {
    const unsigned int z[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_status, z, sizeof z) != cudaSuccess) return FA4_ERR_CUDA;
  }
  return h[0] == 0 ? FA4_OK : static_cast<fa4_status>(h[0]);
}

fa4_status fa4_exp2_eval(const float* x, float* y_emu, float* y_mufu, int64_t n,
                         fa4_stream_t stream) {
  using namespace fa4;
  if (n < 0) return FA4_ERR_INVALID_ARG;
  if (n == 0) return FA4_OK;
  if (!x || !y_emu || !y_mufu) return FA4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y_emu) |
       reinterpret_cast<uintptr_t>(y_mufu)) & 3u)
    return FA4_ERR_MISALIGNED;
  fa4_status st = check_device();
  if (st != FA4_OK) return st;
  const int64_t blocks64 = (n + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(blocks64 < 152 * 8 ? blocks64 : 152 * 8);
  exp2_eval_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, y_emu, y_mufu, n);
  return cudaGetLastError() == cudaSuccess ? FA4_OK : FA4_ERR_CUDA;
}

}  // extern "C"
