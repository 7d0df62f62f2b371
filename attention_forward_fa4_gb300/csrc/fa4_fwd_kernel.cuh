// fa4_fwd_kernel.cuh -- warp-specialised attention forward for sm_103a.
//
// A work tile is two 128-row query tiles of one (batch, head) -- M = 256
// rows -- walking every key block of 128 keys once; a persistent grid of
// one CTA per SM visits the work tiles in turn ("FlashAttention-4:
// Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware
// Scaling", Table 1 / §3.1.1 tile M = 256, N = 128; §3.1.2 two output
// tiles per CTA). Roles, one per warp group (§3.1.2, Method (1); "How
// FlashAttention 4 Works", the Load / MMA / Softmax / Correction /
// Epilogue split):
//
//   warps 0-3   softmax WG for tile 0: one thread owns one row (TMEM lane)
//   warps 4-7   softmax WG for tile 1; both also run the epilogue
//   warps 8-11  correction WG: rescales O in TMEM when a row group's
//               reference max moves (conditional rescale, §3.1.4); groups
//               that need no rescale never wait for it

//   warp 12     TMA load warp: Q once, then K_j / V_j into a ring of slots
//               (whole warp, one elected lane issues each copy)
//   warp 13     MMA warp: the whole warp runs the issue loop with uniform
//               operands; one elected lane issues every tcgen05.mma
//   warps 14-15 idle
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   S_t  = Q_t K_j^T   fp32, columns [128 t, 128 t + 128)
//   P_t  (BF16, two per column) aliases the first 64 columns of S_t; in
//        the persistent grid at head dim 64 it has its own columns
//        [384 + 64 t, 448 + 64 t) instead (see OwnP)
//   O_t  fp32, columns [256 + D t, 256 + D t + D)
//
// The MMA thread issues the two tiles' work in ping-pong order (see
// mma_role): each softmax WG works on its tile while the tensor core runs
// the other tile's P*V and next S.
//
// Every mbarrier wait is bounded (about half a second of SM cycles). On
// expiry the waiting thread raises a CTA-wide abort flag and a device
// status word; every role then leaves its loop, in-flight TMA copies and
// MMAs are drained, and TMEM is freed before the CTA exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "fa4_exp2.cuh"
#include "fa4_ptx.cuh"

// Tunables (compile-time):
//   FA4_P_SLICES     1: P is stored and released to P*V as one 128-key block;
//                    2: in two 64-key halves so P*V starts on the first half
//                    while the second is being exponentiated.
//   FA4_WAIT_SPIN    0: waits poll mbarrier.try_wait (the thread may be
//                    suspended for a system-dependent time); 1: poll
//                    mbarrier.test_wait (never suspended); 2: try_wait with a
//                    100 us suspend-time hint; 3, 4, 5: test_wait with a 32,
//                    256 or 1024 ns nanosleep back-off.
#ifndef FA4_P_SLICES
#define FA4_P_SLICES 1
#endif
#ifndef FA4_WAIT_SPIN
#define FA4_WAIT_SPIN 0
#endif


namespace fa4 {

#ifdef FA4_PROF
// Light phase profile (diagnostic builds only): cycle sums added once per
// role at exit. [0..5] softmax of the tile-0 warp 0: load, decide, exp,
// store, wait for S, steps; [8..13] MMA warp: wait for the softmax,
// P*V issue, between P*V and S, S issue, steps.
__device__ unsigned long long g_prof[32];
#define FA4_PROF_CLK(x) const unsigned x = static_cast<unsigned>(clock())
#else
#define FA4_PROF_CLK(x)
#endif

constexpr int kBM = 128;          // query rows per tile = TMEM lanes
constexpr int kBN = 128;          // keys per block
constexpr int kThreads = 512;     // 16 warps
constexpr int kWarpLoad = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
// A wait gives up after this many SM cycles (about 0.5 s at 2 GHz).
constexpr long long kWaitLimitCycles = 1ll << 30;

enum : unsigned { kStatusTimeout = 5u };
enum : unsigned { kRoleLoad = 0, kRoleMma = 1, kRoleSoftmax = 2, kRoleCorrection = 3, kRoleFlush = 4, kRoleDqRead = 5 };

struct FwdParams {
  __nv_bfloat16* o;            // [B, Sq, Hq, D]
  float* lse;                  // [B, Hq, Sq]
  int B, Hq, Hkv, Sq, Sk;
  int group;                   // Hq / Hkv
  int n_qblk;                  // ceil(Sq / 256)
  int head_chunk;              // (b, h) pairs interleaved by the tile order
  float scale_log2;            // scale * log2(e)
  float tau;                   // rescale threshold, log2 units
  unsigned long long* stats;   // optional rescale counters [2]
  unsigned int* status;        // device status word [4]
  unsigned long long* trace;   // optional per-role cycle trace (see trace_mark)
  int trace_ctas;              // CTAs (by blockIdx.x) that record a trace
  int strict_order;            // 1: S_t(j+1) waits for P_t(j) V_j to complete
  int n_tiles;                 // n_qblk * B * Hq * n_splits work tiles
  // Key-range split: work tile id = (query tile pair) * n_splits + split;
  // split s covers key blocks [s * split_blocks, (s + 1) * split_blocks).
  // With o_part set, each split writes its normalised partial output
  // o_part[s][B][Sq][Hq][D] and lse_part[s][B][Hq][Sq] (fp32) instead of
  // o / lse; a merge kernel combines them.
  int n_splits;
  int split_blocks;
  float* o_part;
  float* lse_part;
  float out_scale;             // multiplies O in the epilogue (V's dequantisation scale; 1 for BF16)
  // 1: a correction warpgroup rescales O_t when a row group's reference max
  // moves; 0: the softmax warp of that row group does it itself.
  int correction_wg;
  // Diagnostic: when > 0 the softmax warps first wait on a barrier that
  // nothing completes and give up after this many SM cycles, so the kernel
  // takes its timeout path (abort, drain, free tensor memory, exit).
  long long test_stall_cycles;
};

// ------------------------------------------------------------ cycle trace
// Optional diagnostic: when FwdParams::trace is set, CTAs with
// blockIdx.x < trace_ctas record the SM cycle counter at fixed points of
// each role, for key block j < kTraceSteps and query tile t of the CTA's
// first work tile:
//   trace[((cta * kTraceEvents + event) * kTraceSteps + j) * 2 + t].
// The MMA thread, lane 0 of the first softmax warp of each tile and lane 0
// of the first correction warp record. Only the kernels instantiated with
// TRACE = true contain the marks (the host picks them when a trace buffer
// is passed); in the others they compile to nothing, because even untaken
// checks at every mark cost about 8 % of forward throughput.
constexpr int kTraceSteps = 128;
enum TraceEvent : int {
  kTrMmaSWait = 0,     // MMA: starts waiting for the S_t slot / K_j
  kTrMmaSIssued,       // MMA: S_t = Q_t K_j^T issued and committed
  kTrMmaPvWait,        // MMA: starts waiting for o_ready[t]
  kTrMmaPvIssued,      // MMA: O_t += P_t V_j issued and committed
  kTrSmSReady,         // softmax: S_t visible (s_full passed)
  kTrSmLoaded,         // softmax: S row in registers
  kTrSmExpDone,        // softmax: P computed and packed (before the TMEM stores)
  kTrSmArrived,        // softmax: P stored, barrier arrived
  kTrCoWake,           // correction: p_full passed
  kTrCoArrived,        // correction: o_ready arrived
  kTrMmaSGo,           // MMA: S_t dependencies met (before issuing)
  kTrMmaPvGo,          // MMA: P_t / O_t dependencies met (before issuing)
  kTrSmArrivedQ1,      // softmax warps 2-4 of the tile: P stored
  kTrSmArrivedQ2,
  kTrSmArrivedQ3,
  kTrSmMaxDone,        // softmax: block max known, rescale decided
  kTrMmaCommitted,     // MMA: slot-release commits of key block j issued
  kTrMmaVReady,        // MMA: V_j in shared memory (before any P_t V_j)
  kTrLoadIssued,       // load warp: V_j copy issued (t = 0) / K_j copy issued (t = 1)
  kTrSmMaxLoop,        // softmax: block max reduced (before the warp vote)
  kTrSmCDone,          // softmax: the correction warps have taken the last step's flags
  kTraceEvents
};

template <bool TRACE>
__device__ __forceinline__ void trace_mark(const FwdParams& p, int ev, int j, int t, int iter = 0) {
  if constexpr (!TRACE) return;
  if (p.trace != nullptr && iter == 0 && static_cast<int>(blockIdx.x) < p.trace_ctas && j < kTraceSteps) {
    uint64_t c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    p.trace[((static_cast<size_t>(blockIdx.x) * kTraceEvents + ev) * kTraceSteps + j) * 2 + t] = c;
  }
}

// As trace_mark, recorded by lane 0 of a warp whose lanes all run the role.
template <bool TRACE>
__device__ __forceinline__ void trace_mark_lane0(const FwdParams& p, int ev, int j, int t, int iter = 0) {
  if ((threadIdx.x & 31) == 0) trace_mark<TRACE>(p, ev, j, t, iter);
}

// FP8: Q, K, V (and P) in e4m3 -- one byte per element, so a d = 128 row is
// a single 128-byte swizzle panel.
template <int D, bool FP8 = false>
struct Smem {
  static_assert(!FP8 || D == 128, "the FP8 forward is built for head dim 128");
  static constexpr int kTileBytes = kBM * D * (FP8 ? 1 : 2);  // one 128 x D tile
  static constexpr int kPanelBytes = kBM * 128;          // 128 rows x 128 B
  static constexpr int kPanels = FP8 ? 1 : D / 64;
  static constexpr int kSlots = (D == 128 && !FP8) ? 4 : 8;   // K/V ring depth
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + 2 * kTileBytes;
  static constexpr int kBars = kRing + kSlots * kTileBytes;
  // barrier ids
  static constexpr int bQ = 0;
  static constexpr int bKvFull = 1;
  static constexpr int bKvEmpty = bKvFull + kSlots;
  static constexpr int bSFull = bKvEmpty + kSlots;       // [2]
  static constexpr int bPFull = bSFull + 2;              // [2]
  static constexpr int bOReady = bPFull + 2;             // [2]
  static constexpr int bPvDone = bOReady + 2;            // [2]
  static constexpr int bCDone = bPvDone + 2;             // [2 tiles][2 buffers]
  static constexpr int bPHalf = bCDone + 4;              // [2 tiles][2 halves]
  static constexpr int bQEmpty = bPHalf + 4;             // Q tiles free for the next work tile
  static constexpr int bOFree = bQEmpty + 1;             // [2] epilogue has read O_t
  static constexpr int bDrain = bOFree + 2;
  static constexpr int bStall = bDrain + 1;              // never completed (timeout test)
  static constexpr int bSFree = bStall + 1;              // [2] softmax has read S_t (own-P layout)
  static constexpr int kNumBars = bSFree + 2;
  // Rescale hand-off from softmax to correction, double-buffered by step
  // parity: alpha float [2 buffers][2 tiles][128], flags int [2][2][4].
  static constexpr int kAlpha = kBars + kNumBars * 8;
  static constexpr int kFlags = kAlpha + 4 * kBM * 4;
  static constexpr int kMisc = kFlags + 16 * 4;          // tmem base, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;           // slack for 1 KB alignment
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
  // At head dim 64 the two O tiles leave 128 columns free, so P_t can have
  // its own 64 columns instead of aliasing S_t ("own P", see OwnP below).
  static constexpr bool kPColsFree = (D == 64 && !FP8);
  static constexpr uint32_t kColP0 = 256 + 2 * D, kColP1 = 256 + 2 * D + 64;
  static_assert(!kPColsFree || kColP1 + 64 <= 512, "P columns beyond tensor memory");
};

// Own P: P_t in its own tensor-memory columns. The next S_t MMA then only
// waits until the softmax has read S_t into registers, not for the P*V that
// reads P_t, so S_t(j+1) is computed while softmax_t(j) runs; every P*V
// commits pv_done, which the softmax waits for before it overwrites P_t or
// rescales O_t. Used by the persistent grid at head dim 64 (short
// sequences), where it measured faster; with one CTA per work tile the
// MMA warp's extra waits and commits cost more than the overlap gains.
template <int D, bool PERSIST, bool FP8>
struct OwnP {
  static constexpr bool value = Smem<D, FP8>::kPColsFree && PERSIST;
  static constexpr uint32_t col(int t) {
    return value ? (t == 0 ? Smem<D, FP8>::kColP0 : Smem<D, FP8>::kColP1)
                 : (t == 0 ? Smem<D, FP8>::kColS0 : Smem<D, FP8>::kColS1);
  }
};

// ------------------------------------------------------------ bounded waits
struct Waiter {
  volatile int* abort;
  unsigned int* status;
  unsigned role;

  __device__ __forceinline__ bool slow(uint32_t bar, uint32_t parity, unsigned id,
                                       bool honour_abort, long long limit = kWaitLimitCycles) const {
    // Poll first; the (cheap, SM-local) cycle counter is only read every
    // 1024 failed polls.
    long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
      bool done;
      if (FA4_WAIT_SPIN == 1) {
        done = mbar_test_wait(bar, parity);
      } else if (FA4_WAIT_SPIN == 2) {
        done = mbar_try_wait_hint(bar, parity, 100000u);
      } else if (FA4_WAIT_SPIN >= 3) {
        done = mbar_test_wait(bar, parity);
        if (!done) __nanosleep(FA4_WAIT_SPIN == 3 ? 32 : (FA4_WAIT_SPIN == 4 ? 256 : 1024));
      } else {
        done = mbar_try_wait(bar, parity);
      }
      if (done) return true;
      if ((it & (FA4_WAIT_SPIN == 2 ? 15u : 1023u)) == 0u) {
        if (honour_abort && *abort) return false;
        const long long now = clock64();
        if (t0 == 0) t0 = now;
        if (now - t0 > limit) {
          *abort = 1;
          if (atomicCAS(status, 0u, kStatusTimeout) == 0u) {
            status[1] = role;
            status[2] = id;
            status[3] = blockIdx.x;
          }
          __threadfence();
          return false;
        }
      }
    }
  }
  // Returns false if the CTA is aborting (this wait or another one expired).
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, unsigned id) const {
    return mbar_try_wait(bar, parity) || slow(bar, parity, id, true);
  }
  // As wait(), giving up after `limit` SM cycles instead of the default.
  __device__ __forceinline__ bool wait_for(uint32_t bar, uint32_t parity, unsigned id,
                                           long long limit) const {
    return mbar_try_wait(bar, parity) || slow(bar, parity, id, true, limit);
  }
  // Used only while draining: waits for hardware-driven completions (TMA
  // bytes, MMA commits) even after an abort, still bounded.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, unsigned id) const {
    return mbar_try_wait(bar, parity) || slow(bar, parity, id, false);
  }
  // Warp-wide forms for a role that a whole warp runs: every lane waits and
  // the outcome is made uniform, so the warp stays converged for the
  // elect.sync issues that follow.
  __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, unsigned id) const {
    const bool ok = mbar_try_wait(bar, parity) || slow(bar, parity, id, true);
    return __all_sync(0xffffffffu, ok);
  }
  __device__ __forceinline__ bool drain_warp(uint32_t bar, uint32_t parity, unsigned id) const {
    const bool ok = mbar_try_wait(bar, parity) || slow(bar, parity, id, false);
    return __all_sync(0xffffffffu, ok);
  }
};

// ------------------------------------------------------------ tile geometry
// A work tile is two 128-row query tiles of one (batch, head). The grid is
// persistent: with G = gridDim.x, CTA c visits work tiles in snake order
// c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... Causal tiles are numbered heaviest
// first, so the pairs a CTA takes from consecutive rounds add up to about
// the same work on every CTA.
// Without PERSIST the grid has one CTA per work tile and each CTA takes
// exactly its own tile (the loops below then run once, with every running
// counter starting from zero).
template <bool PERSIST>
__device__ __forceinline__ int tile_of(int k, int n_tiles) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if constexpr (!PERSIST) return k == 0 ? c : n_tiles;
  return k * g + ((k & 1) ? (g - 1 - c) : c);
}

struct Tile {
  int b, h, hk, q0;
  int split;        // key-range split of this work tile
  int kv0;          // first key block of the split
  int nkv[2];       // key blocks each query tile visits (within the split)
  int nkv_max;
};

template <bool CAUSAL>
__device__ __forceinline__ Tile make_tile(const FwdParams& p, int id_split) {
  Tile tl;
  const int id = id_split / p.n_splits;
  tl.split = id_split - id * p.n_splits;
  tl.kv0 = tl.split * p.split_blocks;
  const int n_bh = p.B * p.Hq;
  const int per_chunk = p.head_chunk * p.n_qblk;
  const int chunk = id / per_chunk;
  const int rem = id - chunk * per_chunk;
  const int g_eff = min(p.head_chunk, n_bh - chunk * p.head_chunk);
  const int qrank = rem / g_eff;
  const int bh = chunk * p.head_chunk + (rem - qrank * g_eff);
  // Causal: the largest query blocks (most key blocks) go first.
  const int qb = CAUSAL ? (p.n_qblk - 1 - qrank) : qrank;
  tl.b = bh / p.Hq;
  tl.h = bh - tl.b * p.Hq;
  tl.hk = tl.h / p.group;
  tl.q0 = qb * 2 * kBM;
  const int nblk = (p.Sk + kBN - 1) / kBN;
  tl.nkv_max = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = tl.q0 + t * kBM;
    int n = 0;
    if (r0 < p.Sq) {
      if (CAUSAL) {
        const int last_row = min(r0 + kBM - 1, p.Sq - 1);
        const long long kmax = static_cast<long long>(last_row) + p.Sk - p.Sq;  // last allowed key
        n = kmax < 0 ? 0 : min(nblk, static_cast<int>(kmax / kBN) + 1);
      } else {
        n = nblk;
      }
    }
    n = max(0, min(n - tl.kv0, p.split_blocks));   // the split's share
    tl.nkv[t] = n;
    tl.nkv_max = max(tl.nkv_max, n);
  }
  return tl;
}

// ------------------------------------------------------------ load warp
// Q once per work tile (after the previous tile's S MMAs have released the
// Q buffers), then K_j, V_j of every key block into the slot ring; the
// ring's fill counter runs on across work tiles.
template <int D, bool CAUSAL, bool PERSIST, bool TRACE, bool FP8 = false>
__device__ __forceinline__ void load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_v, uint32_t sbase,
                                          const FwdParams& p, const Waiter& w) {
  using L = Smem<D, FP8>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  int fill = 0;     // K/V copies issued so far (ring position)
  int n_q = 0;      // Q copies issued so far
  bool ok = true;
  int iter = 0;
  for (int id = tile_of<PERSIST>(0, p.n_tiles); ok && id < p.n_tiles; id = tile_of<PERSIST>(++iter, p.n_tiles)) {
    const Tile tl = make_tile<CAUSAL>(p, id);
    if (tl.nkv_max == 0) continue;
    if (n_q > 0 && !(ok = w.wait_warp(bar(L::bQEmpty), static_cast<uint32_t>(n_q - 1) & 1u, L::bQEmpty)))
      break;
    mbar_arrive_expect_tx_warp(bar(L::bQ), 2u * L::kTileBytes);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int pn = 0; pn < L::kPanels; ++pn)
        tma_load_4d_warp(sbase + L::kQ + t * L::kTileBytes + pn * L::kPanelBytes, tm_q, bar(L::bQ),
                    pn * 64, tl.h, tl.q0 + t * kBM, tl.b);
    ++n_q;
    for (int idx = 0; idx < 2 * tl.nkv_max; ++idx) {   // K_0, V_0, K_1, V_1, ...
      const int s = fill % L::kSlots;
      const uint32_t n = static_cast<uint32_t>(fill / L::kSlots);
      if (!(ok = w.wait_warp(bar(L::bKvEmpty + s), (n & 1u) ^ 1u, L::bKvEmpty + s))) break;
      mbar_arrive_expect_tx_warp(bar(L::bKvFull + s), L::kTileBytes);
      const CUtensorMap* tm = (idx & 1) ? tm_v : tm_k;
      const int row = (tl.kv0 + (idx >> 1)) * kBN;
#pragma unroll
      for (int pn = 0; pn < L::kPanels; ++pn)
        tma_load_4d_warp(sbase + L::kRing + s * L::kTileBytes + pn * L::kPanelBytes, tm,
                    bar(L::bKvFull + s), pn * 64, tl.hk, row, tl.b);
      ++fill;
      trace_mark_lane0<TRACE>(p, kTrLoadIssued, idx >> 1, (idx & 1) ? 0 : 1, iter);
    }
  }
  if (__any_sync(0xffffffffu, !ok || *w.abort)) {
    // Let every copy this warp started land before the CTA frees its memory.
    if (n_q > 0) w.drain_warp(bar(L::bQ), static_cast<uint32_t>(n_q - 1) & 1u, L::bQ);
    for (int idx = max(0, fill - L::kSlots); idx < fill; ++idx) {
      const int s = idx % L::kSlots;
      w.drain_warp(bar(L::bKvFull + s), static_cast<uint32_t>(idx / L::kSlots) & 1u, L::bKvFull + s);
    }
  }
}

// ------------------------------------------------------------ MMA warp
// Issue order (two-tile ping-pong, "FlashAttention-4" §3.1.2):
//   S_0(0), S_1(0), then for each key block j:
//     O_0 += P_0(j) V_j, S_0(j+1) = Q_0 K_{j+1}^T, O_1 += P_1(j) V_j, S_1(j+1)
// so the tensor core computes tile 1's work while tile 0's softmax runs and
// the other way round. S_t(j+1) overwrites the TMEM columns that P_t(j)
// occupies and is issued right behind the P*V that reads them: the MMAs of
// one issuing thread run through the SM's tensor core in issue order (the
// warp stays converged, so elect.sync picks the same lane for every MMA and
// commit). With FwdParams::strict_order set, S_t(j+1) instead waits for the
// P*V's commit.
//
// Measured on GB300: with the softmax warps busy on every SMSP, a single
// issuing lane whose descriptors live in per-thread registers kept a
// 128 x 128 x 128 MMA group to about 1000 cycles (about 600 with the SM
// otherwise idle); the whole warp computing the same uniform operands and
// one elected lane issuing brought it to about 850.
//
// With own P (OwnP) the order per key block is S_0(j+1), S_1(j+1), then
// O_0 += P_0(j) V_j, O_1 += P_1(j) V_j: the S MMAs only wait until the
// softmax has read S_t(j), and strict order changes nothing.
//
// Phases run on across the CTA's work tiles: the ring position, the count
// of P*V MMAs per query tile and the count of earlier tiles whose O_t the
// epilogue has to read before the next tile's first P*V overwrites it.
template <int D, bool CAUSAL, bool PERSIST, bool TRACE, bool FP8 = false>
__device__ __forceinline__ void mma_role(uint32_t sbase, uint32_t tmem, const FwdParams& p,
                                         const Waiter& w) {
  using L = Smem<D, FP8>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false, false);  // Q, K both K-major
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);     // V is MN-major
  constexpr uint32_t kHi = desc_hi_sw128(1024);                          // 8 rows x 128 B
  const uint32_t col_s[2] = {L::kColS0, L::kColS1};
  const uint32_t col_o[2] = {L::kColO0, L::kColO1};
  constexpr bool kOwnP = OwnP<D, PERSIST, FP8>::value;
  const uint32_t col_p[2] = {OwnP<D, PERSIST, FP8>::col(0), OwnP<D, PERSIST, FP8>::col(1)};
#ifdef FA4_PROF
  unsigned pm_acc[4] = {0, 0, 0, 0}, pm_n = 0, pm_pw = 0;
#endif
  // Low descriptor halves: K-major operands (LBO unused = 16 B), V with the
  // 64-column panel stride as LBO.
  const uint32_t q_lo[2] = {desc_lo_sw128(sbase + L::kQ, 16),
                            desc_lo_sw128(sbase + L::kQ + L::kTileBytes, 16)};
  const uint32_t ring_lo_k = desc_lo_sw128(sbase + L::kRing, 16);
  const uint32_t ring_lo_v = desc_lo_sw128(sbase + L::kRing, L::kPanelBytes);
  constexpr uint32_t kSlotStep = L::kTileBytes >> 4;

  auto issue_s = [&](int t, int slot) {
    const uint32_t k_lo = ring_lo_k + slot * kSlotStep;
    if constexpr (FP8) {
      // e4m3: 32 elements (32 bytes of the 128-byte row) per MMA
      constexpr uint32_t kIdesc8 = idesc_e4m3_f32(kBM, kBN, false, false);
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        const uint32_t off = (kk * 32) >> 4;
        mma_ss_lohi_f8_warp(tmem + col_s[t], q_lo[t] + off, kHi, k_lo + off, kHi, kIdesc8, kk > 0 ? 1u : 0u);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * L::kPanelBytes + (kk & 3) * 32) >> 4;
        mma_ss_lohi_warp(tmem + col_s[t], q_lo[t] + off, kHi, k_lo + off, kHi, kIdescQK, kk > 0 ? 1u : 0u);
      }
    }
    mma_commit_warp(bar(L::bSFull + t));
  };
  // O_t (+)= P_t V; each slice of P is issued once the softmax warps have
  // stored it. `phase` counts this tile's earlier P*V MMAs. Returns false on
  // abort.
  auto issue_pv = [&](int t, int slot, bool first, int phase, bool commit_done) -> bool {
    const uint32_t v_lo = ring_lo_v + slot * kSlotStep;
    constexpr int kSlices = FP8 ? 1 : FA4_P_SLICES;   // the FP8 P is released whole
#pragma unroll
    for (int half = 0; half < kSlices; ++half) {
      if (!w.wait_warp(bar(L::bPHalf + 2 * t + half), static_cast<uint32_t>(phase) & 1u, L::bPHalf + 2 * t + half))
        return false;
      tc_fence_after_sync();
#ifdef FA4_PROF
      pm_pw = static_cast<unsigned>(clock());
#endif
      if constexpr (FP8) {
        // 32 keys per step: 8 TMEM columns of packed e4m3 P, 32 rows (4 KB) of V
        constexpr uint32_t kIdescPv8 = idesc_e4m3_f32(kBM, D, false, true);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_ts_lohi_f8_warp(tmem + col_o[t], tmem + col_p[t] + kk * 8, v_lo + kk * (4096 >> 4), kHi,
                              kIdescPv8, (!first || kk > 0) ? 1u : 0u);
      } else {
#pragma unroll
        for (int k = 0; k < kBN / 16 / FA4_P_SLICES; ++k) {
          // 16 keys per step: 8 TMEM columns of packed P, 16 rows (2 KB) of V.
          const int kk = half * (kBN / 16 / FA4_P_SLICES) + k;
          mma_ts_lohi_warp(tmem + col_o[t], tmem + col_p[t] + kk * 8, v_lo + kk * (2048 >> 4), kHi,
                      kIdescPV, (!first || kk > 0) ? 1u : 0u);
        }
      }
    }
    // pv_done is only needed after a tile's last P*V of a work tile (the
    // epilogue) and, in strict order, before every next S. Any other P*V
    // has completed once the commit of the S MMA issued behind it arrives.
    if (commit_done) mma_commit_warp(bar(L::bPvDone + t));
    return true;
  };
  auto wait_slot = [&](int pos) -> bool {
    const int s = pos % L::kSlots;
    const bool ok = w.wait_warp(bar(L::bKvFull + s), static_cast<uint32_t>(pos / L::kSlots) & 1u,
                           L::bKvFull + s);
    tc_fence_after_sync();
    return ok;
  };

  int cons = 0;                 // ring positions consumed
  int n_q = 0;                  // Q tile pairs consumed
  int n_s[2] = {0, 0};          // S MMAs issued per query tile
  int n_pv[2] = {0, 0};         // P*V MMAs issued per query tile
  int n_epi[2] = {0, 0};        // earlier work tiles whose O_t the epilogue reads
  bool ok = true;
  int iter = 0;
  for (int id = tile_of<PERSIST>(0, p.n_tiles); ok && id < p.n_tiles; id = tile_of<PERSIST>(++iter, p.n_tiles)) {
    const Tile tl = make_tile<CAUSAL>(p, id);
    if (tl.nkv_max == 0) continue;
    if (!(ok = w.wait_warp(bar(L::bQ), static_cast<uint32_t>(n_q) & 1u, L::bQ))) break;
    tc_fence_after_sync();
    ++n_q;
    // S_0(0), S_1(0)
    if (!(ok = wait_slot(cons))) break;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (tl.nkv[t] == 0) continue;
      if constexpr (kOwnP) {
        // the softmax must have read the previous work tile's last S_t
        if (n_s[t] > 0 &&
            !(ok = w.wait_warp(bar(L::bSFree + t), static_cast<uint32_t>(n_s[t] - 1) & 1u, L::bSFree + t)))
          break;
        tc_fence_after_sync();
        ++n_s[t];
      }
      trace_mark_lane0<TRACE>(p, kTrMmaSGo, 0, t, iter);
      issue_s(t, cons % L::kSlots);
      trace_mark_lane0<TRACE>(p, kTrMmaSIssued, 0, t, iter);
    }
    if (kOwnP && !ok) break;
    mma_commit_warp(bar(L::bKvEmpty + cons % L::kSlots));
    ++cons;
    if (tl.nkv_max == 1) mma_commit_warp(bar(L::bQEmpty));     // no further S of this tile
    if constexpr (kOwnP) {
      // P_t has its own columns: per key block j, first S_t(j+1) for both
      // tiles (each as soon as softmax_t(j) has read S_t(j)), then
      // O_t += P_t(j) V_j for both tiles, each followed by a pv_done commit.
      for (int j = 0; ok && j < tl.nkv_max; ++j) {
        const int vpos = cons, kpos = cons + 1;             // V_j, then K_{j+1}
        const bool next = j + 1 < tl.nkv_max;
        if (next) {
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j + 1 >= tl.nkv[t]) continue;
            trace_mark_lane0<TRACE>(p, kTrMmaSWait, j + 1, t, iter);
            if (!(ok = w.wait_warp(bar(L::bSFree + t), static_cast<uint32_t>(n_s[t] - 1) & 1u,
                                   L::bSFree + t)))
              break;
            tc_fence_after_sync();
            if (!k_ready) {
              if (!(ok = wait_slot(kpos))) break;
              k_ready = true;
            }
            trace_mark_lane0<TRACE>(p, kTrMmaSGo, j + 1, t, iter);
            issue_s(t, kpos % L::kSlots);
            ++n_s[t];
            trace_mark_lane0<TRACE>(p, kTrMmaSIssued, j + 1, t, iter);
          }
          if (!ok) break;
          // K_{j+1} was needed by at least one tile (the one with nkv_max blocks).
          mma_commit_warp(bar(L::bKvEmpty + kpos % L::kSlots));
          // The last S MMAs of this work tile are issued: once they complete
          // the Q buffers may take the next tile's queries.
          if (j + 2 == tl.nkv_max) mma_commit_warp(bar(L::bQEmpty));
        }
        if (!(ok = wait_slot(vpos))) break;
        trace_mark_lane0<TRACE>(p, kTrMmaVReady, j, 0, iter);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= tl.nkv[t]) continue;
          trace_mark_lane0<TRACE>(p, kTrMmaPvWait, j, t, iter);
          if (p.correction_wg &&
              !(ok = w.wait_warp(bar(L::bOReady + t), static_cast<uint32_t>(n_pv[t]) & 1u, L::bOReady + t)))
            break;
          if (j == 0 && n_epi[t] > 0 &&     // the previous tile's O_t must have been read out
              !(ok = w.wait_warp(bar(L::bOFree + t), static_cast<uint32_t>(n_epi[t] - 1) & 1u, L::bOFree + t)))
            break;
          tc_fence_after_sync();
          trace_mark_lane0<TRACE>(p, kTrMmaPvGo, j, t, iter);
          if (!(ok = issue_pv(t, vpos % L::kSlots, j == 0, n_pv[t], true))) break;
          ++n_pv[t];
          trace_mark_lane0<TRACE>(p, kTrMmaPvIssued, j, t, iter);
        }
        if (!ok) break;
        mma_commit_warp(bar(L::bKvEmpty + vpos % L::kSlots));
        cons += next ? 2 : 1;
        trace_mark_lane0<TRACE>(p, kTrMmaCommitted, j, 0, iter);
      }
    } else
    for (int j = 0; ok && j < tl.nkv_max; ++j) {
      const int vpos = cons, kpos = cons + 1;             // V_j, then K_{j+1}
      const bool next = j + 1 < tl.nkv_max;
      if (!(ok = wait_slot(vpos))) break;
      trace_mark_lane0<TRACE>(p, kTrMmaVReady, j, 0, iter);
      bool k_ready = false;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= tl.nkv[t]) continue;
        trace_mark_lane0<TRACE>(p, kTrMmaPvWait, j, t, iter);
        FA4_PROF_CLK(pm_a);
        if (p.correction_wg &&
            !(ok = w.wait_warp(bar(L::bOReady + t), static_cast<uint32_t>(n_pv[t]) & 1u, L::bOReady + t)))
          break;
        if (j == 0 && n_epi[t] > 0 &&     // the previous tile's O_t must have been read out
            !(ok = w.wait_warp(bar(L::bOFree + t), static_cast<uint32_t>(n_epi[t] - 1) & 1u, L::bOFree + t)))
          break;
        tc_fence_after_sync();
        trace_mark_lane0<TRACE>(p, kTrMmaPvGo, j, t, iter);
        if (!(ok = issue_pv(t, vpos % L::kSlots, j == 0, n_pv[t], p.strict_order || j + 1 == tl.nkv[t])))
          break;
        ++n_pv[t];
        FA4_PROF_CLK(pm_b);
        trace_mark_lane0<TRACE>(p, kTrMmaPvIssued, j, t, iter);
        if (j + 1 >= tl.nkv[t]) continue;
        trace_mark_lane0<TRACE>(p, kTrMmaSWait, j + 1, t, iter);
        if (!k_ready) {
          if (!(ok = wait_slot(kpos))) break;
          k_ready = true;
        }
        if (p.strict_order) {
          if (!(ok = w.wait_warp(bar(L::bPvDone + t), static_cast<uint32_t>(n_pv[t] - 1) & 1u,
                            L::bPvDone + t)))
            break;
          tc_fence_after_sync();
        }
        trace_mark_lane0<TRACE>(p, kTrMmaSGo, j + 1, t, iter);
        FA4_PROF_CLK(pm_c);
        issue_s(t, kpos % L::kSlots);
#ifdef FA4_PROF
        if (j > 0) {
          const unsigned pm_d = static_cast<unsigned>(clock());
          pm_acc[0] += pm_pw - pm_a;
          pm_acc[1] += pm_b - pm_pw;
          pm_acc[2] += pm_c - pm_b;
          pm_acc[3] += pm_d - pm_c;
          ++pm_n;
        }
#endif
        trace_mark_lane0<TRACE>(p, kTrMmaSIssued, j + 1, t, iter);
      }
      if (!ok) break;
      mma_commit_warp(bar(L::bKvEmpty + vpos % L::kSlots));
      ++cons;
      if (next) {
        // K_{j+1} was needed by at least one tile (the one with nkv_max blocks).
        mma_commit_warp(bar(L::bKvEmpty + kpos % L::kSlots));
        ++cons;
      }
      // The last S MMAs of this work tile are issued: once they complete the
      // Q buffers may take the next tile's queries.
      if (j + 2 == tl.nkv_max) mma_commit_warp(bar(L::bQEmpty));
      trace_mark_lane0<TRACE>(p, kTrMmaCommitted, j, 0, iter);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (tl.nkv[t] > 0) ++n_epi[t];
  }
  // Every MMA issued above has completed once this commit arrives.
  mma_commit_warp(bar(L::bDrain));
  w.drain_warp(bar(L::bDrain), 0u, L::bDrain);
#ifdef FA4_PROF
  if ((threadIdx.x & 31) == 0) {
    for (int i = 0; i < 4; ++i) atomicAdd(&g_prof[8 + i], static_cast<unsigned long long>(pm_acc[i]));
    atomicAdd(&g_prof[12], static_cast<unsigned long long>(pm_n));
  }
#endif
}

// ------------------------------------------------------------ correction WG
template <int D, bool CAUSAL, bool PERSIST, bool TRACE, bool FP8 = false>
__device__ __forceinline__ void correction_role(uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                                const FwdParams& p, const Waiter& w) {
  using L = Smem<D, FP8>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const float* alpha_s = reinterpret_cast<const float*>(smem + L::kAlpha);
  volatile int* flags_s = reinterpret_cast<volatile int*>(smem + L::kFlags);
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t col_o[2] = {L::kColO0, L::kColO1};
  int n_step[2] = {0, 0};       // softmax steps seen per query tile (all work tiles)
  int iter = 0;
  for (int id = tile_of<PERSIST>(0, p.n_tiles); id < p.n_tiles; id = tile_of<PERSIST>(++iter, p.n_tiles)) {
    const Tile tl = make_tile<CAUSAL>(p, id);
    for (int j = 0; j < tl.nkv_max; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= tl.nkv[t]) continue;
        const int cnt = n_step[t]++;
        const int buf = cnt & 1;
        if (!w.wait(bar(L::bPFull + t), static_cast<uint32_t>(cnt) & 1u, L::bPFull + t)) return;
        tc_fence_after_sync();
        if (warp == 8 && lane == 0) trace_mark<TRACE>(p, kTrCoWake, j, t, iter);
        const int fval = flags_s[(buf * 2 + t) * 4 + wq];
        const bool flagged = j > 0 && fval != 0;
        // a set flag is cleared here, so a step that needs no rescale
        // stores nothing before its p_full arrival
        if (fval != 0 && lane == 0) flags_s[(buf * 2 + t) * 4 + wq] = 0;
        const float a = flagged ? alpha_s[(buf * 2 + t) * kBM + r] : 1.0f;
        // this buffer's flags and alpha are read: the softmax may reuse it
        // two steps on
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bCDone + 2 * t + buf));
        if (flagged) {
          // This 32-row group's reference max moved: O_t <- alpha * O_t, then
          // release the group. The previous P*V into O_t has completed: the
          // S MMA issued behind it had completed before the softmax warps
          // arrived on p_full. With its own P columns no S MMA is issued
          // behind it, so wait for its pv_done commit.
          if (OwnP<D, PERSIST, FP8>::value &&
              !w.wait(bar(L::bPvDone + t), static_cast<uint32_t>(cnt - 1) & 1u, L::bPvDone + t))
            return;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t x[16];
            const uint32_t addr = lane_base + col_o[t] + c * 16;
            tmem_ld_x16(addr, x);
            tmem_wait_ld_x16(x);
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * a);
            tmem_st_x16(addr, x);
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::bOReady + t));
        }
        if (warp == 8 && lane == 0) trace_mark<TRACE>(p, kTrCoArrived, j, t, iter);
      }
    }
  }
}

// ------------------------------------------------------------ softmax WGs
// Entry pair pi (columns 2 pi, 2 pi + 1) of a 128-key block goes through the
// software 2^x when pi % PERIOD == PERIOD - 1 (PERIOD = 8: 12.5 % of the
// entries, PERIOD = 4: 25 %); PERIOD = 0 sends every entry through MUFU.EX2.
template <int PERIOD>
__host__ __device__ constexpr bool emulated_pair(int pi) {
  if constexpr (PERIOD <= 0) {
    return false;
  } else {
    return (pi % PERIOD) == PERIOD - 1;
  }
}

// One row's 128 exponentials p = 2^(c s + neg_m) on pairs of entries
// (FFMA2 / FADD2): the row sum of the fp32 p goes to `tot` (two partial
// halves), P is packed for the P*V MMA (BF16 pairs, or e4m3 quads with
// FP8).
template <int EMU_PAIR_PERIOD, bool FP8>
__device__ __forceinline__ void exp_pass(const uint32_t (&s)[128], float2 c2, float neg_m,
                                         uint32_t (&pk)[FP8 ? 32 : 64], float2& tot) {
  const float2 nm2 = make_float2(neg_m, neg_m);
  float2 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int pi = 0; pi < 64; ++pi) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * pi]), __uint_as_float(s[2 * pi + 1])),
                                c2, nm2);
    const float2 pp = emulated_pair<EMU_PAIR_PERIOD>(pi)
                          ? ex2_emulated2(x)
                          : make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
    acc[pi & 3] = __fadd2_rn(acc[pi & 3], pp);
    if constexpr (FP8) {
      const uint32_t h = pack_e4m3x2(pp.x, pp.y);
      pk[pi >> 1] = (pi & 1) ? (pk[pi >> 1] | (h << 16)) : h;
    } else {
      pk[pi] = pack_bf16x2(pp.x, pp.y);
    }
  }
  tot = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
}

template <int D, bool CAUSAL, int EMU_PAIR_PERIOD, bool PERSIST, bool TRACE, bool FP8 = false>
__device__ __forceinline__ void softmax_role(int t, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                             const FwdParams& p, const Waiter& w) {
  using L = Smem<D, FP8>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;                 // row within the tile = TMEM lane
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);
  volatile int* flags_s = reinterpret_cast<volatile int*>(smem + L::kFlags);
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t s_addr = lane_base + (t == 0 ? L::kColS0 : L::kColS1);
  constexpr bool kOwnP = OwnP<D, PERSIST, FP8>::value;
  const uint32_t p_addr = lane_base + OwnP<D, PERSIST, FP8>::col(t);
  const uint32_t o_addr = lane_base + (t == 0 ? L::kColO0 : L::kColO1);
  const float cl2 = p.scale_log2;
  const int shift = p.Sk - p.Sq;
  unsigned n_rescaled = 0, n_steps = 0;
#ifdef FA4_PROF
  unsigned pr_acc[5] = {0, 0, 0, 0, 0}, pr_prev_arrived = 0, pr_n = 0;
#endif
  int n_step = 0;               // steps of this query tile over all work tiles
  int n_fin = 0;                // work tiles in which this query tile saw keys
  bool ok = true;
  int iter = 0;
  if (p.test_stall_cycles > 0)   // diagnostic: a wait nothing ends
    ok = w.wait_for(bar(L::bStall), 0u, L::bStall, p.test_stall_cycles);
  for (int id = tile_of<PERSIST>(0, p.n_tiles); ok && id < p.n_tiles; id = tile_of<PERSIST>(++iter, p.n_tiles)) {
  const Tile tl = make_tile<CAUSAL>(p, id);
  const int row = tl.q0 + t * kBM + r;          // query index
  const int n = t == 0 ? tl.nkv[0] : tl.nkv[1];  // (a runtime index would put Tile in local memory)
  // Keys k < lim_row are visible to this row; lim_min is the tile's smallest.
  const int lim_row = CAUSAL ? max(0, min(p.Sk, row + shift + 1)) : p.Sk;
  const int row_min = tl.q0 + t * kBM;
  const int lim_min = CAUSAL ? max(0, min(p.Sk, row_min + shift + 1)) : p.Sk;
  float m_ref = -INFINITY;      // reference max (log2 units) of the last rescale
  float l = 0.0f;               // running sum of p relative to m_ref

  for (int j = 0; j < n; ++j) {
    if (!(ok = w.wait(bar(L::bSFull + t), static_cast<uint32_t>(n_step) & 1u, L::bSFull + t))) break;
    tc_fence_after_sync();
    FA4_PROF_CLK(pr_t0);
    const bool tracer = (wq == 0 && lane == 0);
    if (tracer) trace_mark<TRACE>(p, kTrSmSReady, j, t, iter);
    uint32_t s[128];
    tmem_ld_x32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_ld_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_ld_x32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
    tmem_ld_x32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
    // Hand-off buffer of this step (the one step n - 2 used; the end of
    // step n - 1 checked that the correction warps have read it).
    const int buf = n_step & 1;
    tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&s[64]));
    tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&s[96]));
    // With its own P columns, the MMA warp may compute the next S_t into
    // these columns as soon as all four warps have read them.
    if constexpr (kOwnP) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bSFree + t));
    }
    // Own P: before this step rescales O_t or overwrites P_t, the previous
    // step's P*V must have completed (the S MMA this step waited for was
    // issued before it, so its commit does not track it). At j = 0 the
    // epilogue of the previous work tile has waited for its last P*V.
    bool pv_prev_done = !kOwnP || j == 0;
    auto wait_pv_prev = [&]() -> bool {
      if (pv_prev_done) return true;
      pv_prev_done = true;
      const bool r = w.wait(bar(L::bPvDone + t), static_cast<uint32_t>(n_step - 1) & 1u, L::bPvDone + t);
      tc_fence_after_sync();
      return r;
    };
    FA4_PROF_CLK(pr_t1);
    if (tracer) trace_mark<TRACE>(p, kTrSmLoaded, j, t, iter);
    const int kb = tl.kv0 + j;           // absolute key block
    const bool masked = (kb + 1) * kBN > lim_min;   // tile-uniform: this block has masked keys
    const int lim = lim_row - kb * kBN;             // this row's first masked column
    if (masked) {
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : __float_as_uint(-INFINITY);
    }
    const float2 c2 = make_float2(cl2, cl2);
    float2 tot;
    // P for the P*V MMA: BF16 pairs (64 columns), or with FP8 e4m3 quads
    // (32 columns; key 4i + j in byte j of column i), rounded from fp32
    uint32_t pk[FP8 ? 32 : 64];
    // Conditional rescale (§3.1.4, Eq. 6): only when the max moved by more
    // than tau, decided per warp so the correction stays warp-uniform. Once
    // decided, the correction warps may read flag / alpha and rescale O_t
    // while the exponentials run; row groups that need no rescale release
    // O_t for the next P*V right away. (Every thread arrives on p_full after
    // its own alpha store; measured faster than one arrival per warp behind
    // a warp barrier.)
#ifdef FA4_PROF
    unsigned pr_t2 = 0;
#endif
    auto release = [&](float m_cand, bool warp_need) {
      if (tracer) trace_mark<TRACE>(p, kTrSmCDone, j, t, iter);
      if (tracer) trace_mark<TRACE>(p, kTrSmMaxDone, j, t, iter);
      if (!p.correction_wg) {
        if (warp_need) {
          const float alpha = (m_cand == -INFINITY) ? 1.0f : ex2_mufu(m_ref - m_cand);
          l *= alpha;
          if (m_cand != -INFINITY) m_ref = m_cand;
          if (j > 0) {
            ++n_rescaled;
            // O_t <- alpha * O_t for this warp's rows. The previous P*V into
            // O_t has completed: the S MMA issued behind it, whose commit this
            // step waited for, tracks it too (with its own P columns, the
            // explicit pv_done wait).
            if constexpr (kOwnP) {
              if (!wait_pv_prev()) ok = false;
            }
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t x[16];
              tmem_ld_x16(o_addr + c * 16, x);
              tmem_wait_ld_x16(x);
#pragma unroll
              for (int i = 0; i < 16; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * alpha);
              tmem_st_x16(o_addr + c * 16, x);
            }
            tmem_wait_st();
            tc_fence_before_sync();
          }
        }
        // No o_ready arrival: the P arrival below comes after this warp's
        // rescale in program order, so the MMA warp waits for P alone.
        if (j > 0) ++n_steps;
#ifdef FA4_PROF
        pr_t2 = static_cast<unsigned>(clock());
#endif
        return;
      }
      // Own P: S_t(j+1) is issued before P_t(j) V_j, so this step may run a
      // whole step ahead of the consumers of p_full and o_ready. Before it
      // arrives on either, the correction warps must have taken the previous
      // step's hand-off (which also frees the buffer this step reuses, two
      // steps on) and the MMA warp its o_ready (its P*V has completed);
      // otherwise a phase could complete twice before its consumer looks.
      // Without own P the next S follows the P*V that waits for o_ready, and
      // the hand-off check stays at the end of the step (below), off the
      // step's path.
      if constexpr (kOwnP) {
        if (n_step >= 1 &&
            !w.wait(bar(L::bCDone + 2 * t + (buf ^ 1)), static_cast<uint32_t>((n_step - 1) >> 1) & 1u,
                    L::bCDone + 2 * t + (buf ^ 1)))
          ok = false;
        if (!wait_pv_prev()) ok = false;
      }
      if (warp_need) {
        const float alpha = (m_cand == -INFINITY) ? 1.0f : ex2_mufu(m_ref - m_cand);
        l *= alpha;
        if (m_cand != -INFINITY) m_ref = m_cand;
        alpha_s[(buf * 2 + t) * kBM + r] = alpha;
        if (j > 0) ++n_rescaled;
      }
      if (lane == 0 && warp_need) flags_s[(buf * 2 + t) * 4 + wq] = 1;
      mbar_arrive(bar(L::bPFull + t));
      __syncwarp();
      if (lane == 0 && (!warp_need || j == 0)) mbar_arrive(bar(L::bOReady + t));
      if (j > 0) ++n_steps;
#ifdef FA4_PROF
      pr_t2 = static_cast<unsigned>(clock());
#endif
    };
    // p = 2^(c*s - m_ref) on pairs of entries (FFMA2 / FADD2); one pair in
    // EMU_PAIR_PERIOD goes through the FMA-pipe emulation (§3.1.3), the rest
    // through MUFU.EX2. The row sum uses the fp32 p; P is stored as BF16.
    auto neg_ref = [&]() { return (m_ref == -INFINITY) ? 0.0f : -m_ref; };
    {
      // block max of the raw scores (scale > 0, so max commutes with it)
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
      for (int c = 8; c < 128; c += 8)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mx[i] = fmax3(mx[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
      const float m_cand = fmaxf(m_ref, fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * cl2);
      if (tracer) trace_mark<TRACE>(p, kTrSmMaxLoop, j, t, iter);
      release(m_cand, __any_sync(0xffffffffu, m_cand > m_ref + p.tau));
      exp_pass<EMU_PAIR_PERIOD, FP8>(s, c2, neg_ref(), pk, tot);
    }
    FA4_PROF_CLK(pr_t3);
    if (tracer) trace_mark<TRACE>(p, kTrSmExpDone, j, t, iter);
    // Own P: the previous P*V must have read P_t before it is overwritten.
    if constexpr (kOwnP) {
      if (!wait_pv_prev()) ok = false;
      if (!ok) break;
    }
    // P goes to the first kPCols columns of S_t (at head dim 64 to its own
    // columns), released to the P*V MMAs in kSlices parts (the FP8 forward
    // always releases it whole)
    constexpr int kPCols = FP8 ? 32 : 64;
    constexpr int kSlices = FP8 ? 1 : FA4_P_SLICES;
    constexpr int kSliceCols = kPCols / kSlices;
#pragma unroll
    for (int half = 0; half < kSlices; ++half) {
#pragma unroll
      for (int q = 0; q < kSliceCols / 32; ++q)
        tmem_st_x32(p_addr + half * kSliceCols + q * 32,
                    *reinterpret_cast<const uint32_t(*)[32]>(&pk[half * kSliceCols + q * 32]));
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bPHalf + 2 * t + half));
    }
    l += tot.x + tot.y;
#ifdef FA4_PROF
    {
      const unsigned pr_t4 = static_cast<unsigned>(clock());
      if (j > 0) {
        pr_acc[0] += pr_t1 - pr_t0;
        pr_acc[1] += pr_t2 - pr_t1;
        pr_acc[2] += pr_t3 - pr_t2;
        pr_acc[3] += pr_t4 - pr_t3;
        pr_acc[4] += pr_t0 - pr_prev_arrived;
        ++pr_n;
      }
      pr_prev_arrived = pr_t4;
    }
#endif
    if (tracer) trace_mark<TRACE>(p, kTrSmArrived, j, t, iter);
    if (lane == 0 && wq > 0) trace_mark<TRACE>(p, kTrSmArrivedQ1 + wq - 1, j, t, iter);
    // The next step reuses the buffer of step n_step - 1: the correction
    // warps must have read it. Checked here, where the warp would otherwise
    // only wait for the next S, rather than on the next step's path.
    if (!kOwnP && p.correction_wg && n_step >= 1 &&
        !(ok = w.wait(bar(L::bCDone + 2 * t + (buf ^ 1)), static_cast<uint32_t>((n_step - 1) >> 1) & 1u,
                      L::bCDone + 2 * t + (buf ^ 1))))
      break;
    ++n_step;
  }

  if (!ok) break;
  // ---- epilogue: O / l -> BF16 -> global, LSE = ln2 * (m_ref + log2 l);
  // with a key-range split, fp32 O / l and LSE of this split into the
  // partial buffers instead.
  const bool row_valid = row < p.Sq;
  const bool has_keys = n > 0 && m_ref != -INFINITY;
  const float inv_l = has_keys ? p.out_scale / l : 0.0f;
  const bool partial = p.o_part != nullptr;
  const int64_t orow_idx = (static_cast<int64_t>(tl.b) * p.Sq + row) * p.Hq + tl.h;
  const int64_t part_off = static_cast<int64_t>(tl.split) * p.B * p.Sq * p.Hq;
  __nv_bfloat16* orow = p.o + orow_idx * static_cast<int64_t>(D);
  float* prow = p.o_part + (part_off + orow_idx) * static_cast<int64_t>(D);
  if (n > 0) {
    // one pv_done commit per work tile (per step in strict order and with
    // own P)
    const uint32_t pv_par = (p.strict_order || kOwnP) ? static_cast<uint32_t>(n_step - 1) & 1u
                                                      : static_cast<uint32_t>(n_fin) & 1u;
    ++n_fin;
    if (!(ok = w.wait(bar(L::bPvDone + t), pv_par, L::bPvDone + t)))
      break;
    tc_fence_after_sync();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t x[32];
      tmem_ld_x32(o_addr + c * 32, x);
      tmem_wait_ld_x32(x);
      if (c == D / 32 - 1) {
        // O_t is read out: the next work tile's first P*V may overwrite it.
        tc_fence_before_sync();
        mbar_arrive(bar(L::bOFree + t));
      }
      if (row_valid && partial) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<float4*>(prow + c * 32)[i] =
              make_float4(__uint_as_float(x[4 * i + 0]) * inv_l, __uint_as_float(x[4 * i + 1]) * inv_l,
                          __uint_as_float(x[4 * i + 2]) * inv_l, __uint_as_float(x[4 * i + 3]) * inv_l);
      } else if (row_valid) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(x[8 * i + 0]) * inv_l, __uint_as_float(x[8 * i + 1]) * inv_l);
          v.y = pack_bf16x2(__uint_as_float(x[8 * i + 2]) * inv_l, __uint_as_float(x[8 * i + 3]) * inv_l);
          v.z = pack_bf16x2(__uint_as_float(x[8 * i + 4]) * inv_l, __uint_as_float(x[8 * i + 5]) * inv_l);
          v.w = pack_bf16x2(__uint_as_float(x[8 * i + 6]) * inv_l, __uint_as_float(x[8 * i + 7]) * inv_l);
          reinterpret_cast<uint4*>(orow + c * 32)[i] = v;
        }
      }
    }
  } else if (row_valid && partial) {
    float4* dst = reinterpret_cast<float4*>(prow);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else if (row_valid) {
    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (row_valid) {
    const float lse_val = has_keys ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    const int64_t li = (static_cast<int64_t>(tl.b) * p.Hq + tl.h) * p.Sq + row;
    if (partial)
      p.lse_part[static_cast<int64_t>(tl.split) * p.B * p.Hq * p.Sq + li] = lse_val;
    else
      p.lse[li] = lse_val;
  }
  }  // work tiles
  if (p.stats != nullptr && lane == 0 && n_steps > 0) {
    atomicAdd(&p.stats[0], static_cast<unsigned long long>(n_rescaled));
    atomicAdd(&p.stats[1], static_cast<unsigned long long>(n_steps));
  }
#ifdef FA4_PROF
  if (t == 0 && wq == 0 && lane == 0) {
    for (int i = 0; i < 5; ++i) atomicAdd(&g_prof[i], static_cast<unsigned long long>(pr_acc[i]));
    atomicAdd(&g_prof[5], static_cast<unsigned long long>(pr_n));
  }
#endif
}

// ------------------------------------------------------------ kernel
template <int D, bool CAUSAL, int EMU_PAIR_PERIOD, bool PERSIST, bool TRACE, bool FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa4_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Smem<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    mbar_init(bar(L::bQ), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bar(L::bKvFull + s), 1);
      mbar_init(bar(L::bKvEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::bSFull + t), 1);
      mbar_init(bar(L::bPFull + t), kBM);
      mbar_init(bar(L::bOReady + t), 4);
      mbar_init(bar(L::bPvDone + t), 1);
      mbar_init(bar(L::bCDone + 2 * t), 4);
      mbar_init(bar(L::bCDone + 2 * t + 1), 4);
      mbar_init(bar(L::bPHalf + 2 * t), 4);
      mbar_init(bar(L::bPHalf + 2 * t + 1), 4);
      mbar_init(bar(L::bOFree + t), kBM);
    }
    mbar_init(bar(L::bQEmpty), 1);
    mbar_init(bar(L::bDrain), 1);
    mbar_init(bar(L::bStall), 1);
    mbar_init(bar(L::bSFree), 4);
    mbar_init(bar(L::bSFree + 1), 4);
    for (int i = 0; i < 16; ++i) reinterpret_cast<volatile int*>(smem + L::kFlags)[i] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Register split (setmaxnreg): 256 softmax threads, 128 correction, 128
  // load/MMA; the total must equal the 512 x 128 the block launches with.
  constexpr int kRegsSoftmax = 184;
  constexpr int kRegsCorrection = D == 128 ? 56 : 64;
  constexpr int kRegsLoadMma = D == 128 ? 88 : 80;
  static_assert(256 * kRegsSoftmax + 128 * kRegsCorrection + 128 * kRegsLoadMma == kThreads * 128,
                "register split must use exactly the launch allocation");
  if (warp < 8) {
    regs_increase<kRegsSoftmax>();
    const Waiter w{abort_flag, p.status, kRoleSoftmax};
    softmax_role<D, CAUSAL, EMU_PAIR_PERIOD, PERSIST, TRACE, FP8>(warp >> 2, sbase, smem, tmem, p, w);
  } else if (warp < 12) {
    regs_decrease<kRegsCorrection>();
    const Waiter w{abort_flag, p.status, kRoleCorrection};
    if (p.correction_wg) correction_role<D, CAUSAL, PERSIST, TRACE, FP8>(sbase, smem, tmem, p, w);
  } else {
    regs_decrease<kRegsLoadMma>();
    if (warp == kWarpLoad) {
      const Waiter w{abort_flag, p.status, kRoleLoad};
      load_role<D, CAUSAL, PERSIST, TRACE, FP8>(&tm_q, &tm_k, &tm_v, sbase, p, w);
    } else if (warp == kWarpMma) {
      const Waiter w{abort_flag, p.status, kRoleMma};
      mma_role<D, CAUSAL, PERSIST, TRACE, FP8>(sbase, tmem, p, w);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa4
