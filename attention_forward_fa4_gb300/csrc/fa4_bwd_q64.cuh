// fa4_bwd_q64.cuh -- attention backward in steps of 64 queries (head dims
// 64 and 128), with the next step's S^T / dP^T MMAs overlapping the current
// step's softmax-side work ("FlashAttention-4: Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling", §3.2: five MMAs
// per tile pair, spread over producer and consumer warps).
//
// One CTA owns a 128-key block of one (batch, kv head) and walks every
// 64-query block of every query head that reads it. Tensor memory (512
// columns, lanes = keys for the transposed products) holds two steps:
//
//   S^T[b]  = K Q^T         SS MMA, M = 128 keys, N = 64    cols 64 b + [0, 64)
//   dP^T[b] = V dO^T        SS MMA                          cols 128 + 64 b + [0, 64)
//   P^T, dS^T (BF16)        compute warps, written over S^T[b]: the warp on
//                           queries 32 c .. 32 c + 31 puts P^T in columns
//                           32 c + [0, 16) and dS^T in 32 c + [16, 32)
//   dQ^T[b] = K^T dS^T      SS MMA, M = 128 (head dim; at 64 the K panel
//                           twice), N = 64 queries, A = K read MN-major, B =
//                           dS from shared memory; into dP^T[b] (already
//                           read), issued first so the read-out starts early
//   dV     += P^T dO        TS MMA, A = P^T from TMEM    cols 256 + [0, D)
//   dK     += dS^T Q        TS MMA, A = dS^T from TMEM   cols 256 + D + [0, D)
//
// With a step's P^T and dS^T both in its S^T columns, the dP^T columns take
// the dQ^T tile, so a step needs 128 columns and two fit beside dV and dK.
// The MMA warp issues step s + 2's S^T and dP^T as soon as step s's dQ^T has
// been read out; the tensor core then works on them (and on step s + 1's
// dV, dK, dQ^T) while the compute warps exponentiate step s + 1.
//
// Q, dO, LSE2 and Delta of a step sit in one of several stages (three at
// head dim 128, six at 64; the stage of step s is loaded once the dK MMA of
// the step that used it before has read it). The dQ^T tile is read out one
// head-dimension row per thread and staged transposed (row = query, 32-
// column blocks, 128-byte swizzle) in a ring of three units for bulk tensor
// reduce-adds into the global fp32 accumulator: a reduce-add reads its
// source in about as long as a step takes, so the next units are staged
// while earlier ones are still being read.
//
// Warps: 0-7 compute (two per TMEM lane quarter, 32 queries each), 8 TMA
// loads, 9 MMA issue, 10 dQ flush (in deterministic mode in key-block
// order), 11 idle, 12-15 dQ^T read-out and staging (one per lane quarter),
// so the compute warps go on to the next step as soon as P^T and dS^T are
// handed over. Every wait is bounded.
#pragma once

#include "fa4_fwd_kernel.cuh"

namespace fa4 {

constexpr int kBwdWarpLoad = 8;
constexpr int kBwdWarpMma = 9;
constexpr int kBwdWarpFlush = 10;

struct BwdParams {
  __nv_bfloat16* dk;        // [B, Sk, Hkv, D]
  __nv_bfloat16* dv;        // [B, Sk, Hkv, D]
  float* dq_acc;            // [B, Sq, Hq, D] fp32, zeroed; receives scale * dS K
  const float* lse2;        // [B * Hq][Sq_pad]
  const float* delta;       // [B * Hq][Sq_pad]
  int B, Hq, Hkv, Sq, Sk, group, Sq_pad, n_kblk;
  float scale, scale_log2;
  unsigned int* status;
  // Deterministic mode (non-null): one int per (batch, query head, 64-query
  // block), zeroed; the dQ tile of key block kb is added only once kb
  // earlier key blocks have added theirs, so the fp32 sums are formed in
  // the same order on every run. CTAs are then numbered key block first.
  int* dq_turn;
  // Deterministic mode: a zeroed counter from which each CTA takes its work
  // number when it starts, so every lower number belongs to a CTA that is
  // already running whatever order the hardware dispatched them in.
  int* cta_ticket;
  // Diagnostic (> 0): the compute warps first wait this many cycles on a
  // barrier nothing completes, so the launch takes the timeout path.
  long long test_stall_cycles;
};

// The CTA's key block and the query blocks it visits.
struct BwdWork {
  int b, g, k0;
  int qb0, n_qb;      // query blocks [qb0, n_qb) of every head in the group
  int steps;          // group * (n_qb - qb0)
};

constexpr int kBwdQ64Threads = 512;
constexpr int kBwdQ64WarpDq = 12;   // first of the four dQ^T read-out warps

// Head dim 128: two 64-column panels per K, V, Q, dO tile; dQ staged in
// halves of 32 queries. Head dim 64: one panel, with K loaded twice (the
// dQ^T MMA's M = 128 then yields the 64 head-dim rows twice, and the
// read-out warps of the duplicate lanes take the step's other 32 queries);
// dQ staged per whole step; six Q/dO stages.
template <int D>
struct BwdQ64Smem {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kPanels = D / 64;
  static constexpr int kKvPanel = 128 * 128;            // 128 rows x 64 BF16
  static constexpr int kQPanel = 64 * 128;              // 64 rows x 64 BF16
  static constexpr int kK = 0;                          // two panels (at D = 64 the same one twice)
  static constexpr int kV = kK + 2 * kKvPanel;
  static constexpr int kDS = kV + kPanels * kKvPanel;   // 128 keys x 64 queries BF16, MN-major
  static constexpr int kUnits = D == 128 ? 2 : 1;       // staged units per step
  static constexpr int kUnitRows = 64 / kUnits;
  static constexpr int kSlots = 3;                      // staging ring of dQ units
  static constexpr int kSlotBlock = kUnitRows * 128;    // [rows x 32 fp32]
  static constexpr int kSlotBytes = (D / 32) * kSlotBlock;
  static constexpr int kStg = kDS + 128 * 128;
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kStage0 = kStg + kSlots * kSlotBytes;
  static constexpr int kQ = 0, kDO = kPanels * kQPanel;
  static constexpr int kStageBytes = 2 * kPanels * kQPanel;
  static constexpr int kLd = kStage0 + kStages * kStageBytes;   // per stage LSE2[64], Delta[64]
  static constexpr int kBars = kLd + kStages * 512;
  // kv; per stage full (Q, dO, LSE2, Delta) and empty (after the dK MMA);
  // per buffer s / dp (S^T, dP^T committed); p_ready (P^T, dS^T written),
  // dq_full / dq_free (dQ^T committed / read out), acc (all MMAs done); per
  // staging slot full / free (handed to / back from the flush warp)
  static constexpr int bKv = 0, bFull = 1, bEmpty = bFull + kStages, bS = bEmpty + kStages,
                       bDP = bS + 2, bPReady = bDP + 2, bDqFull = bPReady + 1, bDqFree = bDqFull + 1,
                       bAcc = bDqFree + 1, bSlotFull = bAcc + 1, bSlotFree = bSlotFull + kSlots,
                       bStall = bSlotFree + kSlots,   // never completed (timeout test)
                       kNumBars = bStall + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;    // tmem base, abort flag, work number
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;          // re-align the base to 1 KB
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr int stage(int s) { return kStage0 + (s % kStages) * kStageBytes; }
  static constexpr int lse(int s) { return kLd + (s % kStages) * 512; }
  static constexpr int delta(int s) { return kLd + (s % kStages) * 512 + 256; }
};

template <bool CAUSAL>
__device__ __forceinline__ BwdWork bwd_q64_work(const BwdParams& p, int id) {
  BwdWork w;
  // Key blocks in groups of G, the groups in key order and every (batch, kv
  // head) inside each group:
  // - causal, G = 24: the longest CTAs (the first key blocks see the most
  //   queries) start first and the grid ends on short ones, while the live
  //   CTAs span few enough heads for their Q, dO and dQ accumulator to stay
  //   in L2. Measured on long causal (TFLOP/s, DRAM bytes per launch):
  //   G = 1 1061 / 2.91 GB, 16 1068 / 1.23 GB, 24 1072 / 0.97 GB,
  //   32 1056 / 0.83 GB, n_kblk (heads outermost) 1028 / 0.63 GB;
  // - deterministic mode, G = 1 (key block outermost: measured fastest for
  //   its turn chain); a lower key block of a head always has a lower work
  //   number, so every CTA whose turn comes earlier is already running;
  // - otherwise G = n_kblk: the key blocks of one (batch, kv head) side by
  //   side (their CTAs share Q and dO in L2).
  const int n_bg = p.B * p.Hkv;
  const int G = p.dq_turn ? 1 : (CAUSAL ? 24 : p.n_kblk);
  const int grp = id / (G * n_bg);
  const int in_grp = min(G, p.n_kblk - grp * G);
  const int rem = id - grp * G * n_bg;
  const int bg = rem / in_grp;
  const int kb = grp * G + rem % in_grp;
  w.b = bg / p.Hkv;
  w.g = bg - w.b * p.Hkv;
  w.k0 = kb * 128;
  w.n_qb = (p.Sq + 63) / 64;
  w.qb0 = 0;
  if (CAUSAL) {
    const long long i_min = static_cast<long long>(w.k0) - (p.Sk - p.Sq);
    w.qb0 = i_min <= 0 ? 0 : static_cast<int>(i_min / 64 < w.n_qb ? i_min / 64 : w.n_qb);
  }
  w.steps = p.group * (w.n_qb - w.qb0);
  return w;
}

// Query block of step s (its head is wk.g * group + s / (n_qb - qb0)). In
// deterministic mode each head's blocks are walked from the last one down:
// every key block then reaches a query block right after the key block
// before it (in whose order the adds must come), instead of two blocks
// ahead of it as an upward walk from each key block's diagonal would put it.
__device__ __forceinline__ int bwd_q64_qb(const BwdWork& wk, const BwdParams& p, int s) {
  const int per_head = wk.n_qb - wk.qb0;
  const int r = s % per_head;
  return p.dq_turn ? wk.n_qb - 1 - r : wk.qb0 + r;
}

template <int D>
__device__ __forceinline__ int bwd_q64_work_id(uint32_t sbase) {
  int id;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(id) : "r"(sbase + BwdQ64Smem<D>::kMisc + 8) : "memory");
  return id;
}

// ------------------------------------------------------------ load warp
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_q64_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                                  const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                                  uint32_t sbase, const BwdParams& p, const Waiter& w) {
  using L = BwdQ64Smem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_q64_work<CAUSAL>(p, bwd_q64_work_id<D>(sbase));
  if (wk.steps == 0) return;
  mbar_arrive_expect_tx_warp(bar(L::bKv), (2u + L::kPanels) * L::kKvPanel);
#pragma unroll
  for (int pn = 0; pn < 2; ++pn)
    tma_load_4d_warp(sbase + L::kK + pn * L::kKvPanel, tm_k, bar(L::bKv), D == 128 ? pn * 64 : 0, wk.g, wk.k0,
                     wk.b);
#pragma unroll
  for (int pn = 0; pn < L::kPanels; ++pn)
    tma_load_4d_warp(sbase + L::kV + pn * L::kKvPanel, tm_v, bar(L::bKv), pn * 64, wk.g, wk.k0, wk.b);
  const int per_head = wk.n_qb - wk.qb0;
  bool ok = true;
  int n = 0;   // stages issued
  for (int s = 0; s < wk.steps; ++s) {
    const int h = wk.g * p.group + s / per_head;
    const int qb = bwd_q64_qb(wk, p, s);
    const int st = s % L::kStages;
    const uint32_t stg = sbase + L::stage(s);
    if (s >= L::kStages &&
        !(ok = w.wait_warp(bar(L::bEmpty + st), static_cast<uint32_t>(s / L::kStages - 1) & 1u,
                           L::bEmpty + st)))
      break;
    mbar_arrive_expect_tx_warp(bar(L::bFull + st), L::kStageBytes + 512u);
#pragma unroll
    for (int pn = 0; pn < L::kPanels; ++pn) {
      tma_load_4d_warp(stg + L::kDO + pn * L::kQPanel, tm_do, bar(L::bFull + st), pn * 64, h, qb * 64, wk.b);
      tma_load_4d_warp(stg + L::kQ + pn * L::kQPanel, tm_q, bar(L::bFull + st), pn * 64, h, qb * 64, wk.b);
    }
    const int64_t row0 = (static_cast<int64_t>(wk.b) * p.Hq + h) * p.Sq_pad + qb * 64;
    bulk_load_warp(sbase + L::lse(s), p.lse2 + row0, 256u, bar(L::bFull + st));
    bulk_load_warp(sbase + L::delta(s), p.delta + row0, 256u, bar(L::bFull + st));
    ++n;
  }
  if (__any_sync(0xffffffffu, !ok || *w.abort)) {
    // Let the copies this warp started land before the CTA exits.
    w.drain_warp(bar(L::bKv), 0u, L::bKv);
    for (int t = max(0, n - L::kStages); t < n; ++t)
      w.drain_warp(bar(L::bFull + t % L::kStages), static_cast<uint32_t>(t / L::kStages) & 1u,
                   L::bFull + t % L::kStages);
  }
}

// ------------------------------------------------------------ MMA warp
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_q64_mma_role(uint32_t sbase, uint32_t tmem, const BwdParams& p,
                                                 const Waiter& w) {
  using L = BwdQ64Smem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_q64_work<CAUSAL>(p, bwd_q64_work_id<D>(sbase));
  if (wk.steps == 0) return;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);   // S^T, dP^T
  constexpr uint32_t kIdescTs = idesc_bf16_f32(128, D, false, true);    // dV, dK
  constexpr uint32_t kIdescDq = idesc_bf16_f32(128, 64, true, true);    // dQ^T: A, B MN-major
  constexpr uint32_t kHi = desc_hi_sw128(1024);
  const uint32_t k_lo = desc_lo_sw128(sbase + L::kK, 16), v_lo = desc_lo_sw128(sbase + L::kV, 16);
  // K^T as an MN-major A operand: M = head dim over the two 64-column panels
  const uint32_t k_mn = desc_lo_sw128(sbase + L::kK, L::kKvPanel);
  // dS as an MN-major B operand: N = the step's 64 queries (one swizzle row)
  const uint32_t ds_mn = desc_lo_sw128(sbase + L::kDS, L::kKvPanel);
  // S^T = K Q^T or dP^T = V dO^T of step s into buffer s % 2, then a commit
  // to that product's barrier
  auto issue_kq = [&](int s, uint32_t a_lo, int col, int opnd, int done) {
    const uint32_t b_lo = desc_lo_sw128(sbase + L::stage(s) + opnd, 16);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t a_off = ((kk >> 2) * L::kKvPanel + (kk & 3) * 32) >> 4;
      const uint32_t b_off = ((kk >> 2) * L::kQPanel + (kk & 3) * 32) >> 4;
      mma_ss_lohi_warp(tmem + col + 64 * (s & 1), a_lo + a_off, kHi, b_lo + b_off, kHi, kIdescS,
                       kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(bar(done + (s & 1)));
  };
  bool ok = w.wait_warp(bar(L::bKv), 0u, L::bKv);
  for (int s = 0; ok && s < 2 && s < wk.steps; ++s) {
    if (!(ok = w.wait_warp(bar(L::bFull + s), 0u, L::bFull + s))) break;
    tc_fence_after_sync();
    issue_kq(s, k_lo, L::kColS, L::kQ, L::bS);
    issue_kq(s, v_lo, L::kColDP, L::kDO, L::bDP);
  }
  for (int s = 0; ok && s < wk.steps; ++s) {
    const int b = s & 1;
    const int st = s % L::kStages;
    if (!(ok = w.wait_warp(bar(L::bPReady), static_cast<uint32_t>(s) & 1u, L::bPReady))) break;
    tc_fence_after_sync();
    // dQ^T = K^T dS^T over the step's dP^T columns, 16 keys per MMA
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lohi_warp(tmem + L::kColDP + 64 * b, k_mn + kk * (2048 >> 4), kHi, ds_mn + kk * (2048 >> 4),
                       kHi, kIdescDq, kk > 0 ? 1u : 0u);
    mma_commit_warp(bar(L::bDqFull));
    // dV += P^T dO and dK += dS^T Q, 16 queries (8 TMEM columns of packed
    // BF16, 2 KB of the MN-major operand) per MMA
    const uint32_t q_mn = desc_lo_sw128(sbase + L::stage(s) + L::kQ, L::kQPanel);
    const uint32_t do_mn = desc_lo_sw128(sbase + L::stage(s) + L::kDO, L::kQPanel);
    const uint32_t pcol = tmem + L::kColS + 64 * b;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ts_lohi_warp(tmem + L::kColDV, pcol + 32 * (kk >> 1) + 8 * (kk & 1), do_mn + kk * (2048 >> 4), kHi,
                       kIdescTs, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ts_lohi_warp(tmem + L::kColDK, pcol + 32 * (kk >> 1) + 16 + 8 * (kk & 1), q_mn + kk * (2048 >> 4),
                       kHi, kIdescTs, (s > 0 || kk > 0) ? 1u : 0u);
    mma_commit_warp(bar(L::bEmpty + st));   // the stage's Q and dO read
    // Step s + 2 reuses this step's columns: S^T at once (dV and dK, issued
    // above, execute first and read P^T and dS^T there), dP^T once the
    // read-out warps have read dQ^T. Waiting for the read-out on every step
    // (the last two too) also keeps dq_full from completing a second phase
    // before those warps have seen the first.
    const bool next = s + 2 < wk.steps;
    if (next) {
      const int st2 = (s + 2) % L::kStages;
      if (!(ok = w.wait_warp(bar(L::bFull + st2), static_cast<uint32_t>((s + 2) / L::kStages) & 1u,
                             L::bFull + st2)))
        break;
      tc_fence_after_sync();
      issue_kq(s + 2, k_lo, L::kColS, L::kQ, L::bS);
    }
    if (!(ok = w.wait_warp(bar(L::bDqFree), static_cast<uint32_t>(s) & 1u, L::bDqFree))) break;
    if (next) {
      tc_fence_after_sync();
      issue_kq(s + 2, v_lo, L::kColDP, L::kDO, L::bDP);
    }
  }
  // Every MMA issued above has completed once this commit arrives (the
  // epilogue waits for it; on abort it is the drain).
  mma_commit_warp(bar(L::bAcc));
  w.drain_warp(bar(L::bAcc), 0u, L::bAcc);
}

// ------------------------------------------------------------ compute warps
// p = 2^(c s - LSE2) for one thread's 32 entries (pairs on FFMA2); with MASK,
// 0 for a key row past Sk and for entries e < lim (above the causal
// diagonal).
template <bool MASK>
__device__ __forceinline__ void bwd_q64_p(const uint32_t (&sv)[32], const float4* lse4, float c2,
                                          bool row_live, int lim, float (&pv)[32]) {
  const float2 c22 = make_float2(c2, c2);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 l4 = lse4[e4];
    const float2 nl[2] = {make_float2(-l4.x, -l4.y), make_float2(-l4.z, -l4.w)};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = 4 * e4 + 2 * u;
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c22, nl[u]);
      float a = ex2_mufu(x.x), bb = ex2_mufu(x.y);
      if (MASK) {
        if (!row_live || e < lim) a = 0.0f;
        if (!row_live || e + 1 < lim) bb = 0.0f;
      }
      pv[e] = a;
      pv[e + 1] = bb;
    }
  }
}

// Warp w owns key rows 32 (w % 4) .. + 31 (its TMEM lane quarter) and
// queries 32 (w / 4) .. + 31 of each step. At the end it writes half of the
// columns of its rows of dK and dV.
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_q64_compute_role(uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                                     const BwdParams& p, const Waiter& w) {
  using L = BwdQ64Smem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3, ch = warp >> 2;
  const int r = wq * 32 + lane;                         // key row = dQ^T head-dim row = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const BwdWork wk = bwd_q64_work<CAUSAL>(p, bwd_q64_work_id<D>(sbase));
  const int kabs = wk.k0 + r;
  const float c2 = p.scale_log2;
  const int shift = p.Sk - p.Sq;
  const int per_head = wk.n_qb - wk.qb0;
  const bool row_live = kabs < p.Sk;
  const bool rows_live = wk.k0 + 128 <= p.Sk;          // every key row of the block exists
  bool ok = true;
  if (p.test_stall_cycles > 0)   // diagnostic: a wait nothing ends
    ok = w.wait_for(bar(L::bStall), 0u, L::bStall, p.test_stall_cycles);
  for (int s = 0; ok && s < wk.steps; ++s) {
    const int b = s & 1;
    const int st = s % L::kStages;
    const int q0 = bwd_q64_qb(wk, p, s) * 64;
    const float4* lse4 = reinterpret_cast<const float4*>(smem + L::lse(s)) + 8 * ch;
    const float4* delta4 = reinterpret_cast<const float4*>(smem + L::delta(s)) + 8 * ch;
    if (!(ok = w.wait(bar(L::bFull + st), static_cast<uint32_t>(s / L::kStages) & 1u, L::bFull + st)))
      break;
    if (!(ok = w.wait(bar(L::bS + b), static_cast<uint32_t>(s >> 1) & 1u, L::bS + b))) break;
    tc_fence_after_sync();
    const uint32_t scol = lane_base + L::kColS + 64 * b + 32 * ch;
    const uint32_t dcol = lane_base + L::kColDP + 64 * b + 32 * ch;
    uint32_t sv[32];
    tmem_ld_x32(scol, sv);
    tmem_wait_ld_x32(sv);
    // P = 2^(c S - LSE2) while dP^T is still being formed; masked entries
    // (keys past Sk, and above the causal diagonal) only on tiles that have
    // any, which is tile-uniform
    float pv[32];
    const bool masked = !rows_live || (CAUSAL && wk.k0 + 127 > q0 + shift);
    if (masked)
      bwd_q64_p<true>(sv, lse4, c2, row_live, CAUSAL ? kabs - shift - q0 - 32 * ch : -1, pv);
    else
      bwd_q64_p<false>(sv, lse4, c2, true, 0, pv);
    uint32_t pk[16], dk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
    // P^T into the first 16 of this warp's own (already read) S^T columns
    tmem_st_x16(scol, pk);
    if (!(ok = w.wait(bar(L::bDP + b), static_cast<uint32_t>(s >> 1) & 1u, L::bDP + b))) break;
    tc_fence_after_sync();
    uint32_t dv[32];
    tmem_ld_x32(dcol, dv);
    tmem_wait_ld_x32(dv);
    // dS = P (dP - Delta) on paired FP32 instructions
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
      const float4 d4 = delta4[e4];
      const float2 nd[2] = {make_float2(-d4.x, -d4.y), make_float2(-d4.z, -d4.w)};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = 4 * e4 + 2 * u;
        const float2 t = __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd[u]);
        const float2 de = __fmul2_rn(make_float2(pv[e], pv[e + 1]), t);
        dk[2 * e4 + u] = pack_bf16x2(de.x, de.y);
      }
    }
    // dS^T into the other 16
    tmem_st_x16(scol + 16, dk);
    // dS for the dQ^T MMA: row = key, the step's 64 queries in one 128-byte
    // swizzle row (16-byte chunk index XOR row within its 8-row group), once
    // the previous step's dQ^T MMA has read the tile
    if (s > 0 && !(ok = w.wait(bar(L::bDqFull), static_cast<uint32_t>(s - 1) & 1u, L::bDqFull))) break;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int chunk = 4 * ch + u;
      const uint32_t addr = sbase + L::kDS + r * 128 + (static_cast<uint32_t>(chunk ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk[4 * u]),
                   "r"(dk[4 * u + 1]), "r"(dk[4 * u + 2]), "r"(dk[4 * u + 3])
                   : "memory");
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before_sync();
    mbar_arrive(bar(L::bPReady));
  }
  // ---- epilogue: this warp's half of dV and scale * dK -> BF16 -> global
  const int64_t orow = (static_cast<int64_t>(wk.b) * p.Sk + kabs) * p.Hkv + wk.g;
  __nv_bfloat16* dv_row = p.dv + orow * D + ch * (D / 2);
  __nv_bfloat16* dk_row = p.dk + orow * D + ch * (D / 2);
  if (ok && wk.steps > 0) {
    if (!w.wait(bar(L::bAcc), 0u, L::bAcc)) return;
    tc_fence_after_sync();
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
      uint32_t x[32], y[32];
      tmem_ld_x32(lane_base + L::kColDV + ch * (D / 2) + 32 * c, x);
      tmem_ld_x32(lane_base + L::kColDK + ch * (D / 2) + 32 * c, y);
      tmem_wait_ld_x32(x);
      tmem_wait_ld_x32(y);
      if (row_live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 a, bb;
          a.x = pack_bf16x2(__uint_as_float(x[8 * i + 0]), __uint_as_float(x[8 * i + 1]));
          a.y = pack_bf16x2(__uint_as_float(x[8 * i + 2]), __uint_as_float(x[8 * i + 3]));
          a.z = pack_bf16x2(__uint_as_float(x[8 * i + 4]), __uint_as_float(x[8 * i + 5]));
          a.w = pack_bf16x2(__uint_as_float(x[8 * i + 6]), __uint_as_float(x[8 * i + 7]));
          bb.x = pack_bf16x2(__uint_as_float(y[8 * i + 0]) * p.scale, __uint_as_float(y[8 * i + 1]) * p.scale);
          bb.y = pack_bf16x2(__uint_as_float(y[8 * i + 2]) * p.scale, __uint_as_float(y[8 * i + 3]) * p.scale);
          bb.z = pack_bf16x2(__uint_as_float(y[8 * i + 4]) * p.scale, __uint_as_float(y[8 * i + 5]) * p.scale);
          bb.w = pack_bf16x2(__uint_as_float(y[8 * i + 6]) * p.scale, __uint_as_float(y[8 * i + 7]) * p.scale);
          reinterpret_cast<uint4*>(dv_row + c * 32)[i] = a;
          reinterpret_cast<uint4*>(dk_row + c * 32)[i] = bb;
        }
      }
    }
  } else if (ok && row_live) {
    // no query reads this key block: zero gradients
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      reinterpret_cast<uint4*>(dv_row)[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(dk_row)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ------------------------------------------------------------ dQ^T read-out warps
// Warp 12 + i reads TMEM lane quarter i of each step's dQ^T, frees the
// columns for the step after next, and stages scale * dQ in a ring slot,
// row = query, in the 32-column block of its head-dim rows: for each query
// the warp's 32 lanes fill one 128-byte row.
// Head dim 128: lanes = head-dim rows 32 i .. + 31, all 64 queries, staged in
// two units of 32 queries. Head dim 64: lanes 64..127 repeat rows 0..63, so
// warp i takes head-dim rows 32 (i % 2) .. + 31 of queries 32 (i / 2) .. + 31,
// and the step is one unit.
template <int D>
__device__ __forceinline__ void bwd_q64_dq_role(uint32_t sbase, uint32_t tmem, int steps,
                                                const BwdParams& p, const Waiter& w) {
  using L = BwdQ64Smem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int wq = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  constexpr int kCols = D == 128 ? 64 : 32;             // queries this warp reads per step
  const int dblk = D == 128 ? wq : (wq & 1);            // 32-column block of dQ
  const int q_first = D == 128 ? 0 : 32 * (wq >> 1);    // first query it reads
  const uint32_t blk = sbase + L::kStg + dblk * L::kSlotBlock + ((lane & 3) << 2);
  for (int s = 0; s < steps; ++s) {
    if (!w.wait(bar(L::bDqFull), static_cast<uint32_t>(s) & 1u, L::bDqFull)) return;
    tc_fence_after_sync();
    uint32_t x[kCols];
    const uint32_t col = lane_base + L::kColDP + 64 * (s & 1) + q_first;
#pragma unroll
    for (int c = 0; c < kCols / 32; ++c) tmem_ld_x32(col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
#pragma unroll
    for (int c = 0; c < kCols / 32; ++c) tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
    tc_fence_before_sync();
    mbar_arrive(bar(L::bDqFree));
#pragma unroll
    for (int hh = 0; hh < L::kUnits; ++hh) {
      const int u = L::kUnits * s + hh;                 // staged unit number
      const int slot = u % L::kSlots;
      if (u >= L::kSlots &&
          !w.wait(bar(L::bSlotFree + slot), static_cast<uint32_t>(u / L::kSlots - 1) & 1u, L::bSlotFree + slot))
        return;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int row = (D == 128 ? 0 : q_first) + j;   // query row within the unit
        const uint32_t addr = blk + slot * L::kSlotBytes + row * 128 +
                              (static_cast<uint32_t>((lane >> 2) ^ (row & 7)) << 4);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(__uint_as_float(x[32 * hh + j]) * p.scale)
                     : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::bSlotFull + slot));
    }
  }
}

// ------------------------------------------------------------ dQ flush warp
// Adds each staged unit (32 queries x 128 columns at head dim 128, 64 x 64
// at 64) to the global fp32 accumulator with one bulk tensor reduce-add per
// 32 columns (rows past Sq are outside the tensor and skipped). Up to two
// units are in flight: a slot is handed back once the reduce-add issued
// after it has been issued and its own source has been read. In
// deterministic mode the lane first waits for its turn on the 64-query
// block's counter and, once the step's last unit has completed, passes the
// turn on.
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_q64_flush_role(const CUtensorMap* tm_dq, uint32_t sbase,
                                                   const BwdParams& p, const Waiter& w) {
  using L = BwdQ64Smem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_q64_work<CAUSAL>(p, bwd_q64_work_id<D>(sbase));
  const int per_head = wk.n_qb - wk.qb0;
  const int lane = threadIdx.x & 31;
  const int kb = wk.k0 / 128;
  bool ok = true;
  for (int u = 0; u < L::kUnits * wk.steps; ++u) {
    const int s = u / L::kUnits, hh = u % L::kUnits;
    const int h = wk.g * p.group + s / per_head;
    const int qb = bwd_q64_qb(wk, p, s);
    const int slot = u % L::kSlots;
    if (!(ok = w.wait(bar(L::bSlotFull + slot), static_cast<uint32_t>(u / L::kSlots) & 1u, L::bSlotFull + slot)))
      break;
    if (lane == 0) {
      int* turn = p.dq_turn ? p.dq_turn + (static_cast<int64_t>(wk.b) * p.Hq + h) * wk.n_qb + qb : nullptr;
      if (turn && hh == 0) {
        // every earlier key block reads this query block (visibility grows
        // with the key index), so the turn of key block kb comes after kb adds
        const long long t0 = clock64();
        while (true) {
          int cur;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cur) : "l"(turn) : "memory");
          if (cur >= kb) break;
          if (*w.abort || clock64() - t0 > kWaitLimitCycles) {
            if (!*w.abort) {
              *w.abort = 1;
              if (atomicCAS(p.status, 0u, kStatusTimeout) == 0u) {
                p.status[1] = kRoleFlush;
                p.status[2] = L::bSlotFull + slot;
                p.status[3] = blockIdx.x;
              }
            }
            ok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      if (ok) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tma_reduce_add_4d(tm_dq, sbase + L::kStg + slot * L::kSlotBytes + c * L::kSlotBlock, 32 * c, h,
                            qb * 64 + L::kUnitRows * hh, wk.b);
        bulk_commit_group();
        if (turn && hh == L::kUnits - 1) {
          bulk_wait_group0();                         // both halves' adds are done in global memory
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(turn, 1);
        } else {
          bulk_wait_group_read<1>();                  // the half-tile before this one has been read
        }
        if (u > 0) mbar_arrive(bar(L::bSlotFree + (u - 1) % L::kSlots));
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;
  }
  // the accumulator must hold every reduce before the CTA exits
  if (lane == 0) bulk_wait_group0();
}

// ------------------------------------------------------------ kernel
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdQ64Threads, 1)
    fa4_bwd_q64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using L = BwdQ64Smem<D>;
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
    *reinterpret_cast<volatile int*>(smem + L::kMisc + 8) =
        p.cta_ticket ? atomicAdd(p.cta_ticket, 1) : static_cast<int>(blockIdx.x);
    mbar_init(bar(L::bKv), 1);
    for (int i = 0; i < L::kStages; ++i) {
      mbar_init(bar(L::bFull + i), 1);
      mbar_init(bar(L::bEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bS + i), 1);
      mbar_init(bar(L::bDP + i), 1);
    }
    mbar_init(bar(L::bPReady), 256);
    mbar_init(bar(L::bDqFull), 1);
    mbar_init(bar(L::bDqFree), 128);
    mbar_init(bar(L::bAcc), 1);
    mbar_init(bar(L::bStall), 1);
    for (int i = 0; i < L::kSlots; ++i) {
      mbar_init(bar(L::bSlotFull + i), 128);
      mbar_init(bar(L::bSlotFree + i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kBwdWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Register split (setmaxnreg): 256 compute threads, 128 load / MMA /
  // flush, 128 dQ^T read-out; the total must equal the 512 x 128 the block
  // launches with.
  constexpr int kRegsCompute = 160, kRegsIssue = 88, kRegsDq = 104;
  static_assert(256 * kRegsCompute + 128 * kRegsIssue + 128 * kRegsDq == kBwdQ64Threads * 128,
                "register split must use exactly the launch allocation");
  if (warp < 8) {
    regs_increase<kRegsCompute>();
    const Waiter w{abort_flag, p.status, kRoleSoftmax};
    bwd_q64_compute_role<D, CAUSAL>(sbase, smem, tmem, p, w);
  } else if (warp < kBwdQ64WarpDq) {
    regs_decrease<kRegsIssue>();
    if (warp == kBwdWarpLoad) {
      const Waiter w{abort_flag, p.status, kRoleLoad};
      bwd_q64_load_role<D, CAUSAL>(&tm_q, &tm_k, &tm_v, &tm_do, sbase, p, w);
    } else if (warp == kBwdWarpMma) {
      const Waiter w{abort_flag, p.status, kRoleMma};
      bwd_q64_mma_role<D, CAUSAL>(sbase, tmem, p, w);
    } else if (warp == kBwdWarpFlush) {
      const Waiter w{abort_flag, p.status, kRoleFlush};
      bwd_q64_flush_role<D, CAUSAL>(&tm_dq, sbase, p, w);
    }
  } else {
    regs_decrease<kRegsDq>();
    const Waiter w{abort_flag, p.status, kRoleDqRead};
    bwd_q64_dq_role<D>(sbase, tmem, bwd_q64_work<CAUSAL>(p, bwd_q64_work_id<D>(sbase)).steps, p, w);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa4
