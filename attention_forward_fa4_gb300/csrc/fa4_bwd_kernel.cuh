// fa4_bwd_kernel.cuh -- attention backward on sm_103a: dQ, dK, dV from Q,
// K, V, dO and the forward's logsumexp, with tcgen05 MMAs into tensor
// memory ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", §3.2: five MMAs per tile pair).
//
// One CTA owns a 128-key block of one (batch, kv head) and walks every
// query block of every query head that reads it. Per step (128 queries x
// 128 keys), with rows of the transposed products on TMEM lanes = keys:
//
//   S^T  = K Q^T            SS MMA          TMEM cols [0, 128)
//   dP^T = V dO^T           SS MMA          TMEM cols [128, 256)
//   P^T  = 2^(c S^T - LSE2) (compute warps, one key row per thread and
//                           half the queries per warp; masked 0)
//   dS^T = P^T o (dP^T - Delta)
//   dV  += P^T dO           TS MMA, A = P^T from TMEM (BF16 over S^T: the
//                           32 queries of each 32-column chunk in its first
//                           16 columns)
//   dK  += dS^T Q           TS MMA, A = dS^T from TMEM (BF16 over dP^T, same)
//   dQ   = dS K             SS MMA, A = dS from shared memory (MN-major,
//                           written by the compute threads), into cols
//                           [0, D) over S^T; read out, staged in shared
//                           memory and added to the global fp32 dQ
//                           accumulator with bulk tensor reduce-adds.
//
// dK and dV accumulate in TMEM (cols [256, 256 + 2D)) over all steps and
// are written once at the end; the GQA group's query heads all pass through
// the CTA, so kv-head gradients need no atomics. Delta_i = sum_e dO O and
// LSE2 = LSE log2(e) (+inf for rows that must contribute nothing) come from
// a preprocessing kernel, padded to whole 128-row blocks.
//
// Warps: 0-7 softmax-side work, dQ read-out and staging, and the dK/dV
// epilogue (two warps per TMEM lane quarter, each on half of the columns);
// 8 TMA loads, 9 MMA issue (both warp-wide with an elected lane); 10 dQ
// flush (bulk reduce-adds; in deterministic mode in key-block order); 11
// idle. Every wait is bounded (Waiter), as in the forward kernel.
#pragma once

#include "fa4_fwd_kernel.cuh"

namespace fa4 {

constexpr int kBwdThreads = 384;
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
  // Deterministic mode (non-null): one int per (batch, query head, query
  // block), zeroed; the dQ tile of key block kb is added only once kb
  // earlier key blocks have added theirs, so the fp32 sums are formed in
  // the same order on every run. CTAs are then numbered key block first.
  int* dq_turn;
  // Deterministic mode: a zeroed counter from which each CTA takes its work
  // number when it starts, so every lower number belongs to a CTA that is
  // already running whatever order the hardware dispatched them in.
  int* cta_ticket;
};

// Q, dO, LSE2 and Delta of a step sit in one of kStages stages (two at
// d = 64, so the next step's copies land while the current step computes;
// one at d = 128, where the space goes to the dQ staging tile). The dQ
// staging tile holds a step's fp32 dQ in 32-column, 128-byte-swizzled
// blocks for the bulk reduce-add into the global accumulator.
template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kPanelBytes = 128 * 128;
  static constexpr int kPanels = D / 64;
  static constexpr int kStages = D == 128 ? 1 : 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kDS = kV + kTileBytes;           // 128 x 128 BF16, two MN-major panels
  static constexpr int kDqStage = kDS + 2 * kPanelBytes;  // (D / 32) x [128 rows x 32 fp32]
  static constexpr int kStage = kDqStage + 128 * D * 4;   // kStages x {Q, dO, LSE2, Delta}
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kQ = 0, kDO = kTileBytes, kLse = 2 * kTileBytes, kDelta = kLse + 512;
  static constexpr int kBars = kStage + kStages * kStageBytes;
  // barriers: kv; per stage Q full / empty and dO (with LSE2, Delta) full /
  // empty -- dO is released after the dV MMA, Q only after dK, so the next
  // step's dO arrives first; sdp, p_ready, dq_full, dq_free, acc, stg (the
  // compute warps' rendezvous around the dQ staging tile)
  static constexpr int bKv = 0, bQ = 1, bDO = 3, bQEmpty = 5, bDOEmpty = 7, bSdp = 9, bPReady = 10,
                       bDqFull = 11, bDqFree = 12, bAcc = 13, bStgFull = 14, bStgFree = 15,
                       kNumBars = 16;
  static constexpr int kMisc = kBars + kNumBars * 8;    // tmem base, abort flag, work number
  static constexpr int kBytes = kMisc + 16;
  // 1 KB of slack re-aligns the base to the 128-byte swizzle's 1 KB period;
  // when it does not fit (d = 128) the kernel requires an aligned base.
  static constexpr int kSlack = (kBytes + 1024 <= 232448) ? 1024 : 0;
  static constexpr int kAlloc = kBytes + kSlack;
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr int stage(int s) { return kStage + (s % kStages) * kStageBytes; }
};

// The CTA's key block and the query blocks it visits.
struct BwdWork {
  int b, g, k0;
  int qb0, n_qb;      // query blocks [qb0, n_qb) of every head in the group
  int steps;          // group * (n_qb - qb0)
};

// The CTA's work number, stored in shared memory by the kernel prologue.
template <int D>
__device__ __forceinline__ int bwd_work_id(uint32_t sbase) {
  int id;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(id) : "r"(sbase + BwdSmem<D>::kMisc + 8) : "memory");
  return id;
}

template <bool CAUSAL>
__device__ __forceinline__ BwdWork bwd_work(const BwdParams& p, int id) {
  BwdWork w;
  // Key blocks of one (batch, kv head) side by side (their CTAs share Q and
  // dO in L2); in deterministic mode key block first, with work numbers
  // taken in start order, so every CTA whose turn comes earlier is already
  // running.
  const int n_bg = p.B * p.Hkv;
  const int kb = p.dq_turn ? id / n_bg : id % p.n_kblk;
  const int bg = p.dq_turn ? id % n_bg : id / p.n_kblk;
  w.b = bg / p.Hkv;
  w.g = bg - w.b * p.Hkv;
  w.k0 = kb * 128;
  w.n_qb = (p.Sq + 127) / 128;
  w.qb0 = 0;
  if (CAUSAL) {
    // the first query that sees key k0: i >= k0 - (Sk - Sq)
    const long long i_min = static_cast<long long>(w.k0) - (p.Sk - p.Sq);
    w.qb0 = i_min <= 0 ? 0 : static_cast<int>(i_min / 128 < w.n_qb ? i_min / 128 : w.n_qb);
  }
  w.steps = p.group * (w.n_qb - w.qb0);
  return w;
}

// ------------------------------------------------------------ load warp
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                              uint32_t sbase, const BwdParams& p, const Waiter& w) {
  using L = BwdSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_work<CAUSAL>(p, bwd_work_id<D>(sbase));
  if (wk.steps == 0) return;
  mbar_arrive_expect_tx_warp(bar(L::bKv), 2u * L::kTileBytes);
#pragma unroll
  for (int pn = 0; pn < L::kPanels; ++pn) {
    tma_load_4d_warp(sbase + L::kK + pn * L::kPanelBytes, tm_k, bar(L::bKv), pn * 64, wk.g, wk.k0, wk.b);
    tma_load_4d_warp(sbase + L::kV + pn * L::kPanelBytes, tm_v, bar(L::bKv), pn * 64, wk.g, wk.k0, wk.b);
  }
  const int per_head = wk.n_qb - wk.qb0;
  bool ok = true;
  int n_do = 0, n_q = 0;        // dO and Q copies issued
  for (int s = 0; s < wk.steps; ++s) {
    const int h = wk.g * p.group + s / per_head;
    const int qb = wk.qb0 + s % per_head;
    const int st = s % L::kStages;
    const uint32_t stg = sbase + L::stage(s);
    const uint32_t par = static_cast<uint32_t>(s / L::kStages - 1) & 1u;
    // dO, LSE2 and Delta of step s, once the stage's previous step
    // (s - kStages) has finished its dV MMA -- with two stages, its dK MMA
    // too (both copies then go out together: measured faster at d = 64)
    const int do_free = L::kStages == 1 ? L::bDOEmpty + st : L::bQEmpty + st;
    if (s >= L::kStages && !(ok = w.wait_warp(bar(do_free), par, do_free))) break;
    mbar_arrive_expect_tx_warp(bar(L::bDO + st), L::kTileBytes + 1024u);
#pragma unroll
    for (int pn = 0; pn < L::kPanels; ++pn)
      tma_load_4d_warp(stg + L::kDO + pn * L::kPanelBytes, tm_do, bar(L::bDO + st), pn * 64, h, qb * 128,
                       wk.b);
    const int64_t row0 = (static_cast<int64_t>(wk.b) * p.Hq + h) * p.Sq_pad + qb * 128;
    bulk_load_warp(stg + L::kLse, p.lse2 + row0, 512u, bar(L::bDO + st));
    bulk_load_warp(stg + L::kDelta, p.delta + row0, 512u, bar(L::bDO + st));
    ++n_do;
    // Q of step s, once that step has finished its dK MMA
    if (L::kStages == 1 && s >= L::kStages && !(ok = w.wait_warp(bar(L::bQEmpty + st), par, L::bQEmpty + st)))
      break;
    mbar_arrive_expect_tx_warp(bar(L::bQ + st), L::kTileBytes);
#pragma unroll
    for (int pn = 0; pn < L::kPanels; ++pn)
      tma_load_4d_warp(stg + L::kQ + pn * L::kPanelBytes, tm_q, bar(L::bQ + st), pn * 64, h, qb * 128, wk.b);
    ++n_q;
  }
  if (__any_sync(0xffffffffu, !ok || *w.abort)) {
    // Let the copies this warp started land before the CTA exits.
    w.drain_warp(bar(L::bKv), 0u, L::bKv);
    for (int t = max(0, n_do - L::kStages); t < n_do; ++t)
      w.drain_warp(bar(L::bDO + t % L::kStages), static_cast<uint32_t>(t / L::kStages) & 1u,
                   L::bDO + t % L::kStages);
    for (int t = max(0, n_q - L::kStages); t < n_q; ++t)
      w.drain_warp(bar(L::bQ + t % L::kStages), static_cast<uint32_t>(t / L::kStages) & 1u,
                   L::bQ + t % L::kStages);
  }
}

// ------------------------------------------------------------ MMA warp
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_mma_role(uint32_t sbase, uint32_t tmem, const BwdParams& p,
                                             const Waiter& w) {
  using L = BwdSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_work<CAUSAL>(p, bwd_work_id<D>(sbase));
  if (wk.steps == 0) return;
  constexpr uint32_t kIdescKmaj = idesc_bf16_f32(128, 128, false, false);   // S^T, dP^T
  constexpr uint32_t kIdescTs = idesc_bf16_f32(128, D, false, true);        // dV, dK
  constexpr uint32_t kIdescDq = idesc_bf16_f32(128, D, true, true);         // dQ: A, B MN-major
  constexpr uint32_t kHi = desc_hi_sw128(1024);
  // K-major views (LBO unused) and MN-major views (LBO = 64-column panel stride).
  const uint32_t k_lo = desc_lo_sw128(sbase + L::kK, 16), v_lo = desc_lo_sw128(sbase + L::kV, 16);
  const uint32_t k_mn = desc_lo_sw128(sbase + L::kK, L::kPanelBytes);
  constexpr uint32_t kStageStep = L::kStageBytes >> 4;   // descriptor units between stages
  const uint32_t ds_mn = desc_lo_sw128(sbase + L::kDS, L::kPanelBytes);
  bool ok = w.wait_warp(bar(L::bKv), 0u, L::bKv);
  tc_fence_after_sync();
  for (int s = 0; ok && s < wk.steps; ++s) {
    const int st = s % L::kStages;
    const uint32_t q_lo = desc_lo_sw128(sbase + L::stage(0) + L::kQ, 16) + st * kStageStep;
    const uint32_t do_lo = desc_lo_sw128(sbase + L::stage(0) + L::kDO, 16) + st * kStageStep;
    const uint32_t q_mn = desc_lo_sw128(sbase + L::stage(0) + L::kQ, L::kPanelBytes) + st * kStageStep;
    const uint32_t do_mn = desc_lo_sw128(sbase + L::stage(0) + L::kDO, L::kPanelBytes) + st * kStageStep;
    const uint32_t par = static_cast<uint32_t>(s / L::kStages) & 1u;
    // dP^T = V dO^T into columns that only the previous step's dK MMA
    // (issued before it) still reads, and S^T = K Q^T (keys on the M side,
    // queries on N) into columns the previous step's dQ has been read out of.
    auto issue_dp = [&]() {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * L::kPanelBytes + (kk & 3) * 32) >> 4;
        mma_ss_lohi_warp(tmem + L::kColDP, v_lo + off, kHi, do_lo + off, kHi, kIdescKmaj, kk > 0 ? 1u : 0u);
      }
    };
    if constexpr (L::kStages == 1) {
      // One Q/dO stage (d = 128): the next step's dO arrives while its Q is
      // still loading (dO is released after dV, Q after dK), so dP^T goes
      // first, ahead of the waits for Q and for the dQ read-out. Measured:
      // +11 % (long causal); with two stages (d = 64) this order lost 3 %.
      if (!(ok = w.wait_warp(bar(L::bDO + st), par, L::bDO + st))) break;
      tc_fence_after_sync();
      issue_dp();
    }
    if (!(ok = w.wait_warp(bar(L::bQ + st), par, L::bQ + st))) break;
    if (L::kStages > 1 && !(ok = w.wait_warp(bar(L::bDO + st), par, L::bDO + st))) break;
    if (s > 0 && !(ok = w.wait_warp(bar(L::bDqFree), static_cast<uint32_t>(s - 1) & 1u, L::bDqFree)))
      break;
    tc_fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * L::kPanelBytes + (kk & 3) * 32) >> 4;
      mma_ss_lohi_warp(tmem + L::kColS, k_lo + off, kHi, q_lo + off, kHi, kIdescKmaj, kk > 0 ? 1u : 0u);
    }
    if constexpr (L::kStages > 1) issue_dp();
    mma_commit_warp(bar(L::bSdp));
    if (!(ok = w.wait_warp(bar(L::bPReady), static_cast<uint32_t>(s) & 1u, L::bPReady))) break;
    tc_fence_after_sync();
    // dV += P^T dO and dK += dS^T Q: 16 queries (8 TMEM columns of packed
    // BF16 -- queries 32 j .. 32 j + 31 at columns 32 j .. 32 j + 15 -- and
    // 2 KB of the MN-major operand) per MMA
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_lohi_warp(tmem + L::kColDV, tmem + L::kColS + 32 * (kk >> 1) + 8 * (kk & 1),
                       do_mn + kk * (2048 >> 4), kHi, kIdescTs, (s > 0 || kk > 0) ? 1u : 0u);
    // dO of this stage read (with two stages the load warp waits for dK)
    if constexpr (L::kStages == 1) mma_commit_warp(bar(L::bDOEmpty + st));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_lohi_warp(tmem + L::kColDK, tmem + L::kColDP + 32 * (kk >> 1) + 8 * (kk & 1),
                       q_mn + kk * (2048 >> 4), kHi, kIdescTs, (s > 0 || kk > 0) ? 1u : 0u);
    mma_commit_warp(bar(L::bQEmpty + st));    // Q of this stage read
    // dQ = dS K over the S^T columns: issued after the dV MMA that reads
    // P^T there (one issuing thread's MMAs execute in order)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lohi_warp(tmem + L::kColS, ds_mn + kk * (2048 >> 4), kHi, k_mn + kk * (2048 >> 4), kHi, kIdescDq,
                       kk > 0 ? 1u : 0u);
    mma_commit_warp(bar(L::bDqFull));
  }
  // Every MMA issued above has completed once this commit arrives (the
  // epilogue waits for it; on abort it is the drain).
  mma_commit_warp(bar(L::bAcc));
  w.drain_warp(bar(L::bAcc), 0u, L::bAcc);
}

// ------------------------------------------------------------ compute warps
// Warps 0-7: warp w owns key rows 32 (w % 4) .. + 31 (its TMEM lane quarter)
// and query columns 64 (w / 4) .. + 63 of each step. Per step it forms P^T
// and dS^T for its 32 x 64 entries, then reads out its half of the step's
// dQ rows (lanes = queries, columns (w / 4) D/2 .. + D/2) and adds them to
// the global accumulator; at the end it writes its half of dK and dV.
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_compute_role(const CUtensorMap* tm_dq, uint32_t sbase,
                                                 uint8_t* smem, uint32_t tmem, const BwdParams& p,
                                                 const Waiter& w) {
  using L = BwdSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3, ch = warp >> 2;             // lane quarter, column half
  const int r = wq * 32 + lane;                         // key row (and dQ query row) = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const BwdWork wk = bwd_work<CAUSAL>(p, bwd_work_id<D>(sbase));
  const int kabs = wk.k0 + r;
  const float c2 = p.scale_log2;
  const int shift = p.Sk - p.Sq;
  const int per_head = wk.n_qb - wk.qb0;
  const bool row_live = kabs < p.Sk;
  bool ok = true;
  for (int s = 0; s < wk.steps; ++s) {
    const int h = wk.g * p.group + s / per_head;
    const int q0 = (wk.qb0 + s % per_head) * 128;
    const int st = s % L::kStages;
    const float4* lse4 = reinterpret_cast<const float4*>(smem + L::stage(s) + L::kLse);
    const float4* delta4 = reinterpret_cast<const float4*>(smem + L::stage(s) + L::kDelta);
    // LSE2 and Delta arrive with dO
    if (!(ok = w.wait(bar(L::bDO + st), static_cast<uint32_t>(s / L::kStages) & 1u, L::bDO + st)))
      break;
    if (!(ok = w.wait(bar(L::bSdp), static_cast<uint32_t>(s) & 1u, L::bSdp))) break;
    tc_fence_after_sync();
    // tile-uniform: every (key, query) pair of the step is visible
    const bool all_visible = !CAUSAL || (wk.k0 + 127 <= q0 + shift);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * ch + cc;                        // 32-query chunk of the step
      uint32_t sv[32], dv[32];
      tmem_ld_x32(lane_base + L::kColS + 32 * c, sv);
      tmem_ld_x32(lane_base + L::kColDP + 32 * c, dv);
      tmem_wait_ld_x32(sv);
      tmem_wait_ld_x32(dv);
      uint32_t pk[16], dk[16];
      // Pairs of entries on the paired FP32 instructions (FFMA2 / FADD2 /
      // FMUL2): p = 2^(c s - LSE2), dS = p (dP - Delta); masked entries 0.
      const float2 c22 = make_float2(c2, c2);
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 l4 = lse4[8 * c + e4];
        const float4 d4 = delta4[8 * c + e4];
        const float2 nl[2] = {make_float2(-l4.x, -l4.y), make_float2(-l4.z, -l4.w)};
        const float2 nd[2] = {make_float2(-d4.x, -d4.y), make_float2(-d4.z, -d4.w)};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = 4 * e4 + 2 * u;
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c22, nl[u]);
          float2 pv = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
          if (!row_live) pv = make_float2(0.0f, 0.0f);
          if (!all_visible) {
            const int lim = kabs - shift - q0 - 32 * c;   // entries e with e < lim are masked
            if (e < lim) pv.x = 0.0f;
            if (e + 1 < lim) pv.y = 0.0f;
          }
          const float2 t = __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd[u]);
          const float2 de = __fmul2_rn(pv, t);
          pk[2 * e4 + u] = pack_bf16x2(pv.x, pv.y);
          dk[2 * e4 + u] = pack_bf16x2(de.x, de.y);
        }
      }
      // P^T over S^T and dS^T over dP^T, in the first 16 of this chunk's own
      // 32 columns (already read; the other warp of the lane quarter works
      // on other columns): query q sits at column 32 (q / 32) + (q % 32) / 2
      tmem_st_x16(lane_base + L::kColS + 32 * c, pk);
      tmem_st_x16(lane_base + L::kColDP + 32 * c, dk);
      // dS for the dQ MMA: MN-major A tile, panel = 64 queries, row = key,
      // 128-byte swizzle (16-byte chunk index XOR row within its 8-row group)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int chunk = 4 * (c & 1) + u;
        const uint32_t addr = sbase + L::kDS + (c >> 1) * L::kPanelBytes + r * 128 +
                              (static_cast<uint32_t>(chunk ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk[4 * u]),
                     "r"(dk[4 * u + 1]), "r"(dk[4 * u + 2]), "r"(dk[4 * u + 3])
                     : "memory");
      }
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before_sync();
    mbar_arrive(bar(L::bPReady));
    // ---- this step's dQ: half of the columns of the lane quarter's rows
    if (!(ok = w.wait(bar(L::bDqFull), static_cast<uint32_t>(s) & 1u, L::bDqFull))) break;
    tc_fence_after_sync();
    constexpr int kHalf = D / 2;
    uint32_t x[kHalf];
#pragma unroll
    for (int c = 0; c < kHalf / 32; ++c)
      tmem_ld_x32(lane_base + L::kColS + ch * kHalf + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
#pragma unroll
    for (int c = 0; c < kHalf / 32; ++c) tmem_wait_ld_x32(*reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
    // dQ is in registers: the next step's S^T may overwrite its columns
    tc_fence_before_sync();
    mbar_arrive(bar(L::bDqFree));
    // Stage scale * dQ in shared memory once the flush warp has handed the
    // tile back from the previous step; the flush warp adds it to the
    // global accumulator.
    if (s > 0 && !(ok = w.wait(bar(L::bStgFree), static_cast<uint32_t>(s - 1) & 1u, L::bStgFree)))
      break;
#pragma unroll
    for (int cl = 0; cl < kHalf / 32; ++cl) {
      const int c = ch * (kHalf / 32) + cl;             // 32-column block of the D columns
      const uint32_t blk = sbase + L::kDqStage + c * 16384 + r * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t addr = blk + (static_cast<uint32_t>(j ^ (r & 7)) << 4);
        const int e = 32 * cl + 4 * j;
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                     "f"(__uint_as_float(x[e]) * p.scale), "f"(__uint_as_float(x[e + 1]) * p.scale),
                     "f"(__uint_as_float(x[e + 2]) * p.scale), "f"(__uint_as_float(x[e + 3]) * p.scale)
                     : "memory");
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(L::bStgFull));
  }
  // ---- epilogue: this warp's half of dV and scale * dK -> BF16 -> global
  constexpr int kHalf = D / 2;
  const int64_t orow = (static_cast<int64_t>(wk.b) * p.Sk + kabs) * p.Hkv + wk.g;
  __nv_bfloat16* dv_row = p.dv + orow * D + ch * kHalf;
  __nv_bfloat16* dk_row = p.dk + orow * D + ch * kHalf;
  if (ok && wk.steps > 0) {
    if (!w.wait(bar(L::bAcc), 0u, L::bAcc)) return;
    tc_fence_after_sync();
#pragma unroll 1
    for (int c = 0; c < kHalf / 32; ++c) {
      uint32_t x[32], y[32];
      tmem_ld_x32(lane_base + L::kColDV + ch * kHalf + 32 * c, x);
      tmem_ld_x32(lane_base + L::kColDK + ch * kHalf + 32 * c, y);
      tmem_wait_ld_x32(x);
      tmem_wait_ld_x32(y);
      if (row_live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 a, b;
          a.x = pack_bf16x2(__uint_as_float(x[8 * i + 0]), __uint_as_float(x[8 * i + 1]));
          a.y = pack_bf16x2(__uint_as_float(x[8 * i + 2]), __uint_as_float(x[8 * i + 3]));
          a.z = pack_bf16x2(__uint_as_float(x[8 * i + 4]), __uint_as_float(x[8 * i + 5]));
          a.w = pack_bf16x2(__uint_as_float(x[8 * i + 6]), __uint_as_float(x[8 * i + 7]));
          b.x = pack_bf16x2(__uint_as_float(y[8 * i + 0]) * p.scale, __uint_as_float(y[8 * i + 1]) * p.scale);
          b.y = pack_bf16x2(__uint_as_float(y[8 * i + 2]) * p.scale, __uint_as_float(y[8 * i + 3]) * p.scale);
          b.z = pack_bf16x2(__uint_as_float(y[8 * i + 4]) * p.scale, __uint_as_float(y[8 * i + 5]) * p.scale);
          b.w = pack_bf16x2(__uint_as_float(y[8 * i + 6]) * p.scale, __uint_as_float(y[8 * i + 7]) * p.scale);
          reinterpret_cast<uint4*>(dv_row + c * 32)[i] = a;
          reinterpret_cast<uint4*>(dk_row + c * 32)[i] = b;
        }
      }
    }
  } else if (ok && row_live) {
    // no query reads this key block: zero gradients
#pragma unroll
    for (int i = 0; i < kHalf / 8; ++i) {
      reinterpret_cast<uint4*>(dv_row)[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(dk_row)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ------------------------------------------------------------ dQ flush warp
// Adds each step's staged dQ tile to the global fp32 accumulator with one
// bulk tensor reduce-add per 32 columns (rows past Sq are outside the
// tensor and skipped), then hands the tile back once the copies have read
// it. In deterministic mode it first waits for its turn on the query
// block's counter and, after the reduce has completed, passes the turn on.
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_flush_role(const CUtensorMap* tm_dq, uint32_t sbase,
                                               const BwdParams& p, const Waiter& w) {
  using L = BwdSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const BwdWork wk = bwd_work<CAUSAL>(p, bwd_work_id<D>(sbase));
  const int per_head = wk.n_qb - wk.qb0;
  const int lane = threadIdx.x & 31;
  const int kb = wk.k0 / 128;
  bool ok = true;
  for (int s = 0; s < wk.steps; ++s) {
    const int h = wk.g * p.group + s / per_head;
    const int qb = wk.qb0 + s % per_head;
    if (!(ok = w.wait(bar(L::bStgFull), static_cast<uint32_t>(s) & 1u, L::bStgFull))) break;
    if (lane == 0) {
      int* turn = p.dq_turn ? p.dq_turn + (static_cast<int64_t>(wk.b) * p.Hq + h) * wk.n_qb + qb : nullptr;
      if (turn) {
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
                p.status[2] = L::bStgFull;
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
          tma_reduce_add_4d(tm_dq, sbase + L::kDqStage + c * 16384, 32 * c, h, qb * 128, wk.b);
        bulk_commit_group();
        if (turn) {
          bulk_wait_group0();                         // the adds are done in global memory
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(turn, 1);
        } else {
          bulk_wait_group_read0();                    // the tile may be rewritten
        }
      }
      mbar_arrive(bar(L::bStgFree));
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;
  }
  // the accumulator must hold every reduce before the CTA exits
  if (lane == 0) bulk_wait_group0();
}

// ------------------------------------------------------------ kernel
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa4_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  if (L::kSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
    // no room to re-align: refuse rather than touch memory past the allocation
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, kStatusMisalignedSmem);
    return;
  }
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bQ + i), 1);
      mbar_init(bar(L::bDO + i), 1);
      mbar_init(bar(L::bQEmpty + i), 1);
      mbar_init(bar(L::bDOEmpty + i), 1);
    }
    mbar_init(bar(L::bSdp), 1);
    mbar_init(bar(L::bPReady), 256);
    mbar_init(bar(L::bDqFull), 1);
    mbar_init(bar(L::bDqFree), 256);
    mbar_init(bar(L::bAcc), 1);
    mbar_init(bar(L::bStgFull), 256);
    mbar_init(bar(L::bStgFree), 1);
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

  if (warp < 8) {
    const Waiter w{abort_flag, p.status, kRoleSoftmax};
    bwd_compute_role<D, CAUSAL>(&tm_dq, sbase, smem, tmem, p, w);
  } else if (warp == kBwdWarpLoad) {
    const Waiter w{abort_flag, p.status, kRoleLoad};
    bwd_load_role<D, CAUSAL>(&tm_q, &tm_k, &tm_v, &tm_do, sbase, p, w);
  } else if (warp == kBwdWarpMma) {
    const Waiter w{abort_flag, p.status, kRoleMma};
    bwd_mma_role<D, CAUSAL>(sbase, tmem, p, w);
  } else if (warp == kBwdWarpFlush) {
    const Waiter w{abort_flag, p.status, kRoleFlush};
    bwd_flush_role<D, CAUSAL>(&tm_dq, sbase, p, w);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa4
