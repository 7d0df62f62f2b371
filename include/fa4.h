/*
 * fa4.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The operation is exact attention forward with a per-row logsumexp,
 * computed tile by tile with an online softmax so that the score matrix S
 * and the probabilities P never reach HBM. It is the forward pass described
 * in "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
 * Asymmetric Hardware Scaling" (Method; §3.1.1-§3.1.4; Table 1, Table 2,
 * Eq. 6) and "How FlashAttention 4 Works" (warp roles, TMA load warp,
 * lazy rescale, cubic 2^x approximation).
 *
 * For every batch b, query head h and query row i, with kv head
 * g = h / (Hq / Hkv):
 *     x_j       = scale * <q[b,i,h,:], k[b,j,g,:]>
 *     valid(j)  = !causal || j <= i + (Sk - Sq)      (bottom-right causal)
 *     O[b,i,h,:] = sum_{valid j} exp(x_j - m) v[b,j,g,:] / sum_{valid j} exp(x_j - m)
 *     LSE[b,h,i] = m + ln sum_{valid j} exp(x_j - m),   m = max_{valid j} x_j
 * A row with no valid key gets O = 0 and LSE = -inf.
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense and contiguous: q, o [B, Sq, Hq, d] BF16;
 *     k, v [B, Sk, Hkv, d] BF16; lse [B, Hq, Sq] fp32 (natural log).
 *   - Pointers are DEVICE pointers owned by the caller; the library keeps
 *     none of them after the call returns and allocates no device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). They validate their arguments first and launch
 *     nothing when validation fails.
 *   - Kernel waits are bounded. A pipeline stage that stalls for longer
 *     than its limit makes the kernel give up cleanly and record
 *     FA4_ERR_TIMEOUT in a per-device status word that fa4_device_status()
 *     reads; the CUDA context stays usable.
 *   - All functions are thread-safe.
 */
#ifndef FA4_H_
#define FA4_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t. */
typedef struct CUstream_st *fa4_stream_t;

typedef enum {
    FA4_OK = 0,
    FA4_ERR_INVALID_ARG = 1,  /* null pointer, bad size, aliasing, bad scale   */
    FA4_ERR_UNSUPPORTED = 2,  /* head dim not in {64,128}; device not cc 10.3  */
    FA4_ERR_MISALIGNED = 3,   /* q/k/v/o not 16-byte aligned, lse not 4-byte   */
    FA4_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed              */
    FA4_ERR_TIMEOUT = 5       /* a kernel pipeline wait ran out (device status) */
} fa4_status;

/* Options of fa4_fwd_ex. Fill with fa4_fwd_default_options() first. */
typedef struct {
    /* Conditional-rescale threshold in log2 units ("FlashAttention-4",
     * §3.1.4, Eq. 6): the running output is only rescaled when a row's new
     * block maximum exceeds the reference maximum by more than tau.
     * 8.0 (= log2 256) is the default; 0.0 gives the eager online softmax.
     * Must be finite and in [0, 64]. */
    float tau;
    /* Software 2^x beside MUFU.EX2 ("FlashAttention-4", §3.1.3): N = 8 or
     * N = 4 runs a Cody-Waite + degree-3 Horner polynomial on one softmax
     * entry pair in N (12.5 % or 25 % of the entries; 1 means 8), 0 sends
     * every entry through MUFU.EX2. Default 0: on GB300, whose MUFU issues
     * twice the exponentials per clock of the B200 the method was tuned
     * for, the all-MUFU path measured faster at both head dimensions. */
    int exp2_emulation;
    /* Optional DEVICE pointer to two uint64 counters, or NULL. When set, the
     * kernel adds [0] += number of (32-row group, key block) steps that
     * rescaled the output, [1] += number of such steps after the first key
     * block of each tile. The caller zeroes them. */
    unsigned long long *rescale_stats;
    /* Optional DEVICE pointer to a cycle trace, or NULL (diagnostic). CTAs
     * with block index < trace_ctas record the SM cycle counter at fixed
     * points of the load/MMA/softmax/correction roles into
     * trace[((cta * FA4_TRACE_EVENTS + event) * FA4_TRACE_STEPS + j) * 2 + t]
     * for key block j < FA4_TRACE_STEPS and query tile t in {0, 1}; the
     * buffer holds trace_ctas * FA4_TRACE_EVENTS * FA4_TRACE_STEPS * 2
     * uint64 values. Events, in order: MMA waits for an S slot, S issued,
     * MMA waits for the corrected O, P*V issued, softmax sees S, S in
     * registers, P computed, P stored, correction wakes, correction done,
     * MMA S dependencies met, MMA P*V dependencies met, P stored by softmax
     * warps 2, 3 and 4 of the tile, softmax block max known, MMA released
     * the key block's slots (t = 0), V_j resident (t = 0), load warp issued
     * V_j (t = 0) / K_j (t = 1). */
    unsigned long long *trace;
    int trace_ctas;
    /* 0 (default): the MMA that computes the next score tile S_t into the
     * tensor-memory columns where the probabilities P_t of the previous
     * key block live is issued right behind the P_t*V MMA that reads them,
     * relying on the tensor core running one thread's MMAs in issue order
     * (the two-tile ping-pong of "FlashAttention-4" §3.1.2). 1: wait for
     * the P_t*V MMA to complete first (slower; the PTX memory model only
     * promises issue order for MMAs into the same accumulator). At head
     * dimension 64 in the persistent grid (grid_mode 2, or chosen
     * automatically) P_t has its own tensor-memory columns, no score MMA
     * overwrites it, and the flag changes nothing. */
    int strict_mma_order;
    /* Grid of CTAs: 0 (default) chooses automatically; 1: one CTA per work
     * tile (two 128-row query tiles of one batch and head), scheduled by the
     * hardware; 2: persistent, one CTA per SM, each taking work tiles in
     * snake order. Both compute identical results. */
    int grid_mode;
    /* Who rescales the output accumulator when a row group's reference
     * maximum moves (the conditional rescale of "FlashAttention-4" §3.1.4):
     * 0 (default): the softmax warp of those 32 rows, before it releases
     * the accumulator to the next P*V -- under tau = 8 rescales are rare
     * (on the GQA stress workload 0.3 % of row-group steps), and on GB300
     * dropping the per-step hand-off measured 2-10 % faster; 1: a separate
     * correction warpgroup, off the softmax's path, as the pages describe
     * (§3.1.2). Both compute identical results. */
    int correction_warpgroup;
    /* Diagnostic, 0 by default (must be >= 0). When positive, the softmax
     * warps of every CTA first wait on a barrier that nothing completes and
     * give up after this many SM cycles: the kernel then takes its timeout
     * path (abort flag, in-flight copies and MMAs drained, tensor memory
     * freed), fa4_device_status reports FA4_ERR_TIMEOUT with role 2
     * (softmax), and O and LSE are left unwritten. It exercises the abort
     * path without a GPU fault; the context stays usable. */
    long long test_stall_cycles;
} fa4_fwd_options;

#define FA4_TRACE_EVENTS 21
#define FA4_TRACE_STEPS 128

/* Default options: tau = 8, exp2_emulation = 0, no counters, no trace,
 * strict_mma_order = 0, grid_mode = 0, correction_warpgroup = 0,
 * test_stall_cycles = 0. */
void fa4_fwd_default_options(fa4_fwd_options *opt);

/*
 * fa4_fwd -- attention forward with default options.
 *
 *   q      [B, Sq, Hq, d]  BF16, device, 16-byte aligned
 *   k, v   [B, Sk, Hkv, d] BF16, device, 16-byte aligned
 *   o      [B, Sq, Hq, d]  BF16, device, 16-byte aligned, written
 *   lse    [B, Hq, Sq]     fp32, device, 4-byte aligned, written
 *   B, Sq, Sk >= 0 (B*Sq == 0 is a no-op; Sk == 0 gives O = 0, LSE = -inf);
 *   Hq, Hkv >= 1 with Hq % Hkv == 0; d in {64, 128};
 *   scale finite and > 0 (usually 1/sqrt(d)); causal 0 or 1.
 *   o and lse must not overlap q, k, v or each other.
 *
 * Returns FA4_OK after the kernel is enqueued, or an error code with
 * nothing launched.
 */
fa4_status fa4_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                   int causal, fa4_stream_t stream);

/* fa4_fwd with explicit options (opt may be NULL for the defaults). */
fa4_status fa4_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                      int causal, const fa4_fwd_options *opt, fa4_stream_t stream);

/*
 * fa4_fwd_host -- the forward with inputs and outputs in HOST memory: on
 * `stream`, copies q, k, v into the device workspace (one cudaMemcpyAsync
 * each), runs the forward there, and copies o and lse back. Meant for
 * callers whose data lives on the host; host buffers should be pinned
 * (page-locked) for the copies to be asynchronous. Same operation as
 * fa4_fwd_ex.
 *
 *   q, k, v          HOST, layouts as fa4_fwd (BF16), read
 *   o, lse           HOST, layouts as fa4_fwd, written once the stream has
 *                    passed this call (synchronise before reading them)
 *   workspace        DEVICE scratch owned by the caller, 256-byte aligned, at
 *                    least fa4_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk,
 *                    d) bytes: device copies of q, k, v, o and lse in that
 *                    order, each starting on a 256-byte boundary; it may be
 *                    reused once the stream has passed this call.
 *   other arguments as fa4_fwd_ex.
 * Every argument is checked before anything is enqueued. Returns
 * FA4_ERR_INVALID_ARG for a missing or small workspace, FA4_ERR_MISALIGNED
 * for a misaligned one, FA4_ERR_CUDA if a copy cannot be enqueued, and
 * otherwise as fa4_fwd_ex.
 */
uint64_t fa4_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d);
fa4_status fa4_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                        int causal, void *workspace, uint64_t workspace_bytes,
                        const fa4_fwd_options *opt, fa4_stream_t stream);

/*
 * fa4_fwd_fp8 -- the same forward with Q, K and V in FP8 (e4m3): both
 * products run on the tensor cores with 8-bit inputs and an fp32
 * accumulator, the softmax stays in fp32, P is rounded to e4m3 for the
 * second product, and O is stored in BF16 ("How FlashAttention 4 Works",
 * the section on where low precision is safe: Q K^T and P V in FP8,
 * softmax in FP32, the output in BF16/FP16).
 *
 * The inputs are scaled codes: the true values are q * q_scale, k * k_scale
 * and v * v_scale. The result is the forward of those true values,
 *     S = scale q_scale k_scale (q k^T),   O = v_scale softmax(S) v,
 * with LSE the natural-log logsumexp of S.
 *
 *   q                [B, Sq, Hq, 128] e4m3 bytes, device, 16-byte aligned
 *   k, v             [B, Sk, Hkv, 128] e4m3 bytes, device, 16-byte aligned
 *   o                [B, Sq, Hq, 128] BF16, written
 *   lse              [B, Hq, Sq] fp32, written
 *   q_scale, k_scale, v_scale  finite and > 0
 *   other arguments as fa4_fwd_ex. Only d = 128 is built; options must keep
 *   exp2_emulation = 0 and trace = NULL.
 * Returns FA4_ERR_UNSUPPORTED for d != 128 or those options,
 * FA4_ERR_INVALID_ARG for a bad scale, otherwise as fa4_fwd_ex.
 */
fa4_status fa4_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                       int causal, float q_scale, float k_scale, float v_scale,
                       const fa4_fwd_options *opt, fa4_stream_t stream);

/*
 * fa4_bwd -- attention backward: the gradients of O = softmax(scale QK^T
 * [+causal]) V with respect to q, k, v for an upstream gradient dout
 * ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
 * Asymmetric Hardware Scaling", §3.2: five MMAs per tile pair -- S, dP,
 * dV += P^T dO, dK += dS^T Q, dQ += dS K -- with
 * dS = P o (dP - rowsum(dO o O))).
 *
 *   q, o, dout       [B, Sq, Hq, d]  BF16, device, 16-byte aligned (o and lse
 *                    are the forward's outputs for these q, k, v)
 *   k, v             [B, Sk, Hkv, d] BF16, device, 16-byte aligned
 *   lse              [B, Hq, Sq]     fp32 natural-log LSE, 4-byte aligned
 *   dq               [B, Sq, Hq, d]  BF16, written
 *   dk, dv           [B, Sk, Hkv, d] BF16, written (a kv head's gradient sums
 *                    over the query heads of its group)
 *   workspace        DEVICE scratch owned by the caller, 16-byte aligned, at
 *                    least fa4_bwd_workspace_bytes(B, Hq, Sq, d) bytes: the
 *                    fp32 dQ accumulator [B, Sq, Hq, d], then LSE log2(e)
 *                    and rowsum(dO o O), each [B, Hq, Sq rounded up to 128],
 *                    then one int per (batch, query head, 64-query block)
 *                    (padded to 16 bytes), then one int (the CTA ticket).
 *   other arguments and rules as fa4_fwd; dq, dk, dv and the workspace
 *   must not overlap each other or any input.
 * Enqueues a memset, a preprocessing kernel, the main kernel and a
 * conversion kernel on `stream`. Sq == 0 gives dk = dv = 0; Sk == 0 gives
 * dq = 0.
 */
uint64_t fa4_bwd_workspace_bytes(int B, int Hq, int Sq, int d);
fa4_status fa4_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                   int Sq, int Sk, int d, float scale, int causal, void *workspace,
                   uint64_t workspace_bytes, fa4_stream_t stream);

/*
 * fa4_bwd_ex -- fa4_bwd with deterministic = 0 (the same) or 1: the tiles
 * of dQ that different key blocks contribute are added to the fp32
 * accumulator in key-block order (each CTA waits for its turn on a per
 * query-block counter kept in the workspace; CTAs number their work in the
 * order they start, from a counter in the workspace, so a CTA only ever
 * waits for CTAs that are already running), so dq is bit-for-bit the same
 * on every run ("FlashAttention-4: Algorithm and Kernel Pipelining
 * Co-Design for Asymmetric Hardware Scaling", §1: a deterministic execution
 * mode for reproducible training). dk and dv are deterministic in both
 * modes (each is accumulated inside one CTA).
 */
fa4_status fa4_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                      const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                      int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                      int deterministic, void *workspace, uint64_t workspace_bytes,
                      fa4_stream_t stream);

/* Options of fa4_bwd_opt. Fill with fa4_bwd_default_options() first. */
typedef struct fa4_bwd_options {
    /* 0 or 1, as fa4_bwd_ex's deterministic. */
    int deterministic;
    /* Diagnostic, >= 0; 0 (the default) disables it. With a positive value
     * the compute warps first wait on a barrier that nothing completes, for
     * that many SM cycles: the wait runs out and the launch takes the
     * timeout path (fa4_device_status reports FA4_ERR_TIMEOUT with role 2;
     * dk and dv are not written). Tests use it; results are meaningless. */
    long long test_stall_cycles;
} fa4_bwd_options;

/* Default options: deterministic = 0, test_stall_cycles = 0. */
void fa4_bwd_default_options(fa4_bwd_options *opt);

/*
 * fa4_bwd_opt -- fa4_bwd with options (NULL: the defaults). Arguments,
 * workspace and return codes as fa4_bwd; FA4_ERR_INVALID_ARG also for
 * deterministic outside {0, 1} or a negative test_stall_cycles.
 */
fa4_status fa4_bwd_opt(const void *q, const void *k, const void *v, const void *o,
                       const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                       int Hq, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                       const fa4_bwd_options *opt, void *workspace, uint64_t workspace_bytes,
                       fa4_stream_t stream);

/*
 * fa4_fwd_splitkv -- the same forward, with the keys cut into num_splits
 * contiguous ranges of whole 128-key blocks that separate CTAs process in
 * parallel, then combined. Meant for shapes with few query tiles and many
 * keys (short Sq, long Sk), where one CTA per query tile would leave SMs
 * idle. The combine is exact: each range yields its softmax-normalised
 * output O_s and logsumexp L_s, and
 *     LSE = log sum_s exp(L_s),   O = sum_s exp(L_s - LSE) O_s
 * is the softmax over the union of the ranges ("FlashAttention-4:
 * Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware
 * Scaling", Method: the output is recovered exactly at the final
 * normalisation; here that normalisation is applied once more across key
 * ranges -- the exchange step a key-parallel forward needs).
 *
 * Arguments as fa4_fwd, plus:
 *   num_splits       1 .. 128 requested ranges (ranges that would start past
 *                    the last key block are dropped; each range holds
 *                    ceil(ceil(Sk / 128) / num_splits) blocks);
 *   workspace        DEVICE scratch owned by the caller, 16-byte aligned,
 *                    not overlapping any other argument, at least
 *                    fa4_fwd_splitkv_workspace_bytes(B, Hq, Sq, d,
 *                    num_splits) bytes. Layout: fp32 partial outputs
 *                    [num_splits][B][Sq][Hq][d], then fp32 partial LSE
 *                    [num_splits][B][Hq][Sq]. Its contents on return are
 *                    unspecified; it may be reused once the stream has
 *                    passed this call.
 *   opt              as fa4_fwd_ex (may be NULL).
 * Enqueues two kernels (the split forward and the combine) on `stream`.
 * Returns FA4_ERR_INVALID_ARG for a bad num_splits or a missing, small or
 * overlapping workspace, FA4_ERR_MISALIGNED for a misaligned one, and
 * otherwise as fa4_fwd_ex.
 */
uint64_t fa4_fwd_splitkv_workspace_bytes(int B, int Hq, int Sq, int d, int num_splits);
fa4_status fa4_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int Hq, int Hkv, int Sq, int Sk, int d, float scale,
                           int causal, int num_splits, void *workspace,
                           uint64_t workspace_bytes, const fa4_fwd_options *opt,
                           fa4_stream_t stream);

/*
 * fa4_fwd_splitkv_static -- fa4_fwd_splitkv without a caller workspace: the
 * partial results go to a scratch array the library holds in device memory
 * (a fixed-size file-scope __device__ array, one per device; nothing is
 * allocated or freed at run time). The pages have no counterpart to this
 * entry point; it exists for callers that cannot hand over a workspace.
 *
 * Arguments as fa4_fwd_splitkv without workspace / workspace_bytes, checked
 * in the same order and with the same status codes. The scratch holds
 * fa4_fwd_splitkv_static_max_bytes() bytes (32 MiB); a call with otherwise
 * valid arguments whose fa4_fwd_splitkv_workspace_bytes(B, Hq, Sq, d,
 * num_splits) exceeds it returns FA4_ERR_INVALID_ARG with nothing launched.
 *
 * The array lives in the library's module, so it takes its 32 MiB of
 * device memory on every device where any entry point of this library has
 * run, whether or not this one is ever called, until the process exits.
 *
 * The first call on each device looks up the scratch's device address
 * (cudaGetSymbolAddress) and caches it for the life of the process; make
 * that first call before any stream capture. The cached address belongs to
 * the device's primary context: do not use the library on a device after
 * cudaDeviceReset (or any other teardown of that context) in the same
 * process. All calls on a device share the one scratch array, so
 * calls whose kernels can overlap in time -- on different streams, or from
 * different host threads without ordering between their streams -- race on
 * it and give undefined results. Calls on one stream are ordered and safe.
 */
uint64_t fa4_fwd_splitkv_static_max_bytes(void);
fa4_status fa4_fwd_splitkv_static(const void *q, const void *k, const void *v, void *o,
                                  float *lse, int B, int Hq, int Hkv, int Sq, int Sk, int d,
                                  float scale, int causal, int num_splits,
                                  const fa4_fwd_options *opt, fa4_stream_t stream);

/*
 * fa4_device_status -- synchronise the current device and return the
 * kernel-side status word: FA4_OK, or FA4_ERR_TIMEOUT if any kernel of
 * this library gave up on a pipeline wait since the last clear. `detail`
 * (may be NULL) receives 4 words: the error code, the waiting role
 * (0 load, 1 mma, 2 softmax -- the backward's compute warps --,
 * 3 correction, 4 the backward's dQ flush warp, 5 the backward's dQ^T
 * read-out warps), the barrier id (an index
 * into the kernel's own barrier table) and the block index. When `clear`
 * is non-zero the word is reset to FA4_OK.
 * Returns FA4_ERR_CUDA if the device cannot be reached.
 */
fa4_status fa4_device_status(int clear, unsigned int *detail);

/*
 * fa4_exp2_eval -- diagnostic: evaluate the kernel's two 2^x paths on n
 * fp32 inputs: y_emu[i] = Cody-Waite + degree-3 polynomial emulation (the paired
 * form the softmax runs),
 * y_mufu[i] = MUFU.EX2 (ex2.approx.ftz.f32). All three pointers are device
 * fp32 arrays of n elements (n >= 0). This is the kernel's own device
 * function ("FlashAttention-4", §3.1.3, Table 2), exported so it can be
 * checked exhaustively over every BF16 input.
 */
fa4_status fa4_exp2_eval(const float *x, float *y_emu, float *y_mufu, int64_t n,
                         fa4_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *fa4_status_string(fa4_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA4_H_ */
