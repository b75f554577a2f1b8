/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward pass and
 * its backward pass (kda_bwd).
 *
 * The entry point mirrors the call printed in "Flashkda Delta Attention",
 * section "Core Kernel API":
 *     fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
 *         initial_state=None, final_state=None, cu_seqlens=None)
 * with the constraints of "MoonshotAI/FlashKDA" (trend summary), section
 * "Kernel API and Constraints": K = V = 128, cu_seqlens only with B = 1,
 * states bf16, fp32 or absent and of matching dtype when both are given;
 * activations are bf16 ("Flashkda Delta Attention", opening summary).
 *
 * Operation (per sequence n and head h; the pages print no formula, so the
 * plain gated-delta-rule reading is taken and the gate form is a reading of
 * the parameter names A_log, dt_bias, lower_bound):
 *     la_t = max(-exp(A_log[h]) * softplus(g_t + dt_bias[h]), lower_bound)
 *     S_t  = (I - beta_t k_t k_t^T) Diag(exp(la_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t  = scale * S_t^T q_t
 * S_0 = initial_state[n, h] (or 0); final_state[n, h] = S at the sequence end.
 * q and k are used as given (no normalisation inside the call); kda_fwd_ex
 * can normalise them first.
 *
 * Every pointer handed to kda_fwd is DEVICE memory owned by the caller; the
 * call reads the inputs, writes out (and final_state) and keeps no reference
 * after it returns.  The call is asynchronous on `stream`: it returns once the
 * work is enqueued.  Scratch memory for the per-chunk intermediates is taken
 * from the stream-ordered allocator (cudaMallocAsync / cudaFreeAsync on
 * `stream`) unless the caller supplies a workspace through kda_fwd_ws.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 1

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* bad shape / dtype / pointer; nothing launched */
    KDA_ERR_UNSUPPORTED = 2,      /* valid but outside the kernels' range (e.g. lower_bound) */
    KDA_ERR_CUDA = 3,             /* a CUDA runtime call failed; see kda_last_error_message */
    KDA_ERR_TIMEOUT = 4,          /* a bounded device-side wait gave up (reported by kda_device_status) */
    KDA_ERR_DEVICE_INPUT = 5      /* malformed device-side input (cu_seqlens) detected on the device */
} kda_status_t;

typedef enum {
    KDA_DTYPE_NONE = 0, /* state absent */
    KDA_DTYPE_BF16 = 1,
    KDA_DTYPE_FP32 = 2
} kda_dtype_t;

/*
 * kda_fwd -- KDA forward pass ("Flashkda Delta Attention", "Core Kernel API").
 *
 *   q, k, g     bf16 [B, T, H, K] contiguous (token-major; packed: B = 1, T = total)
 *   v           bf16 [B, T, H, V]
 *   beta        bf16 [B, T, H]
 *   scale       output scale (commonly K^-0.5)
 *   out         bf16 [B, T, H, V], written (round-to-nearest-even)
 *   A_log       fp32 [H]
 *   dt_bias     fp32 [H, K]
 *   lower_bound clamp of the log-decay; finite, <= 0.  The kernels factor the
 *               in-chunk decays around 16-token sub-blocks, which is exact in
 *               fp32 for lower_bound >= -10; below that the call returns
 *               KDA_ERR_UNSUPPORTED.
 *   initial_state  [N, H, K, V] in initial_dtype, or NULL with KDA_DTYPE_NONE
 *                  (zeros).  S[n][h][c][j]: key channel c, value channel j.
 *   final_state    [N, H, K, V] in final_dtype, written, or NULL with
 *                  KDA_DTYPE_NONE.  May alias initial_state exactly (in place);
 *                  any other overlap is rejected.  When both states are given
 *                  their dtypes must match.
 *   cu_seqlens  int32 [num_seqs + 1] device offsets of packed sequences, or NULL
 *               (then the B rows are the sequences).  Requires B = 1.  Must be
 *               0 = cu[0] <= cu[1] <= ... <= cu[num_seqs] = T; zero-length
 *               sequences are allowed (their final state is their initial
 *               state).  A violation is detected on the device: the call then
 *               skips all work and kda_device_status reports
 *               KDA_ERR_DEVICE_INPUT.
 *   num_seqs    number of packed sequences (ignored when cu_seqlens is NULL)
 *   B, T, H, K, V  sizes; K = V = 128 is required, H >= 1, T >= 0, B >= 1.
 *   stream      CUDA stream (cudaStream_t passed as void*; NULL = legacy default)
 *
 * N = num_seqs with cu_seqlens, else B.
 * Returns KDA_OK once enqueued; argument errors are reported synchronously
 * and launch nothing.
 */
kda_status_t kda_fwd(const void* q, const void* k, const void* v, const void* g,
                     const void* beta, float scale, void* out, const float* A_log,
                     const float* dt_bias, float lower_bound, const void* initial_state,
                     kda_dtype_t initial_dtype, void* final_state, kda_dtype_t final_dtype,
                     const int32_t* cu_seqlens, int32_t num_seqs, int32_t B, int32_t T,
                     int32_t H, int32_t K, int32_t V, void* stream);

/*
 * kda_workspace_size -- bytes of device scratch kda_fwd_ws needs for a
 * problem with these sizes (an upper bound that does not read cu_seqlens),
 * for the recurrence selection in force (kda_set_recurrence_kernel: the
 * segmented path needs room for its per-segment states, so query the size
 * after choosing).  A problem that takes the single-token step (T = 1 without
 * cu_seqlens, automatic selection) uses no scratch: the answer is then 256.
 * Returns 0 and sets the error message for invalid sizes.
 */
size_t kda_workspace_size(int32_t B, int32_t T, int32_t H, int32_t num_seqs, int32_t has_cu_seqlens);

/*
 * kda_fwd_ws -- kda_fwd with caller-provided scratch: `workspace` is device
 * memory of at least kda_workspace_size(...) bytes, 256-byte aligned, owned by
 * the caller and not used by anything else until the enqueued work finishes.
 * Makes no allocation.  Same arguments and errors as kda_fwd otherwise.
 */
kda_status_t kda_fwd_ws(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, float scale, void* out, const float* A_log,
                        const float* dt_bias, float lower_bound, const void* initial_state,
                        kda_dtype_t initial_dtype, void* final_state, kda_dtype_t final_dtype,
                        const int32_t* cu_seqlens, int32_t num_seqs, int32_t B, int32_t T,
                        int32_t H, int32_t K, int32_t V, void* workspace,
                        size_t workspace_bytes, void* stream);

/* kda_fwd_ex flag: scale every row of q and k (one token of one head, K
 * channels) to x / sqrt(sum_c x_c^2 + 1e-6) inside the kernels before use. */
#define KDA_FWD_QK_L2NORM 1u

/*
 * kda_fwd_ex -- kda_fwd with options.  The call printed in "Flashkda Delta
 * Attention", "Core Kernel API", takes q and k as given; callers that hold
 * raw (un-normalised) query/key projections would otherwise run a separate
 * normalisation pass over q and k in HBM first.  With KDA_FWD_QK_L2NORM the
 * chunk kernel (and the single-token step) normalise each row of the staged
 * q / k tiles instead; the normalised rows are rounded to bf16 like the
 * inputs before use.  `flags`: 0 or KDA_FWD_QK_L2NORM (other bits return
 * KDA_ERR_INVALID_ARGUMENT).  `workspace`: as for kda_fwd_ws, or NULL to take
 * scratch from the stream-ordered allocator as kda_fwd does (then
 * workspace_bytes is ignored).  Same arguments and errors as kda_fwd otherwise.
 */
kda_status_t kda_fwd_ex(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, float scale, void* out, const float* A_log,
                        const float* dt_bias, float lower_bound, const void* initial_state,
                        kda_dtype_t initial_dtype, void* final_state, kda_dtype_t final_dtype,
                        const int32_t* cu_seqlens, int32_t num_seqs, int32_t B, int32_t T,
                        int32_t H, int32_t K, int32_t V, uint32_t flags, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * kda_fwd_noalloc -- kda_fwd for callers that must not allocate device memory
 * during the call (no counterpart on the pages).  Some callers cannot: a
 * serving runtime that reserves all GPU memory at start-up and forbids
 * allocation on the request path, a plug-in running under memory pools it does
 * not own, or real-time code that cannot pay for an allocator call.  This
 * entry point allocates nothing: its scratch is a fixed area compiled into
 * the library (kda_noalloc_scratch_bytes(), 64 MiB), which every GPU that
 * loads the library holds until the process exits.  Inputs and outputs are
 * the caller's, exactly as for kda_fwd.
 *   - A problem whose kda_workspace_size exceeds the area is rejected with
 *     KDA_ERR_UNSUPPORTED and a message giving both sizes.  Single-token
 *     problems (T = 1 without cu_seqlens, automatic recurrence selection)
 *     take the single-token step, which uses no scratch, so every batch size
 *     of them is accepted.
 *   - The first call on a device looks up the area's address on that device
 *     (it must be the current device); make that first call before any stream
 *     capture.
 *   - All calls share the one area and it keeps the last call's contents;
 *     calls whose GPU work overlaps (other streams or host threads) race on it
 *     and must be serialised by the caller.
 */
kda_status_t kda_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                             const void* beta, float scale, void* out, const float* A_log,
                             const float* dt_bias, float lower_bound, const void* initial_state,
                             kda_dtype_t initial_dtype, void* final_state,
                             kda_dtype_t final_dtype, const int32_t* cu_seqlens, int32_t num_seqs,
                             int32_t B, int32_t T, int32_t H, int32_t K, int32_t V, void* stream);

/* Size in bytes of the fixed scratch area kda_fwd_noalloc uses. */
size_t kda_noalloc_scratch_bytes(void);

/*
 * kda_bwd -- backward pass of kda_fwd (no counterpart on the pages, which
 * print the forward call only; the operation differentiated is the one stated
 * at the top of this file, q and k used as given).  Computes the gradients of
 *     L = sum(dout * out) + sum(dfinal_state * final_state)
 * with respect to every input (q and k as given, or normalised first with
 * KDA_FWD_QK_L2NORM in flags):
 *   dq, dk, dg     fp32 [B, T, H, K], written
 *   dv             fp32 [B, T, H, V], written
 *   dbeta          fp32 [B, T, H], written
 *   dA_log         fp32 [H], written (sum over all sequences and tokens)
 *   ddt_bias       fp32 [H, K], written (likewise)
 *   dinitial_state fp32 [N, H, K, V], written, or NULL (not wanted)
 * Inputs are those of kda_fwd (same layouts, dtypes and constraints on q, k,
 * v, g, beta, A_log, dt_bias, initial_state, cu_seqlens and the sizes) plus
 *   dout           bf16 [B, T, H, V], the gradient of out
 *   dfinal_state   fp32 [N, H, K, V], or NULL (no final-state term)
 * flags: a combination of
 *   KDA_FWD_QK_L2NORM   the gradients of kda_fwd_ex with that flag: q and k enter
 *                       the recurrence as x / sqrt(|x|^2 + 1e-6) row by row, and
 *                       dq, dk are the gradients with respect to the raw rows (the
 *                       chain rule through that map, dx = (dxhat - xhat (xhat .
 *                       dxhat)) / n).  The normalised rows are used unrounded
 *                       here (the forward rounds them to bf16; that rounding is
 *                       taken as the identity).
 *   KDA_BWD_LOW_MEMORY  keep one fp32 state per 64 tokens (about 1 KB per token
 *                       per head, plus 32 MiB) instead of one per 8 tokens (about
 *                       8 KB); each 64-token chunk is replayed once more during
 *                       the reverse walk.  Same results, bit for bit; slower.
 * Other bits return KDA_ERR_INVALID_ARGUMENT.
 * lower_bound: finite, <= 0 (no other range limit: the backward pass does not
 * use the forward's sub-block factorisation).  The clamp max(pre, lower_bound)
 * passes its gradient to the argument it returns, and to pre at a tie.
 * Arithmetic is fp32 throughout, token by token; the results are
 * deterministic (every sum is taken in a fixed order).
 * All pointers are DEVICE memory owned by the caller, 16-byte aligned (beta:
 * 2-byte, dbeta: 4-byte); outputs must not overlap inputs or one another.
 * `workspace`: device memory of at least kda_bwd_workspace_size(...) bytes,
 * 256-byte aligned, or NULL to take it from the stream-ordered allocator on
 * `stream` (workspace_bytes is then ignored).  The scratch holds fp32 copies
 * of the state every 8 tokens (about 8 KB per token per head), or every 64
 * with KDA_BWD_LOW_MEMORY.
 * Asynchronous on `stream`; argument errors are reported synchronously and
 * launch nothing.  A malformed cu_seqlens (as for kda_fwd) is detected on the
 * device: the affected sequences are skipped and kda_device_status reports
 * KDA_ERR_DEVICE_INPUT; the gradients of that call are then undefined.
 */
kda_status_t kda_bwd(const void* q, const void* k, const void* v, const void* g,
                     const void* beta, float scale, const float* A_log, const float* dt_bias,
                     float lower_bound, const void* initial_state, kda_dtype_t initial_dtype,
                     const void* dout, const float* dfinal_state, const int32_t* cu_seqlens,
                     int32_t num_seqs, int32_t B, int32_t T, int32_t H, int32_t K, int32_t V,
                     float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dA_log,
                     float* ddt_bias, float* dinitial_state, uint32_t flags, void* workspace,
                     size_t workspace_bytes, void* stream);

/* kda_bwd flag: checkpoint the state every 64 tokens instead of every 8. */
#define KDA_BWD_LOW_MEMORY 2u

/* Bytes of device scratch kda_bwd needs for these sizes and flags (does not
 * read cu_seqlens).  Returns 0 and sets the error message for invalid sizes or
 * unknown flag bits. */
size_t kda_bwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t num_seqs,
                              int32_t has_cu_seqlens, uint32_t flags);

/*
 * kda_device_status -- synchronises `stream`, then returns and clears the
 * library's per-device status word: KDA_OK, KDA_ERR_DEVICE_INPUT (malformed
 * cu_seqlens seen by an earlier call), KDA_ERR_TIMEOUT (a bounded
 * device-side wait gave up; that call's outputs are undefined) or KDA_ERR_CUDA
 * (a chunk kernel found its shared-memory area misaligned for its swizzled
 * tensor store and skipped its work, or a low-memory kda_bwd call found no free
 * replay slot, which cannot happen while at most one of its CTAs runs per SM;
 * outputs undefined).
 */
kda_status_t kda_device_status(void* stream);

/* Human-readable name of a status code (static storage). */
const char* kda_status_string(kda_status_t status);

/* Detail of the last error returned on the calling host thread (thread-local). */
const char* kda_last_error_message(void);

/*
 * kda_last_path -- how the calling host thread's last successful kda_fwd /
 * kda_fwd_ws / kda_fwd_noalloc call with a non-empty problem ran (no
 * counterpart on the pages; for benchmarks and diagnostics): 1 = chunk kernel
 * then value-sliced recurrence, 2 = chunk kernel then transposed recurrence,
 * 3 = the fused cooperative launch, 4 = the single-token step (T = 1 without
 * cu_seqlens, chosen automatically: one pass over the states, the workspace
 * is not used), 5 = the segmented path (chunk kernel, per-segment state maps,
 * scan, value-sliced recurrence over the segments); 0 before any such call.
 */
int kda_last_path(void);

/* KDA_ABI_VERSION of the built library. */
int kda_abi_version(void);

/*
 * kda_set_stage_events -- timing hook (no counterpart on the pages).  With
 * count = 4 or 6, every later kda_fwd / kda_fwd_ws call on this process
 * records events[0] before its first kernel, events[1] after the schedule
 * kernels, events[2] after the chunk kernel and events[3] after the recurrence
 * kernel, all on the call's stream; on the segmented path events[3] follows
 * the map pass, events[4] the scan and events[5] the recurrence (recorded only
 * with count = 6).  The single-token step records events[0] and events[1]
 * around its one kernel.  Events are cudaEvent_t created by the caller and
 * must outlive the calls.  count = 0 (or events = NULL) turns the hook off;
 * any other count returns KDA_ERR_INVALID_ARGUMENT.  Not thread-safe; intended
 * for benchmarks.
 */
kda_status_t kda_set_stage_events(void* const* events, int32_t count);

/*
 * kda_set_recurrence_kernel -- selects how the sequential chunk-to-chunk
 * recurrence runs (no counterpart on the pages; every choice computes the same
 * operation to the same tolerance).  kind = 0 (default): chosen per call from
 * the number of (sequence, head) pairs, the chunks per sequence and the SM
 * count, with single-token problems (T = 1, no cu_seqlens) taking the
 * single-token step instead of the chunked path; 1: the value-sliced kernel
 * (state slices of 32..128 value channels, one CTA each); 2: the transposed
 * kernel (one CTA per (sequence, head), state held as S^T); 3: the fused
 * launch (chunk kernel and transposed recurrence in one cooperative kernel,
 * overlapping; used only when the pairs leave at least one SM for the chunk
 * kernel, else kind 2 runs); 4: the segmented path (each sequence's chunks
 * split into 2..32 segments; the affine state map of every segment is found
 * in parallel, the maps are scanned in fp32, and the value-sliced recurrence
 * then runs all segments at once from their entering states; automatic
 * selection takes it for few, long sequences; forced, it falls back to the
 * kind-0 choice between 1 and 2 when the (sequence, head) pairs exceed half
 * the SM count, where the segments could not run side by side).  Process-wide
 * (an atomic setting, safe to change from any thread): it applies to calls
 * that start after it returns, including kda_workspace_size, so a caller that
 * sizes a workspace must not change it between the query and the call.  Any
 * other kind returns KDA_ERR_INVALID_ARGUMENT.
 */
kda_status_t kda_set_recurrence_kernel(int32_t kind);

/*
 * kda_set_wait_limit_ns -- test hook (no counterpart on the pages).  Every
 * device-side wait of the kernels that can give up (an mbarrier wait for a
 * copy or an MMA, or the fused launch's wait for a chunk record) is bounded by
 * this limit, 2e9 ns (2 s) by default.  A wait that runs out records
 * KDA_ERR_TIMEOUT in the status word (see kda_device_status), the CTA stops,
 * waits for its own copies and MMAs in flight (with a separate 4 s limit),
 * frees its tensor memory and exits, and later CTAs of the launch exit at
 * once.  A short limit makes that path run on purpose; the outputs of a call
 * that timed out are undefined, and the next call is unaffected.
 * limit_ns in [1, 2e9]; applies to the current device and to kernels
 * launched after the call (it writes a word of the device's status block).
 */
kda_status_t kda_set_wait_limit_ns(uint64_t limit_ns);

/*
 * kda_selftest_tcgen05 -- diagnostic for the tensor-core building blocks the
 * kernels use (no counterpart on the pages).  Runs one M=128 x N x K bf16 MMA
 * per operand-layout combination (A and B each K-major or MN-major, no
 * swizzle) on device inputs a [128][K] and b [K][N] (row-major bf16), writing
 * d [4][128][N] fp32 (one product per combination, in the order
 * (A K-major, B K-major), (A MN, B MN), (A K, B MN), (A MN, B K)).
 * N must be a multiple of 16 in [16, 256], K a multiple of 16 in [16, 128].
 * Synchronous (returns after the kernel finishes).
 */
kda_status_t kda_selftest_tcgen05(const void* a, const void* b, float* d, int32_t N, int32_t K,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
