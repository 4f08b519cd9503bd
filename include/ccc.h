/*
 * ccc.h -- C ABI of the GB300 (sm_103a) packed, width-4, depthwise causal
 * Conv1d + SiLU ("ccc"): forward with in-place conv_state pool update, the
 * fused backward with a deterministic FP32 weight/bias gradient, and the
 * speculative / single-token decode update of the pool.  Widths 2 and 3 and
 * the no-activation variant are served by the same entry points.
 *
 * The operation (FlashInfer "flashinfer.mamba.causal_conv1d_fn", Parameters
 * and Notes): sequence n owns the packed rows [cu_seqlens[n], cu_seqlens[n+1])
 * of x.  Its history h is three initial values followed by its raw inputs;
 * the initial values are conv_state positions 0:3 of slot cache_indices[n]
 * when has_initial_state[n] is true, zeros otherwise.  For token j and
 * channel c, with FP32 accumulation,
 *
 *     z = bias[c] + w[c][0]*h[j] + w[c][1]*h[j+1] + w[c][2]*h[j+2] + w[c][3]*h[j+3]
 *     out[j][c] = BF16_rne( z * sigmoid(z) )
 *
 * (tap 3 acts on the current token; the sum starts from the bias and the
 * four FMAs follow in the order k = 0, 1, 2, 3).  cache_indices[n] == -1
 * produces a zero output and no state access.  A live sequence with at
 * least one token leaves the last three inputs of its history (unactivated)
 * in its slot at positions 0, 1, 2, oldest first; nothing else in the pool
 * changes.  Rows after
 * cu_seqlens[N] are never written.
 *
 * The backward (FlashInfer "cake_causal_conv1d_train.cake_causal_conv1d_kcp",
 * Returns: dx from one fused kernel, the weight gradient in FP32 with a
 * run-to-run identical result) recomputes z, forms
 * dz = dy * s * (1 + z * (1 - s)) with s = sigmoid(z), and gives
 *
 *     dH[i] = carry + w[c][0]*dz[i] + w[c][1]*dz[i-1] + w[c][2]*dz[i-2] + w[c][3]*dz[i-3]
 *
 * for every history index i (terms with an index outside the sequence are
 * absent; carry = d_final_state[n][i-len] for the three indices past the end,
 * else 0), dx = dH for the input rows, d_init_state = dH for the three initial
 * values, and dweight[c][k] = sum of dz[j]*h[j+k], dbias[c] = sum of dz[j]
 * over all live tokens.  The weight/bias sums use per-run FP32 partials in
 * workspace combined by a reduction in a fixed order, never atomics (Megatron-Core
 * "core.ssm.causal_conv1d", assert_causal_conv1d_deterministic), so repeated
 * calls with the same arguments match bit for bit.
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer.  The library allocates nothing, keeps no
 *    state between calls, never synchronizes the host and never reads device
 *    values on the host (Notes of causal_conv1d_fn: graph-capturable).  Work is
 *    enqueued on `cuda_stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Device pointers are marked [dev]; sizes are in elements unless stated.
 *  - BF16 tensors are raw IEEE bfloat16 (uint16 storage).
 *  - All checks are host-side.  A failed check returns a negative ccc_status
 *    and enqueues nothing.  Device-side values (offsets, slot IDs, flags) are
 *    caller-owned constraints: if invalid, the results are undefined, but
 *    the kernels clamp offsets to [0, rows] and skip slot IDs outside
 *    [0, n_slots), so they do not access memory outside the buffers given.
 *  - rows == 0 or N == 0 returns CCC_OK with no row read or written (with
 *    rows == 0 the row buffers x, out, dy and dx may be NULL); the backward
 *    still zeroes dweight, dbias and d_init_state.
 *  - Concurrent calls on different streams need disjoint live slots, outputs
 *    and workspaces.
 */
#ifndef CCC_H_
#define CCC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { CCC_F32 = 0, CCC_BF16 = 1, CCC_NONE = -1 } ccc_dtype;

/* Activation after the convolution (Megatron-Core "core.ssm.causal_conv1d",
 * causal_conv1d_cp: the caller may ask for an activation or none). */
typedef enum { CCC_ACT_NONE = 0, CCC_ACT_SILU = 1 } ccc_activation;

typedef enum {
    CCC_OK = 0,
    CCC_ERR_NULL = -1,      /* a required pointer is NULL */
    CCC_ERR_SHAPE = -2,     /* a size or stride is invalid (C % 8, state_len < W-1, width, activation, ...) */
    CCC_ERR_DTYPE = -3,     /* unknown dtype code, or a dtype code without its buffer */
    CCC_ERR_ALIGN = -4,     /* x/out/dy/dx/saved_hist not 16-byte aligned, or misaligned element pointers */
    CCC_ERR_WORKSPACE = -5, /* workspace NULL or smaller than ccc_workspace_size() */
    CCC_ERR_ALIAS = -6,     /* an output overlaps another operand */
    CCC_ERR_CUDA = -7       /* a CUDA launch failed (cudaGetLastError after launch) */
} ccc_status;

/*
 * Bytes of device scratch ("workspace") that ccc_fwd (for_bwd = 0) or ccc_bwd
 * (for_bwd != 0) needs for `rows` packed rows, `n_seqs` sequences and
 * `channels` channels.  Pure host arithmetic; no CUDA call.
 *
 * Forward: always 0.  The kernels split the valid rows into runs (equal rows
 * in the forward; equal rows plus a fixed cost per sequence in the backward)
 * and find each run's first sequence themselves, on every call (the role of
 * the chunk map of causal_conv1d_fn, workspace), so no scratch is needed.
 * Backward: the FP32 partial sums of the ordered weight/bias reduction,
 * R x 5 x C floats (rounded up to 256 bytes) with R = min(1216 / ceil(C /
 * 256), ceil(rows / 16)), at least 1 -- so at most max(6,225,920, 20 x C)
 * bytes, and less for small batches.  The value depends only on `rows` and
 * `channels` (0 for invalid sizes or an empty batch), never on device values,
 * so a workspace sized once for a shape can be reused (and captured in a CUDA
 * graph); one sized for more rows also serves fewer.
 */
size_t ccc_workspace_size(int64_t rows, int32_t n_seqs, int32_t channels, int32_t for_bwd);

/*
 * Forward (causal_conv1d_fn).
 *
 *  x            [dev] BF16 [rows][x_row_stride], channels contiguous; 16-byte
 *               aligned; x_row_stride >= C, a multiple of 8.  Rows after
 *               cu_seqlens[N] may be padding.
 *  rows, C      C > 0 and a multiple of 8 (cake_causal_conv1d_kcp, x_local).
 *  weight       [dev] [C][width] contiguous, w_dtype CCC_F32 or CCC_BF16.
 *  width        taps W: 4 (causal_conv1d_fn), or 2 or 3 (causal_conv1d_cp,
 *               weight [D, W]).  Everything written "3" below is W - 1: the
 *               history rows, the state positions read and written, the rows
 *               of saved_hist / d_final_state / d_init_state.
 *  bias         [dev] [C] with b_dtype CCC_F32/CCC_BF16, or NULL with
 *               b_dtype CCC_NONE.
 *  activation   CCC_ACT_SILU (causal_conv1d_fn) or CCC_ACT_NONE (out = z).
 *  conv_state   [dev] BF16 pool, in place, or NULL (zero history, no
 *               write-back).  Element (slot, c, l) is at
 *               st_slot*slot + st_c*c + st_l*l; st_c == 1 or st_l == 1; slots
 *               must not overlap; state_len >= W - 1; n_slots >= 1.
 *  cu_seqlens   [dev] int32 [N+1]: 0, nondecreasing, cu_seqlens[N] <= rows.
 *  cache_indices[dev] int32 [N] slot per sequence, -1 = zero output and no
 *               state access.  Required with a pool; optional without (then
 *               only the -1 rule applies).  Live slots unique, in [0, n_slots).
 *  has_initial_state [dev] uint8/bool [N] or NULL (= all false).
 *  out          [dev] BF16 [rows][out_row_stride], 16-byte aligned, must not
 *               overlap any operand.  Rows after cu_seqlens[N] are not written.
 *  saved_hist   [dev] BF16 [N][3][C] or NULL.  When given, every nonempty
 *               sequence's initial history (what the forward read before it
 *               overwrote the slot; zeros for a -1 request) is stored, for
 *               ccc_bwd.  Rows of empty sequences are not written.
 *  workspace    unused (ccc_workspace_size(..., 0) is 0); may be NULL.
 */
int ccc_fwd(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
            const void *weight, int32_t w_dtype, int32_t width,
            const void *bias, int32_t b_dtype, int32_t activation,
            void *conv_state, int32_t n_slots, int32_t state_len,
            int64_t st_slot, int64_t st_c, int64_t st_l,
            const int32_t *cu_seqlens, int32_t N,
            const int32_t *cache_indices, const uint8_t *has_initial_state,
            void *out, int64_t out_row_stride,
            void *saved_hist,
            void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Backward (cake_causal_conv1d_kcp, Returns: dx from one fused pass and an
 * FP32 weight gradient that repeats bit for bit; core.ssm.causal_conv1d, _exchange_initial_states: the state
 * gradient is what a preceding fragment receives).
 *
 *  x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype,
 *               activation: as in ccc_fwd (the same values the forward saw).
 *               Without activation dz = dy.
 *  saved_hist   [dev] BF16 [N][3][C] from ccc_fwd, or NULL (zero history).
 *  cu_seqlens, N, cache_indices (NULL = all live), has_initial_state (NULL =
 *               all false): as in ccc_fwd.
 *  dy           [dev] BF16 [rows][dy_row_stride], gradient of out; rows after
 *               cu_seqlens[N] are ignored.
 *  d_final_state[dev] FP32 [N][3][C] or NULL: gradient of the three state
 *               values the forward wrote (position order), e.g. the
 *               d_init_state of the fragment that continued this one.
 *  dx           [dev] BF16 [rows][dx_row_stride]; rows after cu_seqlens[N] are
 *               not written; zero for -1 requests.
 *  dweight      [dev] FP32 [C][width], overwritten (not accumulated).
 *  dbias        [dev] FP32 [C] or NULL, overwritten.
 *  d_init_state [dev] FP32 [N][3][C] or NULL: gradient of the initial history
 *               for sequences that read their state (has_initial_state true,
 *               live, nonempty); 0 for every other sequence.
 *  workspace    [dev] >= ccc_workspace_size(rows, N, C, 1) bytes, 256-byte
 *               aligned.
 * Every buffer written must not overlap any other operand.
 */
int ccc_bwd(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
            const void *weight, int32_t w_dtype, int32_t width,
            const void *bias, int32_t b_dtype, int32_t activation,
            const void *saved_hist,
            const int32_t *cu_seqlens, int32_t N,
            const int32_t *cache_indices, const uint8_t *has_initial_state,
            const void *dy, int64_t dy_row_stride,
            const float *d_final_state,
            void *dx, int64_t dx_row_stride,
            float *dweight, float *dbias, float *d_init_state,
            void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Launch options of ccc_fwd_ex / ccc_bwd_ex / ccc_update_ex (ccc_fwd,
 * ccc_bwd and ccc_update are these with options = 0).  Library behaviour,
 * not part of the method.
 *
 * CCC_OPT_OVERLAP_PROLOGUE: launch the call's main kernel as a programmatic
 * dependent of the kernel enqueued just before it on the stream, so that
 * the kernel's prologue -- reading cu_seqlens, cache_indices,
 * has_initial_state, the weight and the bias, and splitting the rows into
 * runs -- can run while that previous kernel finishes.  The kernel then
 * waits for the previous kernel to complete (and its writes to be visible)
 * before it reads x, dy, conv_state, saved_hist or d_final_state, and before
 * it writes anything.  Contract: the kernel enqueued immediately before the
 * call on `cuda_stream` (in stream order, also inside a CUDA graph) must not
 * write cu_seqlens, cache_indices, has_initial_state (num_accepted for
 * ccc_update_ex), weight or bias.  This
 * holds in the usual step order -- the forward after the projection that
 * produces x, the backward after the kernel that produces dy or after this
 * library's forward, a forward after this library's backward -- but not,
 * e.g., right after a kernel that builds cu_seqlens on the device or an
 * optimizer step that updates these taps; leave the option off there.
 * Results are identical with and without it.  Unknown option bits return
 * CCC_ERR_SHAPE.
 */
enum { CCC_OPT_OVERLAP_PROLOGUE = 1 << 0 };

int ccc_fwd_ex(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
               const void *weight, int32_t w_dtype, int32_t width,
               const void *bias, int32_t b_dtype, int32_t activation,
               void *conv_state, int32_t n_slots, int32_t state_len,
               int64_t st_slot, int64_t st_c, int64_t st_l,
               const int32_t *cu_seqlens, int32_t N,
               const int32_t *cache_indices, const uint8_t *has_initial_state,
               void *out, int64_t out_row_stride,
               void *saved_hist,
               void *workspace, size_t workspace_bytes, uint32_t options, void *cuda_stream);

int ccc_bwd_ex(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
               const void *weight, int32_t w_dtype, int32_t width,
               const void *bias, int32_t b_dtype, int32_t activation,
               const void *saved_hist,
               const int32_t *cu_seqlens, int32_t N,
               const int32_t *cache_indices, const uint8_t *has_initial_state,
               const void *dy, int64_t dy_row_stride,
               const float *d_final_state,
               void *dx, int64_t dx_row_stride,
               float *dweight, float *dbias, float *d_init_state,
               void *workspace, size_t workspace_bytes, uint32_t options, void *cuda_stream);

/*
 * Backward without a workspace argument, for callers that cannot allocate
 * device memory (a host framework whose memory pool they cannot reach, a
 * plugin host that forbids device allocation after start-up, a latency-
 * critical path that cannot pay for cudaMalloc's possible device-wide
 * synchronization).  The pages have no counterpart: this is a library
 * convenience, not part of the method.
 *
 * Arguments, results and checks are those of ccc_bwd without `workspace` /
 * `workspace_bytes`.  The scratch is a fixed array of
 * CCC_NOALLOC_SCRATCH_BYTES compiled into the library, held by every GPU the
 * library is loaded on until the process exits; a shape whose
 * ccc_workspace_size(rows, N, C, 1) exceeds it returns CCC_ERR_WORKSPACE with
 * nothing enqueued (that size is at most max(6,225,920, 20 x C) bytes, so
 * every C up to 838,856 fits).  The first call in a CUDA context (normally
 * the device's primary context: once per device, and again after a device
 * reset) looks up the array's device address (cudaGetSymbolAddress) and
 * caches it under the context; make that first call before any stream
 * capture in the context.  All calls share the array and it keeps the last
 * call's contents (nothing in it needs to start at zero), so calls whose GPU
 * work overlaps (other streams, other host threads on the same device) race
 * and must be serialized by the caller.  Nothing is allocated and no
 * allocating routine is called.
 */
#define CCC_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

int ccc_bwd_noalloc(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
                    const void *weight, int32_t w_dtype, int32_t width,
                    const void *bias, int32_t b_dtype, int32_t activation,
                    const void *saved_hist,
                    const int32_t *cu_seqlens, int32_t N,
                    const int32_t *cache_indices, const uint8_t *has_initial_state,
                    const void *dy, int64_t dy_row_stride,
                    const float *d_final_state,
                    void *dx, int64_t dx_row_stride,
                    float *dweight, float *dbias, float *d_init_state,
                    void *cuda_stream);

/*
 * Speculative / single-token decode step (causal_conv1d_fn, Notes: the
 * speculative step that follows a prefill takes an accepted count of 1; the
 * pages define nothing more, so the rule below is this library's reading).
 *
 * Sequence n feeds len = cu_seqlens[n+1] - cu_seqlens[n] new tokens (1 for a
 * plain decode step, the draft tokens for a speculative one).  With
 * a = num_accepted[n] (1 when num_accepted is NULL) -- how many tokens of the
 * slot's previous step were kept -- the W-1 history values before the first
 * new token are conv_state positions a-1 .. a+W-3 of slot cache_indices[n];
 * each token's output is computed exactly as in ccc_fwd; then the step writes
 * history value h[p+1] to position p for p < min(len + W - 2, state_len)
 * (h = the W-1 values read, then the len new tokens), so the next step,
 * keeping a' of these tokens, reads positions a'-1 .. a'+W-3.  A prefill
 * (ccc_fwd) leaves exactly the state this rule expects for a = 1, and one
 * token with a = 1 is the ordinary shift-by-one decode update.  A -1 slot
 * gives zero output and no state access; an empty sequence leaves its slot
 * alone.  No workspace, one kernel launch.
 *
 *  x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype,
 *               activation, out, out_row_stride: as in ccc_fwd.
 *  conv_state   [dev] BF16 pool, required, same layout rules as ccc_fwd;
 *               state_len >= W - 1, and >= len + W - 2 for every position a
 *               later step may read to have been written.  A dense
 *               [slots][C][state_len] pool with state_len <= 8, or a
 *               channel-contiguous one, is moved in 16-byte vectors.
 *  cache_indices[dev] int32 [N], required; live slots unique, in
 *               [0, n_slots).
 *  num_accepted [dev] int32 [N] or NULL; values outside [1, state_len - W
 *               + 2] are clamped into it (caller-owned constraint).
 * Meant for short per-sequence lengths (one warp walks each sequence's
 * tokens); long prompts belong to ccc_fwd.
 */
int ccc_update(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
               const void *weight, int32_t w_dtype, int32_t width,
               const void *bias, int32_t b_dtype, int32_t activation,
               void *conv_state, int32_t n_slots, int32_t state_len,
               int64_t st_slot, int64_t st_c, int64_t st_l,
               const int32_t *cu_seqlens, int32_t N,
               const int32_t *cache_indices, const int32_t *num_accepted,
               void *out, int64_t out_row_stride, void *cuda_stream);

/* ccc_update with launch options (CCC_OPT_OVERLAP_PROLOGUE, above). */
int ccc_update_ex(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
                  const void *weight, int32_t w_dtype, int32_t width,
                  const void *bias, int32_t b_dtype, int32_t activation,
                  void *conv_state, int32_t n_slots, int32_t state_len,
                  int64_t st_slot, int64_t st_c, int64_t st_l,
                  const int32_t *cu_seqlens, int32_t N,
                  const int32_t *cache_indices, const int32_t *num_accepted,
                  void *out, int64_t out_row_stride, uint32_t options, void *cuda_stream);

/*
 * Device-side check of the caller-owned metadata.  The pages leave the
 * values in cu_seqlens, cache_indices (and, for the decode step,
 * num_accepted) unchecked: no host read, no validation synchronization
 * (causal_conv1d_fn, Notes), and invalid values are the caller's fault.
 * The kernels above never read or write outside the buffers they are given
 * whatever those values are (offsets are clamped to [0, rows], slot IDs
 * outside [0, n_slots) are skipped), but their results are then
 * meaningless.  This call finds such values on the device, still without a
 * host synchronization, for callers that want to check a batch (in tests,
 * or once per new batch layout).  The pages have no counterpart.
 *
 * It clears `status` and ORs into status[0] one CCC_CHECK_* bit per kind of
 * violation found (0: every value is valid); nothing traps.  The caller
 * reads status[0] after the stream reaches that point.
 *
 *  rows          rows of the packed x the metadata will be used with.
 *  cu_seqlens    [dev] int32 [N + 1], required.  Checked: cu[0] == 0,
 *                nondecreasing, every offset in [0, rows].
 *  cache_indices [dev] int32 [N] or NULL (not checked).  Checked: every
 *                value is -1 or in [0, n_slots); no live slot appears twice.
 *  num_accepted  [dev] int32 [N] or NULL (not checked).  Checked: every
 *                value in [1, max_accepted] (ccc_update: max_accepted =
 *                state_len - width + 2).
 *  status        [dev] uint32 [status_words], caller-owned, with
 *                status_words >= ccc_check_status_words(n_slots): word 0 is
 *                the result, the rest a bitmap of live slots (scratch).
 * Returns CCC_ERR_NULL / CCC_ERR_SHAPE / CCC_ERR_WORKSPACE (status too
 * small) / CCC_ERR_ALIAS with nothing enqueued; otherwise one memset and one
 * kernel launch on cuda_stream.
 */
enum {
    CCC_CHECK_CU_START = 1 << 0,   /* cu_seqlens[0] != 0 */
    CCC_CHECK_CU_ORDER = 1 << 1,   /* an offset smaller than the one before it */
    CCC_CHECK_CU_RANGE = 1 << 2,   /* an offset outside [0, rows] */
    CCC_CHECK_SLOT_RANGE = 1 << 3, /* a cache index outside [-1, n_slots) */
    CCC_CHECK_SLOT_DUP = 1 << 4,   /* a live slot used by two sequences */
    CCC_CHECK_ACCEPTED = 1 << 5    /* an accepted count outside [1, max_accepted] */
};

/* Words of the status array ccc_check needs: 1 + ceil(n_slots / 32). */
size_t ccc_check_status_words(int32_t n_slots);

int ccc_check(int64_t rows, const int32_t *cu_seqlens, int32_t N,
              const int32_t *cache_indices, int32_t n_slots,
              const int32_t *num_accepted, int32_t max_accepted,
              uint32_t *status, size_t status_words, void *cuda_stream);

/* Name of a ccc_status value ("CCC_OK", ...); "unknown" otherwise. */
const char *ccc_status_string(int status);

/* Number of kernel launches the last successful ccc_fwd / ccc_bwd /
 * ccc_update on this host thread enqueued (for launch accounting; memsets
 * not included). */
int ccc_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CCC_H_ */
