/*
 * ccc_oracle.c -- float64 CPU oracle of the packed depthwise causal Conv1d
 * (+ SiLU), its conv_state pool update, its backward and its speculative
 * decode state update.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA library and never calls it.
 *
 * What is computed (FlashInfer "flashinfer.mamba.causal_conv1d_fn",
 * Parameters and Notes; Megatron-Core "core.ssm.causal_conv1d", Parameters of
 * causal_conv1d_cp: weight [D, W], optional activation, and
 * assert_causal_conv1d_deterministic; FlashInfer
 * "cake_causal_conv1d_train.cake_causal_conv1d_kcp", description and Returns):
 *
 *   The width is W (4 in FlashInfer's contract; 2, 3 or 4 here) and H = W - 1
 *   is the length of the carried history.  Sequence n owns packed rows
 *   [s, e) = [cu[n], cu[n+1]), len = e - s.  Its history is h[0..len+H):
 *   h[0..H) is the initial state (conv_state positions 0:H of slot cache[n]
 *   when has_init[n], else zeros) and h[H + j] = x[s + j].  For every token
 *   j of the sequence and channel c
 *
 *       z_j = b_c + w_c0*h[j] + w_c1*h[j+1] + ... + w_c(W-1)*h[j+W-1]
 *       y_j = z_j / (1 + exp(-z_j))     (SiLU; y_j = z_j without activation)
 *
 *   so tap W-1 multiplies the current token and the bias is added first.
 *   cache[n] == -1 gives an all-zero output and no state access.  Rows after
 *   cu[N] are not written.  A nonempty live sequence writes h[len..len+H),
 *   its final H raw history values, to state positions 0:H of its slot.
 *
 *   Backward, for an upstream gradient dy (and optionally d_final, the
 *   gradient of the H state values the forward wrote):
 *
 *       sig_j = 1 / (1 + exp(-z_j))
 *       dz_j  = dy_j * sig_j * (1 + z_j * (1 - sig_j))    (dz_j = dy_j without activation)
 *       dH[i] = [i >= len] d_final[i - len] + sum_{k=0..W-1, 0<=i-k<len} w_ck dz_{i-k}
 *       dx[s + i - H] = dH[i]  (i >= H),   d_init[i] = dH[i]  (i < H)
 *       dweight[c][k] = sum_n sum_j dz_j h[j + k],   dbias[c] = sum_n sum_j dz_j
 *
 *   The sums of dH are taken in the order written (carry first, then
 *   k = 0, 1, ..., W-1); the same order in the GPU kernels makes a sequence
 *   split into fragments reproduce the unsplit result.
 *
 *   Speculative state update (causal_conv1d_fn, Notes: the speculative
 *   step right after a prefill is given an accepted count of one).  Each step feeds
 *   len >= 1 draft tokens per sequence; a = accepted[n] >= 1 says how many
 *   tokens of the previous step were kept.  Reading: the slot keeps a run of
 *   raw history values in time order, and the previous step left its
 *   h[p + 1] at position p, so the H values before this step's first token
 *   are positions a-1 .. a+H-2.  The step computes z and y as above from
 *   h[0..H) = state[a-1 .. a+H-1) and h[H + j] = x[s + j], then writes
 *   h[p + 1] to position p for p < min(len + H - 1, L): whatever a' in
 *   1..len the next step brings, positions a'-1 .. a'+H-2 then hold the H
 *   values that end at the last kept token.  A prefill leaves its last H
 *   values at positions 0:H, which is that rule's state for a = 1.
 *
 * Readings where the pages are silent (each one listed with its reason in
 * the design notes): state position 0 is the oldest history value; for
 * len < H the final state mixes initial history and x; a -1 request has zero
 * gradient and d_init = 0; d_init is zero for a sequence that did not read
 * state (has_init false) and for empty sequences; dx rows after cu[N] are not
 * written; the speculative update rule above.
 *
 * All BF16 inputs are widened exactly to double.  The output arrays are
 * double; the caller rounds them to FP32 for comparison.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MAX_W 4

/* Exact BF16 -> double: a BF16 value is the upper half of an IEEE binary32. */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* The activation: SiLU (act != 0) or none. */
static double activate(double z, int act) { return act ? z / (1.0 + exp(-z)) : z; }

/* g times d activate / dz at z. */
static double activate_grad(double z, double g, int act) {
    if (!act) return g;
    const double sg = sigmoid(z);
    return g * sg * (1.0 + z * (1.0 - sg));
}

/* Raw BF16 bits of history value i of (sequence n, channel c). */
static uint16_t hist_bits(const uint16_t *init, int H, const uint16_t *x, int64_t x_stride,
                          int64_t s, int32_t c, int64_t i) {
    if (i < H) return init[i];
    return x[(s + i - H) * x_stride + c];
}

/* Pre-activation of token j: the bias, then the W taps in order k = 0..W-1. */
static double pre_activation(double b, const double *wk, int W, const uint16_t *init,
                             const uint16_t *x, int64_t x_stride, int64_t s, int32_t c, int64_t j) {
    double z = b;
    for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(hist_bits(init, W - 1, x, x_stride, s, c, j + k));
    return z;
}

static int width_ok(int W) { return W >= 2 && W <= MAX_W; }

/*
 * Forward.  w: [C][W] taps.  state: contiguous [n_slots][C][L] BF16 pool or
 * NULL (zero history, no write-back).  cache: [N] slot IDs, required with a
 * pool; optional without one (NULL: all sequences live), where only its -1
 * entries matter: a -1 request outputs zeros with or without a pool.
 * has_init: [N] bytes or NULL (all false; ignored without a pool).  out:
 * [rows][C] doubles, only rows of sequences written.  hist (optional):
 * [N][W-1][C] BF16, the initial history each nonempty sequence used (zeros
 * for -1 requests).  act: 1 = SiLU, 0 = none.  Returns 0, or -1 on an
 * invalid argument.
 */
int oracle_fwd(const uint16_t *x, int64_t rows, int32_t C, int64_t x_stride,
               const double *w, int32_t W, const double *bias, int32_t act,
               uint16_t *state, int32_t n_slots, int32_t L,
               const int32_t *cu, int32_t N,
               const int32_t *cache, const uint8_t *has_init,
               double *out, int64_t out_stride, uint16_t *hist) {
    (void)rows;
    if (!width_ok(W)) return -1;
    const int H = W - 1;
    if (state && (!cache || L < H)) return -1;
    for (int32_t n = 0; state && n < N; ++n)
        if (cache[n] != -1 && (cache[n] < 0 || cache[n] >= n_slots)) return -1;
#pragma omp parallel for schedule(static)
    for (int32_t c = 0; c < C; ++c) {
        const double b = bias ? bias[c] : 0.0;
        const double *wk = w + (int64_t)W * c;
        for (int32_t n = 0; n < N; ++n) {
            const int64_t s = cu[n], e = cu[n + 1], len = e - s;
            const int32_t q = cache ? cache[n] : 0;
            if (cache && q == -1) {
                /* -1: zero output, no state access. */
                for (int64_t j = 0; j < len; ++j) out[(s + j) * out_stride + c] = 0.0;
                if (hist && len > 0)
                    for (int i = 0; i < H; ++i) hist[((int64_t)n * H + i) * C + c] = 0;
                continue;
            }
            uint16_t init[MAX_W - 1] = {0, 0, 0};
            if (state && has_init && has_init[n])
                for (int i = 0; i < H; ++i) init[i] = state[((int64_t)q * C + c) * L + i];
            if (hist && len > 0)
                for (int i = 0; i < H; ++i) hist[((int64_t)n * H + i) * C + c] = init[i];
            for (int64_t j = 0; j < len; ++j)
                out[(s + j) * out_stride + c] =
                    activate(pre_activation(b, wk, W, init, x, x_stride, s, c, j), act);
            if (state && len > 0) {
                /* Final H raw history values h[len .. len+H). */
                uint16_t fin[MAX_W - 1];
                for (int i = 0; i < H; ++i) fin[i] = hist_bits(init, H, x, x_stride, s, c, len + i);
                for (int i = 0; i < H; ++i) state[((int64_t)q * C + c) * L + i] = fin[i];
            }
        }
    }
    return 0;
}

/*
 * Backward.  hist: [N][W-1][C] BF16 initial history (as written by the
 * forward) or NULL (zero history).  cache: [N] or NULL (all live).
 * has_init: [N] or NULL (all false; then d_init = 0).  d_final: [N][W-1][C]
 * or NULL.  dx: [rows][C] doubles, rows of sequences written.  dweight
 * [C][W], dbias [C] (overwritten).  d_init: [N][W-1][C] or NULL.
 * abs_dweight [C][W] and abs_dbias [C] (optional) receive the sums of
 * |term|, the conditioning of each reduction.  Returns 0, or -1 on an
 * invalid argument or a failed allocation.
 */
int oracle_bwd(const uint16_t *x, int64_t rows, int32_t C, int64_t x_stride,
               const double *w, int32_t W, const double *bias, int32_t act,
               const uint16_t *hist,
               const int32_t *cu, int32_t N, const int32_t *cache,
               const uint8_t *has_init, const uint16_t *dy, int64_t dy_stride,
               const double *d_final, double *dx, int64_t dx_stride,
               double *dweight, double *dbias, double *d_init,
               double *abs_dweight, double *abs_dbias) {
    (void)rows;
    if (!width_ok(W)) return -1;
    const int H = W - 1;
    int64_t max_len = 0;
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] - cu[n] > max_len) max_len = cu[n + 1] - cu[n];
    int bad = 0;
#pragma omp parallel
    {
        double *dz = (double *)malloc(sizeof(double) * (size_t)(max_len + 1));
        if (!dz) bad = -1;
#pragma omp for schedule(static)
        for (int32_t c = 0; c < C; ++c) {
            if (!dz) continue;
            const double b = bias ? bias[c] : 0.0;
            const double *wk = w + (int64_t)W * c;
            double dw[MAX_W] = {0, 0, 0, 0}, db = 0.0;
            double adw[MAX_W] = {0, 0, 0, 0}, adb = 0.0;
            for (int32_t n = 0; n < N; ++n) {
                const int64_t s = cu[n], e = cu[n + 1], len = e - s;
                const int live = !(cache && cache[n] == -1);
                if (!live || len == 0) {
                    for (int64_t j = 0; j < len; ++j) dx[(s + j) * dx_stride + c] = 0.0;
                    if (d_init)
                        for (int i = 0; i < H; ++i) d_init[((int64_t)n * H + i) * C + c] = 0.0;
                    continue;
                }
                uint16_t init[MAX_W - 1] = {0, 0, 0};
                if (hist)
                    for (int i = 0; i < H; ++i) init[i] = hist[((int64_t)n * H + i) * C + c];
                /* Recompute the pre-activation and form dz. */
                for (int64_t j = 0; j < len; ++j) {
                    const double zz = pre_activation(b, wk, W, init, x, x_stride, s, c, j);
                    dz[j] = activate_grad(zz, bf16_to_f64(dy[(s + j) * dy_stride + c]), act);
                }
                /* Gradient of every history value, carry first, k ascending. */
                for (int64_t i = 0; i < len + H; ++i) {
                    double acc = 0.0;
                    if (i >= len && d_final) acc = d_final[((int64_t)n * H + (i - len)) * C + c];
                    for (int k = 0; k < W; ++k) {
                        const int64_t j = i - k;
                        if (j >= 0 && j < len) acc += wk[k] * dz[j];
                    }
                    if (i >= H) {
                        dx[(s + i - H) * dx_stride + c] = acc;
                    } else if (d_init) {
                        const int read_state = has_init && has_init[n];
                        d_init[((int64_t)n * H + i) * C + c] = read_state ? acc : 0.0;
                    }
                }
                /* Weight and bias gradients. */
                for (int64_t j = 0; j < len; ++j) {
                    for (int k = 0; k < W; ++k) {
                        const double t = dz[j] * bf16_to_f64(hist_bits(init, H, x, x_stride, s, c, j + k));
                        dw[k] += t;
                        adw[k] += fabs(t);
                    }
                    db += dz[j];
                    adb += fabs(dz[j]);
                }
            }
            for (int k = 0; k < W; ++k) dweight[(int64_t)W * c + k] = dw[k];
            dbias[c] = db;
            if (abs_dweight)
                for (int k = 0; k < W; ++k) abs_dweight[(int64_t)W * c + k] = adw[k];
            if (abs_dbias) abs_dbias[c] = adb;
        }
        free(dz);
    }
    return bad;
}

/*
 * Speculative / single-token state update (see the header).  state:
 * contiguous [n_slots][C][L] BF16 pool, read at positions accepted[n]-1 ..
 * accepted[n]+W-3 and updated in place; cache: [N] slot IDs, -1 = zero output
 * and no state access; accepted: [N] or NULL (all 1).  out: [rows][C]
 * doubles, rows of sequences written.  Returns 0, or -1 on an invalid
 * argument (accepted must lie in [1, L - W + 2]).
 */
int oracle_update(const uint16_t *x, int64_t rows, int32_t C, int64_t x_stride,
                  const double *w, int32_t W, const double *bias, int32_t act,
                  uint16_t *state, int32_t n_slots, int32_t L,
                  const int32_t *cu, int32_t N,
                  const int32_t *cache, const int32_t *accepted,
                  double *out, int64_t out_stride) {
    (void)rows;
    if (!width_ok(W)) return -1;
    const int H = W - 1;
    if (!state || !cache || L < H) return -1;
    for (int32_t n = 0; n < N; ++n) {
        if (cache[n] != -1 && (cache[n] < 0 || cache[n] >= n_slots)) return -1;
        if (accepted && (accepted[n] < 1 || accepted[n] > L - H + 1)) return -1;
    }
    int64_t max_len = 0;
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] - cu[n] > max_len) max_len = cu[n + 1] - cu[n];
    int bad = 0;
#pragma omp parallel
    {
        /* The whole history of one (sequence, channel): H state values, then x. */
        uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(max_len + H));
        if (!h) bad = -1;
#pragma omp for schedule(static)
        for (int32_t c = 0; c < C; ++c) {
            if (!h) continue;
            const double b = bias ? bias[c] : 0.0;
            const double *wk = w + (int64_t)W * c;
            for (int32_t n = 0; n < N; ++n) {
                const int64_t s = cu[n], e = cu[n + 1], len = e - s;
                const int32_t q = cache[n];
                if (q == -1) {
                    for (int64_t j = 0; j < len; ++j) out[(s + j) * out_stride + c] = 0.0;
                    continue;
                }
                if (len == 0) continue;
                const int32_t a = accepted ? accepted[n] : 1;
                uint16_t *slot = state + ((int64_t)q * C + c) * L;
                for (int i = 0; i < H; ++i) h[i] = slot[a - 1 + i];
                for (int64_t j = 0; j < len; ++j) h[H + j] = x[(s + j) * x_stride + c];
                for (int64_t j = 0; j < len; ++j) {
                    double z = b;
                    for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(h[j + k]);
                    out[(s + j) * out_stride + c] = activate(z, act);
                }
                for (int64_t p = 0; p < len + H - 1 && p < L; ++p) slot[p] = h[p + 1];
            }
        }
        free(h);
    }
    return bad;
}
