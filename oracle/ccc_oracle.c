/*
 * ccc_oracle.c -- float64 CPU oracle of the packed, width-4, depthwise causal
 * Conv1d + SiLU, its conv_state pool update and its backward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA library and never calls it.
 *
 * What is computed (FlashInfer "flashinfer.mamba.causal_conv1d_fn",
 * Parameters and Notes; Megatron-Core "core.ssm.causal_conv1d",
 * assert_causal_conv1d_deterministic; FlashInfer
 * "cake_causal_conv1d_train.cake_causal_conv1d_kcp", description and Returns):
 *
 *   Sequence n owns packed rows [s, e) = [cu[n], cu[n+1]), len = e - s.
 *   Its history is h[0..len+3): h[0..3) is the initial state (conv_state
 *   positions 0:3 of slot cache[n] when has_init[n], else zeros) and
 *   h[3 + j] = x[s + j].  For every token j of the sequence and channel c
 *
 *       z_j = b_c + w_c0*h[j] + w_c1*h[j+1] + w_c2*h[j+2] + w_c3*h[j+3]
 *       y_j = z_j / (1 + exp(-z_j))                (SiLU)
 *
 *   so tap 3 multiplies the current token and the bias is added first.
 *   cache[n] == -1 gives an all-zero output and no state access.  Rows after
 *   cu[N] are not written.  A nonempty live sequence writes h[len..len+3),
 *   its final three raw history values, to state positions 0:3 of its slot.
 *
 *   Backward, for an upstream gradient dy (and optionally d_final, the
 *   gradient of the three state values the forward wrote):
 *
 *       sig_j = 1 / (1 + exp(-z_j))
 *       dz_j  = dy_j * sig_j * (1 + z_j * (1 - sig_j))
 *       dH[i] = [i >= len] d_final[i - len] + sum_{k=0..3, 0<=i-k<len} w_ck dz_{i-k}
 *       dx[s + i - 3] = dH[i]  (i >= 3),   d_init[i] = dH[i]  (i < 3)
 *       dweight[c][k] = sum_n sum_j dz_j h[j + k],   dbias[c] = sum_n sum_j dz_j
 *
 *   The sums of dH are taken in the order written (carry first, then
 *   k = 0, 1, 2, 3); the same order in the GPU kernels makes a sequence
 *   split into fragments reproduce the unsplit result.
 *
 * Readings where the pages are silent (each one listed with its reason in
 * the design notes): state position 0 is the oldest history value; for
 * len < 3 the final state mixes initial history and x; a -1 request has zero
 * gradient and d_init = 0; d_init is zero for a sequence that did not read
 * state (has_init false) and for empty sequences; dx rows after cu[N] are not
 * written.
 *
 * All BF16 inputs are widened exactly to double.  The output arrays are
 * double; the caller rounds them to FP32 for comparison.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact BF16 -> double: a BF16 value is the upper half of an IEEE binary32. */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Raw BF16 bits of history value i of (sequence n, channel c). */
static uint16_t hist_bits(const uint16_t *init3, const uint16_t *x, int64_t x_stride,
                          int64_t s, int32_t c, int64_t i) {
    if (i < 3) return init3[i];
    return x[(s + i - 3) * x_stride + c];
}

/*
 * Forward.  state: contiguous [n_slots][C][L] BF16 pool or NULL (zero history,
 * no write-back).  cache: [N] or NULL (only allowed without a pool: all
 * sequences live).  has_init: [N] bytes or NULL (all false).  out: [rows][C]
 * doubles, only rows of sequences written.  hist (optional): [N][3][C] BF16,
 * the initial history each nonempty sequence used (zeros for -1 requests).
 * Returns 0, or -1 on an invalid slot.
 */
int oracle_fwd(const uint16_t *x, int64_t rows, int32_t C, int64_t x_stride,
               const double *w, const double *bias,
               uint16_t *state, int32_t n_slots, int32_t L,
               const int32_t *cu, int32_t N,
               const int32_t *cache, const uint8_t *has_init,
               double *out, int64_t out_stride, uint16_t *hist) {
    (void)rows;
    if (state && !cache) return -1;
    for (int32_t n = 0; state && n < N; ++n)
        if (cache[n] != -1 && (cache[n] < 0 || cache[n] >= n_slots)) return -1;
#pragma omp parallel for schedule(static)
    for (int32_t c = 0; c < C; ++c) {
        const double b = bias ? bias[c] : 0.0;
        const double w0 = w[4 * c + 0], w1 = w[4 * c + 1];
        const double w2 = w[4 * c + 2], w3 = w[4 * c + 3];
        for (int32_t n = 0; n < N; ++n) {
            const int64_t s = cu[n], e = cu[n + 1], len = e - s;
            const int32_t q = state ? cache[n] : 0;
            if (state && q == -1) {
                /* -1: zero output, no state access. */
                for (int64_t j = 0; j < len; ++j) out[(s + j) * out_stride + c] = 0.0;
                if (hist && len > 0)
                    for (int i = 0; i < 3; ++i) hist[((int64_t)n * 3 + i) * C + c] = 0;
                continue;
            }
            uint16_t init3[3] = {0, 0, 0};
            if (state && has_init && has_init[n])
                for (int i = 0; i < 3; ++i)
                    init3[i] = state[((int64_t)q * C + c) * L + i];
            if (hist && len > 0)
                for (int i = 0; i < 3; ++i) hist[((int64_t)n * 3 + i) * C + c] = init3[i];
            for (int64_t j = 0; j < len; ++j) {
                const double h0 = bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + 0));
                const double h1 = bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + 1));
                const double h2 = bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + 2));
                const double h3 = bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + 3));
                double z = b;
                z += w0 * h0;
                z += w1 * h1;
                z += w2 * h2;
                z += w3 * h3;
                out[(s + j) * out_stride + c] = silu(z);
            }
            if (state && len > 0) {
                /* Final three raw history values h[len], h[len+1], h[len+2]. */
                uint16_t fin[3];
                for (int i = 0; i < 3; ++i) fin[i] = hist_bits(init3, x, x_stride, s, c, len + i);
                for (int i = 0; i < 3; ++i) state[((int64_t)q * C + c) * L + i] = fin[i];
            }
        }
    }
    return 0;
}

/*
 * Backward.  hist: [N][3][C] BF16 initial history (as written by the
 * forward) or NULL (zero history).  cache: [N] or NULL (all live).
 * has_init: [N] or NULL (all false; then d_init = 0).  d_final: [N][3][C] or
 * NULL.  dx: [rows][C] doubles, rows of sequences written.  dweight [C][4],
 * dbias [C] (overwritten).  d_init: [N][3][C] or NULL.  abs_dweight [C][4] and
 * abs_dbias [C] (optional) receive the sums of |term|, the conditioning of
 * each reduction.
 */
int oracle_bwd(const uint16_t *x, int64_t rows, int32_t C, int64_t x_stride,
               const double *w, const double *bias, const uint16_t *hist,
               const int32_t *cu, int32_t N, const int32_t *cache,
               const uint8_t *has_init, const uint16_t *dy, int64_t dy_stride,
               const double *d_final, double *dx, int64_t dx_stride,
               double *dweight, double *dbias, double *d_init,
               double *abs_dweight, double *abs_dbias) {
    (void)rows;
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
            double wk[4];
            for (int k = 0; k < 4; ++k) wk[k] = w[4 * c + k];
            double dw[4] = {0, 0, 0, 0}, db = 0.0;
            double adw[4] = {0, 0, 0, 0}, adb = 0.0;
            for (int32_t n = 0; n < N; ++n) {
                const int64_t s = cu[n], e = cu[n + 1], len = e - s;
                const int live = !(cache && cache[n] == -1);
                if (!live || len == 0) {
                    for (int64_t j = 0; j < len; ++j) dx[(s + j) * dx_stride + c] = 0.0;
                    if (d_init)
                        for (int i = 0; i < 3; ++i) d_init[((int64_t)n * 3 + i) * C + c] = 0.0;
                    continue;
                }
                uint16_t init3[3] = {0, 0, 0};
                if (hist)
                    for (int i = 0; i < 3; ++i) init3[i] = hist[((int64_t)n * 3 + i) * C + c];
                /* Recompute the pre-activation and form dz. */
                for (int64_t j = 0; j < len; ++j) {
                    double zz = b;
                    for (int k = 0; k < 4; ++k)
                        zz += wk[k] * bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + k));
                    const double sg = sigmoid(zz);
                    const double g = bf16_to_f64(dy[(s + j) * dy_stride + c]);
                    dz[j] = g * sg * (1.0 + zz * (1.0 - sg));
                }
                /* Gradient of every history value, carry first, k ascending. */
                for (int64_t i = 0; i < len + 3; ++i) {
                    double acc = 0.0;
                    if (i >= len && d_final) acc = d_final[((int64_t)n * 3 + (i - len)) * C + c];
                    for (int k = 0; k < 4; ++k) {
                        const int64_t j = i - k;
                        if (j >= 0 && j < len) acc += wk[k] * dz[j];
                    }
                    if (i >= 3) {
                        dx[(s + i - 3) * dx_stride + c] = acc;
                    } else if (d_init) {
                        const int read_state = has_init && has_init[n];
                        d_init[((int64_t)n * 3 + i) * C + c] = read_state ? acc : 0.0;
                    }
                }
                /* Weight and bias gradients. */
                for (int64_t j = 0; j < len; ++j) {
                    for (int k = 0; k < 4; ++k) {
                        const double t = dz[j] * bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + k));
                        dw[k] += t;
                        adw[k] += fabs(t);
                    }
                    db += dz[j];
                    adb += fabs(dz[j]);
                }
            }
            for (int k = 0; k < 4; ++k) dweight[4 * c + k] = dw[k];
            dbias[c] = db;
            if (abs_dweight)
                for (int k = 0; k < 4; ++k) abs_dweight[4 * c + k] = adw[k];
            if (abs_dbias) abs_dbias[c] = adb;
        }
        free(dz);
    }
    return bad;
}
