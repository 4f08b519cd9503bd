// ccc_api.cu -- the C ABI declared in include/ccc.h: host-side argument
// checks, workspace carve-up and kernel launches.  No device value is read on
// the host and nothing synchronizes (FlashInfer
// "flashinfer.mamba.causal_conv1d_fn", Notes), so every call can be captured
// in a CUDA graph once out and workspace are supplied.
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "ccc.h"
#include "ccc_internal.h"

namespace {

using ccc::ceil_div;

thread_local int g_last_launches = 0;

constexpr size_t kAlignWs = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte span [lo, hi) of a buffer, or empty.
struct Span {
    uintptr_t lo = 0, hi = 0;
    bool empty() const { return hi <= lo; }
};

Span span(const void *p, size_t bytes) {
    Span s;
    if (p && bytes) {
        s.lo = reinterpret_cast<uintptr_t>(p);
        s.hi = s.lo + bytes;
    }
    return s;
}

bool overlap(const Span &a, const Span &b) {
    return !a.empty() && !b.empty() && a.lo < b.hi && b.lo < a.hi;
}

// Rows of a [rows][stride] BF16 matrix with C used columns, in bytes.
size_t mat_bytes(int64_t rows, int64_t stride, int C) {
    return rows > 0 ? static_cast<size_t>(((rows - 1) * stride + C) * 2) : 0;
}

int dtype_size(int code) { return code == CCC_F32 ? 4 : (code == CCC_BF16 ? 2 : 0); }

bool width_ok(int width) { return width >= 2 && width <= 4; }

bool activation_ok(int act) { return act == CCC_ACT_NONE || act == CCC_ACT_SILU; }

// Pool layout check: strides non-negative, channel or history axis
// contiguous, and distinct (slot, c, l) never share an element (sorted-stride
// criterion: each stride exceeds the span of the smaller dimensions).
bool state_layout_ok(int n_slots, int C, int L, int64_t s_slot, int64_t s_c, int64_t s_l) {
    if (s_slot < 0 || s_c < 0 || s_l < 0) return false;
    if (s_c != 1 && s_l != 1) return false;
    struct D { int64_t stride, extent; } d[3] = {{s_slot, n_slots}, {s_c, C}, {s_l, L}};
    std::sort(d, d + 3, [](const D &a, const D &b) { return a.stride < b.stride; });
    int64_t span_below = 0;
    for (const D &e : d) {
        if (e.extent > 1 && e.stride <= span_below) return false;
        span_below += (e.extent - 1) * e.stride;
    }
    return true;
}

// Per-device launch facts, queried once per device (host calls, no sync).
// They are properties of the hardware and the compiled kernel, so they stay
// valid across device resets and contexts.
struct DeviceFacts {
    int sms = 0;
    int fwd_ctas = 0;
};

DeviceFacts device_facts() {
    static std::mutex mu;
    static DeviceFacts cached[64];
    static const DeviceFacts fallback{152, ccc::kFwdMinBlocks};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fallback;
    std::lock_guard<std::mutex> lock(mu);
    DeviceFacts &f = cached[dev];
    if (f.sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        f.fwd_ctas = ccc::fwd_ctas_per_sm();
        f.sms = n;
    }
    return f;
}

}  // namespace

extern "C" {

size_t ccc_workspace_size(int64_t rows, int32_t n_seqs, int32_t channels, int32_t for_bwd) {
    if (rows < 0 || n_seqs < 0 || channels <= 0 || channels % 8) return 0;
    if (rows == 0 || n_seqs == 0) return 0;
    if (!for_bwd) return 0;  // the forward splits its work in-kernel: no scratch
    const int R = ccc::bwd_runs(rows, channels);
    return round_up(static_cast<size_t>(R) * 5 * channels * sizeof(float), kAlignWs);
}

const char *ccc_status_string(int status) {
    switch (status) {
        case CCC_OK: return "CCC_OK";
        case CCC_ERR_NULL: return "CCC_ERR_NULL";
        case CCC_ERR_SHAPE: return "CCC_ERR_SHAPE";
        case CCC_ERR_DTYPE: return "CCC_ERR_DTYPE";
        case CCC_ERR_ALIGN: return "CCC_ERR_ALIGN";
        case CCC_ERR_WORKSPACE: return "CCC_ERR_WORKSPACE";
        case CCC_ERR_ALIAS: return "CCC_ERR_ALIAS";
        case CCC_ERR_CUDA: return "CCC_ERR_CUDA";
        default: return "unknown";
    }
}

int ccc_last_launch_count(void) { return g_last_launches; }

int ccc_fwd(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
            const void *weight, int32_t w_dtype, int32_t width,
            const void *bias, int32_t b_dtype, int32_t activation,
            void *conv_state, int32_t n_slots, int32_t state_len,
            int64_t st_slot, int64_t st_c, int64_t st_l,
            const int32_t *cu_seqlens, int32_t N,
            const int32_t *cache_indices, const uint8_t *has_initial_state,
            void *out, int64_t out_row_stride,
            void *saved_hist,
            void *workspace, size_t workspace_bytes, void *cuda_stream) {
    return ccc_fwd_ex(x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype, activation, conv_state,
                      n_slots, state_len, st_slot, st_c, st_l, cu_seqlens, N, cache_indices, has_initial_state, out,
                      out_row_stride, saved_hist, workspace, workspace_bytes, 0u, cuda_stream);
}

int ccc_fwd_ex(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
               const void *weight, int32_t w_dtype, int32_t width,
               const void *bias, int32_t b_dtype, int32_t activation,
               void *conv_state, int32_t n_slots, int32_t state_len,
               int64_t st_slot, int64_t st_c, int64_t st_l,
               const int32_t *cu_seqlens, int32_t N,
               const int32_t *cache_indices, const uint8_t *has_initial_state,
               void *out, int64_t out_row_stride,
               void *saved_hist,
               void *workspace, size_t workspace_bytes, uint32_t options, void *cuda_stream) {
    if (options & ~static_cast<uint32_t>(CCC_OPT_OVERLAP_PROLOGUE)) return CCC_ERR_SHAPE;
    // ---- shapes and dtypes
    if (rows < 0 || N < 0 || C <= 0 || C % 8 != 0) return CCC_ERR_SHAPE;
    if (rows > INT32_MAX) return CCC_ERR_SHAPE;  // cu_seqlens is int32
    if (x_row_stride < C || out_row_stride < C || x_row_stride % 8 || out_row_stride % 8) return CCC_ERR_SHAPE;
    if (x_row_stride > INT32_MAX || out_row_stride > INT32_MAX) return CCC_ERR_SHAPE;
    if (w_dtype != CCC_F32 && w_dtype != CCC_BF16) return CCC_ERR_DTYPE;
    if (bias ? (b_dtype != CCC_F32 && b_dtype != CCC_BF16) : (b_dtype != CCC_NONE)) return CCC_ERR_DTYPE;
    if (!width_ok(width) || !activation_ok(activation)) return CCC_ERR_SHAPE;
    const int H = width - 1;
    if (conv_state) {
        if (state_len < H || n_slots < 1) return CCC_ERR_SHAPE;
        if (!state_layout_ok(n_slots, C, state_len, st_slot, st_c, st_l)) return CCC_ERR_SHAPE;
    }
    // ---- pointers
    if (!weight || !cu_seqlens || (rows > 0 && (!x || !out))) return CCC_ERR_NULL;  // x, out: none if no rows
    if (conv_state && !cache_indices) return CCC_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16) || (saved_hist && !aligned(saved_hist, 16))) return CCC_ERR_ALIGN;
    if (!aligned(weight, dtype_size(w_dtype)) || (bias && !aligned(bias, dtype_size(b_dtype)))) return CCC_ERR_ALIGN;
    if ((conv_state && !aligned(conv_state, 2)) || !aligned(cu_seqlens, 4) ||
        (cache_indices && !aligned(cache_indices, 4)))
        return CCC_ERR_ALIGN;
    const size_t ws_need = ccc_workspace_size(rows, N, C, 0);
    if (ws_need && (!workspace || workspace_bytes < ws_need)) return CCC_ERR_WORKSPACE;
    if (ws_need && !aligned(workspace, kAlignWs)) return CCC_ERR_ALIGN;
    // ---- aliasing: every written buffer against every other operand
    const Span s_x = span(x, mat_bytes(rows, x_row_stride, C));
    const Span s_out = span(out, mat_bytes(rows, out_row_stride, C));
    const Span s_w = span(weight, static_cast<size_t>(C) * width * dtype_size(w_dtype));
    const Span s_b = span(bias, bias ? static_cast<size_t>(C) * dtype_size(b_dtype) : 0);
    Span s_st;
    if (conv_state) {
        const int64_t last = (n_slots - 1) * st_slot + (C - 1) * st_c + (state_len - 1) * st_l;
        s_st = span(conv_state, static_cast<size_t>(last + 1) * 2);
    }
    const Span s_cu = span(cu_seqlens, static_cast<size_t>(N + 1) * 4);
    const Span s_ci = span(cache_indices, static_cast<size_t>(N) * 4);
    const Span s_hi = span(has_initial_state, static_cast<size_t>(N));
    const Span s_h = span(saved_hist, static_cast<size_t>(N) * H * C * 2);
    const Span s_ws = span(workspace, ws_need);
    const Span *all[] = {&s_x, &s_out, &s_w, &s_b, &s_st, &s_cu, &s_ci, &s_hi, &s_h, &s_ws};
    const Span *written[] = {&s_out, &s_st, &s_h, &s_ws};
    for (const Span *wsp : written)
        for (const Span *o : all)
            if (o != wsp && overlap(*wsp, *o)) return CCC_ERR_ALIAS;

    g_last_launches = 0;
    if (rows == 0 || N == 0) return CCC_OK;

    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    ccc::FwdArgs a = {};
    a.x = static_cast<const uint16_t *>(x);
    a.rows = rows;
    a.C = C;
    a.xs = static_cast<int>(x_row_stride);
    a.w = weight;
    a.w_bf16 = w_dtype == CCC_BF16;
    a.b = bias;
    a.b_kind = bias ? (b_dtype == CCC_F32 ? 1 : 2) : 0;
    a.width = width;
    a.act = activation;
    a.state = static_cast<uint16_t *>(conv_state);
    a.n_slots = n_slots;
    a.st_slot = st_slot;
    a.st_c = st_c;
    a.st_l = st_l;
    a.state_vec = conv_state && st_c == 1 && st_slot % 8 == 0 && st_l % 8 == 0 && aligned(conv_state, 16);
    a.cu = cu_seqlens;
    a.N = N;
    a.cache = cache_indices;
    a.has_init = has_initial_state;
    a.out = static_cast<uint16_t *>(out);
    a.os = static_cast<int>(out_row_stride);
    a.hist = static_cast<uint16_t *>(saved_hist);
    a.slabs = ccc::slabs_of(C, ccc::kFwdVec);
    a.taps_vec = ccc::kFwdVec == 8 && aligned(weight, 16) && (!bias || aligned(bias, 16));
    const DeviceFacts facts = device_facts();
    a.runs = ccc::runs_per_slab(static_cast<int64_t>(facts.sms) * facts.fwd_ctas * ccc::kWarpsPerCta * ccc::kFwdWaves,
                                a.slabs);
    if (ccc::launch_fwd(a, st, (options & CCC_OPT_OVERLAP_PROLOGUE) != 0) != cudaSuccess) return CCC_ERR_CUDA;
    g_last_launches = 1;
    return CCC_OK;
}

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
            void *workspace, size_t workspace_bytes, void *cuda_stream) {
    return ccc_bwd_ex(x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype, activation, saved_hist,
                      cu_seqlens, N, cache_indices, has_initial_state, dy, dy_row_stride, d_final_state, dx,
                      dx_row_stride, dweight, dbias, d_init_state, workspace, workspace_bytes, 0u, cuda_stream);
}

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
               void *workspace, size_t workspace_bytes, uint32_t options, void *cuda_stream) {
    if (options & ~static_cast<uint32_t>(CCC_OPT_OVERLAP_PROLOGUE)) return CCC_ERR_SHAPE;
    if (rows < 0 || N < 0 || C <= 0 || C % 8 != 0) return CCC_ERR_SHAPE;
    if (rows > INT32_MAX) return CCC_ERR_SHAPE;
    if (x_row_stride < C || dy_row_stride < C || dx_row_stride < C || x_row_stride % 8 || dy_row_stride % 8 ||
        dx_row_stride % 8)
        return CCC_ERR_SHAPE;
    if (x_row_stride > INT32_MAX || dy_row_stride > INT32_MAX || dx_row_stride > INT32_MAX) return CCC_ERR_SHAPE;
    if (w_dtype != CCC_F32 && w_dtype != CCC_BF16) return CCC_ERR_DTYPE;
    if (bias ? (b_dtype != CCC_F32 && b_dtype != CCC_BF16) : (b_dtype != CCC_NONE)) return CCC_ERR_DTYPE;
    if (!width_ok(width) || !activation_ok(activation)) return CCC_ERR_SHAPE;
    const int H = width - 1;
    if (!weight || !cu_seqlens || !dweight || (rows > 0 && (!x || !dy || !dx))) return CCC_ERR_NULL;
    if (!aligned(x, 16) || !aligned(dy, 16) || !aligned(dx, 16) || (saved_hist && !aligned(saved_hist, 16)) ||
        (d_final_state && !aligned(d_final_state, 16)) || (d_init_state && !aligned(d_init_state, 16)))
        return CCC_ERR_ALIGN;
    if (!aligned(weight, dtype_size(w_dtype)) || (bias && !aligned(bias, dtype_size(b_dtype))) ||
        !aligned(dweight, 4) || (dbias && !aligned(dbias, 4)) || !aligned(cu_seqlens, 4) ||
        (cache_indices && !aligned(cache_indices, 4)))
        return CCC_ERR_ALIGN;
    const size_t ws_need = ccc_workspace_size(rows, N, C, 1);
    if (ws_need && (!workspace || workspace_bytes < ws_need)) return CCC_ERR_WORKSPACE;
    if (ws_need && !aligned(workspace, kAlignWs)) return CCC_ERR_ALIGN;

    const Span s_x = span(x, mat_bytes(rows, x_row_stride, C));
    const Span s_dy = span(dy, mat_bytes(rows, dy_row_stride, C));
    const Span s_dx = span(dx, mat_bytes(rows, dx_row_stride, C));
    const Span s_w = span(weight, static_cast<size_t>(C) * width * dtype_size(w_dtype));
    const Span s_b = span(bias, bias ? static_cast<size_t>(C) * dtype_size(b_dtype) : 0);
    const Span s_h = span(saved_hist, static_cast<size_t>(N) * H * C * 2);
    const Span s_cu = span(cu_seqlens, static_cast<size_t>(N + 1) * 4);
    const Span s_ci = span(cache_indices, static_cast<size_t>(N) * 4);
    const Span s_hi = span(has_initial_state, static_cast<size_t>(N));
    const Span s_df = span(d_final_state, static_cast<size_t>(N) * H * C * 4);
    const Span s_dw = span(dweight, static_cast<size_t>(C) * width * 4);
    const Span s_db = span(dbias, static_cast<size_t>(C) * 4);
    const Span s_di = span(d_init_state, static_cast<size_t>(N) * H * C * 4);
    const Span s_ws = span(workspace, ws_need);
    const Span *all[] = {&s_x, &s_dy, &s_dx, &s_w, &s_b, &s_h, &s_cu, &s_ci, &s_hi, &s_df, &s_dw, &s_db, &s_di, &s_ws};
    const Span *written[] = {&s_dx, &s_dw, &s_db, &s_di, &s_ws};
    for (const Span *wsp : written)
        for (const Span *o : all)
            if (o != wsp && overlap(*wsp, *o)) return CCC_ERR_ALIAS;

    g_last_launches = 0;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (rows == 0 || N == 0) {  // no token: the gradients are zero (every sequence is empty)
        if (cudaMemsetAsync(dweight, 0, static_cast<size_t>(C) * width * sizeof(float), st) != cudaSuccess)
            return CCC_ERR_CUDA;
        if (dbias && cudaMemsetAsync(dbias, 0, static_cast<size_t>(C) * sizeof(float), st) != cudaSuccess)
            return CCC_ERR_CUDA;
        if (d_init_state && N > 0 &&
            cudaMemsetAsync(d_init_state, 0, static_cast<size_t>(N) * H * C * sizeof(float), st) != cudaSuccess)
            return CCC_ERR_CUDA;
        return CCC_OK;
    }

    ccc::BwdArgs a = {};
    a.x = static_cast<const uint16_t *>(x);
    a.rows = rows;
    a.C = C;
    a.xs = static_cast<int>(x_row_stride);
    a.w = weight;
    a.w_bf16 = w_dtype == CCC_BF16;
    a.b = bias;
    a.b_kind = bias ? (b_dtype == CCC_F32 ? 1 : 2) : 0;
    a.width = width;
    a.act = activation;
    a.hist = static_cast<const uint16_t *>(saved_hist);
    a.cu = cu_seqlens;
    a.N = N;
    a.cache = cache_indices;
    a.has_init = has_initial_state;
    a.dy = static_cast<const uint16_t *>(dy);
    a.dys = static_cast<int>(dy_row_stride);
    a.d_final = d_final_state;
    a.dx = static_cast<uint16_t *>(dx);
    a.dxs = static_cast<int>(dx_row_stride);
    a.d_init = d_init_state;
    a.part = static_cast<float *>(workspace);
    a.slabs = ccc::bwd_slabs(C);
    a.taps_vec = ccc::kBwdVec == 8 && ccc::kBwdRing > 0 && aligned(weight, 16) && (!bias || aligned(bias, 16));
    a.runs = ccc::bwd_runs(rows, C);
    if (ccc::launch_bwd(a, st, (options & CCC_OPT_OVERLAP_PROLOGUE) != 0, device_facts().sms) != cudaSuccess)
        return CCC_ERR_CUDA;
    if (ccc::launch_reduce(a.part, a.runs, C, width, dweight, dbias, st) != cudaSuccess) return CCC_ERR_CUDA;
    g_last_launches = 2;
    return CCC_OK;
}

int ccc_update(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
               const void *weight, int32_t w_dtype, int32_t width,
               const void *bias, int32_t b_dtype, int32_t activation,
               void *conv_state, int32_t n_slots, int32_t state_len,
               int64_t st_slot, int64_t st_c, int64_t st_l,
               const int32_t *cu_seqlens, int32_t N,
               const int32_t *cache_indices, const int32_t *num_accepted,
               void *out, int64_t out_row_stride, void *cuda_stream) {
    return ccc_update_ex(x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype, activation, conv_state,
                         n_slots, state_len, st_slot, st_c, st_l, cu_seqlens, N, cache_indices, num_accepted, out,
                         out_row_stride, 0u, cuda_stream);
}

int ccc_update_ex(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
                  const void *weight, int32_t w_dtype, int32_t width,
                  const void *bias, int32_t b_dtype, int32_t activation,
                  void *conv_state, int32_t n_slots, int32_t state_len,
                  int64_t st_slot, int64_t st_c, int64_t st_l,
                  const int32_t *cu_seqlens, int32_t N,
                  const int32_t *cache_indices, const int32_t *num_accepted,
                  void *out, int64_t out_row_stride, uint32_t options, void *cuda_stream) {
    if (options & ~static_cast<uint32_t>(CCC_OPT_OVERLAP_PROLOGUE)) return CCC_ERR_SHAPE;
    if (rows < 0 || N < 0 || C <= 0 || C % 8 != 0) return CCC_ERR_SHAPE;
    if (rows > INT32_MAX) return CCC_ERR_SHAPE;
    if (x_row_stride < C || out_row_stride < C || x_row_stride % 8 || out_row_stride % 8) return CCC_ERR_SHAPE;
    if (x_row_stride > INT32_MAX || out_row_stride > INT32_MAX) return CCC_ERR_SHAPE;
    if (w_dtype != CCC_F32 && w_dtype != CCC_BF16) return CCC_ERR_DTYPE;
    if (bias ? (b_dtype != CCC_F32 && b_dtype != CCC_BF16) : (b_dtype != CCC_NONE)) return CCC_ERR_DTYPE;
    if (!width_ok(width) || !activation_ok(activation)) return CCC_ERR_SHAPE;
    if (!weight || !cu_seqlens || !conv_state || !cache_indices || (rows > 0 && (!x || !out))) return CCC_ERR_NULL;
    if (state_len < width - 1 || n_slots < 1) return CCC_ERR_SHAPE;
    if (!state_layout_ok(n_slots, C, state_len, st_slot, st_c, st_l)) return CCC_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(conv_state, 2) || !aligned(cu_seqlens, 4) ||
        !aligned(cache_indices, 4) || (num_accepted && !aligned(num_accepted, 4)))
        return CCC_ERR_ALIGN;
    if (!aligned(weight, dtype_size(w_dtype)) || (bias && !aligned(bias, dtype_size(b_dtype)))) return CCC_ERR_ALIGN;
    const Span s_x = span(x, mat_bytes(rows, x_row_stride, C));
    const Span s_out = span(out, mat_bytes(rows, out_row_stride, C));
    const Span s_w = span(weight, static_cast<size_t>(C) * width * dtype_size(w_dtype));
    const Span s_b = span(bias, bias ? static_cast<size_t>(C) * dtype_size(b_dtype) : 0);
    const int64_t last = (n_slots - 1) * st_slot + (C - 1) * st_c + (state_len - 1) * st_l;
    const Span s_st = span(conv_state, static_cast<size_t>(last + 1) * 2);
    const Span s_cu = span(cu_seqlens, static_cast<size_t>(N + 1) * 4);
    const Span s_ci = span(cache_indices, static_cast<size_t>(N) * 4);
    const Span s_na = span(num_accepted, static_cast<size_t>(N) * 4);
    const Span *all[] = {&s_x, &s_out, &s_w, &s_b, &s_st, &s_cu, &s_ci, &s_na};
    const Span *written[] = {&s_out, &s_st};
    for (const Span *wsp : written)
        for (const Span *o : all)
            if (o != wsp && overlap(*wsp, *o)) return CCC_ERR_ALIAS;

    g_last_launches = 0;
    if (rows == 0 || N == 0) return CCC_OK;
    ccc::UpdArgs a = {};
    a.x = static_cast<const uint16_t *>(x);
    a.rows = rows;
    a.C = C;
    a.xs = static_cast<int>(x_row_stride);
    a.w = weight;
    a.w_bf16 = w_dtype == CCC_BF16;
    a.b = bias;
    a.b_kind = bias ? (b_dtype == CCC_F32 ? 1 : 2) : 0;
    a.width = width;
    a.act = activation;
    a.state = static_cast<uint16_t *>(conv_state);
    a.n_slots = n_slots;
    a.L = state_len;
    a.st_slot = st_slot;
    a.st_c = st_c;
    a.st_l = st_l;
    a.state_vec = st_c == 1 && st_slot % 8 == 0 && st_l % 8 == 0 && aligned(conv_state, 16);
    a.state_stage = !a.state_vec && st_l == 1 && st_c == state_len && st_slot % 8 == 0 &&
                    state_len <= ccc::update_stage_max_len() && aligned(conv_state, 16);
    a.cu = cu_seqlens;
    a.N = N;
    a.cache = cache_indices;
    a.accepted = num_accepted;
    a.out = static_cast<uint16_t *>(out);
    a.os = static_cast<int>(out_row_stride);
    a.slabs = ccc::update_slabs(C);
    a.groups = ccc::update_groups(N, a.slabs, device_facts().sms);
    if (ccc::launch_update(a, static_cast<cudaStream_t>(cuda_stream), (options & CCC_OPT_OVERLAP_PROLOGUE) != 0) !=
        cudaSuccess)
        return CCC_ERR_CUDA;
    g_last_launches = 1;
    return CCC_OK;
}

}  // extern "C"
