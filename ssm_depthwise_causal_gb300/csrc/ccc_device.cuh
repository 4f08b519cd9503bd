// ccc_device.cuh -- device-side building blocks shared by the forward and
// backward kernels of the packed width-4 causal depthwise Conv1d + SiLU.
//
// Data layout (FlashInfer "flashinfer.mamba.causal_conv1d_fn", Parameters):
// activations are BF16 [rows][C] with channels contiguous, so one lane owns
// VEC consecutive channels (VEC = 8 -> one 16-byte vector per row, VEC = 4 ->
// 8 bytes) and a warp covers a 32*VEC-channel slab of every row it touches:
// each row access of a warp is one fully-used, contiguous 256/512-byte span.
// FP32 math runs on packed float2 pairs (sm_100+ FFMA2/FADD2/FMUL2), two
// channels per instruction.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ccc_internal.h"

namespace ccc {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kCtaThreads = kWarpsPerCta * 32;

// ---------------------------------------------------------------- raw I/O --

// NV packed bf16x2 words = 2*NV channels of one row.
template <int NV>
struct Raw {
    uint32_t u[NV];
};

template <int NV>
__device__ __forceinline__ Raw<NV> raw_zero() {
    Raw<NV> r;
#pragma unroll
    for (int i = 0; i < NV; ++i) r.u[i] = 0u;
    return r;
}

// Read-only (non-coherent) vector load: x and dy are never written by the
// kernels that read them.
template <int NV>
__device__ __forceinline__ Raw<NV> ld_ro(const void *p) {
    Raw<NV> r;
    if constexpr (NV == 4) {
        const uint4 t = __ldg(reinterpret_cast<const uint4 *>(p));
        r.u[0] = t.x; r.u[1] = t.y; r.u[2] = t.z; r.u[3] = t.w;
    } else {
        static_assert(NV == 2, "VEC must be 4 or 8");
        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
        r.u[0] = t.x; r.u[1] = t.y;
    }
    return r;
}

// Coherent vector load (for buffers the same kernel may also write).
template <int NV>
__device__ __forceinline__ Raw<NV> ld_rw(const void *p) {
    Raw<NV> r;
    if constexpr (NV == 4) {
        const uint4 t = *reinterpret_cast<const uint4 *>(p);
        r.u[0] = t.x; r.u[1] = t.y; r.u[2] = t.z; r.u[3] = t.w;
    } else {
        const uint2 t = *reinterpret_cast<const uint2 *>(p);
        r.u[0] = t.x; r.u[1] = t.y;
    }
    return r;
}

// Streaming (evict-first) store: outputs are not re-read by this kernel.
template <int NV>
__device__ __forceinline__ void st_stream(void *p, const Raw<NV> &r) {
    if constexpr (NV == 4) {
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(r.u[0], r.u[1], r.u[2], r.u[3]));
    } else {
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(r.u[0], r.u[1]));
    }
}

template <int NV>
__device__ __forceinline__ void st_plain(void *p, const Raw<NV> &r) {
    if constexpr (NV == 4) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(r.u[0], r.u[1], r.u[2], r.u[3]);
    } else {
        *reinterpret_cast<uint2 *>(p) = make_uint2(r.u[0], r.u[1]);
    }
}

// bf16x2 word -> two floats (exact: a BF16 value is the top half of an FP32).
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// two floats -> bf16x2 word, round-to-nearest-even; .x goes to the low half
// (the lower channel, as stored in memory).
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int NV>
__device__ __forceinline__ void unpack(const Raw<NV> &r, float2 (&f)[NV]) {
#pragma unroll
    for (int i = 0; i < NV; ++i) f[i] = bf2_to_f2(r.u[i]);
}

// ------------------------------------------------- asynchronous copies --
//
// Per-lane global -> shared copies (PTX cp.async): the bytes land in shared
// memory without passing through registers, so a lane can keep several rows
// in flight while it computes on earlier ones.  `valid == false` zero-fills
// the destination without reading global memory.

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? BYTES : 0;
    if constexpr (BYTES == 16) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
    } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(BYTES), "r"(n)
                     : "memory");
    }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most `pending` of this thread's committed copy groups are
// still in flight (pending is a small runtime value < 8).
__device__ __forceinline__ void cp_async_wait(int pending) {
    switch (pending) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

template <int NV>
__device__ __forceinline__ Raw<NV> ld_shared(const unsigned char *p) {
    Raw<NV> r;
    if constexpr (NV == 4) {
        const uint4 t = *reinterpret_cast<const uint4 *>(p);
        r.u[0] = t.x; r.u[1] = t.y; r.u[2] = t.z; r.u[3] = t.w;
    } else {
        const uint2 t = *reinterpret_cast<const uint2 *>(p);
        r.u[0] = t.x; r.u[1] = t.y;
    }
    return r;
}

// Per-lane ring over a contiguous row stream [S0, S1) of NT tensors: stage k
// holds rows S0 + k*U .. S0 + k*U + U-1 (zero-filled past S1) in slot k % P.
// Each lane copies -- and later reads -- only its own VB bytes of a row, so
// in-order completion of its cp.async groups is all the synchronisation
// needed: no barrier, no cross-lane wait.  `src[t]` points at the lane's
// bytes of row 0 of tensor t, `stride[t]` is that tensor's row stride in
// elements.  Shared layout per warp: [P][U][NT][32 lanes][VB].
template <int NV, int U, int P, int NT>
struct LaneRing {
    static constexpr int VB = NV * 4;
    static constexpr int kWarpBytes = P * U * NT * 32 * VB;
    uint32_t base;  // shared address of this lane's bytes in stage 0, row 0, tensor 0
    int S0, S1;
    int issued;     // stages issued so far
    const uint16_t *src[NT];
    int stride[NT];

    __device__ __forceinline__ void start(int s0, int s1) {
        cp_async_wait(0);  // nothing of a previous stream may still land
        S0 = s0;
        S1 = s1;
        issued = 0;
    }

    __device__ __forceinline__ void issue(bool act) {
        const int slot = issued % P;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = S0 + issued * U + u;
            const bool ok = act && r < S1;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint32_t dst = base + static_cast<uint32_t>(((slot * U + u) * NT + t) * 32 * VB);
                cp_async<VB>(dst, ok ? src[t] + static_cast<int64_t>(r) * stride[t] : src[t], ok);
            }
        }
        cp_async_commit();
        ++issued;
    }

    // Keep the stages from the one holding row r on issued, P deep.
    __device__ __forceinline__ void top_up(int r, bool act) {
        const int k = (r - S0) / U;
        while (issued < k + P && S0 + issued * U < S1) issue(act);
    }

    // Row r of tensor t (r in [S0, S1), stage already issued).
    __device__ __forceinline__ Raw<NV> get(int r, int t) const {
        const int j = r - S0, k = j / U;
        cp_async_wait(issued - 1 - k);
        const uint32_t addr = base + static_cast<uint32_t>((((k % P) * U + j % U) * NT + t) * 32 * VB);
        Raw<NV> v;
        if constexpr (NV == 4) {
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3])
                         : "r"(addr));
        } else {
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.u[0]), "=r"(v.u[1]) : "r"(addr));
        }
        return v;
    }
};

// ------------------------------------------------------------------ math --

// Documented PTX approximations (PTX ISA: ex2.approx.ftz.f32, rcp.approx.ftz.f32).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(z) = 1 / (1 + 2^(-z*log2(e))) on a pair.  Saturates cleanly:
// z -> -inf gives 2^+big = inf and rcp(inf) = 0; z -> +inf gives 1.
__device__ __forceinline__ float2 sigmoid2(float2 z) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    const float2 m = __fmul2_rn(z, make_float2(kNegLog2e, kNegLog2e));
    float2 d = make_float2(ex2_approx(m.x), ex2_approx(m.y));
    d = __fadd2_rn(d, make_float2(1.0f, 1.0f));
    return make_float2(rcp_approx(d.x), rcp_approx(d.y));
}

__device__ __forceinline__ float2 f2_zero() { return make_float2(0.0f, 0.0f); }

// dz = dy * s * (1 + z * (1 - s)), s = sigmoid(z), for the recomputed
// pre-activation z = b + w0 h0 + w1 h1 + w2 h2 + w3 hc (bias first, then the
// four FMAs in tap order, exactly as the forward).
__device__ __forceinline__ float2 silu_grad(float2 b, float2 w0, float2 w1, float2 w2, float2 w3, float2 h0,
                                            float2 h1, float2 h2, float2 hc, float2 gy) {
    float2 z = __ffma2_rn(w0, h0, b);
    z = __ffma2_rn(w1, h1, z);
    z = __ffma2_rn(w2, h2, z);
    z = __ffma2_rn(w3, hc, z);
    const float2 s = sigmoid2(z);
    const float2 one = make_float2(1.0f, 1.0f);
    const float2 oms = __ffma2_rn(s, make_float2(-1.0f, -1.0f), one);  // 1 - s
    const float2 f = __ffma2_rn(z, oms, one);
    return __fmul2_rn(gy, __fmul2_rn(s, f));
}


// ------------------------------------------------------ taps and bias --

// Weights [C][4] FP32 or BF16 and bias [C] FP32 / BF16 / none, read once per
// lane into packed pairs: w_k[v] holds tap k of channels c0+2v, c0+2v+1.
template <int NV>
__device__ __forceinline__ void load_taps(const void *w, int w_bf16, const void *b, int b_kind,
                                          int c0, bool act, float2 (&w0)[NV], float2 (&w1)[NV],
                                          float2 (&w2)[NV], float2 (&w3)[NV], float2 (&bb)[NV]) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float t[2][4], bv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = c0 + 2 * v + h;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float val = 0.0f;
                if (act) {
                    if (w_bf16) {
                        val = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(w)[4 * c + k]);
                    } else {
                        val = __ldg(reinterpret_cast<const float *>(w) + 4 * c + k);
                    }
                }
                t[h][k] = val;
            }
            float bval = 0.0f;
            if (act && b_kind == 1) bval = __ldg(reinterpret_cast<const float *>(b) + c);
            if (act && b_kind == 2) bval = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(b)[c]);
            bv[h] = bval;
        }
        w0[v] = make_float2(t[0][0], t[1][0]);
        w1[v] = make_float2(t[0][1], t[1][1]);
        w2[v] = make_float2(t[0][2], t[1][2]);
        w3[v] = make_float2(t[0][3], t[1][3]);
        bb[v] = make_float2(bv[0], bv[1]);
    }
}

// Taps [C][W] (FP32 or BF16) and bias [C] (FP32 / BF16 / none) for a
// width-W kernel, read once per lane: wt[k][v] holds tap k of channels
// c0+2v, c0+2v+1 (Megatron-Core "core.ssm.causal_conv1d", causal_conv1d_cp:
// weight [D, W]).
template <int NV, int W>
__device__ __forceinline__ void load_taps_w(const void *w, int w_bf16, const void *b, int b_kind, int c0,
                                            bool act, float2 (&wt)[W][NV], float2 (&bb)[NV]) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float t[2][W], bv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = c0 + 2 * v + h;
#pragma unroll
            for (int k = 0; k < W; ++k) {
                float val = 0.0f;
                if (act) {
                    if (w_bf16) {
                        val = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(w)[W * c + k]);
                    } else {
                        val = __ldg(reinterpret_cast<const float *>(w) + W * c + k);
                    }
                }
                t[h][k] = val;
            }
            float bval = 0.0f;
            if (act && b_kind == 1) bval = __ldg(reinterpret_cast<const float *>(b) + c);
            if (act && b_kind == 2) bval = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(b)[c]);
            bv[h] = bval;
        }
#pragma unroll
        for (int k = 0; k < W; ++k) wt[k][v] = make_float2(t[0][k], t[1][k]);
        bb[v] = make_float2(bv[0], bv[1]);
    }
}

// Pre-activation of one channel pair for a width-W stencil: the bias, then
// tap k on history row k (k < W-1, oldest first), then tap W-1 on the
// current row -- the FMA order of FlashInfer causal_conv1d_fn (bias added
// before the FMAs).  hw[k] is history row k of this pair.
template <int W, int NV>
__device__ __forceinline__ float2 conv_pre(const float2 (&wt)[W][NV], float2 b, const float2 (&hw)[W - 1][NV],
                                           float2 hc, int v) {
    float2 z = b;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) z = __ffma2_rn(wt[k][v], hw[k][v], z);
    return __ffma2_rn(wt[W - 1][v], hc, z);
}

// Output of the activation: SiLU z * sigmoid(z), or z itself.
template <bool ACT>
__device__ __forceinline__ float2 activate2(float2 z) {
    if constexpr (ACT) {
        return __fmul2_rn(z, sigmoid2(z));
    } else {
        return z;
    }
}

// dz = dy * d act / dz: dy * s * (1 + z * (1 - s)) with s = sigmoid(z) for
// SiLU, dy itself without activation.
template <bool ACT>
__device__ __forceinline__ float2 activate2_grad(float2 z, float2 gy) {
    if constexpr (ACT) {
        const float2 s = sigmoid2(z);
        const float2 one = make_float2(1.0f, 1.0f);
        const float2 oms = __ffma2_rn(s, make_float2(-1.0f, -1.0f), one);  // 1 - s
        const float2 f = __ffma2_rn(z, oms, one);
        return __fmul2_rn(gy, __fmul2_rn(s, f));
    } else {
        return gy;
    }
}

// ---------------------------------------------------------- work items --
//
// A work item is (sequence n, first row r0, rows nr <= B) inside one
// sequence; items of a sequence are consecutive B-row chunks in order, and
// items are numbered sequence by sequence.  For n_seqs <= 32 every warp
// derives the numbering itself from cu_seqlens with one shuffle scan, so
// small batches need no scratch; otherwise the chunk-map kernel has written
// (n, r0) pairs and the count to the workspace, afresh on each call
// (causal_conv1d_fn, workspace).
// `empty_items` gives each empty sequence one zero-row item (the backward
// needs one to zero that sequence's d_init_state).

// Row indices fit in 32 bits (the host rejects rows > INT32_MAX: cu_seqlens
// is int32); every address is formed in 64 bits from them.
struct Item {
    int n;
    int s, e, r0;
    int nr;
};

// The decoder keeps three registers per lane for the in-kernel numbering
// (lane n < N holds sequence n's clamped start, end and inclusive item
// prefix); the chunk map, offsets and sizes are read from the kernel
// parameters at each call, so they cost no registers across the loop.
template <int B>
struct ItemDecoder {
    int ls, le, lincl;  // register scan state (no map)
    int total;

    __device__ __forceinline__ static int clamp_row(int v, int64_t rows) {
        return v < 0 ? 0 : (v > rows ? static_cast<int>(rows) : v);
    }

    // The map is written by the chunk-map kernel while this grid may already
    // be resident (programmatic dependent launch), so it is not read-only over
    // this kernel's lifetime: it is read with L2-coherent loads (ld.global.cg),
    // never through the non-coherent read-only path.
    __device__ __forceinline__ void init(const int32_t *map, int cap, const int32_t *cu, int N, int64_t rows,
                                         bool empty_items, int lane) {
        if (map) {
            const int cnt = __ldcg(map);
            total = cnt < cap ? cnt : cap;
            ls = le = lincl = 0;
            return;
        }
        int s = 0, e = 0, ni = 0;
        if (lane < N) {
            s = clamp_row(__ldg(cu + lane), rows);
            e = clamp_row(__ldg(cu + lane + 1), rows);
            if (e < s) e = s;
            ni = (e - s + B - 1) / B;
            if (empty_items && ni == 0) ni = 1;
        }
        int incl = ni;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += t;
        }
        ls = s;
        le = e;
        lincl = incl;
        total = __shfl_sync(kFull, incl, 31);
    }

    // Sequence and first row of item `it` (all 32 lanes, same `it`).
    __device__ __forceinline__ void head(int it, const int32_t *map, int &n, int &r0) const {
        if (map) {
            n = __ldcg(map + 1 + 2 * it);
            r0 = __ldcg(map + 2 + 2 * it);
        } else {
            // Sequences whose items all precede `it` form a lane prefix.
            n = __popc(__ballot_sync(kFull, lincl <= it));
            const int s = __shfl_sync(kFull, ls, n), e = __shfl_sync(kFull, le, n);
            const int incl = __shfl_sync(kFull, lincl, n);
            const int ni = max((e - s + B - 1) / B, 1);
            r0 = s + (it - (incl - ni)) * B;
        }
    }

    __device__ __forceinline__ Item get(int it, const int32_t *map, const int32_t *cu, int64_t rows) const {
        Item t;
        head(it, map, t.n, t.r0);
        if (map) {
            t.s = clamp_row(__ldg(cu + t.n), rows);
            t.e = clamp_row(__ldg(cu + t.n + 1), rows);
            if (t.e < t.s) t.e = t.s;
            t.r0 = t.r0 < t.s ? t.s : (t.r0 > t.e ? t.e : t.r0);
        } else {
            t.s = __shfl_sync(kFull, ls, t.n);
            t.e = __shfl_sync(kFull, le, t.n);
        }
        const int left = t.e - t.r0;
        t.nr = left < B ? left : B;
        return t;
    }
};

// ------------------------------------------------ mbarrier + bulk copies --
//
// Shared-memory mbarriers (PTX mbarrier.*) and the bulk-copy engine
// (cp.async.bulk, global -> shared, completion counted in bytes on an
// mbarrier).  Every wait is bounded: after kSpinLimit polls (each one a
// try_wait that may suspend for up to kSuspendNs) it gives up and returns
// false, so a broken handshake ends the kernel instead of hanging the GPU.

constexpr int kSpinLimit = 1 << 22;
constexpr uint32_t kSuspendNs = 1000;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// true once the barrier phase with this parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// One bulk copy global -> shared; `bytes` and both addresses are multiples of
// 16.  Completion is reported to `bar` as `bytes` transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Ask the bulk-copy engine to bring `bytes` (a multiple of 16, 16-byte
// aligned) into L2; nothing is written to shared memory and nothing waits.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------- programmatic launch --

// Wait until the preceding kernel in the stream has finished and its writes
// are visible (no-op when this grid was not launched as a programmatic
// dependent).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream (launched as a programmatic dependent)
// to be scheduled; it still waits in grid_dependency_wait() for our writes.
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ccc
