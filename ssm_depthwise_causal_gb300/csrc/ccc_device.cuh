// ccc_device.cuh -- device-side building blocks shared by the forward,
// backward and decode-update kernels of the packed causal depthwise Conv1d.
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

// ------------------------------------------------------ taps and bias --

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

// The same taps and bias, read through shared memory when the taps and the
// bias are 16-byte aligned (VEC = 8).  A lane's taps are VEC*W consecutive
// values, so a warp's are one contiguous block of its slab: the warp copies
// that block into `buf` (this warp's own shared memory, >= 32 * VEC * W * 4
// bytes) with 16-byte copies (cp.async, or loads and stores), consecutive
// lanes on consecutive chunks (a few fully used 512-byte requests), then
// each lane reads its own chunks back; the bias is read directly (whole
// 16-byte vectors).
// Per-lane global loads of the taps touch a different 128-byte line per lane
// and instruction; with some 40 of them per warp and 16 warps per SM they
// kept every warp waiting ~10 us at the start of each kernel.  Chunk j of
// lane l is stored at NC*l + (j ^ swz(l)) so that the read-back is free of
// bank conflicts (NC = chunks per lane: 2W for FP32 taps, W for BF16).
template <int NC>
__device__ __forceinline__ int tap_swizzle(int l) {
    if constexpr (NC == 8) return l & 7;
    if constexpr (NC == 4) return (l >> 1) & 3;
    if constexpr (NC == 2) return (l >> 2) & 1;
    return 0;
}

// The copy itself, as one cp.async commit group per lane (global -> shared
// without registers), so it can be issued early and overlap other work;
// read_staged_taps reads the block back once every lane has waited for its
// group (cp.async.wait_group) and the warp has synchronized.
template <int NV, int W, int ESZ>
__device__ __forceinline__ void issue_taps_copy(const void *w, int slab_c0, int C, int lane, uint32_t buf) {
    constexpr int VEC = 2 * NV;
    constexpr int NC = VEC * W * ESZ / 16;  // 16-byte chunks per lane
    static_assert(VEC * W * ESZ % 16 == 0, "a lane's taps must be whole 16-byte chunks");
    const int nch = C - slab_c0 < 32 * VEC ? C - slab_c0 : 32 * VEC;
    const int bytes = nch * W * ESZ;  // a multiple of 16 (C % 8 == 0)
    const unsigned char *src = static_cast<const unsigned char *>(w) + static_cast<int64_t>(slab_c0) * W * ESZ;
    for (int off = lane * 16; off < bytes; off += 32 * 16) {
        const int g = off >> 4, l = g / NC, j = g % NC;
        cp_async<16>(buf + static_cast<uint32_t>(16 * (NC * l + (j ^ tap_swizzle<NC>(l)))), src + off, true);
    }
    cp_async_commit();
}

template <int NV, int W, int ESZ>
__device__ __forceinline__ void read_staged_taps(const unsigned char *buf, int lane, bool act, float2 (&wt)[W][NV]) {
    constexpr int VEC = 2 * NV;
    constexpr int NC = VEC * W * ESZ / 16;
    uint32_t words[4 * NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (act) q = *reinterpret_cast<const uint4 *>(buf + 16 * (NC * lane + (j ^ tap_swizzle<NC>(lane))));
        words[4 * j] = q.x;
        words[4 * j + 1] = q.y;
        words[4 * j + 2] = q.z;
        words[4 * j + 3] = q.w;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            float t[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = (2 * v + h) * W + k;  // value index: [channel][tap]
                if constexpr (ESZ == 4) {
                    t[h] = __uint_as_float(words[idx]);
                } else {
                    const uint32_t u = words[idx >> 1];
                    t[h] = __uint_as_float((idx & 1) ? (u & 0xffff0000u) : (u << 16));
                }
            }
            wt[k][v] = make_float2(t[0], t[1]);
        }
    }
}

// The synchronous form: the warp's block copied with plain 16-byte loads
// and stores, then read back.
template <int NV, int W, int ESZ>
__device__ __forceinline__ void stage_taps(const void *w, int slab_c0, int C, int lane, bool act,
                                           unsigned char *buf, float2 (&wt)[W][NV]) {
    constexpr int VEC = 2 * NV;
    constexpr int NC = VEC * W * ESZ / 16;
    const int nch = C - slab_c0 < 32 * VEC ? C - slab_c0 : 32 * VEC;
    const int bytes = nch * W * ESZ;
    const unsigned char *src = static_cast<const unsigned char *>(w) + static_cast<int64_t>(slab_c0) * W * ESZ;
    for (int off = lane * 16; off < bytes; off += 32 * 16) {
        const int g = off >> 4, l = g / NC, j = g % NC;
        *reinterpret_cast<uint4 *>(buf + 16 * (NC * l + (j ^ tap_swizzle<NC>(l)))) =
            __ldg(reinterpret_cast<const uint4 *>(src + off));
    }
    __syncwarp();
    read_staged_taps<NV, W, ESZ>(buf, lane, act, wt);
    __syncwarp();  // every lane has read before the buffer is reused
}

// Issue the copy of this warp's taps into `buf` (see issue_taps_copy).
template <int NV, int W>
__device__ __forceinline__ void issue_taps(const void *w, int w_bf16, int slab_c0, int C, int lane, uint32_t buf) {
    static_assert(NV == 4, "staged taps need 8 channels per lane");
    if (w_bf16) {
        issue_taps_copy<NV, W, 2>(w, slab_c0, C, lane, buf);
    } else {
        issue_taps_copy<NV, W, 4>(w, slab_c0, C, lane, buf);
    }
}

// Read them back: every lane has waited for its copy group; the warp
// synchronizes here (before and after, so `buf` may be reused afterwards).
template <int NV, int W>
__device__ __forceinline__ void take_taps(int w_bf16, int lane, bool act, const unsigned char *buf,
                                          float2 (&wt)[W][NV]) {
    __syncwarp();
    if (w_bf16) {
        read_staged_taps<NV, W, 2>(buf, lane, act, wt);
    } else {
        read_staged_taps<NV, W, 4>(buf, lane, act, wt);
    }
    __syncwarp();
}

// Bias of this lane's channels: 32 (FP32) or 16 (BF16) contiguous,
// 16-byte aligned bytes.
template <int NV>
__device__ __forceinline__ void load_bias_vec(const void *b, int b_kind, int c0, bool act, float2 (&bb)[NV]) {
    static_assert(NV == 4, "vector bias loads need 8 channels per lane");
#pragma unroll
    for (int v = 0; v < NV; ++v) bb[v] = f2_zero();
    if (act && b_kind == 1) {
        const uint4 lo = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(b) + c0));
        const uint4 hi = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(b) + c0 + 4));
        bb[0] = make_float2(__uint_as_float(lo.x), __uint_as_float(lo.y));
        bb[1] = make_float2(__uint_as_float(lo.z), __uint_as_float(lo.w));
        bb[2] = make_float2(__uint_as_float(hi.x), __uint_as_float(hi.y));
        bb[3] = make_float2(__uint_as_float(hi.z), __uint_as_float(hi.w));
    } else if (act && b_kind == 2) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(b) + c0));
        bb[0] = bf2_to_f2(q.x);
        bb[1] = bf2_to_f2(q.y);
        bb[2] = bf2_to_f2(q.z);
        bb[3] = bf2_to_f2(q.w);
    }
}


// Taps (staged, synchronously) and bias in one call.
template <int NV, int W>
__device__ __forceinline__ void load_taps_staged(const void *w, int w_bf16, const void *b, int b_kind, int slab_c0,
                                                 int C, int c0, bool act, int lane, unsigned char *buf,
                                                 float2 (&wt)[W][NV], float2 (&bb)[NV]) {
    static_assert(NV == 4, "staged taps need 8 channels per lane");
    if (w_bf16) {
        stage_taps<NV, W, 2>(w, slab_c0, C, lane, act, buf, wt);
    } else {
        stage_taps<NV, W, 4>(w, slab_c0, C, lane, act, buf, wt);
    }
    load_bias_vec<NV>(b, b_kind, c0, act, bb);
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

// Slot of the row `back` rows before row u in an RS-slot ring of rows (row
// k of a walk in slot k % RS); u and back are compile-time constants at every
// use, so the ring never costs a register move.
template <int RS>
__device__ __forceinline__ constexpr int slot(int u, int back) { return (u - back + 2 * RS) % RS; }

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

// ---------------------------------------------------------- work split --
//
// The valid rows of a packed batch are contiguous: sequence n owns rows
// [cu[n], cu[n+1]) and together they fill [0, T), T = cu[N].  Run r of R
// takes the rows [r*T/R, (r+1)*T/R) -- equal shares whatever the length mix
// -- plus the empty sequences positioned in that range (the last run also
// those at T).  With a walk cost a > 0 the shares are of cost instead: a
// sequence costs its rows plus a, and run r takes the rows whose cost lies
// in [r*K/R, (r+1)*K/R), K = T + a*N.  Turning cu_seqlens into these balanced pieces of work
// happens at the start of every kernel, on the device, every call (the
// chunk-map role of FlashInfer "flashinfer.mamba.causal_conv1d_fn",
// workspace; no scratch and no extra launch here): the warp finds the
// sequence holding its first row with a 32-way search over cu_seqlens, then
// walks forward.
//
// A boundary that falls inside the first H = W-1 rows of a sequence is moved
// back to that sequence's first row (both runs apply the same rule), so a run
// that starts inside a sequence starts at least H rows in: the H rows before
// it are then rows of x, never initial state -- which only the run holding
// the sequence's first row reads (and, in the forward, overwrites).
//
// The walker hands out segments in row order: at most B rows of one
// sequence, clipped to the run.  Consecutive segments of one sequence form a
// walk; a walk starts at the run's first row or at a sequence's first row,
// and every segment but a walk's last has exactly B rows.  Empty sequences
// come out as zero-row segments when asked for (the backward zeroes their
// d_init_state).

// Row indices fit in 32 bits (the host rejects rows > INT32_MAX: cu_seqlens
// is int32); every address is formed in 64 bits from them.
//
// Batches of up to CAP sequences (1024 in the forward, 256 in the
// backward) have their metadata staged in shared memory by the whole CTA
// at the kernel's start -- the clamped
// offsets, the slots and the flags, one coalesced load -- so the walker's
// searches and every per-sequence lookup cost shared-memory latency instead
// of a chain of dependent global loads before the first row is read.
// Larger batches read them from global memory as they go.  CAP is a
// multiple of 128; every member is a multiple of 128 bytes long.
template <int CAP>
struct SeqMeta {
    static_assert(CAP % 128 == 0, "CAP must be a multiple of 128");
    int cu[CAP + 32];           // clamped to [0, rows]
    int cache[CAP];             // slot, or -2 without cache_indices
    unsigned char flag[CAP];    // has_initial_state (0 without it)
};

// All threads of the CTA call this (it ends with __syncthreads); returns
// whether the batch's metadata now sits in `m`.
template <int CAP>
__device__ __forceinline__ bool stage_meta(SeqMeta<CAP> &m, const int32_t *cu, int N, int64_t rows,
                                           const int32_t *cache, const uint8_t *has_init) {
    const bool staged = N > 0 && N <= CAP;
    if (staged) {
        for (int i = threadIdx.x; i <= N; i += blockDim.x) {
            const int v = __ldg(cu + i);
            m.cu[i] = v < 0 ? 0 : (v > rows ? static_cast<int>(rows) : v);
            if (i < N) {
                m.cache[i] = cache ? __ldg(cache + i) : -2;
                m.flag[i] = has_init ? (__ldg(has_init + i) != 0) : 0;
            }
        }
    }
    __syncthreads();
    return staged;
}

struct Item {
    int n;
    int s, e, r0;
    int nr;
};

template <int B>
struct RunWalker {
    int N;
    int H;           // history rows: boundaries never fall in a sequence's first H rows
    int R_lo, R_hi;  // this run's rows (R_hi before the move above; see next())
    bool last;       // the last run (also takes empty sequences at T)
    bool empties;    // hand out empty sequences
    int n;           // current sequence
    int s, e;        // its rows (clamped)
    int r;           // its next row to hand out
    bool fresh;      // nothing of sequence n handed out yet
    int cbase;       // lane j caches the clamped cu[cbase + j]
    int cval;
    const int *scu;  // the clamped offsets in shared memory, or nullptr

    __device__ __forceinline__ static int clamp_row(int v, int64_t rows) {
        return v < 0 ? 0 : (v > rows ? static_cast<int>(rows) : v);
    }

    // Clamped cu[i], 0 <= i <= N: from shared memory when staged.
    __device__ __forceinline__ int cu_val(const int32_t *cu, int64_t rows, int i) const {
        return scu ? scu[i] : clamp_row(__ldg(cu + i), rows);
    }

    __device__ __forceinline__ void refill(const int32_t *cu, int64_t rows, int base, int lane) {
        cbase = base;
        const int idx = base + lane;
        cval = idx <= N ? cu_val(cu, rows, idx) : static_cast<int>(rows);
    }

    // Clamped cu[i] for cbase <= i < cbase + 32 (all lanes, same i).
    __device__ __forceinline__ int cu_at(int i) const { return __shfl_sync(kFull, cval, i - cbase); }

    // Clamped cu[i] for any i in [0, N] (all lanes, same i).
    __device__ __forceinline__ int cu_get(const int32_t *cu, int64_t rows, int i, int lane) {
        if (i < cbase || i >= cbase + 32) refill(cu, rows, i, lane);
        return cu_at(i);
    }

    // First n in [0, N] with cu[n] + alpha * n > c (cu clamped; true at n = N
    // whenever c < T + alpha * N): the same 32-way ballot search as in init.
    __device__ __forceinline__ int first_cost_above(const int32_t *cu, int64_t rows, int64_t c, int alpha,
                                                    int lane) {
        int lo = 0, hi = N;
        while (hi - lo >= 32) {
            const int step = (hi - lo + 31) / 32;
            const int idx = min(lo + lane * step, hi);
            const int64_t key = static_cast<int64_t>(cu_val(cu, rows, idx)) + static_cast<int64_t>(alpha) * idx;
            const unsigned m = __ballot_sync(kFull, key > c);
            if (m == 0) {
                lo = min(lo + 31 * step, hi) + 1;
            } else {
                const int j = __ffs(m) - 1;
                const int new_hi = min(lo + j * step, hi);
                if (j > 0) lo = min(lo + (j - 1) * step, hi) + 1;
                hi = new_hi;
            }
        }
        refill(cu, rows, lo, lane);
        const int64_t key = static_cast<int64_t>(cval) + static_cast<int64_t>(alpha) * (lo + lane);
        const unsigned m = __ballot_sync(kFull, lane <= hi - lo && key > c);
        return m ? lo + __ffs(m) - 1 : hi;
    }

    // The row at cost c of the weighted split, where sequence n costs its
    // rows plus `alpha` charged at its start: c falls in the last sequence n*
    // with cu[n*] + alpha * n* <= c, at row cu[n*] + (c - cu[n*] - alpha *
    // (n* + 1)) clamped to the sequence.  Nondecreasing in c; c >= total
    // gives T.
    __device__ __forceinline__ int row_at_cost(const int32_t *cu, int64_t rows, int64_t c, int64_t total, int T,
                                               int alpha, int lane) {
        if (c >= total) return T;
        const int f = first_cost_above(cu, rows, c, alpha, lane);
        const int ns = f > 0 ? f - 1 : 0;
        const int s0 = cu_get(cu, rows, ns, lane), e0 = cu_get(cu, rows, ns + 1, lane);
        const int len = e0 > s0 ? e0 - s0 : 0;
        int64_t off = c - (static_cast<int64_t>(s0) + static_cast<int64_t>(alpha) * (ns + 1));
        off = off < 0 ? 0 : (off > len ? len : off);
        return s0 + static_cast<int>(off);
    }

    // Run `run` of `runs`.  All 32 lanes call with the same arguments.
    // walk_rows = 0: runs of equal row counts; > 0: runs of equal cost, a
    // sequence costing its rows plus walk_rows (what a walk's start and end
    // cost in rows' worth of time), so runs that cross many short sequences
    // get fewer rows.  `staged`: the clamped offsets (stage_meta), or
    // nullptr to read cu_seqlens from global memory.
    __device__ __forceinline__ void init(const int32_t *cu, int n_seqs, int64_t rows, int run, int runs,
                                         int hist_rows, bool want_empty, int lane, int walk_rows = 0,
                                         const int *staged = nullptr) {
        scu = staged;
        N = n_seqs;
        H = hist_rows;
        empties = want_empty;
        last = run == runs - 1;
        fresh = true;
        s = e = r = 0;
        n = 0;
        refill(cu, rows, 0, lane);
        if (N <= 0) {
            R_lo = R_hi = 0;
            return;
        }
        const int T = cu_get(cu, rows, N, lane);
        if (walk_rows > 0) {
            // Both neighbours of a boundary compute it from the same cost.
            const int64_t total = static_cast<int64_t>(T) + static_cast<int64_t>(walk_rows) * N;
            R_lo = row_at_cost(cu, rows, static_cast<int64_t>(run) * total / runs, total, T, walk_rows, lane);
            R_hi = row_at_cost(cu, rows, static_cast<int64_t>(run + 1) * total / runs, total, T, walk_rows, lane);
        } else {
            R_lo = static_cast<int>(static_cast<int64_t>(run) * T / runs);
            R_hi = static_cast<int>(static_cast<int64_t>(run + 1) * T / runs);
        }
        // n_a = first n in [0, N) with cu[n+1] >= R_lo (exists: cu[N] = T).
        int lo = 0, hi = N - 1;
        while (hi - lo >= 32) {
            const int step = (hi - lo + 31) / 32;
            const int idx = min(lo + lane * step, hi);
            const int v = cu_val(cu, rows, idx + 1);
            const unsigned m = __ballot_sync(kFull, v >= R_lo);
            if (m == 0) {
                lo = min(lo + 31 * step, hi) + 1;
            } else {
                const int j = __ffs(m) - 1;
                const int new_hi = min(lo + j * step, hi);
                if (j > 0) lo = min(lo + (j - 1) * step, hi) + 1;
                hi = new_hi;
            }
        }
        // hi - lo < 32: lane j tests n = lo + j with cu[lo + j + 1].
        refill(cu, rows, lo + 1, lane);
        const unsigned m = __ballot_sync(kFull, lane <= hi - lo && cval >= R_lo);
        const int n_a = m ? lo + __ffs(m) - 1 : hi;
        // A nonempty sequence ending exactly at R_lo belongs to the previous
        // run; one holding R_lo within its first H rows starts this run.
        n = n_a;
        if (n < N) {
            const int sa = cu_get(cu, rows, n, lane), ea = cu_get(cu, rows, n + 1, lane);
            if (ea == R_lo && sa < R_lo) {
                ++n;
            } else if (sa < R_lo && ea > R_lo && R_lo - sa < H) {
                R_lo = sa;
            }
        }
        if (n < N) load_seq(cu, rows, lane);
    }

    __device__ __forceinline__ void load_seq(const int32_t *cu, int64_t rows, int lane) {
        s = cu_get(cu, rows, n, lane);
        e = cu_get(cu, rows, n + 1, lane);
        if (e < s) e = s;
        r = s > R_lo ? s : R_lo;
        if (r > e) r = e;
        fresh = true;
    }

    // The next segment; false when the run is done.  `cont`: the segment
    // continues the previous one's walk (same sequence, next rows).
    // `more`: another segment of this walk follows it.
    __device__ __forceinline__ bool next(const int32_t *cu, int64_t rows, int lane, Item &t, bool &cont,
                                         bool &more) {
        while (n < N) {
            if (fresh) {
                if (!(s < R_hi || (last && s == R_hi))) return false;  // starts past the run
                if (s < R_hi && e > R_hi && R_hi - s < H) return false;  // the next run starts at s
            }
            const int stop = e < R_hi ? e : R_hi;
            if (s == e) {  // empty sequence
                if (fresh && empties) {
                    t.n = n; t.s = s; t.e = e; t.r0 = s; t.nr = 0;
                    cont = false;
                    more = false;
                    fresh = false;
                    ++n;
                    if (n < N) load_seq(cu, rows, lane);
                    return true;
                }
            } else if (r < stop) {
                t.n = n; t.s = s; t.e = e; t.r0 = r;
                t.nr = stop - r < B ? stop - r : B;
                cont = !fresh;
                fresh = false;
                r += t.nr;
                more = r < stop;
                return true;
            }
            if (e > R_hi) return false;  // the sequence continues in the next run
            ++n;
            if (n < N) load_seq(cu, rows, lane);
        }
        return false;
    }
};

// ------------------------------------------------------- L2 prefetch --

// Ask L2 to fetch `bytes` (a multiple of 16) at the 16-byte aligned `p`.
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
