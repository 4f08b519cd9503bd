// ccc_update.cu -- the speculative / single-token decode step: the causal
// depthwise Conv1d (+ SiLU) of a few new tokens per sequence from the
// history held in the conv_state pool, and the pool update for the next step.
//
// FlashInfer "flashinfer.mamba.causal_conv1d_fn" (Notes): the speculative step
// right after a prefill is given an accepted count of one.  Reading of that rule
// (the pages give no more): slot q keeps raw history values in time order;
// the previous step left value h[p + 1] of its own history at position p.
// For sequence n with a = num_accepted[n] (1 if none given) and len new
// tokens, the W-1 values before the first new token are positions
// a-1 .. a+W-3, the tokens compute exactly as in the prefill (bias first,
// then taps k = 0..W-1, tap W-1 on the current token, FP32, BF16 RNE out),
// and the step writes h[p + 1] to position p for p < min(len + W-2, L):
// positions 0..W-3 get the 2nd .. last read value, positions W-2 .. get the
// new tokens.  The next step, keeping a' of these len tokens, then reads
// positions a'-1 .. a'+W-3 -- the W-1 values that end at its last kept
// token.  With one token and a = 1 this is the ordinary shift-by-one decode
// update, and a prefill's write (last W-1 values at 0:W-1) is the state
// this rule expects for a = 1.  A -1 slot gives zero output and no state
// access; an empty sequence leaves its slot alone.
//
// Two kernels.  For a dense history-contiguous pool ([slots][C][L] with
// L <= 8: the common serving layout) `update_block_kernel` gives every
// (sequence, 256-channel slab) pair its own warp: lane l holds the 8 channels
// c0 .. c0+7 of the slot, whose 8 L values are consecutive in memory
// (16 L bytes, 16-byte aligned), in L vector registers.  Picking position p
// of a channel pair, and rebuilding the block after the step, are byte
// permutes with compile-time selectors, so the block never goes through
// shared memory.  A warp's only dependent round trips are the sequence's
// offsets / slot / accepted count, then the block and its new tokens; with
// one warp per pair those trips overlap across warps instead of queueing
// inside one.  The block is written back (every position; the
// ones not rewritten keep their bits) before the outputs are computed, which
// frees its registers for the arithmetic.
//
// Any other layout takes `update_kernel`: a CTA per (slab, group of
// sequences), its 8 warps taking the group's sequences in turn, reading and
// writing the W-1 positions it needs -- one 16-byte vector per lane and
// position for a channel-contiguous pool, single elements otherwise.
//
// In both kernels the slab's taps and bias are staged once per CTA in shared
// memory (one channel per thread).  Reads of a slot precede every write to
// it in the lane's program order, and no other lane touches the same
// elements (live slots are unique, lanes' channels disjoint), so the in-place
// update needs no synchronisation.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

constexpr int kUpdVec = 8;
#ifndef CCC_UPD_UNROLL
#define CCC_UPD_UNROLL 2
#endif
#ifndef CCC_UPD_CTAS_PER_SM
#define CCC_UPD_CTAS_PER_SM 4
#endif
constexpr int kUpdUnroll = CCC_UPD_UNROLL;
// CTAs the sequence groups of update_kernel are sized for, per SM (more
// groups: more CTAs, fewer requests per warp).
constexpr int kUpdCtasPerSm = CCC_UPD_CTAS_PER_SM;
#ifdef CCC_UPD_BLOCK_MIN_BLOCKS
constexpr int upd_block_min_blocks(int) { return CCC_UPD_BLOCK_MIN_BLOCKS; }
#else
// Resident CTAs per SM update_block_kernel is compiled for: the register cap
// under which a lane's block (4 LS words) and its new tokens stay unspilled.
constexpr int upd_block_min_blocks(int ls) { return ls <= 4 ? 4 : (ls <= 6 ? 3 : 2); }
#endif
constexpr int kUpdBlockMaxL = 8;  // longest history update_block_kernel keeps in registers
constexpr int kUpdSlab = 32 * kUpdVec;

// Element (slot q, channels c0.., position p) of any pool layout.
template <int NV>
__device__ __forceinline__ Raw<NV> state_get(const UpdArgs &a, int q, int p, int c0) {
    const uint16_t *base = a.state + static_cast<int64_t>(q) * a.st_slot + static_cast<int64_t>(p) * a.st_l;
    if (a.state_vec) return ld_rw<NV>(base + c0);
    Raw<NV> r;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const uint32_t lo = base[static_cast<int64_t>(c0 + 2 * v) * a.st_c];
        const uint32_t hi = base[static_cast<int64_t>(c0 + 2 * v + 1) * a.st_c];
        r.u[v] = lo | (hi << 16);
    }
    return r;
}

template <int NV>
__device__ __forceinline__ void state_put(const UpdArgs &a, int q, int p, int c0, const Raw<NV> &r) {
    uint16_t *base = a.state + static_cast<int64_t>(q) * a.st_slot + static_cast<int64_t>(p) * a.st_l;
    if (a.state_vec) {
        st_plain<NV>(base + c0, r);
        return;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        base[static_cast<int64_t>(c0 + 2 * v) * a.st_c] = static_cast<uint16_t>(r.u[v] & 0xffffu);
        base[static_cast<int64_t>(c0 + 2 * v + 1) * a.st_c] = static_cast<uint16_t>(r.u[v] >> 16);
    }
}

// One request: its rows [s, e) (clamped to [0, rows]), slot q and accepted
// count (loaded, not yet clamped); n = -1 for none.
struct Req {
    int n, s, e, q, acc;
};

__device__ __forceinline__ Req load_req(const UpdArgs &a, int n, int n_end) {
    Req r{-1, 0, 0, -1, 1};
    if (n < n_end) {
        const int64_t rows = a.rows;
        r.n = n;
        r.s = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n)), int64_t{0}), rows));
        r.e = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n + 1)), static_cast<int64_t>(r.s)), rows));
        r.q = __ldg(a.cache + n);
        if (a.accepted) r.acc = __ldg(a.accepted + n);
    }
    return r;
}

// The slab's taps 0..W-1 and bias as FP32, one channel per thread of the
// CTA, read from global memory (load) and then stored to shared memory
// (store, after the caller has issued its own loads).
template <int W>
struct TapStage {
    float t[W + 1];
    __device__ __forceinline__ void load(const UpdArgs &a, int slab) {
        const int c = slab * kUpdSlab + static_cast<int>(threadIdx.x);
        const bool ok = c < a.C;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            float v = 0.0f;
            if (ok) {
                v = a.w_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.w)[W * c + k])
                             : __ldg(reinterpret_cast<const float *>(a.w) + W * c + k);
            }
            t[k] = v;
        }
        float bv = 0.0f;
        if (ok && a.b_kind == 1) bv = __ldg(reinterpret_cast<const float *>(a.b) + c);
        if (ok && a.b_kind == 2) bv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.b)[c]);
        t[W] = bv;
    }
    __device__ __forceinline__ void store(float (&s_tap)[W + 1][kUpdSlab]) const {
#pragma unroll
        for (int k = 0; k <= W; ++k) s_tap[k][threadIdx.x] = t[k];
    }
};

// One new token of a lane's 8 channels: y from the history hw (oldest
// first) and the token xr, then hw shifts by one.
template <int W, bool ACT, int NV>
__device__ __forceinline__ Raw<NV> update_token(const float2 (&wt)[W][NV], const float2 (&bb)[NV],
                                                float2 (&hw)[W - 1][NV], const Raw<NV> &xr) {
    constexpr int H = W - 1;
    float2 hc[NV];
    unpack<NV>(xr, hc);
    Raw<NV> y;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        y.u[v] = f2_to_bf2(activate2<ACT>(conv_pre<W, NV>(wt, bb[v], hw, hc[v], v)));
#pragma unroll
        for (int k = 0; k + 1 < H; ++k) hw[k][v] = hw[k + 1][v];
        hw[H - 1][v] = hc[v];
    }
    return y;
}

// Any pool layout: a CTA per (slab, group of sequences), each warp looping
// over its sequences (the group's w-th, (w+8)-th, ...).
template <int W, bool ACT>
__global__ void __launch_bounds__(kCtaThreads, kUpdMinBlocks) update_kernel(const UpdArgs a) {
    constexpr int VEC = kUpdVec, NV = VEC / 2, U = kUpdUnroll;
    constexpr int H = W - 1;
    __shared__ __align__(16) float s_tap[W + 1][kUpdSlab];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slab = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.slabs));
    const int grp = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.slabs));
    const int n_beg = static_cast<int>(static_cast<int64_t>(grp) * a.N / a.groups);
    const int n_end = static_cast<int>(static_cast<int64_t>(grp + 1) * a.N / a.groups);

    int n = n_beg + warp;
    Req cur = load_req(a, n, n_end);
    {
        TapStage<W> ts;
        ts.load(a, slab);
        ts.store(s_tap);
    }
    __syncthreads();
    // Only offsets, slots, accepted counts, taps and bias read above; launched
    // as a programmatic dependent (CCC_OPT_OVERLAP_PROLOGUE) wait here for the
    // previous kernel before touching the pool, x or out.  (A no-op otherwise.)
    grid_dependency_wait();
    if (cur.n < 0) return;  // whole warp, after the CTA barrier

    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;
    float2 wt[W][NV], bb[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) wt[k][v] = reinterpret_cast<const float2 *>(&s_tap[k][lane * VEC])[v];
        bb[v] = reinterpret_cast<const float2 *>(&s_tap[W][lane * VEC])[v];
    }

    while (true) {
        const Req nx = load_req(a, n + kWarpsPerCta, n_end);  // one sequence ahead
        const int len = cur.e - cur.s;
        const int q = cur.q;
        const uint16_t *xrow = a.x + static_cast<int64_t>(cur.s) * a.xs + c0;
        uint16_t *orow = a.out + static_cast<int64_t>(cur.s) * a.os + c0;
        const bool pool = len > 0 && q >= 0 && q < a.n_slots;
        const int acc = min(max(cur.acc, 1), a.L - H + 1);
        const int n_write = len >= a.L ? a.L : min(len + H - 1, a.L);  // positions written

        if (len > 0 && q == -1) {  // padded request: zero output, no state access
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < len; ++r) st_stream<NV>(orow + static_cast<int64_t>(r) * a.os, z);
            }
        } else if (len > 0 && act) {
            Raw<NV> hr[H];  // the W-1 values before the first new token
#pragma unroll
            for (int p = 0; p < H; ++p) hr[p] = pool ? state_get<NV>(a, q, acc - 1 + p, c0) : raw_zero<NV>();
            // Positions 0 .. W-3: the 2nd .. last value just read.
            if (pool) {
#pragma unroll
                for (int p = 0; p + 1 < H; ++p)
                    if (p < n_write) state_put<NV>(a, q, p, c0, hr[p + 1]);
            }
            float2 hw[H][NV];
#pragma unroll
            for (int p = 0; p < H; ++p) unpack<NV>(hr[p], hw[p]);
            for (int base = 0; base < len; base += U) {
                Raw<NV> xr[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    xr[u] = base + u < len ? ld_ro<NV>(xrow + static_cast<int64_t>(base + u) * a.xs) : raw_zero<NV>();
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + u;
                    if (j >= len) break;
                    st_stream<NV>(orow + static_cast<int64_t>(j) * a.os, update_token<W, ACT, NV>(wt, bb, hw, xr[u]));
                    // token j is history value H + j: position H - 1 + j
                    if (pool && j < n_write - (H - 1)) state_put<NV>(a, q, H - 1 + j, c0, xr[u]);
                }
            }
        }
        n += kWarpsPerCta;
        if (nx.n < 0) break;
        cur = nx;
    }
}

// Pre-activation of the lane's channel pair v for one token: taps and bias
// from the CTA's shared copy, history hv (oldest first), token xc -- the
// same FMA order as every other kernel (conv_pre).
template <int W>
__device__ __forceinline__ float2 pair_pre(const float (&s_tap)[W + 1][kUpdSlab], int lane, int v,
                                          const float2 (&hv)[W - 1], float2 xc) {
    float2 wv[W][1], h1[W - 1][1];
#pragma unroll
    for (int k = 0; k < W; ++k) wv[k][0] = reinterpret_cast<const float2 *>(&s_tap[k][lane * kUpdVec])[v];
#pragma unroll
    for (int k = 0; k + 1 < W; ++k) h1[k][0] = hv[k];
    const float2 b = reinterpret_cast<const float2 *>(&s_tap[W][lane * kUpdVec])[v];
    return conv_pre<W, 1>(wv, b, h1, xc, 0);
}

// Pair word (channels 2v, 2v+1 of the lane at position p) of a lane's
// channel-major block: element ch * LS + p is half (ch * LS + p) & 1 of word
// (ch * LS + p) >> 1.  p and v are compile-time constants at every use.
template <int LS>
__device__ __forceinline__ uint32_t block_pair(const uint32_t (&u)[4 * LS], int p, int v) {
    const int e0 = 2 * v * LS + p, e1 = (2 * v + 1) * LS + p;
    const unsigned sel = ((e0 & 1) ? 0x32u : 0x10u) | (((e1 & 1) ? 0x76u : 0x54u) << 8);
    return __byte_perm(u[e0 >> 1], u[e1 >> 1], sel);
}

// Dense history-contiguous pool with L = LS <= 8: a warp per (sequence,
// slab), lane l owning channels c0 .. c0+7 and their whole 16*LS-byte block.
template <int W, bool ACT, int LS>
__global__ void __launch_bounds__(kCtaThreads, upd_block_min_blocks(LS)) update_block_kernel(const UpdArgs a) {
    constexpr int VEC = kUpdVec, NV = VEC / 2;
    constexpr int H = W - 1;
    constexpr int T0 = LS - H + 1;  // new tokens a slot keeps raw: positions H-1 .. LS-1
    constexpr int NW = 4 * LS;      // 32-bit words of a lane's block
    static_assert(LS >= H && LS <= kUpdBlockMaxL, "history length of the register block");
    __shared__ __align__(16) float s_tap[W + 1][kUpdSlab];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slab = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.slabs));
    const int grp = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.slabs));
    const Req r = load_req(a, grp * kWarpsPerCta + warp, a.N);
    TapStage<W> ts;
    ts.load(a, slab);
    // Only offsets, slots, accepted counts, taps and bias read so far;
    // launched as a programmatic dependent (CCC_OPT_OVERLAP_PROLOGUE) wait
    // here for the previous kernel before touching the pool, x or out.  (A
    // no-op otherwise.)
    grid_dependency_wait();

    // The block and the first T0 new tokens, loaded before the CTA barrier.
    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;
    const int len = r.e - r.s;
    const int q = r.q;
    const bool pool = r.n >= 0 && len > 0 && q >= 0 && q < a.n_slots;
    uint16_t *blk_g = a.state + static_cast<int64_t>(pool ? q : 0) * a.st_slot + static_cast<int64_t>(c0) * LS;
    uint32_t blk[NW];
#pragma unroll
    for (int k = 0; k < LS; ++k) {
        uint4 t = make_uint4(0u, 0u, 0u, 0u);
        if (pool && act) t = *reinterpret_cast<const uint4 *>(blk_g + 8 * k);
        blk[4 * k] = t.x; blk[4 * k + 1] = t.y; blk[4 * k + 2] = t.z; blk[4 * k + 3] = t.w;
    }
    const uint16_t *xrow = a.x + static_cast<int64_t>(r.s) * a.xs + c0;
    Raw<NV> tok[T0];
#pragma unroll
    for (int j = 0; j < T0; ++j)
        tok[j] = (r.n >= 0 && act && q != -1 && j < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(j) * a.xs)
                                                         : raw_zero<NV>();
    ts.store(s_tap);
    __syncthreads();
    if (r.n < 0 || len <= 0 || !act) return;
    uint16_t *orow = a.out + static_cast<int64_t>(r.s) * a.os + c0;
    if (q == -1) {  // padded request: zero output, no state access
        const Raw<NV> z = raw_zero<NV>();
        for (int j = 0; j < len; ++j) st_stream<NV>(orow + static_cast<int64_t>(j) * a.os, z);
        return;
    }

    // The W-1 values before the first new token: positions acc-1 .. acc+H-2.
    // Without accepted counts acc = 1; otherwise they are picked by selects
    // over the T0 possible offsets (the empty asm hides each candidate's
    // origin, so the compiler cannot fold the selects into a run-time index
    // of the block, which would put the block in local memory).
    Raw<NV> hr[H];
#pragma unroll
    for (int i = 0; i < H; ++i)
#pragma unroll
        for (int v = 0; v < NV; ++v) hr[i].u[v] = block_pair<LS>(blk, i, v);
    if (T0 > 1 && a.accepted) {
        const int acc = min(max(r.acc, 1), T0);
#pragma unroll
        for (int a0 = 1; a0 < T0; ++a0) {
#pragma unroll
            for (int i = 0; i < H; ++i)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    uint32_t cand = block_pair<LS>(blk, a0 + i, v);
                    asm("" : "+r"(cand));
                    hr[i].u[v] = acc - 1 == a0 ? cand : hr[i].u[v];
                }
        }
    }

    // The new block: position p < n_write gets history value h[p + 1] (the
    // 2nd .. last value read, then the new tokens); the others keep their
    // bits.  Word w of the block holds elements 2w, 2w+1 (channel e / LS,
    // position e % LS): one byte permute gathers both new halves, and a
    // mask per position keeps the old half where nothing is written.
    if (pool) {
        const int n_write = len >= LS ? LS : min(len + H - 1, LS);
        uint32_t keep_lo[LS], keep_hi[LS];
#pragma unroll
        for (int p = 0; p < LS; ++p) {
            keep_lo[p] = p < n_write ? 0u : 0x0000ffffu;
            keep_hi[p] = p < n_write ? 0u : 0xffff0000u;
        }
        uint32_t nb[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int e0 = 2 * w, e1 = 2 * w + 1;
            const int ch0 = e0 / LS, p0 = e0 % LS, ch1 = e1 / LS, p1 = e1 % LS;
            const uint32_t src0 = p0 < H - 1 ? hr[p0 + 1].u[ch0 >> 1] : tok[p0 - H + 1].u[ch0 >> 1];
            const uint32_t src1 = p1 < H - 1 ? hr[p1 + 1].u[ch1 >> 1] : tok[p1 - H + 1].u[ch1 >> 1];
            const unsigned sel = ((ch0 & 1) ? 0x32u : 0x10u) | (((ch1 & 1) ? 0x76u : 0x54u) << 8);
            const uint32_t fresh = __byte_perm(src0, src1, sel);
            const uint32_t keep = keep_lo[p0] | keep_hi[p1];
            nb[w] = (blk[w] & keep) | (fresh & ~keep);
        }
#pragma unroll
        for (int k = 0; k < LS; ++k)
            *reinterpret_cast<uint4 *>(blk_g + 8 * k) = make_uint4(nb[4 * k], nb[4 * k + 1], nb[4 * k + 2], nb[4 * k + 3]);
    }

    // The block's registers are dead from here on: keep the taps' shared
    // loads below its stores.
    asm volatile("" ::: "memory");

    // The first min(len, T0) tokens (held in registers), channel pair by
    // channel pair: each pair's taps, history and outputs are its own.
    Raw<NV> y[T0];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float2 hv[H];
#pragma unroll
        for (int i = 0; i < H; ++i) hv[i] = bf2_to_f2(hr[i].u[v]);
#pragma unroll
        for (int j = 0; j < T0; ++j) {
            if (j < len) {
                const float2 xc = bf2_to_f2(tok[j].u[v]);
                y[j].u[v] = f2_to_bf2(activate2<ACT>(pair_pre<W>(s_tap, lane, v, hv, xc)));
#pragma unroll
                for (int i = 0; i + 1 < H; ++i) hv[i] = hv[i + 1];
                hv[H - 1] = xc;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < T0; ++j)
        if (j < len) st_stream<NV>(orow + static_cast<int64_t>(j) * a.os, y[j]);

    // Tokens past what the slot keeps (a step longer than the pool allows):
    // one at a time, the history kept as raw BF16 values (exact).
    if (len > T0) {
        Raw<NV> hraw[H];  // history values T0 .. T0+H-1: the read values, then tokens
#pragma unroll
        for (int i = 0; i < H; ++i) hraw[i] = T0 + i < H ? hr[T0 + i] : tok[T0 + i - H];
        for (int j = T0; j < len; ++j) {
            const Raw<NV> xr = ld_ro<NV>(xrow + static_cast<int64_t>(j) * a.xs);
            Raw<NV> yj;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float2 hv[H];
#pragma unroll
                for (int i = 0; i < H; ++i) hv[i] = bf2_to_f2(hraw[i].u[v]);
                yj.u[v] = f2_to_bf2(activate2<ACT>(pair_pre<W>(s_tap, lane, v, hv, bf2_to_f2(xr.u[v]))));
            }
            st_stream<NV>(orow + static_cast<int64_t>(j) * a.os, yj);
#pragma unroll
            for (int i = 0; i + 1 < H; ++i) hraw[i] = hraw[i + 1];
            hraw[H - 1] = xr;
        }
    }
}

using UpdKernel = void (*)(const UpdArgs);

// update_block_kernel for (W, ACT) and history length ls (nullptr if none).
template <int W, bool ACT>
UpdKernel update_block_kernel_l(int ls) {
    switch (ls) {
        case 1: if constexpr (W - 1 <= 1) return update_block_kernel<W, ACT, (W - 1 <= 1 ? 1 : 8)>; else return nullptr;
        case 2: if constexpr (W - 1 <= 2) return update_block_kernel<W, ACT, (W - 1 <= 2 ? 2 : 8)>; else return nullptr;
        case 3: return update_block_kernel<W, ACT, 3>;
        case 4: return update_block_kernel<W, ACT, 4>;
        case 5: return update_block_kernel<W, ACT, 5>;
        case 6: return update_block_kernel<W, ACT, 6>;
        case 7: return update_block_kernel<W, ACT, 7>;
        case 8: return update_block_kernel<W, ACT, 8>;
        default: return nullptr;
    }
}

// ls > 0: update_block_kernel with that history length; 0: update_kernel.
UpdKernel update_kernel_for(int width, int act, int ls) {
    switch (width * 2 + (act ? 1 : 0)) {
        case 4: return ls ? update_block_kernel_l<2, false>(ls) : update_kernel<2, false>;
        case 5: return ls ? update_block_kernel_l<2, true>(ls) : update_kernel<2, true>;
        case 6: return ls ? update_block_kernel_l<3, false>(ls) : update_kernel<3, false>;
        case 7: return ls ? update_block_kernel_l<3, true>(ls) : update_kernel<3, true>;
        case 8: return ls ? update_block_kernel_l<4, false>(ls) : update_kernel<4, false>;
        case 9: return ls ? update_block_kernel_l<4, true>(ls) : update_kernel<4, true>;
        default: return nullptr;
    }
}

}  // namespace

int update_slabs(int C) { return slabs_of(C, kUpdVec); }

int update_stage_max_len() { return kUpdBlockMaxL; }

// Sequence groups per slab for update_kernel: enough CTAs for about
// kUpdCtasPerSm per SM, each warp with at least one request.
int update_groups(int N, int slabs, int sms) {
    const int64_t want = (static_cast<int64_t>(kUpdCtasPerSm) * sms + slabs - 1) / slabs;
    const int64_t most = ceil_div(N, kWarpsPerCta);
    const int64_t g = want < most ? want : most;
    return static_cast<int>(g < 1 ? 1 : g);
}

cudaError_t launch_update(const UpdArgs &a, cudaStream_t st, bool overlap) {
    const int ls = a.state_stage ? a.L : 0;
    const UpdKernel kern = update_kernel_for(a.width, a.act, ls);
    if (!kern) return cudaErrorInvalidValue;
    // CTA b: slab b % slabs and, for update_block_kernel, sequences
    // 8 (b / slabs) .. 8 (b / slabs) + 7 (one per warp); for update_kernel,
    // sequence group b / slabs.
    const int64_t groups = ls > 0 ? ceil_div(a.N, kWarpsPerCta) : a.groups;
    const int64_t ctas = static_cast<int64_t>(a.slabs) * groups;
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kCtaThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace ccc
