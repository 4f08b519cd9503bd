// ccc_update.cu -- the speculative / single-token decode step: the causal
// depthwise Conv1d (+ SiLU) of a few new tokens per sequence from the
// history held in the conv_state pool, and the pool update for the next step.
//
// FlashInfer "flashinfer.mamba.causal_conv1d_fn" (Notes): after a prefill,
// the first speculative update uses accepted count 1.  Reading of that rule
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
// Mapping.  One warp per (sequence, 32*VEC-channel slab); the 8 warps of a
// CTA take 8 consecutive sequences on the same slab, so the slab's taps and
// bias are staged once per CTA in shared memory (tap-major, coalesced global
// reads) instead of once per warp.  A warp reads the window (registers),
// walks the sequence's tokens U at a time and writes the slot.  Reads of the
// slot precede every write to it in the warp's program order, and no other
// warp touches the slot's channels (live slots are unique; slabs are
// disjoint), so the in-place update needs no synchronisation beyond the
// warp.  For a dense history-contiguous pool ([slots][C][L], L <=
// kUpdStageL) the warp copies the slot's whole [256 ch][L] block with
// coalesced 16-byte loads and transposes it into a position-major [L][256]
// copy in shared memory, where every position of the lane's 8 channels is one
// conflict-free 16-byte vector; the block goes back the same way (positions
// not written keep their bits).  A channel-contiguous pool is read and
// written one 16-byte vector per lane and position; any other layout element
// by element.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

constexpr int kUpdVec = 8;
constexpr int kUpdUnroll = 4;
constexpr int kUpdStageL = 8;  // longest history the shared-memory path stages

// Element (slot q, channels c0.., position p) for the general layouts.
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

// LS > 0: the pool is dense history-contiguous with L = LS (a compile-time
// constant, so the block transposition below is straight-line code); LS = 0:
// any other layout, L from the arguments.
template <int W, bool ACT, int LS>
__global__ void __launch_bounds__(kCtaThreads, kUpdMinBlocks) update_kernel(const UpdArgs a) {
    constexpr int VEC = kUpdVec, NV = VEC / 2, U = kUpdUnroll;
    constexpr int H = W - 1;
    static_assert(LS == 0 || (LS >= H && LS <= kUpdStageL), "staged history length");
    constexpr int SLAB = 32 * VEC;
    __shared__ __align__(16) float s_tap[W + 1][SLAB];  // taps 0..W-1 and the bias of this slab
    __shared__ __align__(16) uint16_t s_blk[kWarpsPerCta][(LS > 0 ? LS : 1) * SLAB];  // position-major
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slab = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.slabs));
    const int n = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.slabs)) * kWarpsPerCta + warp;

    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;
    uint16_t *blk = s_blk[warp];

    // Every load that does not depend on another is issued before the CTA
    // barrier: this warp's offsets, slot and accepted count, the slab's taps
    // and bias (one channel per thread), then the new tokens and the slot's
    // block, so the step costs two dependent memory round trips.
    // Offsets are clamped to [0, rows] so a bad value cannot leave the buffers.
    const bool has_n = n < a.N;
    const int64_t rows = a.rows;
    int s = 0, e = 0, q = -1, acc = 1;
    if (has_n) {
        s = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n)), int64_t{0}), rows));
        e = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n + 1)), static_cast<int64_t>(s)), rows));
        q = __ldg(a.cache + n);
        if (a.accepted) acc = __ldg(a.accepted + n);
    }
    float tv[W + 1];
    {
        const int c = slab * SLAB + static_cast<int>(threadIdx.x);
        const bool ok = c < a.C;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            float t = 0.0f;
            if (ok) {
                t = a.w_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.w)[W * c + k])
                             : __ldg(reinterpret_cast<const float *>(a.w) + W * c + k);
            }
            tv[k] = t;
        }
        float bv = 0.0f;
        if (ok && a.b_kind == 1) bv = __ldg(reinterpret_cast<const float *>(a.b) + c);
        if (ok && a.b_kind == 2) bv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.b)[c]);
        tv[W] = bv;
    }
    const int len = e - s;
    const bool work = has_n && len > 0 && q != -1;
    const uint16_t *xrow = a.x + static_cast<int64_t>(s) * a.xs + c0;
    uint16_t *orow = a.out + static_cast<int64_t>(s) * a.os + c0;
    Raw<NV> xr0[U];  // the first U new tokens (independent of the state)
#pragma unroll
    for (int u = 0; u < U; ++u)
        xr0[u] = (work && act && u < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(u) * a.xs) : raw_zero<NV>();

    const bool pool = work && q >= 0 && q < a.n_slots;
    acc = min(max(acc, 1), a.L - H + 1);
    const int n_write = min(len + H - 1, a.L);  // positions written
    constexpr bool kStaged = LS > 0;
    const bool staged = kStaged && pool;
    const int L = kStaged ? LS : a.L;
    // The staged block: this slab's channels x L positions of slot q,
    // contiguous (channel-major) in a dense history-contiguous pool.
    const int slab_ch = min(SLAB, a.C - slab * SLAB);
    const int blk_vecs = slab_ch * L / 8;  // 16-byte vectors in the block
    uint16_t *gblk = pool ? a.state + static_cast<int64_t>(q) * a.st_slot + static_cast<int64_t>(slab) * SLAB * L
                          : nullptr;
    uint4 bvec[kStaged ? LS : 1];  // vector lane + 32 k of the block
    if constexpr (kStaged) {
#pragma unroll
        for (int k = 0; k < LS; ++k) {
            const int i = lane + 32 * k;
            bvec[k] = (staged && i < blk_vecs) ? reinterpret_cast<const uint4 *>(gblk)[i] : make_uint4(0u, 0u, 0u, 0u);
        }
    }

#pragma unroll
    for (int k = 0; k <= W; ++k) s_tap[k][threadIdx.x] = tv[k];
    __syncthreads();
    if (!has_n || len == 0) return;  // whole warp, after the CTA barrier
    if (q == -1) {  // padded request: zero output, no state access
        if (act) {
            const Raw<NV> z = raw_zero<NV>();
            for (int r = 0; r < len; ++r) st_stream<NV>(orow + static_cast<int64_t>(r) * a.os, z);
        }
        return;
    }

    // The W-1 values before the first new token.
    Raw<NV> hr[H];
#pragma unroll
    for (int p = 0; p < H; ++p) hr[p] = raw_zero<NV>();
    if (staged) {
        // channel-major global block -> position-major blk[p][ch].  Vector
        // i + 32k of the block starts at element 8 i + 256 k; with L known at
        // compile time every (channel, position) below is a constant plus
        // the lane's own start.
        if constexpr (kStaged) {
            const int ch_l = (8 * lane) / LS, p_l = (8 * lane) % LS;
#pragma unroll
            for (int k = 0; k < LS; ++k) {  // the block holds slab_ch * LS / 8 <= 32 * LS vectors
                const int i = lane + 32 * k;
                if (i < blk_vecs) {
                    const uint4 v = bvec[k];
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        // element 8 i + t = 8 lane + (256 k + t)
                        const int d = 256 * k + t;
                        const int pp = p_l + d % LS, cc = ch_l + d / LS;
                        const int p = pp >= LS ? pp - LS : pp, ch = pp >= LS ? cc + 1 : cc;
                        blk[p * SLAB + ch] = static_cast<uint16_t>(t & 1 ? w4[t >> 1] >> 16 : w4[t >> 1] & 0xffffu);
                    }
                }
            }
        }
        __syncwarp();
        if (act)
#pragma unroll
            for (int p = 0; p < H; ++p) hr[p] = ld_rw<NV>(blk + (acc - 1 + p) * SLAB + lane * VEC);
    } else if (pool && act) {
#pragma unroll
        for (int p = 0; p < H; ++p) hr[p] = state_get<NV>(a, q, acc - 1 + p, c0);
    }

    // Positions 0 .. W-3: the 2nd .. last value just read.
    if (pool && act) {
#pragma unroll
        for (int p = 0; p + 1 < H; ++p) {
            if (p < n_write) {
                if (staged) {
                    st_plain<NV>(blk + p * SLAB + lane * VEC, hr[p + 1]);
                } else {
                    state_put<NV>(a, q, p, c0, hr[p + 1]);
                }
            }
        }
    }

    float2 wt[W][NV], bb[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) wt[k][v] = reinterpret_cast<const float2 *>(&s_tap[k][lane * VEC])[v];
        bb[v] = reinterpret_cast<const float2 *>(&s_tap[W][lane * VEC])[v];
    }
    float2 hw[H][NV];
#pragma unroll
    for (int p = 0; p < H; ++p) unpack<NV>(hr[p], hw[p]);

    for (int base = 0; base < len; base += U) {
        Raw<NV> xr[U];
        if (base == 0) {
#pragma unroll
            for (int u = 0; u < U; ++u) xr[u] = xr0[u];
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u)
                xr[u] = (act && base + u < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(base + u) * a.xs)
                                                : raw_zero<NV>();
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = base + u;
            if (j >= len) break;
            float2 hc[NV];
            unpack<NV>(xr[u], hc);
            Raw<NV> y;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                y.u[v] = f2_to_bf2(activate2<ACT>(conv_pre<W, NV>(wt, bb[v], hw, hc[v], v)));
#pragma unroll
                for (int k = 0; k + 1 < H; ++k) hw[k][v] = hw[k + 1][v];
                hw[H - 1][v] = hc[v];
            }
            if (act) {
                st_stream<NV>(orow + static_cast<int64_t>(j) * a.os, y);
                // token j is history value H + j: position H - 1 + j
                const int p = H - 1 + j;
                if (pool && p < n_write) {
                    if (staged) {
                        st_plain<NV>(blk + p * SLAB + lane * VEC, xr[u]);
                    } else {
                        state_put<NV>(a, q, p, c0, xr[u]);
                    }
                }
            }
        }
    }

    if (staged) {
        // position-major blk -> channel-major global block, whole (positions
        // not written keep the bits they were read with)
        __syncwarp();
        if constexpr (kStaged) {
            const int ch_l = (8 * lane) / LS, p_l = (8 * lane) % LS;
#pragma unroll
            for (int k = 0; k < LS; ++k) {
                const int i = lane + 32 * k;
                if (i < blk_vecs) {
                    uint32_t w4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int d = 256 * k + t;
                        const int pp = p_l + d % LS, cc = ch_l + d / LS;
                        const int p = pp >= LS ? pp - LS : pp, ch = pp >= LS ? cc + 1 : cc;
                        const uint32_t h = blk[p * SLAB + ch];
                        w4[t >> 1] |= t & 1 ? h << 16 : h;
                    }
                    reinterpret_cast<uint4 *>(gblk)[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
        }
    }
}

using UpdKernel = void (*)(const UpdArgs);

// The instantiation for (W, ACT) and a staged history length ls (0: none).
template <int W, bool ACT>
UpdKernel update_kernel_l(int ls) {
    switch (ls) {
        case 0: return update_kernel<W, ACT, 0>;
        case 1: if constexpr (W - 1 <= 1) return update_kernel<W, ACT, (W - 1 <= 1 ? 1 : 0)>; else return nullptr;
        case 2: if constexpr (W - 1 <= 2) return update_kernel<W, ACT, (W - 1 <= 2 ? 2 : 0)>; else return nullptr;
        case 3: return update_kernel<W, ACT, 3>;
        case 4: return update_kernel<W, ACT, 4>;
        case 5: return update_kernel<W, ACT, 5>;
        case 6: return update_kernel<W, ACT, 6>;
        case 7: return update_kernel<W, ACT, 7>;
        case 8: return update_kernel<W, ACT, 8>;
        default: return nullptr;
    }
}

UpdKernel update_kernel_for(int width, int act, int ls) {
    switch (width * 2 + (act ? 1 : 0)) {
        case 4: return update_kernel_l<2, false>(ls);
        case 5: return update_kernel_l<2, true>(ls);
        case 6: return update_kernel_l<3, false>(ls);
        case 7: return update_kernel_l<3, true>(ls);
        case 8: return update_kernel_l<4, false>(ls);
        case 9: return update_kernel_l<4, true>(ls);
        default: return nullptr;
    }
}

}  // namespace

int update_slabs(int C) { return slabs_of(C, kUpdVec); }

int update_stage_max_len() { return kUpdStageL; }

cudaError_t launch_update(const UpdArgs &a, cudaStream_t st) {
    const UpdKernel kern = update_kernel_for(a.width, a.act, a.state_stage ? a.L : 0);
    if (!kern) return cudaErrorInvalidValue;
    // CTA b: slab b % slabs, sequences (b / slabs) * 8 + warp.
    const int64_t ctas = static_cast<int64_t>(a.slabs) * ceil_div(a.N, kWarpsPerCta);
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(ctas));
    kern<<<grid, kCtaThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ccc
