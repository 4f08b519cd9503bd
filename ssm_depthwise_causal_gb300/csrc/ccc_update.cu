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
// Mapping.  A CTA owns one 32*VEC-channel slab and a contiguous group of
// sequences; its 8 warps take the group's sequences in turn (warp w: the
// group's w-th, (w+8)-th, ... sequence).  The slab's taps and bias are staged
// once per CTA in shared memory (coalesced global reads).  For each of its
// sequences a warp reads the window, walks the new tokens U at a time and
// writes the slot.  Reads of the slot precede every write to it in the
// warp's program order, and no other warp touches the slot's channels (live
// slots are unique; slabs are disjoint), so the in-place update needs no
// synchronisation beyond the warp.
//
// For a dense history-contiguous pool ([slots][C][L], L <= kUpdStageL) the
// warp moves the slot's whole [256 ch][L] block: cp.async lands it (and the
// first U new tokens) in shared memory with coalesced 16-byte copies, the
// warp transposes it into a position-major [L][256] copy where every
// position of a lane's 8 channels is one conflict-free 16-byte vector, and
// writes the block back the same way (positions not written keep their
// bits).  The copies for a warp's next sequence are issued as soon as the
// current one has been transposed, and the offsets, slot and accepted count
// are loaded two sequences ahead, so a warp's memory round trips overlap its
// arithmetic.  A channel-contiguous pool is read and written one 16-byte
// vector per lane and position; any other layout element by element.
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
// CTAs the sequence groups are sized for, per SM (more groups: more CTAs,
// fewer requests per warp).
constexpr int kUpdCtasPerSm = CCC_UPD_CTAS_PER_SM;
constexpr int kUpdStageL = 8;  // longest history the shared-memory path stages
constexpr int kUpdSlab = 32 * kUpdVec;

// Element (slot q, channels c0.., position p) for the unstaged layouts.
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

// The request's slot block is staged (dense pool, live slot, new tokens).
__device__ __forceinline__ bool req_staged(const UpdArgs &a, const Req &r) {
    return r.n >= 0 && r.e > r.s && r.q >= 0 && r.q < a.n_slots;
}

// LS > 0: the pool is dense history-contiguous with L = LS (a compile-time
// constant, so the block transposition below is straight-line code); LS = 0:
// any other layout, L from the arguments.
template <int W, bool ACT, int LS>
__global__ void __launch_bounds__(kCtaThreads, kUpdMinBlocks) update_kernel(const UpdArgs a) {
    constexpr int VEC = kUpdVec, NV = VEC / 2, U = kUpdUnroll;
    constexpr int H = W - 1;
    constexpr int SLAB = kUpdSlab;
    constexpr bool kStaged = LS > 0;
    constexpr int LB = kStaged ? LS : 1;
    static_assert(LS == 0 || (LS >= H && LS <= kUpdStageL), "staged history length");
    __shared__ __align__(16) float s_tap[W + 1][SLAB];  // taps 0..W-1 and the bias
    // Dynamic shared memory (staged layout only), per warp: the landing copy
    // of a slot block (channel-major), the working copy (position-major) and
    // the first U new tokens.
    extern __shared__ __align__(16) uint16_t upd_dyn[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slab = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.slabs));
    const int grp = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.slabs));
    const int n_beg = static_cast<int>(static_cast<int64_t>(grp) * a.N / a.groups);
    const int n_end = static_cast<int>(static_cast<int64_t>(grp + 1) * a.N / a.groups);

    // Requests in flight: the current one and the next two (loads issued
    // before the taps' barrier).
    int n = n_beg + warp;
    Req cur = load_req(a, n, n_end);
    Req nx1 = load_req(a, n + kWarpsPerCta, n_end);

    // The slab's taps and bias, one channel per thread (FP32 in shared memory).
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
            s_tap[k][threadIdx.x] = t;
        }
        float bv = 0.0f;
        if (ok && a.b_kind == 1) bv = __ldg(reinterpret_cast<const float *>(a.b) + c);
        if (ok && a.b_kind == 2) bv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.b)[c]);
        s_tap[W][threadIdx.x] = bv;
    }
    __syncthreads();
    if (cur.n < 0) return;  // whole warp, after the CTA barrier

    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;
    const int slab_ch = min(SLAB, a.C - slab * SLAB);
    const int blk_vecs = kStaged ? slab_ch * LS / 8 : 0;  // 16-byte vectors in a slot's block
    uint16_t *raw = upd_dyn + warp * (2 * LB + U) * SLAB;
    uint16_t *blk = raw + LB * SLAB;
    uint16_t *sx = blk + LB * SLAB;
    const uint32_t raw_sa = smem_addr(raw), sx_sa = smem_addr(sx);

    // cp.async of request r's block and first U new tokens (staged layout).
    auto issue = [&](const Req &r) {
        if constexpr (kStaged) {
            if (req_staged(a, r)) {
                const uint16_t *g = a.state + static_cast<int64_t>(r.q) * a.st_slot + static_cast<int64_t>(slab) * SLAB * LS;
#pragma unroll
                for (int k = 0; k < LS; ++k) {
                    const int i = lane + 32 * k;
                    if (i < blk_vecs) cp_async<16>(raw_sa + 16 * i, g + 8 * i, true);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const bool ok = act && r.s + u < r.e;
                    cp_async<16>(sx_sa + 2 * (u * SLAB + lane * VEC),
                                 ok ? a.x + static_cast<int64_t>(r.s + u) * a.xs + c0 : a.x, ok);
                }
            }
            cp_async_commit();
        }
    };
    issue(cur);

    while (true) {
        const Req nx2 = load_req(a, n + 2 * kWarpsPerCta, n_end);  // used two iterations on
        const int len = cur.e - cur.s;
        const int q = cur.q;
        const uint16_t *xrow = a.x + static_cast<int64_t>(cur.s) * a.xs + c0;
        uint16_t *orow = a.out + static_cast<int64_t>(cur.s) * a.os + c0;
        const bool pool = len > 0 && q >= 0 && q < a.n_slots;
        const bool staged = kStaged && pool;
        const int acc = min(max(cur.acc, 1), a.L - H + 1);
        const int n_write = min(len + H - 1, a.L);  // positions written

        Raw<NV> xr0[U];  // the first U new tokens
        Raw<NV> hr[H];   // the W-1 values before them
#pragma unroll
        for (int p = 0; p < H; ++p) hr[p] = raw_zero<NV>();
        if constexpr (kStaged) {
            cp_async_wait(0);
            __syncwarp();
            if (staged) {
                // channel-major raw -> position-major blk.  Vector i + 32 k of
                // the block starts at element 8 i + 256 k; with L known at
                // compile time every (channel, position) is a constant plus
                // the lane's own start.
                const int ch_l = (8 * lane) / LS, p_l = (8 * lane) % LS;
#pragma unroll
                for (int k = 0; k < LS; ++k) {
                    const int i = lane + 32 * k;
                    if (i < blk_vecs) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(raw + 8 * i);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const int d = 256 * k + t;
                            const int pp = p_l + d % LS, cc = ch_l + d / LS;
                            const int p = pp >= LS ? pp - LS : pp, ch = pp >= LS ? cc + 1 : cc;
                            blk[p * SLAB + ch] = static_cast<uint16_t>(t & 1 ? w4[t >> 1] >> 16 : w4[t >> 1] & 0xffffu);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) xr0[u] = ld_rw<NV>(sx + u * SLAB + lane * VEC);
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    xr0[u] = (act && q != -1 && u < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(u) * a.xs)
                                                         : raw_zero<NV>();
            }
            __syncwarp();  // the landing buffers are free: start the next request's copies
            issue(nx1);
            if (staged && act)
#pragma unroll
                for (int p = 0; p < H; ++p) hr[p] = ld_rw<NV>(blk + (acc - 1 + p) * SLAB + lane * VEC);
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u)
                xr0[u] = (act && q != -1 && u < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(u) * a.xs)
                                                     : raw_zero<NV>();
            if (pool && act)
#pragma unroll
                for (int p = 0; p < H; ++p) hr[p] = state_get<NV>(a, q, acc - 1 + p, c0);
        }

        if (len > 0 && q == -1) {  // padded request: zero output, no state access
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < len; ++r) st_stream<NV>(orow + static_cast<int64_t>(r) * a.os, z);
            }
        } else if (len > 0) {
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
            if constexpr (kStaged) {
                if (staged) {
                    // position-major blk -> channel-major global block, whole
                    // (positions not written keep the bits they were read with)
                    __syncwarp();
                    uint16_t *g = a.state + static_cast<int64_t>(q) * a.st_slot + static_cast<int64_t>(slab) * SLAB * LS;
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
                            reinterpret_cast<uint4 *>(g)[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
            }
        }
        __syncwarp();  // blk is rewritten by the next request's transposition
        n += kWarpsPerCta;
        if (nx1.n < 0) break;
        cur = nx1;
        nx1 = nx2;
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

// Sequence groups per slab: enough CTAs for about two per SM, each warp with
// at least one request.
int update_groups(int N, int slabs, int sms) {
    const int64_t want = (static_cast<int64_t>(kUpdCtasPerSm) * sms + slabs - 1) / slabs;
    const int64_t most = ceil_div(N, kWarpsPerCta);
    const int64_t g = want < most ? want : most;
    return static_cast<int>(g < 1 ? 1 : g);
}

cudaError_t launch_update(const UpdArgs &a, cudaStream_t st) {
    const int ls = a.state_stage ? a.L : 0;
    const UpdKernel kern = update_kernel_for(a.width, a.act, ls);
    if (!kern) return cudaErrorInvalidValue;
    const size_t dyn = ls > 0 ? static_cast<size_t>(kWarpsPerCta) * (2 * ls + kUpdUnroll) * kUpdSlab * 2 : 0;
    if (dyn > 0) {
        // Opt in to this much dynamic shared memory (with the static taps it
        // can pass the 48 KB default), once per device and instantiation
        // (width, activation, staged length).
        static bool attr_set[64][6][kUpdStageL + 1] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const int slot = (a.width - 2) * 2 + (a.act ? 1 : 0);
        if (dev < 0 || dev >= 64 || !attr_set[dev][slot][ls]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev][slot][ls] = true;
        }
    }
    // CTA b: slab b % slabs, sequence group b / slabs.
    const int64_t ctas = static_cast<int64_t>(a.slabs) * a.groups;
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    kern<<<dim3(static_cast<unsigned>(ctas)), kCtaThreads, dyn, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ccc
