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
// Mapping.  One warp per (sequence, 32*VEC-channel slab): it reads the
// window (registers), walks the sequence's tokens U at a time and writes the
// slot.  Reads of the slot precede every write to it in the warp's program
// order, and no other warp touches the slot's channels (live slots are
// unique; slabs are disjoint), so the in-place update needs no
// synchronisation.  For a dense history-contiguous pool ([slots][C][L],
// L <= kUpdStageL) the warp moves the slot's whole [256 ch][L] block with
// coalesced 16-byte copies through shared memory (lanes then pick single
// positions there); a channel-contiguous pool is read and written one
// 16-byte vector per lane and position; any other layout element by element.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

constexpr int kUpdVec = 8;
constexpr int kUpdUnroll = 4;
constexpr int kUpdStageL = 8;  // longest history the shared-memory path stages
constexpr int kUpdStageBytes = 32 * kUpdVec * kUpdStageL * 2;  // per warp

// Position p of this lane's VEC channels from the staged [256 ch][L] block.
template <int NV>
__device__ __forceinline__ Raw<NV> staged_get(const uint16_t *blk, int L, int lane, int p) {
    Raw<NV> r;
    const uint16_t *c = blk + lane * 2 * NV * L + p;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const uint32_t lo = c[(2 * v) * L];
        const uint32_t hi = c[(2 * v + 1) * L];
        r.u[v] = lo | (hi << 16);
    }
    return r;
}

template <int NV>
__device__ __forceinline__ void staged_put(uint16_t *blk, int L, int lane, int p, const Raw<NV> &r) {
    uint16_t *c = blk + lane * 2 * NV * L + p;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        c[(2 * v) * L] = static_cast<uint16_t>(r.u[v] & 0xffffu);
        c[(2 * v + 1) * L] = static_cast<uint16_t>(r.u[v] >> 16);
    }
}

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

template <int W, bool ACT>
__global__ void __launch_bounds__(kCtaThreads, 2) update_kernel(const UpdArgs a) {
    constexpr int VEC = kUpdVec, NV = VEC / 2, U = kUpdUnroll;
    constexpr int H = W - 1;
    __shared__ __align__(16) uint16_t stage_all[kWarpsPerCta][kUpdStageBytes / 2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp;
    if (gw >= static_cast<int64_t>(a.slabs) * a.N) return;  // whole warp
    const int n = static_cast<int>(gw / a.slabs), slab = static_cast<int>(gw % a.slabs);
    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;
    uint16_t *blk = stage_all[warp];

    // Offsets clamped to [0, rows] so a bad value cannot leave the buffers.
    const int64_t rows = a.rows;
    const int s = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n)), int64_t{0}), rows));
    const int e = static_cast<int>(min(max(static_cast<int64_t>(__ldg(a.cu + n + 1)), static_cast<int64_t>(s)), rows));
    const int len = e - s;
    if (len == 0) return;
    const int q = __ldg(a.cache + n);
    const uint16_t *xrow = a.x + static_cast<int64_t>(s) * a.xs + c0;
    uint16_t *orow = a.out + static_cast<int64_t>(s) * a.os + c0;
    if (q == -1) {  // padded request: zero output, no state access
        if (act) {
            const Raw<NV> z = raw_zero<NV>();
            for (int r = 0; r < len; ++r) st_stream<NV>(orow + static_cast<int64_t>(r) * a.os, z);
        }
        return;
    }
    const bool pool = q >= 0 && q < a.n_slots;
    int acc = a.accepted ? __ldg(a.accepted + n) : 1;
    acc = min(max(acc, 1), a.L - H + 1);
    const int n_write = min(len + H - 1, a.L);  // positions written
    const bool staged = pool && a.state_stage;
    // The staged block: this slab's channels [slab*256, +256) x L positions of
    // slot q, contiguous in a dense history-contiguous pool.
    const int slab_ch = min(32 * VEC, a.C - slab * 32 * VEC);
    const int blk_vecs = slab_ch * a.L / 8;  // 16-byte vectors in the block
    uint16_t *gblk = pool ? a.state + static_cast<int64_t>(q) * a.st_slot + static_cast<int64_t>(slab) * 32 * VEC * a.L
                          : nullptr;

    // The W-1 values before the first new token.
    Raw<NV> hr[H];
#pragma unroll
    for (int p = 0; p < H; ++p) hr[p] = raw_zero<NV>();
    if (staged) {
        for (int i = lane; i < blk_vecs; i += 32)
            reinterpret_cast<uint4 *>(blk)[i] = reinterpret_cast<const uint4 *>(gblk)[i];
        __syncwarp();
        if (act)
#pragma unroll
            for (int p = 0; p < H; ++p) hr[p] = staged_get<NV>(blk, a.L, lane, acc - 1 + p);
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
                    staged_put<NV>(blk, a.L, lane, p, hr[p + 1]);
                } else {
                    state_put<NV>(a, q, p, c0, hr[p + 1]);
                }
            }
        }
    }

    float2 wt[W][NV], bb[NV];
    load_taps_w<NV, W>(a.w, a.w_bf16, a.b, a.b_kind, c0, act, wt, bb);
    float2 hw[H][NV];
#pragma unroll
    for (int p = 0; p < H; ++p) unpack<NV>(hr[p], hw[p]);

    for (int base = 0; base < len; base += U) {
        Raw<NV> xr[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            xr[u] = (act && base + u < len) ? ld_ro<NV>(xrow + static_cast<int64_t>(base + u) * a.xs) : raw_zero<NV>();
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
                        staged_put<NV>(blk, a.L, lane, p, xr[u]);
                    } else {
                        state_put<NV>(a, q, p, c0, xr[u]);
                    }
                }
            }
        }
    }

    if (staged) {
        // Write the block back whole (positions not written keep the bits
        // they were read with).
        __syncwarp();
        for (int i = lane; i < blk_vecs; i += 32)
            reinterpret_cast<uint4 *>(gblk)[i] = reinterpret_cast<const uint4 *>(blk)[i];
    }
}

using UpdKernel = void (*)(const UpdArgs);

UpdKernel update_kernel_for(int width, int act) {
    switch (width * 2 + (act ? 1 : 0)) {
        case 4: return update_kernel<2, false>;
        case 5: return update_kernel<2, true>;
        case 6: return update_kernel<3, false>;
        case 7: return update_kernel<3, true>;
        case 8: return update_kernel<4, false>;
        case 9: return update_kernel<4, true>;
        default: return nullptr;
    }
}

}  // namespace

int update_slabs(int C) { return slabs_of(C, kUpdVec); }

int update_stage_max_len() { return kUpdStageL; }

cudaError_t launch_update(const UpdArgs &a, cudaStream_t st) {
    const UpdKernel kern = update_kernel_for(a.width, a.act);
    if (!kern) return cudaErrorInvalidValue;
    const int64_t warps = static_cast<int64_t>(a.slabs) * a.N;
    const dim3 grid(static_cast<unsigned>(ceil_div(warps, kWarpsPerCta)));
    kern<<<grid, kCtaThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ccc
