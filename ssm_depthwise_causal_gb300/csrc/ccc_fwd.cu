// ccc_fwd.cu -- forward kernel: packed causal depthwise Conv1d (+ SiLU)
// with the conv_state gather/scatter fused in.
//
// FlashInfer "flashinfer.mamba.causal_conv1d_fn" (Parameters): for token j of
// sequence n and channel c, z = bias + w0*h[j] + w1*h[j+1] + w2*h[j+2] +
// w3*h[j+3] (bias first, then the four FMAs, tap 3 on the current token),
// out = BF16(z * sigmoid(z)); h starts with three state values (slot
// cache_indices[n], positions 0:3, when has_initial_state[n]) or zeros; a -1
// slot gives zero output and no state access; each nonempty live sequence
// leaves its last three raw history values in positions 0:3.  The kernel is
// a template over the width W (2..4: W-1 history rows and state positions,
// Megatron-Core "core.ssm.causal_conv1d", causal_conv1d_cp: weight [D, W])
// and the activation (SiLU or none, the same page's `activation`); W = 4
// with SiLU is FlashInfer's contract.
//
// Mapping.  A warp owns one task: a 32*VEC-channel slab and a run of rows
// (RunWalker: equal shares of the valid rows).  Lane l holds channels
// [c0, c0+VEC) with c0 = (slab*32 + l)*VEC, keeps the H = W-1 previous rows in
// registers as FP32 pairs, and streams its rows U at a time (U independent
// 16-byte loads in flight per lane before any math; lanes 0..U-1 also ask L2
// to prefetch the warp's slab a few rows ahead).  The window is carried from
// one segment to the next along a sequence, so the H rows before a walk are
// re-read (from L2: the neighbouring run) only where a run starts inside a
// sequence.  The rows before a sequence's first row come from the state slot
// (or are zeros).  The warp whose run holds a sequence's first row is the
// only one that touches that slot: it reads the initial history and, after
// its own rows, writes the final values (for len >= H these are x's last H
// rows, re-read from global; for shorter sequences they mix the initial
// history and x), so the read always precedes the write in program order and
// no other warp can race with it.
//
// The grid is one resident wave of CTAs of 8 warps; warp g takes slab
// g % slabs and run g / slabs.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

// State positions 0..H-1 of slot q (position 0 = oldest).
template <int NV, int H>
__device__ __forceinline__ void gather_state(const uint16_t *state, int64_t st_slot, int64_t st_c, int64_t st_l,
                                             bool vec, int q, int c0, Raw<NV> (&hr)[H]) {
    const uint16_t *base = state + static_cast<int64_t>(q) * st_slot;
    if (vec) {
#pragma unroll
        for (int p = 0; p < H; ++p) hr[p] = ld_rw<NV>(base + p * st_l + c0);
    } else {
#pragma unroll
        for (int p = 0; p < H; ++p) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const uint32_t lo = base[(c0 + 2 * v) * st_c + p * st_l];
                const uint32_t hi = base[(c0 + 2 * v + 1) * st_c + p * st_l];
                hr[p].u[v] = lo | (hi << 16);
            }
        }
    }
}

// One state position p of slot q for this lane's channels.
template <int NV>
__device__ __forceinline__ void put_state(uint16_t *state, int64_t st_slot, int64_t st_c, int64_t st_l, bool vec,
                                          int q, int p, int c0, const Raw<NV> &val) {
    uint16_t *base = state + static_cast<int64_t>(q) * st_slot + static_cast<int64_t>(p) * st_l;
    if (vec) {
        st_plain<NV>(base + c0, val);
    } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            base[(c0 + 2 * v) * st_c] = static_cast<uint16_t>(val.u[v] & 0xffffu);
            base[(c0 + 2 * v + 1) * st_c] = static_cast<uint16_t>(val.u[v] >> 16);
        }
    }
}

// One output row: y = act(conv_pre) for the VEC channels of this lane, then
// the history window moves one row on (hw[0] oldest .. hw[H-1] newest).
template <int W, bool ACT, int NV>
__device__ __forceinline__ Raw<NV> fwd_row(const float2 (&wt)[W][NV], const float2 (&bb)[NV],
                                           float2 (&hw)[W - 1][NV], const Raw<NV> &xr) {
    float2 hc[NV];
    unpack<NV>(xr, hc);
    Raw<NV> y;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        y.u[v] = f2_to_bf2(activate2<ACT>(conv_pre<W, NV>(wt, bb[v], hw, hc[v], v)));
#pragma unroll
        for (int k = 0; k + 1 < W - 1; ++k) hw[k][v] = hw[k + 1][v];
        hw[W - 2][v] = hc[v];
    }
    return y;
}

template <int VEC, int U, int W, bool ACT>
__global__ void __launch_bounds__(kCtaThreads, kFwdMinBlocks) fwd_kernel(const FwdArgs a) {
    constexpr int NV = VEC / 2;
    constexpr int H = W - 1;  // history rows
    __shared__ SeqMeta<kFwdStageSeqs> meta;  // (before any exit: the whole CTA stages it)
    __shared__ __align__(16) unsigned char taps_buf[kWarpsPerCta][32 * VEC * W * 4];
    const bool staged = stage_meta(meta, a.cu, a.N, a.rows, a.cache, a.has_init);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kWarpsPerCta + warp;  // this warp's task
    if (gw >= a.slabs * a.runs) return;               // (whole warp) no task in the last CTA
    const int slab = gw % a.slabs, run = gw / a.slabs;
    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const bool full = (slab + 1) * 32 * VEC <= a.C;  // warp-uniform: all lanes have channels
    const int c0 = act ? cv * VEC : 0;
    const int rows_i = static_cast<int>(a.rows);  // host-checked <= 2^31 - 1

    // Taps: with aligned taps the warp's block is copied (cp.async) into its
    // shared buffer while the run search below runs, then read back.
    float2 wt[W][NV], bb[NV];
    if (a.taps_vec) {
        issue_taps<NV, W>(a.w, a.w_bf16, slab * 32 * VEC, a.C, lane, smem_addr(taps_buf[warp]));
        load_bias_vec<NV>(a.b, a.b_kind, c0, act, bb);
    } else {
        load_taps_w<NV, W>(a.w, a.w_bf16, a.b, a.b_kind, c0, act, wt, bb);
    }

    RunWalker<kFwdChunk> walk;
    walk.init(a.cu, a.N, a.rows, run, a.runs, H, false, lane, kFwdWalkRows, staged ? meta.cu : nullptr);
    if (a.taps_vec) {
        cp_async_wait(0);
        take_taps<NV, W>(a.w_bf16, lane, act, taps_buf[warp], wt);
    }

    // Everything above reads only the offsets, slots, flags, taps and bias.
    // Launched as a programmatic dependent (CCC_OPT_OVERLAP_PROLOGUE) it may
    // have run while the previous kernel finished; wait for that kernel
    // before reading x, the pool or the saved history, or writing anything.
    // (A no-op for an ordinary launch.)
    grid_dependency_wait();

    // The H rows before the current one, oldest first.  (With 3-row batches
    // the window comes back to the same registers every batch; a ring
    // indexed by walk row, as in the backward, measured no faster here.)
    float2 hw[H][NV];

    Item t;
    bool cont, more;
    int q = -2;
    bool has_init_n = false;
    while (walk.next(a.cu, a.rows, lane, t, cont, more)) {
        if (!cont) {  // a new sequence (or the run's first rows): its slot and flag
            if (staged) {
                q = meta.cache[t.n];
                has_init_n = meta.flag[t.n] != 0;
            } else {
                q = a.cache ? __ldg(a.cache + t.n) : -2;
                has_init_n = a.has_init != nullptr && __ldg(a.has_init + t.n) != 0;
            }
        }
        const int nr = t.nr;
        if (nr <= 0) continue;
        const int o0 = t.r0 - t.s, L = t.e - t.s;
        const uint16_t *xrow = a.x + static_cast<int64_t>(t.r0) * a.xs + c0;
        uint16_t *orow = a.out + static_cast<int64_t>(t.r0) * a.os + c0;

        if (q == -1) {  // padded request: zero output, no state access
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < nr; ++r) st_stream<NV>(orow + static_cast<int64_t>(r) * a.os, z);
                if (o0 == 0 && a.hist)
#pragma unroll
                    for (int p = 0; p < H; ++p)
                        st_plain<NV>(a.hist + (static_cast<int64_t>(t.n) * H + p) * a.C + c0, z);
            }
            continue;
        }
        const bool pool = a.state != nullptr && q >= 0 && q < a.n_slots;
        const bool rd = o0 == 0 && pool && has_init_n;

        if (!cont) {
            // The H history rows before r0 (raw BF16 bits): the initial
            // state (or zeros) for a sequence's first rows, else x rows.
            Raw<NV> hr[H];
#pragma unroll
            for (int p = 0; p < H; ++p) hr[p] = raw_zero<NV>();
            if (o0 == 0) {
                if (rd && act) gather_state<NV, H>(a.state, a.st_slot, a.st_c, a.st_l, a.state_vec, q, c0, hr);
                if (a.hist && act)
#pragma unroll
                    for (int p = 0; p < H; ++p)
                        st_plain<NV>(a.hist + (static_cast<int64_t>(t.n) * H + p) * a.C + c0, hr[p]);
            } else if (act) {
#pragma unroll
                for (int p = 0; p < H; ++p) hr[p] = ld_ro<NV>(xrow - static_cast<int64_t>(H - p) * a.xs);
            }
#pragma unroll
            for (int p = 0; p < H; ++p) unpack<NV>(hr[p], hw[p]);
        }

        int base = 0;
        if (full) {
            // Every lane active and the batch inside the segment: no guards.
            const uint16_t *xp = xrow;
            uint16_t *op = orow;
            for (; base + U <= nr; base += U) {
                if constexpr (kFwdPrefetch > 0) {
                    // lanes 0..U-1: the warp's slab of row r0+base+PF+lane into L2
                    // (as a difference: rows may be 2^31 - 1)
                    const int ahead = kFwdPrefetch + lane;
                    if (lane < U && ahead < rows_i - (t.r0 + base))
                        prefetch_l2(xp + static_cast<int64_t>(ahead) * a.xs - c0 + slab * 32 * VEC, 32 * VEC * 2);
                }
                Raw<NV> cur[U];
                const uint16_t *lp = xp;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    cur[u] = ld_ro<NV>(lp);
                    lp += a.xs;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    st_stream<NV>(op, fwd_row<W, ACT, NV>(wt, bb, hw, cur[u]));
                    op += a.os;
                }
                xp = lp;
            }
        }
        for (; base < nr; base += U) {  // remainder, or a partly filled slab
            Raw<NV> cur[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                cur[u] = (act && base + u < nr) ? ld_ro<NV>(xrow + static_cast<int64_t>(base + u) * a.xs)
                                                : raw_zero<NV>();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (base + u >= nr) break;
                const Raw<NV> y = fwd_row<W, ACT, NV>(wt, bb, hw, cur[u]);
                if (act) st_stream<NV>(orow + static_cast<int64_t>(base + u) * a.os, y);
            }
        }

        // Final H raw history values h[L .. L+H) -> positions 0:H, by the
        // warp that read the initial ones (read before write; the values
        // come from x, whoever computes those rows).
        if (o0 == 0 && pool && L > 0 && act) {
            Raw<NV> init[H];
#pragma unroll
            for (int p = 0; p < H; ++p) init[p] = raw_zero<NV>();
            if (rd && L < H)  // still unwritten
                gather_state<NV, H>(a.state, a.st_slot, a.st_c, a.st_l, a.state_vec, q, c0, init);
            Raw<NV> fin[H];
#pragma unroll
            for (int p = 0; p < H; ++p) {
                const int idx = L < H ? L + p : H;  // history index L + p (>= H past the initial values)
                if (L >= H - p) {
                    fin[p] = ld_ro<NV>(a.x + (static_cast<int64_t>(t.e) - H + p) * a.xs + c0);
                } else {
                    fin[p] = init[0];
#pragma unroll
                    for (int j = 1; j < H; ++j)
                        if (idx == j) fin[p] = init[j];
                }
            }
#pragma unroll
            for (int p = 0; p < H; ++p) put_state<NV>(a.state, a.st_slot, a.st_c, a.st_l, a.state_vec, q, p, c0, fin[p]);
        }
    }
    // Let a kernel launched as this one's programmatic dependent start its
    // prologue (it waits for this grid's writes before reading them).
    grid_dependents_launch();
}

}  // namespace

// Rows per batch: a multiple of the history length where that is cheap (the
// sliding window then returns to the same registers every batch).
constexpr int fwd_unroll(int W) { return W == 4 ? kFwdUnrollW4 : kFwdUnroll; }

template <int W, bool ACT>
constexpr auto fwd_kernel_of() {
    return fwd_kernel<kFwdVec, fwd_unroll(W), W, ACT>;
}

using FwdKernel = void (*)(const FwdArgs);

// The instantiation for (width, activation); nullptr for an unsupported pair.
FwdKernel fwd_kernel_for(int width, int act) {
    switch (width * 2 + (act ? 1 : 0)) {
        case 4: return fwd_kernel_of<2, false>();
        case 5: return fwd_kernel_of<2, true>();
        case 6: return fwd_kernel_of<3, false>();
        case 7: return fwd_kernel_of<3, true>();
        case 8: return fwd_kernel_of<4, false>();
        case 9: return fwd_kernel_of<4, true>();
        default: return nullptr;
    }
}

int fwd_ctas_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_kernel_for(4, 1), kCtaThreads, 0) != cudaSuccess ||
        n < 1)
        n = kFwdMinBlocks;
    return n;
}

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t st, bool overlap) {
    const FwdKernel kern = fwd_kernel_for(a.width, a.act);
    if (!kern) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(static_cast<int64_t>(a.slabs) * a.runs, kWarpsPerCta)));
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
