// ccc_bwd.cu -- fused backward: dx, d_init_state and per-warp-task FP32
// dweight/dbias partials in one pass, then an ordered reduction.
//
// FlashInfer "cake_causal_conv1d_train.cake_causal_conv1d_kcp" (Returns): one
// kernel produces the input gradient and deterministic FP32 weight-gradient
// partials; Megatron-Core "core.ssm.causal_conv1d"
// (assert_causal_conv1d_deterministic): each warp task writes its own
// partial row to scratch and a second kernel adds the rows in a fixed order
// (no atomics), so the result does not depend on scheduling.
//
// Per token j of a live sequence (history index i = j for the 3 initial
// values, i = j + 3 for input rows):
//   z_j  = b + w0 h[j] + w1 h[j+1] + w2 h[j+2] + w3 h[j+3]        (recomputed)
//   dz_j = dy_j * s * (1 + z_j * (1 - s)),  s = sigmoid(z_j)
//   dH[i] = carry(i) + w0 dz_i + w1 dz_{i-1} + w2 dz_{i-2} + w3 dz_{i-3}
// with dz outside [0, len) taken as 0 and carry(i) = d_final_state[i - len]
// for the three indices past the end (the gradient of the state this
// sequence wrote).  The FMAs run carry first, then k = 0..3, exactly as in
// the forward's fragment rule, so a document split into fragments whose
// backward is chained through d_init_state -> d_final_state gives the
// unsplit dx and d_init_state bit for bit.
//
// Mapping.  As in the forward: a warp owns a 32*VEC-channel slab, a lane
// owns VEC channels, and each warp walks a run of rows (an equal share of
// the valid rows' cost, RunWalker).  Along one sequence the lane walks
// i = o0, o0+1, ... without a break: it keeps a sliding window of 3 history rows and the 3
// previous dz values in registers, emits dx for row i-3 once dz_i is known,
// and accumulates dz_j * h[j+k] and dz_j of its own rows into 5*VEC FP32
// registers.  Only where a walk starts inside a sequence does it re-read the
// 3 rows before it, and only where it stops before the sequence end does it
// read 3 rows past it (both from L2: the neighbouring warp's run).
//
// Widths and activation.  The kernel is a template over the width W (2..4:
// W-1 history rows, W-1 initial-state gradients, W taps; Megatron-Core
// causal_conv1d_cp, weight [D, W]) and the activation (SiLU, or none: then
// dz = dy); W = 4 with SiLU is the contract above, and "3" reads W-1.
//
// Determinism.  The number of runs per slab R is fixed by the host
// arguments rows and C only (never by the device or by device values); the warp
// with task (slab, run r) walks rows [r*T/R, (r+1)*T/R) (T = cu_seqlens[N])
// in order and writes partial[r][k][c] for its channels, so every partial sum
// has a fixed operand order; the reduce kernel then sums the R partials of
// every (k, c) in order r = 0..R-1.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

// Sliding windows as rings.  Row k of a walk keeps its history value and its
// dz in slot k % RS of two RS-slot rings (RS = the batch size U >= W).  A
// walk's batches start at multiples of U from the walk's first row, so row
// u of a batch always sits in slot u: every index below is a compile-time
// constant and nothing moves between rows.
// dz of row u for one channel pair: the pre-activation (bias, then tap k on
// history row u-H+k, then tap H on the current row -- the forward's operand
// order) through the activation's derivative.
template <int W, bool ACT, int RS, int NV>
__device__ __forceinline__ float2 ring_dz(const float2 (&wt)[W][NV], float2 b, const float2 (&hr)[RS][NV], float2 hc,
                                          float2 gy, int u, int v) {
    if constexpr (ACT) {
        float2 z = b;
#pragma unroll
        for (int k = 0; k < W - 1; ++k) z = __ffma2_rn(wt[k][v], hr[slot<RS>(u, W - 1 - k)][v], z);
        z = __ffma2_rn(wt[W - 1][v], hc, z);
        return activate2_grad<true>(z, gy);
    } else {
        return gy;
    }
}

// dH of row u: the carry first, then tap k on dz of row u-k (k = 0: dz).
template <int W, int RS, int NV>
__device__ __forceinline__ float2 ring_dh(const float2 (&wt)[W][NV], float2 carry, float2 dz,
                                          const float2 (&dr)[RS][NV], int u, int v) {
    float2 c = __ffma2_rn(wt[0][v], dz, carry);
#pragma unroll
    for (int k = 1; k < W; ++k) c = __ffma2_rn(wt[k][v], dr[slot<RS>(u, k)][v], c);
    return c;
}

// The weight / bias partial sums of row u: dz * h[u-H+k] for k < H, dz * h[u],
// and dz itself.
template <int W, int RS, int NV>
__device__ __forceinline__ void ring_partials(float2 (&g)[W][NV], float2 (&gb)[NV], float2 dz,
                                              const float2 (&hr)[RS][NV], float2 hc, int u, int v) {
#pragma unroll
    for (int k = 0; k < W - 1; ++k) g[k][v] = __ffma2_rn(dz, hr[slot<RS>(u, W - 1 - k)][v], g[k][v]);
    g[W - 1][v] = __ffma2_rn(dz, hc, g[W - 1][v]);
    gb[v] = __fadd2_rn(gb[v], dz);
}

// P = 0: each lane loads its U rows of x and dy straight into registers.
// P > 0: each lane streams the rows of its walk through a P-stage ring of
// U-row batches in shared memory (cp.async), keeping up to P-1 batches in
// flight ahead of the math.  CW: warps per CTA (kWarpsPerCta for a grid that
// fills every SM, 1 for a smaller one, whose one-warp CTAs the block
// scheduler then spreads over the SMs instead of packing 8 tasks on one).
template <int VEC, int U, int P, int W, bool ACT, int CW>
__global__ void __launch_bounds__(kCtaThreads, kBwdMinBlocks) bwd_kernel(const BwdArgs a) {
    constexpr int NV = VEC / 2;
    constexpr int H = W - 1;                            // history rows
    constexpr int VB = VEC * 2;                         // bytes per lane per row
    constexpr int RING_WARP = P * U * 2 * 32 * VB;      // ring bytes per warp
    static_assert(P == 0 || kBwdChunk % U == 0, "segments must be whole batches");
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    __shared__ SeqMeta<kBwdStageSeqs> meta;  // (before any exit: the whole CTA stages it)
    const bool staged = stage_meta(meta, a.cu, a.N, a.rows, a.cache, a.has_init);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * CW + warp;  // this warp's task
    if (gw >= a.slabs * a.runs) return;               // (whole warp) no task in the last CTA
    const int slab = gw % a.slabs, run = gw / a.slabs;
    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const bool full = (slab + 1) * 32 * VEC <= a.C;  // warp-uniform: all lanes have channels
    const int c0 = act ? cv * VEC : 0;
    const int rows_i = static_cast<int>(a.rows);  // host-checked <= 2^31 - 1

    float2 wt[W][NV], bb[NV];
    if (a.taps_vec) {  // through this warp's ring slice (not in use yet)
        load_taps_staged<NV, W>(a.w, a.w_bf16, a.b, a.b_kind, slab * 32 * VEC, a.C, c0, act, lane,
                                dyn_smem + warp * RING_WARP, wt, bb);
    } else {
        load_taps_w<NV, W>(a.w, a.w_bf16, a.b, a.b_kind, c0, act, wt, bb);
    }

    float2 g[W][NV], gb[NV];  // sum dz*h[j+k], sum dz
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) g[k][v] = f2_zero();
        gb[v] = f2_zero();
    }

    // This warp's run: a fixed share of the batch's cost (its rows plus a
    // fixed cost per sequence; the same for every slab), so the operand
    // order of every partial sum is fixed.
    RunWalker<kBwdChunk> walk;
    walk.init(a.cu, a.N, a.rows, run, a.runs, H, true, lane, kBwdWalkRows, staged ? meta.cu : nullptr);

    // Everything above reads only the offsets, slots, flags, taps and bias.
    // Launched as a programmatic dependent (CCC_OPT_OVERLAP_PROLOGUE) it may
    // have run while the previous kernel finished; wait for that kernel
    // before reading x, dy, the saved history or the final-state gradient,
    // or writing anything.  (A no-op for an ordinary launch.)
    grid_dependency_wait();

    // The rings of history values and dz, carried from one segment to the
    // next along a walk (slot = walk row % RS).
    constexpr int RS = U;
    static_assert(RS >= W, "the ring must hold the current row and the W-1 before it");
    float2 hring[RS][NV], dring[RS][NV];
    bool live = true, read_state = false;

    // Ring state (P > 0): batch b of the current walk holds rows
    // [walk start + b*U, ... + U) of x and dy, in stage b % P.
    const uint32_t ring = smem_addr(dyn_smem + warp * RING_WARP) + lane * VB;
    const unsigned char *ring_p = dyn_smem + warp * RING_WARP + lane * VB;
    int p_row = 0, p_end = 0, issued = 0, consumed = 0;
    int st_in = 0, st_out = 0;            // ring stage of the next issue / the next batch consumed
    const uint16_t *px = a.x, *pg = a.dy;  // this lane's bytes of row p_row
    auto issue = [&]() {
        if constexpr (kBwdPrefetch > 0) {
            // lanes 0..2U-1: the warp's slab of x / dy rows PF ahead into L2
            const int64_t pr = static_cast<int64_t>(p_row) + kBwdPrefetch + (lane >> 1);
            if (full && lane < 2 * U && pr < p_end) {
                const uint16_t *base_ptr = (lane & 1) ? a.dy + static_cast<int64_t>(pr) * a.dys
                                                      : a.x + static_cast<int64_t>(pr) * a.xs;
                prefetch_l2(base_ptr + slab * 32 * VEC, 32 * VEC * 2);
            }
        }
        const uint32_t stage = ring + static_cast<uint32_t>(st_in * U * 2 * 32 * VB);
        // (row arithmetic as differences: p_end may be 2^31 - 1)
        if (act && p_end - p_row >= U) {  // the whole batch inside the walk: plain copies
            const uint16_t *qx = px, *qg = pg;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t off = static_cast<uint32_t>((u * 2) * 32 * VB);
                cp_async<VB>(stage + off, qx, true);
                cp_async<VB>(stage + off + 32 * VB, qg, true);
                qx += a.xs;
                qg += a.dys;
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = act && u < p_end - p_row;
                const uint32_t off = static_cast<uint32_t>((u * 2) * 32 * VB);
                cp_async<VB>(stage + off, ok ? px + static_cast<int64_t>(u) * a.xs : a.x, ok);
                cp_async<VB>(stage + off + 32 * VB, ok ? pg + static_cast<int64_t>(u) * a.dys : a.dy, ok);
            }
        }
        cp_async_commit();
        ++issued;
        st_in = st_in + 1 == (P > 0 ? P : 1) ? 0 : st_in + 1;
        p_row = p_end - p_row > U ? p_row + U : p_end;  // saturates: never past p_end
        px += static_cast<int64_t>(U) * a.xs;
        pg += static_cast<int64_t>(U) * a.dys;
    };

    Item t;
    bool cont, next_cont;
    while (walk.next(a.cu, a.rows, lane, t, cont, next_cont)) {
        if (!cont) {  // a new walk: the sequence's flags
            if (staged) {
                live = meta.cache[t.n] != -1;
                read_state = meta.flag[t.n] != 0;
            } else {
                live = !(a.cache && __ldg(a.cache + t.n) == -1);
                read_state = a.has_init != nullptr && __ldg(a.has_init + t.n) != 0;
            }
        }
        const int nr = t.nr;
        const int o0 = t.r0 - t.s, L = t.e - t.s;
        float *dinit = a.d_init ? a.d_init + static_cast<int64_t>(t.n) * H * a.C + c0 : nullptr;

        if (!live || L == 0) {  // zero gradient, no contribution
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < nr; ++r) st_stream<NV>(a.dx + static_cast<int64_t>(t.r0 + r) * a.dxs + c0, z);
                if (o0 == 0 && dinit)
#pragma unroll
                    for (int p = 0; p < H; ++p)
#pragma unroll
                        for (int v = 0; v < NV; ++v)
                            reinterpret_cast<float2 *>(dinit + p * a.C)[v] = f2_zero();
            }
            continue;
        }

        if constexpr (P > 0) {
            if (!cont) {
                // A new walk: the rows it will load are [t.r0, p_end) -- to the
                // end of the sequence, or H rows past the run where the
                // sequence goes on beyond it.
                cp_async_wait(0);
                p_row = t.r0;
                p_end = t.e - walk.R_hi > H ? walk.R_hi + H : t.e;  // min(R_hi + H, e) without overflow
                issued = consumed = 0;
                st_in = st_out = 0;
                px = a.x + static_cast<int64_t>(p_row) * a.xs + c0;
                pg = a.dy + static_cast<int64_t>(p_row) * a.dys + c0;
                while (issued < P - 1 && p_row < p_end) issue();
                if constexpr (kBwdNextWalkPrefetch) {
                    // Ask L2 for what the next sequence's walk will wait on
                    // first -- its first P-1 batches of x and dy and its saved
                    // history -- so that walk starts on L2 hits (lanes 0..2U-1:
                    // x rows, 2U..4U-1: dy rows, 4U..4U+H-1: history rows).
                    // (only after a short walk: L2 turns over in about 60 rows'
                    // time, so rows prefetched before a long walk would be gone)
                    const int n2 = t.n + 1, s2 = t.e;
                    if (full && n2 < a.N && s2 < walk.R_hi && p_end - t.r0 <= kBwdPrefetchWalkMax) {
                        const int j = lane & (2 * U - 1);
                        if (lane < 4 * U && j < rows_i - s2) {
                            const uint16_t *src = lane < 2 * U ? a.x + static_cast<int64_t>(s2 + j) * a.xs
                                                               : a.dy + static_cast<int64_t>(s2 + j) * a.dys;
                            prefetch_l2(src + slab * 32 * VEC, 32 * VEC * 2);
                        } else if (a.hist && lane >= 4 * U && lane < 4 * U + H) {
                            prefetch_l2(a.hist + (static_cast<int64_t>(n2) * H + (lane - 4 * U)) * a.C + slab * 32 * VEC,
                                        32 * VEC * 2);
                        }
                    }
                }
            }
        }
        if (!cont) {
            // History rows o0-H .. o0-1 (the initial history at a sequence's start).
            Raw<NV> hr[H];
#pragma unroll
            for (int p = 0; p < H; ++p) hr[p] = raw_zero<NV>();
            if (act) {
                if (o0 > 0) {
#pragma unroll
                    for (int p = 0; p < H; ++p) hr[p] = ld_ro<NV>(a.x + static_cast<int64_t>(t.r0 - H + p) * a.xs + c0);
                } else if (a.hist) {
#pragma unroll
                    for (int p = 0; p < H; ++p)
                        hr[p] = ld_ro<NV>(a.hist + (static_cast<int64_t>(t.n) * H + p) * a.C + c0);
                }
            }
            // history row p (oldest first) is walk row p - H: slot RS - H + p
#pragma unroll
            for (int p = 0; p < H; ++p) unpack<NV>(hr[p], hring[slot<RS>(0, H - p)]);
#pragma unroll
            for (int p = 0; p < RS; ++p)
#pragma unroll
                for (int v = 0; v < NV; ++v) dring[p][v] = f2_zero();
        }

        // i = o0 + k.  Rows k < nr are this segment's; when no segment of the
        // walk follows, H more steps finish dx of the last H rows (loading
        // x / dy past the segment while still inside the sequence).
        const int iters = nr + (next_cont ? 0 : H);
        const int nload = L - o0 < iters ? L - o0 : iters;  // steps with i < L
        for (int base = 0; base < iters; base += U) {
            // Steady state: every step of the batch loads a row, is one of
            // this segment's tokens and emits dx of the row H back (no carry:
            // all i < L).  Such batches run guard-free; the first batch of a
            // walk and the tail take the general path.
            const bool fast = full && (cont || base >= H) && base + U <= nload && base + U <= nr;
            Raw<NV> xr[U], gr[U];
            if constexpr (P == 0) {
                if (fast) {  // all lanes, all rows: unconditional loads, stepping row pointers
                    if constexpr (kBwdPrefetch > 0) {
                        // lanes 0..2U-1: the warp's slab of x / dy rows PF ahead into L2
                        const int64_t pr = static_cast<int64_t>(t.r0) + base + kBwdPrefetch + (lane >> 1);
                        if (lane < 2 * U && pr < t.e) {
                            const uint16_t *pp = (lane & 1) ? a.dy + static_cast<int64_t>(pr) * a.dys
                                                            : a.x + static_cast<int64_t>(pr) * a.xs;
                            prefetch_l2(pp + slab * 32 * VEC, 32 * VEC * 2);
                        }
                    }
                    const uint16_t *xp = a.x + static_cast<int64_t>(t.r0 + base) * a.xs + c0;
                    const uint16_t *gp = a.dy + static_cast<int64_t>(t.r0 + base) * a.dys + c0;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        xr[u] = ld_ro<NV>(xp);
                        gr[u] = ld_ro<NV>(gp);
                        xp += a.xs;
                        gp += a.dys;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const bool ld = act && base + u < nload;
                        const int64_t row = static_cast<int64_t>(t.r0) + base + u;
                        xr[u] = ld ? ld_ro<NV>(a.x + static_cast<int64_t>(row) * a.xs + c0) : raw_zero<NV>();
                        gr[u] = ld ? ld_ro<NV>(a.dy + static_cast<int64_t>(row) * a.dys + c0) : raw_zero<NV>();
                    }
                }
            } else {
                if (base < nload) {  // the next batch of the walk (zero-filled past p_end)
                    if (issued - consumed == P - 1) {
                        cp_async_wait(P - 2);  // steady state: the oldest of P-1 batches in flight
                    } else {
                        cp_async_wait(issued - consumed - 1);
                    }
                    const unsigned char *src = ring_p + st_out * U * 2 * 32 * VB;
                    st_out = st_out + 1 == P ? 0 : st_out + 1;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        xr[u] = ld_shared<NV>(src + (u * 2) * 32 * VB);
                        gr[u] = ld_shared<NV>(src + (u * 2 + 1) * 32 * VB);
                    }
                    ++consumed;
                    if (p_row < p_end) issue();
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) xr[u] = gr[u] = raw_zero<NV>();
                }
            }

            if (fast) {
                uint16_t *dxp = a.dx + static_cast<int64_t>(t.r0 + base - H) * a.dxs + c0;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float2 hc[NV], gy[NV];
                    unpack<NV>(xr[u], hc);
                    unpack<NV>(gr[u], gy);
                    Raw<NV> o;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const float2 dz = ring_dz<W, ACT, RS, NV>(wt, bb[v], hring, hc[v], gy[v], u, v);
                        ring_partials<W, RS, NV>(g, gb, dz, hring, hc[v], u, v);
                        // no carry (same op as the general path)
                        o.u[v] = f2_to_bf2(ring_dh<W, RS, NV>(wt, f2_zero(), dz, dring, u, v));
                        hring[u][v] = hc[v];
                        dring[u][v] = dz;
                    }
                    st_stream<NV>(dxp, o);
                    dxp += a.dxs;
                }
                continue;
            }

#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = base + u;
                if (k >= iters) break;
                const int64_t i = static_cast<int64_t>(o0) + k;  // up to L + H - 1 (L may be 2^31 - 1)
                float2 hc[NV], dz[NV];
                unpack<NV>(xr[u], hc);
                if (k < nload) {
                    float2 gy[NV];
                    unpack<NV>(gr[u], gy);
#pragma unroll
                    for (int v = 0; v < NV; ++v) dz[v] = ring_dz<W, ACT, RS, NV>(wt, bb[v], hring, hc[v], gy[v], u, v);
                } else {
#pragma unroll
                    for (int v = 0; v < NV; ++v) dz[v] = f2_zero();
                }
                if (k < nr) {  // this segment's own token: weight / bias partials
#pragma unroll
                    for (int v = 0; v < NV; ++v) ring_partials<W, RS, NV>(g, gb, dz[v], hring, hc[v], u, v);
                }
                // dH[i] is complete now.  i < H: an initial-history gradient.
                // Otherwise it is dx of row i-H, ours unless this is the first
                // step of a walk that starts inside a sequence (then the
                // previous run finished that row).
                const bool emit_init = i < H && dinit != nullptr;
                const bool emit_dx = i >= H && (cont || k >= H);
                if (emit_dx || emit_init) {
                    const bool carry = i >= L && a.d_final != nullptr;
                    const float2 *cp = carry ? reinterpret_cast<const float2 *>(
                                                   a.d_final + (static_cast<int64_t>(t.n) * H + (i - L)) * a.C + c0)
                                             : nullptr;
                    float2 acc[NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        acc[v] = ring_dh<W, RS, NV>(wt, (carry && act) ? __ldg(cp + v) : f2_zero(), dz[v], dring, u, v);
                    if (act) {
                        if (emit_dx) {
                            Raw<NV> o;
#pragma unroll
                            for (int v = 0; v < NV; ++v) o.u[v] = f2_to_bf2(acc[v]);
                            st_stream<NV>(a.dx + (t.s + i - H) * a.dxs + c0, o);
                        } else {
                            float2 *dp = reinterpret_cast<float2 *>(dinit + i * a.C);
#pragma unroll
                            for (int v = 0; v < NV; ++v) dp[v] = read_state ? acc[v] : f2_zero();
                        }
                    }
                }
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    hring[u][v] = hc[v];
                    dring[u][v] = dz[v];
                }
            }
        }
    }

    // Let the reduce kernel get scheduled while this warp stores its sums.
    grid_dependents_launch();

    // partial[run][k][c0 .. c0+VEC) for k = 0..W-1 (taps) and 4 (bias).
    if (act) {
        float *pp = a.part + static_cast<int64_t>(run) * 5 * a.C + c0;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
#pragma unroll
            for (int k = 0; k < W; ++k) reinterpret_cast<float2 *>(pp + k * a.C)[v] = g[k][v];
            reinterpret_cast<float2 *>(pp + 4 * a.C)[v] = gb[v];
        }
    }
}

// Ordered reduction of the G partial rows part[g][k][c] (k = 0..W-1 taps, 4
// the bias) into dweight[c][k] and dbias[c].  A CTA owns one k and 128
// consecutive channels, 4 per lane (16-byte loads); its warp w (of
// m = min(8, G)) sums the contiguous block of rows [w*G/m, (w+1)*G/m) in row
// order (the first row, then each next one added) -- the rows are loaded
// kRedBatch at a time before they are added, so a warp waits for one round
// trip per batch, not per row, and a block of up to kRedBatch rows (every
// block while G <= 128) for one -- and warp 0 adds the m block sums in block
// order.  The order of every addition depends
// only on G and C, so the result is the same bit for bit on every run.  The
// partials are written by the backward grid, which may still be running when
// this grid becomes resident (programmatic dependent launch): they are read
// after griddepcontrol.wait, with L2-coherent loads.
constexpr int kRedChannels = 128;  // channels per CTA (4 per lane)
constexpr int kRedBatch = 16;      // rows loaded before they are added

__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__global__ void __launch_bounds__(256) reduce_kernel(const float *part, int G, int C, int W, float *dweight,
                                                     float *dbias) {
    grid_dependency_wait();  // the backward's partials
    grid_dependents_launch();  // (a dependent's prologue may overlap this kernel)
    __shared__ float4 blk[kWarpsPerCta][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cblocks = (C + kRedChannels - 1) / kRedChannels;
    const int k = static_cast<int>(blockIdx.x) / cblocks;
    const int c = (static_cast<int>(blockIdx.x) % cblocks) * kRedChannels + 4 * lane;  // C % 8 == 0: c..c+3 < C
    if ((k >= W && k < 4) || (k == 4 && !dbias)) return;  // whole CTA: no such output
    const int m = G < kWarpsPerCta ? G : kWarpsPerCta;
    if (warp < m && c < C) {
        const int g0 = static_cast<int>(static_cast<int64_t>(warp) * G / m);
        const int g1 = static_cast<int>(static_cast<int64_t>(warp + 1) * G / m);
        const int64_t step = static_cast<int64_t>(5) * C / 4;  // one partial row, in float4
        const float4 *p = reinterpret_cast<const float4 *>(part + static_cast<int64_t>(k) * C + c);
        float4 v[kRedBatch];
#pragma unroll
        for (int u = 0; u < kRedBatch; ++u)  // the first batch (g0 < g1: m <= G)
            v[u] = g0 + u < g1 ? __ldcg(p + (g0 + u) * step) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 s = v[0];
#pragma unroll
        for (int u = 1; u < kRedBatch; ++u)
            if (g0 + u < g1) s = f4_add(s, v[u]);
        for (int g = g0 + kRedBatch; g < g1; g += kRedBatch) {
#pragma unroll
            for (int u = 0; u < kRedBatch; ++u)
                v[u] = g + u < g1 ? __ldcg(p + (g + u) * step) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < kRedBatch; ++u)
                if (g + u < g1) s = f4_add(s, v[u]);
        }
        blk[warp][lane] = s;
    }
    __syncthreads();
    if (warp == 0 && c < C) {
        float4 s = blk[0][lane];
        for (int w = 1; w < m; ++w) s = f4_add(s, blk[w][lane]);
        if (k < 4) {
            dweight[W * c + k] = s.x;
            dweight[W * (c + 1) + k] = s.y;
            dweight[W * (c + 2) + k] = s.z;
            dweight[W * (c + 3) + k] = s.w;
        } else {  // (dbias is only 4-byte aligned)
            dbias[c] = s.x;
            dbias[c + 1] = s.y;
            dbias[c + 2] = s.z;
            dbias[c + 3] = s.w;
        }
    }
}

using BwdKernel = void (*)(const BwdArgs);

template <int W, bool ACT>
constexpr BwdKernel bwd_kernel_of(bool one_warp) {
    return one_warp ? bwd_kernel<kBwdVec, kBwdUnroll, kBwdRing, W, ACT, 1>
                    : bwd_kernel<kBwdVec, kBwdUnroll, kBwdRing, W, ACT, kWarpsPerCta>;
}

// The instantiation for (width, activation, CTA size); nullptr for an
// unsupported pair.
BwdKernel bwd_kernel_for(int width, int act, bool one_warp) {
    switch (width * 2 + (act ? 1 : 0)) {
        case 4: return bwd_kernel_of<2, false>(one_warp);
        case 5: return bwd_kernel_of<2, true>(one_warp);
        case 6: return bwd_kernel_of<3, false>(one_warp);
        case 7: return bwd_kernel_of<3, true>(one_warp);
        case 8: return bwd_kernel_of<4, false>(one_warp);
        case 9: return bwd_kernel_of<4, true>(one_warp);
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t st, bool overlap, int sms) {
    // Where spreading the tasks evenly would leave every SM fewer than 8 of
    // them, one-warp CTAs, which the block scheduler spreads over all SMs
    // (a tiny batch's 65 tasks on 65 SMs, not on 9 SMs in 8-warp CTAs).
    // Which warp runs a task changes nothing it computes.
    const int64_t tasks = static_cast<int64_t>(a.slabs) * a.runs;
    const bool one_warp = tasks <= static_cast<int64_t>(sms) * (kWarpsPerCta - 1);
    const int cw = one_warp ? 1 : kWarpsPerCta;
    const BwdKernel kern = bwd_kernel_for(a.width, a.act, one_warp);
    if (!kern) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(tasks, cw)));
    cfg.blockDim = dim3(static_cast<unsigned>(32 * cw));
    cfg.stream = st;
    constexpr int P = kBwdRing;
    const size_t ring_bytes = static_cast<size_t>(P) * kBwdUnroll * 2 * 32 * kBwdVec * 2 * cw;
    if (ring_bytes > 48 * 1024) {
        // Opt in to more than 48 KB of dynamic shared memory.  Set on every
        // launch (a host-side attribute, no device work): no flag shared
        // between host threads, and nothing stale after a device reset or in
        // another context.
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ring_bytes));
        if (e != cudaSuccess) return e;
    }
    cfg.dynamicSmemBytes = ring_bytes;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// The reduce is a programmatic dependent launch: it may become resident
// while the backward grid drains (the backward triggers it after its walks)
// and waits for the partials with griddepcontrol.wait.
cudaError_t launch_reduce(const float *part, int G, int C, int width, float *dweight, float *dbias,
                          cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(5 * ceil_div(C, kRedChannels)));  // (k, 128-channel block)
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reduce_kernel, part, G, C, width, dweight, dbias);
}

}  // namespace ccc
