// ccc_bwd.cu -- fused backward: dx, d_init_state and per-CTA FP32
// dweight/dbias partials in one pass, then an ordered reduction.
//
// FlashInfer "cake_causal_conv1d_train.cake_causal_conv1d_kcp" (Returns): one
// kernel produces the input gradient and deterministic FP32 weight-gradient
// partials; Megatron-Core "core.ssm.causal_conv1d"
// (assert_causal_conv1d_deterministic): partials go to a per-block workspace
// and are combined by an ordered reduction instead of atomics, so the result
// does not depend on scheduling.
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
// owns VEC channels, and each warp walks a contiguous run of work items.
// Along consecutive items of one sequence the lane walks i = o0, o0+1, ...
// without a break: it keeps a sliding window of 3 history rows and the 3
// previous dz values in registers, emits dx for row i-3 once dz_i is known,
// and accumulates dz_j * h[j+k] and dz_j of its own rows into 5*VEC FP32
// registers.  Only where a walk starts inside a sequence does it re-read the
// 3 rows before it, and only where it stops before the sequence end does it
// read 3 rows past it (both from L2: the neighbouring warp's run).
//
// Determinism.  The number of runs per slab R is fixed by (rows, N, C) only;
// the warp with task (slab, run r) walks items [r*total/R, (r+1)*total/R) in
// order and writes partial[r][k][c] for its channels, so every partial sum
// has a fixed operand order; the reduce kernel then sums the R partials of
// every (k, c) in order r = 0..R-1.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

// P = 0: each lane loads its U rows of x and dy straight into registers.
// P > 0: each lane streams the rows of its walk through a P-stage ring of
// U-row batches in shared memory (cp.async), keeping up to P-1 batches in
// flight ahead of the math.
template <int VEC, int U, int P>
__global__ void __launch_bounds__(kCtaThreads, kBwdMinBlocks) bwd_kernel(const BwdArgs a) {
    constexpr int NV = VEC / 2;
    constexpr int VB = VEC * 2;                         // bytes per lane per row
    constexpr int RING_WARP = P * U * 2 * 32 * VB;      // ring bytes per warp
    static_assert(P == 0 || kBwdChunk % U == 0, "items must be whole batches");
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kWarpsPerCta + warp;  // this warp's task
    if (gw >= a.slabs * a.runs) return;               // (whole warp) no task in the last CTA
    const int slab = gw % a.slabs, run = gw / a.slabs;
    const int cv = slab * 32 + lane;
    const bool act = cv < a.C / VEC;
    const bool full = (slab + 1) * 32 * VEC <= a.C;  // warp-uniform: all lanes have channels
    const int c0 = act ? cv * VEC : 0;

    float2 w0[NV], w1[NV], w2[NV], w3[NV], bb[NV];
    load_taps<NV>(a.w, a.w_bf16, a.b, a.b_kind, c0, act, w0, w1, w2, w3, bb);

    float2 g0[NV], g1[NV], g2[NV], g3[NV], gb[NV];  // sum dz*h[j+k], sum dz
#pragma unroll
    for (int v = 0; v < NV; ++v) g0[v] = g1[v] = g2[v] = g3[v] = gb[v] = f2_zero();

    grid_dependency_wait();  // the chunk map, when one was built

    ItemDecoder<kBwdChunk> dec;
    dec.init(a.map, a.cap, a.cu, a.N, a.rows, true, lane);

    // This warp's run: a contiguous, fixed range of items (same for every
    // slab), so the operand order of every partial sum is fixed.
    const int lo = static_cast<int>(static_cast<int64_t>(run) * dec.total / a.runs);
    const int hi = static_cast<int>(static_cast<int64_t>(run + 1) * dec.total / a.runs);

    // The run's last item (sequence, row after it): where its final walk
    // stops reading ahead.
    int last_n = -1, last_end = 0;
    if (lo < hi) {
        const Item l = dec.get(hi - 1, a.map, a.cu, a.rows);
        last_n = l.n;
        last_end = l.r0 + l.nr;
    }

    // Sliding windows, carried from one item to the next when the next item
    // continues the same sequence: history rows h[i..i+2] and dz_{i-1..i-3}.
    float2 h0[NV], h1[NV], h2[NV], d1[NV], d2[NV], d3[NV];
    Item cur = {};
    bool live = true, read_state = false;

    // Ring state (P > 0): batch b of the current walk holds rows
    // [walk start + b*U, ... + U) of x and dy, in stage b % P.
    const uint32_t ring = smem_addr(dyn_smem + warp * RING_WARP) + lane * VB;
    const unsigned char *ring_p = dyn_smem + warp * RING_WARP + lane * VB;
    int p_row = 0, p_end = 0, issued = 0, consumed = 0;
    auto issue = [&]() {
        if constexpr (kBwdPrefetch > 0) {
            // lanes 0..2U-1: the warp's slab of x / dy rows PF ahead into L2
            const int pr = p_row + kBwdPrefetch + (lane >> 1);
            if (full && lane < 2 * U && pr < p_end) {
                const uint16_t *base_ptr = (lane & 1) ? a.dy + static_cast<int64_t>(pr) * a.dys
                                                      : a.x + static_cast<int64_t>(pr) * a.xs;
                prefetch_l2(base_ptr + slab * 32 * VEC, 32 * VEC * 2);
            }
        }
        const int st = issued % (P > 0 ? P : 1);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int row = p_row + u;
            const bool ok = act && row < p_end;
            const uint32_t off = static_cast<uint32_t>(((st * U + u) * 2) * 32 * VB);
            cp_async<VB>(ring + off, ok ? a.x + static_cast<int64_t>(row) * a.xs + c0 : a.x, ok);
            cp_async<VB>(ring + off + 32 * VB, ok ? a.dy + static_cast<int64_t>(row) * a.dys + c0 : a.dy, ok);
        }
        cp_async_commit();
        ++issued;
        p_row += U;
    };

    for (int it = lo; it < hi; ++it) {
        // The next item of the same sequence is the next B rows: only a new
        // sequence needs the chunk map / offsets (and its flags) again.
        const bool cont = it > lo && cur.r0 + cur.nr < cur.e;
        if (cont) {
            cur.r0 += cur.nr;
            cur.nr = min(kBwdChunk, cur.e - cur.r0);
        } else {
            cur = dec.get(it, a.map, a.cu, a.rows);
            live = !(a.cache && __ldg(a.cache + cur.n) == -1);
            read_state = a.has_init != nullptr && __ldg(a.has_init + cur.n) != 0;
        }
        const Item t = cur;
        const bool next_cont = it + 1 < hi && t.r0 + t.nr < t.e;
        const int nr = t.nr;
        const int o0 = t.r0 - t.s, L = t.e - t.s;
        float *dinit = a.d_init ? a.d_init + static_cast<int64_t>(t.n) * 3 * a.C + c0 : nullptr;

        if (!live || L == 0) {  // zero gradient, no contribution
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < nr; ++r) st_stream<NV>(a.dx + static_cast<int64_t>(t.r0 + r) * a.dxs + c0, z);
                if (o0 == 0 && dinit)
#pragma unroll
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int v = 0; v < NV; ++v)
                            reinterpret_cast<float2 *>(dinit + p * a.C)[v] = f2_zero();
            }
            continue;
        }

        if constexpr (P > 0) {
            if (!cont) {
                // A new walk: the rows it will load are [t.r0, p_end) -- to the
                // end of the sequence, or for the run's last sequence to 3 rows
                // past the run (within the sequence).
                cp_async_wait(0);
                p_row = t.r0;
                p_end = t.n == last_n ? min(last_end + 3, t.e) : t.e;
                issued = consumed = 0;
                while (issued < P - 1 && p_row < p_end) issue();
            }
        }
        if (!cont) {
            // History rows o0-3 .. o0-1 (the initial history for a first item).
            Raw<NV> hr[3];
#pragma unroll
            for (int p = 0; p < 3; ++p) hr[p] = raw_zero<NV>();
            if (act) {
                if (o0 > 0) {
#pragma unroll
                    for (int p = 0; p < 3; ++p) hr[p] = ld_ro<NV>(a.x + static_cast<int64_t>(t.r0 - 3 + p) * a.xs + c0);
                } else if (a.hist) {
#pragma unroll
                    for (int p = 0; p < 3; ++p)
                        hr[p] = ld_ro<NV>(a.hist + (static_cast<int64_t>(t.n) * 3 + p) * a.C + c0);
                }
            }
            unpack<NV>(hr[0], h0);
            unpack<NV>(hr[1], h1);
            unpack<NV>(hr[2], h2);
#pragma unroll
            for (int v = 0; v < NV; ++v) d1[v] = d2[v] = d3[v] = f2_zero();
        }

        // i = o0 + k.  Rows k < nr are this item's; when the next item does
        // not continue the walk, 3 more steps finish dx of the last 3 rows
        // (loading x / dy past the item while still inside the sequence).
        const int iters = nr + (next_cont ? 0 : 3);
        const int nload = L - o0 < iters ? L - o0 : iters;  // steps with i < L
        for (int base = 0; base < iters; base += U) {
            // Steady state: every step of the batch loads a row, is one of
            // this item's tokens and emits dx of the row 3 back (no carry:
            // all i < L).  Such batches run guard-free; the first batch of a
            // walk and the tail take the general path.
            const bool fast = full && (cont || base >= 3) && base + U <= nload && base + U <= nr;
            Raw<NV> xr[U], gr[U];
            if constexpr (P == 0) {
                if (fast) {  // all lanes, all rows: unconditional loads, stepping row pointers
                    if constexpr (kBwdPrefetch > 0) {
                        // lanes 0..2U-1: the warp's slab of x / dy rows PF ahead into L2
                        const int pr = t.r0 + base + kBwdPrefetch + (lane >> 1);
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
                        const int row = t.r0 + base + u;
                        xr[u] = ld ? ld_ro<NV>(a.x + static_cast<int64_t>(row) * a.xs + c0) : raw_zero<NV>();
                        gr[u] = ld ? ld_ro<NV>(a.dy + static_cast<int64_t>(row) * a.dys + c0) : raw_zero<NV>();
                    }
                }
            } else {
                if (base < nload) {  // the next batch of the walk (zero-filled past p_end)
                    cp_async_wait(issued - consumed - 1);
                    const unsigned char *src = ring_p + (consumed % P) * U * 2 * 32 * VB;
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
                uint16_t *dxp = a.dx + static_cast<int64_t>(t.r0 + base - 3) * a.dxs + c0;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float2 hc[NV], gy[NV], dz[NV];
                    unpack<NV>(xr[u], hc);
                    unpack<NV>(gr[u], gy);
                    Raw<NV> o;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        dz[v] = silu_grad(bb[v], w0[v], w1[v], w2[v], w3[v], h0[v], h1[v], h2[v], hc[v], gy[v]);
                        g0[v] = __ffma2_rn(dz[v], h0[v], g0[v]);
                        g1[v] = __ffma2_rn(dz[v], h1[v], g1[v]);
                        g2[v] = __ffma2_rn(dz[v], h2[v], g2[v]);
                        g3[v] = __ffma2_rn(dz[v], hc[v], g3[v]);
                        gb[v] = __fadd2_rn(gb[v], dz[v]);
                        float2 c = __ffma2_rn(w0[v], dz[v], f2_zero());  // no carry (same op as the general path)
                        c = __ffma2_rn(w1[v], d1[v], c);
                        c = __ffma2_rn(w2[v], d2[v], c);
                        c = __ffma2_rn(w3[v], d3[v], c);
                        o.u[v] = f2_to_bf2(c);
                        d3[v] = d2[v];
                        d2[v] = d1[v];
                        d1[v] = dz[v];
                        h0[v] = h1[v];
                        h1[v] = h2[v];
                        h2[v] = hc[v];
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
                const int i = o0 + k;
                float2 hc[NV], dz[NV];
                unpack<NV>(xr[u], hc);
                if (k < nload) {
                    float2 gy[NV];
                    unpack<NV>(gr[u], gy);
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        dz[v] = silu_grad(bb[v], w0[v], w1[v], w2[v], w3[v], h0[v], h1[v], h2[v], hc[v], gy[v]);
                } else {
#pragma unroll
                    for (int v = 0; v < NV; ++v) dz[v] = f2_zero();
                }
                if (k < nr) {  // this item's own token: weight / bias partials
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        g0[v] = __ffma2_rn(dz[v], h0[v], g0[v]);
                        g1[v] = __ffma2_rn(dz[v], h1[v], g1[v]);
                        g2[v] = __ffma2_rn(dz[v], h2[v], g2[v]);
                        g3[v] = __ffma2_rn(dz[v], hc[v], g3[v]);
                        gb[v] = __fadd2_rn(gb[v], dz[v]);
                    }
                }
                // dH[i] is complete now.  i < 3: an initial-history gradient.
                // Otherwise it is dx of row i-3, ours unless this is the first
                // step of a walk that starts inside a sequence (then the
                // previous item's owner finished that row).
                const bool emit_init = i < 3 && dinit != nullptr;
                const bool emit_dx = i >= 3 && (cont || k >= 3);
                if (emit_dx || emit_init) {
                    const bool carry = i >= L && a.d_final != nullptr;
                    const float2 *cp = carry ? reinterpret_cast<const float2 *>(
                                                   a.d_final + (static_cast<int64_t>(t.n) * 3 + (i - L)) * a.C + c0)
                                             : nullptr;
                    float2 acc[NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float2 c = (carry && act) ? __ldg(cp + v) : f2_zero();
                        c = __ffma2_rn(w0[v], dz[v], c);
                        c = __ffma2_rn(w1[v], d1[v], c);
                        c = __ffma2_rn(w2[v], d2[v], c);
                        c = __ffma2_rn(w3[v], d3[v], c);
                        acc[v] = c;
                    }
                    if (act) {
                        if (emit_dx) {
                            Raw<NV> o;
#pragma unroll
                            for (int v = 0; v < NV; ++v) o.u[v] = f2_to_bf2(acc[v]);
                            st_stream<NV>(a.dx + static_cast<int64_t>(t.s + i - 3) * a.dxs + c0, o);
                        } else {
                            float2 *dp = reinterpret_cast<float2 *>(dinit + static_cast<int64_t>(i) * a.C);
#pragma unroll
                            for (int v = 0; v < NV; ++v) dp[v] = read_state ? acc[v] : f2_zero();
                        }
                    }
                }
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    d3[v] = d2[v];
                    d2[v] = d1[v];
                    d1[v] = dz[v];
                    h0[v] = h1[v];
                    h1[v] = h2[v];
                    h2[v] = hc[v];
                }
            }
        }
    }

    // Let the reduce kernel get scheduled while this warp stores its sums.
    grid_dependents_launch();

    // partial[run][k][c0 .. c0+VEC) for k = 0..3 (taps) and 4 (bias).
    if (act) {
        float *pp = a.part + static_cast<int64_t>(run) * 5 * a.C + c0;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            reinterpret_cast<float2 *>(pp + 0 * a.C)[v] = g0[v];
            reinterpret_cast<float2 *>(pp + 1 * a.C)[v] = g1[v];
            reinterpret_cast<float2 *>(pp + 2 * a.C)[v] = g2[v];
            reinterpret_cast<float2 *>(pp + 3 * a.C)[v] = g3[v];
            reinterpret_cast<float2 *>(pp + 4 * a.C)[v] = gb[v];
        }
    }
}

// dweight[c][k] = sum_{r=0..runs-1} part[r][k][c] (k < 4), dbias[c] likewise
// with k = 4: one thread per output, fixed order.
// The partials are written by the backward grid, which may still be running
// when this grid becomes resident (programmatic dependent launch): they are
// read with L2-coherent loads, not through the read-only path.
__global__ void __launch_bounds__(256) reduce_kernel(const float *part, int G, int C, float *dweight,
                                                     float *dbias) {
    grid_dependency_wait();  // the backward's partials
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 5 * C) return;
    const int k = idx / C, c = idx % C;
    const float *p = part + static_cast<int64_t>(k) * C + c;
    float s = __ldcg(p);
    for (int g = 1; g < G; ++g) s += __ldcg(p + static_cast<int64_t>(g) * 5 * C);
    if (k < 4) {
        dweight[4 * c + k] = s;
    } else if (dbias) {
        dbias[c] = s;
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(static_cast<int64_t>(a.slabs) * a.runs, kWarpsPerCta)));
    cfg.blockDim = dim3(kCtaThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    constexpr int P = kBwdRing;
    constexpr size_t ring_bytes = static_cast<size_t>(P) * kBwdUnroll * 2 * 32 * kBwdVec * 2 * kWarpsPerCta;
    auto kern = bwd_kernel<kBwdVec, kBwdUnroll, P>;
    if (ring_bytes > 48 * 1024) {
        // Opt in to more than 48 KB of dynamic shared memory, once per device.
        static bool attr_set[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ring_bytes));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    cfg.dynamicSmemBytes = ring_bytes;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_reduce(const float *part, int G, int C, float *dweight, float *dbias, bool pdl,
                          cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(5 * static_cast<int64_t>(C), 256)));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, reduce_kernel, part, G, C, dweight, dbias);
}

}  // namespace ccc
