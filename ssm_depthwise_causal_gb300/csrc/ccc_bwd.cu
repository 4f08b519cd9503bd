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
// Mapping.  As in the forward: a warp owns (item, 32*VEC-channel slab), a
// lane owns VEC channels.  For an item of nr rows starting at sequence offset
// o0 the lane walks i = o0 .. o0+nr+2: it needs x rows o0-3 .. o0+nr+2 and dy
// rows o0 .. o0+nr+2 (a 3-row halo on each side, served by L2), keeps a
// sliding window of 3 history rows and 3 past dz values in registers, emits
// dx for row i-3 once dz_i is known, and accumulates dz_j * h[j+k] and dz_j
// of its own rows into 5*VEC FP32 registers.
//
// Determinism.  The grid is (slabs, G) with G fixed by (rows, N, C) only;
// warp w of CTA (x, y) takes items y*8+w, y*8+w+8G, ... in order, so every
// partial sum has a fixed operand order.  At the end each CTA folds its 8
// warps in shared memory in warp order and writes partial[y][k][c]; the
// reduce kernel then sums the G partials of every (k, c) in order y = 0..G-1.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

template <int VEC, int U>
__global__ void __launch_bounds__(kCtaThreads, 2) bwd_kernel(const BwdArgs a) {
    constexpr int NV = VEC / 2;
    constexpr int SLAB = 32 * VEC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cv = blockIdx.x * 32 + lane;
    const bool act = cv < a.C / VEC;
    const int c0 = act ? cv * VEC : 0;

    float2 w0[NV], w1[NV], w2[NV], w3[NV], bb[NV];
    load_taps<NV>(a.w, a.w_bf16, a.b, a.b_kind, c0, act, w0, w1, w2, w3, bb);

    float2 g0[NV], g1[NV], g2[NV], g3[NV], gb[NV];  // sum dz*h[j+k], sum dz
#pragma unroll
    for (int v = 0; v < NV; ++v) g0[v] = g1[v] = g2[v] = g3[v] = gb[v] = f2_zero();

    grid_dependency_wait();  // the chunk map, when one was built

    ItemDecoder dec;
    dec.init(a.map, a.cap, a.cu, a.N, a.rows, kBwdChunk, true, lane);
    const int step = gridDim.y * kWarpsPerCta;

    for (int it = blockIdx.y * kWarpsPerCta + warp; it < dec.total; it += step) {
        const Item t = dec.get(it);
        const int nr = t.nr;
        const int64_t o0 = t.r0 - t.s, L = t.e - t.s;
        const bool live = !(a.cache && __ldg(a.cache + t.n) == -1);
        float *dinit = a.d_init ? a.d_init + static_cast<int64_t>(t.n) * 3 * a.C + c0 : nullptr;

        if (!live || L == 0) {  // zero gradient, no contribution
            if (act) {
                const Raw<NV> z = raw_zero<NV>();
                for (int r = 0; r < nr; ++r) st_stream<NV>(a.dx + (t.r0 + r) * a.dxs + c0, z);
                if (o0 == 0 && dinit)
#pragma unroll
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int v = 0; v < NV; ++v)
                            reinterpret_cast<float2 *>(dinit + p * a.C)[v] = f2_zero();
            }
            continue;
        }
        const bool read_state = a.has_init != nullptr && __ldg(a.has_init + t.n) != 0;

        // History rows o0-3 .. o0-1 (initial history for the first item).
        float2 h0[NV], h1[NV], h2[NV];
        {
            Raw<NV> hr[3];
#pragma unroll
            for (int p = 0; p < 3; ++p) hr[p] = raw_zero<NV>();
            if (act) {
                if (o0 > 0) {
#pragma unroll
                    for (int p = 0; p < 3; ++p) hr[p] = ld_ro<NV>(a.x + (t.r0 - 3 + p) * a.xs + c0);
                } else if (a.hist) {
#pragma unroll
                    for (int p = 0; p < 3; ++p)
                        hr[p] = ld_ro<NV>(a.hist + (static_cast<int64_t>(t.n) * 3 + p) * a.C + c0);
                }
            }
            unpack<NV>(hr[0], h0);
            unpack<NV>(hr[1], h1);
            unpack<NV>(hr[2], h2);
        }
        float2 d1[NV], d2[NV], d3[NV];  // dz_{i-1}, dz_{i-2}, dz_{i-3}
#pragma unroll
        for (int v = 0; v < NV; ++v) d1[v] = d2[v] = d3[v] = f2_zero();

        const int iters = nr + 3;                                       // i = o0 .. o0+nr+2
        const int nload = static_cast<int>(L - o0 < iters ? L - o0 : iters);  // rows with i < L
        for (int base = 0; base < iters; base += U) {
            Raw<NV> xr[U], gr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ld = act && base + u < nload;
                xr[u] = ld ? ld_ro<NV>(a.x + (t.r0 + base + u) * a.xs + c0) : raw_zero<NV>();
                gr[u] = ld ? ld_ro<NV>(a.dy + (t.r0 + base + u) * a.dys + c0) : raw_zero<NV>();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = base + u;
                if (k >= iters) break;
                const int64_t i = o0 + k;
                float2 hc[NV], dz[NV];
                unpack<NV>(xr[u], hc);
                if (k < nload) {
                    float2 gy[NV];
                    unpack<NV>(gr[u], gy);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float2 z = bb[v];
                        z = __ffma2_rn(w0[v], h0[v], z);
                        z = __ffma2_rn(w1[v], h1[v], z);
                        z = __ffma2_rn(w2[v], h2[v], z);
                        z = __ffma2_rn(w3[v], hc[v], z);
                        const float2 s = sigmoid2(z);
                        const float2 oms = __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(-s.x, -s.y));
                        const float2 f = __ffma2_rn(z, oms, make_float2(1.0f, 1.0f));
                        dz[v] = __fmul2_rn(gy[v], __fmul2_rn(s, f));
                    }
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
                const bool emit_dx = k >= 3;
                const bool emit_init = o0 == 0 && k < 3 && dinit != nullptr;
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
                            st_stream<NV>(a.dx + (t.r0 + k - 3) * a.dxs + c0, o);
                        } else {
                            float2 *dp = reinterpret_cast<float2 *>(dinit + i * a.C);
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

    // Let the reduce kernel get scheduled while this CTA folds its warps.
    grid_dependents_launch();

    // Fold the 8 warps' partials in warp order, write partial[y][k][c].
    __shared__ float red[kWarpsPerCta][5][SLAB];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int cl = lane * VEC + 2 * v;
        red[warp][0][cl] = g0[v].x; red[warp][0][cl + 1] = g0[v].y;
        red[warp][1][cl] = g1[v].x; red[warp][1][cl + 1] = g1[v].y;
        red[warp][2][cl] = g2[v].x; red[warp][2][cl + 1] = g2[v].y;
        red[warp][3][cl] = g3[v].x; red[warp][3][cl + 1] = g3[v].y;
        red[warp][4][cl] = gb[v].x; red[warp][4][cl + 1] = gb[v].y;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 5 * SLAB; idx += kCtaThreads) {
        const int k = idx / SLAB, cl = idx % SLAB;
        float s = red[0][k][cl];
#pragma unroll
        for (int w = 1; w < kWarpsPerCta; ++w) s += red[w][k][cl];
        const int c = blockIdx.x * SLAB + cl;
        if (c < a.C) a.part[(static_cast<int64_t>(blockIdx.y) * 5 + k) * a.C + c] = s;
    }
}

// dweight[c][k] = sum_{g=0..G-1} part[g][k][c] (k < 4), dbias[c] likewise
// with k = 4: one thread per output, fixed order.
__global__ void __launch_bounds__(256) reduce_kernel(const float *__restrict__ part, int G, int C,
                                                     float *__restrict__ dweight, float *__restrict__ dbias) {
    grid_dependency_wait();  // the backward's partials
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 5 * C) return;
    const int k = idx / C, c = idx % C;
    const float *p = part + static_cast<int64_t>(k) * C + c;
    float s = p[0];
    for (int g = 1; g < G; ++g) s += p[static_cast<int64_t>(g) * 5 * C];
    if (k < 4) {
        dweight[4 * c + k] = s;
    } else if (dbias) {
        dbias[c] = s;
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, int grid_y, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(a.C, 32 * kBwdVec)), static_cast<unsigned>(grid_y));
    cfg.blockDim = dim3(kCtaThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, bwd_kernel<kBwdVec, 4>, a);
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
