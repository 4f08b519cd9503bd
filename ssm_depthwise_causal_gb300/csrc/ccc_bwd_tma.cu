// ccc_bwd_tma.cu -- the fused backward with a bulk-copy producer warp.
//
// Same method and the same result bits as ccc_bwd.cu (FlashInfer
// "cake_causal_conv1d_train.cake_causal_conv1d_kcp", Returns: fused dx +
// deterministic FP32 dweight; Megatron-Core "core.ssm.causal_conv1d",
// assert_causal_conv1d_deterministic: ordered per-block partials), with a
// different way of feeding the math.
//
// A CTA owns one task: a column of NC*128 channels and a run of consecutive
// work items, i.e. the contiguous packed row range [S0, S1) those items cover
// (plus the 3 history rows before it when the run starts inside a sequence,
// and the up-to-3 rows after it that finish the last rows' dx).  Warp NC is
// the producer: it streams that row range of x and dy into a P-stage ring of
// R-row stages in shared memory with one bulk copy per row and tensor
// (cp.async.bulk, completion counted in bytes on the stage's "full"
// mbarrier).  Warps 0..NC-1 are consumers: each walks the items of the run on
// its 128-channel slab exactly like the register-fed kernel, reading its 8
// bytes of each row from shared memory, and releases a stage (its "empty"
// mbarrier) once its walk has moved past it.  The consumers therefore hold no
// global loads in flight and do no global address arithmetic for x and dy;
// the memory-level parallelism comes from the P-1 stages the producer keeps
// in flight.
//
// Determinism: the number of runs per column is a constant of (rows, N, C);
// consumer warp w of task (column, run r) writes partial[r][k][c] for its
// channels, and the reduce kernel sums the runs in order r = 0..R-1.  The
// per-element arithmetic (operation and operand order) is that of the
// register-fed kernel, so dx, d_init_state and the partial sums are bitwise
// the same for the same run split.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

constexpr int kVec = 4;     // channels per lane
constexpr int kNV = 2;      // float2 pairs per lane
constexpr int kSlab = 128;  // channels per consumer warp

template <int NC, int R, int P>
struct Ring {
    static constexpr int kColW = NC * kSlab;                  // channels per column
    static constexpr int kRowBytes = kColW * 2;               // one tensor row of a column
    static constexpr int kStageBytes = R * 2 * kRowBytes;     // x and dy rows of one stage
    static constexpr int kBarOffset = P * kStageBytes;        // barriers after the stages
    static constexpr int kSmemBytes = kBarOffset + 2 * P * 8;
};

// Consumer-side view of the ring for one warp's walk.
template <int NC, int R, int P>
struct StageReader {
    using RG = Ring<NC, R, P>;
    uint32_t lane_base;  // smem address of stage 0, row 0, x, this lane's 8 bytes
    uint32_t bars;       // smem address of full[0]; empty[s] = bars + 8 * (P + s)
    int S0;              // first row of the stream
    int k_full;          // stages 0 .. k_full-1 are known to be full
    int k_rel;           // stages 0 .. k_rel-1 have been released
    bool ok;             // false after a wait timed out

    // Make sure the stage holding row r has landed.
    __device__ __forceinline__ void need(int r) {
        const int k = (r - S0) / R;
        while (ok && k_full <= k) {
            ok = mbar_wait(bars + 8 * (k_full % P), (k_full / P) & 1);
            ++k_full;
        }
    }

    // The walk will not read rows before r again: release the stages
    // entirely before it -- but only stages this warp has waited on, so each
    // warp arrives on a stage's "empty" barrier exactly once per fill, in
    // order (a warp that skipped rows of a -1 request releases those stages
    // after need() has walked past them).
    __device__ __forceinline__ void release_before(int r, int lane) {
        const int k = min((r - S0) / R, k_full);
        if (k_rel < k) {
            __syncwarp();
            for (; k_rel < k; ++k_rel)
                if (lane == 0) mbar_arrive(bars + 8 * (P + k_rel % P));
        }
    }

    // End of the walk: wait for and release every remaining stage of the
    // stream in order, so the producer can always finish.
    __device__ __forceinline__ void drain(int nst, int lane) {
        for (int k = k_rel; k < nst && ok; ++k) {
            while (ok && k_full <= k) {
                ok = mbar_wait(bars + 8 * (k_full % P), (k_full / P) & 1);
                ++k_full;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (P + k % P));
        }
        k_rel = nst;
    }

    __device__ __forceinline__ Raw<kNV> row(int r, int tensor) const {
        const int j = r - S0;
        const uint32_t addr = lane_base + static_cast<uint32_t>(((j / R) % P) * RG::kStageBytes +
                                                                ((j % R) * 2 + tensor) * RG::kRowBytes);
        Raw<kNV> v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.u[0]), "=r"(v.u[1]) : "r"(addr));
        return v;
    }
};

template <int NC, int R, int P, int U>
__global__ void __launch_bounds__((NC + 1) * 32, kBwdTmaMinBlocks) bwd_tma_kernel(const BwdArgs a) {
    using RG = Ring<NC, R, P>;
    constexpr int NV = kNV;
    static_assert(2 * R <= 32, "one producer lane per row and tensor");
    extern __shared__ __align__(128) unsigned char smem[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cols = a.slabs;  // columns of NC*128 channels
    if (static_cast<int>(blockIdx.x) >= cols * a.runs) return;  // whole CTA
    const int col = blockIdx.x % cols, run = blockIdx.x / cols;
    const int col_c0 = col * RG::kColW;
    const int col_ch = min(RG::kColW, a.C - col_c0);      // channels present in this column
    const int nact = (col_ch + kSlab - 1) / kSlab;          // consumer warps with channels

    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + RG::kBarOffset;
    if (threadIdx.x == 0) {
        for (int s = 0; s < P; ++s) {
            mbar_init(bars + 8 * s, 1);             // full: the producer's expect_tx arrive
            mbar_init(bars + 8 * (P + s), nact);    // empty: one arrive per active consumer
        }
        mbar_init_fence();
    }
    __syncthreads();

    grid_dependency_wait();  // the chunk map, when one was built

    ItemDecoder<kBwdChunk> dec;
    dec.init(a.map, a.cap, a.cu, a.N, a.rows, true, lane);
    const int lo = static_cast<int>(static_cast<int64_t>(run) * dec.total / a.runs);
    const int hi = static_cast<int>(static_cast<int64_t>(run + 1) * dec.total / a.runs);

    // The run's row stream [S0, S1).
    int S0 = 0, S1 = 0;
    if (lo < hi) {
        const Item f = dec.get(lo, a.map, a.cu, a.rows);
        const Item l = dec.get(hi - 1, a.map, a.cu, a.rows);
        S0 = f.r0 > f.s ? f.r0 - 3 : f.r0;     // history rows of a walk that starts inside a sequence
        S1 = min(l.r0 + l.nr + 3, l.e);         // rows that finish the last rows' dx
        if (S1 < S0) S1 = S0;
    }

    // ------------------------------------------------------------ producer
    if (warp == NC) {
        const int nst = (S1 - S0 + R - 1) / R;
        const uint32_t row_bytes = static_cast<uint32_t>(col_ch) * 2;
        bool ok = true;
        for (int k = 0; k < nst && ok; ++k) {
            const int s = k % P;
            if (k >= P) ok = mbar_wait(bars + 8 * (P + s), ((k / P) - 1) & 1);
            if (!ok) break;
            const int r0 = S0 + k * R;
            const int nrows = min(R, S1 - r0);
            if (lane == 0) mbar_arrive_expect_tx(bars + 8 * s, static_cast<uint32_t>(nrows) * 2 * row_bytes);
            __syncwarp();
            if (lane < 2 * nrows) {
                const int q = lane >> 1, tensor = lane & 1;
                const int r = r0 + q;
                const uint16_t *src = tensor ? a.dy + static_cast<int64_t>(r) * a.dys + col_c0
                                             : a.x + static_cast<int64_t>(r) * a.xs + col_c0;
                const uint32_t dst = sbase + static_cast<uint32_t>(s * RG::kStageBytes + (q * 2 + tensor) * RG::kRowBytes);
                bulk_g2s(dst, src, row_bytes, bars + 8 * s);
            }
        }
        // Do not leave while copies into this CTA's shared memory may be in
        // flight: wait (bounded) for the last stages issued to land.
        const int issued = ok ? nst : 0;
        for (int k = max(0, issued - P); k < issued; ++k) mbar_wait(bars + 8 * (k % P), (k / P) & 1);
        return;
    }

    // ------------------------------------------------------------ consumers
    if (warp >= nact) return;
    const int c0 = col_c0 + warp * kSlab + lane * kVec;
    const bool act = c0 < a.C;
    const bool full = (warp + 1) * kSlab <= col_ch;  // warp-uniform: all lanes have channels

    float2 w0[NV], w1[NV], w2[NV], w3[NV], bb[NV];
    load_taps<NV>(a.w, a.w_bf16, a.b, a.b_kind, act ? c0 : 0, act, w0, w1, w2, w3, bb);
    float2 g0[NV], g1[NV], g2[NV], g3[NV], gb[NV];  // sum dz*h[j+k], sum dz
#pragma unroll
    for (int v = 0; v < NV; ++v) g0[v] = g1[v] = g2[v] = g3[v] = gb[v] = f2_zero();

    StageReader<NC, R, P> src;
    src.lane_base = sbase + static_cast<uint32_t>((warp * kSlab + lane * kVec) * 2);
    src.bars = bars;
    src.S0 = S0;
    src.k_full = 0;
    src.k_rel = 0;
    src.ok = true;

    float2 h0[NV], h1[NV], h2[NV], d1[NV], d2[NV], d3[NV];
    Item cur = {};
    bool live = true, read_state = false;

    for (int it = lo; it < hi && src.ok; ++it) {
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

        if (!cont) {
            // History rows o0-3 .. o0-1: from the stream when the walk starts
            // inside a sequence, else the saved initial history (or zeros).
            Raw<NV> hr[3];
#pragma unroll
            for (int p = 0; p < 3; ++p) hr[p] = raw_zero<NV>();
            if (o0 > 0) {
                src.need(t.r0 - 1);
#pragma unroll
                for (int p = 0; p < 3; ++p) hr[p] = src.row(t.r0 - 3 + p, 0);
            } else if (a.hist && act) {
#pragma unroll
                for (int p = 0; p < 3; ++p) hr[p] = ld_ro<NV>(a.hist + (static_cast<int64_t>(t.n) * 3 + p) * a.C + c0);
            }
            unpack<NV>(hr[0], h0);
            unpack<NV>(hr[1], h1);
            unpack<NV>(hr[2], h2);
#pragma unroll
            for (int v = 0; v < NV; ++v) d1[v] = d2[v] = d3[v] = f2_zero();
        }

        const int iters = nr + (next_cont ? 0 : 3);
        const int nload = L - o0 < iters ? L - o0 : iters;  // steps with i < L
        for (int base = 0; base < iters && src.ok; base += U) {
            const bool fast = full && (cont || base >= 3) && base + U <= nload && base + U <= nr;
            // Rows before the next row this walk reads are done with (in the
            // tail steps past a sequence's end that row is the next
            // sequence's first, which must stay resident).
            src.release_before(t.r0 + min(base, nload), lane);
            Raw<NV> xr[U], gr[U];
            if (base < nload) {
                src.need(t.r0 + min(base + U, nload) - 1);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const bool ld = fast || base + u < nload;
                    xr[u] = ld ? src.row(t.r0 + base + u, 0) : raw_zero<NV>();
                    gr[u] = ld ? src.row(t.r0 + base + u, 1) : raw_zero<NV>();
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) xr[u] = gr[u] = raw_zero<NV>();
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
                        float2 c = __ffma2_rn(w0[v], dz[v], f2_zero());
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
                if (k < nr) {
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        g0[v] = __ffma2_rn(dz[v], h0[v], g0[v]);
                        g1[v] = __ffma2_rn(dz[v], h1[v], g1[v]);
                        g2[v] = __ffma2_rn(dz[v], h2[v], g2[v]);
                        g3[v] = __ffma2_rn(dz[v], hc[v], g3[v]);
                        gb[v] = __fadd2_rn(gb[v], dz[v]);
                    }
                }
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

    // Release what is left so the producer can finish, then let the reduce
    // kernel get scheduled.
    src.drain((S1 - S0 + R - 1) / R, lane);
    grid_dependents_launch();

    // partial[run][k][c0 .. c0+4): NaN if a wait timed out, so a failed
    // handshake shows in dweight instead of passing silently.
    if (act) {
        if (!src.ok) {
            const float nan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int v = 0; v < NV; ++v) g0[v] = g1[v] = g2[v] = g3[v] = gb[v] = make_float2(nan, nan);
        }
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

}  // namespace

cudaError_t launch_bwd_tma(const BwdArgs &a, bool pdl, cudaStream_t st) {
    constexpr int NC = kBwdTmaWarps, R = kBwdTmaRows, P = kBwdTmaStages, U = kBwdUnroll;
    using RG = Ring<NC, R, P>;
    auto kern = bwd_tma_kernel<NC, R, P, U>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RG::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(a.slabs) * a.runs));
    cfg.blockDim = dim3((NC + 1) * 32);
    cfg.dynamicSmemBytes = RG::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace ccc
