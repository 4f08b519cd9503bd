// ccc_chunkmap.cu -- device chunk-map builder: cu_seqlens -> work items.
//
// FlashInfer "flashinfer.mamba.causal_conv1d_fn" (workspace, Notes): for
// larger batches the sequence offsets are turned into a list of
// (sequence, token-chunk) work items in device scratch on every call,
// without any host read of the offsets, so the call stays capturable in a
// CUDA graph while cu_seqlens changes in place between replays.
//
// Output layout (int32): map[0] = item count, then for item i the pair
// (map[1 + 2i], map[2 + 2i]) = (sequence n, first row r0).  Items of a
// sequence are its consecutive B-row chunks; sequences appear in order.
// One CTA of 1024 threads: each thread owns a contiguous block of sequences,
// a block-wide exclusive scan of the per-block item counts gives each block
// its first item, then every warp writes the items of its 32 blocks with all
// lanes storing in parallel (so one very long sequence is written 32 items at
// a time, not by one thread).  Items past `cap` are dropped, so an invalid
// cu_seqlens can never write outside the map.
#include "ccc_device.cuh"
#include "ccc_internal.h"

namespace ccc {

namespace {

constexpr int kMapThreads = 1024;

__device__ __forceinline__ int row_clamp(int v, int64_t rows) {
    return v < 0 ? 0 : (v > rows ? static_cast<int>(rows) : v);
}

// Offsets of up to kSmemSeqs sequences are staged in shared memory with one
// coalesced pass, so the scan and the item writes read no global memory.
constexpr int kSmemSeqs = 8192;

__global__ void __launch_bounds__(kMapThreads) chunkmap_kernel(const int32_t *__restrict__ cu, int N,
                                                               int64_t rows, int B, int empty_items,
                                                               int32_t *__restrict__ map, int cap) {
    // Let the consumer kernel start its prologue (tap loads); it waits for
    // this grid's writes in grid_dependency_wait().
    grid_dependents_launch();

    __shared__ int warp_tot[32];
    __shared__ int s_cu[kSmemSeqs + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool staged = N <= kSmemSeqs;
    if (staged) {
        for (int i = tid; i <= N; i += kMapThreads) s_cu[i] = row_clamp(__ldg(cu + i), rows);
        __syncthreads();
    }
    auto off_of = [&](int n) { return staged ? s_cu[n] : row_clamp(__ldg(cu + n), rows); };

    const int per = (N + kMapThreads - 1) / kMapThreads;
    const int n0 = min(tid * per, N), n1 = min(n0 + per, N);

    auto items_of = [&](int n) {
        const int s = off_of(n), e = off_of(n + 1);
        const int len = e > s ? e - s : 0;
        int ni = (len + B - 1) / B;
        if (empty_items && ni == 0) ni = 1;
        return ni;
    };

    int local = 0;
    for (int n = n0; n < n1; ++n) local += items_of(n);

    // Block exclusive scan of `local`.
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(kFull, v, off);
            if (lane >= off) v += t;
        }
        warp_tot[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int base = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - local;

    // Each warp writes the items of its 32 sequence blocks, one block at a
    // time, all lanes in parallel.
    for (int owner = 0; owner < 32; ++owner) {
        int off = __shfl_sync(kFull, base, owner);
        const int on0 = __shfl_sync(kFull, n0, owner), on1 = __shfl_sync(kFull, n1, owner);
        for (int n = on0; n < on1; ++n) {
            const int s = off_of(n);
            const int ni = items_of(n);
            for (int i = lane; i < ni; i += 32) {
                const int idx = off + i;
                if (idx < cap) {
                    map[1 + 2 * idx] = n;
                    map[2 + 2 * idx] = s + i * B;
                }
            }
            off += ni;
        }
    }
    if (tid == kMapThreads - 1) {
        const int total = base + local;
        map[0] = total < cap ? total : cap;
    }
}

}  // namespace

cudaError_t launch_chunkmap(const int32_t *cu, int N, int64_t rows, int B, int empty_items,
                            int32_t *map, int cap, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kMapThreads);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, chunkmap_kernel, cu, N, rows, B, empty_items, map, cap);
}

}  // namespace ccc
