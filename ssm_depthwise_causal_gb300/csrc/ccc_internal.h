// ccc_internal.h -- launch interface between the C-ABI layer (ccc_api.cu)
// and the kernels (ccc_chunkmap.cu, ccc_fwd.cu, ccc_bwd.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ccc {

// Tuning constants.  Each can be overridden at compile time (-DCCC_...) for
// sweeps; the defaults are the measured choice on GB300.
#ifndef CCC_FWD_CHUNK
#define CCC_FWD_CHUNK 64
#endif
#ifndef CCC_BWD_CHUNK
#define CCC_BWD_CHUNK 64
#endif
#ifndef CCC_FWD_VEC
#define CCC_FWD_VEC 8
#endif
#ifndef CCC_BWD_VEC
#define CCC_BWD_VEC 8
#endif
#ifndef CCC_FWD_UNROLL
#define CCC_FWD_UNROLL 4
#endif
#ifndef CCC_BWD_UNROLL
#define CCC_BWD_UNROLL 4
#endif
#ifndef CCC_FWD_MIN_BLOCKS
#define CCC_FWD_MIN_BLOCKS 2
#endif
#ifndef CCC_BWD_MIN_BLOCKS
#define CCC_BWD_MIN_BLOCKS 1
#endif
#ifndef CCC_UPD_MIN_BLOCKS
#define CCC_UPD_MIN_BLOCKS 2
#endif
#ifndef CCC_BWD_TARGET_WARPS
#define CCC_BWD_TARGET_WARPS 1216
#endif
#ifndef CCC_BWD_RING
#define CCC_BWD_RING 3
#endif
#ifndef CCC_BWD_TMA
#define CCC_BWD_TMA 0
#endif
#ifndef CCC_FWD_RING
#define CCC_FWD_RING 0
#endif
#ifndef CCC_FWD_PREFETCH
#define CCC_FWD_PREFETCH 4
#endif
#ifndef CCC_BWD_PREFETCH
#define CCC_BWD_PREFETCH 0
#endif
#ifndef CCC_BWD_TMA_WARPS
#define CCC_BWD_TMA_WARPS 4
#endif
#ifndef CCC_BWD_TMA_ROWS
#define CCC_BWD_TMA_ROWS 16
#endif
#ifndef CCC_BWD_TMA_STAGES
#define CCC_BWD_TMA_STAGES 3
#endif
#ifndef CCC_BWD_TMA_MIN_BLOCKS
#define CCC_BWD_TMA_MIN_BLOCKS 2
#endif

// Rows per work item.  Long enough that the 3-row halo an item re-reads
// (forward: left; backward: left and right) is a few percent of its rows and
// is served from L2, short enough that a lognormal mix of short sequences
// still yields many items.
constexpr int kFwdChunk = CCC_FWD_CHUNK;
constexpr int kBwdChunk = CCC_BWD_CHUNK;
// Above this many sequences the items come from the device chunk map.
constexpr int kMaxInlineSeqs = 32;
// Channels per lane (8: one 16-byte vector per row).  The backward's
// per-lane state (taps, bias, two sliding windows, five partial sums) then
// needs ~200 registers, so it runs one 256-thread CTA per SM and takes its
// memory-level parallelism from the shared-memory ring below instead of from
// more warps.
constexpr int kFwdVec = CCC_FWD_VEC;
constexpr int kBwdVec = CCC_BWD_VEC;
// Rows loaded ahead per lane before the math (independent loads in flight).
constexpr int kFwdUnroll = CCC_FWD_UNROLL;
constexpr int kBwdUnroll = CCC_BWD_UNROLL;
// Resident CTAs per SM the register budget is sized for.
constexpr int kFwdMinBlocks = CCC_FWD_MIN_BLOCKS;
constexpr int kBwdMinBlocks = CCC_BWD_MIN_BLOCKS;
// Decode update: resident CTAs per SM the register budget is sized for.
constexpr int kUpdMinBlocks = CCC_UPD_MIN_BLOCKS;
// Forward: stages of the per-lane shared-memory ring (0 = load rows straight
// into registers).
constexpr int kFwdRing = CCC_FWD_RING;
// Rows ahead of the current batch whose slabs the kernels ask to be brought
// into L2 (cp.async.bulk.prefetch.L2, one row slab per lane); 0 = off.
constexpr int kFwdPrefetch = CCC_FWD_PREFETCH;
constexpr int kBwdPrefetch = CCC_BWD_PREFETCH;
// Backward: stages of the per-lane shared-memory ring (0 = load rows
// straight into registers).
constexpr int kBwdRing = CCC_BWD_RING;
// Backward fed by a bulk-copy producer warp (ccc_bwd_tma.cu): consumer
// warps per CTA (128 channels each), rows per shared-memory stage, stages,
// resident CTAs per SM.
constexpr bool kBwdTma = CCC_BWD_TMA != 0;
constexpr int kBwdTmaWarps = CCC_BWD_TMA_WARPS;
constexpr int kBwdTmaRows = CCC_BWD_TMA_ROWS;
constexpr int kBwdTmaStages = CCC_BWD_TMA_STAGES;
constexpr int kBwdTmaMinBlocks = CCC_BWD_TMA_MIN_BLOCKS;
// Backward warps the work split is sized for: 152 SMs x 1 resident CTA x 8
// warps, i.e. one full wave on GB300.  Fixed, not queried, so the reduction
// order -- and with it every bit of dweight / dbias -- depends only on
// (rows, N, C).
constexpr int kBwdTargetWarps = CCC_BWD_TARGET_WARPS;

// Warps per CTA of the forward and backward kernels.
constexpr int kWarpsPerCta = 8;

// Upper bound on the number of work items: the sum over sequences of
// max(1, ceil(len / B)) is at most ceil(rows / B) + N.
inline int64_t item_capacity(int64_t rows, int64_t N, int B) { return (rows + B - 1) / B + N; }

struct FwdArgs {
    const uint16_t *x;
    int64_t rows;
    int C;
    int xs;  // row strides in elements (host-checked < 2^31)
    const void *w;
    int w_bf16;
    const void *b;
    int b_kind;  // 0 none, 1 FP32, 2 BF16
    int width;   // taps W (2..4); W-1 history rows
    int act;     // 1 SiLU, 0 none
    uint16_t *state;
    int n_slots;
    int64_t st_slot, st_c, st_l;
    int state_vec;  // channel axis contiguous and 16-byte aligned rows
    const int32_t *cu;
    int N;
    const int32_t *cache;
    const uint8_t *has_init;
    uint16_t *out;
    int os;
    uint16_t *hist;
    const int32_t *map;  // nullptr: items derived in-kernel
    int cap;
    int slabs, runs;     // work split (see runs_per_slab)
};

struct BwdArgs {
    const uint16_t *x;
    int64_t rows;
    int C;
    int xs;  // row strides in elements (host-checked < 2^31)
    const void *w;
    int w_bf16;
    const void *b;
    int b_kind;
    int width;   // taps W (2..4); W-1 history rows
    int act;     // 1 SiLU, 0 none
    const uint16_t *hist;
    const int32_t *cu;
    int N;
    const int32_t *cache;
    const uint8_t *has_init;
    const uint16_t *dy;
    int dys;
    const float *d_final;
    uint16_t *dx;
    int dxs;
    float *d_init;
    float *part;  // [runs][5][C]: rows 0..W-1 taps, row 4 bias
    const int32_t *map;
    int cap;
    int slabs, runs;
};

// The speculative / single-token decode update (ccc_update.cu).
struct UpdArgs {
    const uint16_t *x;
    int64_t rows;
    int C;
    int xs;
    const void *w;
    int w_bf16;
    const void *b;
    int b_kind;
    int width;
    int act;
    uint16_t *state;
    int n_slots;
    int L;
    int64_t st_slot, st_c, st_l;
    int state_vec;    // channel axis contiguous, 16-byte aligned rows
    int state_stage;  // dense history-contiguous pool, L <= update_stage_max_len()
    const int32_t *cu;
    int N;
    const int32_t *cache;
    const int32_t *accepted;
    uint16_t *out;
    int os;
    int slabs;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Work split of both kernels.  Every warp owns one task: a 32*VEC-channel
// slab and a run of consecutive items, runs_per_slab runs per slab; warp g
// (global index) takes slab g % slabs and run g / slabs, so the 8 warps of a
// CTA cover neighbouring slabs of the same rows.  The grid is
// ceil(slabs * runs / 8) CTAs -- sized to one resident wave, so no CTA waits
// for a second wave with a whole run of work.
inline int slabs_of(int C, int vec) { return static_cast<int>(ceil_div(C, 32 * vec)); }

inline int runs_per_slab(int64_t target_warps, int slabs, int64_t cap) {
    int64_t r = target_warps / slabs;
    if (r > cap) r = cap;
    return static_cast<int>(r < 1 ? 1 : r);
}

// Backward task split: `slabs` task columns (a slab of 32*VEC channels per
// warp, or a column of kBwdTmaWarps*128 channels per CTA for the bulk-copy
// kernel) times `runs` runs per column; runs is also the number of FP32
// partial rows per channel.  Both depend only on (rows, N, C).
// The bulk-copy backward (when built in) serves the width-4 SiLU contract of
// causal_conv1d_fn; the other widths and the no-activation variant always
// take the register-fed kernel.
inline bool bwd_uses_tma(int width, int act) { return kBwdTma && width == 4 && act == 1; }

inline int bwd_columns(int C, bool tma) {
    return tma ? static_cast<int>(ceil_div(C, kBwdTmaWarps * 128)) : slabs_of(C, kBwdVec);
}

inline int bwd_runs(int64_t rows, int N, int C, bool tma) {
    const int64_t target = tma ? int64_t{152} * kBwdTmaMinBlocks : kBwdTargetWarps;
    return runs_per_slab(target, bwd_columns(C, tma), item_capacity(rows, N, kBwdChunk));
}

cudaError_t launch_chunkmap(const int32_t *cu, int N, int64_t rows, int B, int empty_items,
                            int32_t *map, int cap, cudaStream_t st);
cudaError_t launch_fwd(const FwdArgs &a, bool pdl, cudaStream_t st);
cudaError_t launch_bwd(const BwdArgs &a, bool pdl, cudaStream_t st);
cudaError_t launch_bwd_tma(const BwdArgs &a, bool pdl, cudaStream_t st);
// Resident forward CTAs per SM on the current device (occupancy query).
int fwd_ctas_per_sm();
cudaError_t launch_reduce(const float *part, int G, int C, int width, float *dweight, float *dbias,
                          bool pdl, cudaStream_t st);
int update_slabs(int C);
int update_stage_max_len();
cudaError_t launch_update(const UpdArgs &a, cudaStream_t st);

}  // namespace ccc
