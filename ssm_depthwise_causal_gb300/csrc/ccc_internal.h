// ccc_internal.h -- launch interface between the C-ABI layer (ccc_api.cu)
// and the kernels (ccc_fwd.cu, ccc_bwd.cu, ccc_update.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ccc {

// Tuning constants.  Each can be overridden at compile time (-DCCC_...) for
// sweeps; the defaults are the measured choice on GB300.
#ifndef CCC_FWD_CHUNK
#define CCC_FWD_CHUNK 128
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
#ifndef CCC_FWD_UNROLL_W4
#define CCC_FWD_UNROLL_W4 3
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
#ifndef CCC_BWD_MIN_RUN_ROWS
#define CCC_BWD_MIN_RUN_ROWS 16
#endif
#ifndef CCC_BWD_RING
#define CCC_BWD_RING 3
#endif
#ifndef CCC_FWD_PREFETCH
#define CCC_FWD_PREFETCH 4
#endif
#ifndef CCC_BWD_PREFETCH
#define CCC_BWD_PREFETCH 0
#endif
#ifndef CCC_FWD_WALK_ROWS
#define CCC_FWD_WALK_ROWS 0
#endif
#ifndef CCC_BWD_WALK_ROWS
#define CCC_BWD_WALK_ROWS 10
#endif
#ifndef CCC_BWD_NEXT_WALK_PREFETCH
#define CCC_BWD_NEXT_WALK_PREFETCH 1
#endif
#ifndef CCC_BWD_PREFETCH_WALK_MAX
#define CCC_BWD_PREFETCH_WALK_MAX 96
#endif
#ifndef CCC_FWD_WAVES
#define CCC_FWD_WAVES 1
#endif
#ifndef CCC_FWD_STAGE_SEQS
#define CCC_FWD_STAGE_SEQS 1024
#endif
#ifndef CCC_BWD_STAGE_SEQS
#define CCC_BWD_STAGE_SEQS 256
#endif

// Rows per segment of a walk (RunWalker).  The segment length only bounds
// the inner loop (and is a multiple of the backward's batch so a walk's
// batches stay aligned across segments).  Forward: 128 (64 left the dense
// 16384 x 4096 forward 1.4 % slower; 256 and 1024 gained nothing more).
constexpr int kFwdChunk = CCC_FWD_CHUNK;
constexpr int kBwdChunk = CCC_BWD_CHUNK;
// Channels per lane (8: one 16-byte vector per row).  The backward's
// per-lane state (taps, bias, two sliding windows, five partial sums) then
// needs ~200 registers, so it runs one 256-thread CTA per SM and takes its
// memory-level parallelism from the shared-memory ring below instead of from
// more warps.
constexpr int kFwdVec = CCC_FWD_VEC;
constexpr int kBwdVec = CCC_BWD_VEC;
// Rows loaded ahead per lane before the math (independent loads in flight).
// The width-4 forward takes 3 rows per batch: its 3-row window then comes
// back to the same registers every batch (no register shuffling).
constexpr int kFwdUnroll = CCC_FWD_UNROLL;
constexpr int kFwdUnrollW4 = CCC_FWD_UNROLL_W4;

constexpr int kBwdUnroll = CCC_BWD_UNROLL;
// Resident CTAs per SM the register budget is sized for.
constexpr int kFwdMinBlocks = CCC_FWD_MIN_BLOCKS;
constexpr int kBwdMinBlocks = CCC_BWD_MIN_BLOCKS;
// Decode update: resident CTAs per SM the register budget is sized for.
constexpr int kUpdMinBlocks = CCC_UPD_MIN_BLOCKS;
// Rows ahead of the current batch whose slabs the kernels ask to be brought
// into L2 (cp.async.bulk.prefetch.L2, one row slab per lane); 0 = off.
constexpr int kFwdPrefetch = CCC_FWD_PREFETCH;
constexpr int kBwdPrefetch = CCC_BWD_PREFETCH;
// What a sequence start costs a kernel, in rows' worth of time (the run
// split balances rows plus this per sequence, RunWalker::init; 0 = rows
// only).  Measured: a walk of the backward (ring refill, initial history,
// guarded first and last batches) costs about as much as 8-11 rows, and
// the weight takes its slowest run on the packed mix from ~3 % above the
// mean to ~0 (backward 0.5 % faster); a walk of the forward costs 2-3 rows,
// too little to pay for the two extra searches of a weighted split.
constexpr int kFwdWalkRows = CCC_FWD_WALK_ROWS;
constexpr int kBwdWalkRows = CCC_BWD_WALK_ROWS;
// Backward: at each walk start, ask L2 for the next sequence's first rows
// and saved history (what its walk start waits on).
constexpr bool kBwdNextWalkPrefetch = CCC_BWD_NEXT_WALK_PREFETCH != 0;
// ... only when the current walk loads at most this many rows.
constexpr int kBwdPrefetchWalkMax = CCC_BWD_PREFETCH_WALK_MAX;
// Backward: stages of the per-lane shared-memory ring (0 = load rows
// straight into registers).
constexpr int kBwdRing = CCC_BWD_RING;
// Backward warps the work split is sized for: 152 SMs x 1 resident CTA x 8
// warps, i.e. one full wave on GB300.  Fixed, not queried, so the reduction
// order -- and with it every bit of dweight / dbias -- depends only on the
// host arguments (rows, C), never on the device or on device values.
constexpr int kBwdTargetWarps = CCC_BWD_TARGET_WARPS;
// ... but never more runs per slab than one per this many rows of the
// batch: a small batch then writes (and the reduce re-reads) a few partial
// rows instead of ~1216 / slabs of them.
constexpr int kBwdMinRunRows = CCC_BWD_MIN_RUN_ROWS;

// Warps per CTA of the forward and backward kernels.
constexpr int kWarpsPerCta = 8;
// Forward: resident waves of warps the rows are split over (1: every warp
// has one run and the grid is one wave).
constexpr int kFwdWaves = CCC_FWD_WAVES;
// Sequences whose offsets, slots and flags a CTA stages in shared memory
// (multiples of 128).  The backward's is small so that its copy ring plus
// this stays within the 100 KB shared-memory carveout.
constexpr int kFwdStageSeqs = CCC_FWD_STAGE_SEQS;
constexpr int kBwdStageSeqs = CCC_BWD_STAGE_SEQS;

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
    int slabs, runs;     // work split (see runs_per_slab)
    int taps_vec;        // weight and bias 16-byte aligned: taps read through shared memory
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
    int slabs, runs;
    int taps_vec;  // weight and bias 16-byte aligned: taps read through shared memory
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
    int groups;  // sequence groups per slab (CTA b: slab b % slabs, group b / slabs)
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Work split of both kernels.  Every warp owns one task: a 32*VEC-channel
// slab and a run of rows (an equal share of the valid rows, see RunWalker),
// runs_per_slab runs per slab; warp g
// (global index) takes slab g % slabs and run g / slabs, so the 8 warps of a
// CTA cover neighbouring slabs of the same rows.  The grid is
// ceil(slabs * runs / 8) CTAs -- sized to one resident wave, so no CTA waits
// for a second wave with a whole run of work.
inline int slabs_of(int C, int vec) { return static_cast<int>(ceil_div(C, 32 * vec)); }

inline int runs_per_slab(int64_t target_warps, int slabs) {
    const int64_t r = target_warps / slabs;
    return static_cast<int>(r < 1 ? 1 : r);
}

// Backward task split: slabs of 32*VEC channels times `runs` runs per slab;
// runs is also the number of FP32 partial rows per channel.  Both depend
// only on the host arguments rows and C: runs = min(1216 / slabs,
// ceil(rows / kBwdMinRunRows)), at least 1.
inline int bwd_slabs(int C) { return slabs_of(C, kBwdVec); }

inline int bwd_runs(int64_t rows, int C) {
    const int by_width = runs_per_slab(kBwdTargetWarps, bwd_slabs(C));
    const int64_t by_rows = ceil_div(rows < 1 ? 1 : rows, kBwdMinRunRows);
    return by_rows < by_width ? static_cast<int>(by_rows) : by_width;
}

// `overlap`: launch as a programmatic dependent of the previous kernel in
// the stream (the prologue may run while that kernel finishes; the kernel
// waits for it before touching activations, history, state or outputs).
cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t st, bool overlap);
// sms: the device's SM count (a grid of at most 7 tasks per SM runs as
// one-warp CTAs).
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t st, bool overlap, int sms);
// Resident forward CTAs per SM on the current device (occupancy query).
int fwd_ctas_per_sm();
cudaError_t launch_reduce(const float *part, int G, int C, int width, float *dweight, float *dbias,
                          cudaStream_t st);
int update_slabs(int C);
int update_stage_max_len();
int update_groups(int N, int slabs, int sms);
cudaError_t launch_update(const UpdArgs &a, cudaStream_t st, bool overlap);

}  // namespace ccc
