// ccc_check.cu -- device-side check of the caller-owned metadata (offsets,
// slot IDs, accepted counts) declared in include/ccc.h as ccc_check.  The
// pages leave those values unchecked (FlashInfer
// "flashinfer.mamba.causal_conv1d_fn", Notes: they are the caller's to get
// right, and the library neither reads them on the host nor synchronizes to
// validate them); this kernel checks them on the device, still without a
// host synchronization, and reports through a status word, never trapping.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ccc.h"

namespace {

constexpr int kCheckThreads = 256;
constexpr int kCheckMaxCtas = 1024;

// One thread per offset i in [0, N] (grid-stride), which also checks
// sequence i's slot and accepted count.  A live slot q sets bit q of the
// bitmap in status[1 ..]; finding it already set means a second sequence
// uses the slot.  Each warp ORs its violations into status[0] once.
__global__ void check_kernel(int64_t rows, const int32_t *__restrict__ cu, int N,
                             const int32_t *__restrict__ cache, int n_slots,
                             const int32_t *__restrict__ accepted, int max_accepted, uint32_t *status) {
    uint32_t bits = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i <= N; i += stride) {
        const int v = cu[i];
        if (i == 0 && v != 0) bits |= CCC_CHECK_CU_START;
        if (v < 0 || v > rows) bits |= CCC_CHECK_CU_RANGE;
        if (i > 0 && v < cu[i - 1]) bits |= CCC_CHECK_CU_ORDER;
        if (i < N) {
            if (cache) {
                const int q = cache[i];
                if (q != -1 && (q < 0 || q >= n_slots)) {
                    bits |= CCC_CHECK_SLOT_RANGE;
                } else if (q >= 0) {
                    const uint32_t m = 1u << (q & 31);
                    if (atomicOr(status + 1 + (q >> 5), m) & m) bits |= CCC_CHECK_SLOT_DUP;
                }
            }
            if (accepted) {
                const int a = accepted[i];
                if (a < 1 || a > max_accepted) bits |= CCC_CHECK_ACCEPTED;
            }
        }
    }
    bits = __reduce_or_sync(0xffffffffu, bits);
    if ((threadIdx.x & 31) == 0 && bits) atomicOr(status, bits);
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || !an || !bn) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" {

size_t ccc_check_status_words(int32_t n_slots) {
    return 1 + (n_slots > 0 ? (static_cast<size_t>(n_slots) + 31) / 32 : 0);
}

int ccc_check(int64_t rows, const int32_t *cu_seqlens, int32_t N,
              const int32_t *cache_indices, int32_t n_slots,
              const int32_t *num_accepted, int32_t max_accepted,
              uint32_t *status, size_t status_words, void *cuda_stream) {
    if (rows < 0 || N < 0 || (cache_indices && n_slots < 0) || (num_accepted && max_accepted < 1))
        return CCC_ERR_SHAPE;
    if (!cu_seqlens || !status) return CCC_ERR_NULL;
    if (!aligned4(cu_seqlens) || !aligned4(status) || (cache_indices && !aligned4(cache_indices)) ||
        (num_accepted && !aligned4(num_accepted)))
        return CCC_ERR_ALIGN;
    const size_t words = cache_indices ? ccc_check_status_words(n_slots) : 1;
    if (status_words < words) return CCC_ERR_WORKSPACE;
    const size_t sb = words * 4;
    if (overlap(status, sb, cu_seqlens, (static_cast<size_t>(N) + 1) * 4) ||
        overlap(status, sb, cache_indices, static_cast<size_t>(N) * 4) ||
        overlap(status, sb, num_accepted, static_cast<size_t>(N) * 4))
        return CCC_ERR_ALIAS;
    const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemsetAsync(status, 0, sb, st) != cudaSuccess) return CCC_ERR_CUDA;
    const int64_t want = (static_cast<int64_t>(N) + kCheckThreads) / kCheckThreads;  // ceil((N + 1) / threads)
    const int ctas = static_cast<int>(want < kCheckMaxCtas ? want : kCheckMaxCtas);
    check_kernel<<<ctas, kCheckThreads, 0, st>>>(rows, cu_seqlens, N, cache_indices, n_slots, num_accepted,
                                                 max_accepted, status);
    return cudaGetLastError() == cudaSuccess ? CCC_OK : CCC_ERR_CUDA;
}

}  // extern "C"
