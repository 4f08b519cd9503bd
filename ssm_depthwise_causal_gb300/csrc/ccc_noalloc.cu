// ccc_noalloc.cu -- ccc_bwd_noalloc: the backward without a caller-supplied
// workspace, for callers that cannot allocate device memory.
//
// Some callers of the backward have no way to obtain a device buffer for the
// scratch it needs: code running inside a host framework whose memory pool
// it has no handle to, plugin hosts that forbid device allocation after
// start-up, and latency-critical paths that cannot pay for cudaMalloc, which
// may synchronize the whole device.  This entry point serves them from a
// fixed scratch array compiled into the library instead.
//
// The scratch is one file-scope __device__ array of kScratchBytes.  Every GPU
// on which the library's module is loaded holds it until the process exits.
// The name `g_scratch` in host code is only a host-side stand-in for the
// device symbol, never a device address.  The device address is looked up
// with cudaGetSymbolAddress, with the caller's device current, at set-up:
// the first call made in a CUDA context (normally the device's primary
// context, so once per device; again after a device reset, which replaces
// that context, or in any other context the caller makes current), and
// cached under the context's unique ID, which the driver never reuses within
// a process.  That first call in a context should come before any stream
// capture in it.
//
// Every call uses the same array and leaves its contents behind for the next
// call.  Nothing in it has to start at zero: the backward writes every
// partial sum before the reduction reads it.  The backward's scratch is
// R x 5 x C floats (R partial rows, R x ceil(C / 256) <= 1216 and R >= 1), at
// most max(6,225,920, 20 x C) bytes, so every C up to 838,856 fits; larger C
// is refused before any CUDA call.  Two calls whose work overlaps on the GPU
// (different streams, or different host threads on the same device) race on
// the array; callers must serialize them.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ccc.h"

namespace {

constexpr size_t kScratchBytes = CCC_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Driver entry points, fetched through the runtime so the library needs no
// link against the driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

std::once_flag g_entry_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

void load_entry_points() {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
}

// Unique ID of the context current on this thread; 0 when there is none yet
// (or it cannot be read).
unsigned long long current_context_id() {
    std::call_once(g_entry_once, load_entry_points);
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Cache of looked-up addresses: context ID -> device address of g_scratch.
struct Entry {
    unsigned long long ctx_id;
    void *addr;
};
constexpr int kCacheEntries = 64;
std::mutex g_cache_mu;
Entry g_cache[kCacheEntries] = {};
int g_cache_next = 0;

// Device address of g_scratch in the current context (looked up on the
// first call in each context).
int scratch_address(void **out) {
    unsigned long long id = current_context_id();
    if (id == 0) {
        // No context on this thread yet: the lookup below makes the current
        // device's primary context current (as any runtime call would).
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return CCC_ERR_CUDA;
        id = current_context_id();
        if (id == 0) {  // cannot key it: use the fresh lookup uncached
            *out = p;
            return CCC_OK;
        }
    }
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (const Entry &e : g_cache) {
        if (e.ctx_id == id) {
            *out = e.addr;
            return CCC_OK;
        }
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return CCC_ERR_CUDA;
    g_cache[g_cache_next] = Entry{id, p};
    g_cache_next = (g_cache_next + 1) % kCacheEntries;
    *out = p;
    return CCC_OK;
}

}  // namespace

extern "C" int ccc_bwd_noalloc(const void *x, int64_t rows, int32_t C, int64_t x_row_stride,
                               const void *weight, int32_t w_dtype, int32_t width,
                               const void *bias, int32_t b_dtype, int32_t activation,
                               const void *saved_hist,
                               const int32_t *cu_seqlens, int32_t N,
                               const int32_t *cache_indices, const uint8_t *has_initial_state,
                               const void *dy, int64_t dy_row_stride,
                               const float *d_final_state,
                               void *dx, int64_t dx_row_stride,
                               float *dweight, float *dbias, float *d_init_state,
                               void *cuda_stream) {
    const size_t need = ccc_workspace_size(rows, N, C, 1);
    if (need > kScratchBytes) return CCC_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&ws);
        if (rc != CCC_OK) return rc;
    }
    return ccc_bwd(x, rows, C, x_row_stride, weight, w_dtype, width, bias, b_dtype, activation, saved_hist,
                   cu_seqlens, N,
                   cache_indices, has_initial_state, dy, dy_row_stride, d_final_state, dx, dx_row_stride,
                   dweight, dbias, d_init_state, ws, need > 0 ? kScratchBytes : 0, cuda_stream);
}
