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
// device symbol, never a device address: the address is fetched once per
// device with cudaGetSymbolAddress (with that device current) on the first
// call made on that device, and cached.  That first call on a device should
// therefore come before any stream capture on it.
//
// Every call uses the same array and leaves its contents behind for the next
// call.  Nothing in it has to start at zero: the backward writes every
// partial sum before the reduction reads it.  The backward's scratch is
// R x 5 x C floats with R x ceil(C / 256) <= 1216, at most about 6.2 MB, so
// every shape fits; the size check stays as a guard.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads on the
// same device) race on the array; callers must serialize them.
#include <mutex>

#include <cuda_runtime.h>

#include "ccc.h"

namespace {

constexpr size_t kScratchBytes = CCC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set up on first use).
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CCC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return CCC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
