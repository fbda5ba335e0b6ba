// noalloc.cu -- RMSNorm backward for callers that cannot allocate device
// memory: the same kernels as rmsnorm_bwd, with the dgamma partial rows kept
// in a fixed scratch array that lives in this file instead of a
// caller-provided workspace.
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gbnorm.h"

namespace {

constexpr size_t kScratchBytes = (size_t)GBNORM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDev = 64;

// One copy per device, reserved when the library's device code is loaded on
// that device and held until the process exits.  Host code must not pass
// this name to a kernel: on the host it is only a stand-in for the symbol.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDev];
std::atomic<int> g_ready[kMaxDev];

// Device address of this device's scratch, looked up once per device with
// that device current.
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GBNORM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return GBNORM_ERR_UNSUPPORTED;
    if (!g_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_ready[dev].load(std::memory_order_relaxed)) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
                return GBNORM_ERR_CUDA;
            g_addr[dev] = p;
            g_ready[dev].store(1, std::memory_order_release);
        }
    }
    *out = g_addr[dev];
    return GBNORM_OK;
}

}  // namespace

extern "C" int rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *gamma,
                                   const float *rstd, void *dx, float *dgamma, int64_t M, int64_t N,
                                   int dtype, gbnorm_stream_t stream) {
    // Shapes whose partial rows do not fit the fixed scratch are refused
    // before anything is enqueued (0 = invalid arguments: rmsnorm_bwd below
    // reports which).
    const size_t need = norm_bwd_workspace_size(0, M, N, dtype);
    if (need > kScratchBytes) return GBNORM_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int s = scratch_address(&scratch);
    if (s != GBNORM_OK) return s;
    // The kernels overwrite every partial-row entry they later read, so the
    // scratch needs no clearing between calls.
    return rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, scratch, kScratchBytes, M, N, dtype, stream);
}
