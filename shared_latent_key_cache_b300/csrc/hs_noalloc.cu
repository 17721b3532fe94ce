// hs_noalloc.cu -- li_hs_select_noalloc: hierarchical selection whose scratch
// memory is a fixed array owned by this library instead of a workspace the
// caller allocates.
//
// Some callers cannot allocate device memory at the point where they run the
// indexer: a plugin inside a serving engine whose device memory is owned by
// the engine's own pool, or a latency-critical decode loop that must not pay
// for cudaMalloc (which can synchronise the device).  For them this entry point
// uses `g_hs_scratch`, a file-scope device array of kHsScratchBytes that every
// GPU loading the library holds until the process exits, and allocates
// nothing.
//
// The host cannot pass `g_hs_scratch` to a kernel by name: in host code that
// name is a host-side stand-in, not a device address.  The device address is
// looked up once per device with cudaGetSymbolAddress (on the first call made
// while that device is current) and cached.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "li_internal.cuh"

namespace li {
namespace {

constexpr size_t kHsScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr int kMaxDev = 64;

static __device__ __align__(256) unsigned char g_hs_scratch[kHsScratchBytes];

std::atomic<void *> g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of g_hs_scratch on the current device (nullptr on failure).
void *hs_scratch_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return nullptr;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p != nullptr)
        return p;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_hs_scratch) != cudaSuccess || addr == nullptr)
            return nullptr;
        g_scratch_addr[dev].store(addr, std::memory_order_release);
        p = addr;
    }
    return p;
}

} // namespace
} // namespace li

extern "C" {

int li_hs_select_noalloc(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                         int abs_t, const float *q_abs_scale, const float *w, const float *beta,
                         int B, int G, int H, int r, int L, int m, int k, int32_t *cand,
                         int32_t *idx, void *stream)
{
    // the same argument checks as li_hs_select first, without touching CUDA, so
    // that both entry points report the same status for the same bad call;
    // only then the size limit of the built-in scratch
    const int st = li::hs_check_args(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, B,
                                     G, H, r, L, m, k, cand, idx);
    if (st != LI_OK)
        return st;
    const size_t need = li_hs_workspace_size(B, G, L, m, k);
    if (need == 0)
        return LI_ERR_INVALID_ARG;
    if (need > li::kHsScratchBytes)
        return LI_ERR_WORKSPACE;     // these sizes need more scratch than the built-in array holds
    void *ws = li::hs_scratch_ptr();
    if (ws == nullptr)
        return LI_ERR_CUDA;
    return li_hs_select(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, B, G, H, r, L,
                        m, k, cand, idx, ws, li::kHsScratchBytes, stream);
}

} // extern "C"
