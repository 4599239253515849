// scan_static.cu -- sdm_scan_noalloc: the recurrence with its scratch in a fixed
// device array that the library owns, for callers that cannot allocate device memory.
//
// Some hosts give this code no way to allocate: a plugin inside an application that
// owns all device memory through its own pool or budget, or a latency-critical loop
// where cudaMalloc/cudaFree would synchronise the device and stall other work. For
// them this entry point keeps the scan's scratch (the collision codes, the forwarding
// masks and the per-token progress flags of the row blocks: the minimal scan workspace,
// sdm_scan_min_workspace_bytes; the forwarding ring too when the whole workspace fits)
// in g_scan_scratch below, a file-scope device array of SDM_SCAN_NOALLOC_MAX_BYTES that
// every GPU loading the library holds until exit.
//
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; that first call
// should come before any stream capture. The cached address is not looked up again,
// so it is stale after a cudaDeviceReset of that device (documented in the header). The array is shared by every call: each call
// rewrites the codes it uses and clears the flags it uses (cudaMemsetAsync on the
// caller's stream) before reading them, and calls whose work overlaps on the GPU race
// on it.
#include <cuda_runtime.h>

#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

static __device__ __align__(256) unsigned char g_scan_scratch[SDM_SCAN_NOALLOC_MAX_BYTES];

// Device address of g_scan_scratch on the current device (looked up once per device).
static int static_scratch(void** out)
{
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SDM_ECUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scan_scratch) != cudaSuccess || p == nullptr)
            return SDM_ECUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return SDM_OK;
}

}  // namespace sdm

extern "C" int sdm_scan_noalloc(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                                const void* v, const float* alpha, const float* beta,
                                void* banks, float* y, int B, int T, int* dev_status,
                                void* stream)
{
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    const size_t need = sdm_scan_min_workspace_bytes(cfg, B, T);
    if (need == 0)  // the shape itself is not accepted: report why
        return sdm_scan(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, nullptr, 0, dev_status,
                        stream);
    if (need > (size_t)SDM_SCAN_NOALLOC_MAX_BYTES)
        return SDM_EWORKSPACE;
    if (B == 0 || T == 0)
        return SDM_OK;
    void* ws = nullptr;
    const int rc = sdm::static_scratch(&ws);
    if (rc != SDM_OK)
        return rc;
    return sdm_scan(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws,
                    (size_t)SDM_SCAN_NOALLOC_MAX_BYTES, dev_status, stream);
}
