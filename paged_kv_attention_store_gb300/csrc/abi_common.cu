// Host-side pieces shared by the entry points: status names and the cached SM count.
#include <mutex>

#include "nv_common.cuh"

namespace nvkv_host {

int sm_count()
{
    static std::mutex mu;
    static int cached[64];
    static bool have[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && have[dev])
        return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (dev < 64) {
        cached[dev] = n;
        have[dev] = true;
    }
    return n;
}

}  // namespace nvkv_host

extern "C" const char *nv_status_string(int status)
{
    switch (status) {
    case NV_OK: return "NV_OK";
    case NV_ERR_NULL: return "NV_ERR_NULL: a required pointer is NULL";
    case NV_ERR_SHAPE: return "NV_ERR_SHAPE: a size is negative or inconsistent";
    case NV_ERR_ALIGN: return "NV_ERR_ALIGN: a pointer or stride breaks the 16-byte rule";
    case NV_ERR_UNSUPPORTED: return "NV_ERR_UNSUPPORTED: shape outside what the kernels implement";
    case NV_ERR_WORKSPACE: return "NV_ERR_WORKSPACE: workspace missing or too small";
    case NV_ERR_CUDA: return "NV_ERR_CUDA: the CUDA runtime reported an error";
    default: return "unknown nv_status";
    }
}
