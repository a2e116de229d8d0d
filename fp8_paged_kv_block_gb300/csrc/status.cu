// status.cu -- status codes, per-thread error text, device queries.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace {
thread_local char g_last_error[512] = "";
}

extern "C" const char* pa_status_string(pa_status status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULLPTR: return "PA_ERR_NULLPTR: a required pointer is NULL";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid shape, size, layout or dtype";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call or kernel launch failed";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: configuration not built";
    }
    return "unknown pa_status";
}

extern "C" const char* pa_last_error(void) { return g_last_error; }

namespace pa {

pa_status fail(pa_status st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

pa_status check_launch(const char* what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return PA_OK;
}

// SM count of the current device (cached per device id).
int device_sm_count()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace pa
