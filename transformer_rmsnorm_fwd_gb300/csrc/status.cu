// Per-thread error message and device-property caches of libliger.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>

#include "common.cuh"

namespace liger {

static thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_msg[0] = '\0'; }

int check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(LIGER_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return LIGER_OK;
}

static constexpr int kMaxDev = 64;
// 0 = not yet read; racing threads store the same value
static std::atomic<int> g_sms[kMaxDev];
static std::atomic<int> g_smem[kMaxDev];

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev >= kMaxDev) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 148;
    }
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        g_sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int max_smem_optin() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    int v = g_smem[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) v = 0;
        g_smem[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace liger

extern "C" const char* liger_last_error(void) { return liger::g_msg; }
