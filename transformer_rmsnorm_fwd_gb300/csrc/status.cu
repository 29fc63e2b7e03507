// Per-thread error message and device-property caches of libliger.
#include <stdarg.h>
#include <stdio.h>

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
static int g_sms[kMaxDev] = {0};
static int g_smem[kMaxDev] = {0};

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev >= kMaxDev) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 148;
    }
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

int max_smem_optin() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (g_smem[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) n = 0;
        g_smem[dev] = n;
    }
    return g_smem[dev];
}

}  // namespace liger

extern "C" const char* liger_last_error(void) { return liger::g_msg; }
