// Per-thread error message and device-property caches of libliger.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

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

// ------------------------------------------------------ device status
// The library-owned error words, read and cleared on the caller's stream by
// one thread (atomic exchange), the values landing in g_taken for the copy
// back to the host.
constexpr int kWords = 4;
static const char* const kFamily[kWords] = {"RMSNorm (staged kernels)", "FusedLinearSwiGLU",
                                            "fused RMSNorm+QKV+RoPE", "RoPE (staged kernel)"};

struct Words {
    int* w[kWords];
};

static __device__ int g_taken[kWords];

__global__ void take_error_words(Words w) {
    for (int i = 0; i < kWords; ++i) g_taken[i] = atomicExch(w.w[i], 0);
}

__global__ void set_error_word(int* a) { atomicExch(a, 1); }

static std::mutex g_status_mu;   // one g_taken per device: one reader at a time

static int error_words(Words& w) {
    if (int rc = rmsnorm_err_word(&w.w[0])) return rc;
    if (int rc = lsw_err_word(&w.w[1])) return rc;
    if (int rc = qkv_err_word(&w.w[2])) return rc;
    return rope_err_word(&w.w[3]);
}

}  // namespace liger

extern "C" const char* liger_last_error(void) { return liger::g_msg; }

extern "C" int liger_device_status(void* stream) {
    using namespace liger;
    clear_error();
    Words w;
    if (int rc = error_words(w)) return rc;
    cudaStream_t st = as_stream(stream);
    int h[kWords] = {0};
    {
        std::lock_guard<std::mutex> lock(g_status_mu);
        take_error_words<<<1, 1, 0, st>>>(w);
        if (int rc = check_launch("device_status")) return rc;
        cudaError_t e = cudaMemcpyFromSymbolAsync(h, g_taken, sizeof(h), 0, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return fail(LIGER_ERR_CUDA, "device_status: %s", cudaGetErrorString(e));
    }
    char names[256] = "";
    size_t n = 0;
    for (int i = 0; i < kWords; ++i)
        if (h[i]) n += snprintf(names + n, sizeof(names) - n, "%s%s", n ? ", " : "", kFamily[i]);
    if (n) return fail(LIGER_ERR_CUDA, "a bounded wait expired in: %s; the outputs of that call are incomplete", names);
    return LIGER_OK;
}

extern "C" int liger_device_status_mark(int which, void* stream) {
    using namespace liger;
    clear_error();
    if (which < 0 || which >= kWords)
        return fail(LIGER_ERR_SHAPE, "device_status_mark: which=%d (0 to %d)", which, kWords - 1);
    Words w;
    if (int rc = error_words(w)) return rc;
    set_error_word<<<1, 1, 0, as_stream(stream)>>>(w.w[which]);
    return check_launch("device_status_mark");
}
