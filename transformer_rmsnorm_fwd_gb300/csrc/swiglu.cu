// SwiGLU activation forward and backward.
//
// Operator: the FusedLinearSwiGLU paragraph of the page "Liger-Kernel核心技术：
// RollingBuffer与融合算子详解", section "算子融合": SiLU of the gate branch
// times the up branch, computed in registers.  silu(g) = g * sigmoid(g); the
// backward is its derivative.
//
// GB300 design: purely HBM-bound (bf16: 6 bytes/element forward, 10 bytes
// backward).  16-byte vector loads/stores, two vectors in flight per thread
// per iteration, a persistent grid of (SMs x resident blocks) striding over
// the vectors, and evict-first stores for outputs nobody re-reads here.
// The backward never marks its pointers restrict and never uses the
// read-only path, so dgate == gate and dup == up (in place) are safe: each
// element is read and then written by the same thread.
#include "common.cuh"

namespace liger {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

// sigmoid: accurate exp / division for fp32 storage, the fast hardware
// exp2 / reciprocal for bf16 storage (its rounding dominates by far).
template <typename T> __device__ __forceinline__ float sigm(float g);
template <> __device__ __forceinline__ float sigm<float>(float g) { return 1.0f / (1.0f + expf(-g)); }
template <> __device__ __forceinline__ float sigm<__nv_bfloat16>(float g) {
    return __fdividef(1.0f, 1.0f + __expf(-g));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) swiglu_fwd_kernel(const T* gate, const T* up, T* y, int64_t n) {
    constexpr int EPV = Vec<T>::N;
    const int64_t nvec = n / EPV;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 g[kUnroll], u[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            g[k] = ldg16(gate + (i + k * stride) * EPV);
            u[k] = ldg16(up + (i + k * stride) * EPV);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            float fg[EPV], fu[EPV];
            unpack(g[k], fg);
            unpack(u[k], fu);
#pragma unroll
            for (int e = 0; e < EPV; ++e) fg[e] = fg[e] * sigm<T>(fg[e]) * fu[e];
            stg16_cs(y + (i + k * stride) * EPV, pack(fg));
        }
    }
    for (; i < nvec; i += stride) {
        float fg[EPV], fu[EPV];
        unpack(ldg16(gate + i * EPV), fg);
        unpack(ldg16(up + i * EPV), fu);
#pragma unroll
        for (int e = 0; e < EPV; ++e) fg[e] = fg[e] * sigm<T>(fg[e]) * fu[e];
        stg16_cs(y + i * EPV, pack(fg));
    }
    // tail elements (n not a multiple of the vector width)
    const int64_t t = nvec * EPV + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) {
        const float g = ldf(gate + t);
        stf(y + t, g * sigm<T>(g) * ldf(up + t));
    }
}

template <typename T>
__device__ __forceinline__ void swiglu_grad(float g, float u, float d, float& dg, float& du) {
    const float s = sigm<T>(g);
    du = d * (g * s);
    dg = d * u * s * (1.0f + g * (1.0f - s));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(const T* dy, const T* gate, const T* up, T* dgate,
                                                              T* dup, int64_t n) {
    constexpr int EPV = Vec<T>::N;
    const int64_t nvec = n / EPV;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 g[kUnroll], u[kUnroll], d[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int64_t o = (i + k * stride) * EPV;
            g[k] = ldg16(gate + o);
            u[k] = ldg16(up + o);
            d[k] = ldg16(dy + o);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            float fg[EPV], fu[EPV], fd[EPV], og[EPV], ou[EPV];
            unpack(g[k], fg);
            unpack(u[k], fu);
            unpack(d[k], fd);
#pragma unroll
            for (int e = 0; e < EPV; ++e) swiglu_grad<T>(fg[e], fu[e], fd[e], og[e], ou[e]);
            const int64_t o = (i + k * stride) * EPV;
            stg16_cs(dgate + o, pack(og));
            stg16_cs(dup + o, pack(ou));
        }
    }
    for (; i < nvec; i += stride) {
        float fg[EPV], fu[EPV], fd[EPV], og[EPV], ou[EPV];
        unpack(ldg16(gate + i * EPV), fg);
        unpack(ldg16(up + i * EPV), fu);
        unpack(ldg16(dy + i * EPV), fd);
#pragma unroll
        for (int e = 0; e < EPV; ++e) swiglu_grad<T>(fg[e], fu[e], fd[e], og[e], ou[e]);
        stg16_cs(dgate + i * EPV, pack(og));
        stg16_cs(dup + i * EPV, pack(ou));
    }
    const int64_t t = nvec * EPV + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) {
        float og, ou;
        swiglu_grad<T>(ldf(gate + t), ldf(up + t), ldf(dy + t), og, ou);
        stf(dgate + t, og);
        stf(dup + t, ou);
    }
}

template <typename K>
unsigned grid_for(K kern, int64_t n, int epv) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t need = std::max<int64_t>(1, ceil_div(ceil_div(n, epv), kThreads));
    return static_cast<unsigned>(std::min<int64_t>(need, static_cast<int64_t>(sm_count()) * per_sm));
}

int check(const void* const* ptrs, int np, int64_t n, int dtype, const char* who) {
    if (dtype != LIGER_F32 && dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "%s: dtype %d", who, dtype);
    if (n < 0) return fail(LIGER_ERR_SHAPE, "%s: n=%lld", who, (long long)n);
    if (n == 0) return LIGER_OK;
    for (int i = 0; i < np; ++i)
        if (!ptrs[i]) return fail(LIGER_ERR_NULL, "%s: null tensor pointer", who);
    for (int i = 0; i < np; ++i)
        if (!aligned16(ptrs[i])) return fail(LIGER_ERR_ALIGN, "%s: tensors must be 16-byte aligned", who);
    return LIGER_OK;
}

}  // namespace
}  // namespace liger

using namespace liger;

extern "C" int liger_swiglu_fwd(const void* gate, const void* up, void* y, int64_t n, int dtype, void* stream) {
    clear_error();
    const void* p[3] = {gate, up, y};
    if (int rc = check(p, 3, n, dtype, "swiglu_fwd")) return rc;
    if (n == 0) return LIGER_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == LIGER_F32) {
        swiglu_fwd_kernel<float><<<grid_for(swiglu_fwd_kernel<float>, n, 4), kThreads, 0, st>>>(
            static_cast<const float*>(gate), static_cast<const float*>(up), static_cast<float*>(y), n);
    } else {
        using B = __nv_bfloat16;
        swiglu_fwd_kernel<B><<<grid_for(swiglu_fwd_kernel<B>, n, 8), kThreads, 0, st>>>(
            static_cast<const B*>(gate), static_cast<const B*>(up), static_cast<B*>(y), n);
    }
    return check_launch("swiglu_fwd");
}

extern "C" int liger_swiglu_bwd(const void* dy, const void* gate, const void* up, void* dgate, void* dup, int64_t n,
                                int dtype, void* stream) {
    clear_error();
    const void* p[5] = {dy, gate, up, dgate, dup};
    if (int rc = check(p, 5, n, dtype, "swiglu_bwd")) return rc;
    if (n == 0) return LIGER_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == LIGER_F32) {
        swiglu_bwd_kernel<float><<<grid_for(swiglu_bwd_kernel<float>, n, 4), kThreads, 0, st>>>(
            static_cast<const float*>(dy), static_cast<const float*>(gate), static_cast<const float*>(up),
            static_cast<float*>(dgate), static_cast<float*>(dup), n);
    } else {
        using B = __nv_bfloat16;
        swiglu_bwd_kernel<B><<<grid_for(swiglu_bwd_kernel<B>, n, 8), kThreads, 0, st>>>(
            static_cast<const B*>(dy), static_cast<const B*>(gate), static_cast<const B*>(up), static_cast<B*>(dgate),
            static_cast<B*>(dup), n);
    }
    return check_launch("swiglu_bwd");
}
