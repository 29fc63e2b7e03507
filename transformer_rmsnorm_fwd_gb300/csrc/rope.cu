// RoPE forward / backward, in place on Q and K.
//
// Operator: the FusedRoPE paragraph of the page "Liger-Kernel核心技术：
// RollingBuffer与融合算子详解", section "算子融合" (the rotation angle comes
// from the token position, generated in the kernel, no stored table) and the
// RoPE step of the fused-kernel listing on the page "Liger-Kernel底层优化：
// 新一代内核级推理加速引擎介绍" (pairs (i, i + D/2)).  Frequency schedule
// theta^(-2i/D) (standard RoPE; the pages give none).
//
// GB300 design (HBM-bound: every element read and written once):
//  * one block per position s (and batch group): its D/2 angles are formed
//    once in shared memory and reused by every head of Q and K and, when the
//    positions are implicit (p = s), by every batch row -- 160x reuse at
//    Llama-3-8B shapes -- so the fp64 angle work is negligible;
//  * the inverse frequencies theta^(-2i/D) are computed on the host in
//    double precision and passed as a kernel parameter;
//  * angle phi = p * inv_freq in double, reduced modulo 2 pi in double
//    (two-term 2 pi), then sincosf on the reduced single-precision angle:
//    the result is accurate to ~1 ulp of fp32 at any position, where a plain
//    fp32 p * inv_freq would err by ~p ulp;
//  * each thread rotates 16-byte vectors of the two halves of a head; a warp
//    covers four heads with full 128-byte lines.
#include <math.h>

#include "common.cuh"

namespace liger {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxHalf = 256;   // head_dim <= 512
constexpr int kBatchGroup = 8;

struct InvFreq {
    double v[kMaxHalf];
};

__device__ __forceinline__ float2 angle_cs(double p, double inv_freq, float sign) {
    const double two_pi_hi = 6.283185307179586232;      // nearest double to 2 pi
    const double two_pi_lo = 2.4492935982947064e-16;    // 2 pi - two_pi_hi
    const double phi = p * inv_freq;
    const double k = rint(phi * 0.15915494309189535);   // 1 / (2 pi)
    double r = fma(-k, two_pi_hi, phi);
    r = fma(-k, two_pi_lo, r);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    return make_float2(c, sign * s);
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) rope_kernel(T* q, T* k, const int32_t* __restrict__ pos, int B, int S,
                                                        int Hq, int Hk, int D, const __grid_constant__ InvFreq f,
                                                        float sign) {
    extern __shared__ float2 cs[];   // [nb_angles][D/2] (cos, +-sin)
    const int half = D >> 1;
    const int s = blockIdx.x;
    const int b0 = blockIdx.y * kBatchGroup;
    const int nb = min(kBatchGroup, B - b0);
    const int na = pos ? nb : 1;     // distinct angle rows in this block
    for (int t = threadIdx.x; t < na * half; t += kThreads) {
        const int bl = t / half, i = t - bl * half;
        const double p = pos ? static_cast<double>(pos[static_cast<int64_t>(b0 + bl) * S + s]) : static_cast<double>(s);
        cs[t] = angle_cs(p, f.v[i], sign);
    }
    __syncthreads();
    const int H = Hq + Hk;
    if (VEC) {
        constexpr int EPV = Vec<T>::N;
        const int vph = half / EPV;                 // vectors per half head
        const int ntask = nb * H * vph;
        for (int t = threadIdx.x; t < ntask; t += kThreads) {
            const int bl = t / (H * vph);
            const int rem = t - bl * H * vph;
            const int h = rem / vph, v = rem - h * vph;
            const int64_t bs = static_cast<int64_t>(b0 + bl) * S + s;
            T* base = h < Hq ? q + (bs * Hq + h) * D : k + (bs * Hk + (h - Hq)) * D;
            T* pa = base + v * EPV;
            T* pb = pa + half;
            float a[EPV], bv[EPV];
            unpack(ldg16(pa), a);
            unpack(ldg16(pb), bv);
            const float2* c = cs + (pos ? bl : 0) * half + v * EPV;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const float2 r = c[e];
                const float x0 = a[e], x1 = bv[e];
                a[e] = x0 * r.x - x1 * r.y;
                bv[e] = x1 * r.x + x0 * r.y;
            }
            stg16(pa, pack(a));
            stg16(pb, pack(bv));
        }
    } else {
        const int ntask = nb * H * half;
        for (int t = threadIdx.x; t < ntask; t += kThreads) {
            const int bl = t / (H * half);
            const int rem = t - bl * H * half;
            const int h = rem / half, i = rem - h * half;
            const int64_t bs = static_cast<int64_t>(b0 + bl) * S + s;
            T* base = h < Hq ? q + (bs * Hq + h) * D : k + (bs * Hk + (h - Hq)) * D;
            const float2 r = cs[(pos ? bl : 0) * half + i];
            const float x0 = ldf(base + i), x1 = ldf(base + i + half);
            stf(base + i, x0 * r.x - x1 * r.y);
            stf(base + i + half, x1 * r.x + x0 * r.y);
        }
    }
}

int rope_run(void* q, void* k, const int32_t* pos, int64_t B, int64_t S, int64_t Hq, int64_t Hk, int64_t D,
             double theta, int dtype, void* stream, float sign, const char* who) {
    clear_error();
    if (dtype != LIGER_F32 && dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "%s: dtype %d", who, dtype);
    if (B < 0 || S < 0 || Hq < 0 || Hk < 0 || D <= 0 || (D & 1) || D > 2 * kMaxHalf || S > 2147483647LL ||
        B > 2147483647LL || Hq + Hk > (1 << 20))
        return fail(LIGER_ERR_SHAPE, "%s: batch=%lld seq=%lld heads=%lld/%lld head_dim=%lld (even, <= %d)", who,
                    (long long)B, (long long)S, (long long)Hq, (long long)Hk, (long long)D, 2 * kMaxHalf);
    if (!(theta > 0.0) || !isfinite(theta)) return fail(LIGER_ERR_SHAPE, "%s: theta must be > 0", who);
    if (B == 0 || S == 0 || Hq + Hk == 0) return LIGER_OK;
    if ((Hq > 0 && !q) || (Hk > 0 && !k)) return fail(LIGER_ERR_NULL, "%s: q/k required for nonzero head counts", who);
    if ((q && !aligned16(q)) || (k && !aligned16(k)))
        return fail(LIGER_ERR_ALIGN, "%s: q and k must be 16-byte aligned", who);
    if (pos && (reinterpret_cast<uintptr_t>(pos) & 3)) return fail(LIGER_ERR_ALIGN, "%s: pos must be 4-byte aligned", who);
    const int half = static_cast<int>(D / 2);
    InvFreq f;
    for (int i = 0; i < half; ++i) f.v[i] = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
    const int nbg = static_cast<int>(ceil_div(B, kBatchGroup));
    if (nbg > 65535) return fail(LIGER_ERR_SHAPE, "%s: batch too large", who);
    dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(nbg));
    const size_t smem = static_cast<size_t>(pos ? kBatchGroup : 1) * half * sizeof(float2);
    cudaStream_t st = as_stream(stream);
    const int epv = dtype == LIGER_F32 ? 4 : 8;
    const bool vec = (half % epv) == 0;
    if (dtype == LIGER_F32) {
        auto kern = vec ? rope_kernel<float, true> : rope_kernel<float, false>;
        kern<<<grid, kThreads, smem, st>>>(static_cast<float*>(q), static_cast<float*>(k), pos, (int)B, (int)S, (int)Hq,
                                           (int)Hk, (int)D, f, sign);
    } else {
        using Bf = __nv_bfloat16;
        auto kern = vec ? rope_kernel<Bf, true> : rope_kernel<Bf, false>;
        kern<<<grid, kThreads, smem, st>>>(static_cast<Bf*>(q), static_cast<Bf*>(k), pos, (int)B, (int)S, (int)Hq,
                                           (int)Hk, (int)D, f, sign);
    }
    return check_launch(who);
}

}  // namespace
}  // namespace liger

extern "C" int liger_rope_fwd(void* q, void* k, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                              int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream) {
    return liger::rope_run(q, k, pos, batch, seq, n_q_heads, n_k_heads, head_dim, theta, dtype, stream, 1.0f,
                           "rope_fwd");
}

extern "C" int liger_rope_bwd(void* dq, void* dk, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                              int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream) {
    return liger::rope_run(dq, dk, pos, batch, seq, n_q_heads, n_k_heads, head_dim, theta, dtype, stream, -1.0f,
                           "rope_bwd");
}
