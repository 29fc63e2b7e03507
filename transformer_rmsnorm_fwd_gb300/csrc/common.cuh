// Shared helpers of libliger: status handling, 16-byte vector access for
// fp32 / bf16 storage, and launch sizing for the GB300 SM count.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "liger.h"

namespace liger {

// ---------------------------------------------------------------- status
// Records a message for liger_last_error() and returns the code.
int fail(int code, const char* fmt, ...);
void clear_error();
// Maps a pending launch error (cudaGetLastError) to LIGER_ERR_CUDA.
int check_launch(const char* what);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device addresses (current device) of the library-owned words in which kernels
// without a per-call workspace header record an expired bounded wait: the staged
// RMSNorm kernels, FusedLinearSwiGLU's GEMMs, the fused QKV GEMM and the staged
// RoPE kernel.
int rmsnorm_err_word(int** out);
int lsw_err_word(int** out);
int qkv_err_word(int** out);
int rope_err_word(int** out);

// SM count of the current device (cached per device).
int sm_count();
// Maximum dynamic shared memory per block (opt-in) of the current device.
int max_smem_optin();

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ------------------------------------------------------- vector storage
// A 16-byte vector holds 4 fp32 or 8 bf16 elements.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
};

__device__ __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
    f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
    f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}
// The same as pairs, for the packed fp32x2 arithmetic (__ffma2_rn, __fmul2_rn)
__device__ __forceinline__ void unpack2(const uint4& u, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}
__device__ __forceinline__ void unpack2(const uint4& u, float2 (&f)[4]) {
    f[0] = make_float2(bf_lo(u.x), bf_hi(u.x));
    f[1] = make_float2(bf_lo(u.y), bf_hi(u.y));
    f[2] = make_float2(bf_lo(u.z), bf_hi(u.z));
    f[3] = make_float2(bf_lo(u.w), bf_hi(u.w));
}
// round-to-nearest-even pair -> packed bf16x2 (low half = first element)
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack2(const float2 (&f)[2]) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
}
__device__ __forceinline__ uint4 pack2(const float2 (&f)[4]) {
    return make_uint4(pack_bf2(f[0].x, f[0].y), pack_bf2(f[1].x, f[1].y), pack_bf2(f[2].x, f[2].y),
                      pack_bf2(f[3].x, f[3].y));
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7]));
}

// scalar access
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// 16-byte loads / stores.  ldg_nc: read-only path, only for buffers no
// thread of the same kernel writes.
__device__ __forceinline__ uint4 ldg16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
// 16-byte load asking L2 to fetch the whole 256-byte block around it from DRAM
// (for a thread whose next load falls in the same 256 bytes)
__device__ __forceinline__ uint4 ldg16_pf256(const void* p) {
    uint4 r;
    asm volatile("ld.global.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}
__device__ __forceinline__ uint4 ldg16_nc(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void stg16(void* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }
// 16 bytes of quiet NaNs in the storage type (written where a kernel gave up)
template <typename T> __device__ __forceinline__ uint4 nan16();
template <> __device__ __forceinline__ uint4 nan16<float>() { return make_uint4(0x7FC00000u, 0x7FC00000u, 0x7FC00000u, 0x7FC00000u); }
template <> __device__ __forceinline__ uint4 nan16<__nv_bfloat16>() { return make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u); }
// streaming load (evict-first): data read once by this kernel
__device__ __forceinline__ uint4 ldg16_cs(const void* p) {
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
// streaming store (evict-first): output that is not re-read by this kernel
__device__ __forceinline__ void stg16_cs(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace liger
