// RMSNorm forward and backward.
//
// Operator: the RMSNorm step of the fused RMSNorm + QKV + RoPE kernel on the
// page "Liger-Kernel底层优化：新一代内核级推理加速引擎介绍", section
// "融合内核是如何工作的？来看一段简化版实现": rstd = 1/sqrt(mean(x^2) + eps),
// y = x * rstd * w.  The backward is the derivative of that forward.
//
// GB300 design (HBM-bound, ~2 bytes/element each way in bf16):
//  * forward (rows of whole 16-byte vectors that fit the ring): one warp per
//    row, each warp a ring of row buffers in shared memory filled by 1-D bulk
//    copies (cp.async.bulk, completion on an mbarrier), so several rows per
//    warp are in flight without registers; one warp-shuffle reduction, no
//    block barrier.  Other widths: the row held in registers (warp per row)
//    or a block per row.
//  * backward (the same rows): a persistent block per contiguous group of
//    rows, its (dy, x) rows brought into a ring of 6 buffers by bulk copies;
//    each thread owns fixed 16-byte column vectors and keeps its share of dw
//    in fp32 registers across the group's rows (no atomics); the dot products
//    of two rows are reduced together (shuffles, one block barrier), then the
//    two rows are read again from shared memory for dx (and, in fp32, dw); in
//    bf16 the products come straight from the packed words through the
//    mixed-precision fma (exact, so no widening instructions for dy and w)
//    and dw is summed before the barrier; the other float arithmetic runs on
//    column pairs with the packed fp32x2 instructions.
//    Other widths: the row in registers, or a generic loop.
//  * dw: per-block partial rows (workspace) summed by a second kernel in a
//    fixed order, so dw is deterministic.
#include <atomic>

#include "common.cuh"
#include "mbarrier.cuh"

namespace liger {
namespace {

constexpr int kFwdThreads = 256;
constexpr int kMaxPartials = 1024;

template <typename T, int VPL>
__global__ void __launch_bounds__(kFwdThreads, 2) rmsnorm_fwd_warp(const T* x, const T* __restrict__ w, T* y,
                                                                 float* __restrict__ rstd, int64_t rows, int cols,
                                                                 float eps) {
    constexpr int EPV = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int nvec = cols / EPV;
    const float inv_cols = 1.0f / static_cast<float>(cols);
    for (int64_t r = warp0; r < rows; r += nwarps) {
        const T* xr = x + r * cols;
        uint4 xv[VPL];   // the row stays packed in registers: 4 registers per 16-byte vector
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = j * 32 + lane;
            xv[j] = v < nvec ? ldg16(xr + static_cast<int64_t>(v) * EPV) : make_uint4(0, 0, 0, 0);
        }
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            float f[EPV];
            unpack(xv[j], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss = fmaf(f[e], f[e], ss);
        }
        ss = warp_sum(ss);
        const float rs = 1.0f / sqrtf(ss * inv_cols + eps);
        T* yr = y + r * cols;
        // w is re-read per row through L1 (every warp of the SM reads the same
        // cols elements), which keeps it out of the register budget
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = j * 32 + lane;
            if (v < nvec) {
                float f[EPV], g[EPV];
                unpack(xv[j], f);
                unpack(ldg16_nc(w + static_cast<int64_t>(v) * EPV), g);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = (f[e] * rs) * g[e];
                stg16(yr + static_cast<int64_t>(v) * EPV, pack(f));
            }
        }
        if (rstd != nullptr && lane == 0) rstd[r] = rs;
    }
}

// Any cols (scalar, two passes over the row): one block per row.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_fwd_generic(const T* x, const T* __restrict__ w, T* y,
                                                           float* __restrict__ rstd, int64_t rows, int cols,
                                                           float eps) {
    __shared__ float red[32];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const T* xr = x + r * cols;
        float ss = 0.f;
        for (int j = threadIdx.x; j < cols; j += blockDim.x) {
            const float f = ldf(xr + j);
            ss = fmaf(f, f, ss);
        }
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        const float rs = 1.0f / sqrtf(tot / static_cast<float>(cols) + eps);
        T* yr = y + r * cols;
        for (int j = threadIdx.x; j < cols; j += blockDim.x) stf(yr + j, (ldf(xr + j) * rs) * ldf(w + j));
        if (rstd != nullptr && threadIdx.x == 0) rstd[r] = rs;
        __syncthreads();
    }
}

// ------------------------------------------------------------------ bwd
template <typename T, int VPT>
__global__ void __launch_bounds__(256) rmsnorm_bwd_block(const T* dy, const T* __restrict__ x,
                                                         const T* __restrict__ w, const float* __restrict__ rstd,
                                                         T* dx, float* __restrict__ part, int64_t rows, int cols,
                                                         int64_t rows_per_block) {
    constexpr int EPV = Vec<T>::N;
    __shared__ float red[2][32];
    const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, wid = tid >> 5, NW = NT >> 5;
    const int nvec = cols / EPV;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per_block;
    const int64_t r1 = min(rows, r0 + rows_per_block);
    uint4 wv[VPT];
    float dwa[VPT][EPV];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = j * NT + tid;
        wv[j] = v < nvec ? ldg16_nc(w + static_cast<int64_t>(v) * EPV) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < EPV; ++e) dwa[j][e] = 0.f;
    }
    const float inv_cols = 1.0f / static_cast<float>(cols);
    uint4 nx[VPT], ndy[VPT];
    float nrs = 0.f;
    auto fetch = [&](int64_t r) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * NT + tid;
            const int64_t off = r * cols + static_cast<int64_t>(v) * EPV;
            nx[j] = v < nvec ? ldg16(x + off) : make_uint4(0, 0, 0, 0);
            ndy[j] = v < nvec ? ldg16(dy + off) : make_uint4(0, 0, 0, 0);
        }
        nrs = rstd[r];
    };
    if (r0 < r1) fetch(r0);
    for (int64_t r = r0; r < r1; ++r) {
        uint4 cx[VPT], cdy[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            cx[j] = nx[j];
            cdy[j] = ndy[j];
        }
        const float rs = nrs;
        if (r + 1 < r1) fetch(r + 1);
        float gx = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float fx[EPV], fd[EPV], fw[EPV];
            unpack(cx[j], fx);
            unpack(cdy[j], fd);
            unpack(wv[j], fw);
#pragma unroll
            for (int e = 0; e < EPV; ++e) gx = fmaf(fd[e] * fw[e], fx[e], gx);
        }
        gx = warp_sum(gx);
        if (lane == 0) red[r & 1][wid] = gx;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < NW; ++i) tot += red[r & 1][i];
        const float c = rs * rs * rs * inv_cols * tot;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * NT + tid;
            if (v < nvec) {
                float fx[EPV], fd[EPV], fw[EPV], o[EPV];
                unpack(cx[j], fx);
                unpack(cdy[j], fd);
                unpack(wv[j], fw);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    o[e] = rs * (fd[e] * fw[e]) - c * fx[e];
                    dwa[j][e] = fmaf(fd[e] * fx[e], rs, dwa[j][e]);
                }
                stg16(dx + r * cols + static_cast<int64_t>(v) * EPV, pack(o));
            }
        }
    }
    float* pr = part + static_cast<int64_t>(blockIdx.x) * cols;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = j * NT + tid;
        if (v < nvec) {
#pragma unroll
            for (int e = 0; e < EPV; e += 4) {
                float q[4] = {dwa[j][e], dwa[j][e + 1], dwa[j][e + 2], dwa[j][e + 3]};
                stg16(pr + static_cast<int64_t>(v) * EPV + e, pack(q));
            }
        }
    }
}

// Any cols (scalar): one block per row group, partial dw accumulated in the
// block's own workspace row (no other block touches it).
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_bwd_generic(const T* dy, const T* __restrict__ x,
                                                           const T* __restrict__ w, const float* __restrict__ rstd,
                                                           T* dx, float* __restrict__ part, int64_t rows, int cols,
                                                           int64_t rows_per_block) {
    __shared__ float red[32];
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per_block;
    const int64_t r1 = min(rows, r0 + rows_per_block);
    float* pr = part + static_cast<int64_t>(blockIdx.x) * cols;
    for (int j = threadIdx.x; j < cols; j += blockDim.x) pr[j] = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        const float rs = rstd[r];
        float gx = 0.f;
        for (int j = threadIdx.x; j < cols; j += blockDim.x)
            gx = fmaf(ldf(dy + r * cols + j) * ldf(w + j), ldf(x + r * cols + j), gx);
        gx = warp_sum(gx);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = gx;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        const float c = rs * rs * rs / static_cast<float>(cols) * tot;
        for (int j = threadIdx.x; j < cols; j += blockDim.x) {
            const float fx = ldf(x + r * cols + j), fd = ldf(dy + r * cols + j);
            stf(dx + r * cols + j, rs * (fd * ldf(w + j)) - c * fx);
            pr[j] = fmaf(fd * fx, rs, pr[j]);
        }
        __syncthreads();
    }
}

// dw[j] = sum_b part[b, j] in ascending b: 8 slices of the partial rows per
// 32 columns, combined in slice order.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_dw_reduce(const float* __restrict__ part, T* __restrict__ dw,
                                                         int nparts, int cols) {
    __shared__ float red[8][33];
    const int cl = threadIdx.x & 31, sl = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + cl;
    const int per = (nparts + 7) / 8;
    const int b0 = sl * per, b1 = min(nparts, b0 + per);
    float s = 0.f;
    if (col < cols)
        for (int b = b0; b < b1; ++b) s += part[static_cast<int64_t>(b) * cols + col];
    red[sl][cl] = s;
    __syncthreads();
    if (sl == 0 && col < cols) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += red[i][cl];
        stf(dw + col, t);
    }
}

// The same sum for rows of a multiple of 4 columns, 4 columns per thread:
// block of 32 warps over 128 columns, warp w summing the partial rows w, w +
// 32, ... in ascending order, the 32 slice sums then combined in slice order
// (deterministic for a given number of partial rows).  Many independent
// 16-byte loads per SM instead of one 4-byte chain per thread.
template <typename T>
__global__ void __launch_bounds__(1024) rmsnorm_dw_reduce4(const float* __restrict__ part, T* __restrict__ dw,
                                                           int nparts, int cols) {
    __shared__ float4 red[32][32];
    const int lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
    const int n4 = cols >> 2;
    const int c4 = blockIdx.x * 32 + lane;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < n4) {
        const float4* p = reinterpret_cast<const float4*>(part) + c4;
#pragma unroll 4
        for (int b = sl; b < nparts; b += 32) {
            const float4 v = p[static_cast<int64_t>(b) * n4];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
    }
    red[sl][lane] = s;
    __syncthreads();
    if (sl == 0 && c4 < n4) {
        float4 t = red[0][lane];
        for (int i = 1; i < 32; ++i) {
            const float4 v = red[i][lane];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        T* o = dw + static_cast<int64_t>(c4) * 4;
        stf(o, t.x);
        stf(o + 1, t.y);
        stf(o + 2, t.z);
        stf(o + 3, t.w);
    }
}

// dw from nparts partial rows, with the 4-column form where the rows allow it.
template <typename T>
void launch_dw_reduce(const float* part, T* dw, int nparts, int cols, cudaStream_t st) {
    if (cols % 4 == 0)
        rmsnorm_dw_reduce4<T><<<static_cast<unsigned>(ceil_div(cols / 4, 32)), 1024, 0, st>>>(part, dw, nparts, cols);
    else
        rmsnorm_dw_reduce<T><<<static_cast<unsigned>(ceil_div(cols, 32)), 256, 0, st>>>(part, dw, nparts, cols);
}

// ------------------------------------------------- rows staged by bulk copy
// Rows travel HBM -> shared memory by 1-D bulk copies (cp.async.bulk) into a
// ring of `nst` buffers per warp (forward) or per block (backward), so that
// several rows per warp are in flight without holding them in registers.
// Every wait is bounded; on expiry the kernel records it in g_stage_err
// (read back and cleared by liger_device_status), waits (bounded) for the
// copies it issued, writes NaN into the outputs it did not finish (the
// forward's remaining rows of y and rstd; the backward's remaining rows of dx
// and its partial row of dw, so that dw is NaN) and stops.
static __device__ int g_stage_err;

struct Stage {
    uint8_t* base;     // shared buffers
    uint32_t bar0;     // first mbarrier (8 bytes each)
};

template <typename T>
__global__ void rmsnorm_fwd_staged(const T* x, const T* __restrict__ w, T* y, float* __restrict__ rstd,
                                   int64_t rows, int cols, float eps, int nst) {
    constexpr int EPV = Vec<T>::N;
    extern __shared__ __align__(128) uint8_t sm[];
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rb = static_cast<uint32_t>(cols) * sizeof(T);      // row bytes (multiple of 16)
    const int nvec = cols / EPV;
    uint8_t* wbuf = sm;
    uint8_t* ring = sm + rb + static_cast<size_t>(warp) * nst * rb;
    const uint32_t bars = smem_u32(sm + static_cast<size_t>(rb) * (1 + nw * nst));
    const uint32_t wbar = bars + 8u * nw * nst;
    const uint32_t mybar = bars + 8u * warp * nst;
    if (lane == 0)
        for (int s = 0; s < nst; ++s) mbar_init(mybar + 8u * s, 1);
    if (threadIdx.x == 0) mbar_init(wbar, 1);
    mbar_init_fence();
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_expect_tx(wbar, rb);
        bulk_g2s(smem_u32(wbuf), w, rb, wbar);
    }
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nw + warp;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * nw;
    if (lane == 0)
        for (int s = 0; s < nst; ++s) {
            const int64_t r = gw + s * stride;
            if (r < rows) {
                mbar_expect_tx(mybar + 8u * s, rb);
                bulk_g2s(smem_u32(ring + s * rb), x + r * cols, rb, mybar + 8u * s);
            }
        }
    bool ok = __all_sync(0xffffffffu, mbar_wait(wbar, 0));
    const float inv_cols = 1.0f / static_cast<float>(cols);
    int it = 0;
    int s = 0;          // it % nst, kept without a division (nst is a runtime value)
    uint32_t ph = 0;    // (it / nst) & 1
    int64_t r = gw;
    for (; ok && r < rows; r += stride, ++it) {
        if (!__all_sync(0xffffffffu, mbar_wait(mybar + 8u * s, ph))) {
            ok = false;
            break;
        }
        const uint8_t* xb = ring + s * rb;
        float ss = 0.f;
        for (int v = lane; v < nvec; v += 32) {
            float f[EPV];
            unpack(*reinterpret_cast<const uint4*>(xb + v * 16), f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss = fmaf(f[e], f[e], ss);
        }
        ss = warp_sum(ss);
        const float rs = 1.0f / sqrtf(ss * inv_cols + eps);
        T* yr = y + r * cols;
        for (int v = lane; v < nvec; v += 32) {
            float f[EPV], g[EPV];
            unpack(*reinterpret_cast<const uint4*>(xb + v * 16), f);
            unpack(*reinterpret_cast<const uint4*>(wbuf + v * 16), g);
#pragma unroll
            for (int e = 0; e < EPV; ++e) f[e] = (f[e] * rs) * g[e];
            stg16(yr + static_cast<int64_t>(v) * EPV, pack(f));
        }
        if (rstd != nullptr && lane == 0) rstd[r] = rs;
        __syncwarp();
        if (lane == 0) {
            const int64_t rn = r + nst * stride;
            if (rn < rows) {
                fence_proxy_async_smem();   // the reads above happen before the copy overwrites the buffer
                mbar_expect_tx(mybar + 8u * s, rb);
                bulk_g2s(smem_u32(ring + s * rb), x + rn * cols, rb, mybar + 8u * s);
            }
        }
        if (++s == nst) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (!ok) {
        if (lane == 0) {
            atomicExch(&g_stage_err, 1);
            // copies already issued into this warp's ring: the next phase of each buffer
            for (int sb = 0; sb < nst; ++sb) {
                const int64_t first = static_cast<int64_t>(it) + ((sb - it % nst) + nst) % nst;  // next use of buffer sb
                if (gw + first * stride < rows) mbar_wait(mybar + 8u * sb, static_cast<uint32_t>(first / nst) & 1u);
            }
        }
        // the rows this warp did not finish: NaN
        for (; r < rows; r += stride) {
            for (int v = lane; v < nvec; v += 32) stg16(y + r * cols + static_cast<int64_t>(v) * EPV, nan16<T>());
            if (rstd != nullptr && lane == 0) rstd[r] = __int_as_float(0x7FC00000);
        }
    }
}

// Shared memory of the staged forward for nw warps and nst buffers per warp.
inline size_t fwd_staged_smem(int rb, int nw, int nst) {
    return static_cast<size_t>(rb) * (1 + nw * nst) + 8u * (nw * nst + 1);
}

template <typename T>
int launch_fwd(const void* x, const void* w, void* y, float* rstd, int64_t rows, int cols, float eps,
               cudaStream_t st) {
    constexpr int EPV = Vec<T>::N;
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* yp = static_cast<T*>(y);
    const int sms = sm_count();
    if (cols % EPV == 0) {
        // staged path: 8 (or fewer) warps per block, 2..4 row buffers per warp
        const int rb = cols * static_cast<int>(sizeof(T));
        const size_t cap = static_cast<size_t>(max_smem_optin());
        for (int nw = 8; nw >= 2; nw >>= 1) {
            int nst = 4;
            while (nst >= 2 && fwd_staged_smem(rb, nw, nst) > cap) --nst;
            if (nst < 2) continue;
            const size_t smem = fwd_staged_smem(rb, nw, nst);
            auto kern = rmsnorm_fwd_staged<T>;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess)
                return check_launch("rmsnorm_fwd_staged attribute");
            int per_sm = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nw * 32, smem);
            if (per_sm < 1) per_sm = 1;
            const int64_t grid = std::min<int64_t>(ceil_div(rows, nw), static_cast<int64_t>(sms) * per_sm);
            kern<<<static_cast<unsigned>(grid), nw * 32, smem, st>>>(xp, wp, yp, rstd, rows, cols, eps, nst);
            return check_launch("rmsnorm_fwd_staged");
        }
    }
    if (cols % EPV == 0) {
        const int nvec = cols / EPV;
        const int64_t need_blocks = ceil_div(rows, kFwdThreads / 32);
        auto go = [&](auto kern) {
            int per_sm = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFwdThreads, 0);
            if (per_sm < 1) per_sm = 1;
            const int64_t grid = std::min<int64_t>(need_blocks, static_cast<int64_t>(sms) * per_sm);
            kern<<<static_cast<unsigned>(grid), kFwdThreads, 0, st>>>(xp, wp, yp, rstd, rows, cols, eps);
            return check_launch("rmsnorm_fwd");
        };
        if (nvec <= 32) return go(rmsnorm_fwd_warp<T, 1>);
        if (nvec <= 64) return go(rmsnorm_fwd_warp<T, 2>);
        if (nvec <= 128) return go(rmsnorm_fwd_warp<T, 4>);
        if (nvec <= 256) return go(rmsnorm_fwd_warp<T, 8>);
        if (nvec <= 512) return go(rmsnorm_fwd_warp<T, 16>);
        if (nvec <= 1024) return go(rmsnorm_fwd_warp<T, 32>);
    }
    const int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(sms) * 8);
    rmsnorm_fwd_generic<T><<<static_cast<unsigned>(grid), 256, 0, st>>>(xp, wp, yp, rstd, rows, cols, eps);
    return check_launch("rmsnorm_fwd_generic");
}

constexpr int kBwdStagedMaxThreads = 256;
// (dy, x) row buffers of a staged backward block: two in use, four in flight (with rows of
// at most 8 KB the ring takes at most 96 KB, two blocks per SM; measured faster at the
// power-capped clock of a long step than a ring of 4 with three blocks per SM)
constexpr int kBwdRing = 6;
constexpr size_t kBwdStagedSmemMax = 100u * 1024u;

// Row r of dy and x into ring buffer s (one mbarrier per buffer).
template <typename T>
__device__ __forceinline__ void bwd_issue_row(uint8_t* sm, uint32_t bars, const T* dy, const T* x, int64_t r, int s,
                                              uint32_t rb, int cols) {
    const uint32_t bar = bars + 8u * static_cast<uint32_t>(s);
    uint8_t* dst = sm + static_cast<size_t>(s) * 2 * rb;
    mbar_expect_tx(bar, 2 * rb);
    bulk_g2s(smem_u32(dst), dy + r * cols, rb, bar);
    bulk_g2s(smem_u32(dst + rb), x + r * cols, rb, bar);
}

// Two products of packed bf16 pairs in fp32: (a.lo b.lo + c.x, a.hi b.hi + c.y), each
// rounded once (the product of two bf16 values is exact in fp32).  The mixed-precision
// fma takes the bf16 halves of the packed words as they are, so neither operand is
// widened to fp32 by separate instructions first.
__device__ __forceinline__ float2 fma_bf2(uint32_t a, uint32_t b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %4;\n\t"
        "fma.rn.f32.bf16 %1, ah, bh, %5;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(a), "r"(b), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ uint32_t word(const uint4& u, int e) {
    return e == 0 ? u.x : e == 1 ? u.y : e == 2 ? u.z : u.w;
}

// Staged backward, two rows per block barrier: the block reduces the dot
// products of its rows i and i + 1 together (two independent shuffle trees,
// one barrier), then reads both rows again from shared memory for dx (and, in
// fp32, dw), so no row is held in registers across the barrier.  After the
// barrier of rows (i, i + 1) every thread is past rows (i - 2, i - 1), whose
// buffers thread 0 refills with rows i - 2 + nst and i - 1 + nst (a ring of
// nst = kBwdRing = 6 buffers, a compile-time constant so that slot and phase
// are masks and shifts rather than divisions).  Each
// block takes a contiguous group of rows (rows interleaved across blocks
// measured no faster).
// In bf16 the products are formed from the packed words by the mixed-precision
// fma (no separate widening of dy and w, nor of x before the barrier): before
// the barrier q = dy x feeds both the dot product (w q) and the dw sums (q rstd,
// rstd fetched a pair of rows ahead); after it dx = rstd (w dy) - c x.  Every
// product of two bf16 values is exact in fp32, so the results are those of the
// widened arithmetic bit for bit.
template <typename T, int VPT>
__global__ void __launch_bounds__(kBwdStagedMaxThreads, 3) rmsnorm_bwd_staged2(const T* dy, const T* __restrict__ x,
                                                           const T* __restrict__ w, const float* __restrict__ rstd,
                                                           T* dx, float* __restrict__ part, int64_t rows, int cols,
                                                           int64_t rows_per_block) {
    constexpr int nst = kBwdRing;   // ring slots: slot and phase arithmetic on a constant
    constexpr int EPV = Vec<T>::N;
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ float red[2][2][32];
    const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, wid = tid >> 5, NW = NT >> 5;
    const int nvec = cols / EPV;
    const uint32_t rb = static_cast<uint32_t>(cols) * sizeof(T);   // row bytes (multiple of 16)
    const uint32_t bars = smem_u32(sm + static_cast<size_t>(nst) * 2 * rb);
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per_block;
    const int64_t nr = min(rows, r0 + rows_per_block) - r0;   // this block's rows: r0 + i, i < nr
    auto row_of = [&](int64_t i) { return r0 + i; };
    if (tid == 0)
        for (int s = 0; s < nst; ++s) mbar_init(bars + 8u * s, 1);
    mbar_init_fence();
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < nst && s < nr; ++s) bwd_issue_row(sm, bars, dy, x, row_of(s), s, rb, cols);
    int64_t issued = nst;   // rows 0 .. issued-1 have been asked for (thread 0's view; same on all threads)
    // arithmetic on pairs of columns with the packed fp32x2 instructions (half the
    // floating-point instruction count of scalar code)
    constexpr int NP = EPV / 2;
    constexpr bool MX = sizeof(T) == 2;   // bf16: products from the packed words (mixed-precision fma)
    float2 wf[VPT][NP], dwa[VPT][NP];
    uint4 wraw[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = j * NT + tid;
        wraw[j] = v < nvec ? ldg16_nc(w + static_cast<int64_t>(v) * EPV) : make_uint4(0, 0, 0, 0);
        unpack2(wraw[j], wf[j]);
#pragma unroll
        for (int e = 0; e < NP; ++e) dwa[j][e] = make_float2(0.f, 0.f);
    }
    const float inv_cols = 1.0f / static_cast<float>(cols);
    const float2 nz2 = make_float2(-0.f, -0.f);
    // bf16: rstd of the current pair of rows (the dw sums use it before the barrier), fetched a
    // pair ahead
    float rsc0 = 0.f, rsc1 = 0.f;
    if (MX) {
        rsc0 = nr > 0 ? rstd[row_of(0)] : 0.f;
        rsc1 = nr > 1 ? rstd[row_of(1)] : 0.f;
    }
    bool ok = true;
    int64_t i = 0;
    int it = 0;
    for (; i < nr; i += 2, ++it) {
        float rsn0 = 0.f, rsn1 = 0.f;
        if (MX) {
            rsn0 = i + 2 < nr ? rstd[row_of(i + 2)] : 0.f;
            rsn1 = i + 3 < nr ? rstd[row_of(i + 3)] : 0.f;
        }
        const bool two = i + 1 < nr;
        const int s0 = static_cast<int>(i % nst), s1 = static_cast<int>((i + 1) % nst);
        bool got = mbar_wait(bars + 8u * s0, static_cast<uint32_t>(i / nst) & 1u);
        if (two) got = got && mbar_wait(bars + 8u * s1, static_cast<uint32_t>((i + 1) / nst) & 1u);
        const uint8_t* b0 = sm + static_cast<size_t>(s0) * 2 * rb;
        const uint8_t* b1 = sm + static_cast<size_t>(s1) * 2 * rb;
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        if (got) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = j * NT + tid;
                if (v < nvec) {
                    if constexpr (MX) {
                        // q = dy x in fp32 (exact); the dot product takes w q and the dw sums
                        // q rstd, both here, before the barrier
                        const float2 r0 = make_float2(rsc0, rsc0), r1 = make_float2(rsc1, rsc1);
                        const uint4 ud = *reinterpret_cast<const uint4*>(b0 + static_cast<size_t>(v) * 16);
                        const uint4 ux = *reinterpret_cast<const uint4*>(b0 + rb + static_cast<size_t>(v) * 16);
#pragma unroll
                        for (int e = 0; e < NP; ++e) {
                            const float2 q = fma_bf2(word(ud, e), word(ux, e), nz2);
                            a0 = __ffma2_rn(wf[j][e], q, a0);
                            dwa[j][e] = __ffma2_rn(q, r0, dwa[j][e]);
                        }
                        if (two) {
                            const uint4 vd = *reinterpret_cast<const uint4*>(b1 + static_cast<size_t>(v) * 16);
                            const uint4 vx = *reinterpret_cast<const uint4*>(b1 + rb + static_cast<size_t>(v) * 16);
#pragma unroll
                            for (int e = 0; e < NP; ++e) {
                                const float2 q = fma_bf2(word(vd, e), word(vx, e), nz2);
                                a1 = __ffma2_rn(wf[j][e], q, a1);
                                dwa[j][e] = __ffma2_rn(q, r1, dwa[j][e]);
                            }
                        }
                    } else {
                        float2 fx[NP], fd[NP];
                        unpack2(*reinterpret_cast<const uint4*>(b0 + static_cast<size_t>(v) * 16), fd);
                        unpack2(*reinterpret_cast<const uint4*>(b0 + rb + static_cast<size_t>(v) * 16), fx);
#pragma unroll
                        for (int e = 0; e < NP; ++e) a0 = __ffma2_rn(__fmul2_rn(fd[e], wf[j][e]), fx[e], a0);
                        if (two) {
                            unpack2(*reinterpret_cast<const uint4*>(b1 + static_cast<size_t>(v) * 16), fd);
                            unpack2(*reinterpret_cast<const uint4*>(b1 + rb + static_cast<size_t>(v) * 16), fx);
#pragma unroll
                            for (int e = 0; e < NP; ++e) a1 = __ffma2_rn(__fmul2_rn(fd[e], wf[j][e]), fx[e], a1);
                        }
                    }
                }
            }
        }
        float g0 = a0.x + a0.y, g1 = a1.x + a1.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g0 += __shfl_xor_sync(0xffffffffu, g0, o);
            g1 += __shfl_xor_sync(0xffffffffu, g1, o);
        }
        if (lane == 0) {
            red[it & 1][0][wid] = g0;
            red[it & 1][1][wid] = g1;
        }
        // both rows' partial sums are published, and every thread is past rows i-2, i-1
        if (!__syncthreads_and(got ? 1 : 0)) {
            ok = false;
            break;
        }
        if (tid == 0 && i >= 2) {
            fence_proxy_async_smem();   // the reads of those buffers happen before the copies overwrite them
            if (i - 2 + nst < nr)
                bwd_issue_row(sm, bars, dy, x, row_of(i - 2 + nst), static_cast<int>((i - 2) % nst), rb, cols);
            if (i - 1 + nst < nr)
                bwd_issue_row(sm, bars, dy, x, row_of(i - 1 + nst), static_cast<int>((i - 1) % nst), rb, cols);
        }
        if (i >= 2) issued = i + nst;
        float t0 = 0.f, t1 = 0.f;
        for (int q = 0; q < NW; ++q) {
            t0 += red[it & 1][0][q];
            t1 += red[it & 1][1][q];
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (rr == 1 && !two) break;
            const int64_t r = row_of(i + rr);
            const float rs = MX ? (rr ? rsc1 : rsc0) : rstd[r];
            const float c = rs * rs * rs * inv_cols * (rr ? t1 : t0);
            const float2 rs2 = make_float2(rs, rs), nc2 = make_float2(-c, -c);
            const uint8_t* bb = rr ? b1 : b0;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = j * NT + tid;
                if (v < nvec && MX) {
                    // dx = rs (w dy) - c x, with w dy formed from the packed words
                    const uint4 ud = *reinterpret_cast<const uint4*>(bb + static_cast<size_t>(v) * 16);
                    const uint4 ux = *reinterpret_cast<const uint4*>(bb + rb + static_cast<size_t>(v) * 16);
                    float2 fx[NP], o[NP];
                    unpack2(ux, fx);
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        const float2 u = fma_bf2(word(wraw[j], e), word(ud, e), nz2);
                        o[e] = __ffma2_rn(nc2, fx[e], __fmul2_rn(rs2, u));
                    }
                    stg16(dx + r * cols + static_cast<int64_t>(v) * EPV, pack2(o));
                } else if (v < nvec) {
                    float2 fx[NP], fd[NP], o[NP];
                    unpack2(*reinterpret_cast<const uint4*>(bb + static_cast<size_t>(v) * 16), fd);
                    unpack2(*reinterpret_cast<const uint4*>(bb + rb + static_cast<size_t>(v) * 16), fx);
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        // dx = rs (dy w) - c x;  dw += (dy x) rs
                        o[e] = __ffma2_rn(nc2, fx[e], __fmul2_rn(rs2, __fmul2_rn(fd[e], wf[j][e])));
                        dwa[j][e] = __ffma2_rn(__fmul2_rn(fd[e], fx[e]), rs2, dwa[j][e]);
                    }
                    stg16(dx + r * cols + static_cast<int64_t>(v) * EPV, pack2(o));
                }
            }
        }
        if (MX) {
            rsc0 = rsn0;
            rsc1 = rsn1;
        }
    }
    float* pr = part + static_cast<int64_t>(blockIdx.x) * cols;
    if (!ok) {
        if (tid == 0) {
            atomicExch(&g_stage_err, 1);
            // copies in flight: rows i .. issued-1
            for (int64_t ii = i; ii < min(issued, nr); ++ii)
                mbar_wait(bars + 8u * static_cast<uint32_t>(ii % nst), static_cast<uint32_t>(ii / nst) & 1u);
        }
        // the unfinished rows of dx and this block's partial row of dw: NaN
        for (int64_t ii = i; ii < nr; ++ii)
            for (int v = tid; v < nvec; v += NT)
                stg16(dx + row_of(ii) * cols + static_cast<int64_t>(v) * EPV, nan16<T>());
        for (int64_t c = static_cast<int64_t>(tid) * 4; c < cols; c += static_cast<int64_t>(NT) * 4)
            stg16(pr + c, nan16<float>());
        return;
    }
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = j * NT + tid;
        if (v < nvec) {
#pragma unroll
            for (int e = 0; e < NP; e += 2) {
                const float2 q2[2] = {dwa[j][e], dwa[j][e + 1]};
                stg16(pr + static_cast<int64_t>(v) * EPV + 2 * e, pack2(q2));
            }
        }
    }
}

inline size_t bwd_staged_smem(int rb, int nst) { return static_cast<size_t>(nst) * 2 * rb + 8u * nst; }

int64_t bwd_partials(int64_t rows) {
    return std::max<int64_t>(1, std::min<int64_t>({rows, static_cast<int64_t>(sm_count()) * 2, kMaxPartials}));
}

template <typename T>
int launch_bwd(const void* dy, const void* x, const void* w, const float* rstd, void* dx, void* dw, float* part,
               int64_t rows, int cols, cudaStream_t st) {
    constexpr int EPV = Vec<T>::N;
    const int64_t P = bwd_partials(rows);
    const int64_t rpb = ceil_div(rows, P);
    const int64_t grid = ceil_div(rows, rpb);
    int64_t grid_used = grid;   // partial rows written (the staged path uses its own grid)
    const T* dyp = static_cast<const T*>(dy);
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* dxp = static_cast<T*>(dx);
    bool done = false;
    const int rbytes = cols * static_cast<int>(sizeof(T));
    if (cols % EPV == 0 && cols / EPV <= 2 * kBwdStagedMaxThreads && bwd_staged_smem(rbytes, kBwdRing) <= kBwdStagedSmemMax) {
        // staged path: a ring of kBwdRing (dy, x) row pairs, two rows in use, the rest in flight
        const int nvec = cols / EPV;
        const size_t ssm = bwd_staged_smem(rbytes, kBwdRing);
        auto go = [&](auto kern, int vpt) -> int {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm)) !=
                cudaSuccess)
                return check_launch("rmsnorm_bwd_staged attribute");
            const int nt = static_cast<int>(std::min<int64_t>(kBwdStagedMaxThreads, ceil_div(ceil_div(nvec, vpt), 32) * 32));
            int per_sm = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nt, ssm);
            if (per_sm < 1) per_sm = 1;
            const int64_t P2 = std::max<int64_t>(1, std::min<int64_t>({rows, static_cast<int64_t>(sm_count()) * per_sm,
                                                                       kMaxPartials}));
            const int64_t rpb2 = ceil_div(rows, P2);
            grid_used = ceil_div(rows, rpb2);
            kern<<<static_cast<unsigned>(grid_used), nt, ssm, st>>>(dyp, xp, wp, rstd, dxp, part, rows, cols, rpb2);
            done = true;
            return check_launch("rmsnorm_bwd_staged");
        };
        int rc0 = LIGER_OK;
        // one column vector per thread up to kBwdStagedMaxThreads vectors (more warps per SM)
        if (nvec <= kBwdStagedMaxThreads) rc0 = go(rmsnorm_bwd_staged2<T, 1>, 1);
        else rc0 = go(rmsnorm_bwd_staged2<T, 2>, 2);
        if (rc0) return rc0;
    }
    if (!done && cols % EPV == 0) {
        const int nvec = cols / EPV;
        auto go = [&](auto kern, int vpt) {
            const int nt = static_cast<int>(std::min<int64_t>(256, ceil_div(ceil_div(nvec, vpt), 32) * 32));
            kern<<<static_cast<unsigned>(grid), nt, 0, st>>>(dyp, xp, wp, rstd, dxp, part, rows, cols, rpb);
            done = true;
        };
        if (nvec <= 256) go(rmsnorm_bwd_block<T, 1>, 1);
        else if (nvec <= 512) go(rmsnorm_bwd_block<T, 2>, 2);
        else if (nvec <= 1024) go(rmsnorm_bwd_block<T, 4>, 4);
        else if (nvec <= 2048) go(rmsnorm_bwd_block<T, 8>, 8);
    }
    if (!done)
        rmsnorm_bwd_generic<T><<<static_cast<unsigned>(grid), 256, 0, st>>>(dyp, xp, wp, rstd, dxp, part, rows, cols,
                                                                            rpb);
    int rc = check_launch("rmsnorm_bwd");
    if (rc) return rc;
    launch_dw_reduce<T>(part, static_cast<T*>(dw), static_cast<int>(grid_used), cols, st);
    return check_launch("rmsnorm_dw_reduce");
}

int check_common(int64_t rows, int64_t cols, int dtype) {
    if (dtype != LIGER_F32 && dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "rmsnorm: dtype %d", dtype);
    if (rows < 0 || cols <= 0 || cols > (1 << 30))
        return fail(LIGER_ERR_SHAPE, "rmsnorm: rows=%lld cols=%lld", (long long)rows, (long long)cols);
    return LIGER_OK;
}

}  // namespace

int rmsnorm_err_word(int** out) {
    static std::atomic<int*> addr[64];   // per device; racing threads store the same address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(LIGER_ERR_CUDA, "no CUDA device");
    int* a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&a), g_stage_err) != cudaSuccess)
            return check_launch("rmsnorm error word");
        addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return LIGER_OK;
}

}  // namespace liger

using namespace liger;

extern "C" int liger_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t rows, int64_t cols,
                                 float eps, int dtype, void* stream) {
    clear_error();
    if (int rc = check_common(rows, cols, dtype)) return rc;
    if (rows == 0) return LIGER_OK;
    if (!x || !w || !y) return fail(LIGER_ERR_NULL, "rmsnorm_fwd: x, w and y are required");
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (rstd && (reinterpret_cast<uintptr_t>(rstd) & 3)))
        return fail(LIGER_ERR_ALIGN, "rmsnorm_fwd: tensors must be 16-byte aligned");
    if (!(eps >= 0.f)) return fail(LIGER_ERR_SHAPE, "rmsnorm_fwd: eps must be >= 0");
    cudaStream_t st = as_stream(stream);
    return dtype == LIGER_F32 ? launch_fwd<float>(x, w, y, rstd, rows, (int)cols, eps, st)
                              : launch_fwd<__nv_bfloat16>(x, w, y, rstd, rows, (int)cols, eps, st);
}

extern "C" size_t liger_rmsnorm_bwd_workspace(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>(std::min<int64_t>(rows, kMaxPartials)) * static_cast<size_t>(cols) * sizeof(float);
}

extern "C" int liger_rmsnorm_bwd(const void* dy, const void* x, const void* w, const float* rstd, void* dx, void* dw,
                                 void* ws, size_t ws_bytes, int64_t rows, int64_t cols, int dtype, void* stream) {
    clear_error();
    if (int rc = check_common(rows, cols, dtype)) return rc;
    if (!dw || (rows > 0 && (!dy || !x || !w || !dx || !rstd)))
        return fail(LIGER_ERR_NULL, "rmsnorm_bwd: dy, x, w, rstd, dx and dw are required");
    if (!aligned16(dy) || !aligned16(x) || !aligned16(w) || !aligned16(dx) || !aligned16(dw) ||
        (reinterpret_cast<uintptr_t>(rstd) & 3))
        return fail(LIGER_ERR_ALIGN, "rmsnorm_bwd: tensors must be 16-byte aligned");
    const size_t need = liger_rmsnorm_bwd_workspace(rows, cols);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
        return fail(LIGER_ERR_WORKSPACE, "rmsnorm_bwd: workspace of %zu bytes (16-byte aligned) required, got %zu",
                    need, ws_bytes);
    cudaStream_t st = as_stream(stream);
    if (rows == 0) {
        // dw of an empty batch is zero
        const size_t bytes = static_cast<size_t>(cols) * (dtype == LIGER_F32 ? 4 : 2);
        if (cudaMemsetAsync(dw, 0, bytes, st) != cudaSuccess) return check_launch("rmsnorm_bwd memset");
        return LIGER_OK;
    }
    float* part = static_cast<float*>(ws);
    return dtype == LIGER_F32 ? launch_bwd<float>(dy, x, w, rstd, dx, dw, part, rows, (int)cols, st)
                              : launch_bwd<__nv_bfloat16>(dy, x, w, rstd, dx, dw, part, rows, (int)cols, st);
}

// ------------------------------------------------ backward without workspace
// For callers that cannot hand this library a device buffer at call time
// (see liger_rmsnorm_bwd_noalloc in liger.h), the dw partial sums live in a
// fixed array of device memory that the library itself reserves.  Host code
// must not pass the array's name to a kernel (on the host that name is only a
// stand-in); its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current.
#include <mutex>

namespace liger {
namespace {

constexpr size_t kNoAllocBytes = LIGER_RMSNORM_BWD_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_part[kNoAllocBytes / sizeof(float)];

constexpr int kNoAllocMaxDev = 64;
static float* g_noalloc_addr[kNoAllocMaxDev] = {nullptr};
static std::mutex g_noalloc_mu;

int noalloc_scratch(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return fail(LIGER_ERR_CUDA, "rmsnorm_bwd_noalloc: no current CUDA device");
    if (dev >= kNoAllocMaxDev) return fail(LIGER_ERR_CUDA, "rmsnorm_bwd_noalloc: device %d not supported", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_part);
        if (e != cudaSuccess || p == nullptr)
            return fail(LIGER_ERR_CUDA, "rmsnorm_bwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        g_noalloc_addr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_addr[dev];
    return LIGER_OK;
}

// Same kernels as launch_bwd, with at most max_parts partial rows.
template <typename T>
int launch_bwd_noalloc(const void* dy, const void* x, const void* w, const float* rstd, void* dx, void* dw,
                       float* part, int64_t rows, int cols, int64_t max_parts, cudaStream_t st) {
    constexpr int EPV = Vec<T>::N;
    const int64_t P = std::max<int64_t>(1, std::min(bwd_partials(rows), max_parts));
    const int64_t rpb = ceil_div(rows, P);
    const int64_t grid = ceil_div(rows, rpb);
    const T* dyp = static_cast<const T*>(dy);
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* dxp = static_cast<T*>(dx);
    bool done = false;
    if (cols % EPV == 0) {
        const int nvec = cols / EPV;
        auto go = [&](auto kern, int vpt) {
            const int nt = static_cast<int>(std::min<int64_t>(256, ceil_div(ceil_div(nvec, vpt), 32) * 32));
            kern<<<static_cast<unsigned>(grid), nt, 0, st>>>(dyp, xp, wp, rstd, dxp, part, rows, cols, rpb);
            done = true;
        };
        if (nvec <= 256) go(rmsnorm_bwd_block<T, 1>, 1);
        else if (nvec <= 512) go(rmsnorm_bwd_block<T, 2>, 2);
        else if (nvec <= 1024) go(rmsnorm_bwd_block<T, 4>, 4);
        else if (nvec <= 2048) go(rmsnorm_bwd_block<T, 8>, 8);
    }
    if (!done)
        rmsnorm_bwd_generic<T><<<static_cast<unsigned>(grid), 256, 0, st>>>(dyp, xp, wp, rstd, dxp, part, rows, cols,
                                                                            rpb);
    int rc = check_launch("rmsnorm_bwd_noalloc");
    if (rc) return rc;
    launch_dw_reduce<T>(part, static_cast<T*>(dw), static_cast<int>(grid), cols, st);
    return check_launch("rmsnorm_dw_reduce");
}

}  // namespace
}  // namespace liger

extern "C" int liger_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* w, const float* rstd, void* dx,
                                         void* dw, int64_t rows, int64_t cols, int dtype, void* stream) {
    clear_error();
    if (int rc = check_common(rows, cols, dtype)) return rc;
    if (static_cast<size_t>(cols) * sizeof(float) > kNoAllocBytes)
        return fail(LIGER_ERR_WORKSPACE,
                    "rmsnorm_bwd_noalloc: cols=%lld needs more than the %zu-byte built-in scratch (max cols %zu)",
                    (long long)cols, kNoAllocBytes, kNoAllocBytes / sizeof(float));
    if (!dw || (rows > 0 && (!dy || !x || !w || !dx || !rstd)))
        return fail(LIGER_ERR_NULL, "rmsnorm_bwd_noalloc: dy, x, w, rstd, dx and dw are required");
    if (!aligned16(dy) || !aligned16(x) || !aligned16(w) || !aligned16(dx) || !aligned16(dw) ||
        (reinterpret_cast<uintptr_t>(rstd) & 3))
        return fail(LIGER_ERR_ALIGN, "rmsnorm_bwd_noalloc: tensors must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    if (rows == 0) {
        const size_t bytes = static_cast<size_t>(cols) * (dtype == LIGER_F32 ? 4 : 2);
        if (cudaMemsetAsync(dw, 0, bytes, st) != cudaSuccess) return check_launch("rmsnorm_bwd_noalloc memset");
        return LIGER_OK;
    }
    float* part = nullptr;
    if (int rc = noalloc_scratch(&part)) return rc;
    const int64_t max_parts = static_cast<int64_t>(kNoAllocBytes / (static_cast<size_t>(cols) * sizeof(float)));
    return dtype == LIGER_F32
               ? launch_bwd_noalloc<float>(dy, x, w, rstd, dx, dw, part, rows, (int)cols, max_parts, st)
               : launch_bwd_noalloc<__nv_bfloat16>(dy, x, w, rstd, dx, dw, part, rows, (int)cols, max_parts, st);
}
