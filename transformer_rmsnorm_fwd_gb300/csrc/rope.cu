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
//  * staged form (16-byte vectors, the common case): one block per tile of
//    consecutive tokens of one batch row (about 32 KB of Q and K rows); the
//    tile is brought into shared memory by 1-D bulk copies issued at the
//    block's start, while the threads form the tile's angles, so a whole
//    tile per block is in flight without registers: the kernel keeps HBM
//    busy at the power-capped SM clock of a long training step, where a
//    register-bound form loses a quarter of its bandwidth;
//  * otherwise (scalar elements, or a tile that does not fit): one block per
//    group of npos positions (4 at head_dim 128, so that each thread forms
//    one angle) and batch group: the angles are formed once in shared memory
//    and reused by every head of Q and K and, when the positions are
//    implicit (p = s), by every batch row;
//  * the inverse frequencies theta^(-2i/D) are computed on the host in
//    double precision and passed as a kernel parameter;
//  * angle phi = p * inv_freq in double, reduced modulo 2 pi in double
//    (two-term 2 pi), then sincosf on the reduced single-precision angle:
//    the result is accurate to ~1 ulp of fp32 at any position, where a plain
//    fp32 p * inv_freq would err by ~p ulp;
//  * each thread rotates 16-byte vectors (half-split pairing: the two halves
//    of a head; interleaved pairing: four adjacent pairs); a warp covers
//    whole 128-byte lines; the block's (vector, token) tasks are dealt to the
//    threads in turn, so every thread gets the same share whatever the head
//    counts (40 heads of 128 give 320 vector slots per token).
// The extended entry points add the interleaved pairing (2i, 2i+1), per-token
// strides (Q and K as views into a packed QKV buffer) and caller-supplied
// cos/sin tables (for scaled frequency schedules).
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "mbarrier.cuh"
#include "rope_angle.cuh"

namespace liger {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxHalf = 256;   // head_dim <= 512
constexpr int kBatchGroup = 8;

struct InvFreq {
    double v[kMaxHalf];
};

struct RopeArgs {
    void* q;
    void* k;
    const int32_t* pos;
    const float* cos_tab;   // [n_tab, D/2] or null
    const float* sin_tab;
    int64_t n_tab;
    int64_t q_ts, k_ts;     // elements between consecutive tokens (b, s)
    int B, S, Hq, Hk, D, npos;
    float sign;
};

// VEC: 16-byte vectors (else scalar); INTER: interleaved pairs (2i, 2i+1).
template <typename T, bool VEC, bool INTER>
__global__ void __launch_bounds__(kThreads) rope_kernel(const RopeArgs a, const __grid_constant__ InvFreq f) {
    extern __shared__ float2 cs[];   // [npos][nb_angles][D/2] (cos, +-sin)
    T* q = static_cast<T*>(a.q);
    T* k = static_cast<T*>(a.k);
    const int D = a.D, half = D >> 1, S = a.S, Hq = a.Hq, Hk = a.Hk;
    const int s0 = blockIdx.x * a.npos;
    const int np = min(a.npos, S - s0);
    const int b0 = blockIdx.y * kBatchGroup;
    const int nb = min(kBatchGroup, a.B - b0);
    const int na = a.pos ? nb : 1;     // distinct angle rows per position in this block
    for (int t = threadIdx.x; t < np * na * half; t += kThreads) {
        const int row = t / half, i = t - row * half;
        const int pp = row / na, bl = row - pp * na;
        const int64_t p = a.pos ? static_cast<int64_t>(a.pos[static_cast<int64_t>(b0 + bl) * S + s0 + pp])
                                : static_cast<int64_t>(s0 + pp);
        if (a.cos_tab != nullptr) {
            const int64_t pc = p < 0 ? 0 : (p >= a.n_tab ? a.n_tab - 1 : p);   // positions outside the table clamp
            cs[t] = make_float2(a.cos_tab[pc * half + i], a.sign * a.sin_tab[pc * half + i]);
        } else {
            cs[t] = angle_cs(static_cast<double>(p), f.v[i], a.sign);
        }
    }
    __syncthreads();
    const int H = Hq + Hk;
    auto head_base = [&](int bl, int pp, int h) -> T* {
        const int64_t bs = static_cast<int64_t>(b0 + bl) * S + s0 + pp;
        return h < Hq ? q + bs * a.q_ts + static_cast<int64_t>(h) * D
                      : k + bs * a.k_ts + static_cast<int64_t>(h - Hq) * D;
    };
    if (VEC) {
        constexpr int EPV = Vec<T>::N;
        // half-split: a slot is the pair of vectors (v, v + D/2) of a head; interleaved:
        // one vector.  The block's work is nslot x (positions x batch rows) tasks, dealt
        // to the threads in turn (task t: slot t mod nslot, row t / nslot), so that every
        // thread gets the same share whatever the head counts (40 heads of 128 at 8
        // vectors per head: 320 slots, 1.25 per thread per row); a thread steps through
        // its tasks by adding kThreads to (slot, row) instead of dividing.
        const int vph = INTER ? D / EPV : half / EPV;
        const int nslot = H * vph;
        const int ntask = nslot * np * nb;
        int slot = threadIdx.x, row = 0;
        while (slot >= nslot) {
            slot -= nslot;
            ++row;
        }
        for (int t = threadIdx.x; t < ntask; t += kThreads) {
            const int h = slot / vph, v = slot - h * vph;
            const int pp = row / nb, bl = row - pp * nb;
            const bool isq = h < Hq;
            T* hb = isq ? q + static_cast<int64_t>(h) * D + v * EPV : k + static_cast<int64_t>(h - Hq) * D + v * EPV;
            const int64_t ts = isq ? a.q_ts : a.k_ts;
            const int coff = INTER ? (v * EPV) >> 1 : v * EPV;   // first angle index of this slot
            slot += kThreads;
            while (slot >= nslot) {
                slot -= nslot;
                ++row;
            }
            T* pa = hb + (static_cast<int64_t>(b0 + bl) * S + s0 + pp) * ts;
            const float4* c4 = reinterpret_cast<const float4*>(cs + (pp * na + (a.pos ? bl : 0)) * half + coff);
            if (INTER) {
                float e[EPV];
                unpack(ldg16(pa), e);
#pragma unroll
                for (int j = 0; j < EPV / 2; j += 2) {
                    const float4 r = c4[j >> 1];   // two (cos, sin) pairs
                    float x0 = e[2 * j], x1 = e[2 * j + 1];
                    e[2 * j] = x0 * r.x - x1 * r.y;
                    e[2 * j + 1] = x1 * r.x + x0 * r.y;
                    x0 = e[2 * j + 2];
                    x1 = e[2 * j + 3];
                    e[2 * j + 2] = x0 * r.z - x1 * r.w;
                    e[2 * j + 3] = x1 * r.z + x0 * r.w;
                }
                stg16(pa, pack(e));
            } else {
                T* pb = pa + half;
                float av[EPV], bv[EPV];
                // the two halves of a head sit in one 256-byte block: ask L2 for all of it
                unpack(ldg16_pf256(pa), av);
                unpack(ldg16_pf256(pb), bv);
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const float4 r = c4[e >> 1];
                    float x0 = av[e], x1 = bv[e];
                    av[e] = x0 * r.x - x1 * r.y;
                    bv[e] = x1 * r.x + x0 * r.y;
                    x0 = av[e + 1];
                    x1 = bv[e + 1];
                    av[e + 1] = x0 * r.z - x1 * r.w;
                    bv[e + 1] = x1 * r.z + x0 * r.w;
                }
                stg16(pa, pack(av));
                stg16(pb, pack(bv));
            }
        }
    } else {
        const int per_pos = nb * H * half;
        const int ntask = np * per_pos;
        for (int t = threadIdx.x; t < ntask; t += kThreads) {
            const int pp = t / per_pos;
            int rem = t - pp * per_pos;
            const int bl = rem / (H * half);
            rem -= bl * H * half;
            const int h = rem / half, i = rem - h * half;
            T* base = head_base(bl, pp, h);
            const float2 r = cs[(pp * na + (a.pos ? bl : 0)) * half + i];
            T* pa = INTER ? base + 2 * i : base + i;
            T* pb = INTER ? base + 2 * i + 1 : base + i + half;
            const float x0 = ldf(pa), x1 = ldf(pb);
            stf(pa, x0 * r.x - x1 * r.y);
            stf(pb, x1 * r.x + x0 * r.y);
        }
    }
}

// ------------------------------------------------------------ staged form
// One block per tile of npos consecutive tokens of one batch row.  Thread 0
// bulk-copies the tile's Q and K token rows into shared memory (two 1-D copies
// per token, all counted on one mbarrier) while every thread forms the tile's
// angles; the threads then rotate 16-byte vectors read from shared memory and
// store them in place.  A whole tile (about 32 KB) is in flight per block
// without holding it in registers, so the loads do not wait on the issue rate
// of the threads, whatever the SM clock.  The angle table is laid out
// [token][element of a vector][vector] so that the threads of a quarter warp,
// which hold consecutive vectors of a head, read consecutive words.
// The wait is bounded; on expiry the kernel records it in g_rope_err (read and
// cleared by liger_device_status), waits (bounded) for its copies, writes NaN
// into its tile and stops.
static __device__ int g_rope_err;

template <typename T, bool INTER>
__global__ void __launch_bounds__(kThreads) rope_staged_kernel(const RopeArgs a, const __grid_constant__ InvFreq f) {
    constexpr int EPV = Vec<T>::N;
    constexpr int APV = INTER ? EPV / 2 : EPV;   // angles per 16-byte vector
    extern __shared__ __align__(128) uint8_t sm[];
    T* q = static_cast<T*>(a.q);
    T* k = static_cast<T*>(a.k);
    const int D = a.D, half = D >> 1, S = a.S, Hq = a.Hq, Hk = a.Hk, H = Hq + Hk;
    const int s0 = blockIdx.x * a.npos;
    const int np = min(a.npos, S - s0);
    const int64_t b = blockIdx.y;
    const uint32_t qrow = static_cast<uint32_t>(Hq * D) * sizeof(T), krow = static_cast<uint32_t>(Hk * D) * sizeof(T);
    const uint32_t rowb = qrow + krow;                        // a multiple of 16
    uint8_t* tile = sm;                                       // [npos][rowb]
    float2* cs = reinterpret_cast<float2*>(sm + static_cast<size_t>(a.npos) * rowb);   // [npos][APV][vph]
    const uint32_t bar = smem_u32(cs + a.npos * half);
    const int vph = half / APV;                               // vectors per head (half-split: per half)
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_expect_tx(bar, static_cast<uint32_t>(np) * rowb);
        for (int pp = 0; pp < np; ++pp) {
            const int64_t bs = b * S + s0 + pp;
            if (qrow) bulk_g2s(smem_u32(tile + static_cast<size_t>(pp) * rowb), q + bs * a.q_ts, qrow, bar);
            if (krow) bulk_g2s(smem_u32(tile + static_cast<size_t>(pp) * rowb + qrow), k + bs * a.k_ts, krow, bar);
        }
    }
    for (int t = threadIdx.x; t < np * half; t += kThreads) {
        const int pp = t / half, i = t - pp * half;
        const int64_t p = a.pos ? static_cast<int64_t>(a.pos[b * S + s0 + pp]) : static_cast<int64_t>(s0 + pp);
        float2 r;
        if (a.cos_tab != nullptr) {
            const int64_t pc = p < 0 ? 0 : (p >= a.n_tab ? a.n_tab - 1 : p);   // positions outside the table clamp
            r = make_float2(a.cos_tab[pc * half + i], a.sign * a.sin_tab[pc * half + i]);
        } else {
            r = angle_cs(static_cast<double>(p), f.v[i], a.sign);
        }
        const int v = i / APV, e = i - v * APV;
        cs[pp * half + e * vph + v] = r;
    }
    const bool got = mbar_wait(bar, 0);
    if (!__syncthreads_and(got ? 1 : 0)) {
        if (threadIdx.x == 0) {
            atomicExch(&g_rope_err, 1);
            mbar_wait(bar, 0);   // the copies still in flight into this block's shared memory
        }
        __syncthreads();
        const int nv = H * (D / EPV);
        for (int t = threadIdx.x; t < np * nv; t += kThreads) {
            const int pp = t / nv, slot = t - pp * nv, h = slot / (D / EPV), v = slot - h * (D / EPV);
            const int64_t bs = b * S + s0 + pp;
            T* dst = h < Hq ? q + bs * a.q_ts + static_cast<int64_t>(h) * D : k + bs * a.k_ts + static_cast<int64_t>(h - Hq) * D;
            stg16(dst + v * EPV, nan16<T>());
        }
        return;
    }
    const int nslot = H * vph;
    const int ntask = nslot * np;
    // task t = (token pp, head h, vector v): pp and the slot advance with the thread's
    // stride instead of being divided out of t, and h, v come from a shift and a mask when
    // vph is a power of two (every power-of-two head size)
    const bool vpow2 = (vph & (vph - 1)) == 0;
    const int vsh = __ffs(vph) - 1;
    int pp = static_cast<int>(threadIdx.x) / nslot, slot = static_cast<int>(threadIdx.x) - pp * nslot;
    for (int t = threadIdx.x; t < ntask; t += kThreads) {
        const int h = vpow2 ? slot >> vsh : slot / vph;
        const int v = vpow2 ? slot & (vph - 1) : slot - h * vph;
        const int64_t bs = b * S + s0 + pp;
        T* dst = h < Hq ? q + bs * a.q_ts + static_cast<int64_t>(h) * D : k + bs * a.k_ts + static_cast<int64_t>(h - Hq) * D;
        const uint8_t* src = tile + static_cast<size_t>(pp) * rowb + static_cast<size_t>(h * D) * sizeof(T);
        const float2* ang = cs + pp * half + v;
        if (INTER) {
            float e8[EPV];
            unpack(*reinterpret_cast<const uint4*>(src + v * 16), e8);
#pragma unroll
            for (int j = 0; j < APV; ++j) {
                const float2 r = ang[j * vph];
                const float x0 = e8[2 * j], x1 = e8[2 * j + 1];
                e8[2 * j] = x0 * r.x - x1 * r.y;
                e8[2 * j + 1] = x1 * r.x + x0 * r.y;
            }
            stg16(dst + v * EPV, pack(e8));
        } else {
            float av[EPV], bv[EPV];
            unpack(*reinterpret_cast<const uint4*>(src + v * 16), av);
            unpack(*reinterpret_cast<const uint4*>(src + static_cast<size_t>(half) * sizeof(T) + v * 16), bv);
#pragma unroll
            for (int j = 0; j < APV; ++j) {
                const float2 r = ang[j * vph];
                const float x0 = av[j], x1 = bv[j];
                av[j] = x0 * r.x - x1 * r.y;
                bv[j] = x1 * r.x + x0 * r.y;
            }
            stg16(dst + v * EPV, pack(av));
            stg16(dst + half + v * EPV, pack(bv));
        }
        slot += kThreads;
        while (slot >= nslot) {
            slot -= nslot;
            ++pp;
        }
    }
}

// Tokens per block of the staged form: a tile of about 32 KB, at most 4096
// angles; 0 when one token row does not fit the shared memory.
int staged_tokens(int64_t row_bytes, int half, int64_t S) {
    const int64_t cap = max_smem_optin();
    int64_t np = std::max<int64_t>(1, std::min<int64_t>({(32 << 10) / std::max<int64_t>(row_bytes, 1), 4096 / half, S}));
    if (static_cast<int64_t>(np) * (row_bytes + 8 * half) + 8 > cap) return 0;
    return static_cast<int>(np);
}

int rope_run(void* q, void* k, const int32_t* pos, int64_t B, int64_t S, int64_t Hq, int64_t Hk, int64_t D,
             int64_t q_ts, int64_t k_ts, int pairing, const float* cos_tab, const float* sin_tab, int64_t n_tab,
             double theta, int dtype, void* stream, float sign, bool strict_align, const char* who) {
    clear_error();
    if (dtype != LIGER_F32 && dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "%s: dtype %d", who, dtype);
    if (B < 0 || S < 0 || Hq < 0 || Hk < 0 || D <= 0 || (D & 1) || D > 2 * kMaxHalf || S > 2147483647LL ||
        B > 2147483647LL || Hq + Hk > (1 << 20))
        return fail(LIGER_ERR_SHAPE, "%s: batch=%lld seq=%lld heads=%lld/%lld head_dim=%lld (even, <= %d)", who,
                    (long long)B, (long long)S, (long long)Hq, (long long)Hk, (long long)D, 2 * kMaxHalf);
    if (pairing != 0 && pairing != 1) return fail(LIGER_ERR_SHAPE, "%s: pairing must be 0 or 1", who);
    if ((q_ts < Hq * D) || (k_ts < Hk * D))
        return fail(LIGER_ERR_SHAPE, "%s: token strides %lld/%lld smaller than heads*head_dim", who,
                    (long long)q_ts, (long long)k_ts);
    if ((cos_tab == nullptr) != (sin_tab == nullptr) || (cos_tab && n_tab <= 0))
        return fail(LIGER_ERR_SHAPE, "%s: cos and sin tables go together, with n_tab > 0", who);
    if (!cos_tab && (!(theta > 0.0) || !isfinite(theta))) return fail(LIGER_ERR_SHAPE, "%s: theta must be > 0", who);
    if (B == 0 || S == 0 || Hq + Hk == 0) return LIGER_OK;
    if ((Hq > 0 && !q) || (Hk > 0 && !k)) return fail(LIGER_ERR_NULL, "%s: q/k required for nonzero head counts", who);
    const size_t esz = dtype == LIGER_F32 ? 4 : 2;
    const bool q16 = !q || aligned16(q), k16 = !k || aligned16(k);
    if (strict_align && (!q16 || !k16)) return fail(LIGER_ERR_ALIGN, "%s: q and k must be 16-byte aligned", who);
    if ((q && reinterpret_cast<uintptr_t>(q) % esz) || (k && reinterpret_cast<uintptr_t>(k) % esz))
        return fail(LIGER_ERR_ALIGN, "%s: q and k must be aligned to their element size", who);
    if ((pos && (reinterpret_cast<uintptr_t>(pos) & 3)) ||
        (cos_tab && ((reinterpret_cast<uintptr_t>(cos_tab) | reinterpret_cast<uintptr_t>(sin_tab)) & 3)))
        return fail(LIGER_ERR_ALIGN, "%s: pos and tables must be 4-byte aligned", who);
    const int half = static_cast<int>(D / 2);
    InvFreq f;
    for (int i = 0; i < half; ++i)
        f.v[i] = cos_tab ? 0.0 : pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
    const int nbg = static_cast<int>(ceil_div(B, kBatchGroup));
    if (nbg > 65535) return fail(LIGER_ERR_SHAPE, "%s: batch too large", who);
    // positions per block: enough that every thread forms one angle (head_dim 128: 4)
    const int npos = std::max(1, std::min(16, kThreads / half));
    dim3 grid(static_cast<unsigned>(ceil_div(S, npos)), static_cast<unsigned>(nbg));
    const size_t smem = static_cast<size_t>(npos) * (pos ? kBatchGroup : 1) * half * sizeof(float2);
    cudaStream_t st = as_stream(stream);
    const int epv = dtype == LIGER_F32 ? 4 : 8;
    // 16-byte vectors need every head start aligned: strides and head_dim in whole vectors
    const bool vec = (pairing ? (D % epv) : (half % epv)) == 0 && q_ts % epv == 0 && k_ts % epv == 0 && q16 && k16;
    RopeArgs a{q, k, pos, cos_tab, sin_tab, n_tab, q_ts, k_ts, (int)B, (int)S, (int)Hq, (int)Hk, (int)D, npos, sign};
    if (vec && B <= 65535) {
        const int64_t row_bytes = (Hq + Hk) * D * static_cast<int64_t>(esz);
        int nps = staged_tokens(row_bytes, half, S);
        // small problems: fewer tokens per block, so that at least two blocks per SM share the work
        if (nps > 1) {
            const int64_t per = ceil_div(B * S, 2 * static_cast<int64_t>(sm_count()));
            nps = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(nps, per)));
        }
        if (nps > 0) {
            a.npos = nps;
            const size_t ssm = static_cast<size_t>(nps) * (row_bytes + 8 * half) + 8;
            dim3 g2(static_cast<unsigned>(ceil_div(S, static_cast<int64_t>(nps))), static_cast<unsigned>(B));
            auto go2 = [&](auto kern) -> int {
                if (ssm > 48u * 1024u &&
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm)) !=
                        cudaSuccess)
                    return check_launch(who);
                kern<<<g2, kThreads, ssm, st>>>(a, f);
                return check_launch(who);
            };
            if (dtype == LIGER_F32)
                return pairing ? go2(rope_staged_kernel<float, true>) : go2(rope_staged_kernel<float, false>);
            using Bf = __nv_bfloat16;
            return pairing ? go2(rope_staged_kernel<Bf, true>) : go2(rope_staged_kernel<Bf, false>);
        }
    }
    auto go = [&](auto kern) { kern<<<grid, kThreads, smem, st>>>(a, f); };
    if (dtype == LIGER_F32) {
        if (pairing) vec ? go(rope_kernel<float, true, true>) : go(rope_kernel<float, false, true>);
        else vec ? go(rope_kernel<float, true, false>) : go(rope_kernel<float, false, false>);
    } else {
        using Bf = __nv_bfloat16;
        if (pairing) vec ? go(rope_kernel<Bf, true, true>) : go(rope_kernel<Bf, false, true>);
        else vec ? go(rope_kernel<Bf, true, false>) : go(rope_kernel<Bf, false, false>);
    }
    return check_launch(who);
}

}  // namespace

int rope_err_word(int** out) {
    static std::atomic<int*> addr[64];   // per device; racing threads store the same address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(LIGER_ERR_CUDA, "no CUDA device");
    int* p = addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_rope_err) != cudaSuccess)
            return check_launch("rope error word");
        addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return LIGER_OK;
}

}  // namespace liger

extern "C" int liger_rope_fwd(void* q, void* k, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                              int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream) {
    return liger::rope_run(q, k, pos, batch, seq, n_q_heads, n_k_heads, head_dim, n_q_heads * head_dim,
                           n_k_heads * head_dim, 0, nullptr, nullptr, 0, theta, dtype, stream, 1.0f, true, "rope_fwd");
}

extern "C" int liger_rope_bwd(void* dq, void* dk, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                              int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream) {
    return liger::rope_run(dq, dk, pos, batch, seq, n_q_heads, n_k_heads, head_dim, n_q_heads * head_dim,
                           n_k_heads * head_dim, 0, nullptr, nullptr, 0, theta, dtype, stream, -1.0f, true, "rope_bwd");
}

extern "C" int liger_rope_fwd_ex(void* q, void* k, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                                 int64_t n_k_heads, int64_t head_dim, int64_t q_token_stride, int64_t k_token_stride,
                                 int pairing, const float* cos_tab, const float* sin_tab, int64_t n_tab, double theta,
                                 int dtype, void* stream) {
    return liger::rope_run(q, k, pos, batch, seq, n_q_heads, n_k_heads, head_dim, q_token_stride, k_token_stride,
                           pairing, cos_tab, sin_tab, n_tab, theta, dtype, stream, 1.0f, false, "rope_fwd_ex");
}

extern "C" int liger_rope_bwd_ex(void* dq, void* dk, const int32_t* pos, int64_t batch, int64_t seq,
                                 int64_t n_q_heads, int64_t n_k_heads, int64_t head_dim, int64_t q_token_stride,
                                 int64_t k_token_stride, int pairing, const float* cos_tab, const float* sin_tab,
                                 int64_t n_tab, double theta, int dtype, void* stream) {
    return liger::rope_run(dq, dk, pos, batch, seq, n_q_heads, n_k_heads, head_dim, q_token_stride, k_token_stride,
                           pairing, cos_tab, sin_tab, n_tab, theta, dtype, stream, -1.0f, false, "rope_bwd_ex");
}
