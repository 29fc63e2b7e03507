// Fused RMSNorm + QKV projection + RoPE (forward).
//
// Operator: the fused kernel on the page "Liger-Kernel底层优化：新一代内核级推理
// 加速引擎介绍", section "融合内核是如何工作的": RMSNorm of the hidden row, the
// Q, K and V projections of the normalised row with their biases, RoPE on q
// and k, with nothing written in between.
//
//   r_t = 1 / sqrt(mean_i x_ti^2 + eps)
//   q_t = RoPE_p(r_t * x_t diag(w) W_q^T + b_q),  k_t likewise,  v_t = r_t * x_t diag(w) W_v^T + b_v
//
// GB300 design.  The normalisation scales each row by r_t and each feature by
// w_i.  r_t acts on the output row, so it is applied to the fp32 accumulator
// in the GEMM epilogue.  w_i acts on the contraction index, so it is folded
// into the weights once per call: W' = bf16(W diag(w)), Q, K and V rows
// concatenated into one [N, H] operand (a weight pass of 2 N H bytes each way;
// a caller whose weights do not change can keep the folded copy and skip it).
// The normalised activations and the un-rotated q, k therefore never reach
// HBM: per call the data path is
//   1. qkv_fold   (optional): W' and the fp32 bias row           HBM-bound
//   2. qkv_prep:  r_t per token (one read of x) and, without caller tables,
//                 the token's cos/sin row (angle reduced mod 2 pi in fp32 with
//                 an exact product and a two-constant 2 pi)
//   3. tc_gemm_kernel<EPI_QKV_ROPE>: x W'^T on tcgen05, epilogue scales by r_t,
//                 adds the bias, rotates q and k heads in registers, writes
//                 q, k, v in their [B, S, heads, D] layouts.
#include "rope_angle.cuh"
#include "tc_gemm.cuh"

namespace liger {
namespace {

constexpr int kMaxHalfQkv = 128;   // head_dim <= 256

struct InvFreqQkv {
    double v[kMaxHalfQkv];   // theta^(-2i/D)
    float hi[kMaxHalfQkv];   // fl(v)
    float lo[kMaxHalfQkv];   // fl(v - hi)
};

static __device__ int g_qkv_err;

int qkv_err_addr(int** out) {
    static std::atomic<int*> addr[64];   // per device; racing threads store the same address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(LIGER_ERR_CUDA, "no CUDA device");
    int* a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&a), g_qkv_err) != cudaSuccess)
            return check_launch("rmsnorm_qkv_rope error word");
        addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return LIGER_OK;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct QkvLayout {
    size_t wf, bias, rstd, cos, sin, total;
};

QkvLayout qkv_layout(int64_t T, int64_t H, int64_t N, int64_t D) {
    QkvLayout l{};
    size_t o = 0;
    l.wf = o;
    o += round256(static_cast<size_t>(N) * static_cast<size_t>(H) * 2);
    l.bias = o;
    o += round256(static_cast<size_t>(N) * 4);
    l.rstd = o;
    o += round256(static_cast<size_t>(T) * 4);
    l.cos = o;
    o += round256(static_cast<size_t>(T) * static_cast<size_t>(D / 2) * 4);
    l.sin = o;
    o += round256(static_cast<size_t>(T) * static_cast<size_t>(D / 2) * 4);
    l.total = o;
    return l;
}

// W'[n, :] = bf16(W[n, :] * w) for the rows of W_q, W_k, W_v in turn; bias[n]
// in fp32 (0 where the projection has none).  One 16-byte vector per thread.
__global__ void qkv_fold(const __nv_bfloat16* __restrict__ wn, const __nv_bfloat16* __restrict__ Wq,
                         const __nv_bfloat16* __restrict__ Wk, const __nv_bfloat16* __restrict__ Wv,
                         const __nv_bfloat16* __restrict__ bq, const __nv_bfloat16* __restrict__ bk,
                         const __nv_bfloat16* __restrict__ bv, __nv_bfloat16* __restrict__ wf,
                         float* __restrict__ bias, int64_t nq, int64_t nk, int64_t H) {
    const int64_t N = nq + 2 * nk;
    const int64_t hv = H / 8;
    const int64_t nvec = N * hv;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / hv, kv = i - n * hv;
        const __nv_bfloat16* src = n < nq ? Wq + n * H : (n < nq + nk ? Wk + (n - nq) * H : Wv + (n - nq - nk) * H);
        float a[8], g[8];
        unpack(ldg16_nc(src + kv * 8), a);
        unpack(ldg16(wn + kv * 8), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] *= g[e];
        stg16(wf + n * H + kv * 8, pack(a));   // read by the GEMM next: leave it in L2
    }
    for (int64_t n = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; n < N;
         n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const __nv_bfloat16* b = n < nq ? bq : (n < nq + nk ? bk : bv);
        const int64_t o = n < nq ? n : (n < nq + nk ? n - nq : n - nq - nk);
        bias[n] = b ? __bfloat162float(b[o]) : 0.f;
    }
}

// One warp per token: r_t from the row's sum of squares (fp32, 16-byte
// loads), and, when make_tab, the token's cos/sin row at position
// pos ? pos[t] : t % S.
__global__ void __launch_bounds__(256) qkv_prep(const __nv_bfloat16* __restrict__ x, int64_t T, int64_t H, float eps,
                                                float* __restrict__ rstd, const int32_t* __restrict__ pos, int64_t S,
                                                int half, int make_tab, float* __restrict__ cos_t,
                                                float* __restrict__ sin_t, const __grid_constant__ InvFreqQkv f) {
    const int lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x * 8LL + (threadIdx.x >> 5);
    if (t >= T) return;
    const __nv_bfloat16* row = x + t * H;
    float ss = 0.f;
    for (int64_t c = lane * 8; c < H; c += 256) {
        float a[8];
        unpack(ldg16(row + c), a);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(a[e], a[e], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) rstd[t] = rsqrtf(ss / static_cast<float>(H) + eps);
    if (make_tab) {
        const int64_t p = pos ? static_cast<int64_t>(pos[t]) : t % S;
        for (int i = lane; i < half; i += 32) {
            const float2 cs = angle_cs32(p, f.hi[i], f.lo[i], f.v[i], 1.0f);
            cos_t[t * half + i] = cs.x;
            sin_t[t * half + i] = cs.y;
        }
    }
}

}  // namespace

// exported to liger_device_status, which reads and clears the word
int qkv_err_word(int** out) { return qkv_err_addr(out); }

}  // namespace liger

using namespace liger;
using namespace liger::tc;

extern "C" size_t liger_rmsnorm_qkv_rope_workspace(int64_t tokens, int64_t hidden, int64_t n_q_heads,
                                                   int64_t n_k_heads, int64_t head_dim) {
    if (tokens < 0 || hidden <= 0 || n_q_heads < 0 || n_k_heads < 0 || head_dim <= 0) return 0;
    return qkv_layout(tokens, hidden, (n_q_heads + 2 * n_k_heads) * head_dim, head_dim).total;
}

extern "C" int liger_rmsnorm_qkv_rope_fwd(const void* x, const void* w_norm, const void* Wq, const void* Wk,
                                          const void* Wv, const void* bq, const void* bk, const void* bv,
                                          const int32_t* pos, const float* cos_tab, const float* sin_tab,
                                          int64_t n_tab, void* q, void* k, void* v, float* rstd, void* ws,
                                          size_t ws_bytes, int64_t batch, int64_t seq, int64_t hidden,
                                          int64_t n_q_heads, int64_t n_k_heads, int64_t head_dim, double eps,
                                          double theta, int flags, int dtype, void* stream) {
    clear_error();
    const char* who = "rmsnorm_qkv_rope_fwd";
    if (dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "%s: bf16 only (tensor-core path)", who);
    const int64_t B = batch, S = seq, H = hidden, Hq = n_q_heads, Hk = n_k_heads, D = head_dim;
    if (B < 0 || S < 0 || H < 64 || H % 8 || H > (1 << 30) || Hq < 0 || Hk < 0 || Hq + Hk == 0 ||
        (D != 64 && D != 128 && D != 256) || (Hq + 2 * Hk) * D > (1 << 30) || B * S > (int64_t{1} << 31) - 1)
        return fail(LIGER_ERR_SHAPE, "%s: batch=%lld seq=%lld hidden=%lld heads=%lld/%lld head_dim=%lld "
                    "(hidden >= 64 and a multiple of 8; head_dim 64, 128 or 256)", who, (long long)B, (long long)S,
                    (long long)H, (long long)Hq, (long long)Hk, (long long)D);
    if (flags & ~1) return fail(LIGER_ERR_SHAPE, "%s: unknown flags 0x%x", who, flags);
    if ((cos_tab == nullptr) != (sin_tab == nullptr) || (cos_tab && n_tab <= 0))
        return fail(LIGER_ERR_SHAPE, "%s: cos and sin tables go together, with n_tab > 0", who);
    if (!cos_tab && (!(theta > 0.0) || !isfinite(theta))) return fail(LIGER_ERR_SHAPE, "%s: theta must be > 0", who);
    if (!(eps >= 0.0) || !isfinite(eps)) return fail(LIGER_ERR_SHAPE, "%s: eps must be >= 0", who);
    const int64_t T = B * S, nq = Hq * D, nk = Hk * D, N = nq + 2 * nk;
    const QkvLayout L = qkv_layout(T, H, N, D);
    if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255))
        return fail(LIGER_ERR_WORKSPACE, "%s: workspace of %zu bytes (256-byte aligned) required, got %zu", who,
                    L.total, ws_bytes);
    const bool fold = !(flags & 1);
    if (fold && (!w_norm || (nq > 0 && !Wq) || (nk > 0 && (!Wk || !Wv))))
        return fail(LIGER_ERR_NULL, "%s: norm weight and projection weights required", who);
    if (T == 0) return LIGER_OK;
    if (!x || (nq > 0 && !q) || (nk > 0 && (!k || !v))) return fail(LIGER_ERR_NULL, "%s: null tensor pointer", who);
    auto a16 = [](const void* p) { return p == nullptr || aligned16(p); };
    if (!a16(x) || !a16(w_norm) || !a16(Wq) || !a16(Wk) || !a16(Wv) || !a16(q) || !a16(k) || !a16(v) ||
        !a16(cos_tab) || !a16(sin_tab))
        return fail(LIGER_ERR_ALIGN, "%s: tensors and tables must be 16-byte aligned", who);
    if ((pos && (reinterpret_cast<uintptr_t>(pos) & 3)) || (rstd && (reinterpret_cast<uintptr_t>(rstd) & 3)) ||
        (bq && (reinterpret_cast<uintptr_t>(bq) & 1)) || (bk && (reinterpret_cast<uintptr_t>(bk) & 1)) ||
        (bv && (reinterpret_cast<uintptr_t>(bv) & 1)))
        return fail(LIGER_ERR_ALIGN, "%s: pos/rstd/biases must be aligned to their element size", who);
    cudaStream_t st = as_stream(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __nv_bfloat16* wf = reinterpret_cast<__nv_bfloat16*>(wsb + L.wf);
    float* bias = reinterpret_cast<float*>(wsb + L.bias);
    float* rs = rstd ? rstd : reinterpret_cast<float*>(wsb + L.rstd);
    float* cos_t = reinterpret_cast<float*>(wsb + L.cos);
    float* sin_t = reinterpret_cast<float*>(wsb + L.sin);
    const int half = static_cast<int>(D / 2);
    // 1. fold the norm weight into the projection weights
    if (fold) {
        const int64_t nvec = N * (H / 8);
        const int grid = static_cast<int>(std::min<int64_t>(ceil_div(nvec, 256), int64_t{sm_count()} * 8));
        qkv_fold<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w_norm),
                                       static_cast<const __nv_bfloat16*>(Wq), static_cast<const __nv_bfloat16*>(Wk),
                                       static_cast<const __nv_bfloat16*>(Wv), static_cast<const __nv_bfloat16*>(bq),
                                       static_cast<const __nv_bfloat16*>(bk), static_cast<const __nv_bfloat16*>(bv),
                                       wf, bias, nq, nk, H);
        if (int rc = check_launch("rmsnorm_qkv_rope fold")) return rc;
    }
    // 2. rstd per token and, without caller tables, the token's cos/sin row
    InvFreqQkv f;
    for (int i = 0; i < half; ++i) {
        f.v[i] = cos_tab ? 0.0 : pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
        f.hi[i] = static_cast<float>(f.v[i]);
        f.lo[i] = static_cast<float>(f.v[i] - static_cast<double>(f.hi[i]));
    }
    qkv_prep<<<static_cast<unsigned>(ceil_div(T, 8)), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), T, H, static_cast<float>(eps), rs, pos, S, half, cos_tab ? 0 : 1,
        cos_t, sin_t, f);
    if (int rc = check_launch("rmsnorm_qkv_rope prep")) return rc;
    // 3. the projection GEMM with the scale / bias / RoPE epilogue
    CUtensorMap mX, mW;
    int rc;
    if ((rc = make_map(&mX, x, H, T, H, BK, BM))) return rc;
    if ((rc = make_map(&mW, wf, H, N, H, BK, B_BOX_ROWS))) return rc;
    int* d_err = nullptr;
    if ((rc = qkv_err_addr(&d_err))) return rc;
    EpiParams e{};
    e.err = d_err;
    e.M = static_cast<int>(T);
    e.N = static_cast<int>(N);
    e.rs = rs;
    e.bias = bias;
    e.hd = static_cast<int>(D);
    e.nq = static_cast<int>(nq);
    e.nk = static_cast<int>(nk);
    e.out = static_cast<__nv_bfloat16*>(q);
    e.out2 = static_cast<__nv_bfloat16*>(k);
    e.out3 = static_cast<__nv_bfloat16*>(v);
    if (cos_tab) {
        e.cos_t = cos_tab;
        e.sin_t = sin_tab;
        e.tab_row = pos;
        e.n_tab = static_cast<int>(std::min<int64_t>(n_tab, INT32_MAX));
        e.tab_mod = static_cast<int>(S);
    } else {
        e.cos_t = cos_t;
        e.sin_t = sin_t;
        e.tab_row = nullptr;
        e.tab_mod = INT32_MAX;   // row t of the per-token table
    }
    e.ld_tab = half;
    // groups of 8 tile columns: a wave of resident tiles shares ~19 row blocks of
    // x and 8 column blocks of W' through L2 (measured at seq 32768, hidden
    // 4096, N 12288: 9 % faster than streaming x past an L2-resident W', 20 %
    // faster than the reverse)
    e.raster = RASTER_N_GROUPS;
    e.hint_a = HINT_NORMAL;
    e.hint_b = HINT_NORMAL;
    return launch_gemm<0, 0, EPI_QKV_ROPE, 1>(mX, mW, static_cast<int>(T), static_cast<int>(N), static_cast<int>(H), e,
                                           st);
}
