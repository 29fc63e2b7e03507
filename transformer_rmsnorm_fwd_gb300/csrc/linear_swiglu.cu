// FusedLinearSwiGLU: the gate and up projections of the MLP and the SwiGLU
// activation in one tensor-core kernel, and its backward.
//
// Operator: the FusedLinearSwiGLU paragraph of the page "Liger-Kernel核心技术：
// RollingBuffer与融合算子详解", section "算子融合": x @ W_g and x @ W_u computed
// together, SiLU and the product taken in registers, only the result written.
//
//   forward:  h = silu(X W_g^T) * (X W_u^T)        X [T, H], W_g, W_u [I, H], h [T, I]
//   backward: g = X W_g^T, u = X W_u^T (recomputed), s = sigmoid(g)
//             dG = dh u s (1 + g (1 - s)),  dU = dh g s
//             dX = dG W_g + dU W_u,  dW_g = dG^T X,  dW_u = dU^T X
//
// GB300 design (all tensor-core, tcgen05):
//  * forward: one persistent GEMM whose 256 B rows per stage are 128 gate rows
//    and the matching 128 up rows (two TMA boxes), so a 128 x 256 accumulator
//    tile holds g and u for 128 output columns; the epilogue writes silu(g) u
//    and nothing else -- g and u never reach HBM;
//  * backward: the same GEMM recomputes g and u and its epilogue forms dG and
//    dU from dh (the only [T, I] intermediates, in the workspace); dX is one
//    GEMM over K = 2I that reads (dG, W_g) for the first half of its k-blocks
//    and (dU, W_u) for the second; dW_g and dW_u are two GEMMs with both
//    operands MN-major.
#include <atomic>

#include "tc_gemm.cuh"

namespace liger {

// Error word of the GEMMs launched here (bounded-wait expiry codes); these
// entry points take no workspace header, so it is a module variable, read
// back and cleared by liger_device_status.
static __device__ int g_lsw_err;

int lsw_err_word(int** out) {
    static std::atomic<int*> addr[64];   // per device; racing threads store the same address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(LIGER_ERR_CUDA, "no CUDA device");
    int* a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&a), g_lsw_err) != cudaSuccess)
            return check_launch("fused_linear_swiglu error word");
        addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return LIGER_OK;
}

namespace {

int check_shapes(int64_t T, int64_t H, int64_t I, int dtype, const char* who) {
    if (dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "%s: bf16 only (tensor-core path)", who);
    if (T < 0 || H < 64 || I < 8 || H % 8 || I % 8 || T > (int64_t{1} << 31) || H > (1 << 30) || I > (1 << 30))
        return fail(LIGER_ERR_SHAPE, "%s: T=%lld H=%lld I=%lld (H >= 64, H and I multiples of 8)", who, (long long)T,
                    (long long)H, (long long)I);
    return LIGER_OK;
}

}  // namespace
}  // namespace liger

using namespace liger;
using namespace liger::tc;

namespace liger {
namespace {

int fwd_impl(const void* X, const void* Wg, const void* Wu, void* out, void* g_save, void* u_save, int64_t T,
             int64_t H, int64_t I, int dtype, void* stream, const char* who) {
    using namespace tc;
    if (int rc = check_shapes(T, H, I, dtype, who)) return rc;
    if (T == 0) return LIGER_OK;
    if (!X || !Wg || !Wu || !out) return fail(LIGER_ERR_NULL, "%s: null tensor pointer", who);
    if (!aligned16(X) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(out) || (g_save && !aligned16(g_save)) ||
        (u_save && !aligned16(u_save)))
        return fail(LIGER_ERR_ALIGN, "%s: tensors must be 16-byte aligned", who);
    CUtensorMap mG, mU;
    int rc;
    if ((rc = make_map(&mG, Wg, H, I, H, BK, BN / 2))) return rc;
    if ((rc = make_map(&mU, Wu, H, I, H, BK, BN / 2))) return rc;
    int* d_err = nullptr;
    if ((rc = lsw_err_word(&d_err))) return rc;
    EpiParams e{};
    e.err = d_err;
    e.M = static_cast<int>(T);
    e.N = static_cast<int>(I);
    e.out = static_cast<__nv_bfloat16*>(out);
    e.out2 = static_cast<__nv_bfloat16*>(g_save);
    e.out3 = static_cast<__nv_bfloat16*>(u_save);
    e.ldo = I;
    e.bsplit = 1;
    e.raster = RASTER_M_FASTEST;
    e.hint_a = HINT_EVICT_LAST;    // X: reused by every column tile
    e.hint_b = HINT_EVICT_FIRST;   // weights: streamed once per launch
    const int ntile_n = static_cast<int>(ceil_div(I, BN / 2));
    // launches over rows_in_l2 rows of X, each sweeping all of W_g, W_u over rows that stay in L2
    const int64_t sub = rows_in_l2(H, T);
    for (int64_t m0 = 0; m0 < T; m0 += sub) {
        const int ml = static_cast<int>(std::min<int64_t>(sub, T - m0));
        CUtensorMap mX;
        if ((rc = make_map(&mX, static_cast<const __nv_bfloat16*>(X) + m0 * H, H, ml, H, BK, BM))) return rc;
        EpiParams f = e;
        f.M = ml;
        f.out = e.out + m0 * I;
        if (e.out2 != nullptr) f.out2 = e.out2 + m0 * I;
        if (e.out3 != nullptr) f.out3 = e.out3 + m0 * I;
        if ((rc = launch_gemm<0, 0, EPI_SWIGLU, 1>(mX, mG, ml, ntile_n * BN, static_cast<int>(H), f, as_stream(stream),
                                                   0, &mX, &mU)))
            return rc;
    }
    return LIGER_OK;
}

// dX = dG W_g + dU W_u (one GEMM over K = 2I) and dW_g = dG^T X, dW_u = dU^T X,
// from dG and dU [T, I] bf16.
int grads_from_dgdu(const void* X, const void* Wg, const void* Wu, const __nv_bfloat16* dG,
                    const __nv_bfloat16* dU, void* dX, void* dWg, void* dWu, int64_t T, int64_t H, int64_t I,
                    int* d_err, cudaStream_t st) {
    using namespace tc;
    int rc;
    CUtensorMap mdG_k, mdU_k, mG_mn, mU_mn;
    if ((rc = make_map(&mdG_k, dG, I, T, I, BK, BM))) return rc;
    if ((rc = make_map(&mdU_k, dU, I, T, I, BK, BM))) return rc;
    if ((rc = make_map(&mG_mn, Wg, H, I, H, MN_BOX, BK))) return rc;
    if ((rc = make_map(&mU_mn, Wu, H, I, H, MN_BOX, BK))) return rc;
    const int nkb1 = static_cast<int>(ceil_div(I, BK));
    EpiParams d{};
    d.err = d_err;
    d.M = static_cast<int>(T);
    d.N = static_cast<int>(H);
    d.out = static_cast<__nv_bfloat16*>(dX);
    d.ldo = H;
    d.ksplit_nkb = nkb1;
    d.raster = RASTER_N_GROUPS;
    if ((rc = launch_gemm<0, 1, EPI_STORE, 1>(mdG_k, mG_mn, static_cast<int>(T), static_cast<int>(H), 2 * nkb1 * BK,
                                              d, st, 0, &mdU_k, &mU_mn)))
        return rc;
    CUtensorMap mdG_mn, mdU_mn, mX_mn;
    if ((rc = make_map(&mdG_mn, dG, I, T, I, MN_BOX, BK))) return rc;
    if ((rc = make_map(&mdU_mn, dU, I, T, I, MN_BOX, BK))) return rc;
    if ((rc = make_map(&mX_mn, X, H, T, H, MN_BOX, BK))) return rc;
    EpiParams w{};
    w.err = d_err;
    w.M = static_cast<int>(I);
    w.N = static_cast<int>(H);
    w.ldo = H;
    w.out_write = 1;
    // n fastest touches all of X in every wave: fine while X stays in L2 (up to 32 MiB), above
    // that groups of 8 column blocks of it do (each dG / dU block is then read once per group)
    w.raster = T * H * 2 > (int64_t{32} << 20) ? RASTER_N_GROUPS : RASTER_N_FASTEST;
    w.hint_a = HINT_EVICT_FIRST;
    w.hint_b = HINT_EVICT_LAST;   // X: reused by every row block
    // dW_g and dW_u in one launch: the row blocks of dU^T follow those of dG^T (2 x 43
    // row blocks at intermediate 11008: 1376 tiles fill 18.1 waves of the 76 CTA pairs,
    // where two launches of 688 tiles fill 9.05 waves each)
    const int mt = static_cast<int>(ceil_div(I, static_cast<int64_t>(TileCfg<1>::TM)));
    w.out = static_cast<__nv_bfloat16*>(dWg);
    w.out2 = static_cast<__nv_bfloat16*>(dWu);
    w.msplit_mt = mt;
    w.M2 = static_cast<int>(I);
    return launch_gemm<1, 1, EPI_ACCUM, 1>(mdG_mn, mX_mn, mt * TileCfg<1>::TM + static_cast<int>(I),
                                           static_cast<int>(H), static_cast<int>(T), w, st, 0, &mdU_mn, &mX_mn);
}

}  // namespace
}  // namespace liger

extern "C" int liger_fused_linear_swiglu_fwd(const void* X, const void* Wg, const void* Wu, void* out, int64_t T,
                                             int64_t H, int64_t I, int dtype, void* stream) {
    clear_error();
    return fwd_impl(X, Wg, Wu, out, nullptr, nullptr, T, H, I, dtype, stream, "fused_linear_swiglu_fwd");
}

extern "C" int liger_fused_linear_swiglu_fwd_save(const void* X, const void* Wg, const void* Wu, void* out, void* g,
                                                  void* u, int64_t T, int64_t H, int64_t I, int dtype,
                                                  void* stream) {
    clear_error();
    if (T > 0 && (!g || !u)) return fail(LIGER_ERR_NULL, "fused_linear_swiglu_fwd_save: g and u are required");
    return fwd_impl(X, Wg, Wu, out, g, u, T, H, I, dtype, stream, "fused_linear_swiglu_fwd_save");
}

extern "C" size_t liger_fused_linear_swiglu_workspace(int64_t T, int64_t I) {
    if (T <= 0 || I <= 0) return 0;
    return 2 * ((static_cast<size_t>(T) * static_cast<size_t>(I) * 2 + 255) & ~static_cast<size_t>(255));
}

extern "C" int liger_fused_linear_swiglu_bwd(const void* X, const void* Wg, const void* Wu, const void* dH, void* dX,
                                             void* dWg, void* dWu, void* ws, size_t ws_bytes, int64_t T, int64_t H,
                                             int64_t I, int dtype, void* stream) {
    clear_error();
    if (int rc = check_shapes(T, H, I, dtype, "fused_linear_swiglu_bwd")) return rc;
    if (!Wg || !Wu || !dWg || !dWu || (T > 0 && (!X || !dH || !dX)))
        return fail(LIGER_ERR_NULL, "fused_linear_swiglu_bwd: null tensor pointer");
    if (!aligned16(X) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(dH) || !aligned16(dX) || !aligned16(dWg) ||
        !aligned16(dWu))
        return fail(LIGER_ERR_ALIGN, "fused_linear_swiglu_bwd: tensors must be 16-byte aligned");
    const size_t need = liger_fused_linear_swiglu_workspace(T, I);
    if (need > 0 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)))
        return fail(LIGER_ERR_WORKSPACE, "fused_linear_swiglu_bwd: workspace of %zu bytes (256-byte aligned) "
                    "required, got %zu", need, ws_bytes);
    cudaStream_t st = as_stream(stream);
    if (T == 0) {
        const size_t wb = static_cast<size_t>(I * H) * 2;
        if (cudaMemsetAsync(dWg, 0, wb, st) != cudaSuccess || cudaMemsetAsync(dWu, 0, wb, st) != cudaSuccess)
            return check_launch("fused_linear_swiglu_bwd memset");
        return LIGER_OK;
    }
    int* d_err = nullptr;
    if (int rc0 = lsw_err_word(&d_err)) return rc0;
    __nv_bfloat16* dG = static_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* dU = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + need / 2);
    int rc;
    // 1. recompute g, u; dG, dU from dh (in launches over rows_in_l2 rows of X, as the forward)
    CUtensorMap mG_k, mU_k;
    if ((rc = make_map(&mG_k, Wg, H, I, H, BK, BN / 2))) return rc;
    if ((rc = make_map(&mU_k, Wu, H, I, H, BK, BN / 2))) return rc;
    EpiParams e{};
    e.err = d_err;
    e.M = static_cast<int>(T);
    e.N = static_cast<int>(I);
    e.out = dG;
    e.out2 = dU;
    e.ldo = I;
    e.src = static_cast<const __nv_bfloat16*>(dH);
    e.lds = I;
    e.bsplit = 1;
    e.raster = RASTER_M_FASTEST;
    e.hint_a = HINT_EVICT_LAST;
    e.hint_b = HINT_EVICT_FIRST;
    const int ntile_n = static_cast<int>(ceil_div(I, BN / 2));
    const int64_t sub = rows_in_l2(H, T);
    for (int64_t m0 = 0; m0 < T; m0 += sub) {
        const int ml = static_cast<int>(std::min<int64_t>(sub, T - m0));
        CUtensorMap mX_k;
        if ((rc = make_map(&mX_k, static_cast<const __nv_bfloat16*>(X) + m0 * H, H, ml, H, BK, BM))) return rc;
        EpiParams f = e;
        f.M = ml;
        f.out = dG + m0 * I;
        f.out2 = dU + m0 * I;
        f.src = static_cast<const __nv_bfloat16*>(dH) + m0 * I;
        if ((rc = launch_gemm<0, 0, EPI_SWIGLU_BWD, 1>(mX_k, mG_k, ml, ntile_n * BN, static_cast<int>(H), f, st, 0,
                                                       &mX_k, &mU_k)))
            return rc;
    }
    // 2. dX = dG W_g + dU W_u (K = 2I: k-blocks of the second product follow those of the first);
    // 3. dW_g = dG^T X, dW_u = dU^T X (both operands MN-major, K = T)
    return grads_from_dgdu(X, Wg, Wu, dG, dU, dX, dWg, dWu, T, H, I, d_err, st);
}

extern "C" int liger_fused_linear_swiglu_bwd_saved(const void* X, const void* Wg, const void* Wu, const void* dH,
                                                   const void* g, const void* u, void* dX, void* dWg, void* dWu,
                                                   void* ws, size_t ws_bytes, int64_t T, int64_t H, int64_t I,
                                                   int dtype, void* stream) {
    clear_error();
    const char* who = "fused_linear_swiglu_bwd_saved";
    if (int rc = check_shapes(T, H, I, dtype, who)) return rc;
    if (!Wg || !Wu || !dWg || !dWu || (T > 0 && (!X || !dH || !g || !u || !dX)))
        return fail(LIGER_ERR_NULL, "%s: null tensor pointer", who);
    if (!aligned16(X) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(dH) || !aligned16(g) || !aligned16(u) ||
        !aligned16(dX) || !aligned16(dWg) || !aligned16(dWu))
        return fail(LIGER_ERR_ALIGN, "%s: tensors must be 16-byte aligned", who);
    const size_t need = liger_fused_linear_swiglu_workspace(T, I);
    if (need > 0 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)))
        return fail(LIGER_ERR_WORKSPACE, "%s: workspace of %zu bytes (256-byte aligned) required, got %zu", who, need,
                    ws_bytes);
    cudaStream_t st = as_stream(stream);
    if (T == 0) {
        const size_t wb = static_cast<size_t>(I * H) * 2;
        if (cudaMemsetAsync(dWg, 0, wb, st) != cudaSuccess || cudaMemsetAsync(dWu, 0, wb, st) != cudaSuccess)
            return check_launch("fused_linear_swiglu_bwd_saved memset");
        return LIGER_OK;
    }
    int* d_err = nullptr;
    if (int rc0 = lsw_err_word(&d_err)) return rc0;
    __nv_bfloat16* dG = static_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* dU = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + need / 2);
    // 1. dG, dU from dh and the saved g, u (the elementwise SwiGLU backward)
    if (int rc = liger_swiglu_bwd(dH, g, u, dG, dU, T * I, LIGER_BF16, stream)) return rc;
    // 2-3. as in the backward with recompute
    return grads_from_dgdu(X, Wg, Wu, dG, dU, dX, dWg, dWu, T, H, I, d_err, st);
}
