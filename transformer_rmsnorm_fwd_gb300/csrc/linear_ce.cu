// Fused linear cross-entropy, forward and backward, token-chunked.
//
// Operator: the FusedCrossEntropyLoss paragraph of the page "Liger-Kernel核心
// 技术：RollingBuffer与融合算子详解", section "算子融合" -- softmax and NLL in one
// step on the classifier-head output, the softmax never stored -- with the
// online softmax merge (running maximum and rescaled normaliser per tile) of
// the page "Liger-Kernel内核级优化：FlashAttention与RollingBuffer详解".
//
// bf16 path (tensor cores), per chunk of C tokens (rows t0 .. t0+C):
//   1. Z_c = X_c W^T on tcgen05; the epilogue never stores z: per 256-wide
//      vocab tile it keeps the row max m and sum s of exp(z - m), writes
//      P = exp(z - m) in bf16 to the [C x V] chunk buffer, and the logit at
//      the label in fp32;
//   2. one block per row merges the (m, s) of all vocab tiles into lse, the
//      row's loss term, and rewrites P in place into the softmax part of D,
//      S = scale * P * exp(m_tile - lse) (bf16);
//   3. dX_c = S W on tcgen05 (W read MN-major); the epilogue subtracts the
//      one-hot part, scale * W[label], in fp32; ignored rows written +0;
//   4. dW (+)= S^T X_c on tcgen05 (both operands MN-major); the epilogue
//      subtracts scale * X_t for the tokens labelled with the row (the chunk's
//      labels sorted once, indexed by a [V+1] start table) in fp32, and
//      prefetches and accumulates across chunks in
//      an fp32 [V x H] workspace, the last chunk writing W's dtype.
// Keeping the one-hot term out of the bf16 operand matters: rounding
// -scale to bf16 at every label would cost up to 2^-9 relative on the rows of
// dW and dX that dominate their magnitude.
// The full [T x V] logits never exist; per chunk only [C x V] bf16 does.
//
// fp32 path (and bf16 with H not a multiple of 8): the same steps with an
// fp32 SIMT GEMM and an fp32 [C x V] chunk buffer holding z, then D.  TF32
// tensor cores would miss the 1e-5 fp32 tolerance, so fp32 stays on FMA.
#include <math.h>

#include <atomic>

#include "tc_gemm.cuh"

namespace liger {

namespace {

constexpr int kVT = tc::BN;   // vocab tile of the (m, s) partials
constexpr int kMaxSortKeys = 8192;      // label keys sorted per block (shared memory)
constexpr int64_t kAutoChunkTC = 8192;   // tensor-core path: most rows per chunk chosen automatically
constexpr int64_t kMaxChunkTC = 65536;   // tensor-core path: most rows per chunk a caller may ask for
// The dX GEMM's K is the whole vocabulary: over 150 k vocabulary rows the tiles of a
// wave drift apart along K and stop sharing their D and W slices through L2 (it read
// 4-6x its operand bytes from DRAM).  Above this many vocabulary rows it runs in
// launches over equal slabs of at most this many rows (0: one launch), the partial sums
// kept in an fp32 [chunk x H] buffer; each launch starts the wave's tiles together.
constexpr int64_t kDxSlabRows = 65536;

// vocabulary rows per dX launch: V itself, or equal slabs (multiples of 256) of at most kDxSlabRows
int64_t dx_slab(int64_t V) {
    if (kDxSlabRows <= 0 || V <= kDxSlabRows) return V;
    const int64_t n = (V + kDxSlabRows - 1) / kDxSlabRows;
    return ((V + n - 1) / n + 255) / 256 * 256;
}

struct Hdr {
    unsigned long long n_valid;
    int bad;
    int err;
    float scale;   // the gradient scale, when it is formed on the device (no host wait)
};

struct Layout {
    bool tc;
    int64_t C, ldp, nvt, nchunks;
    int seg;   // label-sort segment: the chunk (C <= 8192, indices relative to it) or 8192 tokens (absolute)
    size_t lse, lossrow, zlab, hdr, labs, keys, lstart, part, scr, acc, dxacc, total;
};

inline size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool use_tc(int64_t H, int64_t V, int dtype) { return dtype == LIGER_BF16 && H % 8 == 0 && H >= 64 && V >= 256; }

Layout layout(int64_t T, int64_t H, int64_t V, int64_t chunk, int dtype) {
    Layout L{};
    L.tc = use_tc(H, V, dtype);
    int64_t C;
    if (chunk > 0) C = chunk;
    // automatic: at most half the tokens (never all T rows at once, for T > 128), at most kAutoChunkTC rows
    else if (L.tc) {
        C = std::min<int64_t>(kAutoChunkTC, std::max<int64_t>(128, (T + 1) / 2));
        // large chunks in whole 256-row tiles of the CTA-pair GEMMs (7373 tokens: 3840 + 3533
        // rows, 15 + 14 row tiles, rather than 2 x 3687 rows in 15 + 15)
        if (C >= 1024) C = std::min<int64_t>(kAutoChunkTC, (C + 255) / 256 * 256);
    }
    else C = std::max<int64_t>(128, (int64_t{1} << 26) / std::max<int64_t>(V, 1));
    if (L.tc) {
        C = std::min<int64_t>(C, kMaxChunkTC);
        // above one label-sort block, whole blocks (the chunk's labels are sorted block by block)
        if (C > kMaxSortKeys && C < T) C = (C / kMaxSortKeys) * kMaxSortKeys;
    }
    C = std::max<int64_t>(1, std::min(C, std::max<int64_t>(T, 1)));
    L.C = C;
    L.seg = static_cast<int>(std::min<int64_t>(C, kMaxSortKeys));
    L.nchunks = T > 0 ? ceil_div(T, C) : 0;
    L.ldp = L.tc ? ((V + 7) / 8) * 8 : V;
    L.nvt = ceil_div(V, kVT);
    size_t o = 0;
    L.lse = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.lossrow = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.zlab = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.hdr = o; o = up256(o + sizeof(Hdr));
    // the labels with bad ones replaced by ignore_index (the entry points that do not wait)
    L.labs = o; o = up256(o + sizeof(int64_t) * static_cast<size_t>(T));
    // every chunk's sorted label keys and start table, made in one pass before the chunks
    L.keys = o; o = up256(o + (L.tc ? sizeof(unsigned long long) * static_cast<size_t>(std::max<int64_t>(T, 1)) : 0));
    L.lstart = o; o = up256(o + (L.tc ? sizeof(int) * static_cast<size_t>(ceil_div(std::max<int64_t>(T, 1), L.seg) * (V + 1)) : 0));
    L.part = o; o = up256(o + (L.tc ? sizeof(float2) * static_cast<size_t>(C * L.nvt) : 0));
    L.scr = o; o = up256(o + static_cast<size_t>(C) * static_cast<size_t>(L.ldp) * (L.tc ? 2 : 4));
    const bool need_acc = L.nchunks > 1 && dtype == LIGER_BF16;
    L.acc = o; o = up256(o + (need_acc ? sizeof(float) * static_cast<size_t>(V * H) : 0));
    const bool dx_slabs = L.tc && dx_slab(V) < V;
    L.dxacc = o; o = up256(o + (dx_slabs ? sizeof(float) * static_cast<size_t>(C * H) : 0));
    L.total = o;
    return L;
}

// Workspace of the waiting tensor-core entry points, which run their GEMMs on the
// tokens that are not ignored only: the ordinary layout's lse, loss_row and header
// first (lse and loss_row of every token, as documented), then the region the
// variant runs in for those tokens (at most the ordinary layout's size), then
// their X rows, their dX rows, their labels and the index maps.
struct CompactLayout {
    size_t core, xc, dxc, labc, idx, inv, cnt, total;
};

constexpr int kCompactBlock = 1024;   // tokens per block of the compaction's index pass

// core_at: where the ordinary layout's per-call part ends (after lse, loss_row, z_label
// and the header); core_total: the ordinary layout's size for all T tokens
CompactLayout compact_regions(size_t core_at, size_t core_total, int64_t T, int64_t H, size_t esz) {
    const size_t t = static_cast<size_t>(std::max<int64_t>(T, 1));
    CompactLayout C{};
    size_t o = core_at;
    C.core = o; o = up256(o + core_total);
    C.xc = o; o = up256(o + t * static_cast<size_t>(H) * esz);
    C.dxc = o; o = up256(o + t * static_cast<size_t>(H) * esz);
    C.labc = o; o = up256(o + t * sizeof(int64_t));
    C.idx = o; o = up256(o + t * sizeof(int64_t));
    C.inv = o; o = up256(o + t * sizeof(int));
    C.cnt = o; o = up256(o + sizeof(int) * static_cast<size_t>(ceil_div(static_cast<int64_t>(t), int64_t{kCompactBlock})));
    C.total = o;
    return C;
}

CompactLayout compact_layout(int64_t T, int64_t H, int64_t V, int64_t chunk, int dtype) {
    const Layout L = layout(T, H, V, chunk, dtype);
    return compact_regions(L.labs, L.total, T, H, dtype == LIGER_F32 ? 4 : 2);
}

// ---------------------------------------------------------------- kernels
// ---- compaction of the tokens that are not ignored (stable: their order is kept)
__global__ void __launch_bounds__(kCompactBlock) compact_count(const int64_t* __restrict__ labels, int64_t T,
                                                               int64_t ignore, int* __restrict__ cnt) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kCompactBlock + threadIdx.x;
    const int c = __syncthreads_count(t < T && labels[t] != ignore);
    if (threadIdx.x == 0) cnt[blockIdx.x] = c;
}

// cnt[0, nb) -> exclusive prefix sums, in place (one block of 1024 threads)
__global__ void __launch_bounds__(1024) compact_scan(int* cnt, int64_t nb) {
    __shared__ int sums[1024];
    const int64_t per = (nb + 1023) / 1024;
    const int64_t b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
    int s = 0;
    for (int64_t b = b0; b < b1; ++b) s += cnt[b];
    sums[threadIdx.x] = s;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int v = threadIdx.x >= o ? sums[threadIdx.x - o] : 0;
        __syncthreads();
        sums[threadIdx.x] += v;
        __syncthreads();
    }
    int run = threadIdx.x ? sums[threadIdx.x - 1] : 0;
    for (int64_t b = b0; b < b1; ++b) {
        const int c = cnt[b];
        cnt[b] = run;
        run += c;
    }
}

// idx[p] = t and lab_c[p] = labels[t] for the p-th token that is not ignored; inv[t] = p, or -1
__global__ void __launch_bounds__(kCompactBlock) compact_index(const int64_t* __restrict__ labels, int64_t T,
                                                               int64_t ignore, const int* __restrict__ off,
                                                               int64_t* __restrict__ idx, int* __restrict__ inv,
                                                               int64_t* __restrict__ lab_c) {
    __shared__ int wsum[kCompactBlock / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kCompactBlock + threadIdx.x;
    const int64_t y = t < T ? labels[t] : ignore;
    const bool v = t < T && y != ignore;
    const unsigned m = __ballot_sync(0xffffffffu, v);
    if (lane == 0) wsum[wid] = __popc(m);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < wid; ++w) before += wsum[w];
    const int p = off[blockIdx.x] + before + __popc(m & ((1u << lane) - 1u));
    if (v) {
        idx[p] = t;
        lab_c[p] = y;
    }
    if (t < T) inv[t] = v ? p : -1;
}

// rows (16-byte vectors, hv per row): dst[r] = src[idx[r]], r < n
__global__ void gather_rows(const uint4* __restrict__ src, const int64_t* __restrict__ idx, int64_t n, int64_t hv,
                            uint4* __restrict__ dst) {
    for (int64_t r = blockIdx.x; r < n; r += gridDim.x) {
        const uint4* s = src + idx[r] * hv;
        uint4* d = dst + r * hv;
        for (int64_t v = threadIdx.x; v < hv; v += blockDim.x) d[v] = ldg16_nc(s + v);
    }
}

// rows back in place: dst[t] = src[inv[t]], or +0 where inv[t] < 0 (an ignored token)
__global__ void scatter_rows(const uint4* __restrict__ src, const int* __restrict__ inv, int64_t T, int64_t hv,
                             uint4* __restrict__ dst) {
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int p = inv[t];
        uint4* d = dst + t * hv;
        if (p < 0) {
            for (int64_t v = threadIdx.x; v < hv; v += blockDim.x) d[v] = make_uint4(0, 0, 0, 0);
        } else {
            const uint4* s = src + static_cast<int64_t>(p) * hv;
            for (int64_t v = threadIdx.x; v < hv; v += blockDim.x) d[v] = ldg16_nc(s + v);
        }
    }
}

// lse and loss_row of every token from those of the tokens that were run (+0 where ignored),
// and the run's kernel error word into the entry point's header
__global__ void scatter_rowvals(const float* __restrict__ lse_c, const float* __restrict__ loss_c,
                                const int* __restrict__ inv, int64_t T, float* __restrict__ lse,
                                float* __restrict__ loss, const int* core_err, int* err) {
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int p = inv[t];
        lse[t] = p < 0 ? 0.f : lse_c[p];
        loss[t] = p < 0 ? 0.f : loss_c[p];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && *core_err != 0) atomicExch(err, *core_err);
}

// Counts the labels that are not ignore_index and flags any outside [0, V).  With
// lab_out set, also writes the labels with every bad one replaced by ignore_index
// (and not counted), so that no later kernel indexes with it.
__global__ void label_scan(const int64_t* __restrict__ labels, int64_t T, int64_t V, int64_t ignore, Hdr* hdr,
                           int64_t* __restrict__ lab_out) {
    unsigned long long cnt = 0;
    int bad = 0;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t y = labels[t];
        if (y != ignore && (y < 0 || y >= V)) {
            bad = 1;
            if (lab_out != nullptr) y = ignore;
        }
        if (lab_out != nullptr) lab_out[t] = y;
        if (y != ignore) ++cnt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (cnt) atomicAdd(&hdr->n_valid, cnt);
        if (bad) atomicOr(&hdr->bad, 1);
    }
}

// The gradient scale from the device-side count: grad_scale / n_valid (mean; 0 when
// nothing is valid) or grad_scale (sum)
__global__ void ce_scale(Hdr* hdr, int reduction, float grad_scale) {
    const unsigned long long n = hdr->n_valid;
    hdr->scale = reduction == 0 ? (n > 0 ? static_cast<float>(static_cast<double>(grad_scale) / static_cast<double>(n))
                                         : 0.0f)
                                : grad_scale;
}

template <int NT>
__device__ __forceinline__ float block_reduce(float v, bool is_max, float* sh) {
    v = is_max ? warp_max(v) : warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    float r = is_max ? -INFINITY : 0.f;
    for (int i = 0; i < NT / 32; ++i) r = is_max ? fmaxf(r, sh[i]) : r + sh[i];
    return r;
}

// Sort the (label << 32 | token) keys of each segment of seg tokens (ignored
// tokens -> ~0), one block per segment (bitonic, in shared memory), for the
// one-hot correction of the dW epilogue.  Segment b covers tokens
// [b*seg, min(n, (b+1)*seg)) and its sorted keys go to out[b*seg ...]; the
// token index in a key is absolute (b*seg + i) or relative to the segment (i).
__global__ void __launch_bounds__(1024) sort_label_keys(const int64_t* __restrict__ labels, int64_t n, int seg,
                                                        int64_t ignore, int absolute,
                                                        unsigned long long* __restrict__ out) {
    extern __shared__ unsigned long long sk[];
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * seg;
    const int cnt = static_cast<int>(n - b0 < seg ? n - b0 : seg);
    int npow2 = 1;
    while (npow2 < cnt) npow2 <<= 1;
    const unsigned base = absolute ? static_cast<unsigned>(b0) : 0u;
    for (int i = threadIdx.x; i < npow2; i += 1024) {
        unsigned long long key = ~0ull;
        if (i < cnt) {
            const int64_t y = labels[b0 + i];
            if (y != ignore) key = (static_cast<unsigned long long>(y) << 32) | (base + static_cast<unsigned>(i));
        }
        sk[i] = key;
    }
    __syncthreads();
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < npow2; i += 1024) {
                const int p = i ^ j;
                if (p > i) {
                    const bool up = (i & k) == 0;
                    const unsigned long long a = sk[i], b = sk[p];
                    if ((a > b) == up) {
                        sk[i] = b;
                        sk[p] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < cnt; i += 1024) out[b0 + i] = sk[i];
}

// Start tables of every segment (blockIdx.y): lstart[s*(V+1) + v] = first index
// of label v among segment s's sorted keys, v in [0, V], plus s*seg when the
// indices are absolute -- so the tokens of segment s labelled v are
// keys[lstart[v] .. lstart[v+1]) of the array the table's indices refer to.
__global__ void label_starts(const unsigned long long* __restrict__ keys, int64_t n, int seg, int V, int absolute,
                             int* __restrict__ lstart) {
    const int64_t b0 = static_cast<int64_t>(blockIdx.y) * seg;
    const int cnt = static_cast<int>(n - b0 < seg ? n - b0 : seg);
    const unsigned long long* k = keys + b0;
    int* ls = lstart + static_cast<int64_t>(blockIdx.y) * (V + 1);
    const int base = absolute ? static_cast<int>(b0) : 0;
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v <= V; v += gridDim.x * blockDim.x) {
        const unsigned long long key = static_cast<unsigned long long>(v) << 32;
        int lo = 0, hi = cnt;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (k[mid] < key) lo = mid + 1;
            else hi = mid;
        }
        ls[v] = base + lo;
    }
}

// Sorted keys and start tables of all nseg segments of seg tokens, in two launches.
int sort_labels(const int64_t* labels, int64_t n, int seg, int64_t ignore, int V, bool absolute,
                unsigned long long* keys, int* lstart, cudaStream_t st) {
    const int64_t nseg = ceil_div(n, static_cast<int64_t>(seg));
    if (nseg <= 0) return LIGER_OK;
    int npow2 = 1;
    while (npow2 < seg) npow2 <<= 1;
    sort_label_keys<<<static_cast<unsigned>(nseg), 1024, sizeof(unsigned long long) * npow2, st>>>(
        labels, n, seg, ignore, absolute ? 1 : 0, keys);
    if (int rc = check_launch("sort_label_keys")) return rc;
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>(ceil_div(V + 1, 256), 2 * sm_count())),
                    static_cast<unsigned>(nseg));
    label_starts<<<grid, 256, 0, st>>>(keys, n, seg, V, absolute ? 1 : 0, lstart);
    return check_launch("label_starts");
}

// Merge the per-tile (m, s) of one chunk row into lse and rewrite P in place
// into the softmax part of D, scale * P * exp(m_tile - lse) (the one-hot part
// is applied exactly, in fp32, by the dX / dW GEMM epilogues).  P null: lse
// and the loss term only.
constexpr int kRowThreads = 256;
__global__ void __launch_bounds__(kRowThreads) dlogits_bf16(const int64_t* __restrict__ labels, int64_t ignore,
                                                            const float2* __restrict__ part, int nvt,
                                                            const float* __restrict__ zlab, __nv_bfloat16* P,
                                                            int64_t ldp, int V, float scale,
                                                            const float* __restrict__ scale_dev,
                                                            float* __restrict__ lse, float* __restrict__ lossrow) {
    extern __shared__ float fac[];   // [nvt]
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int64_t y = labels[row];
    __nv_bfloat16* prow = P + row * ldp;
    const int nv8 = (V + 7) / 8;
    if (y == ignore) {
        if (P != nullptr)
            for (int k = threadIdx.x; k < nv8; k += kRowThreads)
                stg16(prow + static_cast<int64_t>(k) * 8, make_uint4(0, 0, 0, 0));
        if (threadIdx.x == 0) {
            lse[row] = 0.f;
            lossrow[row] = 0.f;
        }
        return;
    }
    const float2* pr = part + row * nvt;
    float m = -INFINITY;
    for (int j = threadIdx.x; j < nvt; j += kRowThreads) m = fmaxf(m, pr[j].x);
    m = block_reduce<kRowThreads>(m, true, red);
    float s = 0.f;
    for (int j = threadIdx.x; j < nvt; j += kRowThreads) {
        const float2 p = pr[j];
        s += p.y * expf(p.x - m);
    }
    s = block_reduce<kRowThreads>(s, false, red);
    const float l = m + logf(s);
    const float sc = scale_dev != nullptr ? *scale_dev : scale;   // scale_dev: formed on the device
    for (int j = threadIdx.x; j < nvt; j += kRowThreads) fac[j] = sc * expf(pr[j].x - l);
    if (threadIdx.x == 0) {
        lse[row] = l;
        lossrow[row] = l - zlab[row];
    }
    if (P == nullptr) return;   // lse and the loss term only
    __syncthreads();
    for (int k = threadIdx.x; k < nv8; k += kRowThreads) {
        const int col = k * 8;
        const float f = fac[col / kVT];
        float v[8];
        unpack(ldg16(prow + col), v);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] *= f;
        stg16(prow + col, pack(v));
    }
}

// fp32 path: z row -> lse, loss term, D (fp32, in place).
__global__ void __launch_bounds__(kRowThreads) dlogits_f32(const int64_t* __restrict__ labels, int64_t ignore,
                                                           float* Z, int64_t ldz, int V, float scale,
                                                           const float* __restrict__ scale_dev,
                                                           float* __restrict__ lse, float* __restrict__ lossrow) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int64_t y = labels[row];
    float* z = Z + row * ldz;
    if (y == ignore) {
        for (int v = threadIdx.x; v < V; v += kRowThreads) z[v] = 0.f;
        if (threadIdx.x == 0) {
            lse[row] = 0.f;
            lossrow[row] = 0.f;
        }
        return;
    }
    float m = -INFINITY;
    for (int v = threadIdx.x; v < V; v += kRowThreads) m = fmaxf(m, z[v]);
    m = block_reduce<kRowThreads>(m, true, red);
    float s = 0.f;
    for (int v = threadIdx.x; v < V; v += kRowThreads) s += expf(z[v] - m);
    s = block_reduce<kRowThreads>(s, false, red);
    const float l = m + logf(s);
    const float zy = z[y];
    __syncthreads();   // every thread has read z[y] before it is overwritten
    if (threadIdx.x == 0) {
        lse[row] = l;
        lossrow[row] = l - zy;
    }
    const float sc = scale_dev != nullptr ? *scale_dev : scale;   // scale_dev: formed on the device
    for (int v = threadIdx.x; v < V; v += kRowThreads) z[v] = sc * (expf(z[v] - l) - (v == y ? 1.0f : 0.0f));
}

// loss = sum of the row terms (fixed order, fp64) / n_valid; NaN if a
// tensor-core kernel recorded an error.
// dev_denom 0: divide by denom; 1 (mean) / 2 (sum): the denominator from the device-side
// count, and NaN when a label was bad
__global__ void __launch_bounds__(1024) loss_final(const float* __restrict__ lossrow, int64_t T, double denom,
                                                   const Hdr* hdr, float* loss, int dev_denom) {
    __shared__ double red[32];
    double s = 0.0;
    for (int64_t t = threadIdx.x; t < T; t += 1024) s += static_cast<double>(lossrow[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int i = 0; i < 32; ++i) tot += red[i];
        if (dev_denom != 0) denom = dev_denom == 1 ? static_cast<double>(hdr->n_valid) : 1.0;
        float r = denom > 0.0 ? static_cast<float>(tot / denom) : 0.0f;
        if (hdr->err != 0 || (dev_denom != 0 && hdr->bad != 0)) r = __int_as_float(0x7fc00000);
        *loss = r;
    }
}

// Generic SIMT GEMM, C[m, n] = sum_k A(m, k) B(k, n), fp32 accumulation.
// A(m, k) = A[m*sam + k*sak], B(k, n) = B[k*sbk + n*sbn].
//  mode 0: outf[m, n]  = acc          mode 2: outf[m, n] += acc
//  mode 1: outT[m, n]  = acc          mode 3: outT[m, n]  = acc + outf[m, n]
// mode 1 writes +0 on rows whose label is ignore_index (labels may be NULL).
// SBT x SBT output tiles (64, or 32 when 64-wide tiles would leave SMs idle), 256
// threads each holding (SBT/16)^2 of them; k steps of SKT (16, or 64 with the small
// tiles: fewer load-then-synchronise rounds, more loads in flight in each).
constexpr int SB = 64, SK = 16;
template <typename TA, typename TB, typename TO, int MODE, int SBT, int SKT>
__global__ void __launch_bounds__(256) simt_gemm(int M, int N, int K, const TA* __restrict__ A, int64_t sam,
                                                 int64_t sak, const TB* __restrict__ B, int64_t sbk, int64_t sbn,
                                                 float* outf, TO* outT, int64_t ldo, const int64_t* __restrict__ labels,
                                                 int64_t ignore) {
    constexpr int RT = SBT / 16;
    __shared__ float As[SKT][SBT + 1], Bs[SKT][SBT + 1];
    const int m0 = blockIdx.y * SBT, n0 = blockIdx.x * SBT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[RT][RT] = {};
    const bool ak = sak == 1, bn = sbn == 1;
    for (int k0 = 0; k0 < K; k0 += SKT) {
        // consecutive threads take consecutive elements of each operand's contiguous
        // dimension (k when sak == 1, else m; n when sbn == 1, else k), so the loads coalesce
        // whichever operand is transposed
        for (int i = threadIdx.x; i < SBT * SKT; i += 256) {
            const int mm = ak ? i / SKT : i % SBT, kk = ak ? i % SKT : i / SBT;
            const int gm = m0 + mm, gk = k0 + kk;
            As[kk][mm] = (gm < M && gk < K) ? ldf(A + gm * sam + gk * sak) : 0.f;
            const int nn = bn ? i % SBT : i / SKT, kb = bn ? i / SBT : i % SKT;
            const int gn = n0 + nn, gk2 = k0 + kb;
            Bs[kb][nn] = (gn < N && gk2 < K) ? ldf(B + gk2 * sbk + gn * sbn) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SKT; ++kk) {
            float a[RT], b[RT];
#pragma unroll
            for (int i = 0; i < RT; ++i) a[i] = As[kk][ty * RT + i], b[i] = Bs[kk][tx * RT + i];
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int j = 0; j < RT; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) {
        const int gm = m0 + ty * RT + i;
        if (gm >= M) continue;
        const bool zero = MODE == 1 && labels != nullptr && labels[gm] == ignore;
#pragma unroll
        for (int j = 0; j < RT; ++j) {
            const int gn = n0 + tx * RT + j;
            if (gn >= N) continue;
            const int64_t o = static_cast<int64_t>(gm) * ldo + gn;
            if (MODE == 0) outf[o] = acc[i][j];
            else if (MODE == 1) stf(outT + o, zero ? 0.f : acc[i][j]);
            else if (MODE == 2) outf[o] += acc[i][j];
            else stf(outT + o, acc[i][j] + outf[o]);
        }
    }
}

template <typename TA, typename TB, typename TO, int MODE>
int simt(int M, int N, int K, const TA* A, int64_t sam, int64_t sak, const TB* B, int64_t sbk, int64_t sbn,
         float* outf, TO* outT, int64_t ldo, const int64_t* labels, int64_t ignore, cudaStream_t st) {
    if (M == 0 || N == 0) return LIGER_OK;
    const int64_t tiles64 = ceil_div(N, SB) * ceil_div(M, SB);
    if (tiles64 < sm_count()) {   // too few 64-wide tiles to fill the GPU: 32-wide ones
        dim3 grid(static_cast<unsigned>(ceil_div(N, SB / 2)), static_cast<unsigned>(ceil_div(M, SB / 2)));
        simt_gemm<TA, TB, TO, MODE, SB / 2, 4 * SK><<<grid, 256, 0, st>>>(M, N, K, A, sam, sak, B, sbk, sbn, outf, outT, ldo,
                                                                  labels, ignore);
        return check_launch("simt_gemm");
    }
    dim3 grid(static_cast<unsigned>(ceil_div(N, SB)), static_cast<unsigned>(ceil_div(M, SB)));
    if (grid.y > 65535) return fail(LIGER_ERR_SHAPE, "linear_ce: SIMT grid too large");
    simt_gemm<TA, TB, TO, MODE, SB, SK><<<grid, 256, 0, st>>>(M, N, K, A, sam, sak, B, sbk, sbn, outf, outT, ldo, labels,
                                                          ignore);
    return check_launch("simt_gemm");
}

// ----------------------------------------------------------- orchestration
struct Args {
    const void* X;
    const void* W;
    const int64_t* labels;
    int64_t T, H, V, ignore;
    int reduction;
    float grad_scale;
    float* loss;
    void* dX;
    void* dW;
    uint8_t* ws;
    int dtype;
    cudaStream_t st;
    const float* scale_dev;   // non-null: the gradient scale is read from the device (no host wait)
};

template <typename TI>
int run_simt(const Args& a, const Layout& L, float scale) {
    const TI* X = static_cast<const TI*>(a.X);
    const TI* W = static_cast<const TI*>(a.W);
    TI* dX = static_cast<TI*>(a.dX);
    TI* dW = static_cast<TI*>(a.dW);
    float* lse = reinterpret_cast<float*>(a.ws + L.lse);
    float* lossrow = reinterpret_cast<float*>(a.ws + L.lossrow);
    float* Z = reinterpret_cast<float*>(a.ws + L.scr);
    float* acc = reinterpret_cast<float*>(a.ws + L.acc);
    const bool f32 = a.dtype == LIGER_F32;
    const int H = static_cast<int>(a.H), V = static_cast<int>(a.V);
    int rc;
    for (int64_t c = 0; c < L.nchunks; ++c) {
        const int64_t t0 = c * L.C;
        const int cl = static_cast<int>(std::min(L.C, a.T - t0));
        const bool first = c == 0, last = c == L.nchunks - 1;
        if ((rc = simt<TI, TI, TI, 0>(cl, V, H, X + t0 * H, H, 1, W, 1, H, Z, (TI*)nullptr, V, nullptr, 0, a.st)))
            return rc;
        dlogits_f32<<<cl, kRowThreads, 0, a.st>>>(a.labels + t0, a.ignore, Z, V, V, scale, a.scale_dev, lse + t0,
                                                  lossrow + t0);
        if ((rc = check_launch("dlogits_f32"))) return rc;
        if (dX && (rc = simt<float, TI, TI, 1>(cl, H, V, Z, V, 1, W, H, 1, nullptr, dX + t0 * H, H, a.labels + t0,
                                               a.ignore, a.st)))
            return rc;
        if (dW) {
            const TI* Xc = X + t0 * H;
            if (f32) {
                float* dWf = reinterpret_cast<float*>(dW);
                rc = first ? simt<float, TI, float, 0>(V, H, cl, Z, 1, V, Xc, H, 1, dWf, nullptr, H, nullptr, 0, a.st)
                           : simt<float, TI, float, 2>(V, H, cl, Z, 1, V, Xc, H, 1, dWf, nullptr, H, nullptr, 0, a.st);
            } else if (first && last) {
                rc = simt<float, TI, TI, 1>(V, H, cl, Z, 1, V, Xc, H, 1, nullptr, dW, H, nullptr, 0, a.st);
            } else if (first) {
                rc = simt<float, TI, TI, 0>(V, H, cl, Z, 1, V, Xc, H, 1, acc, nullptr, H, nullptr, 0, a.st);
            } else if (!last) {
                rc = simt<float, TI, TI, 2>(V, H, cl, Z, 1, V, Xc, H, 1, acc, nullptr, H, nullptr, 0, a.st);
            } else {
                rc = simt<float, TI, TI, 3>(V, H, cl, Z, 1, V, Xc, H, 1, acc, dW, H, nullptr, 0, a.st);
            }
            if (rc) return rc;
        }
    }
    return LIGER_OK;
}

int ensure_sort_attr() {
    // per device: function attributes belong to each device's context (racing threads set the same value)
    static std::atomic<bool> done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return check_launch("sort_label_keys device");
    if (!done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(sort_label_keys, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(unsigned long long) * kMaxSortKeys)) != cudaSuccess)
            return check_launch("sort_label_keys attribute");
        done[dev].store(true, std::memory_order_release);
    }
    return LIGER_OK;
}

// Z = X_c W^T for the cl rows at Xc with the logits epilogue e (its labels, zlab,
// part and p_out set for row 0 of the chunk), in launches over rows_in_l2 rows: each
// launch sweeps the whole vocabulary over its rows of X (an 8192-row chunk at hidden
// 4096 takes two launches, reading W twice but each X row once)
int launch_logits(const __nv_bfloat16* Xc, int cl, int H, int V, const CUtensorMap& mW_k, const tc::EpiParams& e,
                  int64_t ldp, int64_t nvt, cudaStream_t st) {
    using namespace tc;
    const int64_t sub = rows_in_l2(H, cl);
    for (int64_t s0 = 0; s0 < cl; s0 += sub) {
        const int sl = static_cast<int>(std::min<int64_t>(sub, cl - s0));
        CUtensorMap mX;
        if (int rc = make_map(&mX, Xc + s0 * H, H, sl, H, BK, BM)) return rc;   // A (K-major)
        EpiParams f = e;
        f.M = sl;
        f.labels = e.labels + s0;
        f.zlab = e.zlab + s0;
        f.part = e.part + s0 * nvt;
        if (e.p_out != nullptr) f.p_out = e.p_out + s0 * ldp;
        if (int rc = launch_gemm<0, 0, EPI_LOGITS, 1>(mX, mW_k, sl, V, H, f, st)) return rc;
    }
    return LIGER_OK;
}

int run_tc(const Args& a, const Layout& L, float scale) {
    using namespace tc;
    if (int rc = ensure_sort_attr()) return rc;
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.X);
    const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.W);
    float* lse = reinterpret_cast<float*>(a.ws + L.lse);
    float* lossrow = reinterpret_cast<float*>(a.ws + L.lossrow);
    float* zlab = reinterpret_cast<float*>(a.ws + L.zlab);
    Hdr* hdr = reinterpret_cast<Hdr*>(a.ws + L.hdr);
    float2* part = reinterpret_cast<float2*>(a.ws + L.part);
    __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(a.ws + L.scr);
    float* acc = reinterpret_cast<float*>(a.ws + L.acc);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(a.ws + L.keys);
    int* lstart = reinterpret_cast<int*>(a.ws + L.lstart);
    const int H = static_cast<int>(a.H), V = static_cast<int>(a.V);
    int rc;
    CUtensorMap mW_k, mW_mn;
    if ((rc = make_map(&mW_k, W, H, V, H, BK, B_BOX_ROWS))) return rc;          // B of Z = X W^T  (K-major)
    if ((rc = make_map(&mW_mn, W, H, V, H, MN_BOX, BK))) return rc;     // B of dX = D W   (MN-major)
    const size_t fac_smem = sizeof(float) * static_cast<size_t>(L.nvt);
    // label keys: one segment per chunk (indices relative to the chunk) up to 8192 rows, else
    // 8192-token segments with absolute indices, several per chunk
    const bool rel = L.seg == L.C;
    if (a.dW && (rc = sort_labels(a.labels, a.T, L.seg, a.ignore, V, !rel, keys, lstart, a.st))) return rc;
    for (int64_t c = 0; c < L.nchunks; ++c) {
        const int64_t t0 = c * L.C;
        const int cl = static_cast<int>(std::min(L.C, a.T - t0));
        const bool first = c == 0, last = c == L.nchunks - 1;
        const __nv_bfloat16* Xc = X + t0 * H;
        CUtensorMap mX_mn, mD_k, mD_mn;
        if ((rc = make_map(&mX_mn, Xc, H, cl, H, MN_BOX, BK))) return rc;  // B of dW (MN-major)
        if ((rc = make_map(&mD_k, P, V, cl, L.ldp, BK, BM))) return rc;  // A of dX (K-major)
        if ((rc = make_map(&mD_mn, P, V, cl, L.ldp, MN_BOX, BK))) return rc;  // A of dW (MN-major)

        EpiParams e{};
        e.err = &hdr->err;
        e.ignore_index = a.ignore;
        e.labels = a.labels + t0;
        // 1. logits -> P, (m, s) partials, z at label
        e.M = cl;
        e.N = V;
        e.raster = RASTER_M_FASTEST;
        e.hint_a = HINT_EVICT_LAST;    // X_c: reused by every vocab tile, keep in L2
        e.hint_b = HINT_EVICT_FIRST;   // W: streamed once per chunk
        e.p_out = P;
        e.ldp = L.ldp;
        e.part = part;
        e.nvt = static_cast<int>(L.nvt);
        e.zlab = zlab + t0;
        if ((rc = launch_logits(Xc, cl, H, V, mW_k, e, L.ldp, L.nvt, a.st))) return rc;
        // 2. lse, loss terms, P -> D in place
        dlogits_bf16<<<cl, kRowThreads, fac_smem, a.st>>>(a.labels + t0, a.ignore, part, static_cast<int>(L.nvt),
                                                          zlab + t0, P, L.ldp, V, scale, a.scale_dev, lse + t0,
                                                          lossrow + t0);
        if ((rc = check_launch("dlogits_bf16"))) return rc;
        // 3. dX_c = D W, minus scale * W[label] in fp32
        if (a.dX && dx_slab(V) < V) {
            // over vocabulary slabs, summed in fp32; the last slab subtracts scale * W[label]
            // and writes dX in bf16
            float* dxacc = reinterpret_cast<float*>(a.ws + L.dxacc);
            const int64_t slab = dx_slab(V);
            for (int64_t v0 = 0; v0 < V; v0 += slab) {
                const int vl = static_cast<int>(std::min<int64_t>(slab, V - v0));
                const bool s_first = v0 == 0, s_last = v0 + vl >= V;
                CUtensorMap mDs_k, mWs_mn;
                if ((rc = make_map(&mDs_k, P + v0, vl, cl, L.ldp, BK, BM))) return rc;     // A: D[:, slab] (K-major)
                if ((rc = make_map(&mWs_mn, W + v0 * H, H, vl, H, MN_BOX, BK))) return rc;  // B: W[slab, :] (MN-major)
                EpiParams d = e;
                d.p_out = nullptr;
                d.M = cl;
                d.N = H;
                d.raster = RASTER_N_GROUPS;
                d.hint_a = HINT_NORMAL;
                d.hint_b = HINT_NORMAL;
                d.acc = dxacc;
                d.lda = H;
                d.acc_read = s_first ? 0 : 1;
                d.acc_write = s_last ? 0 : 1;
                d.out_write = s_last ? 1 : 0;
                d.out = static_cast<__nv_bfloat16*>(a.dX) + t0 * H;
                d.ldo = H;
                d.keys = nullptr;
                d.corr_src = s_last ? W : nullptr;
                d.ld_corr = H;
                d.corr_scale = scale;
                d.scale_ptr = a.scale_dev;
                if ((rc = launch_gemm<0, 1, EPI_ACCUM, 1>(mDs_k, mWs_mn, cl, H, vl, d, a.st))) return rc;
            }
        } else if (a.dX) {
            EpiParams d = e;
            d.M = cl;
            d.N = H;
            d.out = static_cast<__nv_bfloat16*>(a.dX) + t0 * H;
            d.ldo = H;
            d.raster = RASTER_N_GROUPS;
            d.hint_a = HINT_NORMAL;        // D and W: reused within a wave of tiles
            d.hint_b = HINT_NORMAL;
            d.corr_src = W;
            d.ld_corr = H;
            d.corr_scale = scale;
            d.scale_ptr = a.scale_dev;
            if ((rc = launch_gemm<0, 1, EPI_STORE, 1>(mD_k, mW_mn, cl, H, V, d, a.st))) return rc;
        }
        // 4. dW (+)= D^T X_c, minus scale * X_t in fp32 for each token t labelled with the row
        if (a.dW) {
            EpiParams d = e;
            d.ld_corr = H;
            d.corr_scale = scale;
            d.scale_ptr = a.scale_dev;
            d.nkeys = cl;
            if (rel) {
                d.corr_src = Xc;
                d.keys = keys + t0;               // this chunk's keys (token indices relative to the chunk)
                d.lstart = lstart + c * (V + 1);
            } else {
                d.corr_src = X;                   // absolute token indices
                d.keys = keys;
                d.lstart = lstart + (t0 / L.seg) * (V + 1);
                d.nseg = static_cast<int>(ceil_div(static_cast<int64_t>(cl), static_cast<int64_t>(L.seg)));
                d.lstride = V + 1;
            }
            d.M = V;
            d.N = H;
            // n fastest touches all of X_c in every wave: fine while X_c stays in L2 (up to
            // 32 MiB), above that groups of 8 column blocks of it do (at the price of reading
            // each D block once per group)
            d.raster = static_cast<int64_t>(cl) * H * 2 > (int64_t{32} << 20) ? RASTER_N_GROUPS : RASTER_N_FASTEST;
            d.hint_a = HINT_NORMAL;        // D^T (evict-first measured ~1 % slower with CTA-pair tiles)
            d.hint_b = HINT_EVICT_LAST;    // X_c: reused by every vocab row block, keep in L2
            d.labels = nullptr;
            d.acc = acc;
            d.lda = H;
            d.out = static_cast<__nv_bfloat16*>(a.dW);
            d.ldo = H;
            d.acc_read = first ? 0 : 1;
            d.acc_write = last ? 0 : 1;
            d.out_write = last ? 1 : 0;
            if ((rc = launch_gemm<1, 1, EPI_ACCUM, 1>(mD_mn, mX_mn, V, H, cl, d, a.st))) return rc;
        }
    }
    return LIGER_OK;
}

// Where a layout keeps its per-token lse and loss terms and its header.
struct RowVals {
    size_t lse, lossrow, hdr;
};

// A variant's GEMMs on the tokens that are not ignored only (n_valid of T, known on
// the host from the label scan): an ignored token has D = 0, so it adds nothing to
// dW and its dX row, lse and loss term are 0; its logits, which the GEMMs would
// otherwise compute, are not needed.  The tokens are compacted in order (their X
// rows and labels gathered), run_core runs the variant on them in the region C.core
// (its own layout for n_valid tokens, whose lse, loss terms and header sit at cv),
// and dX, lse and the loss terms are put back in place (tv: the full layout's).
template <typename RunCore>
int run_compacted(const Args& a, int64_t n_valid, const CompactLayout& C, const RowVals& tv, const RowVals& cv,
                  RunCore run_core) {
    uint8_t* w8 = a.ws;
    int* cnt = reinterpret_cast<int*>(w8 + C.cnt);
    int64_t* idx = reinterpret_cast<int64_t*>(w8 + C.idx);
    int* inv = reinterpret_cast<int*>(w8 + C.inv);
    int64_t* labc = reinterpret_cast<int64_t*>(w8 + C.labc);
    const int64_t nb = ceil_div(a.T, static_cast<int64_t>(kCompactBlock));
    compact_count<<<static_cast<unsigned>(nb), kCompactBlock, 0, a.st>>>(a.labels, a.T, a.ignore, cnt);
    compact_scan<<<1, 1024, 0, a.st>>>(cnt, nb);
    compact_index<<<static_cast<unsigned>(nb), kCompactBlock, 0, a.st>>>(a.labels, a.T, a.ignore, cnt, idx, inv, labc);
    const int64_t hv = a.H * 2 / 16;   // 16-byte vectors per bf16 row (H is a multiple of 8 on this path)
    const int rgrid = static_cast<int>(std::min<int64_t>(std::max<int64_t>(n_valid, 1), 8 * sm_count()));
    gather_rows<<<rgrid, 256, 0, a.st>>>(static_cast<const uint4*>(a.X), idx, n_valid, hv,
                                         reinterpret_cast<uint4*>(w8 + C.xc));
    if (int rc = check_launch("linear_ce compaction")) return rc;
    Hdr* hc = reinterpret_cast<Hdr*>(w8 + C.core + cv.hdr);
    if (cudaMemsetAsync(hc, 0, sizeof(Hdr), a.st) != cudaSuccess) return check_launch("linear_ce memset");
    Args b = a;
    b.X = w8 + C.xc;
    b.labels = labc;
    b.T = n_valid;
    b.dX = a.dX ? static_cast<void*>(w8 + C.dxc) : nullptr;
    b.ws = w8 + C.core;
    if (int rc = run_core(b)) return rc;
    if (a.dX) {
        const int tgrid = static_cast<int>(std::min<int64_t>(a.T, 8 * sm_count()));
        scatter_rows<<<tgrid, 256, 0, a.st>>>(reinterpret_cast<const uint4*>(w8 + C.dxc), inv, a.T, hv,
                                              static_cast<uint4*>(a.dX));
    }
    const int vgrid = static_cast<int>(std::min<int64_t>(ceil_div(a.T, int64_t{256}), 4 * sm_count()));
    scatter_rowvals<<<vgrid, 256, 0, a.st>>>(reinterpret_cast<const float*>(w8 + C.core + cv.lse),
                                             reinterpret_cast<const float*>(w8 + C.core + cv.lossrow), inv, a.T,
                                             reinterpret_cast<float*>(w8 + tv.lse),
                                             reinterpret_cast<float*>(w8 + tv.lossrow), &hc->err,
                                             &reinterpret_cast<Hdr*>(w8 + tv.hdr)->err);
    return check_launch("linear_ce scatter");
}

// The token-chunked path on the tokens that are not ignored only.
int run_tc_compact(const Args& a, int64_t n_valid, int64_t chunk, float scale) {
    const Layout Lt = layout(a.T, a.H, a.V, chunk, a.dtype);   // the documented lse / loss_row of every token
    const Layout Lc = layout(n_valid, a.H, a.V, chunk, a.dtype);
    if (Lc.total > Lt.total) return run_tc(a, Lt, scale);   // the region holds any layout of fewer tokens
    return run_compacted(a, n_valid, compact_layout(a.T, a.H, a.V, chunk, a.dtype), RowVals{Lt.lse, Lt.lossrow, Lt.hdr},
                         RowVals{Lc.lse, Lc.lossrow, Lc.hdr}, [&](const Args& b) { return run_tc(b, Lc, scale); });
}

// --------------------------------------- two-pass (vocab-chunked) variant
// The same loss and gradients with no [tokens x vocab] buffer at all: pass 1
// computes only lse (the logits GEMM keeps per-tile (m, s) partials, token
// chunk by token chunk); pass 2 recomputes the logits one vocabulary chunk of
// Vc rows at a time for all T tokens, writes the softmax part of D for that
// chunk ([T x Vc] bf16), accumulates dX += D_c W_c in an fp32 [T x H]
// buffer and writes the finished rows dW_c = D_c^T X.  8 T H V flops (the
// logits twice) against 6 T H V for the token-chunked path, and a workspace
// of O(T (H + Vc)) instead of O(C V + V H).
constexpr int64_t kAutoVChunk = 8192;

struct Layout2 {
    int64_t C, nvt, Vc, ldc, nvchunks, nseg;
    size_t lse, lossrow, zlab, hdr, labs, keys, lstart, part, dscr, acc, total;
};

Layout2 layout2(int64_t T, int64_t H, int64_t V, int64_t vchunk) {
    Layout2 L{};
    L.C = std::max<int64_t>(1, std::min<int64_t>(kAutoChunkTC, T));
    L.nvt = ceil_div(V, kVT);
    L.Vc = std::min<int64_t>(vchunk > 0 ? vchunk : kAutoVChunk, V);
    L.ldc = ((L.Vc + 7) / 8) * 8;
    L.nvchunks = ceil_div(V, L.Vc);
    L.nseg = T > 0 ? ceil_div(T, static_cast<int64_t>(kMaxSortKeys)) : 0;
    size_t o = 0;
    L.lse = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.lossrow = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.zlab = o; o = up256(o + sizeof(float) * static_cast<size_t>(T));
    L.hdr = o; o = up256(o + sizeof(Hdr));
    // the labels with bad ones replaced by ignore_index (the entry points that do not wait)
    L.labs = o; o = up256(o + sizeof(int64_t) * static_cast<size_t>(T));
    L.keys = o; o = up256(o + sizeof(unsigned long long) * static_cast<size_t>(T));
    L.lstart = o; o = up256(o + sizeof(int) * static_cast<size_t>(L.nseg * (V + 1)));
    L.part = o; o = up256(o + sizeof(float2) * static_cast<size_t>(L.C * L.nvt));
    L.dscr = o; o = up256(o + 2 * static_cast<size_t>(T) * static_cast<size_t>(L.ldc));
    L.acc = o; o = up256(o + (L.nvchunks > 1 ? sizeof(float) * static_cast<size_t>(T * H) : 0));
    L.total = o;
    return L;
}

int run_two_pass(const Args& a, const Layout2& L, float scale) {
    using namespace tc;
    if (int rc = ensure_sort_attr()) return rc;
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.X);
    const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.W);
    float* lse = reinterpret_cast<float*>(a.ws + L.lse);
    float* lossrow = reinterpret_cast<float*>(a.ws + L.lossrow);
    float* zlab = reinterpret_cast<float*>(a.ws + L.zlab);
    Hdr* hdr = reinterpret_cast<Hdr*>(a.ws + L.hdr);
    float2* part = reinterpret_cast<float2*>(a.ws + L.part);
    __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(a.ws + L.dscr);
    float* acc = reinterpret_cast<float*>(a.ws + L.acc);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(a.ws + L.keys);
    int* lstart = reinterpret_cast<int*>(a.ws + L.lstart);
    const int H = static_cast<int>(a.H), V = static_cast<int>(a.V), T = static_cast<int>(a.T);
    int rc;
    CUtensorMap mW_k;
    if ((rc = make_map(&mW_k, W, H, V, H, BK, B_BOX_ROWS))) return rc;
    // pass 1: lse and the loss terms, token chunk by token chunk (the chunk's X stays in L2)
    const size_t fac_smem = sizeof(float) * static_cast<size_t>(L.nvt);
    for (int64_t t0 = 0; t0 < a.T; t0 += L.C) {
        const int cl = static_cast<int>(std::min(L.C, a.T - t0));
        EpiParams e{};
        e.err = &hdr->err;
        e.ignore_index = a.ignore;
        e.labels = a.labels + t0;
        e.M = cl;
        e.N = V;
        e.raster = RASTER_M_FASTEST;
        e.hint_a = HINT_EVICT_LAST;
        e.hint_b = HINT_EVICT_FIRST;
        e.p_out = nullptr;   // partials and the label logit only
        e.part = part;
        e.nvt = static_cast<int>(L.nvt);
        e.zlab = zlab + t0;
        if ((rc = launch_logits(X + t0 * H, cl, H, V, mW_k, e, 0, L.nvt, a.st))) return rc;
        dlogits_bf16<<<cl, kRowThreads, fac_smem, a.st>>>(a.labels + t0, a.ignore, part, static_cast<int>(L.nvt),
                                                          zlab + t0, nullptr, 0, V, scale, a.scale_dev, lse + t0,
                                                          lossrow + t0);
        if ((rc = check_launch("dlogits_bf16"))) return rc;
    }
    // label keys of all tokens, sorted in segments of kMaxSortKeys, one start table per segment
    if (a.dW && (rc = sort_labels(a.labels, a.T, kMaxSortKeys, a.ignore, V, true, keys, lstart, a.st))) return rc;
    // pass 2: per vocabulary chunk, recompute the logits, D_c, dX +=, dW_c
    CUtensorMap mX_all, mX_mn;
    if ((rc = make_map(&mX_all, X, H, T, H, BK, BM))) return rc;     // A of the recompute (K-major)
    if ((rc = make_map(&mX_mn, X, H, T, H, MN_BOX, BK))) return rc;  // B of dW_c (MN-major)
    for (int64_t c = 0; c < L.nvchunks; ++c) {
        const int64_t c0 = c * L.Vc;
        const int vl = static_cast<int>(std::min(L.Vc, a.V - c0));
        const bool last = c == L.nvchunks - 1;
        const __nv_bfloat16* Wc = W + c0 * H;
        CUtensorMap mWc_k, mWc_mn, mD_k, mD_mn;
        if ((rc = make_map(&mWc_k, Wc, H, vl, H, BK, B_BOX_ROWS))) return rc;
        if ((rc = make_map(&mWc_mn, Wc, H, vl, H, MN_BOX, BK))) return rc;
        if ((rc = make_map(&mD_k, D, vl, T, L.ldc, BK, BM))) return rc;
        if ((rc = make_map(&mD_mn, D, vl, T, L.ldc, MN_BOX, BK))) return rc;
        EpiParams e{};
        e.err = &hdr->err;
        e.ignore_index = a.ignore;
        e.labels = a.labels;
        // a. D_c = scale * softmax part, from the recomputed logits and lse
        e.M = T;
        e.N = vl;
        // groups of 8 column blocks of W_c (16 MB) stay in L2 while X streams past once per
        // group (n fastest needs all 67 MB of W_c in every wave); X reused within a wave
        e.raster = RASTER_N_GROUPS;
        e.hint_a = HINT_NORMAL;
        e.hint_b = HINT_EVICT_LAST;    // W_c: reused by every token block
        e.lse = lse;
        e.corr_scale = scale;
        e.scale_ptr = a.scale_dev;
        e.out = D;
        e.ldo = L.ldc;
        if ((rc = launch_gemm<0, 0, EPI_SOFTMAX, 1>(mX_all, mWc_k, T, vl, H, e, a.st))) return rc;
        // b. dX (+)= D_c W_c in fp32, the one-hot part subtracted once (first chunk)
        if (a.dX) {
            EpiParams d{};
            d.err = &hdr->err;
            d.ignore_index = a.ignore;
            d.labels = a.labels;
            d.corr_src = c == 0 ? W : nullptr;
            d.ld_corr = H;
            d.corr_scale = scale;
            d.scale_ptr = a.scale_dev;
            d.M = T;
            d.N = H;
            d.raster = RASTER_N_GROUPS;
            d.acc = acc;
            d.lda = H;
            d.acc_read = c > 0 ? 1 : 0;
            d.acc_write = last ? 0 : 1;
            d.out_write = last ? 1 : 0;
            d.out = static_cast<__nv_bfloat16*>(a.dX);
            d.ldo = H;
            if ((rc = launch_gemm<0, 1, EPI_ACCUM, 1>(mD_k, mWc_mn, T, H, vl, d, a.st))) return rc;
        }
        // c. dW_c = D_c^T X, minus scale * X_t for the tokens labelled with each row
        if (a.dW) {
            EpiParams d{};
            d.err = &hdr->err;
            d.ignore_index = a.ignore;
            d.corr_src = X;
            d.ld_corr = H;
            d.corr_scale = scale;
            d.scale_ptr = a.scale_dev;
            d.keys = keys;
            d.nkeys = T;
            d.lstart = lstart + c0;
            d.nseg = static_cast<int>(L.nseg);
            d.lstride = V + 1;
            d.M = vl;
            d.N = H;
            d.raster = RASTER_N_FASTEST;
            d.out_write = 1;
            d.out = static_cast<__nv_bfloat16*>(a.dW) + c0 * H;
            d.ldo = H;
            if ((rc = launch_gemm<1, 1, EPI_ACCUM, 1>(mD_mn, mX_mn, vl, H, T, d, a.st))) return rc;
        }
    }
    return LIGER_OK;
}

CompactLayout compact_layout2(int64_t T, int64_t H, int64_t V, int64_t vchunk) {
    const Layout2 L = layout2(T, H, V, vchunk);
    return compact_regions(L.labs, L.total, T, H, 2);
}

// The two-pass path on the tokens that are not ignored only (both passes skip the
// ignored tokens' logits).
int run_two_pass_compact(const Args& a, int64_t n_valid, int64_t vchunk, float scale) {
    const Layout2 Lt = layout2(a.T, a.H, a.V, vchunk);
    const Layout2 Lc = layout2(n_valid, a.H, a.V, vchunk);
    if (Lc.total > Lt.total) return run_two_pass(a, Lt, scale);
    return run_compacted(a, n_valid, compact_layout2(a.T, a.H, a.V, vchunk), RowVals{Lt.lse, Lt.lossrow, Lt.hdr},
                         RowVals{Lc.lse, Lc.lossrow, Lc.hdr}, [&](const Args& b) { return run_two_pass(b, Lc, scale); });
}

}  // namespace
}  // namespace liger

using namespace liger;

extern "C" size_t liger_linear_ce_workspace(int64_t T, int64_t H, int64_t V, int64_t chunk, int dtype) {
    if (T < 0 || H <= 0 || V <= 0 || chunk < 0 || (dtype != LIGER_F32 && dtype != LIGER_BF16)) return 0;
    if (use_tc(H, V, dtype)) return compact_layout(T, H, V, chunk, dtype).total;
    return layout(T, H, V, chunk, dtype).total;
}

namespace liger {
namespace {

struct CommonLayout {
    size_t lse, lossrow, hdr, labs, total;
};

// A pinned host copy of the header for this thread (allocated on first use, kept for
// the thread's lifetime; pinned memory is visible to every device's context).
int pinned_hdr(Hdr** out) {
    thread_local Hdr* buf = nullptr;
    if (buf == nullptr) {
        void* p = nullptr;
        if (cudaMallocHost(&p, sizeof(Hdr)) != cudaSuccess) return check_launch("linear_ce pinned header");
        buf = static_cast<Hdr*>(p);
    }
    *out = buf;
    return LIGER_OK;
}

// Shared tail of both entry points: pointer and workspace checks, the label
// scan (bad labels -> LIGER_ERR_LABEL before any other work), the all-ignored
// case, the gradient scale, the variant's GEMMs, the final loss.
// sync = false: no host wait (capturable in a CUDA graph); bad labels are replaced by
// ignore_index in a workspace copy, the scale and the mean's count stay on the device,
// and the loss is NaN if a label was bad.
template <typename Run>
int ce_entry(const char* who, const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H, int64_t V,
             int64_t ignore_index, int reduction, float grad_scale, float* loss, void* dX, void* dW, void* ws,
             size_t ws_bytes, int dtype, void* stream, const CommonLayout& CL, Run run, bool sync = true) {
    if (!X || !W || !loss || (T > 0 && !labels)) return fail(LIGER_ERR_NULL, "%s: X, W, labels, loss required", who);
    if (!aligned16(X) || !aligned16(W) || (dX && !aligned16(dX)) || (dW && !aligned16(dW)) ||
        (reinterpret_cast<uintptr_t>(loss) & 3) || (reinterpret_cast<uintptr_t>(labels) & 7))
        return fail(LIGER_ERR_ALIGN, "%s: X, W, dX, dW must be 16-byte aligned", who);
    if (!ws || ws_bytes < CL.total || (reinterpret_cast<uintptr_t>(ws) & 255))
        return fail(LIGER_ERR_WORKSPACE, "%s: workspace of %zu bytes (256-byte aligned) required, got %zu", who,
                    CL.total, ws_bytes);
    cudaStream_t st = as_stream(stream);
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    Hdr* hdr = reinterpret_cast<Hdr*>(w8 + CL.hdr);
    if (cudaMemsetAsync(hdr, 0, sizeof(Hdr), st) != cudaSuccess) return check_launch("linear_ce memset");
    if (!sync && T > 0) {
        int64_t* labs = reinterpret_cast<int64_t*>(w8 + CL.labs);
        const int grid = static_cast<int>(std::min<int64_t>(ceil_div(T, 256), 4 * sm_count()));
        label_scan<<<grid, 256, 0, st>>>(labels, T, V, ignore_index, hdr, labs);
        if (int rc = check_launch("label_scan")) return rc;
        ce_scale<<<1, 1, 0, st>>>(hdr, reduction, grad_scale);
        if (int rc = check_launch("ce_scale")) return rc;
        Args a{X, W, labs, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, w8, dtype, st, &hdr->scale};
        if (int rc = run(a, 0.0f, int64_t{-1})) return rc;   // the count stays on the device
        loss_final<<<1, 1024, 0, st>>>(reinterpret_cast<float*>(w8 + CL.lossrow), T, 0.0, hdr, loss,
                                       reduction == 0 ? 1 : 2);
        return check_launch("loss_final");
    }
    Hdr h{};
    if (T > 0) {
        const int grid = static_cast<int>(std::min<int64_t>(ceil_div(T, 256), 4 * sm_count()));
        label_scan<<<grid, 256, 0, st>>>(labels, T, V, ignore_index, hdr, nullptr);
        if (int rc = check_launch("label_scan")) return rc;
        // read through a pinned buffer of this thread: a copy into pageable memory takes the
        // driver's staging path, which can wait behind other copies in flight
        Hdr* hp = nullptr;
        if (int rc = pinned_hdr(&hp)) return rc;
        if (cudaMemcpyAsync(hp, hdr, sizeof(Hdr), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return check_launch("linear_ce label scan");
        h = *hp;
        if (h.bad) return fail(LIGER_ERR_LABEL, "%s: a label is outside [0, %lld) and is not %lld", who,
                               (long long)V, (long long)ignore_index);
    }
    const int64_t n_valid = static_cast<int64_t>(h.n_valid);
    const size_t esz = dtype == LIGER_F32 ? 4 : 2;
    if (n_valid == 0) {
        // nothing to learn from: loss 0, zero gradients (PyTorch would give NaN for the mean)
        bool ok = cudaMemsetAsync(loss, 0, sizeof(float), st) == cudaSuccess;
        if (dX) ok = ok && cudaMemsetAsync(dX, 0, static_cast<size_t>(T * H) * esz, st) == cudaSuccess;
        if (dW) ok = ok && cudaMemsetAsync(dW, 0, static_cast<size_t>(V * H) * esz, st) == cudaSuccess;
        if (T > 0) ok = ok && cudaMemsetAsync(w8 + CL.lse, 0, sizeof(float) * static_cast<size_t>(T), st) == cudaSuccess;
        if (T > 0)
            ok = ok && cudaMemsetAsync(w8 + CL.lossrow, 0, sizeof(float) * static_cast<size_t>(T), st) == cudaSuccess;
        return ok ? LIGER_OK : check_launch("linear_ce memset");
    }
    const float scale = reduction == 0 ? static_cast<float>(static_cast<double>(grad_scale) / static_cast<double>(n_valid))
                                       : grad_scale;
    Args a{X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, w8, dtype, st, nullptr};
    if (int rc = run(a, scale, n_valid)) return rc;
    const double denom = reduction == 0 ? static_cast<double>(n_valid) : 1.0;
    loss_final<<<1, 1024, 0, st>>>(reinterpret_cast<float*>(w8 + CL.lossrow), T, denom, hdr, loss, 0);
    return check_launch("loss_final");
}

}  // namespace
}  // namespace liger

namespace {
int linear_ce_impl(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H, int64_t V,
                   int64_t ignore_index, int reduction, float grad_scale, float* loss, void* dX, void* dW, void* ws,
                   size_t ws_bytes, int64_t chunk, int dtype, void* stream, bool sync) {
    clear_error();
    if (dtype != LIGER_F32 && dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "linear_ce: dtype %d", dtype);
    if (T < 0 || H <= 0 || V <= 0 || chunk < 0 || H > (1 << 30) || V > (1 << 30) || T > (int64_t{1} << 31) ||
        (reduction != 0 && reduction != 1))
        return fail(LIGER_ERR_SHAPE, "linear_ce: T=%lld H=%lld V=%lld chunk=%lld reduction=%d", (long long)T,
                    (long long)H, (long long)V, (long long)chunk, reduction);
    const Layout L = layout(T, H, V, chunk, dtype);
    const size_t total = L.tc ? compact_layout(T, H, V, chunk, dtype).total : L.total;
    const CommonLayout CL{L.lse, L.lossrow, L.hdr, L.labs, total};
    return ce_entry(
        "linear_ce", X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws, ws_bytes, dtype,
        stream, CL,
        [&](const Args& a, float scale, int64_t n_valid) {
            if (L.tc) {
                // some tokens ignored, and their count known on the host: run the others only
                if (n_valid > 0 && n_valid < a.T) return run_tc_compact(a, n_valid, chunk, scale);
                return run_tc(a, L, scale);
            }
            if (dtype == LIGER_F32) return run_simt<float>(a, L, scale);
            return run_simt<__nv_bfloat16>(a, L, scale);
        },
        sync);
}
}  // namespace

extern "C" int liger_linear_ce_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H,
                                       int64_t V, int64_t ignore_index, int reduction, float grad_scale, float* loss,
                                       void* dX, void* dW, void* ws, size_t ws_bytes, int64_t chunk, int dtype,
                                       void* stream) {
    return linear_ce_impl(X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws, ws_bytes,
                          chunk, dtype, stream, true);
}

extern "C" int liger_linear_ce_fwd_bwd_async(const void* X, const void* W, const int64_t* labels, int64_t T,
                                             int64_t H, int64_t V, int64_t ignore_index, int reduction,
                                             float grad_scale, float* loss, void* dX, void* dW, void* ws,
                                             size_t ws_bytes, int64_t chunk, int dtype, void* stream) {
    return linear_ce_impl(X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws, ws_bytes,
                          chunk, dtype, stream, false);
}

extern "C" size_t liger_linear_ce_two_pass_workspace(int64_t T, int64_t H, int64_t V, int64_t vchunk) {
    if (T < 0 || H <= 0 || V <= 0 || vchunk < 0) return 0;
    return compact_layout2(T, H, V, vchunk).total;
}

namespace {
int linear_ce_two_pass_impl(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H, int64_t V,
                            int64_t ignore_index, int reduction, float grad_scale, float* loss, void* dX, void* dW,
                            void* ws, size_t ws_bytes, int64_t vchunk, int dtype, void* stream, bool sync) {
    clear_error();
    if (dtype != LIGER_BF16) return fail(LIGER_ERR_DTYPE, "linear_ce_two_pass: bf16 only (tensor-core path)");
    if (T < 0 || H < 64 || H % 8 || V < 256 || vchunk < 0 || (vchunk % 8) || H > (1 << 30) || V > (1 << 30) ||
        T > (int64_t{1} << 31) - 1 || (reduction != 0 && reduction != 1))
        return fail(LIGER_ERR_SHAPE, "linear_ce_two_pass: T=%lld H=%lld V=%lld vchunk=%lld reduction=%d "
                    "(H >= 64 and a multiple of 8, V >= 256, vchunk a multiple of 8)", (long long)T, (long long)H,
                    (long long)V, (long long)vchunk, reduction);
    const Layout2 L = layout2(T, H, V, vchunk);
    const CommonLayout CL{L.lse, L.lossrow, L.hdr, L.labs, compact_layout2(T, H, V, vchunk).total};
    return ce_entry(
        "linear_ce_two_pass", X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws, ws_bytes,
        dtype, stream, CL,
        [&](const Args& a, float scale, int64_t n_valid) {
            // some tokens ignored, and their count known on the host: run the others only
            if (n_valid > 0 && n_valid < a.T) return run_two_pass_compact(a, n_valid, vchunk, scale);
            return run_two_pass(a, L, scale);
        },
        sync);
}
}  // namespace

extern "C" int liger_linear_ce_two_pass_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t T,
                                                int64_t H, int64_t V, int64_t ignore_index, int reduction,
                                                float grad_scale, float* loss, void* dX, void* dW, void* ws,
                                                size_t ws_bytes, int64_t vchunk, int dtype, void* stream) {
    return linear_ce_two_pass_impl(X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws,
                                   ws_bytes, vchunk, dtype, stream, true);
}

extern "C" int liger_linear_ce_two_pass_fwd_bwd_async(const void* X, const void* W, const int64_t* labels, int64_t T,
                                                      int64_t H, int64_t V, int64_t ignore_index, int reduction,
                                                      float grad_scale, float* loss, void* dX, void* dW, void* ws,
                                                      size_t ws_bytes, int64_t vchunk, int dtype, void* stream) {
    return linear_ce_two_pass_impl(X, W, labels, T, H, V, ignore_index, reduction, grad_scale, loss, dX, dW, ws,
                                   ws_bytes, vchunk, dtype, stream, false);
}
