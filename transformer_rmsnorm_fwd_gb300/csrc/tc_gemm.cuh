// Persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for sm_103a, with the fused epilogues of the linear
// cross-entropy.
//
//   C[m, n] = sum_k A(m, k) * B(n, k)        (bf16 x bf16 -> fp32 in TMEM)
//
// A and B are each read by TMA in 128-byte-swizzled tiles, either K-major
// (K contiguous) or MN-major (M / N contiguous); the layout is a template
// parameter and becomes the operand-major bits of the MMA instruction
// descriptor and the LBO / SBO of the shared-memory descriptors.
//
// Block = 6 warps, one block per SM.  Two modes:
//  * single CTA (PAIR = 0): 128 x 256 tiles, a 4-stage ring of 48 KB stages;
//  * CTA pair (PAIR = 1, the one the library launches): clusters of two
//    CTAs on neighbouring SMs share tcgen05.mma.cta_group::2 (M=256, N=256):
//    each CTA loads 128 rows of A and 128 rows of B (32 KB per k-block
//    instead of 48 KB, so L2->SM traffic per flop drops by a third) into a
//    5-stage ring, both CTAs' copies complete on the leader's barrier, the
//    leader issues the MMAs for both, and its commits are multicast to the
//    pair's barriers; each CTA's TMEM holds its 128 x 256 half.
//   warp 0      TMA producer (one lane);
//   warp 1      TMEM owner and (leader) MMA issuer (one lane): 4 x tcgen05.mma
//               (K=16) per 64-wide k-block, tcgen05.commit frees the ring
//               slot, a second commit hands the accumulator to the epilogue;
//   warps 2..5  epilogue: each thread owns one accumulator row (TMEM lane),
//               reads it with tcgen05.ld 32 columns at a time and applies the
//               fused epilogue; the accumulator is double-buffered in TMEM
//               (2 x 256 columns) so tile i's epilogue overlaps tile i+1's
//               MMAs.  Each warp moves its 32 rows to and from global memory
//               through an 8 KB staging buffer as whole row runs (see
//               store_block), not one 16-byte piece of 32 rows at a time.
// Every mbarrier wait is bounded (about 4 s of %globaltimer, mbarrier.cuh); on expiry the
// waiting role records an error code in *ep.err, stops issuing work, waits
// (bounded) for the copies and MMAs it already issued, and the block frees
// its TMEM and exits.
#pragma once

#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "mbarrier.cuh"

namespace liger {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;          // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MN_BOX = 64;      // MN-major TMA box: 64 (MN) x 64 (K) = 8 KB
constexpr int MN_BOX_BYTES = MN_BOX * BK * 2;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int B_BOX_ROWS = BN / 2;   // K-major B maps: boxes of 128 rows (two per 256-row stage)

// Tile geometry of one CTA (PAIR = 0) or of a CTA pair sharing one
// cta_group::2 MMA (PAIR = 1): the pair computes a 256 x 256 tile, each CTA
// loading 128 rows of A and 128 rows of B and holding its 128 x 256 half of
// the accumulator, so each SM moves 32 KB instead of 48 KB per k-block.
template <int PAIR>
struct TileCfg {
    static constexpr int TM = PAIR ? 2 * BM : BM;        // tile rows
    static constexpr int BNL = PAIR ? BN / 2 : BN;       // B rows held by this CTA
    static constexpr int B_L = BNL * BK * 2;
    static constexpr int STAGE_L = A_BYTES + B_L;
    static constexpr int ST = PAIR ? 5 : STAGES;         // ring depth: 5 measured fastest (3 and 4 leave the MMAs waiting; 6 and 7 were slower)
    static constexpr int EPI_STAGE = 4 * 8192;           // the epilogue warps' staging buffers (8 KB each)
    static constexpr int SMEM = 1024 + ST * STAGE_L + 256 + EPI_STAGE;
};

enum Epi : int {
    EPI_LOGITS = 0,
    EPI_STORE = 1,
    EPI_ACCUM = 2,
    EPI_SWIGLU = 3,
    EPI_SWIGLU_BWD = 4,
    EPI_QKV_ROPE = 5,
    EPI_SOFTMAX = 6
};

// Tile order of the persistent loop: m fastest, n fastest, or groups of
// GROUP_N tile columns with n fastest inside a group (for long-K problems
// where both operands stream from HBM: each wave then shares ~SMs/GROUP_N
// A row-blocks and GROUP_N B column-blocks through L2).
enum Raster : int { RASTER_M_FASTEST = 0, RASTER_N_FASTEST = 1, RASTER_N_GROUPS = 2 };
constexpr int GROUP_N = 8;

enum Err : int { ERR_TMA_EMPTY = 1, ERR_MMA_FULL = 2, ERR_MMA_TMEM = 3, ERR_EPI_TMEM = 4 };

struct EpiParams {
    int M, N;                           // logical problem size (epilogue masks)
    int raster;                         // tile order (Raster)
    int* err;                           // error word (device)
    // EPI_LOGITS: P = exp(z - m_tile) as bf16 (not written if p_out is null),
    // per-(row, n-tile) (m, sum), z at label
    const int64_t* labels;              // [M] (chunk rows)
    int64_t ignore_index;
    __nv_bfloat16* p_out;
    int64_t ldp;
    float2* part;
    int nvt;
    float* zlab;                        // [M]
    // EPI_STORE: bf16 out [M, N] (ldo), rows with label == ignore_index -> +0
    __nv_bfloat16* out;
    int64_t ldo;
    // EPI_ACCUM: fp32 accumulator acc [M, N] (lda); flags.  With labels set, rows
    // labelled ignore_index are written +0 and, if corr_src is set without keys,
    // corr_scale * corr_src[labels[row], :] is subtracted (as EPI_STORE does).
    float* acc;
    int64_t lda;
    int acc_read, acc_write, out_write;
    // one-hot correction applied in fp32 (the bf16 operand carries only the
    // softmax part): EPI_STORE subtracts corr_scale * corr_src[labels[row], :];
    // EPI_ACCUM subtracts corr_scale * corr_src[t, :] for every token t whose
    // label is this row: keys[0, nkeys) = sorted (label << 32 | t), indexed by lstart.
    const __nv_bfloat16* corr_src;
    int64_t ld_corr;
    float corr_scale;
    const float* scale_ptr;             // non-null: corr_scale is read from here (set on the device)
    // The keys may come in nseg sorted segments with one start table each,
    // lstride ints apart (nseg 0 counts as 1).
    const unsigned long long* keys;
    int nkeys;
    const int* lstart;
    int nseg;
    int64_t lstride;
    // EPI_SOFTMAX: out[row, col] = corr_scale * exp(z - lse[row]) (bf16; +0 on rows
    // labelled ignore_index), the softmax part of the logit gradient
    const float* lse;
    // L2 policies (Hint) of the A and B loads; streaming epilogue traffic (P, the
    // fp32 accumulator, dW) always uses evict-first accesses
    int hint_a, hint_b;
    // operand modes: bsplit -- the 256 B rows of a stage are rows [ni*128, +128) of
    // the B map and rows [ni*128, +128) of the B2 map (gate and up weights);
    // ksplit_nkb > 0 -- k-blocks from ksplit_nkb on come from the A2 / B2 maps,
    // their k coordinate restarting at 0 (a sum of two products)
    int bsplit, ksplit_nkb;
    // msplit_mt > 0 (EPI_ACCUM without labels, keys or the fp32 sum) -- row blocks from
    // msplit_mt on come from the A2 map, their row coordinate restarting at 0, and their
    // rows (< M2) go to out2: two products with the same B in one launch (dW_g and
    // dW_u), so that their tiles share waves
    int msplit_mt, M2;
    // EPI_SWIGLU: out[row, ni*128 + j] = silu(acc[j]) * acc[128 + j], j < 128, col < N; with
    // out2 set, g = acc[j] and u = acc[128 + j] also go to out2 and out3 (bf16, same layout).
    // EPI_SWIGLU_BWD: with dh = src[row, col] recomputes g, u from the
    // accumulator and writes out = dg (dh u s (1 + g (1 - s))), out2 = du (dh g s).
    const __nv_bfloat16* src;
    int64_t lds;
    __nv_bfloat16* out2;
    // EPI_QKV_ROPE: y = acc * rs[row] + bias[col] over heads of hd columns (hd divides
    // BN); heads below nq + nk (q, then k) are rotated, pairs (j, j + hd/2), by the
    // angle row cos_t/sin_t[tr] (ld_tab floats), tr = tab_row ? clamp(tab_row[row],
    // 0, n_tab - 1) : row % tab_mod; q -> out [M, nq], k -> out2 [M, nk],
    // v -> out3 [M, N - nq - nk]
    const float* rs;
    const float* bias;
    const float* cos_t;
    const float* sin_t;
    int64_t ld_tab;
    const int32_t* tab_row;
    int n_tab, tab_mod;
    int hd, nq, nk;
    __nv_bfloat16* out3;
};

// ------------------------------------------------------------ PTX wrappers
// L2 eviction policy of an operand's loads (createpolicy, whole access)
enum Hint : int { HINT_NORMAL = 0, HINT_EVICT_FIRST = 1, HINT_EVICT_LAST = 2 };
__device__ __forceinline__ uint64_t make_policy(int hint) {
    uint64_t p = 0;
    if (hint == HINT_EVICT_FIRST)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    else if (hint == HINT_EVICT_LAST)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, dense.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// ---- CTA-pair (cta_group::2) forms
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// address of the same shared-memory object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t o;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(addr), "r"(rank));
    return o;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory completing on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
// arrive once on the mbarrier at this offset in both CTAs of the pair when the MMAs issued so far complete
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load split in two, so that the next chunk's load is in flight while
// this one is used: issue, then wait.  The wait names the destination
// registers as operands, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
// t[k] for a run-time k in [0, 32) by a select tree on the bits of k (keeps t in registers)
__device__ __forceinline__ float select32(const float (&t)[32], int k) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = (k & 16) ? t[i + 16] : t[i];
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool hi = (k & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) a[i] = hi ? a[i + w] : a[i];
    }
    return a[0];
}
// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// near 2^-22, results below the normal range flushed to zero)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// v[0..32) -= s * src[0..32) over the 8-column groups that start below n_left
__device__ __forceinline__ void sub_scaled32(float (&v)[32], const __nv_bfloat16* src, float s, int n_left) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 < n_left) {
            float f[8];
            unpack(ldg16(src + g * 8), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[g * 8 + e] = fmaf(-s, f[e], v[g * 8 + e]);
        }
    }
}

// ---- row-run epilogue stores through a warp-private staging buffer
// An epilogue thread owns one accumulator row, so a direct 16-byte store from
// every lane touches 32 rows: 32 half-filled sectors per warp instruction.
// Instead each lane writes its row's block of NCH 16-byte chunks (NCH = 4:
// 32 bf16 columns, NCH = 8: 32 fp32 columns) into the warp's buffer, and the
// warp moves the block to global memory as whole row runs, 32 / NCH rows per
// instruction (full sectors, 4 or 8 lines).  Loads of a block (the fp32 sum,
// the upstream gradient) take the reverse path.  Chunk j of row r sits in the
// 16-byte slot j ^ swz(r) of the row, which spreads both the per-row accesses
// and the row-run accesses of each quarter warp over all 32 banks.
__device__ __forceinline__ void sts16(uint32_t a, const uint4& v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds16(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}
template <int NCH>
__device__ __forceinline__ uint32_t stage_slot(int r, int j) {
    return NCH == 8 ? static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) << 4))
                    : static_cast<uint32_t>(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}
// number of 16-byte chunks (epc elements each) of a block starting at column c0 that start below n
__device__ __forceinline__ int chunks_below(int c0, int n, int epc, int nch) {
    const int k = n > c0 ? (n - c0 + epc - 1) / epc : 0;
    return k < nch ? k : nch;
}
// this lane's row of the block, to and from the buffer
template <int NCH>
__device__ __forceinline__ void stage_row(uint32_t buf, int lane, const uint4 (&v)[NCH]) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) sts16(buf + stage_slot<NCH>(lane, j), v[j]);
}
template <int NCH>
__device__ __forceinline__ void unstage_row(uint32_t buf, int lane, uint4 (&v)[NCH]) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) v[j] = lds16(buf + stage_slot<NCH>(lane, j));
}
// The block whose row 0, chunk 0 is at blk (rows ld bytes apart) as row runs:
// only rows whose bit is set in `rows` and chunks below nch are written.
// Every lane of the warp calls it, after a __syncwarp that follows the staging.
template <int NCH, bool CS>
__device__ __forceinline__ void store_block(uint32_t buf, int lane, uint8_t* blk, int64_t ld, uint32_t rows, int nch) {
    constexpr int RPI = 32 / NCH;
    const int j = lane % NCH, r0 = lane / NCH;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int r = i * RPI + r0;
        const uint4 v = lds16(buf + stage_slot<NCH>(r, j));
        if (((rows >> r) & 1u) && j < nch) {
            if (CS) stg16_cs(blk + r * ld + j * 16, v);
            else stg16(blk + r * ld + j * 16, v);
        }
    }
}
// Row runs of a block from global memory into registers (zero where masked) ...
template <int NCH, bool CS>
__device__ __forceinline__ void load_block(int lane, const uint8_t* blk, int64_t ld, uint32_t rows, int nch,
                                           uint4 (&v)[NCH]) {
    constexpr int RPI = 32 / NCH;
    const int j = lane % NCH, r0 = lane / NCH;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int r = i * RPI + r0;
        v[i] = make_uint4(0, 0, 0, 0);
        if (((rows >> r) & 1u) && j < nch) v[i] = CS ? ldg16_cs(blk + r * ld + j * 16) : ldg16(blk + r * ld + j * 16);
    }
}
// Row runs of a block gathered from rows of a table: row r of the block is
// table row idx of lane r (every lane passes an in-range idx).
template <int NCH>
__device__ __forceinline__ void gather_block(int lane, const uint8_t* base, int64_t ld, int idx, uint4 (&v)[NCH]) {
    constexpr int RPI = 32 / NCH;
    const int j = lane % NCH, r0 = lane / NCH;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int tr = __shfl_sync(0xffffffffu, idx, i * RPI + r0);
        v[i] = ldg16(base + static_cast<int64_t>(tr) * ld + j * 16);
    }
}
// ... and from those registers into the buffer (then __syncwarp and unstage_row)
template <int NCH>
__device__ __forceinline__ void stage_block(uint32_t buf, int lane, const uint4 (&v)[NCH]) {
    constexpr int RPI = 32 / NCH;
    const int j = lane % NCH, r0 = lane / NCH;
#pragma unroll
    for (int i = 0; i < NCH; ++i) sts16(buf + stage_slot<NCH>(i * RPI + r0, j), v[i]);
}
__device__ __forceinline__ uint4 pack_bf8(const float* f) {
    return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7]));
}

// --------------------------------------------------------------- kernel
// The kernel and its launcher have internal linkage: every translation unit
// that includes this header registers and configures its own copy, so a
// one-time attribute set in one unit never stands in for another's.
namespace {

template <int A_MN, int B_MN, int EPI, int PAIR = 0>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, int M, int N,
                   int K, EpiParams ep) {
    using Cfg = TileCfg<PAIR>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + Cfg::ST * Cfg::STAGE_L;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Cfg::ST + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * Cfg::ST + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * Cfg::ST + 2 + a); };
    const uint32_t slot = bar0 + 8u * (2 * Cfg::ST + 4);
    uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(gbase + Cfg::ST * Cfg::STAGE_L + 8 * (2 * Cfg::ST + 4));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a CTA pair is a cluster of two consecutive blocks; rank 0 issues the MMAs
    const uint32_t crank = PAIR ? cluster_rank() : 0u;
    const bool leader = crank == 0;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int num_m = (M + Cfg::TM - 1) / Cfg::TM, num_n = (N + BN - 1) / BN;
    const int ntiles = num_m * num_n;
    const int nkb = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::ST; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), PAIR ? 8 : 4);   // the epilogue warps of both CTAs
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tmA);
        prefetch_map(&tmB);
        if (ep.bsplit || ep.ksplit_nkb > 0 || ep.msplit_mt > 0) {
            prefetch_map(&tmA2);
            prefetch_map(&tmB2);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();   // both CTAs' barriers initialised before any cross-CTA arrive
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(slot_ptr);

    auto tile_mn = [&](int t, int& mi, int& ni) {
        if (ep.raster == RASTER_N_FASTEST) {
            mi = t / num_n;
            ni = t - mi * num_n;
        } else if (ep.raster == RASTER_N_GROUPS) {
            // groups of GROUP_N tile columns, n fastest inside a group: a wave of
            // resident tiles spans ~SMs/GROUP_N row blocks x GROUP_N column blocks
            const int full = num_n / GROUP_N;
            const int tiles_full = full * num_m * GROUP_N;
            if (t < tiles_full) {
                const int g = t / (num_m * GROUP_N), w = t - g * num_m * GROUP_N;
                mi = w / GROUP_N;
                ni = g * GROUP_N + (w - mi * GROUP_N);
            } else {
                const int width = num_n - full * GROUP_N, w = t - tiles_full;
                mi = w / width;
                ni = full * GROUP_N + (w - mi * width);
            }
        } else {
            ni = t / num_m;
            mi = t - ni * num_m;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_a = make_policy(ep.hint_a), pol_b = make_policy(ep.hint_b);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[Cfg::ST];
            bool issued[Cfg::ST];
            for (int s = 0; s < Cfg::ST; ++s) issued[s] = false, issued_phase[s] = 0;
            bool ok = true;
            const int a_row0 = static_cast<int>(crank) * BM;   // this CTA's rows within the tile
            for (int t = unit; t < ntiles && ok; t += nunits) {
                int mi, ni;
                tile_mn(t, mi, ni);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u)) {
                        atomicExch(ep.err, ERR_TMA_EMPTY);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * Cfg::STAGE_L;
                    const uint32_t sb = sa + A_BYTES;
                    // the pair's loads all complete on the leader's full barrier
                    const uint32_t fb = PAIR && !leader ? map_to_rank(full_bar(stage), 0) : full_bar(stage);
                    if (leader) mbar_expect_tx(full_bar(stage), (PAIR ? 2 : 1) * Cfg::STAGE_L);
                    auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y, uint64_t pol) {
                        if (PAIR) tma_load_2d_pair(dst, m, fb, x, y, pol);
                        else tma_load_2d_hint(dst, m, fb, x, y, pol);
                    };
                    const bool second = ep.ksplit_nkb > 0 && kb >= ep.ksplit_nkb;
                    const bool mhi = ep.msplit_mt > 0 && mi >= ep.msplit_mt;
                    const CUtensorMap* mA = second || mhi ? &tmA2 : &tmA;
                    const CUtensorMap* mB = second ? &tmB2 : &tmB;
                    const int kc = (second ? kb - ep.ksplit_nkb : kb) * BK;
                    const int arow = (mhi ? mi - ep.msplit_mt : mi) * Cfg::TM + a_row0;
                    if (A_MN) {
#pragma unroll
                        for (int j = 0; j < BM / MN_BOX; ++j) load(sa + j * MN_BOX_BYTES, mA, arow + j * MN_BOX, kc, pol_a);
                    } else {
                        load(sa, mA, kc, arow, pol_a);
                    }
                    if (ep.bsplit) {
                        // K-major B maps with 128-row boxes: gate rows, then up rows (one each per CTA of a pair)
                        if (PAIR) {
                            load(sb, leader ? &tmB : &tmB2, kc, ni * (BN / 2), pol_b);
                        } else {
                            load(sb, &tmB, kc, ni * (BN / 2), pol_b);
                            load(sb + B_BYTES / 2, &tmB2, kc, ni * (BN / 2), pol_b);
                        }
                    } else if (B_MN) {
                        const int bcol = ni * BN + static_cast<int>(crank) * Cfg::BNL;
#pragma unroll
                        for (int j = 0; j < Cfg::BNL / MN_BOX; ++j)
                            load(sb + j * MN_BOX_BYTES, mB, bcol + j * MN_BOX, kc, pol_b);
                    } else {
                        const int brow = ni * BN + static_cast<int>(crank) * Cfg::BNL;
#pragma unroll
                        for (int j = 0; j < Cfg::BNL / B_BOX_ROWS; ++j)
                            load(sb + j * (B_BOX_ROWS * BK * 2), mB, kc, brow + j * B_BOX_ROWS, pol_b);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == Cfg::ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every copy already issued land before the block exits
                if (leader) {
                    for (int s = 0; s < Cfg::ST; ++s)
                        if (issued[s]) mbar_wait(full_bar(s), issued_phase[s]);
                } else {
                    // the peer's copies complete on the leader's barriers: give them time to land
                    const uint64_t t0 = globaltimer();
                    while (globaltimer() - t0 < 20000000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (the leader of a pair)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = make_idesc(Cfg::TM, BN, A_MN, B_MN);
            // K-major SW128: rows of 128 B, 8-row groups 1024 B apart (SBO), K step 32 B.
            // MN-major SW128: 64-element MN atoms 8 KB apart (LBO), 8-row K groups 1024 B
            // apart (SBO), K step 16 rows = 2048 B.
            const uint32_t a_lbo = A_MN ? MN_BOX_BYTES : 16u, b_lbo = B_MN ? MN_BOX_BYTES : 16u;
            const uint32_t a_kstep = A_MN ? UMMA_K * 128u : UMMA_K * 2u;
            const uint32_t b_kstep = B_MN ? UMMA_K * 128u : UMMA_K * 2u;
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            bool any = false;
            auto commit = [&](uint32_t bar) {
                if (PAIR) mma_commit_pair(bar);
                else mma_commit(bar);
            };
            for (int t = unit; t < ntiles && ok; t += nunits, ++it) {
                const int as = it & 1;
                const uint32_t aphase = (it >> 1) & 1;
                if (!mbar_wait(tempty_bar(as), aphase ^ 1u)) {
                    atomicExch(ep.err, ERR_MMA_TMEM);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(as * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase)) {
                        atomicExch(ep.err, ERR_MMA_FULL);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + stage * Cfg::STAGE_L;
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t da = smem_desc(sa + k * a_kstep, a_lbo, 1024u);
                        const uint64_t db = smem_desc(sb + k * b_kstep, b_lbo, 1024u);
                        if (PAIR) mma_bf16_pair(d, da, db, idesc, (kb | k) != 0 ? 1u : 0u);
                        else mma_bf16(d, da, db, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    any = true;
                    commit(empty_bar(stage));
                    if (++stage == Cfg::ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit(tfull_bar(as));
            }
            if (!ok && any) {
                // wait for the MMAs already issued: commit to a free barrier and wait on it
                commit(tfull_bar(it & 1));
                mbar_wait(tfull_bar(it & 1), ((it >> 1) & 1));
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int rl = q * 32 + lane;           // accumulator row of this thread
        // this warp's 8 KB staging buffer, after the ring and the barriers
        const uint32_t sbuf = base + Cfg::ST * Cfg::STAGE_L + 256 + static_cast<uint32_t>(warp - 2) * 8192u;
        // hand the accumulator buffer back to the MMA issuer (the leader's barrier)
        auto release_acc = [&](int a) {
            if (PAIR && !leader) mbar_arrive_cluster(map_to_rank(tempty_bar(a), 0));
            else mbar_arrive(tempty_bar(a));
        };
        int it = 0;
        for (int t = unit; t < ntiles; t += nunits, ++it) {
            int mi, ni;
            tile_mn(t, mi, ni);
            const int as = it & 1;
            const uint32_t aphase = (it >> 1) & 1;
            const bool mhi = ep.msplit_mt > 0 && mi >= ep.msplit_mt;   // a row block of the second product
            const int row = (mhi ? mi - ep.msplit_mt : mi) * Cfg::TM + static_cast<int>(crank) * BM + rl;
            const int n0 = ni * BN;
            const bool row_ok = row < (mhi ? ep.M2 : ep.M);
            const float cscale = ep.scale_ptr != nullptr ? *ep.scale_ptr : ep.corr_scale;
            // EPI_ACCUM: everything that does not depend on the accumulator is fetched
            // before waiting for it (label range, first 32 columns of the fp32 sum)
            int k_lo = 0, k_hi = 0;
            uint4 pre[8], pre2[8];   // EPI_ACCUM: fp32 sum blocks c and c + 1, in flight
            const uint32_t rows = __ballot_sync(0xffffffffu, row_ok);   // bit r: row - lane + r is in range
            uint8_t* ablk = nullptr;
            if (EPI == EPI_ACCUM) {
                ablk = reinterpret_cast<uint8_t*>(ep.acc + static_cast<int64_t>(row - lane) * ep.lda + n0);
                if (row_ok && ep.lstart != nullptr) {
                    k_lo = ep.lstart[row];
                    k_hi = ep.lstart[row + 1];
                }
                load_block<8, true>(lane, ablk, ep.lda * 4, ep.acc_read ? rows : 0u, chunks_below(n0, ep.N, 4, 8), pre);
                load_block<8, true>(lane, ablk + 128, ep.lda * 4, ep.acc_read ? rows : 0u, chunks_below(n0 + 32, ep.N, 4, 8),
                                    pre2);
            }
            const bool got = __all_sync(0xffffffffu, mbar_wait(tfull_bar(as), aphase));
            if (!got) {
                if (lane == 0) atomicExch(ep.err, ERR_EPI_TMEM);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(as * BN) + (static_cast<uint32_t>(q * 32) << 16);
            if (EPI == EPI_LOGITS) {
                const int64_t y = row_ok ? ep.labels[row] : ep.ignore_index;
                const bool live = row_ok && y != ep.ignore_index;
                const bool full = n0 + BN <= ep.N;   // no column of this tile is masked
                const int64_t jy = y - n0;           // the label's column in the tile, if in [0, BN)
                float m = -INFINITY, zl = 0.f;
                bool has_lab = false;
                // Two passes over the tile's TMEM row, each with the next 32 columns'
                // load in flight while the current ones are used.  Pass 1: row max
                // (a tree per 32 columns; max is exact in any order) and z at the label.
                uint32_t ra[32], rb[32];
                auto max_chunk = [&](int c, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
                    if (c + 1 < BN / 32) tmem_ld32_issue(taddr + (c + 1) * 32, nxt);
                    float t[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        t[j] = (full || n0 + c * 32 + j < ep.N) ? __uint_as_float(cur[j]) : -INFINITY;
                    if (jy >= c * 32 && jy < c * 32 + 32) {
                        zl = select32(t, static_cast<int>(jy - c * 32));
                        has_lab = true;
                    }
#pragma unroll
                    for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
                        for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
                    }
                    m = fmaxf(m, t[0]);
                    if (c + 1 < BN / 32) tmem_ld_wait(nxt);
                };
                tmem_ld32_issue(taddr, ra);
                tmem_ld_wait(ra);
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    max_chunk(c, ra, rb);
                    max_chunk(c + 1, rb, ra);
                }
                // Pass 2: P = exp(z - m) (bf16 row runs for labelled rows) and its sum,
                // kept as 8 partial sums so the adds do not form one serial chain.
                const float ml = m * 1.4426950408889634f;
                float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                const uint32_t prows = __ballot_sync(0xffffffffu, live);
                uint8_t* pblk = ep.p_out != nullptr
                                    ? reinterpret_cast<uint8_t*>(ep.p_out + static_cast<int64_t>(row - lane) * ep.ldp + n0)
                                    : nullptr;
                auto exp_chunk = [&](int c, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
                    if (c + 1 < BN / 32) tmem_ld32_issue(taddr + (c + 1) * 32, nxt);
                    float e[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        e[j] = (full || n0 + c * 32 + j < ep.N)
                                   ? ex2_approx(fmaf(__uint_as_float(cur[j]), 1.4426950408889634f, -ml))
                                   : 0.f;
                        ps[j & 7] += e[j];
                    }
                    if (pblk != nullptr) {
                        const uint4 u[4] = {pack_bf8(e), pack_bf8(e + 8), pack_bf8(e + 16), pack_bf8(e + 24)};
                        __syncwarp();   // the previous block's row runs have been read
                        stage_row<4>(sbuf, lane, u);
                        __syncwarp();
                        store_block<4, true>(sbuf, lane, pblk + c * 64, ep.ldp * 2, prows,
                                             chunks_below(n0 + c * 32, ep.N, 8, 4));
                    }
                    if (c + 1 < BN / 32) tmem_ld_wait(nxt);
                };
                tmem_ld32_issue(taddr, ra);
                tmem_ld_wait(ra);
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    exp_chunk(c, ra, rb);
                    exp_chunk(c + 1, rb, ra);
                }
                const float sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
                if (live) {
                    ep.part[static_cast<int64_t>(row) * ep.nvt + ni] = make_float2(m, sum);
                    if (has_lab) ep.zlab[row] = zl;
                }
            } else if (EPI == EPI_STORE) {
                const int64_t y = (row_ok && ep.labels != nullptr) ? ep.labels[row] : ep.ignore_index;
                const bool zero = !row_ok || (ep.labels != nullptr && y == ep.ignore_index);
                const __nv_bfloat16* crow =
                    (ep.corr_src != nullptr && !zero) ? ep.corr_src + y * ep.ld_corr + n0 : nullptr;
                uint8_t* oblk = reinterpret_cast<uint8_t*>(ep.out + static_cast<int64_t>(row - lane) * ep.ldo + n0);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld32(taddr + c * 32, v);
                    if (crow != nullptr) sub_scaled32(v, crow + c * 32, cscale, ep.N - (n0 + c * 32));
                    uint4 u[4] = {pack_bf8(v), pack_bf8(v + 8), pack_bf8(v + 16), pack_bf8(v + 24)};
                    if (zero) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) u[g] = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();   // the previous block's row runs have been read
                    stage_row<4>(sbuf, lane, u);
                    __syncwarp();
                    store_block<4, true>(sbuf, lane, oblk + c * 64, ep.ldo * 2, rows,
                                         chunks_below(n0 + c * 32, ep.N, 8, 4));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
            } else if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) {
                const int o0 = ni * (BN / 2);   // first output (intermediate) column of the tile
                const int64_t orow0 = static_cast<int64_t>(row - lane) * ep.ldo + o0;
                // staging: out at +0, out2 at +2 KB, out3 at +4 KB, the dh block at +6 KB
                const uint32_t s_out = sbuf, s_out2 = sbuf + 2048u, s_out3 = sbuf + 4096u, s_dh = sbuf + 6144u;
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    const int nch = chunks_below(o0 + c * 32, ep.N, 8, 4);
                    uint4 dh[4];
                    if (EPI == EPI_SWIGLU_BWD)
                        load_block<4, false>(lane,
                                             reinterpret_cast<const uint8_t*>(
                                                 ep.src + static_cast<int64_t>(row - lane) * ep.lds + o0 + c * 32),
                                             ep.lds * 2, rows, nch, dh);
                    float gv[32], uv[32];
                    tmem_ld32(taddr + c * 32, gv);
                    tmem_ld32(taddr + BN / 2 + c * 32, uv);
                    __syncwarp();   // the previous block's row runs have been read
                    if (EPI == EPI_SWIGLU_BWD) {
                        stage_block<4>(s_dh, lane, dh);
                        __syncwarp();
                        unstage_row<4>(s_dh, lane, dh);   // now this lane's row
                    }
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float a[8], b[8];
                        if (EPI == EPI_SWIGLU) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float x = gv[g * 8 + e];
                                a[e] = x * __fdividef(1.0f, 1.0f + __expf(-x)) * uv[g * 8 + e];
                            }
                            sts16(s_out + stage_slot<4>(lane, g), pack(a));
                            if (ep.out2 != nullptr) {   // keep g and u for a backward without recompute
                                sts16(s_out2 + stage_slot<4>(lane, g), pack_bf8(gv + g * 8));
                                sts16(s_out3 + stage_slot<4>(lane, g), pack_bf8(uv + g * 8));
                            }
                        } else {
                            float d[8];
                            unpack(dh[g], d);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float x = gv[g * 8 + e], u = uv[g * 8 + e];
                                const float sg = __fdividef(1.0f, 1.0f + __expf(-x));
                                a[e] = d[e] * u * sg * (1.0f + x * (1.0f - sg));
                                b[e] = d[e] * (x * sg);
                            }
                            sts16(s_out + stage_slot<4>(lane, g), pack(a));
                            sts16(s_out2 + stage_slot<4>(lane, g), pack(b));
                        }
                    }
                    __syncwarp();
                    store_block<4, false>(s_out, lane, reinterpret_cast<uint8_t*>(ep.out + orow0 + c * 32), ep.ldo * 2,
                                          rows, nch);
                    if (EPI == EPI_SWIGLU_BWD || ep.out2 != nullptr)
                        store_block<4, false>(s_out2, lane, reinterpret_cast<uint8_t*>(ep.out2 + orow0 + c * 32),
                                              ep.ldo * 2, rows, nch);
                    if (EPI == EPI_SWIGLU && ep.out2 != nullptr)
                        store_block<4, false>(s_out3, lane, reinterpret_cast<uint8_t*>(ep.out3 + orow0 + c * 32),
                                              ep.ldo * 2, rows, nch);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
            } else if (EPI == EPI_SOFTMAX) {
                const int64_t y = row_ok ? ep.labels[row] : ep.ignore_index;
                const bool live = row_ok && y != ep.ignore_index;
                const float l2 = live ? ep.lse[row] * 1.4426950408889634f : 0.f;
                uint8_t* oblk = reinterpret_cast<uint8_t*>(ep.out + static_cast<int64_t>(row - lane) * ep.ldo + n0);
                // the next 32 TMEM columns load while the current ones are used
                uint32_t ra[32], rb[32];
                auto softmax_chunk = [&](int c, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
                    if (c + 1 < BN / 32) tmem_ld32_issue(taddr + (c + 1) * 32, nxt);
                    __syncwarp();   // the previous block's row runs have been read
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float a[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            a[e] = live ? cscale *
                                              ex2_approx(fmaf(__uint_as_float(cur[g * 8 + e]), 1.4426950408889634f, -l2))
                                        : 0.f;
                        sts16(sbuf + stage_slot<4>(lane, g), pack(a));
                    }
                    __syncwarp();
                    store_block<4, false>(sbuf, lane, oblk + c * 64, ep.ldo * 2, rows,
                                          chunks_below(n0 + c * 32, ep.N, 8, 4));
                    if (c + 1 < BN / 32) tmem_ld_wait(nxt);
                };
                tmem_ld32_issue(taddr, ra);
                tmem_ld_wait(ra);
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    softmax_chunk(c, ra, rb);
                    softmax_chunk(c + 1, rb, ra);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
            } else if (EPI == EPI_QKV_ROPE) {
                const float rsv = row_ok ? ep.rs[row] : 0.f;
                int64_t tr = 0;
                if (row_ok) {
                    if (ep.tab_row != nullptr) {
                        const int p = ep.tab_row[row];
                        tr = p < 0 ? 0 : (p >= ep.n_tab ? ep.n_tab - 1 : p);
                    } else {
                        tr = row % ep.tab_mod;
                    }
                }
                const int tr32 = static_cast<int>(tr);   // table row of this lane's token (n_tab < 2^31)
                const int hd = ep.hd, half = hd >> 1;
                // staging: the two 32-column output blocks of a rotated pair at +0 and +2 KB,
                // 16 columns of cos and of sin at +4 and +6 KB
                const uint32_t s_y1 = sbuf, s_y2 = sbuf + 2048u, s_cos = sbuf + 4096u, s_sin = sbuf + 6144u;
#pragma unroll 1
                for (int h0 = 0; h0 < BN; h0 += hd) {
                    const int gc = n0 + h0;   // first column of this head
                    if (gc >= ep.N) break;
                    __nv_bfloat16* hbase;
                    int64_t ldh;
                    if (gc < ep.nq) {
                        hbase = ep.out + gc;
                        ldh = ep.nq;
                    } else if (gc < ep.nq + ep.nk) {
                        hbase = ep.out2 + (gc - ep.nq);
                        ldh = ep.nk;
                    } else {
                        hbase = ep.out3 + (gc - ep.nq - ep.nk);
                        ldh = ep.N - ep.nq - ep.nk;
                    }
                    // this head's columns of the warp's 32 rows
                    uint8_t* hblk = reinterpret_cast<uint8_t*>(hbase + static_cast<int64_t>(row - lane) * ldh);
                    const float* bh = ep.bias + gc;
                    if (gc < ep.nq + ep.nk) {
#pragma unroll 1
                        for (int j = 0; j < half; j += 32) {
                            float a[32], b[32];
                            tmem_ld32(taddr + h0 + j, a);
                            tmem_ld32(taddr + h0 + half + j, b);
                            // cos / sin of 16 pairs at a time: the warp's 32 table rows
                            // gathered as row runs into the buffer, then each lane's own row
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int o0 = j + hh * 16;
                                uint4 gc4[4], gs4[4];
                                gather_block<4>(lane, reinterpret_cast<const uint8_t*>(ep.cos_t + o0), ep.ld_tab * 4,
                                                tr32, gc4);
                                gather_block<4>(lane, reinterpret_cast<const uint8_t*>(ep.sin_t + o0), ep.ld_tab * 4,
                                                tr32, gs4);
                                __syncwarp();   // the buffers' previous contents have been read
                                stage_block<4>(s_cos, lane, gc4);
                                stage_block<4>(s_sin, lane, gs4);
                                __syncwarp();
                                unstage_row<4>(s_cos, lane, gc4);
                                unstage_row<4>(s_sin, lane, gs4);
#pragma unroll
                                for (int g2 = 0; g2 < 2; ++g2) {
                                    const int g = hh * 2 + g2;   // 8 pairs: columns j + 8 g
                                    const int o = j + g * 8;
                                    float cs[8], sn[8], ba[8], bb[8], y1[8], y2[8];
#pragma unroll
                                    for (int h = 0; h < 2; ++h) {
                                        const uint4 c4 = gc4[g2 * 2 + h], s4 = gs4[g2 * 2 + h];
                                        cs[h * 4 + 0] = __uint_as_float(c4.x);
                                        cs[h * 4 + 1] = __uint_as_float(c4.y);
                                        cs[h * 4 + 2] = __uint_as_float(c4.z);
                                        cs[h * 4 + 3] = __uint_as_float(c4.w);
                                        sn[h * 4 + 0] = __uint_as_float(s4.x);
                                        sn[h * 4 + 1] = __uint_as_float(s4.y);
                                        sn[h * 4 + 2] = __uint_as_float(s4.z);
                                        sn[h * 4 + 3] = __uint_as_float(s4.w);
                                    }
                                    *reinterpret_cast<float4*>(ba) = __ldg(reinterpret_cast<const float4*>(bh + o));
                                    *reinterpret_cast<float4*>(ba + 4) =
                                        __ldg(reinterpret_cast<const float4*>(bh + o + 4));
                                    *reinterpret_cast<float4*>(bb) =
                                        __ldg(reinterpret_cast<const float4*>(bh + half + o));
                                    *reinterpret_cast<float4*>(bb + 4) =
                                        __ldg(reinterpret_cast<const float4*>(bh + half + o + 4));
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        const float x1 = fmaf(a[g * 8 + e], rsv, ba[e]);
                                        const float x2 = fmaf(b[g * 8 + e], rsv, bb[e]);
                                        y1[e] = x1 * cs[e] - x2 * sn[e];
                                        y2[e] = x2 * cs[e] + x1 * sn[e];
                                    }
                                    sts16(s_y1 + stage_slot<4>(lane, g), pack(y1));
                                    sts16(s_y2 + stage_slot<4>(lane, g), pack(y2));
                                }
                            }
                            __syncwarp();
                            store_block<4, false>(s_y1, lane, hblk + j * 2, ldh * 2, rows, 4);
                            store_block<4, false>(s_y2, lane, hblk + (half + j) * 2, ldh * 2, rows, 4);
                        }
                    } else {
#pragma unroll 1
                        for (int j = 0; j < hd; j += 32) {
                            float a[32];
                            tmem_ld32(taddr + h0 + j, a);
                            __syncwarp();   // the previous block's row runs have been read
                            {
#pragma unroll
                                for (int g = 0; g < 4; ++g) {
                                    const int o = j + g * 8;
                                    float ba[8], y[8];
                                    *reinterpret_cast<float4*>(ba) = __ldg(reinterpret_cast<const float4*>(bh + o));
                                    *reinterpret_cast<float4*>(ba + 4) =
                                        __ldg(reinterpret_cast<const float4*>(bh + o + 4));
#pragma unroll
                                    for (int e = 0; e < 8; ++e) y[e] = fmaf(a[g * 8 + e], rsv, ba[e]);
                                    sts16(s_y1 + stage_slot<4>(lane, g), pack(y));
                                }
                            }
                            __syncwarp();
                            store_block<4, false>(s_y1, lane, hblk + j * 2, ldh * 2, rows, 4);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
            } else {
                __nv_bfloat16* obase = mhi ? ep.out2 : ep.out;
                uint8_t* oblk = obase != nullptr
                                    ? reinterpret_cast<uint8_t*>(obase + static_cast<int64_t>(row - lane) * ep.ldo + n0)
                                    : nullptr;
                const int64_t ylab = (row_ok && ep.labels != nullptr) ? ep.labels[row] : ep.ignore_index;
                const bool zero_row = ep.labels != nullptr && ylab == ep.ignore_index;
                const __nv_bfloat16* lrow = (ep.labels != nullptr && ep.corr_src != nullptr && ep.keys == nullptr &&
                                             row_ok && !zero_row)
                                                ? ep.corr_src + ylab * ep.ld_corr + n0
                                                : nullptr;
                const int nseg = ep.nseg > 1 ? ep.nseg : 1;
                // staging: the fp32 block at +0 (4 KB), the bf16 block at +4 KB
                const uint32_t s_acc = sbuf, s_out = sbuf + 4096u;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    __syncwarp();   // the previous block's row runs have been read
                    if (ep.acc_read) {
                        uint4(&cur)[8] = (c & 1) ? pre2 : pre;
                        stage_block<8>(s_acc, lane, cur);   // block c, fetched two blocks ahead
                        if (c + 2 < BN / 32)
                            load_block<8, true>(lane, ablk + (c + 2) * 128, ep.lda * 4, rows,
                                                chunks_below(n0 + (c + 2) * 32, ep.N, 4, 8), cur);
                    }
                    float v[32];
                    tmem_ld32(taddr + c * 32, v);
                    for (int sg = 0; sg < nseg; ++sg) {
                        int lo = k_lo, hi = k_hi;
                        if (sg > 0) {
                            lo = row_ok ? ep.lstart[sg * ep.lstride + row] : 0;
                            hi = row_ok ? ep.lstart[sg * ep.lstride + row + 1] : 0;
                        }
                        for (int kk = lo; kk < hi; ++kk) {
                            const int64_t t = static_cast<int64_t>(ep.keys[kk] & 0xFFFFFFFFull);
                            sub_scaled32(v, ep.corr_src + t * ep.ld_corr + n0 + c * 32, cscale,
                                         ep.N - (n0 + c * 32));
                        }
                    }
                    if (lrow != nullptr) sub_scaled32(v, lrow + c * 32, cscale, ep.N - (n0 + c * 32));
                    if (zero_row) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    }
                    if (ep.acc_read) {
                        __syncwarp();
                        uint4 o[8];
                        unstage_row<8>(s_acc, lane, o);
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            float f[4];
                            unpack(o[g], f);
#pragma unroll
                            for (int e = 0; e < 4; ++e) v[g * 4 + e] += f[e];
                        }
                    }
                    if (ep.acc_write) {   // this lane's row only: no other lane reads it before the next barrier
                        uint4 w[8];
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const float f[4] = {v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]};
                            w[g] = pack(f);
                        }
                        stage_row<8>(s_acc, lane, w);
                    }
                    if (ep.out_write) {
                        const uint4 u[4] = {pack_bf8(v), pack_bf8(v + 8), pack_bf8(v + 16), pack_bf8(v + 24)};
                        stage_row<4>(s_out, lane, u);
                    }
                    __syncwarp();
                    if (ep.acc_write)
                        store_block<8, true>(s_acc, lane, ablk + c * 128, ep.lda * 4, rows,
                                             chunks_below(n0 + c * 32, ep.N, 4, 8));
                    if (ep.out_write)
                        store_block<4, true>(s_out, lane, oblk + c * 64, ep.ldo * 2, rows,
                                             chunks_below(n0 + c * 32, ep.N, 8, 4));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(as);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();   // neither CTA exits while the pair's MMAs or copies may touch it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                         : "memory");
    }
}

}  // namespace

// ------------------------------------------------------------ host side
// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Rows of a K-major A operand [M, K] bf16 per launch, for a GEMM whose tiles
// sweep all of B over the same A rows: those rows must stay in L2 meanwhile.
// At most 32 MiB of them (a multiple of 256 rows, at least 256, at most M):
// measured on the 129 MB L2, 33.5 MB of reused rows stayed resident beside
// streamed operands and 67 MB did not (one launch over 67 MB of X rows read
// 12.7x its operand bytes from DRAM).  At K = 4096: 4096 rows.
inline int64_t rows_in_l2(int64_t K, int64_t M) {
    const int64_t r = (int64_t{32} << 20) / (2 * K) / 256 * 256;
    return std::max<int64_t>(1, std::min(M, std::max<int64_t>(256, r)));
}

// 2-D bf16 map over a row-major matrix [outer, inner] with row stride
// `ld` elements, box (box_inner x box_outer), 128-byte swizzle, zero fill.
int make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_inner,
             int box_outer);

// Launch C = A(M x K) * B(N x K) with the given epilogue.  A_MN / B_MN say
// whether each operand is MN-major.  K-major B maps have 128-row boxes
// (B_BOX_ROWS).  PAIR = 1: clusters of two CTAs share cta_group::2 MMAs on
// 256 x 256 tiles.  grid_limit = 0: one block per SM (pairs: as many as fit).
namespace {

template <int A_MN, int B_MN, int EPI, int PAIR = 0>
int launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K, const EpiParams& ep,
                cudaStream_t st, int grid_limit = 0, const CUtensorMap* ma2 = nullptr,
                const CUtensorMap* mb2 = nullptr) {
    using Cfg = TileCfg<PAIR>;
    auto kern = tc_gemm_kernel<A_MN, B_MN, EPI, PAIR>;
    // per instantiation and device: function attributes belong to each device's context.
    // units_of[dev] = 0 until the attribute is set; threads that race here all set the
    // same attribute and store the same count (published with release / acquire).
    constexpr int kDevs = 64;
    static std::atomic<int> units_of[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return check_launch("tc_gemm device");
    int max_units = units_of[dev].load(std::memory_order_acquire);
    if (max_units == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
            return check_launch("tc_gemm attribute");
        if (PAIR) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (sm_count() / 2));
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = Cfg::SMEM;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0)
                return check_launch("tc_gemm cluster occupancy");
            max_units = n;
        } else {
            max_units = sm_count();
        }
        units_of[dev].store(max_units, std::memory_order_release);
    }
    const int tiles = ((M + Cfg::TM - 1) / Cfg::TM) * ((N + BN - 1) / BN);
    int units = max_units;
    if (grid_limit > 0) units = std::min(units, PAIR ? std::max(1, grid_limit / 2) : grid_limit);
    units = std::max(1, std::min(units, tiles));
    if (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * units);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = Cfg::SMEM;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, ma, mb, ma2 ? *ma2 : ma, mb2 ? *mb2 : mb, M, N, K, ep) != cudaSuccess)
            return check_launch("tc_gemm pair launch");
        return check_launch("tc_gemm");
    }
    kern<<<units, THREADS, Cfg::SMEM, st>>>(ma, mb, ma2 ? *ma2 : ma, mb2 ? *mb2 : mb, M, N, K, ep);
    return check_launch("tc_gemm");
}

}  // namespace

}  // namespace tc
}  // namespace liger
