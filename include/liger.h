/*
 * liger.h -- C-ABI of libliger.so: fused decoder-layer operators for one
 * NVIDIA GB300 GPU (sm_103a), hand-written CUDA.
 *
 * Operators (as described on the Liger-Kernel pages):
 *   - RMSNorm forward / backward, a per-row reduction;
 *   - RoPE, rotating Q and K in place (and its variants: interleaved
 *     pairing, strided Q/K views of a packed QKV buffer, caller tables);
 *   - the SwiGLU activation silu(gate) * up and its backward;
 *   - FusedLinearSwiGLU: the gate and up projections and the activation in
 *     one tensor-core GEMM, and its backward;
 *   - the fused RMSNorm + QKV projection + RoPE forward;
 *   - a fused linear cross-entropy that never writes the full [T x V]
 *     logits to device memory (token-chunked, and a two-pass
 *     vocabulary-chunked variant).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc'd or from a
 *     device caching allocator) unless stated otherwise.  Tensors are dense
 *     and row-major (C order).  Float tensor pointers must be 16-byte
 *     aligned.
 *   - The library allocates nothing and frees nothing: the caller owns every
 *     buffer, including workspaces, and must keep them alive until the work
 *     queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls queue work on it and return without waiting, except
 *     liger_linear_ce_fwd_bwd and liger_linear_ce_two_pass_fwd_bwd, which
 *     wait for their label scan (see there).
 *   - `dtype` is LIGER_F32 or LIGER_BF16 and applies to every float tensor
 *     of the call except the ones documented as float (rstd, loss); all
 *     arithmetic is fp32 whatever the storage type.
 *   - Sizes are element counts (int64_t).  Zero-sized problems are valid and
 *     launch nothing.
 *   - Every call returns a status (LIGER_OK = 0 or a negative code below).
 *     Argument checks run before any work is queued: a call that fails them
 *     queues nothing and leaves every output untouched.
 *     liger_last_error() then describes the failure (per calling thread).
 *   - The current CUDA device is the one the pointers belong to.
 *   - Calls may come from several host threads at once, on any streams and
 *     devices, as long as they do not share output or workspace buffers
 *     (liger_rmsnorm_bwd_noalloc shares its scratch array: see there).  The
 *     library's own per-device state (kernel attributes, occupancy, the
 *     tensor-map encoder) is set up on first use and safe to race.
 *   - After a first call on a device, every entry point except
 *     liger_linear_ce_fwd_bwd and liger_linear_ce_two_pass_fwd_bwd (which
 *     wait for their label scan) can be captured in a CUDA graph; their
 *     _async forms do not wait.
 *   - Every wait inside the tensor-core kernels and the staged RMSNorm and
 *     RoPE kernels is bounded (about 4 s); one that expires (never seen in
 *     normal operation) ends the kernel early, its outputs incomplete.  The
 *     linear cross-entropies then return a NaN loss; the RMSNorm and RoPE
 *     kernels write NaN into the rows they did not finish (and into dw);
 *     RMSNorm, RoPE, FusedLinearSwiGLU and the fused RMSNorm + QKV + RoPE
 *     also record the expiry in library-owned device words that
 *     liger_device_status reads back and clears.
 */
#ifndef LIGER_H
#define LIGER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage types */
#define LIGER_F32 0
#define LIGER_BF16 1

/* status codes */
#define LIGER_OK 0
#define LIGER_ERR_NULL (-1)       /* a required pointer is NULL */
#define LIGER_ERR_SHAPE (-2)      /* a size is negative or inconsistent */
#define LIGER_ERR_DTYPE (-3)      /* dtype is not LIGER_F32 / LIGER_BF16 */
#define LIGER_ERR_ALIGN (-4)      /* a float tensor pointer is not 16-byte aligned */
#define LIGER_ERR_LABEL (-5)      /* a label is outside [0, V) and is not ignore_index */
#define LIGER_ERR_WORKSPACE (-6)  /* workspace missing or smaller than required */
#define LIGER_ERR_CUDA (-7)       /* a CUDA runtime call or kernel launch failed */

/* Message for the last failing call on this thread ("" if none). */
const char* liger_last_error(void);

/* Status of the work already queued on the current device.
 *
 * The calls return their status when they queue work, before it runs; an
 * expired bounded wait inside a kernel happens later.  The linear
 * cross-entropies report one through their NaN loss.  The staged RMSNorm
 * kernels, FusedLinearSwiGLU, the fused RMSNorm + QKV + RoPE and the staged
 * RoPE kernel record it in four library-owned device words (one per family,
 * per device).  This call queues a one-thread kernel on `stream` that reads
 * and clears the four words, waits for `stream` (cudaStreamSynchronize), and returns LIGER_OK if
 * none was set, else LIGER_ERR_CUDA with liger_last_error() naming the
 * families whose wait expired.  It covers the work queued on `stream` before
 * it and any other work of the library on the device that has finished by
 * then; an expiry in a kernel still running on another stream shows at a
 * later call.  Each word is cleared when read, so a second call returns
 * LIGER_OK until a new expiry.  A failing CUDA call (no device, an earlier
 * kernel fault) also returns LIGER_ERR_CUDA.  Not for use inside a stream
 * capture (it waits for the stream).
 */
int liger_device_status(void* stream);

/* Marks family `which` (0 = RMSNorm, 1 = FusedLinearSwiGLU, 2 = fused
 * RMSNorm + QKV + RoPE, 3 = RoPE) as an expired wait would, by a one-thread
 * kernel on `stream`, without any wait expiring: for tests of
 * liger_device_status and of the caller's own handling of it.
 * LIGER_ERR_SHAPE for another `which`.
 */
int liger_device_status_mark(int which, void* stream);

/* ------------------------------------------------------------- RMSNorm
 * Source: the RMSNorm step of the fused RMSNorm + QKV + RoPE kernel on the
 * page "Liger-Kernel底层优化：新一代内核级推理加速引擎介绍", section
 * "融合内核是如何工作的？来看一段简化版实现": the row's sum of squares over the
 * hidden size plus epsilon, under an inverse square root, scales the element
 * and the per-feature weight.
 *
 * Forward, per row r of x [rows, cols]:
 *     rstd[r] = 1 / sqrt(mean_j x[r,j]^2 + eps)
 *     y[r,j]  = x[r,j] * rstd[r] * w[j]            (one rounding, at the store)
 *   x, y: [rows, cols] in dtype; w: [cols] in dtype; rstd: [rows] float, may
 *   be NULL (not stored).  y may alias x.
 */
int liger_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t rows, int64_t cols,
                      float eps, int dtype, void* stream);

/* Bytes of workspace liger_rmsnorm_bwd needs (fp32 per-block partial sums of
 * dw): an upper bound valid on any device, min(rows, 1024) * cols * 4. */
size_t liger_rmsnorm_bwd_workspace(int64_t rows, int64_t cols);

/* Backward (the derivative of the forward; the pages give none):
 *     g = dy * w,   s_r = sum_j g[r,j] x[r,j]
 *     dx[r,j] = rstd[r] * g[r,j] - rstd[r]^3 / cols * x[r,j] * s_r
 *     dw[j]   = sum_r dy[r,j] * x[r,j] * rstd[r]
 *   dy, x, dx: [rows, cols]; w, dw: [cols], all in dtype; rstd: [rows] float
 *   as written by the forward.  dx may alias dy.  dw is reduced in a fixed
 *   order (deterministic run to run on one device).
 *   ws: device workspace of at least liger_rmsnorm_bwd_workspace(rows, cols)
 *   bytes, 16-byte aligned; its contents on entry do not matter.
 */
int liger_rmsnorm_bwd(const void* dy, const void* x, const void* w, const float* rstd, void* dx, void* dw,
                      void* ws, size_t ws_bytes, int64_t rows, int64_t cols, int dtype, void* stream);

/* RMSNorm backward that allocates nothing and takes no workspace.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory when they call the backward: code whose
 * operator interface carries only its input and output tensors and has no
 * slot for a scratch buffer, loops that must not call cudaMalloc (it can wait
 * for the whole device to go idle and so stalls other streams), and
 * processes that make every device allocation once, at start-up, under a
 * fixed memory budget.
 *
 * Same operator, arguments and results as liger_rmsnorm_bwd, without ws and
 * ws_bytes.  The per-block fp32 partial sums of dw go to a scratch array of
 * LIGER_RMSNORM_BWD_NOALLOC_SCRATCH_BYTES (16 MiB) that the library reserves
 * in device memory itself: every GPU on which the library is loaded holds
 * that array until the process exits.  The first call on each device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call on a device before any stream capture.  The
 * function calls no cudaMalloc, cudaFree or allocating library routine.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero: a call writes every partial sum it
 *     reads.  Calls whose work can overlap on the GPU (several streams,
 *     several host threads) race on the array: the caller must order them.
 *   - Partial rows: min(rows, 2 x SMs, 1024, 16 MiB / (4 * cols)).
 *     liger_rmsnorm_bwd may split the rows into a different number of
 *     partials (it sizes its grid by the resident blocks per SM), so dw may
 *     differ from it by rounding only (dx too: its row sums may be reduced
 *     in another order).
 *   - cols above 16 MiB / 4 = 4194304 does not fit one partial row: the call
 *     returns LIGER_ERR_WORKSPACE and queues nothing.
 */
#define LIGER_RMSNORM_BWD_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int liger_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* w, const float* rstd, void* dx, void* dw,
                              int64_t rows, int64_t cols, int dtype, void* stream);

/* ---------------------------------------------------------------- RoPE
 * Source: the FusedRoPE paragraph of the page "Liger-Kernel核心技术：
 * RollingBuffer与融合算子详解", section "算子融合" (the angle comes from the
 * token position, generated in the kernel with no stored table), and the
 * RoPE step of the fused-kernel listing on the page "Liger-Kernel底层优化：
 * 新一代内核级推理加速引擎介绍" (feature f is paired by f mod head_dim/2).
 *
 * In place on q [batch, seq, n_q_heads, head_dim] and k [batch, seq,
 * n_k_heads, head_dim]: for each head and pair i in [0, head_dim/2),
 *     phi = p * theta^(-2i/head_dim),   p = pos[b*seq + s] or s if pos is NULL
 *     (a, b) = (v[i], v[i + head_dim/2])
 *     v[i] = a cos(phi) - b sin(phi),   v[i + head_dim/2] = b cos(phi) + a sin(phi)
 * The angle is formed and reduced modulo 2 pi in double precision, then
 * cos/sin are taken in single precision.  head_dim must be even.  pos is an
 * int32 device array [batch, seq] of values >= 0, or NULL.  q (k) may be NULL
 * only when n_q_heads (n_k_heads) is 0.  q and k must not overlap: each block
 * of tokens is read into shared memory, rotated there and written back.
 */
int liger_rope_fwd(void* q, void* k, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                   int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream);

/* Backward: the same rotation by -phi (the transpose of the forward map),
 * applied in place to the incoming gradients dq, dk.  Arguments as above. */
int liger_rope_bwd(void* dq, void* dk, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                   int64_t n_k_heads, int64_t head_dim, double theta, int dtype, void* stream);

/* RoPE variants (the other conventions in use beside the pages' half-split
 * pairing), same rotation and the same in-place semantics:
 *   - pairing 0: pairs (i, i + head_dim/2) (as liger_rope_fwd); pairing 1:
 *     interleaved pairs (2i, 2i+1), angle index i;
 *   - q_token_stride / k_token_stride: elements between consecutive tokens
 *     (b, s) of q / k (>= heads * head_dim), so that q and k can be views into
 *     a packed [batch, seq, (n_q + 2 n_k) * head_dim] QKV buffer; heads of a
 *     token stay contiguous (head h at h * head_dim);
 *   - cos_tab / sin_tab: both NULL (angles from theta as above), or both
 *     [n_tab, head_dim/2] float device tables indexed by position, used as
 *     given (for scaled frequency schedules); theta is then ignored.  Positions
 *     outside [0, n_tab) are clamped to the table; keep them inside.
 *   q and k need only be aligned to their element size here (views into a
 *   packed buffer); 16-byte aligned head starts select the vector path.
 *   The _bwd variant negates the sine (transpose of the forward map).
 */
int liger_rope_fwd_ex(void* q, void* k, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                      int64_t n_k_heads, int64_t head_dim, int64_t q_token_stride, int64_t k_token_stride, int pairing,
                      const float* cos_tab, const float* sin_tab, int64_t n_tab, double theta, int dtype,
                      void* stream);
int liger_rope_bwd_ex(void* dq, void* dk, const int32_t* pos, int64_t batch, int64_t seq, int64_t n_q_heads,
                      int64_t n_k_heads, int64_t head_dim, int64_t q_token_stride, int64_t k_token_stride, int pairing,
                      const float* cos_tab, const float* sin_tab, int64_t n_tab, double theta, int dtype,
                      void* stream);

/* -------------------------------------------------------------- SwiGLU
 * Source: the FusedLinearSwiGLU paragraph of the page "Liger-Kernel核心技术：
 * RollingBuffer与融合算子详解", section "算子融合": SiLU of the gate branch,
 * then an elementwise product with the up branch, in registers.
 *
 * Forward:  y = silu(gate) * up,  silu(g) = g / (1 + exp(-g)).
 *   gate, up, y: n elements in dtype (any shape; the op is pointwise).
 *   y may alias gate or up.
 */
int liger_swiglu_fwd(const void* gate, const void* up, void* y, int64_t n, int dtype, void* stream);

/* Backward (textbook derivative):  s = sigmoid(g)
 *     dup   = dy * g * s
 *     dgate = dy * up * s * (1 + g * (1 - s))
 *   dgate may alias gate and dup may alias up (in-place backward). */
int liger_swiglu_bwd(const void* dy, const void* gate, const void* up, void* dgate, void* dup, int64_t n,
                     int dtype, void* stream);

/* ------------------------------------ fused RMSNorm + QKV projection + RoPE
 * Source: the fused kernel on the page "Liger-Kernel底层优化：新一代内核级推理
 * 加速引擎介绍", section "融合内核是如何工作的" (RMSNorm step, Q/K/V projection
 * with bias, RoPE on q and k, nothing written in between).  Forward only.
 *
 *   r_t = 1 / sqrt(mean_i x[t,i]^2 + eps)                      (rstd, fp32 [T])
 *   q[t] = RoPE_p(r_t (x[t] * w) Wq^T + bq)   [B, S, Hq, D]
 *   k[t] = RoPE_p(r_t (x[t] * w) Wk^T + bk)   [B, S, Hk, D]
 *   v[t] =        r_t (x[t] * w) Wv^T + bv    [B, S, Hk, D]
 * with RoPE as liger_rope_fwd (pairs (i, i + D/2) in every head, angle
 * p * theta^(-2i/D), p = pos[b, s] or s; here the angle is reduced modulo
 * 2 pi in single precision from an exact product, within a few 1e-7 rad for
 * positions below 2^24), or, given cos_tab / sin_tab
 * ([n_tab, D/2] fp32, indexed by position, clamped to the table), those
 * values as given.
 *   x [B*S, H], w_norm [H], Wq [Hq*D, H], Wk and Wv [Hk*D, H] (nn.Linear
 *   layout), biases bq [Hq*D], bk and bv [Hk*D] or NULL (no bias): all bf16,
 *   dense row-major, 16-byte aligned (biases 2-byte).  pos: int32 [B, S] or
 *   NULL.  rstd: fp32 [B*S] output or NULL.  hidden >= 64 and a multiple of
 *   8; head_dim 64, 128 or 256.
 * The norm weight is folded into the projection weights (bf16(W * w)) inside
 * ws, so the normalised rows and the un-rotated q, k never reach device
 * memory.  flags bit 0 set: ws already holds the folded weights and biases of
 * an earlier call with the same w_norm, W and b (they are then not read and
 * may be NULL).
 * ws: liger_rmsnorm_qkv_rope_workspace(B*S, H, Hq, Hk, D) bytes, 256-byte
 * aligned, owned by the caller (the folded weights first, so a workspace
 * sized for more tokens can be reused).  Asynchronous on `stream`.
 * Errors: LIGER_ERR_DTYPE (not bf16), LIGER_ERR_SHAPE, LIGER_ERR_NULL,
 * LIGER_ERR_ALIGN, LIGER_ERR_WORKSPACE, LIGER_ERR_CUDA.  B*S = 0 is a no-op.
 */
size_t liger_rmsnorm_qkv_rope_workspace(int64_t tokens, int64_t hidden, int64_t n_q_heads, int64_t n_k_heads,
                                        int64_t head_dim);
int liger_rmsnorm_qkv_rope_fwd(const void* x, const void* w_norm, const void* Wq, const void* Wk, const void* Wv,
                               const void* bq, const void* bk, const void* bv, const int32_t* pos,
                               const float* cos_tab, const float* sin_tab, int64_t n_tab, void* q, void* k, void* v,
                               float* rstd, void* ws, size_t ws_bytes, int64_t batch, int64_t seq, int64_t hidden,
                               int64_t n_q_heads, int64_t n_k_heads, int64_t head_dim, double eps, double theta,
                               int flags, int dtype, void* stream);

/* ---------------------------------------------- FusedLinearSwiGLU
 * Source: the FusedLinearSwiGLU paragraph of the page "Liger-Kernel核心技术：
 * RollingBuffer与融合算子详解", section "算子融合": x @ W_g and x @ W_u in one
 * kernel, SiLU and the product in registers, only the result written.
 *
 * Forward:  h = silu(X W_g^T) * (X W_u^T)
 *   X [T, H], W_g and W_u [I, H] (nn.Linear layout, no bias), h [T, I]; bf16
 *   only (tcgen05 tensor cores, fp32 accumulation); H >= 64 and H, I multiples
 *   of 8.  The gate and up products never reach device memory.
 *   All tensors dense row-major, 16-byte aligned, device memory owned by the
 *   caller; asynchronous on `stream`.  Errors: LIGER_ERR_DTYPE (not bf16),
 *   LIGER_ERR_SHAPE, LIGER_ERR_NULL, LIGER_ERR_ALIGN, LIGER_ERR_CUDA.  T = 0
 *   is a no-op (X and out may be null).
 */
int liger_fused_linear_swiglu_fwd(const void* X, const void* Wg, const void* Wu, void* out, int64_t T, int64_t H,
                                  int64_t I, int dtype, void* stream);

/* Bytes of workspace the backward needs: dG and dU, [T, I] bf16 each. */
size_t liger_fused_linear_swiglu_workspace(int64_t T, int64_t I);

/* Backward from dH [T, I]: g and u are recomputed (not saved by the forward);
 * with s = sigmoid(g), dG = dH u s (1 + g (1 - s)) and dU = dH g s,
 *     dX = dG W_g + dU W_u [T, H],  dW_g = dG^T X,  dW_u = dU^T X [I, H]
 * (written, not accumulated).  ws: at least
 * liger_fused_linear_swiglu_workspace(T, I) bytes, 256-byte aligned, else
 * LIGER_ERR_WORKSPACE; other errors as the forward.  T = 0 writes zero dW_g and
 * dW_u (X, dH, dX and ws may then be null). */
int liger_fused_linear_swiglu_bwd(const void* X, const void* Wg, const void* Wu, const void* dH, void* dX, void* dWg,
                                  void* dWu, void* ws, size_t ws_bytes, int64_t T, int64_t H, int64_t I, int dtype,
                                  void* stream);

/* The same pair with the activations kept instead of recomputed (memory for
 * speed): liger_fused_linear_swiglu_fwd_save also writes g = X W_g^T and
 * u = X W_u^T ([T, I] bf16, caller-owned, 16-byte aligned; required when
 * T > 0) from the same GEMM, and liger_fused_linear_swiglu_bwd_saved takes
 * them back: dG, dU by the elementwise SwiGLU backward (as liger_swiglu_bwd),
 * then dX and dW_g, dW_u as above -- 8 T H I flops instead of 12, with g and
 * u rounded to bf16 where the recomputing backward uses them in fp32.  Same
 * workspace, arguments and errors otherwise. */
int liger_fused_linear_swiglu_fwd_save(const void* X, const void* Wg, const void* Wu, void* out, void* g, void* u,
                                       int64_t T, int64_t H, int64_t I, int dtype, void* stream);
int liger_fused_linear_swiglu_bwd_saved(const void* X, const void* Wg, const void* Wu, const void* dH, const void* g,
                                        const void* u, void* dX, void* dWg, void* dWu, void* ws, size_t ws_bytes,
                                        int64_t T, int64_t H, int64_t I, int dtype, void* stream);

/* ------------------------------------------------ fused linear + CE
 * Source: the FusedCrossEntropyLoss paragraph of the page "Liger-Kernel核心
 * 技术：RollingBuffer与融合算子详解", section "算子融合" (softmax and NLL
 * merged, the softmax never stored), with the running max / normaliser
 * merge of the online softmax described on the page "Liger-Kernel内核级优化：
 * FlashAttention与RollingBuffer详解".
 *
 *   z_t = W x_t  (fp32 accumulation), lse_t = log sum_v exp(z_t[v])
 *   loss = sum over rows with labels[t] != ignore_index of (lse_t - z_t[labels[t]]),
 *          divided by their count n_valid when reduction = 0 (mean; 0 if
 *          n_valid = 0), not divided when reduction = 1 (sum)
 *   D_t  = s * (softmax(z_t) - onehot(labels[t])),  s = grad_scale / n_valid
 *          (mean) or grad_scale (sum);  D_t = 0 on ignored rows
 *   dX = D W,  dW = D^T X
 *
 *   X: [T, H], W: [V, H] (row-major) in dtype; labels: [T] int64 device array;
 *   loss: one float on the device; dX: [T, H] and dW: [V, H] in dtype, each
 *   may be NULL (not computed).  Rows of dX whose label is ignore_index are
 *   written as +0.0.
 *   On the bf16 tensor-core path, when some labels are ignore_index, the
 *   tokens with the other labels are gathered (in order) into the workspace
 *   and only they go through the GEMMs: an ignored token needs no logits and
 *   adds nothing to dW (6 n_valid H V flops instead of 6 T H V); dX, lse and
 *   the loss terms are then put back in place, 0 on ignored rows.  The chunks
 *   below are chunks of those tokens.
 *   The tokens are processed in chunks of `chunk` rows (0 = automatic:
 *   min(T, 8192, max(128, ceil(T/2)), from 1024 rows on rounded up to a
 *   multiple of 256) on the bf16 tensor-core path; there a
 *   chunk above 8192 rows is rounded down to a multiple of 8192, at most
 *   65536); per chunk the logits
 *   exist only in a [chunk x V] workspace buffer, never as a [T x V] tensor
 *   (T > 128).  dW is accumulated across chunks in fp32.
 *   ws: device workspace of at least liger_linear_ce_workspace(T, H, V,
 *   chunk, dtype) bytes, 256-byte aligned.  On return ws begins with
 *   float lse[T] (0 on ignored rows); float loss_row[T] (lse_t -
 *   z_t[label], 0 on ignored rows) starts at byte offset 4*T rounded up to a
 *   multiple of 256.
 *   Labels are validated on the device before any other work; the call waits
 *   for that scan (one stream synchronisation) and returns LIGER_ERR_LABEL,
 *   with nothing else queued, if a label is outside [0, V) and is not
 *   ignore_index.
 */
size_t liger_linear_ce_workspace(int64_t T, int64_t H, int64_t V, int64_t chunk, int dtype);

int liger_linear_ce_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H, int64_t V,
                            int64_t ignore_index, int reduction, float grad_scale, float* loss, void* dX, void* dW,
                            void* ws, size_t ws_bytes, int64_t chunk, int dtype, void* stream);

/* Two-pass, vocabulary-chunked variant of the same operator (same loss, lse,
 * dX and dW, same arguments and error behaviour), for callers that cannot
 * hold a [chunk x V] buffer and a [V x H] fp32 accumulator: no buffer of the
 * vocabulary's width exists at all.
 *   pass 1: the logits GEMM keeps only per-tile (max, sum-exp) partials and
 *           the label logit (token chunks of up to 8192 rows) -> lse, loss;
 *   pass 2: per chunk of `vchunk` vocabulary rows (0 = automatic: 8192, at
 *           most V), the logits of all T tokens are recomputed and the
 *           softmax part of D for that chunk written to a [T x vchunk] bf16
 *           buffer; dX accumulates D_c W_c in an fp32 [T x H] buffer (when
 *           V > vchunk); the rows dW_c = D_c^T X are finished and written.
 *   8 T H V flops (the logits twice) against 6 T H V for
 *   liger_linear_ce_fwd_bwd; the workspace is O(T (H + vchunk)), not
 *   O(chunk V + V H).  As there, when some labels are ignore_index only the
 *   other tokens (gathered in order) go through both passes (8 n_valid H V
 *   flops); the workspace holds their X and dX rows for that.  bf16 only (tensor cores), H >= 64 and a multiple of 8,
 *   V >= 256, vchunk a multiple of 8.  ws: at least
 *   liger_linear_ce_two_pass_workspace(T, H, V, vchunk) bytes, 256-byte
 *   aligned, with float lse[T] and float loss_row[T] at the same offsets as
 *   above. */
size_t liger_linear_ce_two_pass_workspace(int64_t T, int64_t H, int64_t V, int64_t vchunk);

int liger_linear_ce_two_pass_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H,
                                     int64_t V, int64_t ignore_index, int reduction, float grad_scale, float* loss,
                                     void* dX, void* dW, void* ws, size_t ws_bytes, int64_t vchunk, int dtype,
                                     void* stream);

/* The two linear cross-entropies without their host wait, for callers that
 * capture a training step in a CUDA graph.  Same arguments, workspace and
 * results as liger_linear_ce_fwd_bwd and liger_linear_ce_two_pass_fwd_bwd,
 * except:
 *   - the call queues work only (no stream synchronisation), so it can be
 *     captured once the device has seen one call of either kind;
 *   - labels are checked on the device: a label outside [0, V) that is not
 *     ignore_index does not make the call fail; it is treated as ignored (not
 *     counted in n_valid, its lse, loss term and gradient rows 0) and the
 *     loss is NaN, so the error shows in the result.  Argument errors are
 *     still returned before anything is queued;
 *   - the count n_valid and the gradient scale are formed on the device, so
 *     the GEMMs run over all T tokens (the ignored ones give D = 0).
 * Results are bit-identical to the waiting variant whenever no label is
 * ignored; with ignored labels, lse and dX still are, while dW and the loss
 * are the same sums over a different grouping of the tokens (equal within
 * rounding). */
int liger_linear_ce_fwd_bwd_async(const void* X, const void* W, const int64_t* labels, int64_t T, int64_t H,
                                  int64_t V, int64_t ignore_index, int reduction, float grad_scale, float* loss,
                                  void* dX, void* dW, void* ws, size_t ws_bytes, int64_t chunk, int dtype,
                                  void* stream);
int liger_linear_ce_two_pass_fwd_bwd_async(const void* X, const void* W, const int64_t* labels, int64_t T,
                                           int64_t H, int64_t V, int64_t ignore_index, int reduction,
                                           float grad_scale, float* loss, void* dX, void* dW, void* ws,
                                           size_t ws_bytes, int64_t vchunk, int dtype, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LIGER_H */
