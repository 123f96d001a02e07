/*
 * lapnys.h - C ABI of the GB300 (sm_103a) library for Laplacian-kernel Nystrom
 * attention: forward and backward of
 *
 *     O = Z . A^+ . (C . V),   C = k(L, K),  P = k(Q, L),  A = k(L, L) + eps I,
 *     k(x, y) = exp(-||x - y||_1 / lambda),  Z = P  or  (P - mu) / sqrt(var + eta),
 *
 * with landmarks L average-pooled from K and A^+ the Newton-Schulz iterate
 * X_T (X_0 = alpha A, X_{t+1} = 2 X_t - X_t A X_t, alpha = 1/(|A|_1 |A|_inf)).
 *
 * Defining passages (page title, section):
 *  - kernel: "LaplacianFormer: Rethinking Linear Attention with Laplacian
 *    Kernel" (Dutch summary), Methodology 1; Arabic summary, section 2a.
 *  - Nystrom landmarks by average pooling, Newton-Schulz inverse, eps I:
 *    the same pages, Methodology 2 / section 2c; "[Paper review] SOFT:
 *    Softmax-free Transformer with Linear Complexity", Proposed method
 *    (S-hat = P^T A^+ P, A_0 = alpha A, A_{k+1} = 2 A_k - A_k A A_k, pooling).
 *  - normalised query feature map (centring + diagonal variance): Dutch
 *    summary Methodology 1, Arabic summary section 2b.
 *  - gradient through sgn(x - y) of the L1 distance: Dutch summary
 *    Methodology 1 (non-vanishing gradient), Arabic summary section 2a.
 *
 * Conventions for every entry point
 *  - Tensors q, k, v, out, dout, dq, dk, dv are DEVICE pointers to contiguous
 *    [B][H][N][d] arrays (d innermost), token n = y * grid_w + x on the
 *    grid_h x grid_w grid, 16-byte aligned, all of one element type `dtype`
 *    (LAPNYS_F32 = float, LAPNYS_BF16 = bfloat16).  Arithmetic is float32.
 *  - Landmarks: an mh x mw grid of windows, m = mh * mw; a square m has
 *    mh = mw = sqrt(m), any other m the factor pair shaped most like the token
 *    grid (smallest |log(mh / mw) - log(grid_h / grid_w)|, ties to the smaller
 *    mh).  Landmark a = i * mw + j is the mean of token rows
 *    [floor(i grid_h / mh), floor((i + 1) grid_h / mh)) and columns
 *    [floor(j grid_w / mw), floor((j + 1) grid_w / mw)): equal windows when
 *    mh | grid_h and mw | grid_w, otherwise adaptive windows that still
 *    partition the grid (EINVAL when mh > grid_h or mw > grid_w).
 *  - The caller owns and allocates everything: out, gradients, `ctx` (state
 *    saved by the forward for the backward) and `ws` (scratch).  The library
 *    allocates no device memory and does not synchronise.  Work is ordered on
 *    `stream` (0 = legacy default stream): lapnys_fwd and lapnys_bwd run part
 *    of it (the landmark solver and its reverse) on one high-priority stream
 *    per device that the library creates on its first call there; that part
 *    starts after the work already on `stream` and `stream` waits for it
 *    before the call's last kernel (CUDA events), so to the caller the call
 *    behaves as if all of it were on `stream`.  Calls from several host
 *    threads on one device take turns on that stream (a mutex).  Sizes come
 *    from lapnys_ctx_bytes / lapnys_workspace_bytes.
 *  - Return value: LAPNYS_OK, or an error code.  Argument errors (EINVAL,
 *    ENOSPC, ENOTSUP) are detected on the host before anything is enqueued, so
 *    nothing has been written.  ECUDA reports a failed launch (the CUDA error
 *    is left for cudaGetLastError-style inspection by the caller).
 *  - Not thread-safe only with respect to lapnys_profile_*; the compute entry
 *    points keep no state between calls.
 */
#ifndef LAPNYS_H
#define LAPNYS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LAPNYS_OK = 0,
  LAPNYS_EINVAL = 1,   /* bad dimension, pointer, alignment or parameter */
  LAPNYS_ECUDA = 2,    /* a kernel launch failed */
  LAPNYS_ETIMEOUT = 3, /* a bounded device wait expired (see lapnys_device_status) */
  LAPNYS_ENOSPC = 4,   /* ctx or workspace smaller than the *_bytes functions require */
  LAPNYS_ENOTSUP = 5,  /* valid request outside what this build supports (e.g. d) */
  LAPNYS_ESCRATCH = 6  /* problem too large for the built-in scratch of lapnys_fwd_static */
} lapnys_status;

enum { LAPNYS_F32 = 0, LAPNYS_BF16 = 1 };

/* flags:
 * LAPNYS_NORM   centre each landmark column of P over the slice's N queries and
 *               divide by sqrt(biased variance + 1e-5) (the "injective"
 *               normalised feature map of "LaplacianFormer", Arabic summary 2b);
 * LAPNYS_GAUSS  use the Gaussian kernel k(x, y) = exp(-|x - y|_2^2 / lambda)
 *               (the SOFT review's Proposed method: a symmetric, [0, 1]-valued
 *               Gaussian kernel) instead of the Laplacian kernel
 *               exp(-|x - y|_1 / lambda).  Same ctx, workspace and entry points;
 * LAPNYS_NORM_BATCH  with LAPNYS_NORM only (alone it is LAPNYS_EINVAL): take
 *               the mean and variance of each landmark column over the B * N
 *               queries of all B slices of a head (the same summary's diagonal
 *               estimate read as taken over the batch) instead of per slice; the
 *               backward then couples the B slices of a head through those
 *               statistics, so lapnys_bwd must see the same B as lapnys_fwd. */
enum { LAPNYS_NORM = 1u << 0, LAPNYS_GAUSS = 1u << 1, LAPNYS_NORM_BATCH = 1u << 2 };

/* Limits of this build: d in {16, 32, 64, 128}; 1 <= m <= min(N, 1024); a
 * landmark grid as above; 0 <= iters <= 64; lambda > 0; eps >= 0;
 * B * H * N * d < 2^31. */

/* Bytes of the caller-owned context written by lapnys_fwd and read by
 * lapnys_bwd (landmarks, A, alpha, all Newton-Schulz iterates, W, W-hat,
 * feature-map statistics).  Returns 0 for invalid dimensions. */
size_t lapnys_ctx_bytes(int B, int H, int N, int d, int m, int iters, unsigned flags);

/* Bytes of scratch memory needed by lapnys_fwd (with or without ctx) and by
 * lapnys_bwd for these dimensions.  Returns 0 for invalid dimensions. */
size_t lapnys_workspace_bytes(int B, int H, int N, int d, int m, int iters, unsigned flags);

/* Forward.  Writes out = Z . X_T . (C . V) for every (b, h) slice.
 *  tied_qk: 1 = queries and keys are one tensor (k may be NULL or equal q).
 *  ctx: NULL for inference only; otherwise ctx_bytes >= lapnys_ctx_bytes(...)
 *       and lapnys_bwd can be called with it afterwards.
 *  ws/ws_bytes: scratch, ws_bytes >= lapnys_workspace_bytes(...). */
int lapnys_fwd(const void* q, const void* k, const void* v, void* out,
               int B, int H, int N, int d, int grid_h, int grid_w, int m,
               float lambda, float eps, int iters, int tied_qk, cudaStream_t stream,
               int dtype, unsigned flags, void* ctx, size_t ctx_bytes,
               void* ws, size_t ws_bytes);

/* Inference forward that allocates nothing and takes no workspace.  No passage
 * of the paper corresponds to it: it exists for callers that cannot call
 * cudaMalloc, such as code running inside another framework's memory pool,
 * allocator-free embedded runtimes, or code that must not allocate between
 * two steps.  Same arguments and results as lapnys_fwd with ctx = NULL, minus
 * ctx and ws.
 *  - Scratch: a 32 MiB array compiled into the library (held on every GPU that
 *    loads it, until the process exits).  The forward uses these regions of
 *    it, each rounded up to 256 bytes (f = 4 bytes, mp = 64 ceil(m / 64), S the
 *    token splits of the key pass: about 1216 / (B H ceil(m / 64)), between 1
 *    and ceil(N / 64)):
 *      landmarks (two parts), W, W-hat  4 B H m d f
 *      A, two iterates, A X_t           4 B H m^2 f
 *      alpha record, statistics         B H (4 + 3 m) f
 *      token -> landmark index          N f
 *      key-pass partial sums            B H S mp d f
 *      statistics partials              3 B H S mp f
 *      packed query-pass tiles (bf16, d in {32, 64}, m > 64 only)
 *                                       B H mp (2 d + 1) f
 *    A problem whose regions add up to more than 32 MiB returns
 *    LAPNYS_ESCRATCH before anything is enqueued; use lapnys_fwd with a
 *    workspace instead.
 *  - Every call looks up the array's address in the current context (a
 *    host-side query; nothing is allocated).  The first call in a context may
 *    load the library's device code there: make that first call before any
 *    stream capture.
 *  - Every call shares the one array.  Calls whose work overlaps on the GPU
 *    (other streams, other host threads) race on it and give wrong results:
 *    serialise them, e.g. on one stream.  Each call fully rewrites what it
 *    reads, so leftovers of an earlier call do no harm. */
int lapnys_fwd_static(const void* q, const void* k, const void* v, void* out,
                      int B, int H, int N, int d, int grid_h, int grid_w, int m,
                      float lambda, float eps, int iters, int tied_qk, cudaStream_t stream,
                      int dtype, unsigned flags);

/* Backward of lapnys_fwd for the upstream gradient dout.  Needs the ctx written
 * by the forward with the same q, k, v and parameters.  Writes dq, dk, dv
 * (overwritten, not accumulated).  With tied_qk = 1, dk must be NULL and dq
 * receives the whole gradient of the shared query/key tensor (query path, key
 * path and the landmark-pooling path). */
int lapnys_bwd(const void* q, const void* k, const void* v, const void* dout,
               const void* ctx, void* dq, void* dk, void* dv,
               int B, int H, int N, int d, int grid_h, int grid_w, int m,
               float lambda, float eps, int iters, int tied_qk, cudaStream_t stream,
               int dtype, unsigned flags, void* ws, size_t ws_bytes);

/* Byte offsets of the intermediates inside ctx, for inspection and tests.
 * All float32 unless noted:
 *   L     [B*H][m][d]             landmarks: the fp32 value nearest to each
 *                                 window's exact mean
 *   Llo   [B*H][m][d]             the exact mean minus L (the backward decides
 *                                 sgn(x - l) against the exact mean: by L where
 *                                 x != L, by -sgn(Llo) where x == L)
 *   A     [B*H][m][m]             k(L, L) + eps I
 *   alpha [B*H][4]                alpha, |A|_1, |A|_inf, and in slot 3 the int32
 *                                 jc | (ir << 16) stored bitwise: jc the argmax
 *                                 column of |A|_1, ir the argmax row of |A|_inf
 *   X     [B*H][iters+1][m][m]    Newton-Schulz iterates X_0 .. X_T
 *   Y     [B*H][iters][m][m]      products A X_t
 *   W     [B*H][m][d]             C . V
 *   What  [B*H][m][d]             X_T . W
 *   stats [B*H][3][m]             mu, var, 1/sqrt(var + 1e-5) (LAPNYS_NORM only)
 *   idx   int32 [N]               landmark of each token (same for all slices)
 *   P     [B*H][N][mp]            kernel values k(q_j, l_a) before the feature-map
 *                                 normalisation, rows padded to mp = 64 ceil(m/64)
 *   C     [B*H][N][mp]            kernel values k(l_a, k_j), token-major (the
 *                                 transpose of the m x N matrix C)
 * P and C are what the backward reads instead of recomputing the N x m
 * kernel values. */
typedef struct {
  size_t L, Llo, A, alpha, X, Y, W, What, stats, idx, P, C, total;
} lapnys_ctx_layout;

int lapnys_ctx_offsets(int B, int H, int N, int d, int m, int iters, unsigned flags,
                       lapnys_ctx_layout* out);

/* Landmark pooling alone: L [B*H][m][d] float32 from k, and idx int32 [N]
 * (idx may be NULL).  Same rules as lapnys_fwd. */
int lapnys_pool(const void* k, float* L, int32_t* idx, int B, int H, int N, int d,
                int grid_h, int grid_w, int m, int dtype, cudaStream_t stream);

/* Batched fp32 product C[b] = alpha * op(A[b]) * op(B[b]) + beta * E[b] for
 * b < batch, the building block of the Newton-Schulz solver for m > 64 (the
 * products X_t (A X_t) and their reverse).  Row-major device matrices; op(A)
 * is M x K (A stored K x M when trans_a), op(B) is K x N (B stored N x K when
 * trans_b); E may alias C; E may be NULL when beta == 0.
 *  engine 0: FP32 FMA kernel (any shape).
 *  engine 1: tcgen05 tensor cores, TF32 with the three-term split
 *            hi*hi + hi*lo + lo*hi (fp32-level accuracy); needs M, N, K, the
 *            leading dimensions and strides to be multiples of 4 and 16-byte
 *            aligned pointers, else returns LAPNYS_ENOTSUP.
 * Asynchronous on `stream`. */
int lapnys_matmul(const float* A, const float* B, const float* E, float* C, int batch, int M, int N,
                  int K, int trans_a, int trans_b, int lda, int ldb, int lde, int ldc,
                  long long stride_a, long long stride_b, long long stride_e, long long stride_c,
                  float alpha, float beta, int engine, cudaStream_t stream);

/* ---- the attention block around the path -------------------------------
 * One multi-head layer (the SOFT review, Proposed method: the attention as one
 * layer of a pyramid vision-transformer backbone with embedding width C and H
 * heads):
 *
 *     [Q | K | V] = X W_qkv + b_qkv,   O_h = attention(Q_h, K_h, V_h),
 *     Y = [O_1 | ... | O_H] W_o + b_o,
 *
 * with the attention of lapnys_fwd for every (batch, head).
 *  - x, y, dy, dx: [B][N][C] (token n on the grid as in lapnys_fwd);
 *    w_qkv [C][S*H*d] row-major with column blocks (Q | K | V), S = 3 (tied = 0)
 *    or (Q = K | V), S = 2 (tied = 1), head h at columns h*d .. h*d + d - 1 of
 *    each block; b_qkv [S*H*d]; w_o [H*d][C]; b_o [C].  All DEVICE pointers of
 *    element type `dtype`, 16-byte aligned; b_qkv and b_o may be NULL (no bias).
 *  - C a multiple of 8 (at most 65536), B*N*max(3*H*d, C) < 2^31; the
 *    attention arguments (H, N, d, grid, m, lambda, eps, iters, flags) follow
 *    lapnys_fwd's rules and return its status codes.
 *  - The projections are this library's kernels with float32 accumulation:
 *    bf16 on the tcgen05 tensor cores (bf16 operands read in place, also the
 *    per-head tensors, with the bias, the rounding and the split into heads
 *    in the product's epilogue and the bias gradients summed by the product);
 *    float32 on the FP32 FMA pipe (plain fp32 products).  bf16 also needs
 *    H*d to be a multiple of 8 (else LAPNYS_ENOTSUP).
 *    The calls allocate nothing: every buffer is part of `ws` or ctx.  Q, K,
 *    V, the projected outputs and every gradient are rounded once to `dtype`.
 *  - lapnys_block_fwd writes y; with ctx != NULL it also saves, in ctx, the
 *    attention context and the Q, K, V and head outputs that lapnys_block_bwd
 *    reads (ctx == NULL: inference, they live in ws).
 *  - lapnys_block_bwd writes dx, dw_qkv, dw_o, and db_qkv / db_o unless NULL
 *    (column sums of the output gradients in a fixed order: deterministic).
 *  - Sizes: lapnys_block_ctx_bytes / lapnys_block_workspace_bytes (0 for
 *    invalid arguments); one workspace serves both entry points.
 *  - Errors as for lapnys_fwd; argument errors are found before anything is
 *    enqueued; a failed GEMM or launch returns LAPNYS_ECUDA. */
size_t lapnys_block_ctx_bytes(int B, int N, int C, int H, int d, int m, int iters, int tied,
                              int dtype, unsigned flags);
size_t lapnys_block_workspace_bytes(int B, int N, int C, int H, int d, int m, int iters, int tied,
                                    int dtype, unsigned flags);
int lapnys_block_fwd(const void* x, const void* w_qkv, const void* b_qkv, const void* w_o,
                     const void* b_o, void* y, int B, int N, int C, int H, int d, int grid_h,
                     int grid_w, int m, float lambda, float eps, int iters, int tied,
                     cudaStream_t stream, int dtype, unsigned flags, void* ctx, size_t ctx_bytes,
                     void* ws, size_t ws_bytes);
int lapnys_block_bwd(const void* x, const void* w_qkv, const void* w_o, const void* dy,
                     const void* ctx, void* dx, void* dw_qkv, void* db_qkv, void* dw_o, void* db_o,
                     int B, int N, int C, int H, int d, int grid_h, int grid_w, int m, float lambda,
                     float eps, int iters, int tied, cudaStream_t stream, int dtype,
                     unsigned flags, void* ws, size_t ws_bytes);

/* Synchronises the current device and reports whether a bounded device-side
 * wait (tensor-core pipeline barriers) expired since the last clear:
 * LAPNYS_ETIMEOUT if so (the affected results are invalid), LAPNYS_OK if not,
 * LAPNYS_ECUDA if the device reported an error.  clear != 0 resets the flag. */
int lapnys_device_status(int clear);

/* Self-test of the failure detection (no passage of the paper corresponds to
 * it).  Enqueues on `stream` one CTA that waits, with the bounded wait the
 * tensor-core kernels use but at most `polls` polls (1 <= polls <= 2^22), on
 * an mbarrier that nothing arrives on.  The wait expires, the kernel records the
 * expiry in the device word lapnys_device_status reads and returns, with no copy,
 * MMA or tensor memory in flight: afterwards lapnys_device_status(1) returns
 * LAPNYS_ETIMEOUT (and clears the word) while the context stays usable.
 * LAPNYS_EINVAL for polls out of range (nothing enqueued). */
int lapnys_wait_selftest(int polls, cudaStream_t stream);

/* Human-readable text for a status code (static storage). */
const char* lapnys_strerror(int status);

/* Instrumentation (host side, process-wide, not thread-safe):
 *  lapnys_launch_count: kernels this library has enqueued since load.
 *  lapnys_profile_enable(mode): mode 1 records a CUDA event pair around every
 *    launch from then on (on the launch's stream); mode 2 does the same and
 *    also runs lapnys_fwd / lapnys_bwd entirely on the caller's stream (no
 *    side stream), so that each kernel's time is its own rather than shared
 *    with the kernels that normally overlap it; mode 0 turns both off
 *    (LAPNYS_EINVAL for other values).  lapnys_profile_read, called after the
 *    caller synchronised, adds up elapsed times per kernel name and clears
 *    them.  Up to 4096 launches are recorded between reads; later ones are
 *    counted but not timed.
 *  lapnys_profile_read fills at most max_kernels entries (name pointer with
 *    static storage, launches, total milliseconds) and returns how many kernel
 *    names it found, or -1 if an event query failed.
 *  lapnys_fma_probe: enqueues on `stream` a kernel of 8 CTAs of 256 threads per
 *    SM in which every thread runs `iters` (1 .. 2^24) steps of 8 independent
 *    FP32 FMA chains, scalar (paired = 0) or as packed pairs (paired = 1,
 *    fma.rn.f32x2: two lane-ops per instruction), and stores in *lane_ops the
 *    FP32 lane-ops it executes; timing it gives the measured FP32 FMA rate of
 *    the device.  `sink` is a device float the kernel never writes in
 *    practice (it keeps the chains live).  No passage of the paper corresponds
 *    to it. */
uint64_t lapnys_launch_count(void);
int lapnys_profile_enable(int mode);
int lapnys_profile_read(const char** names, int* launches, double* total_ms, int max_kernels);
int lapnys_fma_probe(int paired, int iters, float* sink, unsigned long long* lane_ops,
                     cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LAPNYS_H */
