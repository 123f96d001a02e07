// Host-side internals of liblapnys: problem description, launch wrapper with
// launch counting and optional per-launch CUDA-event timing, and the launch
// functions each translation unit provides.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

namespace lapnys {

struct Prob {
  int B, H, BH, N, d, gh, gw, m, mh, mw, iters, tied, dtype;  // mh x mw landmark grid
  unsigned flags;
  float lam, eps;
  float ns;       // -log2(e) / lambda: k = exp2(ns * distance)
  float inv_lam;  // 1 / lambda
  int nt;         // landmark tiles of 64
  int mp;         // nt * 64
  int nblk;       // token blocks of 64
  int Sk, Sq, Sb; // token splits of the key pass, statistics pass, backward passes
  int Skt;        // token splits of the tensor-core key pass (0 when it is not used)
  int Stc;        // token splits of the tensor-core backward
  bool norm() const { return flags & 1u; }
  bool gauss() const { return flags & 2u; }  // Gaussian kernel instead of the Laplacian
  bool norm_batch() const { return flags & 4u; }  // statistics over the B slices of a head
};

// the attention entry points' argument checks (LAPNYS_OK or the status they return)
int check_attention(int B, int H, int N, int d, int gh, int gw, int m, float lam, float eps,
                    int iters, int dtype, unsigned flags);

// ---- instrumentation -------------------------------------------------------
int prof_begin(const char* name, cudaStream_t s);
void prof_end(int slot, cudaStream_t s);
void count_launch();

// Every launch is also an NVTX range named like its profiling record (a no-op
// unless a tool such as Nsight Systems is attached).
template <typename Kern, typename... Args>
inline cudaError_t launch(const char* name, Kern kern, dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args... args) {
  nvtxRangePushA(name);
  const int slot = prof_begin(name, st);
  kern<<<grid, block, smem, st>>>(args...);
  cudaError_t e = cudaGetLastError();
  prof_end(slot, st);
  count_launch();
  nvtxRangePop();
  return e;
}

// an NVTX range over a scope (the library's entry points)
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

// opt a kernel into more than 48 KB of dynamic shared memory (once per kernel)
template <typename Kern>
inline cudaError_t allow_smem(Kern kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// ---- launchers (return the first CUDA error, cudaSuccess otherwise) -------
// tensor-core forward passes (bf16, d = 32 or 64, m > 64): the query pass
// reads landmark and W-hat tiles packed by run_pack_q (pack_q_floats floats);
// the key pass writes [BH][Skt][mp][d] partials of W
bool fwd_tc_shape(int d, int m);
bool fwd_tc_ok(const Prob& p);
int key_tc_splits(int BH, int m, int nblk);
size_t pack_q_floats(const Prob& p);
cudaError_t run_pack_q(const Prob& p, const float* L, const float* What, float* pack,
                       cudaStream_t st);
cudaError_t run_query_tc(const Prob& p, const void* q, const float* pack, const float* stats,
                         void* out, float* kvout, cudaStream_t st);
cudaError_t run_key_tc(const Prob& p, const void* k, const void* v, const float* L, float* part,
                       float* kvout, cudaStream_t st);
// the same passes for the Gaussian kernel with the distances on the tensor
// cores too (|x|^2 + |l|^2 - 2 x.l); run_pack_qg writes the landmark records
// (BH * nt * (64 d + 64) floats) at packL and the W-hat tiles at packW
cudaError_t run_pack_qg(const Prob& p, const float* L, const float* What, void* packL, float* packW,
                        cudaStream_t st);
cudaError_t run_query_gtc(const Prob& p, const void* q, const void* packL, const float* packW,
                          const float* stats, void* out, float* kvout, cudaStream_t st);
cudaError_t run_key_gtc(const Prob& p, const void* k, const void* v, const float* L, float* part,
                        float* kvout, cudaStream_t st);
// landmarks: L [BH][m][d] f32 (the fp32 window means), Llo [BH][m][d] (the exact
// means minus L; may be null), idx [N] int32 (may be null)
cudaError_t run_pool(const Prob& p, const void* k, float* L, float* Llo, int32_t* idx,
                     cudaStream_t st);

// gram + alpha + Newton-Schulz, m <= 64: one CTA per slice, everything on chip.
// X has nx slots per slice, Y ny slots; slot of iterate t is t % nx (t % ny).
cudaError_t run_ns_small(const Prob& p, const float* L, float* A, float* alpha, float* X,
                         float* Y, int nx, int ny, cudaStream_t st);
// gram tiles for any m: A = k(L, L) + eps I
cudaError_t run_gram(const Prob& p, const float* L, float* A, cudaStream_t st);
// alpha = 1 / (|A|_1 |A|_inf) and X_0 = alpha A
cudaError_t run_alpha(const Prob& p, const float* A, float* alpha, float* X0, long x_bstride,
                      cudaStream_t st);

// batched C[b] = alpha op(A[b]) op(B[b]) + beta E[b] (fp32, row-major)
cudaError_t run_bgemm(bool ta, bool tb, int batch, int M, int N, int K, const float* A, int lda,
                      long sA, const float* B, int ldb, long sB, float* C, int ldc, long sC,
                      const float* E, int lde, long sE, float alpha, float beta, cudaStream_t st);

// batched C[b] = alpha (op(A1) op(B1) + op(A2) op(B2)) + beta E; sym: C symmetric,
// only tiles on/above the diagonal are computed and mirrored (K2 may be 0)
cudaError_t run_gemm2(bool ta, bool tb, bool sym, int batch, int M, int N, const float* A1, int lda1,
                      long sA1, const float* B1, int ldb1, long sB1, int K1, const float* A2,
                      int lda2, long sA2, const float* B2, int ldb2, long sB2, int K2, float* C,
                      int ldc, long sC, const float* E, int lde, long sE, float alpha, float beta,
                      cudaStream_t st);

// tensor-core (tcgen05, three-term TF32 split) batched product; tc_gemm_ok tells
// whether the shapes, strides and pointers meet its alignment needs
bool tc_gemm_ok(int M, int N, int K, int lda, int ldb, int ldc, int lde, long sA, long sB, long sC,
                long sE, const void* A, const void* B, const void* C, const void* E);
cudaError_t run_tcgemm(bool ta, bool tb, int batch, int M, int N, int K, const float* A, int lda,
                       long sA, const float* B, int ldb, long sB, float* C, int ldc, long sC,
                       const float* E, int lde, long sE, float alpha, float beta, cudaStream_t st);
// value of the device error word set by expired bounded waits (-1 on failure)
int read_wait_error(bool clear);
// device address of that word in the current context (null on failure)
int* wait_error_address();
// one CTA whose bounded wait (at most `polls` polls) expires on purpose and
// sets that word
cudaError_t run_wait_selftest(int polls, cudaStream_t st);
// polls of the bounded waits in the tensor-core kernels
int tc_wait_limit();
// the driver's tensor-map encoder (looked up through the runtime; null when the
// driver lacks it) and a tiled fp32 map: dims / strides (bytes, rank - 1 of
// them) / box as for cuTensorMapEncodeTiled, no swizzle, zero fill out of bounds
void* tensor_map_encoder();
bool encode_tiled_f32(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                      const cuuint64_t* stride, const cuuint32_t* box);
// a tiled bf16 map with the 128-byte swizzle (box rows of 64 elements)
// the same with 128-byte swizzle (the inner box must be 32 floats = 128 bytes)
bool encode_tiled_f32_sw128(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                            const cuuint64_t* stride, const cuuint32_t* box);
bool encode_tiled_bf16_sw128(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                             const cuuint64_t* stride, const cuuint32_t* box);

// ---- bf16 products of the attention block (k_proj.cu) ---------------------
// Geometry: B batch entries of N tokens, embedding width C, H heads of d, S
// projection blocks (3, or 2 when Q = K).  Operand sources (bf16):
enum : int {
  GOP_ROWS_K = 0,    // rows = tokens of [B][N][F], k = feature (contiguous)
  GOP_HEADS_K = 1,   // rows = tokens, k = (s, h, c) of the S tensors [B][H][N][d]
  GOP_W_K = 2,       // rows = n of a weight stored [n][k]
  GOP_TOK_MN = 3,    // rows = features of [B][N][F], k = tokens
  GOP_HEADS_MN = 4,  // rows = (s, h, c) of the tensors [B][H][N][d], k = tokens
  GOP_W_MN = 5,      // rows = n of a weight stored [k][n]
};
// epilogues: bf16 to the per-head tensors (+ bias), bf16 rows [B N][n] (+ bias),
// fp32 rows
enum : int { GEP_HEADS = 0, GEP_ROWS = 1, GEP_F32 = 2 };
struct GemmDims {
  int B, N, C, H, d, S;
};
// the product's needs: C and H d multiples of 8, a tensor-map encoder
bool gemm_bf16_ok(const GemmDims& g);
// ... and for the per-head operands: d = 64 or 128 (a head row holds whole 64-wide
// pieces)
bool gemm_heads_ok(const GemmDims& g);
// fp32 partial tiles the weight-gradient products need (the larger of the two)
size_t gemm_wgrad_floats(const GemmDims& g);
// D[tokens][Nn] = src (tokens x Kf) * w (Kf x Nn): src GOP_ROWS_K (src[0]) or
// GOP_HEADS_K (src[s], Kf = s H d); w GOP_W_K or GOP_W_MN; epilogue epi into
// out[] (GEP_HEADS: out[s] per block of H d columns), bias (bf16, Nn) or null
cudaError_t run_gemm_rows(const char* name, const GemmDims& g, int src_kind,
                          const void* const* src, int Kf, int w_kind, const void* w, int Nn,
                          int epi, void* const* out, const void* bias, cudaStream_t st);
// dw[Mf][Nn] = A^T B over all tokens (A: GOP_TOK_MN or GOP_HEADS_MN with Mf
// features, B likewise with Nn), bf16; db[Nn] = the column sums of B (when not
// null); part holds gemm_wgrad_floats(g) floats
cudaError_t run_gemm_wgrad(const char* name, const GemmDims& g, int a_kind,
                           const void* const* asrc, int Mf, int b_kind, const void* const* bsrc,
                           int Nn, float* part, void* dw, void* db, cudaStream_t st);

// dV = C dW for bf16 tokens (d = 32 / 64) from the kept kernel values C
// [BH][N][mp] and dW [BH][m][d]; writes dv [BH][N][d] in bf16
bool dv_tc_ok(const Prob& p);
// out[BH][N][d] (bf16) = C[BH][N][mp] (fp32, token-major) R[BH][m][d] (fp32): dV = C dW,
// or the forward's O = C W-hat when Q = K (P = C^T).  img: dv_image_floats(p)
// floats of scratch for R^T as the product's operand image.
size_t dv_image_floats(const Prob& p);
cudaError_t run_dv(const Prob& p, const float* C, const float* R, float* img, void* out,
                   const char* name, cudaStream_t st);
// FP32 FMA-rate probe: a grid of 8 CTAs of 256 threads per SM, each thread
// `iters` x 8 independent FMAs (paired: fma.rn.f32x2, two lane-ops each);
// *lane_ops = the FP32 lane-ops the launch executes
cudaError_t run_fma_probe(bool paired, int iters, float* sink, unsigned long long* lane_ops,
                          cudaStream_t st);
// the whole Newton-Schulz iteration (reverse: its exact reverse) of every
// slice in one cluster launch, for ns_cluster_ok(m); buffers as in the ctx and
// workspace layouts ([BH][nx or ny or 1][m][m])
bool ns_cluster_ok(int m);
cudaError_t run_ns_cluster(const Prob& p, bool reverse, const float* A, float* X, float* Y, int nx,
                           int ny, float* G, float* XG, float* Tm, float* dA, cudaStream_t st);

// forward passes; kvout (may be null): the pass's kernel values [BH][N][mp]
cudaError_t run_key_fwd(const Prob& p, const void* k, const void* v, const float* L, float* part,
                        float* kvout, cudaStream_t st);
cudaError_t run_reduce_parts(int BH, int S, int m, int mp, int d, const float* part, float* out,
                             cudaStream_t st);
cudaError_t run_qstats(const Prob& p, const void* q, const float* L, float* spart, cudaStream_t st);
cudaError_t run_stats_final(const Prob& p, const float* spart, float* stats, cudaStream_t st);
// the statistics partials of k_qstats from kernel values P already in memory
cudaError_t run_pstats(const Prob& p, const float* P, float* spart, cudaStream_t st);
// Z = (P - mu) * rsqrt(var + eta), 0 past m, from P and the statistics
cudaError_t run_zmap(const Prob& p, const float* P, const float* stats, float* Z, cudaStream_t st);
cudaError_t run_query_fwd(const Prob& p, const void* q, const float* L, const float* What,
                          const float* stats, void* out, float* kvout, cudaStream_t st);

// backward
// mode 0: query side statistics pass (LAPNYS_NORM only): dWhat and sum dZ, sum dZ*Z partials
// mode 1: query side gradients: dQ partials per landmark tile, dL partials, (no norm) dWhat partials
// mode 2: key side gradients: dK, dV partials per landmark tile, dL partials
struct BwdArgs {
  const void* X;      // q (modes 0, 1) or k (mode 2)
  const void* U;      // dout (modes 0, 1) or v (mode 2)
  const float* L;     // landmarks
  const float* Llo;   // exact landmark means minus L
  const float* R;     // What (modes 0, 1) or dW (mode 2)
  const float* stats; // mu, var, rs [BH][3][m] (norm)
  const float* mdz;   // [BH][2][mp] mean dZ, mean dZ*Z (norm, mode 1)
  float* tok_part;    // [nt][BH][N][d]: dQ (mode 1) or dK (mode 2)
  float* tok_part2;   // [nt][BH][N][d]: dV (mode 2)
  float* lm_part;     // [BH][S][mp][d]: dL
  float* lm_part2;    // [BH][S][mp][d]: dWhat (modes 0, 1)
  float* ns_part;     // [BH][S][2][mp]: sum dZ, sum dZ*Z (mode 0)
  const uint32_t* ties; // [BH][ceil(N / 32)][kTieRec]: tie records (modes 1, 2)
  const float* kv;      // [BH][N][mp]: kernel values P (mode 1) or C (mode 2) of the forward
};
cudaError_t run_bwd_tile(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st);
// modes 1 and 2 with the FMA-pipe sign term (32-token blocks)
cudaError_t run_bwd_pair(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st);
// tie detection for the sign term: run_tie_prep reads the landmarks into
// `scratch` (ties_scratch_bytes); run_ties writes one record of kTieRec words
// per 32-token block of x ([BH][ceil(N / 32)][kTieRec]): word 0 is the number
// of ties n, or kTieExact when the block must take the exact sign path (a value
// out of the fast path's range, or more than kTieRec - 1 ties); words 1..n are
// the ties, ascending, each packed as token-in-block | feature << 5 |
// landmark << 12, for a token value equal to a landmark value
constexpr int kTieRec = 16;
constexpr uint32_t kTieExact = 0x80000000u;
size_t ties_scratch_bytes(int BH, int m, int d);
cudaError_t run_tie_prep(const Prob& p, const float* L, void* scratch, cudaStream_t st);
cudaError_t run_ties(const Prob& p, const void* x, void* scratch, uint32_t* rec, cudaStream_t st);
cudaError_t run_mdz(const Prob& p, const float* ns_part, float* mdz, cudaStream_t st);
cudaError_t run_gram_bwd(const Prob& p, const float* L, const float* Llo, const float* A,
                         const float* dA, float* dLA, cudaStream_t st);
// Newton-Schulz backward for m <= 64 (full ctx: iters + 1 iterates, iters products);
// GT = dLoss/dX_T; writes dA including the alpha term
cudaError_t run_ns_bwd_small(const Prob& p, const float* A, const float* alpha, const float* X,
                             const float* Y, const float* GT, float* dA, cudaStream_t st);
cudaError_t run_alpha_bwd(const Prob& p, const float* A, const float* alpha, const float* G,
                          float* dA, cudaStream_t st);
// dLs = (sum over S splits of dLq and of dLc, plus dLA) / the landmark's window
// size ([BH][S][mp][d] partials): each token's share of its landmark's gradient
cudaError_t run_reduce_dl(const Prob& p, int S, const float* dLq, const float* dLc, const float* dLA,
                          float* dLs, cudaStream_t st);
cudaError_t run_zero(float* x, size_t n, cudaStream_t st);
// token gradients: the token-side partials plus dLs[idx[n]] (idx: the pool's
// token -> landmark map), converted to the tensor type
cudaError_t run_finalize(const Prob& p, const float* dQp, const float* dKp, const float* dVp,
                         const float* dLs, const int32_t* idx, void* dq, void* dk, void* dv,
                         cudaStream_t st);
// the same after the tensor-core backward: nq planes of dQ partials (0: dq was
// written already), nk planes of dK partials, one plane of dV (fp32; null: dv
// was written already)
cudaError_t run_finalize_tc(const Prob& p, int nq, const float* dQp, int nk, const float* dKp,
                            const float* dVp, const float* dLs, const int32_t* idx, void* dq,
                            void* dk, void* dv, cudaStream_t st);

// tensor-core backward tile kernel (bf16 tokens, d = 64): one CTA per token
// range and group of up to 256 landmarks; grid (S, bwd_tc_groups(m), BH)
struct BwdTcArgs {
  const void* X;          // q (mode 1) or k (mode 2)
  const void* U;          // dout (mode 1) or v (mode 2)
  const float* L;         // landmarks (fp32 means) and their low parts
  const float* Llo;
  const float* R;         // What (mode 1) or dW (mode 2)
  const float* stats;     // [BH][3][m] (norm)
  const float* mdz;       // [BH][2][mp] (norm, mode 1)
  const float* kv;        // [BH][N][mp]: P (mode 1) or C (mode 2)
  const uint32_t* ties;   // tie records of x
  void* out;              // dq itself (mode 1, untied, one landmark group), else null
  float* tok_part;        // [NG][BH][N][d] token partials when out is null
  float* lm_part;         // [BH][S][mp][d] dL partials
  float* lm_part2;        // [BH][S][mp][d] dW-hat partials (mode 1 without norm)
  int S;
};
bool bwd_tc_shape(int dtype, int d);
int bwd_tc_groups(int m);
int bwd_tc_splits(int BH, int m, int N);
cudaError_t run_bwd_tc(const Prob& p, int mode, const BwdTcArgs& a, cudaStream_t st);

}  // namespace lapnys
