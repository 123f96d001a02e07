// The attention block around the path: the QKV projection, the per-head
// attention of this library, and the output projection, forward and backward.
//
// "[Paper review] SOFT: Softmax-free Transformer with Linear Complexity",
// Proposed method: the attention is instantiated as one layer of a pyramid
// vision-transformer backbone (embedding width d_e, h heads).  Read as the
// plain multi-head layer: [Q | K | V] = X W_qkv + b_qkv, heads of d columns,
// Y = concat_h(O_h) W_o + b_o.
//
// The six projections are this library's own products.  bf16 layers: the
// tcgen05 GEMM of k_proj.cu, which reads the per-head tensors [B][H][N][d] in
// place and writes them from its epilogue (bias and rounding fused), so no head
// transpose runs between the products, and which sums the bias gradients
// through a row of ones; heads of d = 16 or 32 (a head row narrower than the
// product's 64-wide pieces) go through the layout kernels below and the same
// GEMM on row-major operands.  float32 layers: the FP32 FMA product
// of k_gemm2.cu, with the layout kernels below: the [B*N][S*H*d] <-> [B][H][N][d] head
// transposes fused with the bias addition and the rounding to the element type,
// and fixed-order column sums for the bias gradients.
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "lapnys.h"

namespace lapnys {
namespace {

constexpr int kBlockThreads = 256;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ---- layout kernels ---------------------------------------------------------
// A CTA takes `rpc` consecutive token rows; a thread takes pieces of
// consecutive columns (d is a multiple of 16, so a piece stays inside one head
// row), works out the piece's (block s, head h, offset j) once and walks the
// rows.  Rows are contiguous in the [B*N][W] side, head rows in the
// [B][H][N][d] side; consecutive threads of a head take consecutive pieces.
// Pieces: 4 columns where one side is float32, otherwise 16 bytes of T.
constexpr int kRowsWide = 64;    // rows per CTA when the CTA also sums its columns
constexpr int kRowsNarrow = 16;  // otherwise: more CTAs in flight per SM

template <typename T>
struct Piece {
  static constexpr int n = 16 / (int)sizeof(T);
};

__device__ __forceinline__ void ldp(const float* p, float (&v)[4]) {
  const float4 u = ld4(p);
  v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
}
__device__ __forceinline__ void stp(float* p, const float (&v)[4]) {
  st4(p, make_float4(v[0], v[1], v[2], v[3]));
}
__device__ __forceinline__ void ldp(const __nv_bfloat16* p, float (&v)[4]) {
  const float4 u = ld4(p);
  v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
}
__device__ __forceinline__ void stp(__nv_bfloat16* p, const float (&v)[4]) {
  st4(p, make_float4(v[0], v[1], v[2], v[3]));
}
__device__ __forceinline__ void ldp(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the high half of the bits
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void stp(__nv_bfloat16* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

struct ColMap {
  int s, h, j;
};
__device__ __forceinline__ ColMap col_map(int col, int HD, int d) {
  ColMap c;
  c.s = col / HD;
  const int hc = col - c.s * HD;
  c.h = hc / d;
  c.j = hc - c.h * d;
  return c;
}

// src [rows][S*H*d] float32 (+ bias [S*H*d]) -> dst_s [B][H][N][d] of T
template <typename T>
__global__ void k_split_heads(const float* __restrict__ src, const T* __restrict__ bias,
                              T* __restrict__ d0, T* __restrict__ d1, T* __restrict__ d2, int N,
                              int H, int d, int S, int rows, int rpc) {
  const int HD = H * d, W = S * HD;
  const int r0 = blockIdx.x * rpc, r1 = min(r0 + rpc, rows);
  for (int col = threadIdx.x * 4; col < W; col += blockDim.x * 4) {
    const ColMap c = col_map(col, HD, d);
    T* dst = c.s == 0 ? d0 : (c.s == 1 ? d1 : d2);
    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bias != nullptr) bv = ld4(bias + col);
    int b = r0 / N, n = r0 - b * N;
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      float4 v = ld4(src + (size_t)r * W + col);
      v.x += bv.x; v.y += bv.y; v.z += bv.z; v.w += bv.w;
      st4(dst + (((size_t)b * H + c.h) * N + n) * d + c.j, v);
      if (++n == N) { n = 0; ++b; }
    }
  }
}

// src_s [B][H][N][d] of T -> dst [rows][S*H*d] of T; with part != null also
// part[cta][col] = the column sums of the CTA's rows (in row order)
template <typename T, int P>
__global__ void k_merge_heads(const T* __restrict__ s0, const T* __restrict__ s1,
                              const T* __restrict__ s2, T* __restrict__ dst,
                              float* __restrict__ part, int N, int H, int d, int S, int rows,
                              int rpc) {
  const int HD = H * d, W = S * HD;
  const int r0 = blockIdx.x * rpc, r1 = min(r0 + rpc, rows);
  for (int col = threadIdx.x * P; col < W; col += blockDim.x * P) {
    const ColMap c = col_map(col, HD, d);
    const T* src = c.s == 0 ? s0 : (c.s == 1 ? s1 : s2);
    float acc[P];
#pragma unroll
    for (int i = 0; i < P; ++i) acc[i] = 0.f;
    int b = r0 / N, n = r0 - b * N;
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      float v[P];
      ldp(src + (((size_t)b * H + c.h) * N + n) * d + c.j, v);
      stp(dst + (size_t)r * W + col, v);  // v holds T values: stored exactly
#pragma unroll
      for (int i = 0; i < P; ++i) acc[i] += v[i];
      if (++n == N) { n = 0; ++b; }
    }
    if (part != nullptr)
#pragma unroll
      for (int i = 0; i < P; i += 4)
        st4(part + (size_t)blockIdx.x * W + col + i,
            make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]));
  }
}

// dst [rows][C] of T = src [rows][C] float32 + bias [C] (bias may be null)
template <typename T>
__global__ void k_bias_rows(const float* __restrict__ src, const T* __restrict__ bias,
                            T* __restrict__ dst, int C, int rows, int rpc) {
  const int r0 = blockIdx.x * rpc, r1 = min(r0 + rpc, rows);
  for (int col = threadIdx.x * 4; col < C; col += blockDim.x * 4) {
    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bias != nullptr) bv = ld4(bias + col);
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      float4 v = ld4(src + (size_t)r * C + col);
      v.x += bv.x; v.y += bv.y; v.z += bv.z; v.w += bv.w;
      st4(dst + (size_t)r * C + col, v);
    }
  }
}

// part[cta][col] = sum of G[r][col] over the CTA's rows, in row order
template <typename T>
__global__ void k_colsum_rows(const T* __restrict__ G, float* __restrict__ part, int cols,
                              int rows, int rpc) {
  constexpr int P = 4;
  const int r0 = blockIdx.x * rpc, r1 = min(r0 + rpc, rows);
  for (int col = threadIdx.x * P; col < cols; col += blockDim.x * P) {
    float acc[P];
#pragma unroll
    for (int i = 0; i < P; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      float v[P];
      ldp(G + (size_t)r * cols + col, v);
#pragma unroll
      for (int i = 0; i < P; ++i) acc[i] += v[i];
    }
#pragma unroll
    for (int i = 0; i < P; i += 4)
      st4(part + (size_t)blockIdx.x * cols + col + i,
          make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]));
  }
}

// out[col] = sum of the CTAs' partial sums: CTA (32 columns) x 32 rows of
// lanes; row y adds partials y, y + 32, ... in order, then row 0 adds the 32
// row sums in order (a fixed tree: deterministic)
constexpr int kSumRows = 32;
template <typename T>
__global__ void __launch_bounds__(32 * kSumRows)
    k_colsum_final(const float* __restrict__ part, T* __restrict__ out, int splits, int cols) {
  __shared__ float acc_s[kSumRows][33];
  const int col = blockIdx.x * 32 + threadIdx.x, y = threadIdx.y;
  float acc = 0.f;
  if (col < cols)
    for (int s = y; s < splits; s += kSumRows) acc += part[(size_t)s * cols + col];
  acc_s[y][threadIdx.x] = acc;
  __syncthreads();
  if (y != 0 || col >= cols) return;
  for (int j = 1; j < kSumRows; ++j) acc += acc_s[j][threadIdx.x];
  out[col] = from_f<T>(acc);
}

int row_ctas(int rows, int rpc) { return (rows + rpc - 1) / rpc; }
// threads of a row CTA: one per piece of `piece` columns, at most 512, whole warps
int row_threads(int cols, int piece) {
  int t = ((cols / piece + 31) / 32) * 32;
  return t > 512 ? 512 : t;
}

template <typename T>
cudaError_t split_heads_t(const float* src, const void* bias, void* d0, void* d1, void* d2, int B,
                          int N, int H, int d, int S, cudaStream_t st) {
  const int rows = B * N;
  // wide rows (at least 1024 columns) keep a CTA busy with 64 rows; narrow ones
  // take 16 so that more CTAs are in flight (measured on the 8-head layer)
  const int rpc = S * H * d >= 1024 ? kRowsWide : kRowsNarrow;
  return launch("block_split_heads", k_split_heads<T>, dim3(row_ctas(rows, rpc)),
                dim3(row_threads(S * H * d, 4)), 0, st, src, (const T*)bias, (T*)d0, (T*)d1,
                (T*)d2, N, H, d, S, rows, rpc);
}
template <typename T>
cudaError_t merge_heads_t(const void* s0, const void* s1, const void* s2, void* dst, float* part,
                          int B, int N, int H, int d, int S, cudaStream_t st) {
  const int rows = B * N;
  // measured on the 128 x 128, 8-head layer: with the column sums, 4-column
  // pieces and 64-row CTAs; without, 16-byte pieces and 16-row CTAs
  if (part != nullptr)
    return launch("block_merge_heads", k_merge_heads<T, 4>, dim3(row_ctas(rows, kRowsWide)),
                  dim3(row_threads(S * H * d, 4)), 0, st, (const T*)s0, (const T*)s1,
                  (const T*)s2, (T*)dst, part, N, H, d, S, rows, kRowsWide);
  return launch("block_merge_heads", k_merge_heads<T, Piece<T>::n>,
                dim3(row_ctas(rows, kRowsNarrow)), dim3(row_threads(S * H * d, Piece<T>::n)), 0,
                st, (const T*)s0, (const T*)s1, (const T*)s2, (T*)dst, part, N, H, d, S, rows,
                kRowsNarrow);
}
template <typename T>
cudaError_t bias_rows_t(const float* src, const void* bias, void* dst, int rows, int C,
                        cudaStream_t st) {
  return launch("block_bias_rows", k_bias_rows<T>, dim3(row_ctas(rows, kRowsNarrow)),
                dim3(row_threads(C, 4)), 0, st, src, (const T*)bias, (T*)dst, C, rows,
                kRowsNarrow);
}
template <typename T>
cudaError_t colsum_final_t(const float* part, void* out, int rows, int cols, cudaStream_t st) {
  return launch("block_colsum_final", k_colsum_final<T>, dim3((cols + 31) / 32),
                dim3(32, kSumRows), 0, st, part, (T*)out, row_ctas(rows, kRowsWide), cols);
}
template <typename T>
cudaError_t colsum_t(const void* G, float* part, void* out, int rows, int cols, cudaStream_t st) {
  cudaError_t e = launch("block_colsum", k_colsum_rows<T>, dim3(row_ctas(rows, kRowsWide)),
                         dim3(row_threads(cols, 4)), 0, st, (const T*)G, part, cols, rows,
                         kRowsWide);
  if (e != cudaSuccess) return e;
  return colsum_final_t<T>(part, out, rows, cols, st);
}

#define DT_CALL(dtype, fn, ...) \
  ((dtype) == LAPNYS_BF16 ? fn<__nv_bfloat16>(__VA_ARGS__) : fn<float>(__VA_ARGS__))

// ---- fp32 products -----------------------------------------------------------
// row-major C[M][N] (ldc) = op(A) op(B); op(A) is M x K (A stored K x M when ta),
// op(B) is K x N (B stored N x K when tb), on the FP32 FMA product: plain fp32
// arithmetic.  (The three-term TF32 split of the tensor-core product, about
// 1e-6 relative per product, was measured against the fp64 oracle on a float32
// layer: the attention's backward amplified the output projection's error and
// dX = dQKV W_qkv^T cancels, so dX and dW_qkv missed the fp32 tolerance by 5x.)
cudaError_t gemm_f32(bool ta, bool tb, int M, int N, int K, const void* A, int lda, const void* B,
                     int ldb, void* C, int ldc, cudaStream_t st) {
  return run_gemm2(ta, tb, false, 1, M, N, (const float*)A, lda, 0, (const float*)B, ldb, 0, K,
                   nullptr, 0, 0, nullptr, 0, 0, 0, (float*)C, ldc, 0, nullptr, 0, 0, 1.f, 0.f, st);
}

// ---- sizes ------------------------------------------------------------------
struct BlockLayout {
  // ctx: attention ctx, then the saved q, k (untied), v, and Ot [B*N][H*d]
  size_t c_attn, c_q, c_k, c_v, c_ot, c_total, attn_ctx;
  // forward ws: f32 scratch, O, saved tensors when there is no ctx, attention ws
  size_t f_s32, f_o, f_lite, f_attn, f_total;
  // backward ws: f32 scratch, dO, dq, dk, dv, dqkv, column-sum partials, weight-gradient
  // partials (bf16), attention ws
  size_t b_s32, b_do, b_dq, b_dk, b_dv, b_dqkv, b_part, b_gpart, b_attn, b_total;
  size_t attn_ws;
};

bool block_dims_ok(int B, int N, int C, int H, int d) {
  if (B <= 0 || N <= 0 || C <= 0 || H <= 0 || d <= 0) return false;
  if (C % 8 != 0 || C > (1 << 16)) return false;
  const long long rows = (long long)B * N;
  const long long wide = 3LL * H * d > C ? 3LL * H * d : C;
  return rows * wide < (1LL << 31);
}

BlockLayout block_layout(int B, int N, int C, int H, int d, int m, int iters, int tied, int dtype,
                         unsigned flags) {
  BlockLayout L;
  memset(&L, 0, sizeof(L));
  const size_t es = dtype == LAPNYS_BF16 ? 2 : 4;
  const size_t rows = (size_t)B * N, HD = (size_t)H * d, S = tied ? 2 : 3;
  const size_t head = rows * HD * es;  // one [B][H][N][d] tensor
  L.attn_ctx = lapnys_ctx_bytes(B, H, N, d, m, iters, flags);
  L.attn_ws = lapnys_workspace_bytes(B, H, N, d, m, iters, flags);
  size_t o = 0;
  L.c_attn = o; o = align256(o + L.attn_ctx);
  const size_t saved0 = o;
  L.c_q = o; o = align256(o + head);
  L.c_k = o; o = align256(o + (tied ? 0 : head));
  L.c_v = o; o = align256(o + head);
  L.c_ot = o; o = align256(o + head);
  L.c_total = o;
  const size_t saved = o - saved0;

  const size_t wide = (S * HD > (size_t)C ? S * HD : (size_t)C);
  o = 0;
  L.f_s32 = o; o = align256(o + rows * wide * 4);
  L.f_o = o; o = align256(o + head);
  L.f_lite = o; o = align256(o + saved);
  L.f_attn = o; o = align256(o + L.attn_ws);
  L.f_total = o;

  o = 0;
  L.b_s32 = o; o = align256(o + rows * HD * 4);
  L.b_do = o; o = align256(o + head);
  L.b_dq = o; o = align256(o + head);
  L.b_dk = o; o = align256(o + (tied ? 0 : head));
  L.b_dv = o; o = align256(o + head);
  L.b_dqkv = o; o = align256(o + rows * S * HD * es);
  L.b_part = o; o = align256(o + (size_t)row_ctas((int)rows, kRowsWide) * wide * 4);
  const GemmDims g = {B, N, C, H, d, (int)S};
  L.b_gpart = o; o = align256(o + (dtype == LAPNYS_BF16 ? gemm_wgrad_floats(g) * 4 : 0));
  L.b_attn = o; o = align256(o + L.attn_ws);
  L.b_total = o;
  return L;
}

bool a16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool a16_or_null(const void* p) { return p == nullptr || a16(p); }

#define CKB(x)                                   \
  do {                                           \
    if ((x) != cudaSuccess) return LAPNYS_ECUDA; \
  } while (0)

}  // namespace
}  // namespace lapnys

using namespace lapnys;

extern "C" {

size_t lapnys_block_ctx_bytes(int B, int N, int C, int H, int d, int m, int iters, int tied,
                              int dtype, unsigned flags) {
  if (!block_dims_ok(B, N, C, H, d) || (tied != 0 && tied != 1)) return 0;
  if (dtype != LAPNYS_F32 && dtype != LAPNYS_BF16) return 0;
  if (lapnys_ctx_bytes(B, H, N, d, m, iters, flags) == 0) return 0;
  return block_layout(B, N, C, H, d, m, iters, tied, dtype, flags).c_total;
}

size_t lapnys_block_workspace_bytes(int B, int N, int C, int H, int d, int m, int iters, int tied,
                                    int dtype, unsigned flags) {
  if (!block_dims_ok(B, N, C, H, d) || (tied != 0 && tied != 1)) return 0;
  if (dtype != LAPNYS_F32 && dtype != LAPNYS_BF16) return 0;
  if (lapnys_workspace_bytes(B, H, N, d, m, iters, flags) == 0) return 0;
  const BlockLayout L = block_layout(B, N, C, H, d, m, iters, tied, dtype, flags);
  return L.f_total > L.b_total ? L.f_total : L.b_total;
}

int lapnys_block_fwd(const void* x, const void* w_qkv, const void* b_qkv, const void* w_o,
                     const void* b_o, void* y, int B, int N, int C, int H, int d, int grid_h,
                     int grid_w, int m, float lambda, float eps, int iters, int tied,
                     cudaStream_t stream, int dtype, unsigned flags, void* ctx, size_t ctx_bytes,
                     void* ws, size_t ws_bytes) {
  NvtxScope nvtx_scope("lapnys_block_fwd");
  if (!block_dims_ok(B, N, C, H, d) || (tied != 0 && tied != 1)) return LAPNYS_EINVAL;
  int rc = check_attention(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, dtype, flags);
  if (rc != LAPNYS_OK) return rc;
  if (!x || !w_qkv || !w_o || !y || !ws) return LAPNYS_EINVAL;
  if (!a16(x) || !a16(w_qkv) || !a16(w_o) || !a16(y) || !a16(ws) || !a16_or_null(b_qkv) ||
      !a16_or_null(b_o) || !a16_or_null(ctx))
    return LAPNYS_EINVAL;
  const BlockLayout L = block_layout(B, N, C, H, d, m, iters, tied, dtype, flags);
  if (ws_bytes < L.f_total) return LAPNYS_ENOSPC;
  if (ctx != nullptr && ctx_bytes < L.c_total) return LAPNYS_ENOSPC;

  const int S = tied ? 2 : 3, HD = H * d;
  const int rows = B * N;
  const GemmDims g = {B, N, C, H, d, S};
  const bool bf = dtype == LAPNYS_BF16;
  if (bf && !gemm_bf16_ok(g)) return LAPNYS_ENOTSUP;
  const bool heads = bf && gemm_heads_ok(g);
  char* wb = (char*)ws;
  // saved tensors live in ctx for training, in ws for inference
  char* sb = ctx != nullptr ? (char*)ctx : wb + L.f_lite - L.c_q;
  void* q = sb + L.c_q;
  void* k = tied ? q : (void*)(sb + L.c_k);
  void* v = sb + L.c_v;
  // the attention's output O as the output projection reads it: [B][H][N][d] in
  // place (bf16 with per-head operands), else concatenated rows [B*N][H*d]
  void* ot = sb + L.c_ot;
  float* s32 = (float*)(wb + L.f_s32);
  void* O = heads ? ot : (void*)(wb + L.f_o);

  // [Q | K | V] = X W_qkv (+ b_qkv, split to heads)
  const void* xs[1] = {x};
  if (heads) {
    void* dst[3] = {q, tied ? v : k, v};
    CKB(run_gemm_rows("block_gemm_qkv", g, GOP_ROWS_K, xs, C, GOP_W_MN, w_qkv, S * HD, GEP_HEADS, dst, b_qkv,
                      stream));
  } else {
    if (bf) {
      void* dst[3] = {s32, nullptr, nullptr};
      CKB(run_gemm_rows("block_gemm_qkv", g, GOP_ROWS_K, xs, C, GOP_W_MN, w_qkv, S * HD, GEP_F32, dst, nullptr,
                        stream));
    } else {
      CKB(gemm_f32(false, false, rows, S * HD, C, x, C, w_qkv, S * HD, s32, S * HD, stream));
    }
    CKB(DT_CALL(dtype, split_heads_t, s32, b_qkv, q, tied ? v : k, v, B, N, H, d, S, stream));
  }
  rc = lapnys_fwd(q, tied ? nullptr : k, v, O, B, H, N, d, grid_h, grid_w, m, lambda, eps, iters,
                  tied, stream, dtype, flags, ctx != nullptr ? (char*)ctx + L.c_attn : nullptr,
                  L.attn_ctx, wb + L.f_attn, L.attn_ws);
  if (rc != LAPNYS_OK) return rc;
  // Y = concat_h(O_h) W_o + b_o
  void* ys[3] = {y, nullptr, nullptr};
  if (heads) {
    const void* os[1] = {ot};
    CKB(run_gemm_rows("block_gemm_out", g, GOP_HEADS_K, os, HD, GOP_W_MN, w_o, C, GEP_ROWS, ys, b_o,
                      stream));
    return LAPNYS_OK;
  }
  CKB(DT_CALL(dtype, merge_heads_t, O, nullptr, nullptr, ot, nullptr, B, N, H, d, 1, stream));
  if (bf) {
    const void* os[1] = {ot};
    CKB(run_gemm_rows("block_gemm_out", g, GOP_ROWS_K, os, HD, GOP_W_MN, w_o, C, GEP_ROWS, ys, b_o,
                      stream));
    return LAPNYS_OK;
  }
  CKB(gemm_f32(false, false, rows, C, HD, ot, HD, w_o, C, s32, C, stream));
  CKB(DT_CALL(dtype, bias_rows_t, s32, b_o, y, rows, C, stream));
  return LAPNYS_OK;
}

int lapnys_block_bwd(const void* x, const void* w_qkv, const void* w_o, const void* dy,
                     const void* ctx, void* dx, void* dw_qkv, void* db_qkv, void* dw_o, void* db_o,
                     int B, int N, int C, int H, int d, int grid_h, int grid_w, int m, float lambda,
                     float eps, int iters, int tied, cudaStream_t stream, int dtype,
                     unsigned flags, void* ws, size_t ws_bytes) {
  NvtxScope nvtx_scope("lapnys_block_bwd");
  if (!block_dims_ok(B, N, C, H, d) || (tied != 0 && tied != 1)) return LAPNYS_EINVAL;
  int rc = check_attention(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, dtype, flags);
  if (rc != LAPNYS_OK) return rc;
  if (!x || !w_qkv || !w_o || !dy || !ctx || !dx || !dw_qkv || !dw_o || !ws) return LAPNYS_EINVAL;
  if (!a16(x) || !a16(w_qkv) || !a16(w_o) || !a16(dy) || !a16(ctx) || !a16(dx) || !a16(dw_qkv) ||
      !a16(dw_o) || !a16(ws) || !a16_or_null(db_qkv) || !a16_or_null(db_o))
    return LAPNYS_EINVAL;
  const BlockLayout L = block_layout(B, N, C, H, d, m, iters, tied, dtype, flags);
  if (ws_bytes < L.b_total) return LAPNYS_ENOSPC;

  const int S = tied ? 2 : 3, HD = H * d;
  const int rows = B * N;
  const GemmDims g = {B, N, C, H, d, S};
  const bool bf = dtype == LAPNYS_BF16;
  if (bf && !gemm_bf16_ok(g)) return LAPNYS_ENOTSUP;
  const bool heads = bf && gemm_heads_ok(g);
  const char* cb = (const char*)ctx;
  const void* q = cb + L.c_q;
  const void* k = tied ? q : (const void*)(cb + L.c_k);
  const void* v = cb + L.c_v;
  const void* ot = cb + L.c_ot;
  char* wb = (char*)ws;
  float* s32 = (float*)(wb + L.b_s32);
  void* dO = wb + L.b_do;
  void* dq = wb + L.b_dq;
  void* dk = tied ? nullptr : (void*)(wb + L.b_dk);
  void* dv = wb + L.b_dv;
  void* dqkv = wb + L.b_dqkv;
  float* part = (float*)(wb + L.b_part);
  float* gpart = (float*)(wb + L.b_gpart);
  const void* dys[1] = {dy};
  const void* xs[1] = {x};

  // output projection: dO = dY W_o^T (to heads), dW_o = concat(O)^T dY, db_o = 1^T dY
  if (heads) {
    void* dst[3] = {dO, nullptr, nullptr};
    CKB(run_gemm_rows("block_gemm_do", g, GOP_ROWS_K, dys, C, GOP_W_K, w_o, HD, GEP_HEADS, dst,
                      nullptr, stream));
    const void* os[1] = {ot};
    CKB(run_gemm_wgrad("block_gemm_dwo", g, GOP_HEADS_MN, os, HD, GOP_TOK_MN, dys, C, gpart, dw_o,
                       db_o, stream));
  } else if (bf) {
    void* dst[3] = {s32, nullptr, nullptr};
    CKB(run_gemm_rows("block_gemm_do", g, GOP_ROWS_K, dys, C, GOP_W_K, w_o, HD, GEP_F32, dst,
                      nullptr, stream));
    CKB(DT_CALL(dtype, split_heads_t, s32, nullptr, dO, nullptr, nullptr, B, N, H, d, 1, stream));
    const void* os[1] = {ot};
    CKB(run_gemm_wgrad("block_gemm_dwo", g, GOP_TOK_MN, os, HD, GOP_TOK_MN, dys, C, gpart, dw_o,
                       db_o, stream));
  } else {
    CKB(gemm_f32(false, true, rows, HD, C, dy, C, w_o, C, s32, HD, stream));
    CKB(DT_CALL(dtype, split_heads_t, s32, nullptr, dO, nullptr, nullptr, B, N, H, d, 1, stream));
    CKB(gemm_f32(true, false, HD, C, rows, ot, HD, dy, C, dw_o, C, stream));
    if (db_o != nullptr) CKB(DT_CALL(dtype, colsum_t, dy, part, db_o, rows, C, stream));
  }
  // the attention
  rc = lapnys_bwd(q, tied ? nullptr : k, v, dO, (const char*)ctx + L.c_attn, dq, dk, dv, B, H, N,
                  d, grid_h, grid_w, m, lambda, eps, iters, tied, stream, dtype, flags,
                  wb + L.b_attn, L.attn_ws);
  if (rc != LAPNYS_OK) return rc;
  // QKV projection: dqkv = [dQ | dK | dV], dW_qkv = X^T dqkv, db_qkv, dX = dqkv W_qkv^T
  void* dxs[3] = {dx, nullptr, nullptr};
  if (heads) {
    const void* gs[3] = {dq, tied ? dv : dk, dv};
    CKB(run_gemm_wgrad("block_gemm_dwqkv", g, GOP_TOK_MN, xs, C, GOP_HEADS_MN, gs, S * HD, gpart,
                       dw_qkv, db_qkv,
                       stream));
    CKB(run_gemm_rows("block_gemm_dx", g, GOP_HEADS_K, gs, S * HD, GOP_W_K, w_qkv, C, GEP_ROWS, dxs,
                      nullptr,
                      stream));
    return LAPNYS_OK;
  }
  if (bf) {
    CKB(DT_CALL(dtype, merge_heads_t, dq, tied ? dv : dk, dv, dqkv, nullptr, B, N, H, d, S,
                stream));
    const void* gs[1] = {dqkv};
    CKB(run_gemm_wgrad("block_gemm_dwqkv", g, GOP_TOK_MN, xs, C, GOP_TOK_MN, gs, S * HD, gpart,
                       dw_qkv, db_qkv,
                       stream));
    CKB(run_gemm_rows("block_gemm_dx", g, GOP_ROWS_K, gs, S * HD, GOP_W_K, w_qkv, C, GEP_ROWS, dxs,
                      nullptr,
                      stream));
    return LAPNYS_OK;
  }
  CKB(DT_CALL(dtype, merge_heads_t, dq, tied ? dv : dk, dv, dqkv,
              db_qkv != nullptr ? part : nullptr, B, N, H, d, S, stream));
  CKB(gemm_f32(true, false, C, S * HD, rows, x, C, dqkv, S * HD, dw_qkv, S * HD, stream));
  if (db_qkv != nullptr)
    CKB(DT_CALL(dtype, colsum_final_t, part, db_qkv, rows, S * HD, stream));
  CKB(gemm_f32(false, true, rows, C, S * HD, dqkv, S * HD, w_qkv, S * HD, dx, C, stream));
  return LAPNYS_OK;
}

}  // extern "C"
