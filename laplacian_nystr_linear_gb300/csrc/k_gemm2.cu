// Batched fp32 products for the Newton-Schulz iteration when m > 64, version 2.
//
//   C[b] = alpha (op(A1[b]) op(B1[b]) + op(A2[b]) op(B2[b])) + beta E[b]
//
// The second product is optional (K2 = 0).  With SYM set, C is known to be
// symmetric: only the tiles on and above the diagonal are computed and each
// off-diagonal tile is also written transposed.  The Newton-Schulz iterates
// X_t, the products A X_t and the symmetrised upstream gradients are
// polynomials in the symmetric landmark matrix A, so they commute and every
// product in the iteration X_{t+1} = 2 X_t - X_t A X_t ("SOFT" review,
// Proposed method) and in its reverse is symmetric.
//
// Tile 64 x 64 per CTA of 64 threads; each thread owns an 8 x 8 block (rows
// 4 ty + {0..3}, 32 + 4 ty + {0..3}; columns likewise with tx) so every k step
// is 4 LDS.128 for 64 FFMA.  K is staged 16 at a time, double buffered through
// registers.
#include "common.cuh"
#include "internal.h"

namespace lapnys {

namespace {
constexpr int GBK = 16;
constexpr int GT = 64;  // threads

struct G2Args {
  const float* A1; const float* B1; const float* A2; const float* B2;
  int lda1, ldb1, lda2, ldb2;
  long sA1, sB1, sA2, sB2;
  int K1, K2;
  float* C; int ldc; long sC;
  const float* E; int lde; long sE;
  float alpha, beta;
  int M, N;
};

// element (i, k) of op(A) with op = transpose when TA
template <bool TA>
__device__ __forceinline__ float opA(const float* A, int lda, int i, int k) {
  return TA ? A[(size_t)k * lda + i] : A[(size_t)i * lda + k];
}
}  // namespace

template <bool TA, bool TB, bool SYM, bool VEC>
__global__ void __launch_bounds__(GT, 6) k_gemm2(G2Args g) {
  __shared__ __align__(16) float As[2][GBK][64];
  __shared__ __align__(16) float Bs[2][GBK][64];
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  const int bz = blockIdx.z;
  int bi, bj;
  if (SYM) {
    // upper-triangle tile index -> (row tile, column tile), row <= column
    int t = blockIdx.x, r = 0, nt = (g.M + 63) / 64;
    while (t >= nt - r) {
      t -= nt - r;
      ++r;
    }
    bi = r;
    bj = r + t;
  } else {
    bi = blockIdx.y;
    bj = blockIdx.x;
  }
  const int i0 = bi * 64, j0 = bj * 64;
  const float* A1 = g.A1 + bz * g.sA1;
  const float* B1 = g.B1 + bz * g.sB1;
  const float* A2 = g.A2 ? g.A2 + bz * g.sA2 : nullptr;
  const float* B2 = g.B2 ? g.B2 + bz * g.sB2 : nullptr;
  const int K = g.K1 + g.K2;

  float acc[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int s = 0; s < 8; ++s) acc[r][s] = 0.f;

  // staging registers for one K chunk: 16 A values and 16 B values per thread
  float ra[16], rb[16];
  auto fetch = [&](int k0) {
    const bool second = k0 >= g.K1;
    const float* A = second ? A2 : A1;
    const float* B = second ? B2 : B1;
    const int lda = second ? g.lda2 : g.lda1;
    const int ldb = second ? g.ldb2 : g.ldb1;
    const int kb = second ? k0 - g.K1 : k0;
    const int Kp = second ? g.K2 : g.K1;
    if (VEC) {
      // A: TA ? row k of [k][i] : row i of [i][k];  16 values per thread as 4 float4
      if (!TA) {
        const int i = i0 + tid;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < g.M) v = *reinterpret_cast<const float4*>(A + (size_t)i * lda + kb + 4 * q);
          ra[4 * q] = v.x; ra[4 * q + 1] = v.y; ra[4 * q + 2] = v.z; ra[4 * q + 3] = v.w;
        }
      } else {
        const int k = tid >> 2, ib = i0 + (tid & 3) * 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ib + 4 * q < g.M) v = *reinterpret_cast<const float4*>(A + (size_t)(kb + k) * lda + ib + 4 * q);
          ra[4 * q] = v.x; ra[4 * q + 1] = v.y; ra[4 * q + 2] = v.z; ra[4 * q + 3] = v.w;
        }
      }
      if (TB) {
        const int j = j0 + tid;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j < g.N) v = *reinterpret_cast<const float4*>(B + (size_t)j * ldb + kb + 4 * q);
          rb[4 * q] = v.x; rb[4 * q + 1] = v.y; rb[4 * q + 2] = v.z; rb[4 * q + 3] = v.w;
        }
      } else {
        const int k = tid >> 2, jb = j0 + (tid & 3) * 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (jb + 4 * q < g.N) v = *reinterpret_cast<const float4*>(B + (size_t)(kb + k) * ldb + jb + 4 * q);
          rb[4 * q] = v.x; rb[4 * q + 1] = v.y; rb[4 * q + 2] = v.z; rb[4 * q + 3] = v.w;
        }
      }
    } else {
      // scalar: thread covers row/column tid of the tile, 16 k values
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int kk = kb + q;
        const int i = i0 + tid, j = j0 + tid;
        ra[q] = (i < g.M && kk < Kp) ? opA<TA>(A, lda, i, kk) : 0.f;
        rb[q] = (j < g.N && kk < Kp) ? (TB ? B[(size_t)j * ldb + kk] : B[(size_t)kk * ldb + j]) : 0.f;
      }
    }
  };
  auto stash = [&](int buf) {
    if (VEC && TA) {
      const int k = tid >> 2, ib = (tid & 3) * 16;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st4(&As[buf][k][ib + 4 * q], make_float4(ra[4 * q], ra[4 * q + 1], ra[4 * q + 2], ra[4 * q + 3]));
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) As[buf][q][tid] = ra[q];
    }
    if (VEC && !TB) {
      const int k = tid >> 2, jb = (tid & 3) * 16;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st4(&Bs[buf][k][jb + 4 * q], make_float4(rb[4 * q], rb[4 * q + 1], rb[4 * q + 2], rb[4 * q + 3]));
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) Bs[buf][q][tid] = rb[q];
    }
  };

  const int nchunks = (g.K1 + GBK - 1) / GBK + (g.K2 + GBK - 1) / GBK;
  const int c1 = (g.K1 + GBK - 1) / GBK;
  auto chunk_k0 = [&](int c) { return c < c1 ? c * GBK : g.K1 + (c - c1) * GBK; };
  (void)K;
  fetch(chunk_k0(0));
  stash(0);
  __syncthreads();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) fetch(chunk_k0(c + 1));
#pragma unroll
    for (int k = 0; k < GBK; ++k) {
      const float4 a0 = lds4(&As[buf][k][4 * ty]);
      const float4 a1 = lds4(&As[buf][k][32 + 4 * ty]);
      const float4 b0 = lds4(&Bs[buf][k][4 * tx]);
      const float4 b1 = lds4(&Bs[buf][k][32 + 4 * tx]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int s = 0; s < 8; ++s) acc[r][s] = fmaf(a[r], b[s], acc[r][s]);
    }
    if (c + 1 < nchunks) stash(buf ^ 1);
    __syncthreads();
  }

  float* C = g.C + bz * g.sC;
  const float* E = g.E ? g.E + bz * g.sE : nullptr;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = i0 + (r < 4 ? 4 * ty + r : 32 + 4 * ty + r - 4);
    if (i >= g.M) continue;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int j = j0 + (s < 4 ? 4 * tx + s : 32 + 4 * tx + s - 4);
      if (j >= g.N) continue;
      float v = g.alpha * acc[r][s];
      if (E) v += g.beta * E[(size_t)i * g.lde + j];
      C[(size_t)i * g.ldc + j] = v;
      if (SYM && bi != bj) C[(size_t)j * g.ldc + i] = v;
    }
  }
}

cudaError_t run_gemm2(bool ta, bool tb, bool sym, int batch, int M, int N, const float* A1, int lda1,
                      long sA1, const float* B1, int ldb1, long sB1, int K1, const float* A2,
                      int lda2, long sA2, const float* B2, int ldb2, long sB2, int K2, float* C,
                      int ldc, long sC, const float* E, int lde, long sE, float alpha, float beta,
                      cudaStream_t st) {
  G2Args g;
  g.A1 = A1; g.B1 = B1; g.A2 = A2; g.B2 = B2;
  g.lda1 = lda1; g.ldb1 = ldb1; g.lda2 = lda2; g.ldb2 = ldb2;
  g.sA1 = sA1; g.sB1 = sB1; g.sA2 = sA2; g.sB2 = sB2;
  g.K1 = K1; g.K2 = K2;
  g.C = C; g.ldc = ldc; g.sC = sC;
  g.E = beta == 0.f ? nullptr : E; g.lde = lde; g.sE = sE;
  g.alpha = alpha; g.beta = beta; g.M = M; g.N = N;
  // vector loads need 16-byte aligned rows and whole chunks in each product
  auto al = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  bool vec = (K1 % GBK == 0) && (K2 % GBK == 0) && (lda1 % 4 == 0) && (ldb1 % 4 == 0) && al(A1) &&
             al(B1) && (sA1 % 4 == 0) && (sB1 % 4 == 0);
  if (K2 > 0)
    vec = vec && (lda2 % 4 == 0) && (ldb2 % 4 == 0) && al(A2) && al(B2) && (sA2 % 4 == 0) &&
          (sB2 % 4 == 0);
  // partial tiles in the loaded dimension need whole float4 groups
  if (ta) vec = vec && (M % 4 == 0);
  if (!tb) vec = vec && (N % 4 == 0);
  const int tm = (M + 63) / 64, tn = (N + 63) / 64;
  dim3 grid = sym ? dim3(tm * (tm + 1) / 2, 1, batch) : dim3(tn, tm, batch);
#define G2(TA_, TB_, SY_, VE_)                                                       \
  if (ta == TA_ && tb == TB_ && sym == SY_ && vec == VE_)                           \
    return launch(SY_ ? "gemm_sym" : "gemm", k_gemm2<TA_, TB_, SY_, VE_>, grid, dim3(GT), 0, st, g)
  G2(false, false, false, false); G2(false, false, false, true);
  G2(false, false, true, false);  G2(false, false, true, true);
  G2(false, true, false, false);  G2(false, true, false, true);
  G2(false, true, true, false);   G2(false, true, true, true);
  G2(true, false, false, false);  G2(true, false, false, true);
  G2(true, false, true, false);   G2(true, false, true, true);
  G2(true, true, false, false);   G2(true, true, false, true);
  G2(true, true, true, false);    G2(true, true, true, true);
#undef G2
  return cudaErrorInvalidValue;
}

}  // namespace lapnys
