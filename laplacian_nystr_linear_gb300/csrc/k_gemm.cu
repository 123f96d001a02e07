// Batched fp32 matrix products for the landmark-side linear algebra of
// Laplacian-kernel Nystrom attention when m > 64 (the Newton-Schulz steps
// A_{k+1} = 2 A_k - A_k A A_k of the "SOFT" review, Proposed method, their
// reverse, and the small m x m by m x d products W-hat = A^+ W).
//
// The iteration must stay in fp32 (it is run far from convergence on
// ill-conditioned landmark matrices, where rounding of the products decides
// the result), so these are FFMA kernels: 64 x 64 output tile per CTA,
// K staged through shared memory 16 at a time, 4 x 4 outputs per thread.
#include "common.cuh"
#include "internal.h"

namespace lapnys {

constexpr int kBK = 16;

// C[b] = alpha op(A[b]) op(B[b]) + beta E[b]; op(A) is M x K, op(B) is K x N.
// E may alias C (each element is read and written by the same thread).
template <bool TA, bool TB>
__global__ void __launch_bounds__(kThreads) k_bgemm(const float* __restrict__ A, int lda, long sA,
                                                    const float* __restrict__ B, int ldb, long sB,
                                                    float* C, int ldc, long sC, const float* E,
                                                    int lde, long sE, int M, int N, int K,
                                                    float alpha, float beta) {
  __shared__ __align__(16) float As[TA ? kBK * 68 : 64 * (kBK + 4)];
  __shared__ __align__(16) float Bs[TB ? 64 * (kBK + 4) : kBK * 68];
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64, bz = blockIdx.z;
  A += bz * sA;
  B += bz * sB;
  C += bz * sC;
  if (E != nullptr) E += bz * sE;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int s = 0; s < 4; ++s) acc[r][s] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kBK) {
    for (int e = threadIdx.x; e < 64 * kBK; e += kThreads) {
      if (!TA) {
        const int i = e / kBK, k = e % kBK;
        const bool ok = (i0 + i < M) && (k0 + k < K);
        As[i * (kBK + 4) + k] = ok ? A[(size_t)(i0 + i) * lda + k0 + k] : 0.f;
      } else {
        const int k = e / 64, i = e % 64;
        const bool ok = (i0 + i < M) && (k0 + k < K);
        As[k * 68 + i] = ok ? A[(size_t)(k0 + k) * lda + i0 + i] : 0.f;
      }
      if (!TB) {
        const int k = e / 64, j = e % 64;
        const bool ok = (j0 + j < N) && (k0 + k < K);
        Bs[k * 68 + j] = ok ? B[(size_t)(k0 + k) * ldb + j0 + j] : 0.f;
      } else {
        const int j = e / kBK, k = e % kBK;
        const bool ok = (j0 + j < N) && (k0 + k < K);
        Bs[j * (kBK + 4) + k] = ok ? B[(size_t)(j0 + j) * ldb + k0 + k] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; k += 4) {
      float a[4][4], b[4][4];  // a[r][kk], b[kk][s]
      if (!TA) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float4 v = lds4(As + (4 * ty + r) * (kBK + 4) + k);
          a[r][0] = v.x; a[r][1] = v.y; a[r][2] = v.z; a[r][3] = v.w;
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 v = lds4(As + (k + kk) * 68 + 4 * ty);
          a[0][kk] = v.x; a[1][kk] = v.y; a[2][kk] = v.z; a[3][kk] = v.w;
        }
      }
      if (!TB) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 v = lds4(Bs + (k + kk) * 68 + 4 * tx);
          b[kk][0] = v.x; b[kk][1] = v.y; b[kk][2] = v.z; b[kk][3] = v.w;
        }
      } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float4 v = lds4(Bs + (tx + 16 * s) * (kBK + 4) + k);
          b[0][s] = v.x; b[1][s] = v.y; b[2][s] = v.z; b[3][s] = v.w;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(a[r][kk], b[kk][s], acc[r][s]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = i0 + 4 * ty + r;
      const int j = j0 + (TB ? tx + 16 * s : 4 * tx + s);
      if (i < M && j < N) {
        float v = alpha * acc[r][s];
        if (E != nullptr) v += beta * E[(size_t)i * lde + j];
        C[(size_t)i * ldc + j] = v;
      }
    }
}

cudaError_t run_bgemm(bool ta, bool tb, int batch, int M, int N, int K, const float* A, int lda,
                      long sA, const float* B, int ldb, long sB, float* C, int ldc, long sC,
                      const float* E, int lde, long sE, float alpha, float beta, cudaStream_t st) {
  dim3 grid((N + 63) / 64, (M + 63) / 64, batch);
  if (beta == 0.f) E = nullptr;
#define BG(TA_, TB_)                                                                              \
  return launch("bgemm", k_bgemm<TA_, TB_>, grid, dim3(kThreads), 0, st, A, lda, sA, B, ldb, sB, \
                C, ldc, sC, E, lde, sE, M, N, K, alpha, beta)
  if (!ta && !tb) BG(false, false);
  if (!ta && tb) BG(false, true);
  if (ta && !tb) BG(true, false);
  BG(true, true);
#undef BG
}

}  // namespace lapnys
