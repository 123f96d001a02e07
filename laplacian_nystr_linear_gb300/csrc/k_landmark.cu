// Landmark-side kernels: average-pool landmarks, the landmark matrix
// A = k(L, L) + eps I, the Newton-Schulz scale alpha, the on-chip Newton-Schulz
// solver for m <= 64, and their backward counterparts.
//
// Passages: landmarks are keys chosen by average pooling ("LaplacianFormer",
// Arabic summary 2c.1; "SOFT" review, Proposed method); the landmark matrix is
// inverted by Newton-Schulz, A_0 = alpha A, A_{k+1} = 2 A_k - A_k A A_k
// ("SOFT" review, Proposed method; "LaplacianFormer" Dutch summary,
// Methodology 2), after adding a small eps I (same passages).
#include "common.cuh"
#include "internal.h"

namespace lapnys {

// ---------------------------------------------------------------------------
// pooling: one CTA per (landmark window, slice).  Thread (part p, 4-wide feature
// chunk) sums the window's tokens p, p + P, .. (row-major order inside the
// window), so each token row is read by d / 4 consecutive threads in one
// coalesced piece; the P partial sums of a chunk are then combined in the
// order p = 0, 1, .. by one thread.  Landmark a = wi * mw + wj averages token
// rows [wi gh / mh, (wi + 1) gh / mh) and columns [wj gw / mw, (wj + 1) gw / mw)
// (floors): equal windows when the grid divides, otherwise windows of the
// floor and ceil sizes.
//
// Every sum is kept error-free as a pair s + e (each addition's rounding error,
// by TwoSum, goes into e; two pairs combine by a TwoSum of their s and the sum
// of their e), and the mean is written as hi = the fp32 value nearest to
// (s + e) / n and lo = the rest, (s + e - n hi) / n (n hi is subtracted exactly
// by an FMA).  The sign of x - l in the backward is then decided by hi where
// x != hi and by -sgn(lo) where x == hi, i.e. against the exact mean of the
// window.
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 128;
constexpr int kPoolStage = 16 * 1024;  // a window of at most this many bytes is staged first

// 4 consecutive elements from shared memory (a plain load: the read-only
// global path of ld4 does not address shared memory)
__device__ __forceinline__ float4 sm_ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 sm_ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ void two_sum_acc(float& s, float& e, float v) {
  const float t = s + v;
  const float bp = t - s;
  e += (s - (t - bp)) + (v - bp);
  s = t;
}

__device__ __forceinline__ void mean_hi_lo(float s, float e, float n, float& hi, float& lo) {
  const float sh = s + e;  // renormalise the pair (TwoSum)
  const float bp = sh - s;
  const float sl = (s - (sh - bp)) + (e - bp);
  hi = __fdiv_rn(sh, n);
  const float r = fmaf(-hi, n, sh);  // exact: the remainder of a rounded quotient
  lo = __fdiv_rn(r + sl, n);
}

template <typename T>
__global__ void __launch_bounds__(kPoolThreads) k_pool(const T* __restrict__ K,
                                                       float* __restrict__ L,
                                                       float* __restrict__ Llo,
                                                       int32_t* __restrict__ idx, int N, int d,
                                                       int gh, int gw, int mh, int mw, int m) {
  __shared__ float4 ps[kPoolThreads], pe[kPoolThreads];
  extern __shared__ float4 wsm4[];  // the window's rows (kPoolStage bytes)
  const int a = blockIdx.x, bh = blockIdx.y;
  const int wi = a / mw, wj = a - wi * mw;
  const int C4 = d / 4, P = kPoolThreads / C4;
  const int chunk = threadIdx.x % C4, part = threadIdx.x / C4;
  const int y0 = wi * gh / mh, y1 = (wi + 1) * gh / mh;
  const int x0 = wj * gw / mw, x1 = (wj + 1) * gw / mw;
  const int ww = x1 - x0, nwin = (y1 - y0) * ww;
  const T* Kb = K + (size_t)bh * N * d + chunk * 4;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f), e = s;
  // A window that fits is copied in first (every 16-byte piece of its rows in
  // flight at once), then summed from shared memory in the same order.
  const int rowb = ww * d * (int)sizeof(T);  // bytes of one window row: a multiple of 16
  const bool staged = (y1 - y0) * rowb <= kPoolStage;  // uniform over the CTA
  if (staged) {
    const int per = rowb / 16, total = (y1 - y0) * per;
    const uint8_t* src0 = reinterpret_cast<const uint8_t*>(K + ((size_t)bh * N + (size_t)y0 * gw + x0) * d);
    uint8_t* wsm = reinterpret_cast<uint8_t*>(wsm4);
    for (int id = threadIdx.x; id < total; id += kPoolThreads) {
      const int r = id / per, o = id - r * per;
      cp_async16(smem_addr(wsm + r * rowb + 16 * o), src0 + (size_t)r * gw * d * sizeof(T) + 16 * o,
                 true);
    }
    cp_commit();
    cp_wait_all();
    __syncthreads();
    if (part < P) {
      const T* wb = reinterpret_cast<const T*>(wsm4) + chunk * 4;
#pragma unroll 4
      for (int t = part; t < nwin; t += P) {
        const float4 v = sm_ld4(wb + (size_t)t * d);  // rows of ww tokens, back to back
        two_sum_acc(s.x, e.x, v.x);
        two_sum_acc(s.y, e.y, v.y);
        two_sum_acc(s.z, e.z, v.z);
        two_sum_acc(s.w, e.w, v.w);
      }
      ps[threadIdx.x] = s;
      pe[threadIdx.x] = e;
    }
  } else if (part < P) {
#pragma unroll 4
    for (int t = part; t < nwin; t += P) {
      const int y = y0 + t / ww, x = x0 + t % ww;
      const float4 v = ld4(Kb + ((size_t)y * gw + x) * d);
      two_sum_acc(s.x, e.x, v.x);
      two_sum_acc(s.y, e.y, v.y);
      two_sum_acc(s.z, e.z, v.z);
      two_sum_acc(s.w, e.w, v.w);
    }
    ps[threadIdx.x] = s;
    pe[threadIdx.x] = e;
  }
  if (idx != nullptr && bh == 0 && chunk == 0 && part < P)
    for (int t = part; t < nwin; t += P) idx[(y0 + t / ww) * gw + x0 + t % ww] = a;
  __syncthreads();
  if (part != 0) return;
  for (int q = 1; q < P; ++q) {
    const float4 s2 = ps[q * C4 + chunk], e2 = pe[q * C4 + chunk];
    two_sum_acc(s.x, e.x, s2.x); e.x += e2.x;
    two_sum_acc(s.y, e.y, s2.y); e.y += e2.y;
    two_sum_acc(s.z, e.z, s2.z); e.z += e2.z;
    two_sum_acc(s.w, e.w, s2.w); e.w += e2.w;
  }
  const float n = (float)nwin;
  float4 hi, lo;
  mean_hi_lo(s.x, e.x, n, hi.x, lo.x);
  mean_hi_lo(s.y, e.y, n, hi.y, lo.y);
  mean_hi_lo(s.z, e.z, n, hi.z, lo.z);
  mean_hi_lo(s.w, e.w, n, hi.w, lo.w);
  st4(L + ((size_t)bh * m + a) * d + chunk * 4, hi);
  if (Llo != nullptr) st4(Llo + ((size_t)bh * m + a) * d + chunk * 4, lo);
}

cudaError_t run_pool(const Prob& p, const void* k, float* L, float* Llo, int32_t* idx,
                     cudaStream_t st) {
  dim3 grid(p.m, p.BH);
  if (p.dtype == 1)
    return launch("pool", k_pool<__nv_bfloat16>, grid, dim3(kPoolThreads), kPoolStage, st,
                  (const __nv_bfloat16*)k, L, Llo, idx, p.N, p.d, p.gh, p.gw, p.mh, p.mw, p.m);
  return launch("pool", k_pool<float>, grid, dim3(kPoolThreads), kPoolStage, st, (const float*)k, L,
                Llo, idx, p.N, p.d, p.gh, p.gw, p.mh, p.mw, p.m);
}

// ---------------------------------------------------------------------------
// Shared-memory matrix products for the on-chip solver (m <= 64): row-major
// tiles of 64 x 68 floats, zero past m; op(A) is A[i][k] or, with TA, A[k][i];
// op(B) is B[k][j] or, with TB, B[j][k].
// ---------------------------------------------------------------------------
constexpr int kMS = 68;
constexpr int kNsThreads = 512;  // 16 warps

// The products run on the tensor cores (mma.sync m16n8k8, TF32) at
// fp32-level accuracy: every operand element is split x = hi + lo (hi = x
// rounded to TF32, lo = x - hi) and the product accumulated in fp32 as
// hi*hi + (hi*lo + lo*hi) (the missing lo*lo term and lo's own TF32
// truncation are O(2^-21) relative).  The three terms go to separate
// accumulators, so each k step issues six independent MMAs per warp.
//
// TF32 rounding: nearest, halfway cases away from zero (add half a TF32 ulp to
// the magnitude bits, clear the 13 low bits; a carry into the exponent is the
// correct rounding).  Finite x.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Operand planes: a 64 x 64 matrix (zero past m) kept as {hi, lo} pairs,
// P[i * kMS + k] = split of element (i, k), split once when the element is
// written rather than at every use.  With 68 pairs a row, the 64-bit loads of
// an MMA fragment (4 rows x 4 columns per half-warp, either way round) fall in
// distinct banks.
__device__ __forceinline__ float2 split_pair(float x) {
  uint32_t h, l;
  split_tf32(x, h, l);
  return make_float2(__uint_as_float(h), __uint_as_float(l));
}

// the three partial sums of one 16 x 16 block
struct Acc3 {
  float hh[2][4], hl[2][4], lh[2][4];
  __device__ void zero() {
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) hh[n][c] = hl[n][c] = lh[n][c] = 0.f;
  }
  // hi*hi + (hi*lo + lo*hi)
  __device__ void sum(float (&acc)[2][4]) const {
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[n][c] = hh[n][c] + (hl[n][c] + lh[n][c]);
  }
};

// k step k0 .. k0 + 7 of the 16 x 16 block (rows r0 .., columns c0 ..) of
// op(A) op(B).  Element c of acc[n] sits at row r0 + g + 8 (c / 2), column
// c0 + 8 n + 2 t + c % 2 (g = lane / 4, t = lane % 4).
template <bool TA, bool TB>
__device__ __forceinline__ void unit_kstep(const float2* __restrict__ A, const float2* __restrict__ B,
                                           int r0, int c0, int k0, Acc3& s) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  auto opa = [&](int i, int k) { return TA ? A[k * kMS + i] : A[i * kMS + k]; };
  auto opb = [&](int k, int j) { return TB ? B[j * kMS + k] : B[k * kMS + j]; };
  const float2 a0 = opa(r0 + g, k0 + t), a1 = opa(r0 + g + 8, k0 + t);
  const float2 a2 = opa(r0 + g, k0 + t + 4), a3 = opa(r0 + g + 8, k0 + t + 4);
  const uint32_t ah[4] = {__float_as_uint(a0.x), __float_as_uint(a1.x), __float_as_uint(a2.x),
                          __float_as_uint(a3.x)};
  const uint32_t al[4] = {__float_as_uint(a0.y), __float_as_uint(a1.y), __float_as_uint(a2.y),
                          __float_as_uint(a3.y)};
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const float2 b0 = opb(k0 + t, c0 + 8 * n + g), b1 = opb(k0 + t + 4, c0 + 8 * n + g);
    mma_tf32(s.hh[n], ah, __float_as_uint(b0.x), __float_as_uint(b1.x));
    mma_tf32(s.hl[n], ah, __float_as_uint(b0.y), __float_as_uint(b1.y));
    mma_tf32(s.lh[n], al, __float_as_uint(b0.x), __float_as_uint(b1.x));
  }
}

// one 16 x 16 block of op(A) op(B) over k < K8
template <bool TA, bool TB>
__device__ __forceinline__ void unit_mm(const float2* __restrict__ A, const float2* __restrict__ B,
                                        int r0, int c0, int K8, float (&acc)[2][4]) {
  Acc3 s;
  s.zero();
#pragma unroll
  for (int u = 0; u < 8; ++u)
    if (8 * u < K8) unit_kstep<TA, TB>(A, B, r0, c0, 8 * u, s);
  s.sum(acc);
}

// The same block from fp32 planes (64 x 68 floats, zero past m), each operand
// element split as it is loaded: the forward solver's form.  It holds 64
// registers a thread and 87 KB, so two CTAs share an SM when slices outnumber
// SMs; with pair planes the forward was no faster (the tensor pipe and the
// dependent MMA chains bound both).
template <bool TA, bool TB>
__device__ __forceinline__ void unit_mm_f(const float* __restrict__ A, const float* __restrict__ B,
                                          int r0, int c0, int K8, float (&acc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  float hh[2][4], hl[2][4], lh[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) hh[n][c] = hl[n][c] = lh[n][c] = 0.f;
  auto opa = [&](int i, int k) { return TA ? A[k * kMS + i] : A[i * kMS + k]; };
  auto opb = [&](int k, int j) { return TB ? B[j * kMS + k] : B[k * kMS + j]; };
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int k0 = 8 * u;
    if (k0 < K8) {
      uint32_t ah[4], al[4];
      split_tf32(opa(r0 + g, k0 + t), ah[0], al[0]);
      split_tf32(opa(r0 + g + 8, k0 + t), ah[1], al[1]);
      split_tf32(opa(r0 + g, k0 + t + 4), ah[2], al[2]);
      split_tf32(opa(r0 + g + 8, k0 + t + 4), ah[3], al[3]);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(opb(k0 + t, c0 + 8 * n + g), bh0, bl0);
        split_tf32(opb(k0 + t + 4, c0 + 8 * n + g), bh1, bl1);
        mma_tf32(hh[n], ah, bh0, bh1);
        mma_tf32(hl[n], ah, bl0, bl1);
        mma_tf32(lh[n], al, bh0, bh1);
      }
    }
  }
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[n][c] = hh[n][c] + (hl[n][c] + lh[n][c]);
}

// the 16 x 16 output blocks of an m x m product (R x R of them, R = ceil(m / 16))
struct UnitSet {
  int R, n, K8;
  __device__ explicit UnitSet(int m) : R((m + 15) >> 4), K8((m + 7) & ~7) { n = R * R; }
  __device__ void at(int i, int& r0, int& c0) const {
    r0 = 16 * (i / R);
    c0 = 16 * (i % R);
  }
};

// element c of acc[n] of the block at (r0, c0): its (row, column)
__device__ __forceinline__ void unit_pos(int r0, int c0, int n, int c, int& r, int& j) {
  const int lane = threadIdx.x & 31;
  r = r0 + (lane >> 2) + 8 * (c >> 1);
  j = c0 + 8 * n + 2 * (lane & 3) + (c & 1);
}

// a block's values into a pair plane (two adjacent pairs, 16 bytes, a store)
__device__ __forceinline__ void put_unit(float2* P, int r0, int c0, const float (&v)[2][4]) {
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int r, j;
      unit_pos(r0, c0, n, 2 * h, r, j);
      const float2 p0 = split_pair(v[n][2 * h]), p1 = split_pair(v[n][2 * h + 1]);
      *reinterpret_cast<float4*>(P + r * kMS + j) = make_float4(p0.x, p0.y, p1.x, p1.y);
    }
}
// a block's elements inside the m x m matrix to a row-major global matrix
__device__ __forceinline__ void store_unit(float* g, int m, int r0, int c0, const float (&v)[2][4]) {
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int r, j;
      unit_pos(r0, c0, n, c, r, j);
      if (r < m && j < m) g[r * m + j] = v[n][c];
    }
}
__device__ __forceinline__ void store_mat(float* g, const float* s, int m) {
  const int j = threadIdx.x & 63;
  if (j >= m) return;
  for (int i = threadIdx.x >> 6; i < m; i += kNsThreads / 64) g[i * m + j] = s[i * kMS + j];
}

// alpha = 1 / (|A|_1 |A|_inf) of the m x m tile in shared memory; writes the
// info record {alpha, |A|_1, |A|_inf, argmax column (int bits)} unless info_g is null.
__device__ void alpha_of_tile(const float* As, int m, float* info_g, float* alpha_s) {
  __shared__ float csum[64], rsum[64];
  if (threadIdx.x < 64) {
    float cs = 0.f, rs = 0.f;
    if (threadIdx.x < m)
      for (int i = 0; i < m; ++i) {
        cs += As[i * kMS + threadIdx.x];
        rs += As[threadIdx.x * kMS + i];
      }
    csum[threadIdx.x] = cs;
    rsum[threadIdx.x] = rs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int jc = 0, ir = 0;
    for (int i = 1; i < m; ++i) {
      if (csum[i] > csum[jc]) jc = i;
      if (rsum[i] > rsum[ir]) ir = i;
    }
    const float n1 = csum[jc], ninf = rsum[ir];
    const float al = 1.0f / (n1 * ninf);
    *alpha_s = al;
    if (info_g) {
      info_g[0] = al;
      info_g[1] = n1;
      info_g[2] = ninf;
      info_g[3] = __int_as_float(jc | (ir << 16));
    }
  }
  __syncthreads();
}


// ---------------------------------------------------------------------------
// gram + alpha + Newton-Schulz for m <= 64: one CTA per slice, everything on
// chip; each of the 16 warps takes one 16 x 16 block of each product.
// ---------------------------------------------------------------------------
template <int D, bool GAUSS>
__global__ void __launch_bounds__(kNsThreads) k_ns_small(const float* __restrict__ L, float* __restrict__ A,
                                                       float* __restrict__ alpha, float* __restrict__ X,
                                                       float* __restrict__ Y, int m, int iters, int nx,
                                                       int ny, float ns, float eps) {
  extern __shared__ float4 sm4[];
  float* Ls = reinterpret_cast<float*>(sm4);
  float* As = Ls + tile_floats(D);
  float* Xa = As + 64 * kMS;
  float* Xb = Xa + 64 * kMS;
  float* Ys = Xb + 64 * kMS;
  __shared__ float al_s;
  const int bh = blockIdx.x;
  const int ty = threadIdx.x >> 4;
  const size_t mm = (size_t)m * m;

  if (threadIdx.x < kThreads) load_tile<D>(Ls, L + (size_t)bh * m * D, 0, m);
  __syncthreads();
  if (threadIdx.x < kThreads) {  // the 16 x 16 thread grid of the distance tile
    float dist[4][4];
    dist_tile<D, GAUSS>(Ls, Ls, dist);
    const int tx = threadIdx.x & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = 4 * ty + r, j = tx + 16 * q;
        float v = 0.f;
        if (i < m && j < m) v = exp2_ftz(dist[r][q] * ns) + (i == j ? eps : 0.f);
        As[i * kMS + j] = v;
      }
  }
  __syncthreads();
  store_mat(A + bh * mm, As, m);
  alpha_of_tile(As, m, alpha + (size_t)bh * 4, &al_s);
  const float al = al_s;
  for (int e = threadIdx.x; e < 64 * 64; e += kNsThreads) {
    const int i = e >> 6, j = e & 63;
    Xa[i * kMS + j] = al * As[i * kMS + j];
  }
  __syncthreads();
  store_mat(X + (size_t)bh * nx * mm, Xa, m);
  const UnitSet us(m);
  const int warp = threadIdx.x >> 5;
  for (int t = 0; t < iters; ++t) {
    for (int i = warp; i < us.n; i += kNsThreads / 32) {  // Y_t = A X_t
      int r0, c0;
      us.at(i, r0, c0);
      float acc[2][4];
      unit_mm_f<false, false>(As, Xa, r0, c0, us.K8, acc);
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int r, j;
          unit_pos(r0, c0, n, c, r, j);
          Ys[r * kMS + j] = acc[n][c];
        }
    }
    __syncthreads();
    store_mat(Y + ((size_t)bh * ny + t % ny) * mm, Ys, m);
    for (int i = warp; i < us.n; i += kNsThreads / 32) {  // X_{t+1} = 2 X_t - X_t Y_t
      int r0, c0;
      us.at(i, r0, c0);
      float acc[2][4];
      unit_mm_f<false, false>(Xa, Ys, r0, c0, us.K8, acc);
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int r, j;
          unit_pos(r0, c0, n, c, r, j);
          Xb[r * kMS + j] = 2.f * Xa[r * kMS + j] - acc[n][c];
        }
    }
    __syncthreads();
    store_mat(X + ((size_t)bh * nx + (t + 1) % nx) * mm, Xb, m);
    float* tmp = Xa; Xa = Xb; Xb = tmp;
  }
}

cudaError_t run_ns_small(const Prob& p, const float* L, float* A, float* alpha, float* X, float* Y,
                         int nx, int ny, cudaStream_t st) {
#define NS_SMALL_CASE(DD)                                                                   \
  case DD: {                                                                                \
    const size_t smem = (size_t)(tile_floats(DD) + 4 * 64 * kMS) * sizeof(float);           \
    if (p.gauss()) {                                                                        \
      static bool once = (allow_smem(k_ns_small<DD, true>, smem), true);                    \
      (void)once;                                                                           \
      return launch("ns_small", k_ns_small<DD, true>, dim3(p.BH), dim3(kNsThreads), smem, st, \
                    L, A, alpha, X, Y, p.m, p.iters, nx, ny, p.ns, p.eps);                  \
    }                                                                                       \
    static bool once = (allow_smem(k_ns_small<DD, false>, smem), true);                     \
    (void)once;                                                                             \
    return launch("ns_small", k_ns_small<DD, false>, dim3(p.BH), dim3(kNsThreads), smem, st,  \
                  L, A, alpha, X, Y, p.m, p.iters, nx, ny, p.ns, p.eps);                    \
  }
  switch (p.d) {
    NS_SMALL_CASE(16)
    NS_SMALL_CASE(32)
    NS_SMALL_CASE(64)
    NS_SMALL_CASE(128)
  }
#undef NS_SMALL_CASE
  return cudaErrorInvalidValue;
}


// ---------------------------------------------------------------------------
// gram tiles for any m: grid (column tile, row tile, slice)
// ---------------------------------------------------------------------------
template <int D, bool GAUSS>
__global__ void __launch_bounds__(kThreads) k_gram(const float* __restrict__ L, float* __restrict__ A,
                                                   int m, float ns, float eps) {
  extern __shared__ float4 sm4[];
  float* Xs = reinterpret_cast<float*>(sm4);
  float* Ls = Xs + tile_floats(D);
  const int it = blockIdx.y, jt = blockIdx.x, bh = blockIdx.z;
  const float* Lb = L + (size_t)bh * m * D;
  load_tile<D>(Xs, Lb, it * 64, m);
  load_tile<D>(Ls, Lb, jt * 64, m);
  __syncthreads();
  float dist[4][4];
  dist_tile<D, GAUSS>(Xs, Ls, dist);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = it * 64 + 4 * ty + r, j = jt * 64 + tx + 16 * s;
      if (i < m && j < m)
        A[((size_t)bh * m + i) * m + j] = exp2_ftz(dist[r][s] * ns) + (i == j ? eps : 0.f);
    }
}

cudaError_t run_gram(const Prob& p, const float* L, float* A, cudaStream_t st) {
  dim3 grid(p.nt, p.nt, p.BH);
#define GRAM_CASE(DD)                                                                        \
  case DD: {                                                                                 \
    const size_t smem = 2 * (size_t)tile_floats(DD) * sizeof(float);                         \
    if (p.gauss()) {                                                                         \
      static bool once = (allow_smem(k_gram<DD, true>, smem), true);                         \
      (void)once;                                                                            \
      return launch("gram", k_gram<DD, true>, grid, dim3(kThreads), smem, st, L, A, p.m,     \
                    p.ns, p.eps);                                                            \
    }                                                                                        \
    static bool once = (allow_smem(k_gram<DD, false>, smem), true);                          \
    (void)once;                                                                              \
    return launch("gram", k_gram<DD, false>, grid, dim3(kThreads), smem, st, L, A, p.m, p.ns, \
                  p.eps);                                                                    \
  }
  switch (p.d) {
    GRAM_CASE(16)
    GRAM_CASE(32)
    GRAM_CASE(64)
    GRAM_CASE(128)
  }
#undef GRAM_CASE
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// alpha for any m (m <= 1024): one CTA per slice; also X_0 = alpha A
// ---------------------------------------------------------------------------
// (value, index) pairs: the larger value wins, the lower index on equal values
__device__ __forceinline__ void argmax_pair(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// column sums by a thread per column (rows in order), row sums by a warp per
// row (lanes over the row, a fixed shuffle tree), the two argmaxes by a
// parallel reduction that keeps the lowest index among equal sums
__global__ void __launch_bounds__(kThreads) k_alpha(const float* __restrict__ A, float* __restrict__ info,
                                                    float* __restrict__ X0, long x_bstride, int m) {
  __shared__ float csum[1024], rsum[1024];
  __shared__ float bv[2][kThreads / 32];
  __shared__ int bi[2][kThreads / 32];
  __shared__ float al_s;
  const int bh = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* Ab = A + (size_t)bh * m * m;
  for (int j = threadIdx.x; j < m; j += kThreads) {
    float cs = 0.f;
    for (int i = 0; i < m; ++i) cs += Ab[(size_t)i * m + j];
    csum[j] = cs;
  }
  for (int r = warp; r < m; r += kThreads / 32) {
    float rs = 0.f;
    for (int i = lane; i < m; i += 32) rs += Ab[(size_t)r * m + i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
    if (lane == 0) rsum[r] = rs;
  }
  __syncthreads();
  float cv = -1.f, rv = -1.f;  // sums of positive entries: any real sum beats -1
  int ci = 0, ri = 0;
  for (int j = threadIdx.x; j < m; j += kThreads) {
    argmax_pair(cv, ci, csum[j], j);
    argmax_pair(rv, ri, rsum[j], j);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    argmax_pair(cv, ci, __shfl_xor_sync(0xffffffffu, cv, o), __shfl_xor_sync(0xffffffffu, ci, o));
    argmax_pair(rv, ri, __shfl_xor_sync(0xffffffffu, rv, o), __shfl_xor_sync(0xffffffffu, ri, o));
  }
  if (lane == 0) {
    bv[0][warp] = cv; bi[0][warp] = ci;
    bv[1][warp] = rv; bi[1][warp] = ri;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) {
      argmax_pair(cv, ci, bv[0][w], bi[0][w]);
      argmax_pair(rv, ri, bv[1][w], bi[1][w]);
    }
    const int jc = ci, ir = ri;
    const float n1 = csum[jc], ninf = rsum[ir];
    const float al = 1.0f / (n1 * ninf);
    al_s = al;
    float* o = info + (size_t)bh * 4;
    o[0] = al;
    o[1] = n1;
    o[2] = ninf;
    o[3] = __int_as_float(jc | (ir << 16));
  }
  __syncthreads();
  const float al = al_s;
  float* Xb = X0 + (size_t)bh * x_bstride;
  for (int e = threadIdx.x; e < m * m; e += kThreads) Xb[e] = al * Ab[e];
}

cudaError_t run_alpha(const Prob& p, const float* A, float* alpha, float* X0, long x_bstride,
                      cudaStream_t st) {
  return launch("alpha", k_alpha, dim3(p.BH), dim3(kThreads), 0, st, A, alpha, X0, x_bstride, p.m);
}

// ---------------------------------------------------------------------------
// backward of A = k(L, L) + eps I:
//   dL_A[a][c] = -(1/lambda) sum_{b != a} (dA_ab + dA_ba) A_ab sgn(L_ac - L_bc)
// or, for the Gaussian kernel (dk/dx = -(2/lambda) (x - y) k),
//   dL_A[a][c] = -(2/lambda) sum_{b != a} (dA_ab + dA_ba) A_ab (L_ac - L_bc)
// (landmark values l = hi + lo: equal his compare by their lo parts)
// CTA = kGB landmarks of one slice: their weights w_ab = (dA_ab + dA_ba) A_ab
// (0 at b = a) for every b go to shared memory first (coalesced reads of rows
// and of the 16-wide column strips of dA), then thread (feature c, landmark
// group ag) walks b once, reusing each L_bc for its D / 16 landmarks.  Each
// (a, c) sums over b in ascending order.
// ---------------------------------------------------------------------------
constexpr int kGB = 16;  // landmarks per CTA

template <int D, bool GAUSS>
__global__ void __launch_bounds__(kThreads) k_gram_bwd(const float* __restrict__ L,
                                                       const float* __restrict__ Llo,
                                                       const float* __restrict__ A,
                                                       const float* __restrict__ dA,
                                                       float* __restrict__ dLA, int m,
                                                       float inv_lam) {
  constexpr int LPT = D / 16;           // landmarks per thread: kGB / (kThreads / D)
  constexpr int NG = kThreads / D;      // landmark groups
  extern __shared__ float4 sm4[];
  float* w = reinterpret_cast<float*>(sm4);  // [kGB][m]
  const int a0 = blockIdx.x * kGB, bh = blockIdx.y;
  const float* Lb = L + (size_t)bh * m * D;
  const float* Ab = A + (size_t)bh * m * m;
  const float* dAb = dA + (size_t)bh * m * m;
  for (int e = threadIdx.x; e < kGB * m; e += kThreads) {  // rows a: dA_ab
    const int i = e / m, b = e - i * m, a = a0 + i;
    w[e] = a < m ? dAb[(size_t)a * m + b] : 0.f;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kGB * m; e += kThreads) {  // columns a: + dA_ba, then * A_ab
    const int b = e / kGB, i = e - b * kGB, a = a0 + i;
    if (a < m) {
      const float v = (w[i * m + b] + dAb[(size_t)b * m + a]) * Ab[(size_t)a * m + b];
      w[i * m + b] = b == a ? 0.f : v;
    }
  }
  __syncthreads();
  const int c = threadIdx.x % D, ag = threadIdx.x / D;
  float la[LPT], acc[LPT];
#pragma unroll
  for (int k = 0; k < LPT; ++k) {
    const int a = a0 + ag + NG * k;
    la[k] = a < m ? Lb[(size_t)a * D + c] : 0.f;
    acc[k] = 0.f;
  }
#pragma unroll 4
  for (int b = 0; b < m; ++b) {
    const float lb = __ldg(Lb + (size_t)b * D + c);
#pragma unroll
    for (int k = 0; k < LPT; ++k) {
      const float wv = w[(ag + NG * k) * m + b];
      float t = la[k] - lb;
      if constexpr (GAUSS) {
        acc[k] = fmaf(2.f * t, wv, acc[k]);
      } else {
        if (t == 0.f && Llo != nullptr && a0 + ag + NG * k < m)
          t = __ldg(Llo + ((size_t)bh * m + a0 + ag + NG * k) * D + c) -
              __ldg(Llo + ((size_t)bh * m + b) * D + c);
        // sgn(t) w: w with t's sign bit folded in, 0 where t is 0
        const float sw = __int_as_float(__float_as_int(wv) ^ (__float_as_int(t) & 0x80000000));
        acc[k] += t == 0.f ? 0.f : sw;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < LPT; ++k) {
    const int a = a0 + ag + NG * k;
    if (a < m) dLA[((size_t)bh * m + a) * D + c] = -inv_lam * acc[k];
  }
}

template <int D, bool GAUSS>
static cudaError_t gram_bwd_g(const Prob& p, const float* L, const float* Llo, const float* A,
                              const float* dA, float* dLA, cudaStream_t st) {
  const size_t smem = (size_t)kGB * p.m * sizeof(float);
  static bool once = (allow_smem(k_gram_bwd<D, GAUSS>, (size_t)kGB * 1024 * sizeof(float)), true);
  (void)once;
  return launch("gram_bwd", k_gram_bwd<D, GAUSS>, dim3((p.m + kGB - 1) / kGB, p.BH),
                dim3(kThreads), smem, st, L, Llo, A, dA, dLA, p.m, p.inv_lam);
}

template <int D>
static cudaError_t gram_bwd_t(const Prob& p, const float* L, const float* Llo, const float* A,
                              const float* dA, float* dLA, cudaStream_t st) {
  return p.gauss() ? gram_bwd_g<D, true>(p, L, Llo, A, dA, dLA, st)
                   : gram_bwd_g<D, false>(p, L, Llo, A, dA, dLA, st);
}

cudaError_t run_gram_bwd(const Prob& p, const float* L, const float* Llo, const float* A,
                         const float* dA, float* dLA, cudaStream_t st) {
  switch (p.d) {
    case 16: return gram_bwd_t<16>(p, L, Llo, A, dA, dLA, st);
    case 32: return gram_bwd_t<32>(p, L, Llo, A, dA, dLA, st);
    case 64: return gram_bwd_t<64>(p, L, Llo, A, dA, dLA, st);
    default: return gram_bwd_t<128>(p, L, Llo, A, dA, dLA, st);
  }
}

// ---------------------------------------------------------------------------
// Newton-Schulz backward for m <= 64, one CTA per slice, all on chip.
// Reverse of X_{t+1} = 2 X_t - X_t A X_t with upstream G = dLoss/dX_{t+1},
// the exact adjoint of the forward's own products:
//   XG  = X_t^T G,   Tm = 2 G - G Y_t^T              (phase 1, independent)
//   dA -= XG X_t^T,  G  = Tm - A^T XG                 (phase 2, independent)
// then X_0 = alpha A contributes alpha G and, through alpha = 1/(n1 ninf),
// dalpha = <G, A> spread over the maximising column (n1) and row (ninf).
// GT holds dLoss/dX_T on entry.  Warp w owns the 16 x 16 block w of all four
// products, so its blocks of G (Tm between the phases) and dA stay in fp32
// registers; A, X_t, Y_t, G and XG sit in shared memory as pair planes.  Each
// thread loads its share of X_t (into registers) and of Y_t (by asynchronous
// copies into a staging buffer) one step ahead and splits it into the planes
// at the top of the step.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kNsThreads) k_ns_bwd_small(const float* __restrict__ A,
                                                             const float* __restrict__ info,
                                                             const float* __restrict__ X,
                                                             const float* __restrict__ Y,
                                                             const float* __restrict__ GT,
                                                             float* __restrict__ dA, int m,
                                                             int iters, int nx, int ny) {
  extern __shared__ float4 sm4[];
  float2* Ap = reinterpret_cast<float2*>(sm4);
  float2* Xp2 = Ap + 64 * kMS;      // X_t, two planes: step t - 1's is written during step t
  float2* Yp = Xp2 + 2 * 64 * kMS;  // Y_t
  float2* Gp = Yp + 64 * kMS;
  float2* XGp = Gp + 64 * kMS;
  float* Yr = reinterpret_cast<float*>(XGp + 64 * kMS);  // Y_t as copied: element e at Yr[e]
  __shared__ float red[kNsThreads];
  constexpr int kPer = 64 * 64 / kNsThreads;  // elements of a matrix per thread
  const int bh = blockIdx.x;
  const size_t mm = (size_t)m * m;
  const UnitSet us(m);
  const int warp = threadIdx.x >> 5;
  const bool owner = warp < us.n;
  int r0 = 0, c0 = 0;
  if (owner) us.at(warp, r0, c0);

  float xr[kPer];  // this thread's elements e = tid + 512 q of X_t (those of Y_t go to Yr[e])
  auto fetch = [&](int t) {
    const float* Xg = X + ((size_t)bh * nx + t % nx) * mm;
    const float* Yg = Y + ((size_t)bh * ny + t % ny) * mm;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = threadIdx.x + q * kNsThreads, i = e >> 6, j = e & 63;
      const bool ok = i < m && j < m;
      xr[q] = ok ? Xg[i * m + j] : 0.f;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(Yr + e)),
                   "l"(ok ? Yg + i * m + j : Yg), "r"(ok ? 4 : 0)
                   : "memory");
    }
    cp_commit();
  };
  if (iters > 0) fetch(iters - 1);

  const float* Ab = A + bh * mm;
  const float* Gb = GT + bh * mm;
  for (int e = threadIdx.x; e < 64 * 64; e += kNsThreads) {
    const int i = e >> 6, j = e & 63, o = i * kMS + j;
    const bool ok = i < m && j < m;
    Ap[o] = split_pair(ok ? Ab[i * m + j] : 0.f);
    Gp[o] = split_pair(ok ? Gb[i * m + j] : 0.f);
  }
  float gf[2][4], da[2][4];  // this warp's blocks of G and dA
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int r, j;
      unit_pos(r0, c0, n, c, r, j);
      gf[n][c] = (r < m && j < m) ? Gb[r * m + j] : 0.f;
      da[n][c] = 0.f;
    }
  for (int t = iters - 1; t >= 0; --t) {
    float2* Xt = Xp2 + ((iters - 1 - t) & 1) * 64 * kMS;
    cp_wait_all();  // this thread's own copies of Y_t landed
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = threadIdx.x + q * kNsThreads, o = (e >> 6) * kMS + (e & 63);
      Xt[o] = split_pair(xr[q]);
      Yp[o] = split_pair(Yr[e]);
    }
    __syncthreads();  // X_t, Y_t and G in place; step t + 1 is done with this X plane
    if (t > 0) fetch(t - 1);
    if (owner) {  // gf becomes Tm
      float xg[2][4], gy[2][4];
      unit_mm<true, false>(Xt, Gp, r0, c0, us.K8, xg);
      unit_mm<false, true>(Gp, Yp, r0, c0, us.K8, gy);
      put_unit(XGp, r0, c0, xg);
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) gf[n][c] = 2.f * gf[n][c] - gy[n][c];
    }
    __syncthreads();  // XG in place; phase 1 is done with G and Y_t
    if (owner) {
      float xgx[2][4], axg[2][4];
      unit_mm<false, true>(XGp, Xt, r0, c0, us.K8, xgx);
      unit_mm<true, false>(Ap, XGp, r0, c0, us.K8, axg);
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          da[n][c] -= xgx[n][c];
          gf[n][c] -= axg[n][c];
        }
      put_unit(Gp, r0, c0, gf);
    }
  }
  __syncthreads();  // the pair planes are free
  // X_0 = alpha A, on fp32 planes in the X planes' space
  float* Gs = reinterpret_cast<float*>(Xp2);
  float* As = Gs + 64 * kMS;
  float* dAs = As + 64 * kMS;
  if (owner)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        int r, j;
        unit_pos(r0, c0, n, c, r, j);
        Gs[r * kMS + j] = gf[n][c];
        dAs[r * kMS + j] = da[n][c];
      }
  for (int e = threadIdx.x; e < 64 * 64; e += kNsThreads) {
    const int i = e >> 6, j = e & 63;
    if (i < m && j < m) As[i * kMS + j] = Ab[i * m + j];
  }
  __syncthreads();
  const float* in = info + (size_t)bh * 4;
  const float al = in[0], n1 = in[1], ninf = in[2];
  const int code = __float_as_int(in[3]);
  const int jc = code & 0xffff, ir = code >> 16;
  float part = 0.f;
  for (int e = threadIdx.x; e < 64 * 64; e += kNsThreads) {
    const int i = e >> 6, j = e & 63;
    if (i < m && j < m) part += Gs[i * kMS + j] * As[i * kMS + j];
  }
  red[threadIdx.x] = part;
  __syncthreads();
  for (int w = kNsThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  const float dal = red[0];
  for (int e = threadIdx.x; e < 64 * 64; e += kNsThreads) {
    const int i = e >> 6, j = e & 63;
    if (i >= m || j >= m) continue;
    const int o = i * kMS + j;
    float v = dAs[o] + al * Gs[o];
    if (j == jc) v += dal * (-al / n1);
    if (i == ir) v += dal * (-al / ninf);
    dA[bh * mm + i * m + j] = v;
  }
}

cudaError_t run_ns_bwd_small(const Prob& p, const float* A, const float* alpha, const float* X,
                             const float* Y, const float* GT, float* dA, cudaStream_t st) {
  const size_t smem = 6 * 64 * kMS * sizeof(float2) + 64 * 64 * sizeof(float);
  static bool once = (allow_smem(k_ns_bwd_small, smem), true);
  (void)once;
  return launch("ns_bwd_small", k_ns_bwd_small, dim3(p.BH), dim3(kNsThreads), smem, st, A, alpha,
                X, Y, GT, dA, p.m, p.iters, p.iters + 1, p.iters);
}

// ---------------------------------------------------------------------------
// alpha part of the Newton-Schulz backward for any m: one CTA per slice.
//   dA += alpha G;  dalpha = <G, A>;  dA[:, j*] += dalpha (-alpha / n1);
//   dA[i*, :] += dalpha (-alpha / ninf)
// The slice's m^2 elements are streamed twice (the sum, then the update) by
// 1024 threads, eight independent loads in flight per thread.
// ---------------------------------------------------------------------------
constexpr int kAlphaThreads = 1024;
__global__ void __launch_bounds__(kAlphaThreads) k_alpha_bwd(const float* __restrict__ A,
                                                             const float* __restrict__ info,
                                                             const float* __restrict__ G,
                                                             float* __restrict__ dA, int m) {
  __shared__ float red[kAlphaThreads / 32];
  const int bh = blockIdx.x;
  const size_t mm = (size_t)m * m;
  const float* Ab = A + bh * mm;
  const float* Gb = G + bh * mm;
  float* dAb = dA + bh * mm;
  float part = 0.f;
#pragma unroll 8
  for (size_t e = threadIdx.x; e < mm; e += kAlphaThreads) part += __ldg(Gb + e) * __ldg(Ab + e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
  __syncthreads();
  float dal = 0.f;
  for (int w = 0; w < kAlphaThreads / 32; ++w) dal += red[w];  // fixed order: deterministic
  const float* in = info + (size_t)bh * 4;
  const float al = in[0], n1 = in[1], ninf = in[2];
  const int code = __float_as_int(in[3]);
  const int jc = code & 0xffff, ir = code >> 16;
  const float cj = dal * (-al / n1), ci = dal * (-al / ninf);
#pragma unroll 8
  for (size_t e = threadIdx.x; e < mm; e += kAlphaThreads) {
    const int i = (int)(e / m), j = (int)(e - (size_t)i * m);
    float v = dAb[e] + al * __ldg(Gb + e);
    if (j == jc) v += cj;
    if (i == ir) v += ci;
    dAb[e] = v;
  }
}

cudaError_t run_alpha_bwd(const Prob& p, const float* A, const float* alpha, const float* G,
                          float* dA, cudaStream_t st) {
  return launch("alpha_bwd", k_alpha_bwd, dim3(p.BH), dim3(kAlphaThreads), 0, st, A, alpha, G, dA,
                p.m);
}

}  // namespace lapnys
