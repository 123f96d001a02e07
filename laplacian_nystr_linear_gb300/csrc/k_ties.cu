// Tie detection for the backward sign term of Laplacian-kernel Nystrom
// attention.
//
// The kernel gradient carries sgn(x_c - l_c) per (token, landmark, feature)
// ("LaplacianFormer", Dutch summary Methodology 1: the L1 norm keeps a
// non-vanishing gradient); the backward tile kernels evaluate it as one
// saturated FMA, which reads a tie x_c == l_c as sgn = -1 instead of 0 and is
// exact otherwise, as long as every value lies in {0} u [2^-40, 2^60].  These
// kernels list, ahead of the tile kernels, the ties of every 32-token block as
// (token, feature, landmark) triples; the tile kernels take the fast path and
// then correct the listed terms, which are few (bf16 tokens meet a landmark
// value exactly a few times per block at most).  A block with an out-of-range
// value, or with more ties than a record holds, is marked for the exact path.
//
// k_tie_prep (one CTA per slice and group of 8 feature columns):
//   - flags the slice when a landmark value is out of range;
//   - marks, per feature column, the candidate values in a 2048-bit map keyed
//     by 11 bits of the value (sign, 5 low exponent bits, 5 high mantissa
//     bits).  A bf16 token can only equal a landmark value that bf16
//     represents exactly, so for bf16 tokens only those values are candidates;
//   - sorts each column's candidate values ascending with their landmark
//     indices (the others as +inf).
// k_ties (many CTAs per slice, at most 64 blocks each): streams the tokens 16
// bytes at a time; a value whose key is
// marked is looked up in the sorted column and every landmark holding it gives
// a triple.  Triples are gathered per block in shared memory and written
// sorted, so the corrections are applied in a fixed order.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace lapnys {

namespace {
constexpr int TJ = 32;                              // tokens per block
constexpr int kCols = 8;                            // feature columns per prep CTA
constexpr int kMapWords = 64;                       // 2048-bit map per column (11-bit keys)
constexpr int kMapStride = kMapWords + 1;           // shared-memory column stride: odd, so the
                                                    // columns' words fall in different banks
constexpr float kLo = 9.094947017729282e-13f;        // 2^-40
constexpr float kHi = 1.152921504606846976e18f;      // 2^60
constexpr int kMaxBlocks = 64;                       // blocks per k_ties CTA
constexpr int kCap = kTieRec - 1;                    // triples per record

__device__ __forceinline__ bool out_of_range(float v) {
  const float a = fabsf(v);
  return !(a <= kHi) || (a != 0.f && a < kLo);
}

// 11-bit key of a value's bits (sign, the exponent's low 5 bits, the top 5
// mantissa bits): equal values have equal keys, both zeros get the key of +0
// (they compare equal); a key hit is only a candidate, checked exactly
__device__ __forceinline__ uint32_t tie_key(uint32_t u) {
  u = (u << 1) == 0u ? 0u : u;
  return ((u >> 21) & 0x400u) | ((u >> 18) & 0x3ffu);
}

template <typename T>
__device__ __forceinline__ bool candidate(float l) {
  return !std::is_same<T, __nv_bfloat16>::value || (__float_as_uint(l) & 0xffffu) == 0u;
}

size_t pow2_at_least(int m) {
  size_t P = 1;
  while ((int)P < m) P <<= 1;
  return P;
}
}  // namespace

// scratch: sorted values [BH][P][D] f32, their landmark indices [BH][P][D] i32,
// map [BH][D][kMapWords] u32, bad [BH][D / kCols] i32
size_t ties_scratch_bytes(int BH, int m, int d) {
  const size_t P = pow2_at_least(m);
  return 2 * (size_t)BH * P * d * 4 + (size_t)BH * d * kMapWords * 4 +
         (size_t)BH * (d / kCols) * 4 + 256;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_tie_prep(const float* __restrict__ L,
                                                       float* __restrict__ sorted,
                                                       int* __restrict__ sidx,
                                                       uint32_t* __restrict__ map,
                                                       int* __restrict__ bad, int m, int P, int D) {
  extern __shared__ float4 sm4[];
  const int CP = P + 1;  // column stride: odd, so a row's kCols values fall in different banks
  float* a = reinterpret_cast<float*>(sm4);                        // [kCols][CP] values
  int* ix = reinterpret_cast<int*>(a + kCols * CP);                // [kCols][CP] landmark index
  uint32_t* mp = reinterpret_cast<uint32_t*>(ix + kCols * CP);     // [kCols][kMapWords]
  const int bh = blockIdx.x, cg = blockIdx.y, c0 = cg * kCols, tid = threadIdx.x;
  const float* Lb = L + (size_t)bh * m * D;
  const float inf = __int_as_float(0x7f800000);
  for (int e = tid; e < kCols * kMapWords; e += kThreads) mp[e] = 0u;
  __syncthreads();
  bool b = false;
  for (int e = tid; e < kCols * P; e += kThreads) {  // row-major: kCols consecutive values
    const int i = e / kCols, cc = e % kCols;
    float v = inf;
    if (i < m) {
      const float l = __ldg(Lb + (size_t)i * D + c0 + cc);
      b = b || out_of_range(l);
      if (candidate<T>(l)) {
        v = l;
        const uint32_t k = tie_key(__float_as_uint(l));
        atomicOr(&mp[cc * kMapWords + (k >> 5)], 1u << (k & 31));
      }
    }
    a[cc * CP + i] = v;
    ix[cc * CP + i] = i;
  }
  const int any = __syncthreads_or(b);
  if (tid == 0) bad[bh * (D / kCols) + cg] = any ? 1 : 0;
  // bitonic sort of every column by value, ascending, carrying the indices
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int e = tid; e < kCols * (P / 2); e += kThreads) {
        const int cc = e / (P / 2), t = e % (P / 2);
        const int i = 2 * t - (t & (j - 1));  // lower index of the pair
        float* col = a + cc * CP;
        int* ci = ix + cc * CP;
        const bool up = (i & k) == 0;
        const float x = col[i], y = col[i + j];
        if ((x > y) == up) {
          col[i] = y;
          col[i + j] = x;
          const int t0 = ci[i];
          ci[i] = ci[i + j];
          ci[i + j] = t0;
        }
      }
      __syncthreads();
    }
  }
  for (int e = tid; e < kCols * P; e += kThreads) {
    const int i = e / kCols, cc = e % kCols;
    sorted[((size_t)bh * P + i) * D + c0 + cc] = a[cc * CP + i];
    sidx[((size_t)bh * P + i) * D + c0 + cc] = ix[cc * CP + i];
  }
  for (int e = tid; e < kCols * kMapWords; e += kThreads)
    map[((size_t)bh * D + c0) * kMapWords + e] = mp[e];
}

// four CTAs per SM (the bitmaps take 16 KB at d = 64): the register budget
// that occupancy leaves goes to the loads in flight
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 4) k_ties(const T* __restrict__ X,
                                                   const float* __restrict__ sorted,
                                                   const int* __restrict__ sidx,
                                                   const uint32_t* __restrict__ map,
                                                   const int* __restrict__ bad,
                                                   uint32_t* __restrict__ rec, int N, int P,
                                                   int nblk, int S) {
  extern __shared__ float4 sm4[];
  uint32_t* mp = reinterpret_cast<uint32_t*>(sm4);  // [D][kMapStride]
  __shared__ unsigned oor[kMaxBlocks / 32];         // block holds an out-of-range value
  __shared__ unsigned cnt[kMaxBlocks];              // ties found per block
  __shared__ uint32_t lst[kMaxBlocks][kCap];        // the first kCap triples per block
  constexpr int V = 16 / (int)sizeof(T);  // values per 16-byte load
  constexpr int G = D / V;                // 16-byte groups per token row
  static_assert(kThreads % G == 0, "a thread's columns must stay fixed");
  const int sp = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int b0 = (int)((long long)nblk * sp / S), b1 = (int)((long long)nblk * (sp + 1) / S);
  const T* Xb = X + (size_t)bh * N * D;
  const float* Sb = sorted + (size_t)bh * P * D;
  const int* Ib = sidx + (size_t)bh * P * D;
  bool all = false;
  for (int g = 0; g < D / kCols; ++g) all = all || bad[bh * (D / kCols) + g] != 0;
  for (int e = tid; e < kMaxBlocks; e += kThreads) cnt[e] = 0u;
  if (tid < kMaxBlocks / 32) oor[tid] = 0u;
  if (!all)
    for (int e = tid; e < D * kMapWords / 4; e += kThreads) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(map + (size_t)bh * D * kMapWords) + e);
      uint32_t* o = mp + (4 * e / kMapWords) * kMapStride + (4 * e) % kMapWords;  // one column
      o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
  __syncthreads();
  if (!all) {
    const int c0 = (tid % G) * V;
    const int n_lo = b0 * TJ, n_hi = min(N, b1 * TJ);
    const int total = (n_hi - n_lo) * G;
    // one 16-byte piece (V values of token n, columns c0 ..): flag out-of-range
    // values, look each value's key up in its column's map, and search the
    // sorted column on a hit
    auto scan = [&](int e, uint4 u) {
      const int n = n_lo + e / G, k = n / TJ - b0, j = n % TJ;
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t xb[V];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (V == 8) {
          xb[2 * q] = w[q] << 16;
          xb[2 * q + 1] = w[q] & 0xffff0000u;
        } else {
          xb[q] = w[q];
        }
      }
      bool bad_x = false;
#pragma unroll
      for (int q = 0; q < V; ++q) {
        const float x = __uint_as_float(xb[q]);
        const uint32_t key = tie_key(xb[q]);
        bad_x = bad_x || out_of_range(x);
        if ((mp[(c0 + q) * kMapStride + (key >> 5)] >> (key & 31)) & 1u) {
          // lower bound of x in the column's sorted candidates, then every equal entry
          const float* col = Sb + c0 + q;
          int lo = 0;
          for (int step = P >> 1; step > 0; step >>= 1)
            if (__ldg(col + (size_t)(lo + step - 1) * D) < x) lo += step;
          for (int t = lo; t < P && __ldg(col + (size_t)t * D) == x; ++t) {
            const uint32_t a = (uint32_t)__ldg(Ib + (size_t)t * D + c0 + q);
            const unsigned slot = atomicAdd(&cnt[k], 1u);
            if (slot < (unsigned)kCap) lst[k][slot] = (uint32_t)j | (uint32_t)(c0 + q) << 5 | a << 12;
          }
        }
      }
      if (bad_x) atomicOr(&oor[k >> 5], 1u << (k & 31));
    };
    // four pieces a round per thread (the thread's columns stay c0 ..), the
    // next round's loads issued before this round is scanned
    constexpr int kIn = 4;
    auto load = [&](int e0, uint4 (&u)[kIn]) {
#pragma unroll
      for (int i = 0; i < kIn; ++i) {
        const int e = e0 + i * kThreads;
        if (e < total) {
          const int n = n_lo + e / G;
          u[i] = __ldg(reinterpret_cast<const uint4*>(Xb + (size_t)n * D + c0));
        }
      }
    };
    uint4 u[kIn], un[kIn];
    load(tid, u);
    for (int e0 = tid; e0 < total; e0 += kIn * kThreads) {
      load(e0 + kIn * kThreads, un);
#pragma unroll
      for (int i = 0; i < kIn; ++i)
        if (e0 + i * kThreads < total) scan(e0 + i * kThreads, u[i]);
#pragma unroll
      for (int i = 0; i < kIn; ++i) u[i] = un[i];
    }
  }
  __syncthreads();
  for (int b = b0 + tid; b < b1; b += kThreads) {
    const int k = b - b0;
    uint32_t* r = rec + ((size_t)bh * nblk + b) * kTieRec;
    const unsigned n = cnt[k];
    if (all || ((oor[k >> 5] >> (k & 31)) & 1u) || n > (unsigned)kCap) {
      r[0] = kTieExact;
      continue;
    }
    r[0] = n;
    // insertion sort of the block's triples: a fixed order for the corrections
    for (unsigned i = 0; i < n; ++i) {
      uint32_t best = lst[k][i];
      unsigned at = i;
      for (unsigned t = i + 1; t < n; ++t)
        if (lst[k][t] < best) { best = lst[k][t]; at = t; }
      lst[k][at] = lst[k][i];
      lst[k][i] = best;
      r[1 + i] = best;
    }
  }
}

namespace {
struct TieScratch {
  float* sorted;
  int* sidx;
  uint32_t* map;
  int* bad;
  int P;
};
TieScratch tie_scratch(const Prob& p, void* scratch) {
  TieScratch t;
  t.P = (int)pow2_at_least(p.m);
  t.sorted = reinterpret_cast<float*>(scratch);
  t.sidx = reinterpret_cast<int*>(t.sorted + (size_t)p.BH * t.P * p.d);
  t.map = reinterpret_cast<uint32_t*>(t.sidx + (size_t)p.BH * t.P * p.d);
  t.bad = reinterpret_cast<int*>(t.map + (size_t)p.BH * p.d * kMapWords);
  return t;
}

template <int D, typename T>
cudaError_t ties_t(const Prob& p, const void* x, const TieScratch& t, uint32_t* rec,
                   cudaStream_t st) {
  const size_t smem = (size_t)D * kMapStride * 4;
  static bool once = (allow_smem(k_ties<D, T>, smem), true);
  (void)once;
  const int nblk = (p.N + TJ - 1) / TJ;
  // about four waves of CTAs over the GPU, at most kMaxBlocks blocks each
  int S = (4 * 152 + p.BH - 1) / p.BH;
  if (S < (nblk + kMaxBlocks - 1) / kMaxBlocks) S = (nblk + kMaxBlocks - 1) / kMaxBlocks;
  if (S > nblk) S = nblk;
  if (S < 1) S = 1;
  return launch("ties", k_ties<D, T>, dim3(S, p.BH), dim3(kThreads), smem, st, (const T*)x,
                (const float*)t.sorted, (const int*)t.sidx, (const uint32_t*)t.map,
                (const int*)t.bad, rec, p.N, t.P, nblk, S);
}
}  // namespace

cudaError_t run_tie_prep(const Prob& p, const float* L, void* scratch, cudaStream_t st) {
  const TieScratch t = tie_scratch(p, scratch);
  const size_t smem = (size_t)kCols * (t.P + 1) * 8 + (size_t)kCols * kMapWords * 4;
  if (p.dtype == 1) {
    static bool once = (allow_smem(k_tie_prep<__nv_bfloat16>, 96 * 1024), true);
    (void)once;
    return launch("tie_prep", k_tie_prep<__nv_bfloat16>, dim3(p.BH, p.d / kCols), dim3(kThreads),
                  smem, st, L, t.sorted, t.sidx, t.map, t.bad, p.m, t.P, p.d);
  }
  static bool once = (allow_smem(k_tie_prep<float>, 96 * 1024), true);
  (void)once;
  return launch("tie_prep", k_tie_prep<float>, dim3(p.BH, p.d / kCols), dim3(kThreads), smem, st,
                L, t.sorted, t.sidx, t.map, t.bad, p.m, t.P, p.d);
}

cudaError_t run_ties(const Prob& p, const void* x, void* scratch, uint32_t* rec, cudaStream_t st) {
  const TieScratch t = tie_scratch(p, scratch);
  if (p.dtype == 1) {
    switch (p.d) {
      case 16: return ties_t<16, __nv_bfloat16>(p, x, t, rec, st);
      case 32: return ties_t<32, __nv_bfloat16>(p, x, t, rec, st);
      case 64: return ties_t<64, __nv_bfloat16>(p, x, t, rec, st);
      case 128: return ties_t<128, __nv_bfloat16>(p, x, t, rec, st);
    }
  } else {
    switch (p.d) {
      case 16: return ties_t<16, float>(p, x, t, rec, st);
      case 32: return ties_t<32, float>(p, x, t, rec, st);
      case 64: return ties_t<64, float>(p, x, t, rec, st);
      case 128: return ties_t<128, float>(p, x, t, rec, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace lapnys
