// Device helpers shared by the lapnys kernels (sm_103a).
//
// Tiles: 64 tokens x 64 landmarks per CTA step, 256 threads arranged as a
// 16 x 16 grid (ty = tid / 16, tx = tid % 16).  Row tiles of a [rows][D]
// matrix live in shared memory as float [64][D + 4]; the +4 pad keeps 16-byte
// alignment and spreads rows over the 32 banks.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace lapnys {

constexpr int kTile = 64;      // tokens per token block == landmarks per landmark tile
constexpr int kThreads = 256;  // threads per CTA for the tile kernels
constexpr int kPad = 4;        // row padding (floats) of shared-memory tiles

__host__ __device__ constexpr int row_stride(int D) { return D + kPad; }
__host__ __device__ constexpr int tile_floats(int D) { return kTile * (D + kPad); }

// ---- element loads/stores (4 consecutive elements) ------------------------
__device__ __forceinline__ float4 ld4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// 2^x for the kernel values: the PTX base-2 exponential (ex2.approx) with
// results below 2^-126 flushed to zero (a kernel value that small is taken as
// 0, an absolute difference under 1.2e-38).  Fewer instructions than exp2f,
// which also returns the subnormal results; on the hires16k inputs every kernel
// value came out bit-identical to exp2f's.
__device__ __forceinline__ float exp2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 values as three bf16 planes each, v = p0 + p1 + p2 (+ a remainder
// below 2^-24 |v|): plane p is the bf16 rounding (nearest, ties to even) of what
// the earlier planes leave, the subtractions exact.  Word w[p] packs plane p of
// v0 (low half) and v1 (high half); one packed conversion per plane.
__device__ __forceinline__ void split3_bf16x2(float v0, float v1, uint32_t (&w)[3]) {
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
    w[p] = u;
    v0 -= __uint_as_float(u << 16);
    v1 -= __uint_as_float(u & 0xffff0000u);
  }
}

// Packed pairs of fp32 values (one 64-bit register, .x in the low half) and the
// paired FMA of the sm_100-family FP32 pipe: one issue slot for two lanes'
// worth of FMAs.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// acc[s] += |x - l_s| (s = 0..3) with the differences formed in pairs
// (sub.rn.f32x2: one instruction for two, the same rounded values as two scalar
// subtractions) and the absolute values added one by one: 6 instructions for
// 4 elements instead of 8, 7 % faster in the forward passes' tile loop on a
// GB300 (57.5 against 53.4 elements per cycle per SM)
__device__ __forceinline__ void l1_row4(float (&acc)[4], float x, f32x2 la, f32x2 lb) {
  const f32x2 xx = pack2(x, x);
  const float2 da = unpack2(sub2(xx, la)), db = unpack2(sub2(xx, lb));
  acc[0] += fabsf(da.x);
  acc[1] += fabsf(da.y);
  acc[2] += fabsf(db.x);
  acc[3] += fabsf(db.y);
}
__device__ __forceinline__ float comp(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Load rows [row0, row0 + 64) of a row-major [nrows][D] matrix into a padded
// shared tile; rows at or beyond nrows are zero-filled.
template <int D, typename T>
__device__ __forceinline__ void load_tile(float* s, const T* g, int row0, int nrows) {
  constexpr int C4 = D / 4;
  for (int id = threadIdx.x; id < kTile * C4; id += kThreads) {
    const int r = id / C4, c = (id % C4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < nrows) v = ld4(g + (size_t)(row0 + r) * D + c);
    st4(s + r * row_stride(D) + c, v);
  }
}

// Load rows [row0, row0 + ROWS) of a row-major [nrows][D] matrix into a
// padded shared tile of ROWS rows (zero-filled past nrows).
template <int D, int ROWS, typename T>
__device__ __forceinline__ void load_rows(float* s, const T* g, int row0, int nrows) {
  constexpr int C4 = D / 4;
  for (int id = threadIdx.x; id < ROWS * C4; id += kThreads) {
    const int r = id / C4, c = (id % C4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < nrows) v = ld4(g + (size_t)(row0 + r) * D + c);
    st4(s + r * row_stride(D) + c, v);
  }
}

// CPT consecutive floats from shared memory (CPT = 1, 2 or a multiple of 4)
template <int CPT>
__device__ __forceinline__ void lds_cpt(const float* p, float (&v)[CPT]) {
  if constexpr (CPT % 4 == 0) {
#pragma unroll
    for (int i = 0; i < CPT; i += 4) {
      const float4 t = lds4(p + i);
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
  } else if constexpr (CPT == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  } else {
    v[0] = p[0];
  }
}

// CPT consecutive values to global memory
template <int CPT>
__device__ __forceinline__ void st_cpt(float* p, const float (&v)[CPT]) {
  if constexpr (CPT % 4 == 0) {
#pragma unroll
    for (int i = 0; i < CPT; i += 4) st4(p + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < CPT; ++i) p[i] = v[i];
  }
}
template <int CPT>
__device__ __forceinline__ void st_cpt(__nv_bfloat16* p, const float (&v)[CPT]) {
  if constexpr (CPT % 4 == 0) {
#pragma unroll
    for (int i = 0; i < CPT; i += 4) st4(p + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < CPT; ++i) p[i] = __float2bfloat16_rn(v[i]);
  }
}

// |t| (Laplacian kernel) or t^2 (Gaussian kernel) added to a distance
template <bool GAUSS>
__device__ __forceinline__ float dist_add(float acc, float t) {
  return GAUSS ? fmaf(t, t, acc) : acc + fabsf(t);
}

// four features' terms added to a distance in feature order; for the L1 norm
// the differences are formed in pairs (sub.rn.f32x2, the same rounded values)
template <bool GAUSS>
__device__ __forceinline__ void dist4_add(float& acc, float4 x, float4 l) {
  if (GAUSS) {
    acc = dist_add<true>(acc, x.x - l.x);
    acc = dist_add<true>(acc, x.y - l.y);
    acc = dist_add<true>(acc, x.z - l.z);
    acc = dist_add<true>(acc, x.w - l.w);
  } else {
    const float2 da = unpack2(sub2(pack2(x.x, x.y), pack2(l.x, l.y)));
    const float2 db = unpack2(sub2(pack2(x.z, x.w), pack2(l.z, l.w)));
    acc += fabsf(da.x);
    acc += fabsf(da.y);
    acc += fabsf(db.x);
    acc += fabsf(db.y);
  }
}

// Register-blocked distances between 4 token rows (j = 4*ty + r) and 4
// landmark rows (a = tx + 16*s) of two shared tiles:
//   dist[r][s] = sum_c |X[j][c] - L[a][c]|  (L1), or sum_c (X[j][c] - L[a][c])^2
//   (squared L2, GAUSS)   (c ascending)
template <int D, bool GAUSS = false>
__device__ __forceinline__ void dist_tile(const float* __restrict__ Xs, const float* __restrict__ Ls,
                                          float dist[4][4]) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int s = 0; s < 4; ++s) dist[r][s] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    float4 x[4], l[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] = lds4(Xs + (4 * ty + r) * row_stride(D) + c);
#pragma unroll
    for (int s = 0; s < 4; ++s) l[s] = lds4(Ls + (tx + 16 * s) * row_stride(D) + c);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        dist4_add<GAUSS>(dist[r][s], x[r], l[s]);
      }
  }
}

// ---- warp-level TF32 tensor-core product (mma.sync m16n8k8) ----------------
// Fragments (g = lane / 4, t = lane % 4):
//   A (16 x 8, row-major): a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B (8 x 8):             b0 (t, g), b1 (t + 4, g)
//   C (16 x 8):            c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1)
// x rounded to the nearest TF32 value, halfway cases away from zero: add half
// a TF32 ulp to the magnitude bits and clear the 13 low bits (a carry into the
// exponent is the correct rounding).  Two integer ops on the full-rate pipe.
// Finite x.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  return (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
}
__device__ __forceinline__ void mma_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                           const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- asynchronous copies global -> shared (cp.async, 16 bytes) ------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// four consecutive elements (group c4) of a raw row of T in shared memory,
// as fp32 (the last argument only selects the element type)
__device__ __forceinline__ float4 raw4(const uint8_t* row, int c4, const float*) {
  return *reinterpret_cast<const float4*>(row + 16 * c4);
}
__device__ __forceinline__ float4 raw4(const uint8_t* row, int c4, const __nv_bfloat16*) {
  const uint2 u = *reinterpret_cast<const uint2*>(row + 8 * c4);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// sgn(t) * g with sgn(0) = 0
__device__ __forceinline__ float sgn_times(float t, float g) {
  return t > 0.f ? g : (t < 0.f ? -g : 0.f);
}

}  // namespace lapnys
