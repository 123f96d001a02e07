// Backward tile kernels of Laplacian-kernel Nystrom attention, query side
// (MODE 1) and key side (MODE 2).
//
// The Laplacian kernel k(x, l) = exp(-|x - l|_1 / lambda) has the
// non-vanishing L1 gradient dk/dx_c = -(k / lambda) sgn(x_c - l_c)
// ("LaplacianFormer", Dutch summary Methodology 1; Arabic summary 2a).  With
// an upstream weight g_ja per (token, landmark) pair,
//     dX_jc  = -sum_a g_ja sgn(x_jc - l_ac)      (token side, per landmark tile)
//     dL_ac +=  sum_j g_ja sgn(x_jc - l_ac)      (landmark side, over the split)
// Writing sgn(t) = 2 [t > 0] - 1 for t != 0, the sums become
//     dX_jc  = G_j  - sum_a 2 g_ja [x_jc > l_ac],   G_j = sum_a g_ja
//     dL_ac +=        sum_j 2 g_ja [x_jc > l_ac] - G'_a,  G'_a = sum_j g_ja
// and [x > l] is one saturated FMA, sat(fma(x, 2^64, -2^64 l)), which is exactly
// 0 or 1 whenever x != l and both lie in {0} u [2^-40, 2^60] (the difference is
// then at least 2^-64).  So the sign term costs three FMA-pipe operations per
// (token, landmark, feature) instead of compare/select work on the half-rate
// ALU pipe.  Landmark values are l = hi + lo (hi the fp32 window mean, lo the
// rest of the exact mean), compared by hi; a tie x == hi reads as sgn = -1 on
// the fast path while the exact mean gives -sgn(lo): the fast path then put
// g_ja into dX_jc and -g_ja into dL_ac, and a correction moves g_ja (1 - sgn(lo))
// back for each tie the tie kernels listed for the block (k_ties.cu; a few per
// block at most).  A block with an out-of-range value or too many ties takes an
// exact path with sgn(x - hi), and -sgn(lo) where x == hi.
//
// Gaussian kernel k(x, l) = exp(-|x - l|_2^2 / lambda) (the SOFT review's
// Proposed method): dk/dx_c = -(2 k / lambda) (x_c - l_c), so with the same g
//     dX_jc  = 2 (sum_a g_ja l_ac - G_j x_jc)
//     dL_ac += 2 (sum_j g_ja x_jc - G'_a l_ac)
// two paired FMAs per (token, landmark, feature) and no ties (GAUSS = true).
//
// Work split per CTA: one 64-landmark tile and a contiguous range of 32-token
// blocks; the raw token and upstream rows of the next block are copied into
// shared memory (cp.async) while the current block computes; per block
//   phase 1  (thread = 4 tokens x 2 landmarks)  dot, g from the kernel values
//            the forward kept ([N][mp] rows, copied in with the token rows)
//   phase S  (warp = D/8 features, lane = 8 tokens x 8 landmarks) sign term,
//            both sums as paired FMAs over token pairs (fma.rn.f32x2)
//   phase C  contraction: dW-hat_a += sum_j Z_ja dO_j (query side) or
//            dV_j = sum_a C_ja dW_a (key side)
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace lapnys {

namespace {
constexpr int TJ = 32;            // tokens per block
constexpr int TA = 64;            // landmarks per tile
constexpr int AS = TA + 4;        // row stride of [*][TA] tiles
constexpr int JS = TJ + 4;        // row stride of the transposed token tile
constexpr float kBig = 18446744073709551616.0f;   // 2^64
constexpr float kInvBig = 5.42101086242752217e-20f;  // 2^-64
constexpr float kLo = 9.094947017729282e-13f;        // 2^-40
constexpr float kHi = 1.152921504606846976e18f;      // 2^60

__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ bool out_of_range(float v) {
  const float a = fabsf(v);
  return !(a <= kHi) || (a != 0.f && a < kLo);
}

__device__ __forceinline__ float ldx(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldx(const __nv_bfloat16* p) {
  return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}

// Shared-memory layout (floats).
template <int D>
struct Smem {
  static constexpr int LBt = 0;                    // [D][AS]   -scale * l, transposed
  static constexpr int Rs = LBt + D * AS;          // [TA][D+4] R rows
  static constexpr int Xt = Rs + TA * (D + 4);     // [D][JS]   tokens, transposed
  static constexpr int Us = Xt + D * JS;           // [TJ][D+4] U rows
  static constexpr int Gs = Us + TJ * (D + 4);     // 2g, landmark-major: gt(a, j)
  static constexpr int Zs = Gs + TJ * AS;          // [TJ][ZS]  Z (query side) or C (key side)
  static constexpr int dLs = Zs + TJ * (AS + 4);   // [D][TA]   landmark-side accumulator
  static constexpr int KVs = dLs + D * TA;         // [TJ][AS]  kernel values of the block
  static constexpr int Raw = KVs + TJ * AS;        // raw rows of the next block: X then U
  static constexpr int Stage = Gs;                 // dX staging [TJ][D+4] over Gs (and Zs)
  template <typename T>
  __host__ __device__ static constexpr int raw_pitch() { return D * (int)sizeof(T) + 16; }  // bytes per raw row
  template <typename T>
  __host__ __device__ static constexpr int total() { return Raw + 2 * TJ * raw_pitch<T>() / 4; }
  static_assert(TJ * (D + 4) <= 2 * TJ * AS, "staging must fit in the g and Z tiles");
  static_assert(TA * TJ <= TJ * AS, "the g tile must fit its region");
  // row stride of the Z / C tile: query side AS + 4 (its tensor-core dW-hat
  // reads columns of it), key side AS (its dV reads rows)
};

}  // namespace

// Landmark slot of landmark a (0..63) in the g and scaled-landmark tiles: 4
// floats of padding after the first 32 put the 8-landmark groups read by
// lanes ag and ag + 4 into different banks.
__device__ __forceinline__ int pa(int a) { return a + ((a >> 5) << 2); }

// Slot of g[token j][landmark a] in the landmark-major g tile: one row of 32
// tokens per landmark, rotated by 4 (a / 8 + a % 8) floats (mod 32).  The
// rotation keeps 16-byte pieces whole and spreads over all banks both the
// 16-byte loads of landmarks a, a + 8, ..., a + 56 (sign term) and the scalar
// stores of an mma accumulator fragment (landmarks a, a + 2, a + 4, a + 6 x 8
// tokens).
__device__ __forceinline__ int gt(int a, int j) {
  return a * TJ + ((j + 4 * ((a >> 3) + (a & 7))) & (TJ - 1));
}

// Sign term for the warp's feature columns [cbase, cbase + D/8): lane (jg, ag)
// holds 2g for tokens j0..j0+7 x landmarks al..al+7.  Per feature the lane's
// 8 token partials are reduce-scattered over the 8 lanes of its jg group
// (lane ag keeps token j0 + ag) and its 8 landmark partials over the 4 lanes
// of its ag group (lane jg keeps landmarks al + 2 jg, al + 2 jg + 1), by warp
// shuffles in a fixed order; the token-side result goes to Stage and the
// landmark-side sum into dLs.
template <int D, bool EXACT, bool GAUSS>
__device__ __forceinline__ void sign_cols(int cbase, int j0, int al, int jg, int ag,
                                          const f32x2 (&gp)[4][8], const float* Xt,
                                          const float* LBt, float rowg, float inv_scale,
                                          float* Stage, float* dLs, const float* llo, int nv) {
  constexpr int CW = D / 8;
  constexpr unsigned kFull = 0xffffffffu;
  const bool b2 = ag & 4, b1 = ag & 2, b0 = ag & 1;
  const bool c1 = jg & 2, c0 = jg & 1;
#pragma unroll 1
  for (int ci = 0; ci < CW; ++ci) {
    const int c = cbase + ci;
    float x[8], lb[8];
    {
      const float4 u = lds4(Xt + c * JS + j0);
      const float4 v = lds4(Xt + c * JS + j0 + 4);
      x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
      x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
    }
    {
      const float4 u = lds4(LBt + c * AS + pa(al));
      const float4 v = lds4(LBt + c * AS + pa(al) + 4);
      lb[0] = u.x; lb[1] = u.y; lb[2] = u.z; lb[3] = u.w;
      lb[4] = v.x; lb[5] = v.y; lb[6] = v.z; lb[7] = v.w;
    }
    float pq[8], pl[8];
    if constexpr (GAUSS) {
      // token pair (2 rp, 2 rp + 1): sum_t 2g l_t; landmark t: sum over the
      // lane's tokens of 2g x (even-token, odd-token halves)
      f32x2 PQ[4];
#pragma unroll
      for (int rp = 0; rp < 4; ++rp) PQ[rp] = 0ull;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const f32x2 lt = pack2(lb[t], lb[t]);
        f32x2 PL = 0ull;
#pragma unroll
        for (int rp = 0; rp < 4; ++rp) {
          PQ[rp] = fma2(gp[rp][t], lt, PQ[rp]);
          PL = fma2(gp[rp][t], pack2(x[2 * rp], x[2 * rp + 1]), PL);
        }
        const float2 v = unpack2(PL);
        pl[t] = v.x + v.y;
      }
#pragma unroll
      for (int rp = 0; rp < 4; ++rp) {
        const float2 v = unpack2(PQ[rp]);
        pq[2 * rp] = v.x;
        pq[2 * rp + 1] = v.y;
      }
    } else if (!EXACT) {
      // gp[rp][t] = (2g of tokens 2 rp, 2 rp + 1 at landmark t); the indicator
      // pair p multiplies it into the token pair's sums and into landmark t's
      // (even-token, odd-token) sums
      f32x2 PQ[4];
#pragma unroll
      for (int rp = 0; rp < 4; ++rp) PQ[rp] = 0ull;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        f32x2 PL = 0ull;
#pragma unroll
        for (int rp = 0; rp < 4; ++rp) {
          const f32x2 p = pack2(fma_sat(x[2 * rp], kBig, lb[t]), fma_sat(x[2 * rp + 1], kBig, lb[t]));
          PQ[rp] = fma2(gp[rp][t], p, PQ[rp]);
          PL = fma2(gp[rp][t], p, PL);
        }
        const float2 v = unpack2(PL);
        pl[t] = v.x + v.y;
      }
#pragma unroll
      for (int rp = 0; rp < 4; ++rp) {
        const float2 v = unpack2(PQ[rp]);
        pq[2 * rp] = v.x;
        pq[2 * rp + 1] = v.y;
      }
    } else {
      // exact sgn(x - hi), and -sgn(lo) where x == hi; hi = -lb / scale (a power
      // of two: exact)
#pragma unroll
      for (int t = 0; t < 8; ++t) pq[t] = pl[t] = 0.f;
#pragma unroll
      for (int rp = 0; rp < 4; ++rp)
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float2 g = unpack2(gp[rp][t]);
          const float d0 = x[2 * rp] + lb[t] * inv_scale, d1 = x[2 * rp + 1] + lb[t] * inv_scale;
          float v0 = sgn_times(d0, 0.5f * g.x);
          float v1 = sgn_times(d1, 0.5f * g.y);
          if ((d0 == 0.f || d1 == 0.f) && al + t < nv) {
            const float lo = __ldg(llo + (size_t)(al + t) * D + c);
            const float sl = lo > 0.f ? -1.f : (lo < 0.f ? 1.f : 0.f);
            if (d0 == 0.f) v0 = sl * 0.5f * g.x;
            if (d1 == 0.f) v1 = sl * 0.5f * g.y;
          }
          pq[2 * rp] += v0;
          pq[2 * rp + 1] += v1;
          pl[t] += v0;
          pl[t] += v1;
        }
    }
    // token side: halve the 8 partials three times across lanes ag ^ 4, ^ 2, ^ 1
    float q4[4], q2[2], qs;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = b2 ? pq[k] : pq[k + 4], keep = b2 ? pq[k + 4] : pq[k];
      q4[k] = keep + __shfl_xor_sync(kFull, send, 4);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = b1 ? q4[k] : q4[k + 2], keep = b1 ? q4[k + 2] : q4[k];
      q2[k] = keep + __shfl_xor_sync(kFull, send, 2);
    }
    {
      const float send = b0 ? q2[0] : q2[1], keep = b0 ? q2[1] : q2[0];
      qs = keep + __shfl_xor_sync(kFull, send, 1);
    }
    // landmark side: halve twice across lanes jg ^ 2, jg ^ 1 (lane bits 4, 3)
    float l4[4], l2[2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = c1 ? pl[k] : pl[k + 4], keep = c1 ? pl[k + 4] : pl[k];
      l4[k] = keep + __shfl_xor_sync(kFull, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = c0 ? l4[k] : l4[k + 2], keep = c0 ? l4[k + 2] : l4[k];
      l2[k] = keep + __shfl_xor_sync(kFull, send, 8);
    }
    // fast path: dX = G_j - sum_a 2 g [x > l];  exact path: dX = -sum_a g sgn;
    // Gaussian: dX = sum_a 2 g l - 2 G_j x
    Stage[(j0 + ag) * (D + 4) + c] =
        GAUSS ? qs - 2.f * rowg * Xt[c * JS + j0 + ag] : (EXACT ? -qs : rowg - qs);
    float2* dl = reinterpret_cast<float2*>(dLs + c * TA + al + 2 * jg);
    float2 o = *dl;
    o.x += l2[0];
    o.y += l2[1];
    *dl = o;
  }
}

template <int D, typename T, int MODE, bool NORM, bool GAUSS>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 2 : 1)  // d = 128: shared memory allows one CTA
    k_bwd_pair(const T* __restrict__ X, const T* __restrict__ U, const float* __restrict__ L,
               const float* __restrict__ Llo, const float* __restrict__ R,
               const float* __restrict__ stats,
               const float* __restrict__ mdz, float* __restrict__ tok_part,
               float* __restrict__ tok_part2, float* __restrict__ lm_part,
               float* __restrict__ lm_part2, const uint32_t* __restrict__ tie_rec,
               const float* __restrict__ KV, int N, int m, int mp, int S, int nblk, int BH,
               float inv_lam) {
  constexpr int CW = D / 8;     // features per warp in phase S
  constexpr int CPT = D / 16;   // features per thread in phase C
  constexpr bool kDWhat = (MODE == 1) && !NORM;
  // bf16 inputs: the dot (dO . W-hat or V . dW) and the key-side dV contraction
  // run on the tensor cores in TF32; dW-hat stays in fp32 (it is amplified by
  // the Newton-Schulz reverse, where TF32 rounding would cost ~5e-3 on dK)
  constexpr bool kTC = std::is_same<T, __nv_bfloat16>::value && D >= 32;
  constexpr int ZS = MODE == 1 ? AS + 4 : AS;  // row stride of the Z / C tile
  using SM = Smem<D>;
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  float* LBt = sm + SM::LBt;
  float* Rs = sm + SM::Rs;
  float* Xt = sm + SM::Xt;
  float* Us = sm + SM::Us;
  float* Gs = sm + SM::Gs;
  float* Zs = sm + SM::Zs;
  float* dLs = sm + SM::dLs;
  float* Stage = sm + SM::Stage;
  float* KVs = sm + SM::KVs;
  uint8_t* raw = reinterpret_cast<uint8_t*>(sm + SM::Raw);
  constexpr int RP = SM::template raw_pitch<T>();
  __shared__ float mu_s[TA], rs_s[TA], m0_s[TA], m1_s[TA];
  __shared__ float rowg_s[TJ], colg_s[TA];  // sums of g over the tile's landmarks / block's tokens
  __shared__ uint32_t tie_s[kTieRec];        // this block's ties in this tile (else ~0u)
  __shared__ float tieg_s[kTieRec];          // g of each tie

  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * TA;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nv = min(TA, m - a0);  // valid landmarks in this tile
  const T* Xb = X + (size_t)bh * N * D;
  const T* Ub = U + (size_t)bh * N * D;
  const float* Lb = L + ((size_t)bh * m + a0) * D;

  // ---- landmark range check, R tile, statistics ----
  bool bad_l = false;
  if (!GAUSS)
    for (int e = tid; e < nv * D; e += kThreads)
      if (out_of_range(__ldg(Lb + e))) bad_l = true;
  load_tile<D>(Rs, R + (size_t)bh * m * D, a0, m);
  if (NORM && tid < TA) {
    const int a = a0 + tid;
    const float* stb = stats + (size_t)bh * 3 * m;
    mu_s[tid] = a < m ? stb[a] : 0.f;
    rs_s[tid] = a < m ? stb[2 * m + a] : 0.f;
    m0_s[tid] = mdz[(size_t)bh * 2 * mp + a0 + tid];
    m1_s[tid] = mdz[(size_t)bh * 2 * mp + mp + a0 + tid];
  }
  for (int e = tid; e < D * TA; e += kThreads) dLs[e] = 0.f;
  if constexpr (kTC) {
    // R feeds only TF32 products here: round it once (each thread its own slots)
    __syncthreads();
    for (int e = tid; e < TA * (D + 4); e += kThreads) Rs[e] = __uint_as_float(to_tf32(Rs[e]));
  }
  // landmarks outside {0} u [2^-40, 2^60] force the exact path for the whole CTA;
  // then distances use scale 1 instead of 2^64
  const bool cta_exact = __syncthreads_or(bad_l) != 0;
  // the landmark tile: -scale l for the saturated-FMA sign term, l itself for GAUSS
  const float scale = GAUSS ? -1.f : (cta_exact ? 1.f : kBig);
  const float inv_scale = cta_exact ? 1.f : kInvBig;
  for (int e = tid; e < TA * D; e += kThreads) {
    const int c = e / TA, a = e % TA;
    LBt[c * AS + pa(a)] = a < nv ? -scale * __ldg(Lb + (size_t)a * D + c) : 0.f;
  }
  __syncthreads();

  const int b0 = (int)((long long)nblk * sp / S);
  const int b1 = (int)((long long)nblk * (sp + 1) / S);

  // raw rows of block b (X then U) into shared memory, zero past N
  auto prefetch = [&](int b) {
    if (b >= b1) return;
    const int n0 = b * TJ;
    constexpr int CH = D * (int)sizeof(T) / 16;  // 16-byte pieces per row
    for (int id = tid; id < 2 * TJ * CH; id += kThreads) {
      const int which = id / (TJ * CH), rem = id % (TJ * CH), j = rem / CH, ch = rem % CH;
      const bool ok = n0 + j < N;
      const T* src = (which ? Ub : Xb) + (size_t)(ok ? n0 + j : 0) * D;
      cp_async16(smem_addr(raw + (which * TJ + j) * RP + 16 * ch),
                 reinterpret_cast<const uint8_t*>(src) + 16 * ch, ok);
    }
    cp_commit();
  };
  // kernel values of block b (this tile's 64 landmarks), zero past N
  const float* KVb = KV + (size_t)bh * N * mp + a0;
  auto prefetch_kv = [&](int b) {
    if (b >= b1) return;
    const int n0 = b * TJ;
    for (int id = tid; id < TJ * (TA / 4); id += kThreads) {
      const int j = id / (TA / 4), ch = id % (TA / 4);
      const bool ok = n0 + j < N;
      cp_async16(smem_addr(KVs + j * AS + 4 * ch), KVb + (size_t)(ok ? n0 + j : 0) * mp + 4 * ch, ok);
    }
    cp_commit();
  };
  prefetch(b0);
  prefetch_kv(b0);

  // phase S ownership: warp -> features [warp*CW, +CW); lane (jg, ag) -> tokens
  // 8 jg .. 8 jg + 7 and landmarks 8 ag .. 8 ag + 7
  const int jg = lane >> 3, ag = lane & 7;
  float colg_acc0 = 0.f, colg_acc1 = 0.f;
  // phase C ownership (query side dW-hat): landmarks 4 (tid >> 4) + s, features (tid & 15) CPT ..
  float dw[4][CPT];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int c = 0; c < CPT; ++c) dw[s][c] = 0.f;
  // tensor-core dW-hat (bf16 inputs): warp = landmarks 16 (warp & 3) .., features
  // (warp >> 2) D/2 ..; mma C fragments per 8-feature tile
  constexpr int NT8 = D / 16;
  float dwt[NT8][4];
#pragma unroll
  for (int n = 0; n < NT8; ++n) dwt[n][0] = dwt[n][1] = dwt[n][2] = dwt[n][3] = 0.f;

  for (int b = b0; b < b1; ++b) {
    const int n0 = b * TJ;
    const uint32_t* rb = GAUSS ? nullptr : tie_rec + ((size_t)bh * nblk + b) * kTieRec;
    const uint32_t rh = GAUSS ? 0u : __ldg(rb);
    const bool exact = cta_exact || (rh & kTieExact) != 0;
    const int nties = exact ? 0 : (int)rh;
    cp_wait_all();
    __syncthreads();
    // tokens transposed (Xt[c][j]) and U rows, from the raw copies
    for (int id = tid; id < TJ * (D / 4); id += kThreads) {
      const int c4 = id / TJ, j = id % TJ;
      const float4 v = raw4(raw + j * RP, c4, Xb);
      Xt[(c4 * 4 + 0) * JS + j] = v.x;
      Xt[(c4 * 4 + 1) * JS + j] = v.y;
      Xt[(c4 * 4 + 2) * JS + j] = v.z;
      Xt[(c4 * 4 + 3) * JS + j] = v.w;
    }
    for (int id = tid; id < TJ * (D / 4); id += kThreads) {
      const int j = id / (D / 4), c4 = id % (D / 4);
      st4(Us + j * (D + 4) + 4 * c4, raw4(raw + (TJ + j) * RP, c4, Ub));
    }
    __syncthreads();
    prefetch(b + 1);

    // g and the contraction operand Z (query side) or C (key side) of one
    // (token, landmark) pair from its dot product and kernel value
    auto gz = [&](int j, int a, float dot, float kv, float& g2, float& zc) {
      const bool valid = (n0 + j < N) && (a < nv);
      float g, z;
      if (MODE == 2) {
        g = dot * kv * inv_lam;
        z = kTC ? __uint_as_float(to_tf32(kv)) : kv;  // the key side's dV reads C in TF32
      } else {
        z = NORM ? (kv - mu_s[a]) * rs_s[a] : kv;
        const float dp = NORM ? (dot - m0_s[a] - z * m1_s[a]) * rs_s[a] : dot;
        g = dp * kv * inv_lam;
      }
      g2 = valid ? 2.f * g : 0.f;
      zc = valid ? z : 0.f;
    };
    if constexpr (kTC) {
      // dot[j][a] = sum_c U[j][c] R[a][c] on the tensor cores (R is stored
      // TF32-rounded); g and Z straight from the accumulator fragments
      const int gq = lane >> 2, tg = lane & 3;
      const int jt = (warp >> 2) * 16, wa = (warp & 3) * 16;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
      for (int k0 = 0; k0 < D; k0 += 8) {
        uint32_t af[4];
        af[0] = __float_as_uint(Us[(jt + gq) * (D + 4) + k0 + tg]);
        af[1] = __float_as_uint(Us[(jt + gq + 8) * (D + 4) + k0 + tg]);
        af[2] = __float_as_uint(Us[(jt + gq) * (D + 4) + k0 + tg + 4]);
        af[3] = __float_as_uint(Us[(jt + gq + 8) * (D + 4) + k0 + tg + 4]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          uint32_t bf[2];
          bf[0] = __float_as_uint(Rs[(wa + 8 * n + gq) * (D + 4) + k0 + tg]);
          bf[1] = __float_as_uint(Rs[(wa + 8 * n + gq) * (D + 4) + k0 + tg + 4]);
          mma_16x8x8(acc[n], af, bf);
        }
      }
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int a = wa + 8 * n + 2 * tg;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int j = jt + gq + 8 * hr;
          const float2 kv2 = *reinterpret_cast<const float2*>(KVs + j * AS + a);
          float g0, g1, z0, z1;
          gz(j, a, acc[n][2 * hr], kv2.x, g0, z0);
          gz(j, a + 1, acc[n][2 * hr + 1], kv2.y, g1, z1);
          Gs[gt(a, j)] = g0;
          Gs[gt(a + 1, j)] = g1;
          *reinterpret_cast<float2*>(Zs + j * ZS + a) = make_float2(z0, z1);
        }
      }
    } else {
      // ---- phase 1: thread = tokens 4 warp .. +3, landmarks 2 lane and 2 lane + 1 ----
      const int jb = 4 * warp, la = 2 * lane;
      float kvv[4][2], dot[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float2 k2 = *reinterpret_cast<const float2*>(KVs + (jb + r) * AS + la);
        kvv[r][0] = k2.x;
        kvv[r][1] = k2.y;
        dot[r][0] = dot[r][1] = 0.f;
      }
#pragma unroll 2
      for (int c = 0; c < D; c += 4) {
        const float4 r0 = lds4(Rs + la * (D + 4) + c);
        const float4 r1 = lds4(Rs + (la + 1) * (D + 4) + c);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float4 u4 = lds4(Us + (jb + r) * (D + 4) + c);
          dot[r][0] = fmaf(u4.x, r0.x, dot[r][0]);
          dot[r][0] = fmaf(u4.y, r0.y, dot[r][0]);
          dot[r][0] = fmaf(u4.z, r0.z, dot[r][0]);
          dot[r][0] = fmaf(u4.w, r0.w, dot[r][0]);
          dot[r][1] = fmaf(u4.x, r1.x, dot[r][1]);
          dot[r][1] = fmaf(u4.y, r1.y, dot[r][1]);
          dot[r][1] = fmaf(u4.z, r1.z, dot[r][1]);
          dot[r][1] = fmaf(u4.w, r1.w, dot[r][1]);
        }
      }
      float gv[2][4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float z0, z1;
        gz(jb + r, la, dot[r][0], kvv[r][0], gv[0][r], z0);
        gz(jb + r, la + 1, dot[r][1], kvv[r][1], gv[1][r], z1);
        *reinterpret_cast<float2*>(Zs + (jb + r) * ZS + la) = make_float2(z0, z1);
      }
      st4(Gs + gt(la, jb), make_float4(gv[0][0], gv[0][1], gv[0][2], gv[0][3]));
      st4(Gs + gt(la + 1, jb), make_float4(gv[1][0], gv[1][1], gv[1][2], gv[1][3]));
    }
    __syncthreads();
    prefetch_kv(b + 1);  // this block's kernel values are read

    // ---- per-token and per-landmark sums of g (the tile holds 2g) ----
    if (tid < TJ) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int a = 0; a < TA; a += 2) {
        s0 += Gs[gt(a, tid)];
        s1 += Gs[gt(a + 1, tid)];
      }
      rowg_s[tid] = 0.5f * (s0 + s1);
    } else if (tid < TJ + TA) {
      const int a = tid - TJ;
      float sacc = 0.f;
#pragma unroll
      for (int j = 0; j < TJ; j += 4) {
        const float4 v = lds4(Gs + gt(a, j));
        sacc += (v.x + v.y) + (v.z + v.w);
      }
      colg_s[a] = 0.5f * sacc;
    }

    // ---- phase C: contractions ----
    if constexpr (kDWhat && kTC) {
      // dW-hat[a][c] += sum_j Z[j][a] U[j][c] as (Z_hi + Z_lo)^T U on the tensor
      // cores: bf16 U is exact in TF32 and the split of Z keeps fp32 accuracy
      const int gq = lane >> 2, tg = lane & 3;
      const int am = (warp & 3) * 16, cn = (warp >> 2) * (D / 2);
#pragma unroll
      for (int k0 = 0; k0 < TJ; k0 += 8) {
        const float z[4] = {Zs[(k0 + tg) * ZS + am + gq], Zs[(k0 + tg) * ZS + am + gq + 8],
                            Zs[(k0 + tg + 4) * ZS + am + gq], Zs[(k0 + tg + 4) * ZS + am + gq + 8]};
        uint32_t ah[4], alo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ah[i] = to_tf32(z[i]);
          alo[i] = to_tf32(z[i] - __uint_as_float(ah[i]));
        }
#pragma unroll
        for (int n = 0; n < NT8; ++n) {
          uint32_t bf[2];
          bf[0] = __float_as_uint(Us[(k0 + tg) * (D + 4) + cn + 8 * n + gq]);
          bf[1] = __float_as_uint(Us[(k0 + tg + 4) * (D + 4) + cn + 8 * n + gq]);
          mma_16x8x8(dwt[n], ah, bf);
          mma_16x8x8(dwt[n], alo, bf);
        }
      }
    } else if constexpr (kDWhat) {
      const int ty = tid >> 4, tx = tid & 15;
#pragma unroll 4
      for (int j = 0; j < TJ; ++j) {
        const float4 z4 = lds4(Zs + j * ZS + 4 * ty);
        float uv[CPT];
        lds_cpt<CPT>(Us + j * (D + 4) + tx * CPT, uv);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          dw[0][c] = fmaf(z4.x, uv[c], dw[0][c]);
          dw[1][c] = fmaf(z4.y, uv[c], dw[1][c]);
          dw[2][c] = fmaf(z4.z, uv[c], dw[2][c]);
          dw[3][c] = fmaf(z4.w, uv[c], dw[3][c]);
        }
      }
    }
    if constexpr (MODE == 2 && kTC) {
      // dV[j][c] = sum_a C[j][a] dW[a][c] on the tensor cores (TF32)
      constexpr int NCT2 = D / 32;
      const int gq = lane >> 2, tg = lane & 3;
      const int jt = (warp >> 2) * 16, wc = (warp & 3) * (D / 4);
      float acc[NCT2][4];
#pragma unroll
      for (int n = 0; n < NCT2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll 4
      for (int k0 = 0; k0 < TA; k0 += 8) {
        uint32_t af[4];
        af[0] = __float_as_uint(Zs[(jt + gq) * ZS + k0 + tg]);
        af[1] = __float_as_uint(Zs[(jt + gq + 8) * ZS + k0 + tg]);
        af[2] = __float_as_uint(Zs[(jt + gq) * ZS + k0 + tg + 4]);
        af[3] = __float_as_uint(Zs[(jt + gq + 8) * ZS + k0 + tg + 4]);
#pragma unroll
        for (int n = 0; n < NCT2; ++n) {
          uint32_t bf[2];
          bf[0] = __float_as_uint(Rs[(k0 + tg) * (D + 4) + wc + 8 * n + gq]);
          bf[1] = __float_as_uint(Rs[(k0 + tg + 4) * (D + 4) + wc + 8 * n + gq]);
          mma_16x8x8(acc[n], af, bf);
        }
      }
      const int j1 = n0 + jt + gq, j2 = j1 + 8;
#pragma unroll
      for (int n = 0; n < NCT2; ++n) {
        const int c = wc + 8 * n + 2 * tg;
        if (j1 < N)
          *reinterpret_cast<float2*>(tok_part2 + (((size_t)lt * BH + bh) * N + j1) * D + c) =
              make_float2(acc[n][0], acc[n][1]);
        if (j2 < N)
          *reinterpret_cast<float2*>(tok_part2 + (((size_t)lt * BH + bh) * N + j2) * D + c) =
              make_float2(acc[n][2], acc[n][3]);
      }
    }
    if constexpr (MODE == 2 && !kTC) {
      // dV_j = sum_a C_ja dW_a: thread = tokens {ty, ty + 16}, features tx CPT ..
      const int ty = tid >> 4, tx = tid & 15;
      float v0[CPT], v1[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) v0[c] = v1[c] = 0.f;
#pragma unroll 2
      for (int a = 0; a < TA; a += 4) {
        const float4 c0 = lds4(Zs + ty * ZS + a);
        const float4 c1 = lds4(Zs + (ty + 16) * ZS + a);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float rv[CPT];
          lds_cpt<CPT>(Rs + (a + q) * (D + 4) + tx * CPT, rv);
          const float ck0 = comp(c0, q), ck1 = comp(c1, q);
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            v0[c] = fmaf(ck0, rv[c], v0[c]);
            v1[c] = fmaf(ck1, rv[c], v1[c]);
          }
        }
      }
      if (n0 + ty < N)
        st_cpt<CPT>(tok_part2 + (((size_t)lt * BH + bh) * N + n0 + ty) * D + tx * CPT, v0);
      if (n0 + ty + 16 < N)
        st_cpt<CPT>(tok_part2 + (((size_t)lt * BH + bh) * N + n0 + ty + 16) * D + tx * CPT, v1);
    }

    // ---- phase S: sign term ----
    {
      const int j0 = 8 * jg, al = 8 * ag;
      f32x2 gp[4][8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const ulonglong2 u = *reinterpret_cast<const ulonglong2*>(Gs + gt(al + t, j0));
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(Gs + gt(al + t, j0 + 4));
        gp[0][t] = u.x; gp[1][t] = u.y; gp[2][t] = v.x; gp[3][t] = v.y;
      }
      if (tid < nties) {
        // the tie's correction g (1 - sgn(lo)), read before the g tile becomes
        // staging space
        const uint32_t t = __ldg(rb + 1 + tid);
        const int a = (int)(t >> 12) - a0;
        const bool mine = a >= 0 && a < nv;
        tie_s[tid] = mine ? t : ~0u;
        float corr = 0.f;
        if (mine) {
          const float lo = __ldg(Llo + ((size_t)bh * m + a0 + a) * D + ((t >> 5) & 127u));
          corr = 0.5f * Gs[gt(a, (int)(t & 31u))] * (lo > 0.f ? 0.f : (lo < 0.f ? 2.f : 1.f));
        }
        tieg_s[tid] = corr;
      }
      __syncthreads();  // g and Z tiles are free from here on (staging); sums are ready
      const float rowg = rowg_s[j0 + ag];
      if (!exact) {
        colg_acc0 += colg_s[al + 2 * jg];
        colg_acc1 += colg_s[al + 2 * jg + 1];
      }
      const float* llo = Llo + ((size_t)bh * m + a0) * D;
      if constexpr (GAUSS) {
        sign_cols<D, false, true>(warp * CW, j0, al, jg, ag, gp, Xt, LBt, rowg, inv_scale, Stage,
                                  dLs, llo, nv);
      } else {
        if (exact)
          sign_cols<D, true, false>(warp * CW, j0, al, jg, ag, gp, Xt, LBt, rowg, inv_scale, Stage,
                                    dLs, llo, nv);
        else
          sign_cols<D, false, false>(warp * CW, j0, al, jg, ag, gp, Xt, LBt, rowg, inv_scale,
                                     Stage, dLs, llo, nv);
      }
    }
    __syncthreads();
    if (nties > 0) {
      // ties: the fast path counted sgn(0) as -1; take g back from dX, give it to dL
      if (tid == 0)
        for (int i = 0; i < nties; ++i) {
          const uint32_t t = tie_s[i];
          if (t == ~0u) continue;
          const int j = (int)(t & 31u), c = (int)((t >> 5) & 127u), a = (int)(t >> 12) - a0;
          Stage[j * (D + 4) + c] -= tieg_s[i];
          dLs[c * TA + a] += tieg_s[i];
        }
      __syncthreads();
    }
    // staged token-side results -> per-tile partial rows
    for (int id = tid; id < TJ * (D / 4); id += kThreads) {
      const int j = id / (D / 4), c = (id % (D / 4)) * 4;
      if (n0 + j < N)
        st4(tok_part + (((size_t)lt * BH + bh) * N + n0 + j) * D + c, lds4(Stage + j * (D + 4) + c));
    }
  }

  // ---- landmark-side outputs: dL = accumulated sum - sum of g per landmark ----
  {
    const int al = 8 * ag + 2 * jg;
    float* o = lm_part + ((size_t)bh * S + sp) * mp * D;
#pragma unroll
    for (int ci = 0; ci < CW; ++ci) {
      const int c = warp * CW + ci;
      if (GAUSS) {
        // LBt holds l: dL = sum_j 2 g x - 2 G'_a l
        o[(size_t)(a0 + al) * D + c] = dLs[c * TA + al] - 2.f * colg_acc0 * LBt[c * AS + pa(al)];
        o[(size_t)(a0 + al + 1) * D + c] =
            dLs[c * TA + al + 1] - 2.f * colg_acc1 * LBt[c * AS + pa(al + 1)];
      } else {
        o[(size_t)(a0 + al) * D + c] = dLs[c * TA + al] - colg_acc0;
        o[(size_t)(a0 + al + 1) * D + c] = dLs[c * TA + al + 1] - colg_acc1;
      }
    }
  }
  if constexpr (kDWhat && kTC) {
    const int gq = lane >> 2, tg = lane & 3;
    const int am = (warp & 3) * 16, cn = (warp >> 2) * (D / 2);
    float* o = lm_part2 + (((size_t)bh * S + sp) * mp + a0 + am + gq) * D + cn + 2 * tg;
#pragma unroll
    for (int n = 0; n < NT8; ++n) {
      *reinterpret_cast<float2*>(o + 8 * n) = make_float2(dwt[n][0], dwt[n][1]);
      *reinterpret_cast<float2*>(o + (size_t)8 * D + 8 * n) = make_float2(dwt[n][2], dwt[n][3]);
    }
  } else if constexpr (kDWhat) {
    const int ty = tid >> 4, tx = tid & 15;
    float* o = lm_part2 + (((size_t)bh * S + sp) * mp + a0 + 4 * ty) * D + tx * CPT;
#pragma unroll
    for (int s = 0; s < 4; ++s) st_cpt<CPT>(o + (size_t)s * D, dw[s]);
  }
}

template <int D, typename T, int MODE, bool NORM, bool GAUSS>
static cudaError_t bwd_pair_t2(const Prob& p, const BwdArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)Smem<D>::template total<T>() * sizeof(float);
  static bool once = (allow_smem(k_bwd_pair<D, T, MODE, NORM, GAUSS>, smem), true);
  (void)once;
  static const char* names[3] = {"", "bwd_query", "bwd_key"};
  const int nblk = (p.N + TJ - 1) / TJ;
  return launch(names[MODE], k_bwd_pair<D, T, MODE, NORM, GAUSS>, dim3(p.nt, p.Sb, p.BH), dim3(kThreads),
                smem, st, (const T*)a.X, (const T*)a.U, a.L, a.Llo, a.R, a.stats, a.mdz, a.tok_part,
                a.tok_part2, a.lm_part, a.lm_part2, a.ties, a.kv, p.N, p.m, p.mp,
                p.Sb, nblk, p.BH, p.inv_lam);
}

template <int D, typename T, bool GAUSS>
static cudaError_t bwd_pair_t3(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st) {
  if (mode == 1) {
    if (p.norm()) return bwd_pair_t2<D, T, 1, true, GAUSS>(p, a, st);
    return bwd_pair_t2<D, T, 1, false, GAUSS>(p, a, st);
  }
  return bwd_pair_t2<D, T, 2, false, GAUSS>(p, a, st);
}

template <int D, typename T>
static cudaError_t bwd_pair_t(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st) {
  return p.gauss() ? bwd_pair_t3<D, T, true>(p, mode, a, st) : bwd_pair_t3<D, T, false>(p, mode, a, st);
}

cudaError_t run_bwd_pair(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st) {
  if (p.dtype == 1) {
    switch (p.d) {
      case 16: return bwd_pair_t<16, __nv_bfloat16>(p, mode, a, st);
      case 32: return bwd_pair_t<32, __nv_bfloat16>(p, mode, a, st);
      case 64: return bwd_pair_t<64, __nv_bfloat16>(p, mode, a, st);
      case 128: return bwd_pair_t<128, __nv_bfloat16>(p, mode, a, st);
    }
  } else {
    switch (p.d) {
      case 16: return bwd_pair_t<16, float>(p, mode, a, st);
      case 32: return bwd_pair_t<32, float>(p, mode, a, st);
      case 64: return bwd_pair_t<64, float>(p, mode, a, st);
      case 128: return bwd_pair_t<128, float>(p, mode, a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace lapnys
