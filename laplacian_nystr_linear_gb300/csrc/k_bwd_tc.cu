// Backward tile kernel of Laplacian-kernel Nystrom attention for bf16 tokens
// with d = 64, query side (MODE 1) and key side (MODE 2), one CTA covering up
// to MC landmarks of a slice (all of them for m <= 256), so that each token's
// gradient is finished inside the CTA.
//
// Per (token j, landmark a) the backward needs the upstream weight
//     g_ja = dP_ja P_ja / lambda   (query side, dP from dZ = dO W-hat^T and the
//                                   feature map's reverse)
//     g_ja = dC_aj C_aj / lambda   (key side, dC = dW V^T)
// and then the kernel gradient of the Laplacian kernel k = exp(-|x - l|_1 / lambda)
// ("LaplacianFormer", Dutch summary Methodology 1; Arabic summary 2a), whose L1
// norm has the non-vanishing gradient sgn(x - l):
//     dX_jc  = -sum_a g_ja sgn(x_jc - l_ac)        (token side)
//     dL_ac +=  sum_j g_ja sgn(x_jc - l_ac)        (landmark side)
// With sgn(t) = 2 [t > 0] - 1 for t != 0:
//     dX_jc = G_j - 2 sum_a g_ja [x_jc > l_ac],   G_j = sum_a g_ja
//     dL_ac = 2 sum_j g_ja [x_jc > l_ac] - G'_a,  G'_a = sum_j g_ja
// [x > l] is one saturated FMA, sat(x 2^64 - 2^64 l) (1.0 or 0.0: exact while
// every value lies in {0} u [2^-40, 2^60], which the tie scan checks per block
// and this kernel per landmark group), and the two sums are paired FP32 FMAs
// (fma.rn.f32x2): all on the FMA pipe, with fewer instructions issued than a
// compare on the ALU pipe plus the paired FMAs (measured 7 % less time per
// launch, with identical results).  Landmark values are kept as l = hi + lo (hi the fp32 mean of the
// window, lo the rounding error of the exact mean); x != hi decides the sign
// by hi alone, and a tie x == hi (listed per 32-token block by the tie kernels)
// is corrected to sgn = -sgn(lo), so every sign matches the exact mean.  A block
// whose record overflowed, or that holds a value out of that range, takes an
// exact path with sgn(x - hi) and the same tie rule.  Gaussian kernel exp(-|x - l|_2^2 / lambda) (the SOFT review's Proposed
// method): dX_jc = 2 (sum_a g_ja l_ac - G_j x_jc), dL_ac += 2 (sum_j g_ja x_jc -
// G'_a l_ac), two paired FMAs per two elements and no signs.
//
// Contractions on the tensor cores (tcgen05.mma kind::f16, bf16 operands, f32
// accumulators in tensor memory): tokens are bf16 (exact), the fp32 factors
// are split into bf16 planes (R = hi + lo for the dot products, Z = z1 + z2 +
// z3 for dW-hat), which keeps the products at fp32-level accuracy:
//     dot_ja  = sum_c U_jc R_ac           U = dO, R = W-hat (query) or U = V, R = dW (key)
//     dW-hat += Z^T dO                    (query side without the feature map's
//                                          statistics pass)
// The key side's dV = C dW is a separate product (the kernel values C are
// stored by the forward), so this kernel writes dK, not dV.
//
// Work split: grid (token splits, landmark groups of MC, slices); a CTA of 16
// warps walks its token range in blocks of 16 tokens with a 3-stage pipeline of
// bulk copies (token rows, upstream rows, the forward's kernel values), and per
// block:
//   [g]  each thread reads 4 or 8 dot products of one landmark from tensor
//        memory and forms g (and Z, dO^T for dW-hat) into shared memory;
//   [s]  each thread (feature c = lane + 32 (warp % 2), landmarks of group
//        warp / 2) runs the sign term over the block's tokens; its landmark
//        sums stay in registers for the whole range, its token sums go to one
//        of 8 shared partial rows;
//   [r]  the 8 partials of each (token, feature) are added in a fixed order and
//        the tie corrections applied; the token gradient is written once.
// Every reduction has a fixed order, so results are bitwise reproducible.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int D = 64;
constexpr int TJ = 16;                          // tokens per block
constexpr int NTH = 512;                        // 16 warps
constexpr int FWARPS = D / 32;                  // feature halves in the sign phase
constexpr int NGR = 16 / FWARPS;                // landmark groups in the sign phase
constexpr int NST = 3;                          // load stages
constexpr uint32_t SBO = 128;                   // 8-row groups of a core-matrix operand
constexpr uint32_t LBO_R = 16 * SBO;            // K groups of a 128-row operand
constexpr uint32_t PLANE_R = (D / 8) * LBO_R;   // 128 x 64 bf16 operand: 16 KB
constexpr uint32_t LBO_U = 2 * SBO + 16;        // K groups of the 16-token operand (padded)
constexpr uint32_t TILE_U = (D / 8) * LBO_U;
constexpr uint32_t LBO_Z = 16 * SBO;            // K groups (8 tokens) of a 128-landmark operand
constexpr uint32_t PLANE_Z = (TJ / 8) * LBO_Z;
constexpr uint32_t LBO_DT = (D / 8) * SBO;      // K groups of the 64-feature operand
constexpr uint32_t TILE_DT = (TJ / 8) * LBO_DT;

template <int MC, bool DW>
struct BSmem {
  static constexpr int HF = MC > 128 ? 2 : 1;               // 128-landmark halves
  static constexpr uint32_t Rb = 0;                         // R planes: [hi, lo][HF]
  static constexpr uint32_t kXr = 0;                        // stage: token rows (bf16)
  static constexpr uint32_t kUr = TJ * D * 2;               //        upstream rows (bf16)
  static constexpr uint32_t kPr = 2 * TJ * D * 2;           //        kernel values [TJ][MC]
  static constexpr uint32_t kStage = kPr + TJ * MC * 4;
  static constexpr uint32_t St = Rb + 2 * HF * PLANE_R;
  static constexpr uint32_t Ub = St + NST * kStage;         // dot B operand (tokens x features)
  static constexpr uint32_t Gs = Ub + TILE_U;               // g [2][TJ][MC] (by block parity)
  static constexpr uint32_t Zt = Gs + 2 * TJ * MC * 4;      // Z^T planes [3][HF] (DW)
  static constexpr uint32_t Dt = Zt + (DW ? 3 * HF * PLANE_Z : 0);  // dO^T (DW)
  static constexpr uint32_t Ps = Dt + (DW ? TILE_DT : 0);   // token partials [NGR][TJ][D]
  static constexpr uint32_t total = Ps + NGR * TJ * D * 4;
};

__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

constexpr float kBig = 18446744073709551616.0f;     // 2^64
constexpr float kInvBig = 5.421010862427522e-20f;   // 2^-64
constexpr float kRangeLo = 9.094947017729282e-13f;  // 2^-40
constexpr float kRangeHi = 1.152921504606846976e18f;  // 2^60

__device__ __forceinline__ bool out_of_range(float v) {
  const float a = fabsf(v);
  return !(a <= kRangeHi) || (a != 0.f && a < kRangeLo);
}

__device__ __forceinline__ float sgnf(float v) { return v > 0.f ? 1.f : (v < 0.f ? -1.f : 0.f); }

__device__ __forceinline__ float bf16_at(const uint8_t* row, int c) {
  return __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short*>(row)[c]) << 16);
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// bounded wait for a phase of an mbarrier; on expiry the error word is set
__device__ __forceinline__ bool wait_or_flag(int* err, uint32_t bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  if (!ok) atomicOr(err, 1);
  return ok;
}
}  // namespace

struct BtcArgs {
  const __nv_bfloat16* X;   // q (query side) or k (key side)
  const __nv_bfloat16* U;   // dout (query side) or v (key side)
  const float* L;           // landmarks [BH][m][D] (fp32 means)
  const float* Llo;         // rounding error of those means [BH][m][D]
  const float* R;           // W-hat (query side) or dW (key side) [BH][m][D]
  const float* stats;       // [BH][3][m] (feature-map statistics)
  const float* mdz;         // [BH][2][mp] (column means of dZ and dZ * Z)
  const float* KV;          // P (query side) or C (key side), token-major [BH][N][mp]
  const uint32_t* ties;     // [BH][ceil(N / 32)][kTieRec]
  __nv_bfloat16* out;       // the token gradient itself when the CTA finishes it, else null
  float* tok_part;          // [NG][BH][N][D] token-side partials (when out is null)
  float* lm_part;           // [BH][S][mp][D] landmark-side partials
  float* lm_part2;          // [BH][S][mp][D] dW-hat partials (query side, no statistics pass)
  int* err;
  int N, m, mp, S, nblk, BH;
  float inv_lam;
};

template <int MODE, int MC, bool NORM, bool GAUSS>
__global__ void __launch_bounds__(NTH, 1) k_bwd_tc(BtcArgs a) {
  constexpr bool DW = (MODE == 1) && !NORM;     // dW-hat accumulated here
  constexpr int HF = MC > 128 ? 2 : 1;
  constexpr int LPT = MC / NGR;                 // landmarks per thread in the sign phase
  constexpr int TPT = 4 * HF;                   // tokens per thread in the g phase
  constexpr uint32_t DWCOL = 0, DOTCOL = DW ? HF * 64 : 0;
  constexpr uint32_t kCols = (DOTCOL + 2 * HF * TJ) <= 32 ? 32 : ((DOTCOL + 2 * HF * TJ) <= 64 ? 64
                                : ((DOTCOL + 2 * HF * TJ) <= 128 ? 128 : 256));
  using S = BSmem<MC, DW>;
  static_assert(LPT % 4 == 0, "sign phase works on groups of four landmarks");
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[NST];     // a stage's copies landed
  __shared__ __align__(8) uint64_t dotdone[2];    // dot products of a block in tensor memory
  __shared__ __align__(8) uint64_t wdone;         // dW-hat MMAs of a block done
  __shared__ uint32_t tmem_s;
  __shared__ float gsum_s[TJ];                    // G_j of the block
  __shared__ float colg_s[NTH];                   // per-thread G'_a partials (g phase)
  __shared__ float nc_s[NORM ? 4 * MC : 1];       // mu, rs, mean dZ, mean dZ Z per landmark
  __shared__ uint32_t tie_s[kTieRec];             // the block's tie record

  const int sp = blockIdx.x, gi = blockIdx.y, bh = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int abase = gi * MC;                      // first landmark of the group
  const int mg = min(MC, a.m - abase);            // landmarks of the group
  const int pw = min(MC, a.mp - abase);           // kernel-value columns copied per row
  const int nblk16 = (a.N + TJ - 1) / TJ;
  const int b0 = (int)((long long)nblk16 * sp / a.S), b1 = (int)((long long)nblk16 * (sp + 1) / a.S);
  const int nb = b1 - b0;
  const __nv_bfloat16* Xb = a.X + (size_t)bh * a.N * D;
  const __nv_bfloat16* Ubp = a.U + (size_t)bh * a.N * D;

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) tc::mbar_init(tc::smem_u32(&full[i]), 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&dotdone[i]), 1);
    tc::mbar_init(tc::smem_u32(&wdone), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- R as two bf16 planes (hi, lo) in the K-major A layout, rows past the
  // group zero ----
  {
    const float* Rg = a.R + ((size_t)bh * a.m + abase) * D;
    for (int e = tid; e < HF * 128 * (D / 8); e += NTH) {
      const int row = e / (D / 8), c8 = e % (D / 8);
      float v[8];
      if (row < mg) {
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(Rg + (size_t)row * D + 8 * c8));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(Rg + (size_t)row * D + 8 * c8 + 4));
        v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
        v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint16_t h0 = bf16_bits(v[2 * i]), h1 = bf16_bits(v[2 * i + 1]);
        const uint16_t l0 = bf16_bits(v[2 * i] - __uint_as_float((uint32_t)h0 << 16));
        const uint16_t l1 = bf16_bits(v[2 * i + 1] - __uint_as_float((uint32_t)h1 << 16));
        hw[i] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lw[i] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      const int hf = row >> 7, r = row & 127;
      const uint32_t off = c8 * LBO_R + (r >> 3) * SBO + (r & 7) * 16;
      *reinterpret_cast<uint4*>(sm + S::Rb + hf * PLANE_R + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sm + S::Rb + (HF + hf) * PLANE_R + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }

  // ---- per-thread constants ----
  // g phase: landmark ag of half hf, quarter q; tokens tok0 .. tok0 + TPT - 1
  const int q = warp & 3, wg = warp >> 2;
  const int ghf = HF == 2 ? (wg & 1) : 0;
  const int tok0 = HF == 2 ? 8 * (wg >> 1) : 4 * wg;
  const int ag = 128 * ghf + 32 * q + lane;
  const bool gact = 32 * q < MC;                  // warp-uniform: this warp has landmarks
  if (NORM) {
    for (int e = tid; e < MC; e += NTH) {
      const bool ok = e < mg;
      const float* stb = a.stats + (size_t)bh * 3 * a.m + abase;
      nc_s[e] = ok ? __ldg(stb + e) : 0.f;
      nc_s[MC + e] = ok ? __ldg(stb + 2 * a.m + e) : 0.f;
      nc_s[2 * MC + e] = ok ? __ldg(a.mdz + (size_t)bh * 2 * a.mp + abase + e) : 0.f;
      nc_s[3 * MC + e] = ok ? __ldg(a.mdz + (size_t)bh * 2 * a.mp + a.mp + abase + e) : 0.f;
    }
  }
  colg_s[tid] = 0.f;                              // G'_a over the fast-path blocks
  // sign phase: feature c, landmarks gr * LPT .. gr * LPT + LPT - 1 of the group
  const int c = 32 * (warp % FWARPS) + lane, gr = warp / FWARPS;
  // l: -2^64 hi for the saturated-FMA sign (hi itself for the Gaussian kernel,
  // or when a landmark of the group is out of range: then every block of the CTA
  // takes the exact path)
  float l[LPT];
  bool oor = false;
#pragma unroll
  for (int i = 0; i < LPT; ++i) {
    const int al = gr * LPT + i;
    l[i] = al < mg ? __ldg(a.L + ((size_t)bh * a.m + abase + al) * D + c) : 0.f;
    oor = oor || out_of_range(l[i]);
  }
  const bool cta_exact = !GAUSS && __syncthreads_or(oor);
  const float lscale = (GAUSS || cta_exact) ? 1.f : -kBig;
#pragma unroll
  for (int i = 0; i < LPT; ++i) l[i] *= lscale;
  f32x2 dl2[LPT / 2];
#pragma unroll
  for (int i = 0; i < LPT / 2; ++i) dl2[i] = 0ull;

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  // copies of block b into stage st (warp 0)
  auto issue_loads = [&](int b, int st) {
    const int n0 = b * TJ, nv = min(TJ, a.N - n0);
    uint8_t* sb = sm + S::St + st * S::kStage;
    const uint32_t bar = tc::smem_u32(&full[st]);
    if (lane == 0) tc::mbar_expect_tx(bar, (uint32_t)nv * (2 * D * 2 + (uint32_t)pw * 4));
    __syncwarp();
    if (lane == 0) tc::bulk_g2s(tc::smem_u32(sb + S::kXr), Xb + (size_t)n0 * D, nv * D * 2, bar);
    if (lane == 1) tc::bulk_g2s(tc::smem_u32(sb + S::kUr), Ubp + (size_t)n0 * D, nv * D * 2, bar);
    if (lane < nv)
      tc::bulk_g2s(tc::smem_u32(sb + S::kPr + lane * MC * 4),
                   a.KV + ((size_t)bh * a.N + n0 + lane) * a.mp + abase, (uint32_t)pw * 4, bar);
  };
  // upstream rows of a stage -> the dot's B operand (token rows, zero past N)
  auto convert_u = [&](int st, int nv) {
    const uint8_t* ur = sm + S::St + st * S::kStage + S::kUr;
    if (tid < TJ * (D / 8)) {
      const int j = tid >> 3, c8 = tid & 7;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (j < nv) v = *reinterpret_cast<const uint4*>(ur + j * D * 2 + 16 * c8);
      *reinterpret_cast<uint4*>(sm + S::Ub + c8 * LBO_U + (j >> 3) * SBO + (j & 7) * 16) = v;
    }
  };
  // the dot products of one block into tensor-memory stage ds (thread 0)
  auto issue_dot = [&](int ds) {
    const uint32_t id = tc::idesc_bf16(128, TJ);
    const uint32_t ub = tc::smem_u32(sm + S::Ub);
#pragma unroll
    for (int hf = 0; hf < HF; ++hf)
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          tc::mma_bf16(tmem + DOTCOL + (uint32_t)((ds * HF + hf) * TJ),
                       tc::desc(tc::smem_u32(sm + S::Rb + (p * HF + hf) * PLANE_R) + k16 * 2 * LBO_R,
                                LBO_R, SBO),
                       tc::desc(ub + k16 * 2 * LBO_U, LBO_U, SBO), id, (p > 0 || k16 > 0) ? 1u : 0u);
    tc::commit(tc::smem_u32(&dotdone[ds]));
  };

  // An expired wait (bad) stops the CTA at its next barrier, taken by all
  // threads alike (__syncthreads_or); the copies and MMAs in flight are then
  // waited for (bounded) before the tensor memory is freed.
  bool bad = false, abort = false;
  int ndot = 0, nw = 0;  // dot-product and dW-hat commits issued so far (the same in every thread)
  if (nb > 0) {
    if (warp == 0) {
      issue_loads(b0, 0);
      if (nb > 1) issue_loads(b0 + 1, 1);
    }
    bad |= !wait_or_flag(a.err, tc::smem_u32(&full[0]), 0u);
    convert_u(0, min(TJ, a.N - b0 * TJ));
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(bad)) {
      abort = true;
    } else {
      ndot = 1;
      if (tid == 0) {
        tc::fence_after();
        issue_dot(0);
      }
    }
  }

  // tie record of the 32-token block that block b is half of: its header (all
  // threads) and its tie words (thread k holds word k), loaded one block ahead so
  // that the load's latency hides behind a block's work
  auto rec_of = [&](int b) { return a.ties + ((size_t)bh * a.nblk + (b >> 1)) * kTieRec; };
  uint32_t rh_n = 0u, tw_n = 0u;
  if (!GAUSS && nb > 0) {
    rh_n = __ldg(rec_of(b0));
    if (tid >= 1 && tid < kTieRec) tw_n = __ldg(rec_of(b0) + tid);
  }
  int i = 0;
  for (int b = b0; b < b1 && !abort; ++b, ++i) {
    const int st = i % NST, ds = i & 1;
    const int n0 = b * TJ, nv = min(TJ, a.N - n0);
    const uint8_t* sb = sm + S::St + st * S::kStage;
    const uint32_t rh = rh_n, tw = tw_n;
    if (!GAUSS && b + 1 < b1) {
      rh_n = __ldg(rec_of(b + 1));
      if (tid >= 1 && tid < kTieRec) tw_n = __ldg(rec_of(b + 1) + tid);
    }
    const bool exact = cta_exact || (rh & kTieExact) != 0;
    const int nties = exact ? 0 : (int)rh;
    // g of this block: buffer i & 1 (the previous block's g is still read by its
    // tie corrections while this one is written)
    float* gsb = reinterpret_cast<float*>(sm + S::Gs) + (i & 1) * TJ * MC;

    // ---- [g] g (and Z, dO^T) from the dot products in tensor memory ----
    bad |= !wait_or_flag(a.err, tc::smem_u32(&dotdone[ds]), (uint32_t)(i >> 1) & 1u);
    tc::fence_after();
    if (DW && i > 0) bad |= !wait_or_flag(a.err, tc::smem_u32(&wdone), (uint32_t)(i - 1) & 1u);
    if (gact) {
      uint32_t v[TPT];
      tc::tmem_ld<TPT>(tmem + ((uint32_t)(32 * q) << 16) + DOTCOL + (uint32_t)((ds * HF + ghf) * TJ + tok0), v);
      const float* pr = reinterpret_cast<const float*>(sb + S::kPr);
      float* gs = gsb;
      float z[TPT];
      float cg = 0.f;
      const float mu = NORM ? nc_s[ag] : 0.f, rs = NORM ? nc_s[MC + ag] : 0.f;
      const float m0 = NORM ? nc_s[2 * MC + ag] : 0.f, m1 = NORM ? nc_s[3 * MC + ag] : 0.f;
#pragma unroll
      for (int t = 0; t < TPT; ++t) {
        const int j = tok0 + t;
        const bool valid = j < nv && ag < mg;
        const float kv = valid ? pr[j * MC + ag] : 0.f;
        const float dot = __uint_as_float(v[t]);
        float g, zz;
        if (MODE == 2) {
          g = dot * kv * a.inv_lam;
          zz = 0.f;
        } else {
          zz = NORM ? (kv - mu) * rs : kv;
          const float dp = NORM ? (dot - m0 - zz * m1) * rs : dot;
          g = dp * kv * a.inv_lam;
        }
        g = valid ? g : 0.f;
        z[t] = valid ? zz : 0.f;
        gs[j * MC + ag] = g;
        cg += g;
      }
      if (!exact) colg_s[tid] += cg;
      if constexpr (DW) {
        // Z^T as three bf16 planes z1 + z2 + z3 (row = landmark, k = token)
        const int r = ag & 127;
        uint32_t w[3][TPT / 2];
#pragma unroll
        for (int t = 0; t < TPT; t += 2) {
          uint32_t u[3];
          split3_bf16x2(z[t], z[t + 1], u);
#pragma unroll
          for (int p = 0; p < 3; ++p) w[p][t / 2] = u[p];
        }
        const uint32_t off = (tok0 >> 3) * LBO_Z + (r >> 3) * SBO + (r & 7) * 16 + (tok0 & 7) * 2;
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          uint8_t* dst = sm + S::Zt + (p * HF + ghf) * PLANE_Z + off;
          if constexpr (TPT == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
          else
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[p][0], w[p][1]);
        }
      }
    }
    if constexpr (DW) {
      // dO^T, the B operand of dW-hat (row = feature, k = token)
      if (tid < D * (TJ / 4)) {
        const int cc = tid & (D - 1), j4 = tid / D;
        const uint8_t* ur = sb + S::kUr;
        uint16_t h[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int j = 4 * j4 + t;
          h[t] = j < nv ? reinterpret_cast<const uint16_t*>(ur + j * D * 2)[cc] : (uint16_t)0;
        }
        *reinterpret_cast<uint2*>(sm + S::Dt + (j4 >> 1) * LBO_DT + (cc >> 3) * SBO + (cc & 7) * 16 +
                                  (j4 & 1) * 8) =
            make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
      }
    }
    // next block's upstream rows -> the dot's B operand
    if (b + 1 < b1) {
      bad |= !wait_or_flag(a.err, tc::smem_u32(&full[(i + 1) % NST]), (uint32_t)((i + 1) / NST) & 1u);
      convert_u((i + 1) % NST, min(TJ, a.N - (b + 1) * TJ));
    }
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    if (tid < kTieRec) tie_s[tid] = (tid >= 1 && tid <= nties) ? tw : 0u;
    if (b + 1 < b1) ++ndot;
    if (DW) ++nw;
    if (tid == 0) {
      tc::fence_after();
      if (b + 1 < b1) issue_dot(ds ^ 1);
      if constexpr (DW) {
        const uint32_t id = tc::idesc_bf16(128, D);
        const uint32_t dt = tc::smem_u32(sm + S::Dt);
#pragma unroll
        for (int hf = 0; hf < HF; ++hf)
#pragma unroll
          for (int p = 0; p < 3; ++p)
            tc::mma_bf16(tmem + DWCOL + (uint32_t)(hf * 64),
                         tc::desc(tc::smem_u32(sm + S::Zt + (p * HF + hf) * PLANE_Z), LBO_Z, SBO),
                         tc::desc(dt, LBO_DT, SBO), id, (i > 0 || p > 0) ? 1u : 0u);
        tc::commit(tc::smem_u32(&wdone));
      }
    }
    if (warp == 0 && b + 2 < b1) issue_loads(b + 2, (i + 2) % NST);

    // ---- [s] the sign term ----
    {
      const float* gs = gsb;
      // G_j: warp j sums the block's row j (fixed order)
      if (warp < nv) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < MC / 32; ++k) s += gs[warp * MC + lane + 32 * k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) gsum_s[warp] = s;
      }
      const uint8_t* xr = sb + S::kXr;
      float* ps = reinterpret_cast<float*>(sm + S::Ps) + gr * TJ * D + c;
      const float* gbase = gs + gr * LPT;
      if (GAUSS) {
        for (int j = 0; j < nv; ++j) {
          const float x = bf16_at(xr + j * D * 2, c);
          const f32x2 xx = pack2(x, x);
          f32x2 pa = 0ull, pb = 0ull;
#pragma unroll
          for (int i4 = 0; i4 < LPT / 4; ++i4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gbase + j * MC + 4 * i4);
            const f32x2 ga = pack2(g4.x, g4.y), gb = pack2(g4.z, g4.w);
            pa = fma2(ga, pack2(l[4 * i4], l[4 * i4 + 1]), pa);
            pb = fma2(gb, pack2(l[4 * i4 + 2], l[4 * i4 + 3]), pb);
            dl2[2 * i4] = fma2(ga, xx, dl2[2 * i4]);
            dl2[2 * i4 + 1] = fma2(gb, xx, dl2[2 * i4 + 1]);
          }
          const float2 u = unpack2(pa), w = unpack2(pb);
          ps[j * D] = (u.x + u.y) + (w.x + w.y);
        }
      } else if (!exact) {
        for (int j = 0; j < nv; ++j) {
          const float x = bf16_at(xr + j * D * 2, c);
          f32x2 pa = 0ull, pb = 0ull;
#pragma unroll
          for (int i4 = 0; i4 < LPT / 4; ++i4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gbase + j * MC + 4 * i4);
            const f32x2 ga = pack2(g4.x, g4.y), gb = pack2(g4.z, g4.w);
            const f32x2 ia = pack2(fma_sat(x, kBig, l[4 * i4]), fma_sat(x, kBig, l[4 * i4 + 1]));
            const f32x2 ib = pack2(fma_sat(x, kBig, l[4 * i4 + 2]), fma_sat(x, kBig, l[4 * i4 + 3]));
            pa = fma2(ga, ia, pa);
            pb = fma2(gb, ib, pb);
            dl2[2 * i4] = fma2(ga, ia, dl2[2 * i4]);
            dl2[2 * i4 + 1] = fma2(gb, ib, dl2[2 * i4 + 1]);
          }
          const float2 u = unpack2(pa), w = unpack2(pb);
          ps[j * D] = (u.x + u.y) + (w.x + w.y);
        }
      } else {
        // exact signs: sgn(x - hi), and -sgn(lo) where x == hi; landmark side
        // accumulates half of g sgn so that it combines with the fast path's 2 g [x > l].
        // hi = l / lscale: exact (a power of two, and in range whenever lscale != 1)
        const float unscale = cta_exact ? 1.f : -kInvBig;
        const float* lo_row = a.Llo + ((size_t)bh * a.m + abase + gr * LPT) * D + c;
        for (int j = 0; j < nv; ++j) {
          const float x = bf16_at(xr + j * D * 2, c);
          float s = 0.f;
#pragma unroll
          for (int i4 = 0; i4 < LPT / 4; ++i4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gbase + j * MC + 4 * i4);
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
            float e[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float li = l[4 * i4 + k] * unscale;
              e[k] = x > li ? 1.f : (x < li ? -1.f : 0.f);
              if (x == li && gr * LPT + 4 * i4 + k < mg) e[k] = -sgnf(__ldg(lo_row + (size_t)(4 * i4 + k) * D));
              s = fmaf(gv[k], e[k], s);
            }
            float2 u = unpack2(dl2[2 * i4]), w = unpack2(dl2[2 * i4 + 1]);
            u.x = fmaf(0.5f * gv[0], e[0], u.x);
            u.y = fmaf(0.5f * gv[1], e[1], u.y);
            w.x = fmaf(0.5f * gv[2], e[2], w.x);
            w.y = fmaf(0.5f * gv[3], e[3], w.y);
            dl2[2 * i4] = pack2(u.x, u.y);
            dl2[2 * i4 + 1] = pack2(w.x, w.y);
          }
          ps[j * D] = s;
        }
      }
    }
    __syncthreads();

    // ---- [r] token gradients: the 8 partial rows in a fixed order, the ties ----
    {
      const float* psb = reinterpret_cast<const float*>(sm + S::Ps);
      const float* gs = gsb;
      const int cc = tid & (D - 1);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = (tid >> 6) + 8 * r;
        if (j >= nv) continue;
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NGR; ++k) s += psb[(k * TJ + j) * D + cc];
        float dx;
        if (GAUSS) {
          dx = 2.f * (s - gsum_s[j] * bf16_at(sb + S::kXr + j * D * 2, cc));
        } else if (exact) {
          dx = -s;
        } else {
          dx = gsum_s[j] - 2.f * s;
          // a listed tie x == hi: the fast path took sgn = -1; the exact mean gives
          // -sgn(lo), so take back g (1 - sgn(lo))
          for (int k = 1; k <= nties; ++k) {
            const uint32_t t = tie_s[k];
            const int tj = (int)(t & 31u);
            if ((tj >> 4) != (b & 1) || (tj & 15) != j || (int)((t >> 5) & 127u) != cc) continue;
            const int at = (int)(t >> 12) - abase;
            if (at < 0 || at >= mg) continue;
            const float lo = __ldg(a.Llo + ((size_t)bh * a.m + abase + at) * D + cc);
            dx -= gs[j * MC + at] * (1.f - sgnf(lo));
          }
        }
        if (a.out != nullptr)
          a.out[((size_t)bh * a.N + n0 + j) * D + cc] = __float2bfloat16_rn(dx);
        else
          a.tok_part[(((size_t)gi * a.BH + bh) * a.N + n0 + j) * D + cc] = dx;
      }
      if (!GAUSS && !exact) {
        // the same ties on the landmark side: g (1 - sgn(lo)), halved like dl2
        for (int k = 1; k <= nties; ++k) {
          const uint32_t t = tie_s[k];
          const int tj = (int)(t & 31u);
          const int at = (int)(t >> 12) - abase - gr * LPT;
          if ((tj >> 4) != (b & 1) || (int)((t >> 5) & 127u) != c || at < 0 || at >= LPT ||
              gr * LPT + at >= mg)
            continue;
          const float lo = __ldg(a.Llo + ((size_t)bh * a.m + abase + gr * LPT + at) * D + c);
          const float corr = 0.5f * gs[(tj & 15) * MC + gr * LPT + at] * (1.f - sgnf(lo));
          // select-adds with compile-time indices keep dl2 in registers
#pragma unroll
          for (int p = 0; p < LPT / 2; ++p)
            dl2[p] = fma2(pack2(at == 2 * p ? corr : 0.f, at == 2 * p + 1 ? corr : 0.f),
                          pack2(1.f, 1.f), dl2[p]);
        }
      }
    }
  }

  // ---- drain: the copies and MMAs this CTA issued ----
  if (abort) {
    // the last commits cover every earlier MMA of thread 0
    if (ndot > 0)
      wait_or_flag(a.err, tc::smem_u32(&dotdone[(ndot - 1) & 1]), (uint32_t)((ndot - 1) >> 1) & 1u);
    if (nw > 0) wait_or_flag(a.err, tc::smem_u32(&wdone), (uint32_t)(nw - 1) & 1u);
    if (tid == 0)
      for (int k = i; k < min(nb, i + 2); ++k)
        wait_or_flag(a.err, tc::smem_u32(&full[k % NST]), (uint32_t)(k / NST) & 1u);
  } else if (DW && nb > 0) {
    wait_or_flag(a.err, tc::smem_u32(&wdone), (uint32_t)(nb - 1) & 1u);
  }
  tc::fence_after();
  __syncthreads();

  // ---- landmark-side sums: G'_a over the threads of each landmark ----
  float* colg_m = reinterpret_cast<float*>(sm + S::Ps);  // [4 / HF][MC]
  if (gact) colg_m[(HF == 2 ? (wg >> 1) : wg) * MC + ag] = colg_s[tid];
  __syncthreads();
  if (!abort) {
#pragma unroll
    for (int p = 0; p < LPT / 2; ++p) {
      const float2 u = unpack2(dl2[p]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int al = gr * LPT + 2 * p + h;
        if (al >= mg) continue;
        float cg = 0.f;
#pragma unroll
        for (int k = 0; k < 4 / HF; ++k) cg += colg_m[k * MC + al];
        const float v = h ? u.y : u.x;
        a.lm_part[(((size_t)bh * a.S + sp) * a.mp + abase + al) * D + c] =
            GAUSS ? 2.f * (v - cg * l[2 * p + h]) : 2.f * v - cg;
      }
    }
    if constexpr (DW) {
      // dW-hat partial of this token range: lane quarter q holds landmarks 32 q ..
      constexpr int NCOL = HF == 2 ? 32 : 16;
      const int hf = HF == 2 ? (wg >> 1) : 0, c0 = HF == 2 ? 32 * (wg & 1) : 16 * wg;
      if (gact) {
        uint32_t v[NCOL];
        tc::tmem_ld<NCOL>(tmem + ((uint32_t)(32 * q) << 16) + DWCOL + (uint32_t)(hf * 64 + c0), v);
        const int al = 128 * hf + 32 * q + lane;
        if (al < mg) {
          float* o = a.lm_part2 + (((size_t)bh * a.S + sp) * a.mp + abase + al) * D + c0;
#pragma unroll
          for (int k = 0; k < NCOL; k += 4)
            *reinterpret_cast<float4*>(o + k) =
                nb > 0 ? make_float4(__uint_as_float(v[k]), __uint_as_float(v[k + 1]),
                                     __uint_as_float(v[k + 2]), __uint_as_float(v[k + 3]))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool bwd_tc_shape(int dtype, int d) { return dtype == 1 && d == D; }

int bwd_tc_groups(int m) { return (m + 255) / 256; }

int bwd_tc_splits(int BH, int m, int N) {
  // Token splits per (slice, landmark group), from the dimensions alone (the
  // landmark-side summation order does not depend on the device): the count
  // that minimises rounds x (1 + blocks per CTA) on a 152-SM part, one CTA per
  // SM at a time, where a CTA's fixed cost (R planes, tensor memory, the
  // landmark-side epilogue) is about one 16-token block (measured on the PVT
  // stages: 1216 CTAs of 2-3 blocks and 160 CTAs of 13 blocks were both slower
  // than the minimum of this model); ties go to fewer splits.
  const int ng = bwd_tc_groups(m), nblk16 = (N + TJ - 1) / TJ;
  const long long units = (long long)BH * ng;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= nblk16 && s <= 4096; ++s) {
    const long long rounds = (units * s + 151) / 152;
    const long long cost = rounds * (1 + (nblk16 + s - 1) / s);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

template <int MODE, int MC, bool NORM, bool GAUSS>
static cudaError_t bwd_tc_t(const Prob& p, const BwdTcArgs& h, cudaStream_t st) {
  using SS = BSmem<MC, (MODE == 1) && !NORM>;
  static bool once = (allow_smem(k_bwd_tc<MODE, MC, NORM, GAUSS>, SS::total), true);
  (void)once;
  BtcArgs a;
  a.X = (const __nv_bfloat16*)h.X;
  a.U = (const __nv_bfloat16*)h.U;
  a.L = h.L; a.Llo = h.Llo; a.R = h.R; a.stats = h.stats; a.mdz = h.mdz; a.KV = h.kv;
  a.ties = h.ties; a.out = (__nv_bfloat16*)h.out; a.tok_part = h.tok_part;
  a.lm_part = h.lm_part; a.lm_part2 = h.lm_part2;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidSymbol;
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.S = h.S; a.nblk = (p.N + 31) / 32; a.BH = p.BH;
  a.inv_lam = p.inv_lam;
  static const char* names[3] = {"", "bwd_query", "bwd_key"};
  return launch(names[MODE], k_bwd_tc<MODE, MC, NORM, GAUSS>,
                dim3(h.S, bwd_tc_groups(p.m), p.BH), dim3(NTH), SS::total, st, a);
}

template <int MODE, bool NORM, bool GAUSS>
static cudaError_t bwd_tc_mc(const Prob& p, const BwdTcArgs& h, cudaStream_t st) {
  if (p.m <= 64) return bwd_tc_t<MODE, 64, NORM, GAUSS>(p, h, st);
  if (p.m <= 128) return bwd_tc_t<MODE, 128, NORM, GAUSS>(p, h, st);
  return bwd_tc_t<MODE, 256, NORM, GAUSS>(p, h, st);
}

cudaError_t run_bwd_tc(const Prob& p, int mode, const BwdTcArgs& h, cudaStream_t st) {
  if (!bwd_tc_shape(p.dtype, p.d)) return cudaErrorInvalidValue;
  if (mode == 1) {
    if (p.norm())
      return p.gauss() ? bwd_tc_mc<1, true, true>(p, h, st) : bwd_tc_mc<1, true, false>(p, h, st);
    return p.gauss() ? bwd_tc_mc<1, false, true>(p, h, st) : bwd_tc_mc<1, false, false>(p, h, st);
  }
  return p.gauss() ? bwd_tc_mc<2, false, true>(p, h, st) : bwd_tc_mc<2, false, false>(p, h, st);
}

}  // namespace lapnys
