// Token-side forward passes of the Gaussian-kernel variant on the
// 5th-generation tensor cores (bf16 inputs, d = 32 or 64, m > 64):
//
//   k(x, l) = exp(-|x - l|_2^2 / lambda)   (the SOFT review's Proposed method:
//   a symmetric, [0, 1]-valued Gaussian kernel; read with the caller's lambda)
//
// The squared distance expands to |x|^2 + |l|^2 - 2 x.l, a dense contraction,
// so unlike the L1 distance it runs on the tensor cores: per tile one MMA
// (kind::tf32) forms x.l into TMEM, the warps read it back (tcgen05.ld), form
// exp2(ns (|x|^2 + |l|^2 - 2 x.l)) and write the kernel values as the A operand
// of the second MMA (the contraction with W-hat or V), as in k_fwd_tc.cu.
// The landmarks enter the first MMA rounded to TF32 (l~); their norms are taken
// of the same rounded values, so the distance is |x - l~|^2 exactly in real
// arithmetic (bf16 queries / keys are exact in TF32).
//
//   query pass  persistent CTAs over items of 128 queries (M); per 64-landmark
//               tile: S = X L~^T (N = 64, K = d), P = k, O += Z W-hat (N = d,
//               K = 64).  L~ with its norms and W-hat^T are packed once per
//               forward (k_pack_qg) and fetched by bulk copy a tile ahead.
//   key pass    one CTA per (128-landmark tile, token range, slice); per
//               64-token block: S = L~ K^T, C = k, W += C^T-as-A x V.
//
// Every mbarrier wait is bounded; on expiry the kernel records an error in the
// device word read by lapnys_device_status and carries on.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int QM = 128;                      // rows of both MMAs (queries, or landmarks)
constexpr int TL = 64;                       // landmarks per query tile / keys per key block
constexpr int NTH = 512;                     // threads per CTA
constexpr uint32_t kSbo = 128;               // 8-row groups 128 bytes apart (dense)
constexpr uint32_t kLbo128 = (QM / 8) * kSbo;  // K groups of a 128-row operand
constexpr uint32_t kLbo64 = (TL / 8) * kSbo;   // K groups of a 64-row operand
constexpr uint32_t kTileP = (TL / 4) * kLbo128;  // 128 x 64 A operand of the second MMA
constexpr uint32_t kSboVB = 144;             // key pass V^T: 8-row groups 144 bytes apart
constexpr uint32_t kScol = 128;              // first TMEM column of the two S buffers
// key pass: W += C^T V as kind::f16 MMAs with V exact in bf16 and C as three bf16
// planes (24 significant bits; W is amplified by X_T in W-hat = X_T W)
constexpr uint32_t kLboC = (QM / 8) * kSbo + 16;  // C^T planes: 8-key K groups, 2064 bytes apart
constexpr uint32_t kPlaneC = (TL / 8) * kLboC;
constexpr uint32_t kCols = 256;              // TMEM columns: accumulator [0, d), S at 128, 192

__device__ __forceinline__ float tf32f(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}
// bounded wait for a phase of an mbarrier; on expiry the error word is set
__device__ __forceinline__ bool wait_or_flag(int* err, uint32_t bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  if (!ok) atomicOr(err, 1);
  return ok;
}
__device__ __forceinline__ void bf16x8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}
// byte offset of (row, k) in a K-major operand whose K groups are `lbo` apart
__device__ __forceinline__ uint32_t kmaj(int row, int k, uint32_t lbo, uint32_t sbo) {
  return (uint32_t)(k >> 2) * lbo + (uint32_t)(row >> 3) * sbo + (uint32_t)(row & 7) * 16u +
         (uint32_t)(k & 3) * 4u;
}

template <int D>
struct GQ {
  static constexpr uint32_t kTileX = (D / 4) * kLbo128;      // queries as A of S
  static constexpr uint32_t kTileL = (D / 4) * kLbo64;       // landmarks as B of S
  static constexpr uint32_t kRec = kTileL + TL * 4;          // + |l~|^2 of the 64 landmarks
  static constexpr uint32_t kLboW = (D / 8) * kSbo;          // W-hat^T as B of O
  static constexpr uint32_t kTileW = (TL / 4) * kLboW;
  static constexpr uint32_t Xa = 0;
  static constexpr uint32_t Lb = Xa + kTileX;                // 2 x landmark records
  static constexpr uint32_t Wt = Lb + 2 * kRec;              // 3 x W-hat^T tiles
  static constexpr uint32_t Pa = Wt + 3 * kTileW;            // 2 x A tiles of O
  static constexpr uint32_t Xn = Pa + 2 * kTileP;            // |x|^2 of the item's queries
  static constexpr uint32_t kRow = D * 2 + 16;               // padded raw row
  static constexpr uint32_t Raw = Xn + QM * 4;
  static constexpr uint32_t total = Raw + QM * kRow;
};

template <int D>
struct GK {
  static constexpr uint32_t kTileL = (D / 4) * kLbo128;      // landmarks as A of S
  static constexpr uint32_t kTileK = (D / 4) * kLbo64;       // keys as B of S
  static constexpr uint32_t kLboV = (D / 8) * kSboVB;        // V^T (bf16) as B of W
  static constexpr uint32_t kTileV = (TL / 8) * kLboV;
  static constexpr uint32_t La = 0;
  static constexpr uint32_t Ln = La + kTileL;                // |l~|^2 of the CTA's landmarks
  static constexpr uint32_t Kb = Ln + QM * 4;
  static constexpr uint32_t Kn = Kb + kTileK;                // |k|^2 of the block's keys
  static constexpr uint32_t Vb = Kn + TL * 4;                // 2 x V^T tiles
  static constexpr uint32_t Ca = Vb + 2 * kTileV;            // 2 x 3 C^T planes (A of W)
  static constexpr uint32_t kRow = D * 2 + 16;
  static constexpr uint32_t Raw = Ca + 6 * kPlaneC;          // 2 x (64 key rows, 64 value rows)
  static constexpr uint32_t kRawBuf = 2 * TL * kRow;
  static constexpr uint32_t total = Raw + 2 * kRawBuf;
};
}  // namespace

// ---------------------------------------------------------------------------
// pack, per slice and 64-landmark tile t (zero past m):
//   LB[bh][t]: l~ (TF32-rounded landmarks) as the K-major B operand of S
//              (row = landmark, k = feature), then |l~|^2 of the 64 landmarks
//   WT[bh][t]: W-hat rows of the tile as the K-major B operand of O
//              (row = feature, k = landmark), TF32-rounded
// grid (nt, BH)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) k_pack_qg(const float* __restrict__ L,
                                                      const float* __restrict__ What,
                                                      uint8_t* __restrict__ LB,
                                                      float* __restrict__ WT, int m, int nt) {
  const int t = blockIdx.x, bh = blockIdx.y;
  uint8_t* lb = LB + ((size_t)bh * nt + t) * GQ<D>::kRec;
  float* wt = WT + ((size_t)bh * nt + t) * D * TL;
  for (int e = threadIdx.x; e < TL * D; e += kThreads) {
    const int al = e / D, c = e % D, a = t * TL + al;
    const bool ok = a < m;
    const float l = ok ? tf32f(__ldg(L + ((size_t)bh * m + a) * D + c)) : 0.f;
    const float w = ok ? __ldg(What + ((size_t)bh * m + a) * D + c) : 0.f;
    *reinterpret_cast<float*>(lb + kmaj(al, c, kLbo64, kSbo)) = l;
    wt[(al >> 2) * (GQ<D>::kLboW / 4) + (c >> 3) * (kSbo / 4) + (c & 7) * 4 + (al & 3)] = tf32f(w);
  }
  if (threadIdx.x < TL) {
    const int al = threadIdx.x, a = t * TL + al;
    float s = 0.f;
    if (a < m)
      for (int c = 0; c < D; ++c) {
        const float l = tf32f(__ldg(L + ((size_t)bh * m + a) * D + c));
        s = fmaf(l, l, s);
      }
    reinterpret_cast<float*>(lb + GQ<D>::kTileL)[al] = s;
  }
}

// ---------------------------------------------------------------------------
// query pass
// ---------------------------------------------------------------------------
struct GQArgs {
  const __nv_bfloat16* Q;
  const uint8_t* LB;
  const float* WT;
  const float* stats;  // [BH][3][m] (norm)
  __nv_bfloat16* O;
  float* kvout;        // [BH][N][mp] kernel values P, or null
  int* err;
  int N, m, mp, nt, nb, items;
  float ns;
};

template <int D, bool NORM>
__global__ void __launch_bounds__(NTH, 1) k_query_gtc(GQArgs a) {
  using S = GQ<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[3];   // landmark record and W-hat^T tile landed
  __shared__ __align__(8) uint64_t sdone;     // S = X L~^T of the current tile completed
  __shared__ __align__(8) uint64_t mdone[2];  // O MMAs reading A buffer b completed
  __shared__ uint32_t tmem_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cg = warp >> 2;  // TMEM lanes 32 quarter .., column group
  const uint32_t idS = tc::idesc_tf32(QM, TL), idO = tc::idesc_tf32(QM, D);

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(tc::smem_u32(&full[i]), 1);
    tc::mbar_init(tc::smem_u32(&sdone), 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&mdone[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  // operands of tile g (item `item`, landmark tile t): the landmark record into
  // Lb[g % 2], the W-hat^T tile into Wt[g % 3]
  auto issue_tile = [&](uint32_t g, int item, int t) {
    const int bh = item / a.nb;
    const uint32_t bar = tc::smem_u32(&full[g % 3]);
    tc::mbar_expect_tx(bar, S::kRec + S::kTileW);
    const size_t tile = (size_t)bh * a.nt + t;
    tc::bulk_g2s(tc::smem_u32(sm + S::Lb + (g & 1) * S::kRec), a.LB + tile * S::kRec, S::kRec, bar);
    tc::bulk_g2s(tc::smem_u32(sm + S::Wt + (g % 3) * S::kTileW), a.WT + tile * D * TL, S::kTileW,
                 bar);
  };
  auto prefetch_q = [&](int item) {
    if (item >= a.items) return;
    const int bh = item / a.nb, j0 = (item % a.nb) * QM;
    constexpr int CH = D / 8;
    for (int e = tid; e < QM * CH; e += NTH) {
      const int j = e % QM, ch = e / QM;
      const bool ok = j0 + j < a.N;
      const __nv_bfloat16* src = a.Q + ((size_t)bh * a.N + (ok ? j0 + j : 0)) * D + 8 * ch;
      cp_async16(smem_addr(sm + S::Raw + j * S::kRow + 16 * ch), src, ok);
    }
    cp_commit();
  };

  // An expired wait (bad) stops the CTA at its next barrier, taken by all
  // threads alike (__syncthreads_or): no further copy or MMA is issued, and the
  // copies and MMAs already in flight are waited for (bounded) before the
  // tensor memory is freed.
  uint32_t g = 0;
  bool bad = false, abort = false;
  int last_mma = -1;     // last tile whose contraction MMAs were issued
  int last_s = -1;       // last tile whose distance MMAs were issued (thread 0)
  uint32_t issued = 0;   // tiles whose operand copies were issued (thread 0)
  if (tid == 0 && (int)blockIdx.x < a.items) {
    issue_tile(0, blockIdx.x, 0);
    issued = 1;
  }
  prefetch_q(blockIdx.x);
  for (int item = blockIdx.x; item < a.items; item += gridDim.x) {
    const int bh = item / a.nb, j0 = (item % a.nb) * QM;
    cp_wait_all();
    // this item's rows landed; the previous item's MMAs have completed
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    {
      // raw rows -> A operand of S (bf16 is exact in TF32); lanes take consecutive queries
      constexpr int CH = D / 8;
      for (int e = tid; e < QM * CH; e += NTH) {
        const int j = e % QM, ch = e / QM;
        float f[8];
        bf16x8(*reinterpret_cast<const uint4*>(sm + S::Raw + j * S::kRow + 16 * ch), f);
        *reinterpret_cast<float4*>(sm + S::Xa + kmaj(j, 8 * ch, kLbo128, kSbo)) =
            make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(sm + S::Xa + kmaj(j, 8 * ch + 4, kLbo128, kSbo)) =
            make_float4(f[4], f[5], f[6], f[7]);
      }
    }
    __syncthreads();
    if (tid < QM) {
      // |x|^2 of each query, features in ascending order
      float s = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < D / 4; ++k4) {
        const float4 v = *reinterpret_cast<const float4*>(sm + S::Xa + kmaj(tid, 4 * k4, kLbo128, kSbo));
        s = fmaf(v.x, v.x, s);
        s = fmaf(v.y, v.y, s);
        s = fmaf(v.z, v.z, s);
        s = fmaf(v.w, v.w, s);
      }
      reinterpret_cast<float*>(sm + S::Xn)[tid] = s;
    }
    tc::fence_async_smem();
    __syncthreads();
    prefetch_q(item + gridDim.x);

    for (int t = 0; t < a.nt; ++t, ++g) {
      bad |= !wait_or_flag(a.err, tc::smem_u32(&full[g % 3]), (g / 3) & 1);
      const uint32_t sbuf = kScol + (g & 1) * TL;
      if (tid == 0 && !bad) {
        tc::fence_after();
        const uint32_t xa = tc::smem_u32(sm + S::Xa);
        const uint32_t lb = tc::smem_u32(sm + S::Lb + (g & 1) * S::kRec);
#pragma unroll
        for (int k8 = 0; k8 < D / 8; ++k8)
          tc::mma_ss(tmem + sbuf, tc::desc(xa + k8 * 2 * kLbo128, kLbo128, kSbo),
                     tc::desc(lb + k8 * 2 * kLbo64, kLbo64, kSbo), idS, k8 > 0 ? 1u : 0u);
        tc::commit(tc::smem_u32(&sdone));
        last_s = (int)g;
        // tile g + 1: its landmark record goes where tile g - 1's was (that S MMA
        // completed before tile g - 1's epilogue); its W-hat^T where MMA g - 2 read
        int nitem = item, nt1 = t + 1;
        if (nt1 == a.nt) { nitem = item + gridDim.x; nt1 = 0; }
        if (nitem < a.items) {
          if (g >= 2) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[g & 1]), ((g - 2) >> 1) & 1);
          if (!bad) {
            issue_tile(g + 1, nitem, nt1);
            issued = g + 2;
          }
        }
      }
      // (thread 0 skips the distance MMAs after an expired wait; the others' wait
      // for them then expires too, and the barrier below stops the CTA)
      bad |= !wait_or_flag(a.err, tc::smem_u32(&sdone), g & 1);
      tc::fence_after();
      uint32_t v[16];
      tc::tmem_ld<16>(tmem + ((uint32_t)(32 * quarter) << 16) + sbuf + 16 * cg, v);
      // the A buffer of O for this tile was read by MMA g - 2
      if (g >= 2) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[g & 1]), ((g - 2) >> 1) & 1);
      {
        const int jl = 32 * quarter + lane, j = j0 + jl;
        const int al0 = 16 * cg, ab = t * TL + al0;  // this thread's 16 landmarks
        const float xn = reinterpret_cast<const float*>(sm + S::Xn)[jl];
        const float* ln = reinterpret_cast<const float*>(sm + S::Lb + (g & 1) * S::kRec + S::kTileL);
        float p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float dist = fmaxf(fmaf(-2.f, __uint_as_float(v[i]), xn + ln[al0 + i]), 0.f);
          p[i] = ab + i < a.m ? exp2_ftz(dist * a.ns) : 0.f;
        }
        if (a.kvout != nullptr && j < a.N) {
          float* o = a.kvout + ((size_t)bh * a.N + j) * a.mp + ab;
#pragma unroll
          for (int i = 0; i < 16; i += 4) st4(o + i, make_float4(p[i], p[i + 1], p[i + 2], p[i + 3]));
        }
        if (NORM) {
          const float* st = a.stats + (size_t)bh * 3 * a.m;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const bool ok = ab + i < a.m;
            p[i] = ok ? (p[i] - __ldg(st + ab + i)) * __ldg(st + 2 * a.m + ab + i) : 0.f;
          }
        }
        uint8_t* pa = sm + S::Pa + (g & 1) * kTileP;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(pa + kmaj(jl, al0 + i, kLbo128, kSbo)) =
              make_float4(tf32f(p[i]), tf32f(p[i + 1]), tf32f(p[i + 2]), tf32f(p[i + 3]));
      }
      tc::fence_async_smem();
      tc::fence_before();
      if (__syncthreads_or(bad)) {
        abort = true;
        break;
      }
      if (tid == 0) {
        tc::fence_after();
        const uint32_t pa = tc::smem_u32(sm + S::Pa + (g & 1) * kTileP);
        const uint32_t wb = tc::smem_u32(sm + S::Wt + (g % 3) * S::kTileW);
#pragma unroll
        for (int k8 = 0; k8 < TL / 8; ++k8)
          tc::mma_ss(tmem, tc::desc(pa + k8 * 2 * kLbo128, kLbo128, kSbo),
                     tc::desc(wb + k8 * 2 * S::kLboW, S::kLboW, kSbo), idO,
                     (t > 0 || k8 > 0) ? 1u : 0u);
        tc::commit(tc::smem_u32(&mdone[g & 1]));
      }
      last_mma = (int)g;
    }
    if (abort) break;
    // the item's accumulator: lane quarter w % 4 holds queries 32 (w % 4) .., the
    // four warps of a quarter split the columns
    bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[(g - 1) & 1]), ((g - 1) >> 1) & 1);
    tc::fence_after();
    {
      constexpr int HC = D / 4;
      uint32_t v[HC];
      tc::tmem_ld<HC>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(cg * HC), v);
      const int j = j0 + 32 * quarter + lane;
      if (j < a.N) {
        uint4* o = reinterpret_cast<uint4*>(a.O + ((size_t)bh * a.N + j) * D + cg * HC);
#pragma unroll
        for (int c = 0; c < HC; c += 8) {
          uint4 w;
          const __nv_bfloat162 p0 = __floats2bfloat162_rn(__uint_as_float(v[c]), __uint_as_float(v[c + 1]));
          const __nv_bfloat162 p1 = __floats2bfloat162_rn(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
          const __nv_bfloat162 p3 = __floats2bfloat162_rn(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
          w.x = *reinterpret_cast<const uint32_t*>(&p0);
          w.y = *reinterpret_cast<const uint32_t*>(&p1);
          w.z = *reinterpret_cast<const uint32_t*>(&p2);
          w.w = *reinterpret_cast<const uint32_t*>(&p3);
          o[c / 8] = w;
        }
      }
    }
    tc::fence_before();
  }
  cp_wait_all();
  if (abort) {
    // drain what this CTA issued: the last MMAs (a commit covers every earlier
    // MMA of its thread) and the operand tiles not yet waited for
    if (last_mma >= 0)
      wait_or_flag(a.err, tc::smem_u32(&mdone[last_mma & 1]), ((uint32_t)last_mma >> 1) & 1);
    if (tid == 0) {
      if (last_s > last_mma) wait_or_flag(a.err, tc::smem_u32(&sdone), (uint32_t)last_s & 1);
      for (uint32_t gi = g; gi < issued; ++gi)
        wait_or_flag(a.err, tc::smem_u32(&full[gi % 3]), (gi / 3) & 1);
    }
    tc::fence_before();
  }
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// key pass, grid (128-landmark tile, token range, slice)
// ---------------------------------------------------------------------------
struct GKArgs {
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const float* L;
  float* part;   // [BH][S][mp][d] partial W
  float* kvout;  // [BH][N][mp] kernel values C, or null
  int* err;
  int N, m, mp, S, nblk;
  float ns;
};

template <int D>
__global__ void __launch_bounds__(NTH, 1) k_key_gtc(GKArgs a) {
  using S = GK<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t sdone;     // S = L~ K^T of the current block completed
  __shared__ __align__(8) uint64_t mdone[2];  // W MMAs reading Vb[b], Ca[b] completed
  __shared__ uint32_t tmem_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cg = warp >> 2;
  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * QM;
  const uint32_t idS = tc::idesc_tf32(QM, TL), idW = tc::idesc_bf16(QM, D);
  const __nv_bfloat16* Kb = a.K + (size_t)bh * a.N * D;
  const __nv_bfloat16* Vb = a.V + (size_t)bh * a.N * D;

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    tc::mbar_init(tc::smem_u32(&sdone), 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&mdone[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the CTA's landmarks l~ as the A operand of S (zero past m), and |l~|^2
  for (int e = tid; e < QM * D; e += NTH) {
    const int al = e / D, c = e % D;
    const float l = a0 + al < a.m ? tf32f(__ldg(a.L + ((size_t)bh * a.m + a0 + al) * D + c)) : 0.f;
    *reinterpret_cast<float*>(sm + S::La + kmaj(al, c, kLbo128, kSbo)) = l;
  }
  if (tid < QM) {
    float s = 0.f;
    if (a0 + tid < a.m)
      for (int c = 0; c < D; ++c) {
        const float l = tf32f(__ldg(a.L + ((size_t)bh * a.m + a0 + tid) * D + c));
        s = fmaf(l, l, s);
      }
    reinterpret_cast<float*>(sm + S::Ln)[tid] = s;
  }
  tc::fence_async_smem();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  const int b0 = (int)((long long)a.nblk * sp / a.S), b1 = (int)((long long)a.nblk * (sp + 1) / a.S);
  auto prefetch = [&](int b, int buf) {
    if (b >= b1) return;
    const int n0 = b * TL;
    constexpr int CH = D / 8;
    uint8_t* rb = sm + S::Raw + buf * S::kRawBuf;
    for (int e = tid; e < 2 * TL * CH; e += NTH) {
      const int which = e / (TL * CH), rem = e % (TL * CH), j = rem % TL, ch = rem / TL;
      const bool ok = n0 + j < a.N;
      const __nv_bfloat16* src = (which ? Vb : Kb) + (size_t)(ok ? n0 + j : 0) * D + 8 * ch;
      cp_async16(smem_addr(rb + (which * TL + j) * S::kRow + 16 * ch), src, ok);
    }
    cp_commit();
  };
  prefetch(b0, 0);
  // An expired wait (bad) stops the CTA before its next MMAs, decided by all
  // threads alike (__syncthreads_or); the MMAs already issued and the copies in
  // flight are waited for (bounded) before the tensor memory is freed.
  bool bad = false, abort = false;
  int s_block = -1;  // last block whose distance MMAs were issued
  int i = 0;
  for (int b = b0; b < b1; ++b, ++i) {
    const int buf = i & 1;
    cp_wait_all();
    __syncthreads();  // block b's rows landed; block i - 1's S was read out
    // Vb[buf] and Ca[buf] were last read by MMA i - 2
    if (i >= 2) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[buf]), ((i - 2) >> 1) & 1);
    {
      const uint8_t* rb = sm + S::Raw + buf * S::kRawBuf;
      constexpr int CH = D / 8;
      // keys -> B operand of S (exact); lanes take consecutive keys
      for (int e = tid; e < TL * CH; e += NTH) {
        const int j = e % TL, ch = e / TL;
        float f[8];
        bf16x8(*reinterpret_cast<const uint4*>(rb + j * S::kRow + 16 * ch), f);
        *reinterpret_cast<float4*>(sm + S::Kb + kmaj(j, 8 * ch, kLbo64, kSbo)) =
            make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(sm + S::Kb + kmaj(j, 8 * ch + 4, kLbo64, kSbo)) =
            make_float4(f[4], f[5], f[6], f[7]);
      }
      // values -> bf16 B operand of W (row = feature, k = key); a thread takes a
      // key pair and 8 features, lanes: 8 feature groups x 4 key pairs
      uint8_t* vb = sm + S::Vb + buf * S::kTileV;
      for (int e = tid; e < (TL / 2) * CH; e += NTH) {
        const int ch = e % CH, j = 2 * (e / CH);
        const uint4 u0 = *reinterpret_cast<const uint4*>(rb + (TL + j) * S::kRow + 16 * ch);
        const uint4 u1 = *reinterpret_cast<const uint4*>(rb + (TL + j + 1) * S::kRow + 16 * ch);
        const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w}, w1[4] = {u1.x, u1.y, u1.z, u1.w};
        uint8_t* dst = vb + (j >> 3) * S::kLboV + ch * kSboVB + (j & 7) * 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint32_t*>(dst + (2 * q) * 16) = (w0[q] & 0xffffu) | (w1[q] << 16);
          *reinterpret_cast<uint32_t*>(dst + (2 * q + 1) * 16) = (w0[q] >> 16) | (w1[q] & 0xffff0000u);
        }
      }
      if (tid < TL) {
        // |k|^2 of each key, features in ascending order
        float s = 0.f;
        for (int ch = 0; ch < CH; ++ch) {
          float f[8];
          bf16x8(*reinterpret_cast<const uint4*>(rb + tid * S::kRow + 16 * ch), f);
#pragma unroll
          for (int q = 0; q < 8; ++q) s = fmaf(f[q], f[q], s);
        }
        reinterpret_cast<float*>(sm + S::Kn)[tid] = s;
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    prefetch(b + 1, buf ^ 1);
    if (tid == 0) {
      tc::fence_after();
      const uint32_t la = tc::smem_u32(sm + S::La), kb = tc::smem_u32(sm + S::Kb);
#pragma unroll
      for (int k8 = 0; k8 < D / 8; ++k8)
        tc::mma_ss(tmem + kScol, tc::desc(la + k8 * 2 * kLbo128, kLbo128, kSbo),
                   tc::desc(kb + k8 * 2 * kLbo64, kLbo64, kSbo), idS, k8 > 0 ? 1u : 0u);
      tc::commit(tc::smem_u32(&sdone));
    }
    s_block = i;
    bad |= !wait_or_flag(a.err, tc::smem_u32(&sdone), i & 1);
    tc::fence_after();
    {
      uint32_t v[16];
      tc::tmem_ld<16>(tmem + ((uint32_t)(32 * quarter) << 16) + kScol + 16 * cg, v);
      const int al = 32 * quarter + lane, aa = a0 + al;   // this thread's landmark
      const int jl0 = 16 * cg, n0 = b * TL;               // and 16 keys
      const float lnv = reinterpret_cast<const float*>(sm + S::Ln)[al];
      const float* kn = reinterpret_cast<const float*>(sm + S::Kn);
      float c[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float dist = fmaxf(fmaf(-2.f, __uint_as_float(v[q]), lnv + kn[jl0 + q]), 0.f);
        c[q] = (aa < a.m && n0 + jl0 + q < a.N) ? exp2_ftz(dist * a.ns) : 0.f;
      }
      if (a.kvout != nullptr && aa < a.mp) {
        // keep the kernel values for the backward: lanes write consecutive landmarks of a key row
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int j = n0 + jl0 + q;
          if (j < a.N) a.kvout[((size_t)bh * a.N + j) * a.mp + aa] = c[q];
        }
      }
      // C^T as three bf16 planes (row = landmark al, k = keys jl0 .. jl0 + 15)
      uint8_t* ca = sm + S::Ca + buf * 3 * kPlaneC + (uint32_t)(al >> 3) * kSbo +
                    (uint32_t)(al & 7) * 16u;
      uint32_t pl[3][8];
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        uint32_t w[3];
        split3_bf16x2(c[q], c[q + 1], w);
#pragma unroll
        for (int p = 0; p < 3; ++p) pl[p][q / 2] = w[p];
      }
#pragma unroll
      for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          *reinterpret_cast<uint4*>(ca + p * kPlaneC + (uint32_t)((jl0 >> 3) + h) * kLboC) =
              make_uint4(pl[p][4 * h], pl[p][4 * h + 1], pl[p][4 * h + 2], pl[p][4 * h + 3]);
    }
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    if (tid == 0) {
      tc::fence_after();
      const uint32_t ca = tc::smem_u32(sm + S::Ca + buf * 3 * kPlaneC);
      const uint32_t vbs = tc::smem_u32(sm + S::Vb + buf * S::kTileV);
#pragma unroll
      for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k16 = 0; k16 < TL / 16; ++k16)
          tc::mma_bf16(tmem, tc::desc(ca + p * kPlaneC + k16 * 2 * kLboC, kLboC, kSbo),
                       tc::desc(vbs + k16 * 2 * S::kLboV, S::kLboV, kSboVB), idW,
                       (i > 0 || p > 0 || k16 > 0) ? 1u : 0u);
      tc::commit(tc::smem_u32(&mdone[buf]));
    }
  }
  cp_wait_all();  // the next block's rows, when the loop stopped early
  // the contraction MMAs of blocks < i, and the distance MMAs of block i when the
  // loop stopped after issuing them (a commit covers every earlier MMA)
  if (i > 0) wait_or_flag(a.err, tc::smem_u32(&mdone[(i - 1) & 1]), ((i - 1) >> 1) & 1);
  if (abort && s_block == i) wait_or_flag(a.err, tc::smem_u32(&sdone), (uint32_t)i & 1);
  tc::fence_after();
  if (!abort) {
    constexpr int HC = D / 4;
    uint32_t v[HC];
    tc::tmem_ld<HC>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(cg * HC), v);
    const int al = a0 + 32 * quarter + lane;
    if (al < a.mp) {
      float4* o = reinterpret_cast<float4*>(a.part + (((size_t)bh * a.S + sp) * a.mp + al) * D + cg * HC);
#pragma unroll
      for (int c = 0; c < HC; c += 4)
        o[c / 4] = i > 0 ? make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                       __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
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
cudaError_t run_pack_qg(const Prob& p, const float* L, const float* What, void* packL, float* packW,
                        cudaStream_t st) {
  if (p.d == 32)
    return launch("pack_q", k_pack_qg<32>, dim3(p.nt, p.BH), dim3(kThreads), 0, st, L, What,
                  (uint8_t*)packL, packW, p.m, p.nt);
  if (p.d == 64)
    return launch("pack_q", k_pack_qg<64>, dim3(p.nt, p.BH), dim3(kThreads), 0, st, L, What,
                  (uint8_t*)packL, packW, p.m, p.nt);
  return cudaErrorInvalidValue;
}

// SMs of the current device (the persistent query pass's grid only)
static int sm_count_g() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

template <int D, bool NORM>
static cudaError_t query_gtc_t(const Prob& p, const void* q, const void* packL, const float* packW,
                               const float* stats, void* out, float* kvout, cudaStream_t st) {
  const size_t smem = GQ<D>::total;
  static bool once = (allow_smem(k_query_gtc<D, NORM>, smem), true);
  (void)once;
  GQArgs a;
  a.Q = (const __nv_bfloat16*)q;
  a.LB = (const uint8_t*)packL;
  a.WT = packW;
  a.stats = stats;
  a.O = (__nv_bfloat16*)out;
  a.kvout = kvout;
  a.err = wait_error_address();
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.nt = p.nt;
  a.nb = (p.N + QM - 1) / QM;
  a.items = a.nb * p.BH;
  a.ns = p.ns;
  const int grid = a.items < sm_count_g() ? a.items : sm_count_g();
  return launch("query_fwd", k_query_gtc<D, NORM>, dim3(grid), dim3(NTH), smem, st, a);
}

cudaError_t run_query_gtc(const Prob& p, const void* q, const void* packL, const float* packW,
                          const float* stats, void* out, float* kvout, cudaStream_t st) {
  if (p.d == 32) return p.norm() ? query_gtc_t<32, true>(p, q, packL, packW, stats, out, kvout, st)
                                 : query_gtc_t<32, false>(p, q, packL, packW, stats, out, kvout, st);
  if (p.d == 64) return p.norm() ? query_gtc_t<64, true>(p, q, packL, packW, stats, out, kvout, st)
                                 : query_gtc_t<64, false>(p, q, packL, packW, stats, out, kvout, st);
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t key_gtc_t(const Prob& p, const void* k, const void* v, const float* L,
                             float* part, float* kvout, cudaStream_t st) {
  const size_t smem = GK<D>::total;
  static bool once = (allow_smem(k_key_gtc<D>, smem), true);
  (void)once;
  GKArgs a;
  a.K = (const __nv_bfloat16*)k;
  a.V = (const __nv_bfloat16*)v;
  a.L = L;
  a.part = part;
  a.kvout = kvout;
  a.err = wait_error_address();
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.S = p.Skt; a.nblk = p.nblk;
  a.ns = p.ns;
  const int nt = (p.m + QM - 1) / QM;
  return launch("key_fwd", k_key_gtc<D>, dim3(nt, p.Skt, p.BH), dim3(NTH), smem, st, a);
}

cudaError_t run_key_gtc(const Prob& p, const void* k, const void* v, const float* L, float* part,
                        float* kvout, cudaStream_t st) {
  if (p.d == 32) return key_gtc_t<32>(p, k, v, L, part, kvout, st);
  if (p.d == 64) return key_gtc_t<64>(p, k, v, L, part, kvout, st);
  return cudaErrorInvalidValue;
}

}  // namespace lapnys
