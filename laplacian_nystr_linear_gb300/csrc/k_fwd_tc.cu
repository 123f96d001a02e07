// Token-side forward passes of Laplacian-kernel Nystrom attention (and of its
// Gaussian-kernel variant) with the contractions on the 5th-generation tensor
// cores (bf16 inputs, d = 32 or 64, m > 64):
//
//   query pass   O = Z W-hat,  Z = P or (P - mu) / sqrt(var + eta),  P_ia = k(Q_i, L_a)
//   key pass     W = C V,      C_aj = k(L_a, K_j)
//
// with k(x, y) = exp(-|x - y|_1 / lambda) ("LaplacianFormer", Dutch summary
// Methodology 1; Arabic summary 2a) and the Nystrom product read as
// O = k(Q, L) A^+ (k(L, K) V) ("SOFT" review, Proposed method).
//
// The L1 distances run on the FP32 pipe: each of 512 threads holds a 4 x 4
// block of distances (summed over the features in ascending order) and reads
// both operands from feature-major tiles, one 16-byte load per four values.
// The kernel values, rounded to TF32, go straight into the K-major operand
// layout of the MMA: a thread's 4 x 4 block is half a core matrix (8 rows x 16
// bytes).  One thread then issues the tile's tcgen05.mma (kind::tf32, M = 128)
// into a TMEM accumulator and commits them to an mbarrier while every warp
// moves on to the next tile's distances; a shared-memory operand buffer is
// rewritten only after the MMAs that read it have completed.
//
// Query pass: persistent CTAs over items of 128 queries (M); the landmarks
// come in tiles of 64 (K), each with its W-hat tile, pre-packed in global
// memory (k_pack_q) and fetched by the bulk-copy engine, three tiles ahead of
// their MMAs.  The next item's query rows are copied in (cp.async) while the
// current item computes.
// Key pass: one CTA per (128-landmark tile (M), token range, slice); the
// key / value rows stream in blocks of 64 tokens (K), double buffered; V goes
// into the B operand (bf16 is exact in TF32), C^T into the A operand; the
// accumulated W tile is a per-range partial summed afterwards.
//
// Every mbarrier wait is bounded: on expiry the kernel records an error in the
// device word read by lapnys_device_status and carries on (results are then
// garbage, flagged); it never spins forever.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int QM = 128;                         // queries per query item / landmarks per key tile (M)
constexpr int TL = 64;                          // landmarks per query tile / tokens per key block (K)
constexpr uint32_t kSbo = 128;                  // A: 8-row groups 128 bytes apart
constexpr uint32_t kLboA = (QM / 8) * kSbo + 16;  // A: 4-wide K groups 2064 bytes apart (bank spread)
constexpr uint32_t kTileA = (TL / 4) * kLboA;   // one A tile (M = 128, K = 64)
constexpr uint32_t kSboVB = 144;                // key-pass B (V^T): 8-row groups 144 bytes apart
constexpr int NTH = 512;                        // threads per CTA (4 warps per SM sub-partition)

template <int D>
struct QSmem {
  static constexpr uint32_t Xt = 0;                            // [D][QM] f32, feature-major queries
  static constexpr uint32_t Lt = Xt + D * QM * 4;              // 2 x [D][TL] f32 landmark tiles
  static constexpr uint32_t Wt = Lt + 2 * D * TL * 4;          // 3 x packed W-hat^T tiles (B)
  static constexpr uint32_t Pa = Wt + 3 * D * TL * 4;          // 2 x A tiles (Z, TF32)
  static constexpr uint32_t Raw = Pa + 2 * kTileA;             // next item's query rows (bf16)
  static constexpr uint32_t kRow = D * 2 + 16;                 // padded raw row
  static constexpr uint32_t total = Raw + QM * kRow;
  static constexpr uint32_t kLboB = (D / 8) * kSbo;            // packed B: K groups dense
  static constexpr uint32_t kTileB = D * TL * 4;
};

// key pass: the contraction W += C^T V runs as kind::f16 MMAs on bf16 operands,
// V exact and C as three bf16 planes c1 + c2 + c3 (24 significant bits): W
// enters W-hat = X_T W, whose unconverged directions amplify a single rounding
// of C (TF32: ~2e-4 in W) about a hundredfold.
// A (C^T planes): 8-landmark row groups 144 bytes apart, 8-token K groups 2304
// bytes apart.  A warp's 8-byte plane stores (its 8 x 4 blocks of 4 landmarks x
// 4 tokens) then fall on 16 distinct 8-byte bank slots, two lanes each.
constexpr uint32_t kSboC = 144;
constexpr uint32_t kLboC = (QM / 8) * kSboC;
constexpr uint32_t kPlaneC = (TL / 8) * kLboC;
template <int D>
struct KSmem {
  static constexpr uint32_t Lt = 0;                            // [D][QM] f32, feature-major landmarks
  static constexpr uint32_t Kt = Lt + D * QM * 4;              // 2 x [D][TL] f32, feature-major keys
  static constexpr uint32_t kLboB = (D / 8) * kSboVB;          // B (V^T, bf16): 8-token K groups
  static constexpr uint32_t kTileB = (TL / 8) * kLboB;
  static constexpr uint32_t Vb = Kt + 2 * D * TL * 4;          // 2 x B tiles (V^T)
  static constexpr uint32_t Ca = Vb + 2 * kTileB;              // 2 x 3 A planes (C^T, bf16)
  static constexpr uint32_t kRow = D * 2 + 16;                 // padded raw row
  static constexpr uint32_t Raw = Ca + 6 * kPlaneC;            // 2 x (64 key rows, 64 value rows)
  static constexpr uint32_t kRawBuf = 2 * TL * kRow;
  static constexpr uint32_t total = Raw + 2 * kRawBuf;
};

__host__ __device__ constexpr uint32_t tmem_cols(int d) { return d < 32 ? 32u : (uint32_t)d; }

// x rounded to the nearest TF32 value, halfway cases away from zero (as
// cvt.rna.tf32.f32): add half a TF32 ulp to the magnitude bits and clear the
// 13 low bits; a carry into the exponent is the correct rounding.  Finite x.
__device__ __forceinline__ float tf32f(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

// bounded wait for a phase of an mbarrier; on expiry the error word is set
__device__ __forceinline__ bool wait_or_flag(int* err, uint32_t bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  if (!ok) atomicOr(err, 1);
  return ok;
}

// 8 bf16 values (16 bytes) -> 8 floats
__device__ __forceinline__ void bf16x8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}
}  // namespace

// ---------------------------------------------------------------------------
// pack: per slice and 64-landmark tile t,
//   LT[bh][t][c][a] = L[bh][64 t + a][c]                 (feature-major, f32)
//   WT[bh][t] = W-hat rows 64 t .. 64 t + 63 as the K-major B operand
//               (row = feature c, k = landmark a), TF32-rounded
// zero past m.  grid (nt, BH).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) k_pack_q(const float* __restrict__ L,
                                                     const float* __restrict__ What,
                                                     float* __restrict__ LT, float* __restrict__ WT,
                                                     int m, int nt) {
  const int t = blockIdx.x, bh = blockIdx.y;
  float* lt = LT + ((size_t)bh * nt + t) * D * TL;
  float* wt = WT + ((size_t)bh * nt + t) * D * TL;
  for (int e = threadIdx.x; e < TL * D; e += kThreads) {
    const int al = e / D, c = e % D, a = t * TL + al;
    const bool ok = a < m;
    const float l = ok ? __ldg(L + ((size_t)bh * m + a) * D + c) : 0.f;
    const float w = ok ? __ldg(What + ((size_t)bh * m + a) * D + c) : 0.f;
    lt[c * TL + al] = l;
    wt[(al >> 2) * (QSmem<D>::kLboB / 4) + (c >> 3) * (kSbo / 4) + (c & 7) * 4 + (al & 3)] = tf32f(w);
  }
}

// ---------------------------------------------------------------------------
// query pass
// ---------------------------------------------------------------------------
struct QArgs {
  const __nv_bfloat16* Q;
  const float* LT;
  const float* WT;
  const float* stats;  // [BH][3][m] (norm)
  __nv_bfloat16* O;
  float* kvout;        // [BH][N][mp] kernel values P, or null
  int* err;
  int N, m, mp, nt, nb, items;
  float ns;
};

template <int D, bool NORM, bool GAUSS>
__global__ void __launch_bounds__(NTH, 1) k_query_tc(QArgs a) {
  using S = QSmem<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[3];   // tile operands landed (bulk copies)
  __shared__ __align__(8) uint64_t mdone[2];  // MMAs reading A buffer b completed
  __shared__ uint32_t tmem_s;
  float* Xt = reinterpret_cast<float*>(sm + S::Xt);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ty = tid >> 4, tx = tid & 15;  // queries 4 ty .. 4 ty + 3, landmarks 4 tx .. 4 tx + 3
  constexpr uint32_t kCols = tmem_cols(D);
  const uint32_t id = tc::idesc_tf32(QM, D);

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(tc::smem_u32(&full[i]), 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&mdone[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  // operands of tile g (item `item`, landmark tile t) into its buffers
  auto issue_tile = [&](uint32_t g, int item, int t) {
    const int bh = item / a.nb;
    const uint32_t bar = tc::smem_u32(&full[g % 3]);
    tc::mbar_expect_tx(bar, 2 * S::kTileB);
    const size_t off = ((size_t)bh * a.nt + t) * D * TL;
    tc::bulk_g2s(tc::smem_u32(sm + S::Lt + (g & 1) * S::kTileB), a.LT + off, S::kTileB, bar);
    tc::bulk_g2s(tc::smem_u32(sm + S::Wt + (g % 3) * S::kTileB), a.WT + off, S::kTileB, bar);
  };
  // raw query rows of an item (zero past N)
  auto prefetch_q = [&](int item) {
    if (item >= a.items) return;
    const int bh = item / a.nb, j0 = (item % a.nb) * QM;
    constexpr int CH = D / 8;  // 16-byte pieces per row
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
  int last_mma = -1;     // last tile whose MMAs were issued
  uint32_t issued = 0;   // tiles whose operand copies were issued (thread 0)
  if (tid == 0 && (int)blockIdx.x < a.items) {
    issue_tile(0, blockIdx.x, 0);
    issued = 1;
  }
  prefetch_q(blockIdx.x);
  for (int item = blockIdx.x; item < a.items; item += gridDim.x) {
    const int bh = item / a.nb, j0 = (item % a.nb) * QM;
    // this thread's pieces of the item's rows landed (each thread converts the
    // pieces it copied); the previous item's distances ended before its last
    // tile's barrier, so the query tile is free
    cp_wait_all();
    {
      // raw rows -> feature-major f32 (lanes take consecutive queries)
      constexpr int CH = D / 8;
      for (int e = tid; e < QM * CH; e += NTH) {
        const int j = e % QM, ch = e / QM;
        float f[8];
        bf16x8(*reinterpret_cast<const uint4*>(sm + S::Raw + j * S::kRow + 16 * ch), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) Xt[(8 * ch + i) * QM + j] = f[i];
      }
    }
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    prefetch_q(item + gridDim.x);

    for (int t = 0; t < a.nt; ++t, ++g) {
      bad |= !wait_or_flag(a.err, tc::smem_u32(&full[g % 3]), (g / 3) & 1);
      if (tid == 0 && !bad) {
        // tile g + 1: its landmark buffer was read by tile g - 1's distances
        // (finished before the last barrier), its W-hat buffer by MMA g - 2
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
      const float* Lt = reinterpret_cast<const float*>(sm + S::Lt + (g & 1) * S::kTileB);
      float acc[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[r][s] = 0.f;
      {
        const float* xp = Xt + 4 * ty;
        const float* lp = Lt + 4 * tx;
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
          const float4 x0 = lds4(xp + c * QM), l = lds4(lp + c * TL);
          const float x[4] = {x0.x, x0.y, x0.z, x0.w};
          if (GAUSS) {
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
              for (int s = 0; s < 4; ++s) acc[r][s] = dist_add<GAUSS>(acc[r][s], x[r] - lv[s]);
          } else {
            const f32x2 la = pack2(l.x, l.y), lb = pack2(l.z, l.w);
#pragma unroll
            for (int r = 0; r < 4; ++r) l1_row4(acc[r], x[r], la, lb);
          }
        }
      }
      // the A buffer of this tile was read by MMA g - 2
      if (g >= 2) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[g & 1]), ((g - 2) >> 1) & 1);
      {
        const int ab = t * TL + 4 * tx;  // first landmark of this thread
        float mu[4], rs[4];
        if (NORM) {
          const float* st = a.stats + (size_t)bh * 3 * a.m;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const bool ok = ab + s < a.m;
            mu[s] = ok ? __ldg(st + ab + s) : 0.f;
            rs[s] = ok ? __ldg(st + 2 * a.m + ab + s) : 0.f;
          }
        }
        uint8_t* pa = sm + S::Pa + (g & 1) * kTileA + tx * kLboA + (ty >> 1) * kSbo + (ty & 1) * 64;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int j = j0 + 4 * ty + r;
          float pv[4], z[4];
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const bool ok = ab + s < a.m;
            pv[s] = ok ? exp2_ftz(acc[r][s] * a.ns) : 0.f;
            z[s] = NORM ? (ok ? (pv[s] - mu[s]) * rs[s] : 0.f) : pv[s];
          }
          // keep the kernel value (before normalisation) for the backward
          if (a.kvout != nullptr && j < a.N)
            st4(a.kvout + ((size_t)bh * a.N + j) * a.mp + ab, make_float4(pv[0], pv[1], pv[2], pv[3]));
          *reinterpret_cast<float4*>(pa + r * 16) =
              make_float4(tf32f(z[0]), tf32f(z[1]), tf32f(z[2]), tf32f(z[3]));
        }
      }
      tc::fence_async_smem();
      tc::fence_before();
      if (__syncthreads_or(bad)) {
        abort = true;
        break;
      }
      if (tid == 0) {
        tc::fence_after();
        const uint32_t pa = tc::smem_u32(sm + S::Pa + (g & 1) * kTileA);
        const uint32_t wb = tc::smem_u32(sm + S::Wt + (g % 3) * S::kTileB);
#pragma unroll
        for (int k8 = 0; k8 < TL / 8; ++k8)
          tc::mma_ss(tmem, tc::desc(pa + k8 * 2 * kLboA, kLboA, kSbo),
                     tc::desc(wb + k8 * 2 * S::kLboB, S::kLboB, kSbo), id,
                     (t > 0 || k8 > 0) ? 1u : 0u);
        tc::commit(tc::smem_u32(&mdone[g & 1]));
      }
      last_mma = (int)g;
    }
    if (abort) break;
    // the item's accumulator: lane quarter w % 4 holds queries 32 (w % 4) .., the
    // four warps w, w + 4, w + 8, w + 12 split the columns
    bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[(g - 1) & 1]), ((g - 1) >> 1) & 1);
    tc::fence_after();
    {
      constexpr int HC = D / 4;
      const int q = warp & 3, h = warp >> 2;
      uint32_t v[HC];
      tc::tmem_ld<HC>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HC), v);
      const int j = j0 + 32 * q + lane;
      if (j < a.N) {
        uint4* o = reinterpret_cast<uint4*>(a.O + ((size_t)bh * a.N + j) * D + h * HC);
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
    // drain what this CTA issued: the last MMAs, and operand tiles not yet waited for
    if (last_mma >= 0)
      wait_or_flag(a.err, tc::smem_u32(&mdone[last_mma & 1]), ((uint32_t)last_mma >> 1) & 1);
    if (tid == 0)
      for (uint32_t gi = g; gi < issued; ++gi)
        wait_or_flag(a.err, tc::smem_u32(&full[gi % 3]), (gi / 3) & 1);
    tc::fence_before();
  }
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// key pass, grid (128-landmark tile, token range, slice)
// ---------------------------------------------------------------------------
struct KArgs {
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const float* L;
  float* part;   // [BH][S][mp][d] partial W
  float* kvout;  // [BH][N][mp] kernel values C, or null
  int* err;
  int N, m, mp, S, nblk;
  float ns;
};

template <int D, bool GAUSS>
__global__ void __launch_bounds__(NTH, 1) k_key_tc(KArgs a) {
  using S = KSmem<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t mdone[2];  // MMAs reading operand buffer b completed
  __shared__ uint32_t tmem_s;
  float* Lt = reinterpret_cast<float*>(sm + S::Lt);
  float* Kt = reinterpret_cast<float*>(sm + S::Kt);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // landmarks 4 ty .. 4 ty + 3, tokens 4 tx .. 4 tx + 3; a warp takes 8 x 4 of these blocks
  // (32 landmarks x 16 tokens), so that each of its kernel-value stores writes
  // four whole 128-byte lines of token rows
  const int ty = 8 * (warp & 3) + (lane & 7), tx = 4 * (warp >> 2) + (lane >> 3);
  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * QM;
  constexpr uint32_t kCols = tmem_cols(D);
  const uint32_t id = tc::idesc_bf16(QM, D);
  const __nv_bfloat16* Kb = a.K + (size_t)bh * a.N * D;
  const __nv_bfloat16* Vb = a.V + (size_t)bh * a.N * D;

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&mdone[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the CTA's landmarks, feature-major (zero past m)
  for (int e = tid; e < QM * D; e += NTH) {
    const int al = e % QM, c = e / QM;
    Lt[c * QM + al] = a0 + al < a.m ? __ldg(a.L + ((size_t)bh * a.m + a0 + al) * D + c) : 0.f;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  const int b0 = (int)((long long)a.nblk * sp / a.S), b1 = (int)((long long)a.nblk * (sp + 1) / a.S);
  constexpr int CH = D / 8;
  constexpr int NV = (TL / 2) * CH;  // value tasks (a token pair, 8 features): threads 0 ..
  constexpr int NK = TL * CH;        // key pieces (a token, 8 features): threads NTH / 2 .., two each
  static_assert(NV <= NTH / 2 && NK / 2 <= NTH / 2, "one value task or key-piece pair per thread");
  // Raw key and value rows of block b into raw buffer rbuf (zero past N), one
  // commit group per block (empty past the range).  Each thread copies the
  // pieces it converts afterwards, so its own wait on its copies is all that
  // the conversion needs: no barrier between the copies and the conversion.
  auto prefetch = [&](int b, int rbuf) {
    if (b < b1) {
      const int n0 = b * TL;
      uint8_t* rb = sm + S::Raw + rbuf * S::kRawBuf;
      if (tid < NTH / 2) {
        if (tid < NV) {
          const int ch = tid % CH, j = 2 * (tid / CH);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const bool ok = n0 + j + u < a.N;
            cp_async16(smem_addr(rb + (TL + j + u) * S::kRow + 16 * ch),
                       Vb + (size_t)(ok ? n0 + j + u : 0) * D + 8 * ch, ok);
          }
        }
      } else if (tid - NTH / 2 < NK / 2) {
        const int kp = tid - NTH / 2, j = 2 * (kp % (TL / 2)), ch = kp / (TL / 2);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const bool ok = n0 + j + u < a.N;
          cp_async16(smem_addr(rb + (j + u) * S::kRow + 16 * ch),
                     Kb + (size_t)(ok ? n0 + j + u : 0) * D + 8 * ch, ok);
        }
      }
    }
    cp_commit();
  };
  // the block in raw buffer rbuf -> keys feature-major f32 (Kt buffer kb; lanes
  // take consecutive tokens) and values the bf16 B operand (V^T buffer kb; row =
  // feature, k = token; a task is a token pair and 8 features)
  auto convert = [&](int rbuf, int kb) {
    const uint8_t* rb = sm + S::Raw + rbuf * S::kRawBuf;
    if (tid < NTH / 2) {
      if (tid < NV) {
        const int ch = tid % CH, j = 2 * (tid / CH);
        const uint4 u0 = *reinterpret_cast<const uint4*>(rb + (TL + j) * S::kRow + 16 * ch);
        const uint4 u1 = *reinterpret_cast<const uint4*>(rb + (TL + j + 1) * S::kRow + 16 * ch);
        const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w}, w1[4] = {u1.x, u1.y, u1.z, u1.w};
        uint8_t* dst = sm + S::Vb + kb * S::kTileB + (j >> 3) * S::kLboB + ch * kSboVB + (j & 7) * 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // features 8 ch + 2 q (low halves) and 8 ch + 2 q + 1 (high halves)
          *reinterpret_cast<uint32_t*>(dst + (2 * q) * 16) = (w0[q] & 0xffffu) | (w1[q] << 16);
          *reinterpret_cast<uint32_t*>(dst + (2 * q + 1) * 16) = (w0[q] >> 16) | (w1[q] & 0xffff0000u);
        }
      }
    } else if (tid - NTH / 2 < NK / 2) {
      // a token pair: one 8-byte store per feature
      const int kp = tid - NTH / 2, j = 2 * (kp % (TL / 2)), ch = kp / (TL / 2);
      float f0[8], f1[8];
      bf16x8(*reinterpret_cast<const uint4*>(rb + j * S::kRow + 16 * ch), f0);
      bf16x8(*reinterpret_cast<const uint4*>(rb + (j + 1) * S::kRow + 16 * ch), f1);
      float* kt = Kt + kb * D * TL + j;
#pragma unroll
      for (int q = 0; q < 8; ++q) *reinterpret_cast<float2*>(kt + (8 * ch + q) * TL) = make_float2(f0[q], f1[q]);
    }
  };
  // One barrier a block: block b + 1's operands are converted at the end of
  // block b, before the barrier that precedes block b's MMAs.
  prefetch(b0, 0);
  prefetch(b0 + 1, 1);
  asm volatile("cp.async.wait_group 1;" ::: "memory");  // this thread's pieces of block b0
  convert(0, 0);
  __syncthreads();
  // An expired wait (bad) stops the CTA before its next MMAs, decided by all
  // threads alike (__syncthreads_or); the MMAs already issued and the copies in
  // flight are waited for (bounded) before the tensor memory is freed.
  bool bad = false, abort = false;
  int i = 0;
  float* pend = nullptr;  // the previous block's kernel values, stored during this block's loop
  int pn0 = 0;
  float pv[4][4];
  for (int b = b0; b < b1; ++b, ++i) {
    const int buf = i & 1;
    prefetch(b + 2, buf);  // raw buffer buf held block b, converted before the last barrier

    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) acc[r][s] = 0.f;
    {
      const float* lp = Lt + 4 * ty;
      const float* xp = Kt + buf * D * TL + 4 * tx;
#pragma unroll
      for (int c16 = 0; c16 < D; c16 += 16) {
        if (pend != nullptr) {
          const int s = c16 >> 4;
          if (pn0 + s < a.N)
            st4(pend + (size_t)s * a.mp, make_float4(pv[0][s], pv[1][s], pv[2][s], pv[3][s]));
        }
#pragma unroll 8
        for (int c = c16; c < c16 + 16; ++c) {
          const float4 l0 = lds4(lp + c * QM), x = lds4(xp + c * TL);
          const float lv[4] = {l0.x, l0.y, l0.z, l0.w};
          if (GAUSS) {
            const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
              for (int s = 0; s < 4; ++s) acc[r][s] = dist_add<GAUSS>(acc[r][s], xv[s] - lv[r]);
          } else {
            // |x_s - l_r| = |l_r - x_s|: the pairs run over the keys
            const f32x2 xa = pack2(x.x, x.y), xb = pack2(x.z, x.w);
#pragma unroll
            for (int r = 0; r < 4; ++r) l1_row4(acc[r], lv[r], xa, xb);
          }
        }
      }
      if (pend != nullptr)  // D < 64: the rest of the previous block's values
#pragma unroll
        for (int s = D / 16; s < 4; ++s)
          if (pn0 + s < a.N)
            st4(pend + (size_t)s * a.mp, make_float4(pv[0][s], pv[1][s], pv[2][s], pv[3][s]));
    }
    {
      const int n0 = b * TL;
      float cv[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const bool ok = (a0 + 4 * ty + r < a.m) && (n0 + 4 * tx + s < a.N);
          cv[r][s] = ok ? exp2_ftz(acc[r][s] * a.ns) : 0.f;
        }
      if (a.kvout != nullptr && a0 + 4 * ty < a.mp) {
        // kept for the backward (token-major rows), stored during the next
        // block's distance loop, one token row every 16 features
        pend = a.kvout + ((size_t)bh * a.N + n0 + 4 * tx) * a.mp + a0 + 4 * ty;
        pn0 = n0 + 4 * tx;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int s = 0; s < 4; ++s) pv[r][s] = cv[r][s];
      }
      // the C^T buffer of this block was read by MMA i - 2
      if (i >= 2) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[buf]), ((i - 2) >> 1) & 1);
      // C^T as three bf16 planes (row = landmark 4 ty + r, k = tokens 4 tx .. 4 tx + 3)
      uint8_t* ca = sm + S::Ca + buf * 3 * kPlaneC + (tx >> 1) * kLboC + (ty >> 1) * kSboC +
                    (ty & 1) * 64 + (tx & 1) * 8;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint32_t pl[3][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[3];  // two tokens at a time
          split3_bf16x2(cv[r][2 * h], cv[r][2 * h + 1], w);
#pragma unroll
          for (int p = 0; p < 3; ++p) pl[p][h] = w[p];
        }
#pragma unroll
        for (int p = 0; p < 3; ++p)
          *reinterpret_cast<uint2*>(ca + p * kPlaneC + r * 16) = make_uint2(pl[p][0], pl[p][1]);
      }
    }
    if (b + 1 < b1) {
      // block b + 1's V^T buffer was read by MMA i - 1
      if (i >= 1) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone[buf ^ 1]), ((i - 1) >> 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this thread's pieces of block b + 1
      convert(buf ^ 1, buf ^ 1);
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
      const uint32_t vbs = tc::smem_u32(sm + S::Vb + buf * S::kTileB);
#pragma unroll
      for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k16 = 0; k16 < TL / 16; ++k16)
          tc::mma_bf16(tmem, tc::desc(ca + p * kPlaneC + k16 * 2 * kLboC, kLboC, kSboC),
                       tc::desc(vbs + k16 * 2 * S::kLboB, S::kLboB, kSboVB), id,
                       (i > 0 || p > 0 || k16 > 0) ? 1u : 0u);
      tc::commit(tc::smem_u32(&mdone[buf]));
    }
  }
  if (pend != nullptr && !abort)
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (pn0 + s < a.N)
        st4(pend + (size_t)s * a.mp, make_float4(pv[0][s], pv[1][s], pv[2][s], pv[3][s]));
  cp_wait_all();  // the next block's rows, when the loop stopped early
  // partial W of this range: lane quarter w % 4 holds landmarks 32 (w % 4) .., the
  // four warps w, w + 4, w + 8, w + 12 split the columns (MMAs of blocks < i)
  if (i > 0) wait_or_flag(a.err, tc::smem_u32(&mdone[(i - 1) & 1]), ((i - 1) >> 1) & 1);
  tc::fence_after();
  if (!abort) {
    constexpr int HC = D / 4;
    const int q = warp & 3, h = warp >> 2;
    uint32_t v[HC];
    tc::tmem_ld<HC>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HC), v);
    const int al = a0 + 32 * q + lane;
    if (al < a.mp) {
      float4* o = reinterpret_cast<float4*>(a.part + (((size_t)bh * a.S + sp) * a.mp + al) * D + h * HC);
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
bool fwd_tc_shape(int d, int m) { return (d == 32 || d == 64) && m > kTile; }
bool fwd_tc_ok(const Prob& p) { return p.dtype == 1 && fwd_tc_shape(p.d, p.m); }

// SMs of the current device (the persistent query pass's grid; the items it
// processes, and so its results, do not depend on it)
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

int key_tc_splits(int BH, int m, int nblk) {
  const int nt = (m + QM - 1) / QM;
  // about six waves of one CTA per SM of a 152-SM part; from the dimensions
  // alone, so the summation order (and the workspace size) does not depend on
  // the device
  int s = (6 * 152 + BH * nt / 2) / (BH * nt);
  if (s < 1) s = 1;
  if (s > nblk) s = nblk;
  return s;
}

// landmark and W-hat tiles; the Gaussian variant's landmark records also carry
// the 64 squared norms of each tile
size_t pack_q_floats(const Prob& p) { return 2 * (size_t)p.BH * p.nt * p.d * TL + (size_t)p.BH * p.nt * TL; }

template <int D>
static cudaError_t pack_q_t(const Prob& p, const float* L, const float* What, float* pack,
                            cudaStream_t st) {
  float* LT = pack;
  float* WT = pack + (size_t)p.BH * p.nt * D * TL;
  return launch("pack_q", k_pack_q<D>, dim3(p.nt, p.BH), dim3(kThreads), 0, st, L, What, LT, WT,
                p.m, p.nt);
}

cudaError_t run_pack_q(const Prob& p, const float* L, const float* What, float* pack,
                       cudaStream_t st) {
  if (p.d == 32) return pack_q_t<32>(p, L, What, pack, st);
  if (p.d == 64) return pack_q_t<64>(p, L, What, pack, st);
  return cudaErrorInvalidValue;
}

template <int D, bool NORM, bool GAUSS>
static cudaError_t query_tc_t(const Prob& p, const void* q, const float* pack, const float* stats,
                              void* out, float* kvout, cudaStream_t st) {
  const size_t smem = QSmem<D>::total;
  static bool once = (allow_smem(k_query_tc<D, NORM, GAUSS>, smem), true);
  (void)once;
  QArgs a;
  a.Q = (const __nv_bfloat16*)q;
  a.LT = pack;
  a.WT = pack + (size_t)p.BH * p.nt * D * TL;
  a.stats = stats;
  a.O = (__nv_bfloat16*)out;
  a.kvout = kvout;
  a.err = wait_error_address();
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.nt = p.nt;
  a.nb = (p.N + QM - 1) / QM;
  a.items = a.nb * p.BH;
  a.ns = p.ns;
  const int grid = a.items < sm_count() ? a.items : sm_count();
  return launch("query_fwd", k_query_tc<D, NORM, GAUSS>, dim3(grid), dim3(NTH), smem, st, a);
}

cudaError_t run_query_tc(const Prob& p, const void* q, const float* pack, const float* stats,
                         void* out, float* kvout, cudaStream_t st) {
#define QTC(DD, NN)                                                                   \
  return p.gauss() ? query_tc_t<DD, NN, true>(p, q, pack, stats, out, kvout, st)     \
                   : query_tc_t<DD, NN, false>(p, q, pack, stats, out, kvout, st)
  if (p.d == 32) {
    if (p.norm()) QTC(32, true);
    QTC(32, false);
  }
  if (p.d == 64) {
    if (p.norm()) QTC(64, true);
    QTC(64, false);
  }
#undef QTC
  return cudaErrorInvalidValue;
}

template <int D, bool GAUSS>
static cudaError_t key_tc_t(const Prob& p, const void* k, const void* v, const float* L, float* part,
                            float* kvout, cudaStream_t st) {
  const size_t smem = KSmem<D>::total;
  static bool once = (allow_smem(k_key_tc<D, GAUSS>, smem), true);
  (void)once;
  KArgs a;
  a.K = (const __nv_bfloat16*)k;
  a.V = (const __nv_bfloat16*)v;
  a.L = L;
  a.part = part;
  a.kvout = kvout;
  a.err = wait_error_address();
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.S = p.Skt; a.nblk = p.nblk;
  a.ns = p.ns;
  const int nt = (p.m + QM - 1) / QM;
  return launch("key_fwd", k_key_tc<D, GAUSS>, dim3(nt, p.Skt, p.BH), dim3(NTH), smem, st, a);
}

cudaError_t run_key_tc(const Prob& p, const void* k, const void* v, const float* L, float* part,
                       float* kvout, cudaStream_t st) {
  if (p.d == 32)
    return p.gauss() ? key_tc_t<32, true>(p, k, v, L, part, kvout, st)
                     : key_tc_t<32, false>(p, k, v, L, part, kvout, st);
  if (p.d == 64)
    return p.gauss() ? key_tc_t<64, true>(p, k, v, L, part, kvout, st)
                     : key_tc_t<64, false>(p, k, v, L, part, kvout, st);
  return cudaErrorInvalidValue;
}

}  // namespace lapnys
