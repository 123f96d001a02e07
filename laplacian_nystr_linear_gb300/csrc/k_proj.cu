// Dense bf16 products of the attention block's projections on the tcgen05
// tensor cores, with the block's layout work fused into the operand loads and
// the epilogues.
//
// "[Paper review] SOFT: Softmax-free Transformer with Linear Complexity",
// Proposed method: the attention is one layer of a pyramid backbone, read as
// the plain multi-head layer [Q | K | V] = X W_qkv + b_qkv (heads of d
// columns), Y = concat_h(O_h) W_o + b_o.  Its six products, with T = B N tokens,
// C the embedding width and HD = H d (sizes M x N x K):
//     forward   [Q|K|V] = X W_qkv (+ b, split to heads)    T x S HD x C
//               Y = concat(O) W_o (+ b)                     T x C x HD
//     backward  dO = dY W_o^T (split to heads)              T x HD x C
//               dW_o = concat(O)^T dY, db_o = 1^T dY        HD x C x T
//               dX = concat(dQ|dK|dV) W_qkv^T               T x C x S HD
//               dW_qkv = X^T concat(dQ|dK|dV), db_qkv       C x S HD x T
//
// D[m][n] = sum_k A(m, k) B(n, k), bf16 operands, fp32 accumulators in tensor
// memory.  Operands come by TMA straight from the tensors the block keeps, in
// whichever orientation they are stored, as tiles in the canonical layouts
// with the 128-byte swizzle (TMA rows of 64 bf16, so every copy request moves
// 128 bytes; the swizzle XORs a row's 16-byte chunk index with the row's index
// mod 8, on both the TMA and the tensor-core side):
//   K-major  (the source row holds k contiguously): a 64-wide K step of R rows
//            is R rows of 128 bytes; the MMA's 16-wide slice starts 32 bytes
//            further per slice; 8-row groups 1024 bytes apart (SBO);
//   MN-major (the source row holds m or n contiguously, k = the row): per 64
//            rows of m or n, 64 k-rows of 128 bytes (8 KB, LBO apart); the
//            MMA's 16-wide slice starts 2 KB further; 8-deep K groups 1024
//            bytes apart (SBO).
// So X^T and dY^T of the weight gradients need no transposed copy, and the
// per-head tensors [B][H][N][d] (d = 64 or 128: a head row holds whole 64-wide
// pieces) are read and written in place: the concatenation of heads is never
// materialised.  Tiles of token rows stay inside one batch entry (rows past N
// read as zeros and are not stored).
//
// Epilogues: + bias, round to bf16 and scatter to the per-head tensors (Q|K|V,
// dO); + bias and round to bf16 rows (Y, dX); or fp32 rows (partial tiles of a
// reduction over tokens split into contiguous ranges for the weight gradients,
// which k_gemm_reduce adds in a fixed order and rounds).  The bias gradients are
// the same reduction with a row of ones: one extra M tile whose A operand is a
// constant all-ones tile in shared memory (its first row is kept).
//
// Persistent kernel, one CTA per SM, 192 threads:
//   warp 0     one lane copies each 64-wide K step (A 16 KB + B 32 KB) into a
//              4-stage ring;
//   warp 1     allocates two 256-column accumulators; one lane issues the four
//              M = 128, N = 256, K = 16 MMAs of each K step;
//   warps 2-5  read an item's accumulator (tcgen05.ld, lane quarter = warp % 4,
//              one row per thread) and store it while the next item
//              accumulates in the other one; the item's bias slice is staged
//              in shared memory once.
// Every wait is bounded; after an expired wait a role stops issuing work, the
// error word is set, and the CTA drains what it issued before freeing tensor
// memory.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int BM = 128, BN = 256, BK = 64;
constexpr int NST = 4;
constexpr int NTH = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;     // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;     // 32 KB
constexpr uint32_t STAGE = A_BYTES + B_BYTES;
constexpr uint32_t ONES = NST * STAGE;        // the all-ones A tile
constexpr uint32_t SMEM = ONES + A_BYTES + 1024;  // + alignment slack: 209 KB
constexpr uint32_t BLK64 = 64 * BK * 2;       // one 64-row MN-major block: 8 KB
constexpr uint32_t SW_SBO = 1024;             // 8 rows of 128 bytes
constexpr uint64_t SW128 = 2;                 // descriptor layout type: 128-byte swizzle

__device__ __forceinline__ bool wait_or_flag(int* err, uint32_t bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  if (!ok) atomicOr(err, 1);
  return ok;
}

__device__ __forceinline__ void tma2(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                     uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                     uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma4(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                     int c3, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(mbar)
      : "memory");
}

// shared-memory descriptor of a 128-byte-swizzled tile
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo) {
  return tc::desc(saddr, lbo, SW_SBO) | (SW128 << 61);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// barrier of the 128 epilogue threads (named barrier 1) that also ORs a flag
// over them, so that they all take the same branch after it
__device__ __forceinline__ bool epi_sync_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, 1, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
}  // namespace

struct GemmMaps {
  CUtensorMap a[3], b[3];
};

struct GemmArgs {
  int akind, bkind, epi;
  int wgrad;            // 1: M = features, K = tokens (split reduction); 0: M = tokens
  int B, N, H, d, HD;   // token and head geometry
  int dshift;           // log2(d) (per-head operands)
  int Mf;               // wgrad: feature rows of A (without the ones tile)
  int Nn;               // columns of the product
  int tpb;              // row tiles per batch entry (wgrad 0)
  int mt, nt;           // tiles along M (wgrad: with the ones tile) and N
  int kst;              // K steps (wgrad: over all tokens, per batch entry ceil(N / 64))
  int kpb;              // K steps per batch entry (wgrad)
  int splits;           // contiguous K ranges (wgrad)
  int ones;             // wgrad: M tile of the all-ones rows, or -1
  long long items;
  void* out[3];         // GEP_HEADS: per block s; GEP_ROWS: [B N][ldo]; GEP_F32: [splits][Mrows][Nn]
  const __nv_bfloat16* bias;
  int ldo, Mrows;
  int* err;
};

struct Item {
  int b, t0, m0, n0, ks0, ks1, sp, mtile;
};

__device__ __forceinline__ Item decode(const GemmArgs& a, long long it) {
  Item r;
  if (!a.wgrad) {
    const int nt = (int)(it % a.nt);
    const long long q = it / a.nt;
    r.b = (int)(q / a.tpb);
    r.t0 = (int)(q % a.tpb) * BM;
    r.m0 = 0;
    r.n0 = nt * BN;
    r.ks0 = 0;
    r.ks1 = a.kst;
    r.sp = 0;
    r.mtile = 0;
  } else {
    r.mtile = (int)(it % a.mt);
    const long long q = it / a.mt;
    const int nt = (int)(q % a.nt);
    r.sp = (int)(q / a.nt);
    r.m0 = r.mtile * BM;
    r.n0 = nt * BN;
    r.ks0 = (int)((long long)a.kst * r.sp / a.splits);
    r.ks1 = (int)((long long)a.kst * (r.sp + 1) / a.splits);
    r.b = 0;
    r.t0 = 0;
  }
  return r;
}

// the copies of one operand's tile for one K step into dst; returns its bytes.
// rows0: first row (m or n) of the tile, R: rows; (kb, kt): batch entry and
// first token of the step (wgrad), k0: first feature (otherwise); rt: first
// token row of the tile (otherwise)
template <bool ISSUE>
__device__ __forceinline__ uint32_t load_operand(const CUtensorMap* maps, int kind, uint32_t dst,
                                                 int R, int rows0, int lim, const GemmArgs& a,
                                                 int b, int rt, int k0, int kb, int kt,
                                                 uint32_t bar) {
  switch (kind) {
    case GOP_ROWS_K:  // [B][N][F]: {F, N, B}, box {64, R, 1}
      if (ISSUE) tma3(dst, &maps[0], k0, rt, b, bar);
      return (uint32_t)R * 128;
    case GOP_HEADS_K: {  // [B][H][N][d]: {d, N, H, B}, box {64, R, 1, 1}
      const int s = k0 / a.HD, q = k0 - s * a.HD;
      if (ISSUE) tma4(dst, &maps[s], q & (a.d - 1), rt, q >> a.dshift, b, bar);
      return (uint32_t)R * 128;
    }
    case GOP_W_K:  // [n][k]: {Kf, Nw}, box {64, R}
      if (ISSUE) tma2(dst, &maps[0], k0, rows0, bar);
      return (uint32_t)R * 128;
    case GOP_W_MN:  // [k][n]: {Nw, Kf}, box {64, 64} per 64 rows
      if (ISSUE)
        for (int i = 0; i < R / 64; ++i) tma2(dst + i * BLK64, &maps[0], rows0 + 64 * i, k0, bar);
      return (uint32_t)R * 128;
    case GOP_TOK_MN:  // [B][N][F]: {F, N, B}, box {64, 64, 1} per 64 rows
      if (ISSUE)
        for (int i = 0; i < R / 64; ++i) tma3(dst + i * BLK64, &maps[0], rows0 + 64 * i, kt, kb, bar);
      return (uint32_t)R * 128;
    default: {  // GOP_HEADS_MN: [B][H][N][d]: {d, N, H, B}, box {64, 64, 1, 1} per 64 rows
      uint32_t bytes = 0;
      for (int i = 0; i < R / 64; ++i) {
        const int f = rows0 + 64 * i;
        if (f >= lim) break;
        const int s = f / a.HD, q = f - s * a.HD;
        if (ISSUE) tma4(dst + i * BLK64, &maps[s], q & (a.d - 1), kt, q >> a.dshift, kb, bar);
        bytes += BLK64;
      }
      return bytes;
    }
  }
}

__global__ void __launch_bounds__(NTH, 1) k_gemm_bf16(const __grid_constant__ GemmMaps mp,
                                                       GemmArgs a) {
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[NST];   // a stage's copies landed
  __shared__ __align__(8) uint64_t empty[NST];  // a stage's MMAs done (stage free)
  __shared__ __align__(8) uint64_t accf[2];     // an accumulator's MMAs done
  __shared__ __align__(8) uint64_t acce[2];     // an accumulator read out (128 arrivals)
  __shared__ uint32_t tmem_s;
  __shared__ int issued_s, consumed_s, bad_s;   // for the drain after an expired wait
  __shared__ float bias_s[2][BN];               // an item's bias slice (by accumulator)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool amn = a.akind >= GOP_TOK_MN, bmn = a.bkind >= GOP_TOK_MN;
  // 1024-byte aligned base of the tiles (the swizzle atoms)
  const uint32_t raw_u32 = tc::smem_u32(sm_raw);
  uint8_t* sm = sm_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);

  if (warp == 1) tc::tmem_alloc(&tmem_s, 512);
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(tc::smem_u32(&full[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(&accf[i]), 1);
      tc::mbar_init(tc::smem_u32(&acce[i]), 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    issued_s = 0;
    consumed_s = 0;
    bad_s = 0;
  }
  if (a.ones >= 0) {
    // all-ones A tile (bf16 1.0 = 0x3F80): every layout reads it as ones
    for (int e = tid; e < (int)(A_BYTES / 16); e += NTH)
      reinterpret_cast<uint4*>(sm + ONES)[e] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    tc::fence_async_smem();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int st = 0, issued = 0;
      uint32_t ph = 0;
      bool bad = false;
      for (long long it = blockIdx.x; it < a.items && !bad; it += gridDim.x) {
        const Item r = decode(a, it);
        const bool ones = a.wgrad && r.mtile == a.ones;
        for (int ks = r.ks0; ks < r.ks1; ++ks) {
          if (!wait_or_flag(a.err, tc::smem_u32(&empty[st]), ph ^ 1u)) { bad = true; break; }
          const uint32_t bar = tc::smem_u32(&full[st]);
          const uint32_t sa = tc::smem_u32(sm + st * STAGE), sb = sa + A_BYTES;
          const int kb = a.wgrad ? ks / a.kpb : 0;
          const int kt = a.wgrad ? (ks - kb * a.kpb) * BK : 0;
          const int k0 = ks * BK;
          uint32_t bytes = load_operand<false>(mp.b, a.bkind, sb, BN, r.n0, a.Nn, a, r.b, r.t0, k0,
                                               kb, kt, bar);
          if (!ones)
            bytes += load_operand<false>(mp.a, a.akind, sa, BM, r.m0, a.Mf, a, r.b, r.t0, k0, kb,
                                         kt, bar);
          tc::mbar_expect_tx(bar, bytes);
          if (!ones)
            load_operand<true>(mp.a, a.akind, sa, BM, r.m0, a.Mf, a, r.b, r.t0, k0, kb, kt, bar);
          load_operand<true>(mp.b, a.bkind, sb, BN, r.n0, a.Nn, a, r.b, r.t0, k0, kb, kt, bar);
          ++issued;
          if (++st == NST) { st = 0; ph ^= 1u; }
        }
      }
      issued_s = issued;
      if (bad) atomicOr(&bad_s, 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      int st = 0, consumed = 0;
      uint32_t ph = 0;
      long long li = 0;
      bool bad = false;
      const uint32_t id = tc::idesc_bf16(BM, BN) | (amn ? (1u << 15) : 0u) | (bmn ? (1u << 16) : 0u);
      // LBO: K-major swizzled tiles do not use it (16); MN-major: 64-row blocks
      const uint32_t lbo_a = amn ? BLK64 : 16, lbo_b = bmn ? BLK64 : 16;
      // bytes per 16-wide K slice
      const uint32_t kstep_a = amn ? 16 * 128 : 32, kstep_b = bmn ? 16 * 128 : 32;
      for (long long it = blockIdx.x; it < a.items && !bad; it += gridDim.x, ++li) {
        const Item r = decode(a, it);
        const bool ones = a.wgrad && r.mtile == a.ones;
        const int acc = (int)(li & 1);
        if (!wait_or_flag(a.err, tc::smem_u32(&acce[acc]), (uint32_t)((li >> 1) & 1) ^ 1u)) {
          bad = true;
          break;
        }
        tc::fence_after();
        const uint32_t dt = tmem + (uint32_t)(acc * BN);
        for (int ks = r.ks0; ks < r.ks1; ++ks) {
          if (!wait_or_flag(a.err, tc::smem_u32(&full[st]), ph)) { bad = true; break; }
          tc::fence_after();
          const uint32_t sb = tc::smem_u32(sm + st * STAGE) + A_BYTES;
          const uint32_t sa = ones ? tc::smem_u32(sm + ONES) : tc::smem_u32(sm + st * STAGE);
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16)
            tc::mma_bf16(dt, sdesc(sa + k16 * kstep_a, lbo_a), sdesc(sb + k16 * kstep_b, lbo_b), id,
                         (ks > r.ks0 || k16 > 0) ? 1u : 0u);
          tc::commit(tc::smem_u32(&empty[st]));
          ++consumed;
          if (++st == NST) { st = 0; ph ^= 1u; }
        }
        if (bad) break;
        tc::commit(tc::smem_u32(&accf[acc]));
      }
      consumed_s = consumed;
      if (bad) atomicOr(&bad_s, 1);
    }
  } else {
    // ---------------- epilogue ----------------
    const int et = tid - 64;                      // 0 .. 127
    const int q = warp & 3;                       // TMEM lane quarter
    const int row = 32 * q + lane;                // row of the tile
    long long li = 0;
    bool bad = false;
    for (long long it = blockIdx.x; it < a.items; it += gridDim.x, ++li) {
      const Item r = decode(a, it);
      const int acc = (int)(li & 1);
      // the item's bias slice, while its products finish
      if (a.bias != nullptr)
        for (int j = et; j < BN; j += 128) {
          const int n = r.n0 + j;
          bias_s[acc][j] = n < a.Nn ? __bfloat162float(a.bias[n]) : 0.f;
        }
      bad = !wait_or_flag(a.err, tc::smem_u32(&accf[acc]), (uint32_t)(li >> 1) & 1u);
      if (epi_sync_any(bad)) {      // also publishes bias_s to the four warps
        bad = true;
        break;
      }
      tc::fence_after();
      bool keep;
      size_t rowoff;
      int t = 0;
      if (!a.wgrad) {
        t = r.t0 + row;
        keep = t < a.N;
        rowoff = (size_t)r.b * a.N + t;
      } else if (r.mtile == a.ones) {
        keep = row == 0;
        rowoff = (size_t)a.Mf;
      } else {
        keep = r.m0 + row < a.Mf;
        rowoff = (size_t)(r.m0 + row);
      }
      const int ncols = min(BN, a.Nn - r.n0);
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        if (32 * ch >= ncols) break;              // uniform over the warp
        uint32_t v[32];
        tc::tmem_ld<32>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + 32 * ch), v);
        if (!keep) continue;
        const int n = r.n0 + 32 * ch;
        if (a.epi == GEP_F32) {
          float* o = reinterpret_cast<float*>(a.out[0]) + ((size_t)r.sp * a.Mrows + rowoff) * a.Nn + n;
#pragma unroll
          for (int p = 0; p < 8; ++p)
            if (n + 4 * p < a.Nn)
              reinterpret_cast<float4*>(o)[p] =
                  make_float4(__uint_as_float(v[4 * p]), __uint_as_float(v[4 * p + 1]),
                              __uint_as_float(v[4 * p + 2]), __uint_as_float(v[4 * p + 3]));
          continue;
        }
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
        if (a.bias != nullptr)
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] += bias_s[acc][32 * ch + i];
        __nv_bfloat16* dst;
        if (a.epi == GEP_ROWS) {
          dst = reinterpret_cast<__nv_bfloat16*>(a.out[0]) + rowoff * a.ldo + n;
        } else {
          // 32 columns inside one head (d = 64 or 128)
          const int s = n / a.HD, hq = n - s * a.HD;
          void* os = s == 0 ? a.out[0] : (s == 1 ? a.out[1] : a.out[2]);
          dst = reinterpret_cast<__nv_bfloat16*>(os) +
                (((size_t)r.b * a.H + (hq >> a.dshift)) * a.N + t) * a.d + (hq & (a.d - 1));
        }
#pragma unroll
        for (int p = 0; p < 4; ++p)
          if (n + 8 * p < a.Nn)
            reinterpret_cast<uint4*>(dst)[p] =
                make_uint4(pack_bf16(f[8 * p], f[8 * p + 1]), pack_bf16(f[8 * p + 2], f[8 * p + 3]),
                           pack_bf16(f[8 * p + 4], f[8 * p + 5]), pack_bf16(f[8 * p + 6], f[8 * p + 7]));
      }
      tc::fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&acce[acc])) : "memory");
    }
    if (bad) atomicOr(&bad_s, 1);
  }

  // ---- drain and free the tensor memory ----
  // On a healthy run the epilogue waited for the last MMAs and the MMAs for
  // every copy.  After an expired wait: the last MMA commit (it covers every
  // earlier MMA of the issuing thread), then every copy issued but not consumed.
  __syncthreads();
  if (bad_s && warp == 1 && lane == 0) {
    const int c = consumed_s, n = issued_s;
    if (c > 0) wait_or_flag(a.err, tc::smem_u32(&empty[(c - 1) % NST]), (uint32_t)((c - 1) / NST) & 1u);
    for (int k = c; k < n; ++k)
      wait_or_flag(a.err, tc::smem_u32(&full[k % NST]), (uint32_t)(k / NST) & 1u);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// out[m][n] = sum over splits of part[sp][m][n] (fixed order), rounded to bf16;
// row Mf of the partials (the ones tile) goes to db when db is not null
__global__ void k_gemm_reduce(const float* part, int splits, int Mf, int Mrows, int Nn,
                              __nv_bfloat16* out, __nv_bfloat16* db) {
  const long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  const long long rows = db != nullptr ? Mf + 1 : Mf;
  if (e >= rows * Nn) return;
  const int m = (int)(e / Nn), n = (int)(e % Nn);
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < splits; ++sp) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(part + ((size_t)sp * Mrows + m) * Nn + n));
    s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
  }
  __nv_bfloat16* o = m < Mf ? out + (size_t)m * Nn + n : db + n;
  *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16(s.x, s.y), pack_bf16(s.z, s.w));
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
constexpr int kSmTarget = 152;  // split counts follow from the dimensions alone

bool map_tok(CUtensorMap* t, const void* p, int B, int N, int F, int box_rows) {
  const cuuint64_t dim[3] = {(cuuint64_t)F, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t stride[2] = {(cuuint64_t)F * 2, (cuuint64_t)N * F * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  return encode_tiled_bf16_sw128(t, 3, p, dim, stride, box);
}
bool map_heads(CUtensorMap* t, const void* p, int B, int H, int N, int d, int box_rows) {
  const cuuint64_t dim[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t stride[3] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2, (cuuint64_t)H * N * d * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  return encode_tiled_bf16_sw128(t, 4, p, dim, stride, box);
}
// weight [rows][cols] row-major, boxes of 64 columns x box_rows rows
bool map_w(CUtensorMap* t, const void* p, int rows, int cols, int box_rows) {
  const cuuint64_t dim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  return encode_tiled_bf16_sw128(t, 2, p, dim, stride, box);
}

int log2i(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return s;
}

GemmArgs base_args(const GemmDims& g) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.B = g.B; a.N = g.N; a.H = g.H; a.d = g.d; a.HD = g.H * g.d;
  a.dshift = log2i(g.d);
  a.ones = -1;
  return a;
}

// product over token rows: M = tokens (tiles inside one batch entry), K = Kf features
void rows_shape(GemmArgs& a, const GemmDims& g, int Nn, int Kf) {
  a.wgrad = 0;
  a.Nn = Nn;
  a.tpb = (g.N + BM - 1) / BM;
  a.nt = (Nn + BN - 1) / BN;
  a.mt = g.B * a.tpb;
  a.kst = (Kf + BK - 1) / BK;
  a.items = (long long)a.mt * a.nt;
}

// weight-gradient product: M = Mf features (+ a ones tile), N = Nn, K = all tokens
void wgrad_shape(GemmArgs& a, const GemmDims& g, int Mf, int Nn, bool ones) {
  a.wgrad = 1;
  a.Mf = Mf;
  a.Nn = Nn;
  a.mt = (Mf + BM - 1) / BM + (ones ? 1 : 0);
  a.ones = ones ? a.mt - 1 : -1;
  a.nt = (Nn + BN - 1) / BN;
  a.kpb = (g.N + BK - 1) / BK;
  a.kst = g.B * a.kpb;
  const int tiles = a.mt * a.nt;
  int s = (4 * kSmTarget + tiles / 2) / tiles;
  a.splits = s < 1 ? 1 : (s > a.kst ? a.kst : s);
  a.items = (long long)tiles * a.splits;
  a.Mrows = Mf + (ones ? 1 : 0);
}

cudaError_t go(const char* name, const GemmMaps& mp, GemmArgs& a, cudaStream_t st) {
  static bool once = (allow_smem(k_gemm_bf16, SMEM), true);
  (void)once;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidSymbol;
  if (a.items <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = (int)(a.items < sms ? a.items : sms);
  return launch(name, k_gemm_bf16, dim3(grid), dim3(NTH), (size_t)SMEM, st, mp, a);
}

cudaError_t reduce(const char* name, const GemmArgs& a, const float* part, void* out, void* db,
                   cudaStream_t st) {
  const long long n4 = (long long)(db != nullptr ? a.Mf + 1 : a.Mf) * a.Nn / 4;
  const int th = 256;
  return launch(name, k_gemm_reduce, dim3((unsigned)((n4 + th - 1) / th)), dim3(th), 0, st, part,
                a.splits, a.Mf, a.Mrows, a.Nn, (__nv_bfloat16*)out, (__nv_bfloat16*)db);
}
}  // namespace

bool gemm_bf16_ok(const GemmDims& g) {
  const long long HD = (long long)g.H * g.d;
  return tensor_map_encoder() != nullptr && g.C % 8 == 0 && HD % 8 == 0 && g.B > 0 && g.N > 0;
}

bool gemm_heads_ok(const GemmDims& g) {
  return gemm_bf16_ok(g) && (g.d == 64 || g.d == 128);
}

size_t gemm_wgrad_floats(const GemmDims& g) {
  size_t mx = 0;
  const int HD = g.H * g.d;
  const int shapes[2][2] = {{HD, g.C}, {g.C, g.S * HD}};
  for (const auto& s : shapes)
    for (int ones = 0; ones < 2; ++ones) {
      GemmArgs a = base_args(g);
      wgrad_shape(a, g, s[0], s[1], ones != 0);
      const size_t f = (size_t)a.splits * a.Mrows * a.Nn;
      if (f > mx) mx = f;
    }
  return mx;
}

cudaError_t run_gemm_rows(const char* name, const GemmDims& g, int src_kind,
                          const void* const* src, int Kf, int w_kind, const void* w, int Nn,
                          int epi, void* const* out, const void* bias, cudaStream_t st) {
  GemmMaps mp;
  memset(&mp, 0, sizeof(mp));
  GemmArgs a = base_args(g);
  rows_shape(a, g, Nn, Kf);
  a.akind = src_kind;
  a.bkind = w_kind;
  a.epi = epi;
  bool ok = true;
  if (src_kind == GOP_ROWS_K) {
    ok = map_tok(&mp.a[0], src[0], g.B, g.N, Kf, BM);
  } else {
    for (int s = 0; s < Kf / (g.H * g.d); ++s)
      ok = ok && map_heads(&mp.a[s], src[s], g.B, g.H, g.N, g.d, BM);
  }
  // K-major weight [Nn][Kf]: boxes of 64 k x 256 rows; MN-major [Kf][Nn]: 64 n x 64 k
  ok = ok && (w_kind == GOP_W_K ? map_w(&mp.b[0], w, Nn, Kf, BN) : map_w(&mp.b[0], w, Kf, Nn, BK));
  if (!ok) return cudaErrorInvalidValue;
  for (int s = 0; s < 3; ++s) a.out[s] = out[s];
  a.bias = (const __nv_bfloat16*)bias;
  a.ldo = Nn;
  return go(name, mp, a, st);
}

cudaError_t run_gemm_wgrad(const char* name, const GemmDims& g, int a_kind,
                           const void* const* asrc, int Mf, int b_kind, const void* const* bsrc,
                           int Nn, float* part, void* dw, void* db, cudaStream_t st) {
  GemmMaps mp;
  memset(&mp, 0, sizeof(mp));
  GemmArgs a = base_args(g);
  wgrad_shape(a, g, Mf, Nn, db != nullptr);
  a.akind = a_kind;
  a.bkind = b_kind;
  a.epi = GEP_F32;
  const int HD = g.H * g.d;
  bool ok = true;
  // MN-major: boxes of 64 features x 64 tokens
  if (a_kind == GOP_TOK_MN) {
    ok = map_tok(&mp.a[0], asrc[0], g.B, g.N, Mf, BK);
  } else {
    for (int s = 0; s < Mf / HD; ++s) ok = ok && map_heads(&mp.a[s], asrc[s], g.B, g.H, g.N, g.d, BK);
  }
  if (b_kind == GOP_TOK_MN) {
    ok = ok && map_tok(&mp.b[0], bsrc[0], g.B, g.N, Nn, BK);
  } else {
    for (int s = 0; s < Nn / HD; ++s) ok = ok && map_heads(&mp.b[s], bsrc[s], g.B, g.H, g.N, g.d, BK);
  }
  if (!ok) return cudaErrorInvalidValue;
  a.out[0] = part;
  cudaError_t e = go(name, mp, a, st);
  if (e != cudaSuccess) return e;
  return reduce("block_gemm_reduce", a, part, dw, db, st);
}

}  // namespace lapnys
