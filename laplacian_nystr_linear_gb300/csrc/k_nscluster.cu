// The whole Newton-Schulz iteration of one slice in one thread-block cluster,
// for 64 < m <= 256, on the 5th-generation tensor cores.
//
// Forward ("SOFT" review, Proposed method: A_{k+1} = 2 A_k - A_k A A_k, here
// X_{t+1} = 2 X_t - X_t (A X_t)):
//     Y_t = A X_t,   X_{t+1} = -X_t Y_t + 2 X_t,            t = 0 .. T-1
// Reverse of those products, t = T-1 .. 0, with G = dLoss/dX_{t+1} on entry:
//     XG = X_t^T G,  dA = -XG X_t^T + dA,  Tm = -G Y_t^T + 2 G,  G = -A^T XG + Tm
// (dA starts at zero; G leaves as dLoss/dX_0).
//
// Each product is fp32-accurate: operands are split x = hi + lo (hi = x
// rounded to TF32, lo = x - hi) and accumulated in fp32 as hi*hi + hi*lo +
// lo*hi (kind::tf32 MMAs, accumulator in TMEM).
//
// A cluster of ceil(m / 128) CTAs owns a slice; CTA r computes rows
// [128 r, 128 r + 128) of every product, all m (rounded up to 16) columns in
// one M = 128, N <= 256 MMA accumulator.  Products depend on each other's full
// results, so a cluster barrier (release / acquire) separates consecutive
// products.  Twelve warps (three per SM sub-partition, so each may hold up to
// 168 registers):
//   warp 9, one lane  copies each K-stage (16) of both operands into a 4-stage
//           raw ring in shared memory with TMA (cp.async.bulk.tensor).  An
//           operand whose rows hold K contiguously goes through a 3-D tensor
//           map {k, rows, matrix} in boxes of 16 k (one 64-byte row per copy
//           request, 64-byte swizzle so that the splitters' row-wise reads are
//           free of bank conflicts); one stored [k][row] through a 3-D map
//           {row, k, matrix}.
//   warps 0-7  per stage: split op(A) (lane = row 32 (w % 4) + lane, k-step
//           w / 4) into TF32 hi / lo and write them into TMEM (tcgen05.st),
//           where the MMA reads op(A); split op(B) and store hi / lo into a
//           3-stage ring in the K-major core-matrix layout (8 rows x 16 bytes
//           per core matrix; 8-row groups 144 bytes apart and K groups 32 bytes
//           further apart than dense, which keeps the split stores free of bank
//           conflicts).  Their share of the work is shared-memory reads, the
//           split and the stores: no address arithmetic or copy issue for
//           global memory.
//   warp 8  allocates TMEM (accumulator: columns 0-255; op(A) stages: 32
//           columns each from 256); its first lane issues each stage's six MMAs
//           (2 k-steps x 3 split products, A from TMEM, B from shared memory),
//           commits them to the stage's "free" mbarrier and, after a product's
//           last stage, to the accumulator barrier.
//   all twelve warps then read the accumulator back with tcgen05.ld (warp w
//           reads TMEM lanes 32 (w % 4) .., three warps per lane quarter, each
//           taking every third 32-column piece), transpose 32 x 32 pieces
//           through a small per-warp buffer (in split stages 0-1, idle between
//           a product's last MMA and the next cluster barrier) and write
//           C = alpha acc + beta E in whole lines; E is fetched two pieces
//           ahead.  The stores are made visible to the next product's TMA reads
//           (async proxy) before the cluster barrier.
//
// Every mbarrier wait is bounded: on expiry the CTA records an error in the
// device word read by lapnys_device_status and stops working, but still takes
// part in every cluster barrier, so that the other CTA of its cluster finishes;
// copies it issued are waited for (bounded) before it exits.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace lapnys {

namespace {
constexpr int TM = 128;    // rows per CTA (MMA M)
constexpr int TNMAX = 256; // largest MMA N
constexpr int TK = 16;     // K per stage
constexpr int NSPL = 3;    // split (hi / lo) stages of op(B)
constexpr int NRAW = 4;    // raw (TMA) stages of both operands
constexpr int NSPW = 8;    // splitter warps
constexpr int NSPT = NSPW * 32;
constexpr int NEPW = 4;    // epilogue-only warps (8-11)
constexpr int NTH = NSPT + NEPW * 32;  // 384
constexpr int kMmaWarp = NSPW;         // warp 8
constexpr int kTmaWarp = NSPW + 1;     // warp 9
constexpr uint32_t kSbo = 144;                       // bytes between 8-row groups
constexpr uint32_t kLboB = (TNMAX / 8) * kSbo + 32;  // bytes between 4-wide K groups, B tile
constexpr uint32_t kTileB = (TK / 4) * kLboB;        // B hi (or lo) per stage
constexpr uint32_t kStage = 2 * kTileB;              // B hi, B lo
constexpr uint32_t kAcol = TNMAX;                    // first TMEM column of the op(A) stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRawA = TM * TK * 4;              // raw op(A) box (bytes)
constexpr uint32_t kRawB = TNMAX * TK * 4;           // raw op(B) box
constexpr uint32_t kRawStage = kRawA + kRawB;
constexpr uint32_t kEpiPitch = 36 * 4;               // staged row: 32 floats + 16-byte pad
constexpr uint32_t kEpiWarp = 32 * kEpiPitch;
static_assert(NTH / 32 * kEpiWarp <= 2 * kStage, "epilogue staging fits in two split stages");
static_assert(kAcol + NSPL * 32 <= kTmemCols, "op(A) stages fit in TMEM");
// the raw ring starts 1024-byte aligned (the 64-byte swizzle of its K-contiguous
// boxes is a function of the shared-memory address bits)
constexpr size_t kRawOff = ((size_t)NSPL * kStage + 1023) / 1024 * 1024;
constexpr size_t kSmem = kRawOff + (size_t)NRAW * kRawStage + 1024;
constexpr int kWaitLimit = 1 << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// instruction descriptor: D f32, A/B tf32, both K-major, N, M = 128
__device__ __forceinline__ uint32_t idesc(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
}

// shared-memory matrix descriptor, K-major without swizzle
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((kSbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for this architecture
  return d;
}

// byte offset of the 16-byte piece (row, k4) of a K-major tile
__device__ __forceinline__ uint32_t kmaj_off(int row, int k4, uint32_t lbo) {
  return (uint32_t)k4 * lbo + (uint32_t)(row >> 3) * kSbo + (uint32_t)(row & 7) * 16u;
}

// x rounded to the nearest TF32 value (10 mantissa bits, halfway cases away
// from zero) by integer arithmetic on the bits: add half a TF32 ulp to the
// magnitude and clear the 13 low bits (a carry into the exponent is the
// correct rounding).  Finite inputs only, which the iteration's are.
__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

__device__ __forceinline__ void store_split(uint8_t* hi, uint8_t* lo, uint32_t off, float4 x) {
  float4 h, l;
  h.x = tf32_hi(x.x); l.x = x.x - h.x;
  h.y = tf32_hi(x.y); l.y = x.y - h.y;
  h.z = tf32_hi(x.z); l.z = x.z - h.z;
  h.w = tf32_hi(x.w); l.w = x.w - h.w;
  *reinterpret_cast<float4*>(hi + off) = h;
  *reinterpret_cast<float4*>(lo + off) = l;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  for (int i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}
// D (TMEM) += A (TMEM, lane = row) * B (shared-memory descriptor)
__device__ __forceinline__ void mma_tf32_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                            uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(id), "r"(accumulate)
      : "memory");
}
// this lane's 8 consecutive TMEM columns at taddr (warp-collective)
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ float4 ldcg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}
}  // namespace

// Tensor maps of every operand use in the programs (encoded on the host per
// launch).  A-role maps have 128-row boxes, B-role maps 256-row boxes; "kc":
// rows hold K contiguously (swizzled 64-byte rows), "mn": stored [k][row].  The
// last dimension enumerates the m x m matrices of the buffer.
struct NsMaps {
  CUtensorMap a_kc, a_mn;          // landmark matrix A [BH]: A X (fwd), A^T XG (rev)
  CUtensorMap x_akc, x_amn;        // iterates X [BH * nx]: X Y (fwd), X^T G (rev)
  CUtensorMap x_bmn, x_bkc;        //   as B: A X (fwd), XG X^T (rev)
  CUtensorMap y_bmn, y_bkc;        // products Y [BH * ny]: X Y (fwd), G Y^T (rev)
  CUtensorMap g_akc, g_bmn;        // G [BH]: G Y^T, X^T G (rev)
  CUtensorMap xg_akc, xg_bmn;      // XG [BH]: XG X^T, A^T XG (rev)
};

struct NsArgs {
  float* X;        // [BH][nx][m][m]: iterate t in slot t % nx
  float* Y;        // [BH][ny][m][m]: A X_t in slot t % ny
  float* G;        // reverse only: [BH][m][m]
  float* XG;       // reverse only: [BH][m][m]
  float* Tm;       // reverse only: [BH][m][m]
  float* dA;       // reverse only: [BH][m][m]
  int* err;        // device error word (set when a bounded wait expires)
  int m, iters, nx, ny, reverse;
};

namespace {
// one product of the program: C = alpha op(A) op(B) + beta E (slice-local)
struct Prod {
  const CUtensorMap* ma;  // op(A) rows: map and matrix index
  int za;
  bool ka;                // rows of op(A) hold K contiguously
  const CUtensorMap* mb;  // op(B)^T rows (result columns)
  int zb;
  bool kb;
  float* C;
  const float* E;         // null when beta == 0
  float alpha, beta;
};

__device__ __forceinline__ Prod prod_of(const NsMaps& mp, const NsArgs& a, int s, int bh) {
  const long mm = (long)a.m * a.m;
  const int xs0 = bh * a.nx, ys0 = bh * a.ny;
  auto Xi = [&](int t) { return xs0 + t % a.nx; };
  auto Yi = [&](int t) { return ys0 + t % a.ny; };
  Prod p;
  if (!a.reverse) {
    const int t = s >> 1;
    if ((s & 1) == 0) {  // Y_t = A X_t
      p = Prod{&mp.a_kc, bh, true, &mp.x_bmn, Xi(t), false, a.Y + Yi(t) * mm, nullptr, 1.f, 0.f};
    } else {             // X_{t+1} = -X_t Y_t + 2 X_t
      p = Prod{&mp.x_akc, Xi(t), true, &mp.y_bmn, Yi(t), false, a.X + Xi(t + 1) * mm,
               a.X + Xi(t) * mm, -1.f, 2.f};
    }
  } else {
    const int t = a.iters - 1 - (s >> 2);
    float* G = a.G + bh * mm;
    float* XG = a.XG + bh * mm;
    float* Tm = a.Tm + bh * mm;
    float* dA = a.dA + bh * mm;
    const bool first = t == a.iters - 1;
    switch (s & 3) {
      case 0:  // XG = X_t^T G
        p = Prod{&mp.x_amn, Xi(t), false, &mp.g_bmn, bh, false, XG, nullptr, 1.f, 0.f};
        break;
      case 1:  // dA = -XG X_t^T + dA
        p = Prod{&mp.xg_akc, bh, true, &mp.x_bkc, Xi(t), true, dA, first ? nullptr : dA, -1.f,
                 first ? 0.f : 1.f};
        break;
      case 2:  // Tm = -G Y_t^T + 2 G
        p = Prod{&mp.g_akc, bh, true, &mp.y_bkc, Yi(t), true, Tm, G, -1.f, 2.f};
        break;
      default:  // G = -A^T XG + Tm
        p = Prod{&mp.a_mn, bh, false, &mp.xg_bmn, bh, false, G, Tm, -1.f, 1.f};
        break;
    }
  }
  return p;
}

// issue the TMA copies of stage c (K = 16 c .. 16 c + 15) into one raw slot
__device__ __forceinline__ void issue_stage(uint8_t* raw, const Prod& p, int i0, int c,
                                            uint32_t bar) {
  mbar_expect_tx(bar, kRawStage);
  if (p.ka) tma_load_3d(smem_u32(raw), p.ma, c * TK, i0, p.za, bar);
  else tma_load_3d(smem_u32(raw), p.ma, i0, c * TK, p.za, bar);
  if (p.kb) tma_load_3d(smem_u32(raw + kRawA), p.mb, c * TK, 0, p.zb, bar);
  else tma_load_3d(smem_u32(raw + kRawA), p.mb, 0, c * TK, p.zb, bar);
}

// op(A) of one stage for splitter lane `row` (0..127 of the panel), k-step ah
// (k = 8 ah .. 8 ah + 7): read from the raw slot (load_a), then split and
// written to TMEM columns colh, coll (+0..7) of this warp's lane quarter
// (store_a, warp-collective).  Raw layout: kc box: row r's 16 k values in 64
// bytes at 64 r, its 16-byte piece k4 swizzled to slot k4 ^ ((r / 2) % 4) (the
// 64-byte swizzle: lanes reading one piece of 32 rows then hit every bank once
// per 8 lanes); mn box: value (k, row) at 4 (128 k + row).
__device__ __forceinline__ void load_a(const uint8_t* ra, bool kc, int row, int ah, float (&v)[8]) {
  if (kc) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float4 x = *reinterpret_cast<const float4*>(ra + 64 * row + 16 * ((2 * ah + j) ^ ((row >> 1) & 3)));
      v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
    }
  } else {
    const float* r = reinterpret_cast<const float*>(ra);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = r[TM * (8 * ah + j) + row];
  }
}
__device__ __forceinline__ void store_a(const float (&v)[8], uint32_t colh, uint32_t coll) {
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float h = tf32_hi(v[j]);
    hi[j] = __float_as_uint(h);
    lo[j] = __float_as_uint(v[j] - h);
  }
  tmem_st8(colh, hi);
  tmem_st8(coll, lo);
}

__device__ __forceinline__ void store_transposed(uint8_t* hi, uint8_t* lo, uint32_t lbo, int rb,
                                                 int k4, const float4 (&x)[4]) {
  store_split(hi, lo, kmaj_off(4 * rb + 0, k4, lbo), make_float4(x[0].x, x[1].x, x[2].x, x[3].x));
  store_split(hi, lo, kmaj_off(4 * rb + 1, k4, lbo), make_float4(x[0].y, x[1].y, x[2].y, x[3].y));
  store_split(hi, lo, kmaj_off(4 * rb + 2, k4, lbo), make_float4(x[0].z, x[1].z, x[2].z, x[3].z));
  store_split(hi, lo, kmaj_off(4 * rb + 3, k4, lbo), make_float4(x[0].w, x[1].w, x[2].w, x[3].w));
}

// op(B)^T of one stage (256 rows x 16 k), thread ts of the 256 splitters: four
// 16-byte pieces read from the raw slot (load_b), then split and stored in the
// K-major layout (store_b).  Raw kc box: piece (row, k4) of 16 bytes at
// 64 row + 16 (k4 ^ ((row / 2) % 4)); thread ts takes row ts, pieces k4 = 0..3.
// Raw 3-D box (mn): [16 k][256 rows]; thread ts takes the 4-row block
// rb = ts % 64 at k4 = ts / 64 (four pieces along the rows, transposed).
// Consecutive lanes read consecutive 16-byte words.
__device__ __forceinline__ void load_b(const uint8_t* rbase, bool kc, int ts, float4 (&x)[4]) {
  if (kc) {
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4)
      x[k4] = *reinterpret_cast<const float4*>(rbase + 64 * ts + 16 * (k4 ^ ((ts >> 1) & 3)));
  } else {
    const int rb = ts % (TNMAX / 4), k4 = ts / (TNMAX / 4);
    const float* r = reinterpret_cast<const float*>(rbase);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      x[j] = *reinterpret_cast<const float4*>(r + TNMAX * (4 * k4 + j) + 4 * rb);
  }
}
__device__ __forceinline__ void store_b(const float4 (&x)[4], bool kc, uint8_t* sp, int ts) {
  uint8_t* bhi = sp;
  uint8_t* blo = sp + kTileB;
  if (kc) {
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) store_split(bhi, blo, kmaj_off(ts, k4, kLboB), x[k4]);
  } else {
    const int rb = ts % (TNMAX / 4), k4 = ts / (TNMAX / 4);
    store_transposed(bhi, blo, kLboB, rb, k4, x);
  }
}
}  // namespace

__global__ void __launch_bounds__(NTH, 1)
    k_ns_cluster(const __grid_constant__ NsMaps maps, NsArgs a) {
  extern __shared__ uint8_t tsm_raw[];
  __shared__ __align__(8) uint64_t spl_full[NSPL], spl_free[NSPL], raw_full[NRAW], raw_free[NRAW],
      acc_full, mma_done;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, i0 = TM * blockIdx.x;
  const int m = a.m;
  const int np = (m + 15) & ~15;  // MMA N
  uint8_t* tsm = tsm_raw + ((1024u - (smem_u32(tsm_raw) & 1023u)) & 1023u);
  uint8_t* stage_base = tsm;
  uint8_t* raw_base = tsm + kRawOff;
  uint8_t* epi_base = stage_base;  // split stages 0-1 (see the header)
  const int nchunks = (m + TK - 1) / TK;
  const int nprod = a.reverse ? 4 * a.iters : 2 * a.iters;
  constexpr unsigned kFull = 0xffffffffu;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < NSPL; ++s) {
      mbar_init(smem_u32(&spl_full[s]), NSPW);  // one arrival per splitter warp
      mbar_init(smem_u32(&spl_free[s]), 1);
    }
    for (int s = 0; s < NRAW; ++s) {
      mbar_init(smem_u32(&raw_full[s]), 1);
      mbar_init(smem_u32(&raw_free[s]), NSPW);
    }
    mbar_init(smem_u32(&acc_full), 1);
    mbar_init(smem_u32(&mma_done), 1);
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid == 32 * kTmaWarp) {
    const CUtensorMap* all = &maps.a_kc;
    for (int i = 0; i < (int)(sizeof(NsMaps) / sizeof(CUtensorMap)); ++i)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(all + i)) : "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base_s;
  auto fail = [&]() {
    atomicExch(a.err, 1);
    abort_s = 1;
  };

  int q = 0;       // stages of all earlier products (the same count in every role)
  int issued = 0;  // TMA stages issued (producer lane)
  for (int s = 0; s < nprod; ++s, q += nchunks) {
    const Prod p = prod_of(maps, a, s, bh);
    if (warp < NSPW) {
      // ---- splitters ----
      const int ts = tid;
      const int aq = warp & 3, ah = warp >> 2;  // TMEM lane quarter, op(A) k-step
      const uint32_t alane = (uint32_t)(32 * aq) << 16;
      // Software-pipelined: stage c + 1's raw values are read (and its raw slot
      // released) while stage c's split stores drain, before stage c is
      // published; the waits for stage c + 1 need only earlier stages' MMAs and
      // copies, never stage c's.
      float va[8];
      float4 xb[4];
      auto fetch = [&](int c) -> bool {  // wait for stage c and read it (all lanes)
        const int qq = q + c, u = qq % NSPL, r = qq % NRAW;
        if (__any_sync(kFull, abort_s)) return false;
        const bool ok =
            (qq < NSPL || mbar_wait(smem_u32(&spl_free[u]), (uint32_t)((qq / NSPL - 1) & 1))) &&
            mbar_wait(smem_u32(&raw_full[r]), (uint32_t)((qq / NRAW) & 1));
        if (!__all_sync(kFull, ok)) {
          fail();
          return false;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint8_t* raw = raw_base + r * kRawStage;
        load_a(raw, p.ka, 32 * aq + lane, ah, va);
        load_b(raw + kRawA, p.kb, ts, xb);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&raw_free[r]));  // this warp has read the raw slot
        return true;
      };
      bool ok = nchunks > 0 && fetch(0);
      for (int c = 0; ok && c < nchunks; ++c) {
        const int qq = q + c, u = qq % NSPL;
        const uint32_t col = tmem + alane + kAcol + 32u * u + 8u * ah;
        store_a(va, col, col + 16u);
        store_b(xb, p.kb, stage_base + u * kStage, ts);
        const bool more = c + 1 < nchunks;
        if (more) ok = fetch(c + 1);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        // generic-proxy stores visible to the tensor core's async proxy; TMEM
        // stores ordered before the MMA warp's thread sync
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&spl_full[u]));
      }
    } else if (warp == kTmaWarp) {
      // ---- TMA producer (one lane) ----
      if (lane == 0) {
        for (int c = 0; c < nchunks; ++c) {
          const int qq = q + c, r = qq % NRAW;
          if (abort_s) break;
          if (qq >= NRAW && !mbar_wait(smem_u32(&raw_free[r]), (uint32_t)((qq / NRAW - 1) & 1))) {
            fail();
            break;
          }
          issue_stage(raw_base + r * kRawStage, p, i0, c, smem_u32(&raw_full[r]));
          issued = qq + 1;
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ---- MMA issuer (first lane) ----
      if (lane == 0 && !abort_s) {
        const uint32_t id = idesc(np);
        for (int c = 0; c < nchunks; ++c) {
          const int qq = q + c, u = qq % NSPL;
          if (!mbar_wait(smem_u32(&spl_full[u]), (uint32_t)((qq / NSPL) & 1))) {
            fail();
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t sp = smem_u32(stage_base + u * kStage);
          const uint32_t b_hi = sp, b_lo = sp + kTileB;
          const uint32_t a_hi = tmem + kAcol + 32u * u, a_lo = a_hi + 16u;
#pragma unroll
          for (int k = 0; k < TK / 8; ++k) {
            const uint64_t dbh = make_desc(b_hi + 2 * k * kLboB, kLboB);
            const uint64_t dbl = make_desc(b_lo + 2 * k * kLboB, kLboB);
            mma_tf32_ta(tmem, a_hi + 8u * k, dbh, id, (c > 0 || k > 0) ? 1u : 0u);
            mma_tf32_ta(tmem, a_hi + 8u * k, dbl, id, 1u);
            mma_tf32_ta(tmem, a_lo + 8u * k, dbh, id, 1u);
          }
          mma_commit(smem_u32(&spl_free[u]));
        }
        if (!abort_s) mma_commit(smem_u32(&acc_full));
      }
      __syncwarp();
    }
    {
      // ---- epilogue, all twelve warps: three per TMEM lane quarter, each
      // taking every third 32-column piece ----
      const int quarter = warp & 3, slot = warp >> 2;
      uint8_t* stg = epi_base + warp * kEpiWarp;
      const int c4 = lane & 7;
      const int r0 = i0 + 32 * quarter;
      auto load_e = [&](float4 (&e)[8], int cb) {
        if (!p.E || cb >= np) return;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int row = r0 + 4 * it + (lane >> 3), col = cb + 4 * c4;
          e[it] = row < m && col < m ? ldcg4(p.E + (size_t)row * m + col) : make_float4(0, 0, 0, 0);
        }
      };
      const int npc = (np + 31) / 32;  // 32-column pieces
      float4 e0[8], e1[8];
      load_e(e0, 32 * slot);
      load_e(e1, 32 * (slot + 3));
      const bool ok = !abort_s && mbar_wait(smem_u32(&acc_full), (uint32_t)(s & 1));
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // tcgen05.ld is warp-collective: the whole warp takes the same decision
      if (__all_sync(kFull, ok && !abort_s)) {
        auto piece = [&](int cb, const float4 (&e)[8]) {
          uint32_t v[32];
          const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)cb;
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
              "%26, %27, %28, %29, %30, %31}, [%32];"
              : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
                "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
                "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
                "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
                "=r"(v[31])
              : "r"(taddr));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          // lane = row: stage the 32 x 32 piece, then write it out by whole rows
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(stg + lane * kEpiPitch + 16 * k) =
                make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rl = 4 * it + (lane >> 3);
            const int row = r0 + rl, col = cb + 4 * c4;
            const float4 x = *reinterpret_cast<const float4*>(stg + rl * kEpiPitch + 16 * c4);
            if (row < m && col < m) {
              float4 o = make_float4(p.alpha * x.x, p.alpha * x.y, p.alpha * x.z, p.alpha * x.w);
              if (p.E) {
                o.x += p.beta * e[it].x; o.y += p.beta * e[it].y;
                o.z += p.beta * e[it].z; o.w += p.beta * e[it].w;
              }
              *reinterpret_cast<float4*>(p.C + (size_t)row * m + col) = o;
            }
          }
          __syncwarp();
        };
#pragma unroll 1
        for (int pi = slot; pi < npc; pi += 6) {
          piece(32 * pi, e0);
          load_e(e0, 32 * (pi + 6));
          if (pi + 3 < npc) piece(32 * (pi + 3), e1);
          load_e(e1, 32 * (pi + 9));
        }
      } else if (!ok) {
        fail();
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    // the product is complete in global memory for the whole cluster (and
    // visible to the async proxy that reads it with TMA) before the next one
    // starts; the accumulator is free again
    asm volatile("fence.proxy.async.global;" ::: "memory");
    cluster_sync();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }

  if (warp == kTmaWarp && lane == 0) {
    // drain: every copy issued must have landed before the CTA may exit
    for (int qq = issued > NRAW ? issued - NRAW : 0; qq < issued; ++qq)
      if (!mbar_wait(smem_u32(&raw_full[qq % NRAW]), (uint32_t)((qq / NRAW) & 1)))
        atomicExch(a.err, 1);
  }
  if (warp == kMmaWarp && lane == 0) {
    // tracks every MMA issued above, also after an abort
    mma_commit(smem_u32(&mma_done));
    if (!mbar_wait(smem_u32(&mma_done), 0u)) atomicExch(a.err, 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  __syncwarp();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
}

namespace {
// whether a cluster of `ncta` CTAs of this kernel fits on the current device
bool cluster_fits(int ncta) {
  static std::mutex mu;
  static int fits[64][3] = {};  // per device and cluster size: 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || ncta < 1 || ncta > 2)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  if (fits[dev][ncta] == 0) {
    bool ok = allow_smem(k_ns_cluster, kSmem) == cudaSuccess;
    if (ok) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(ncta, 1);
      cfg.blockDim = dim3(NTH);
      cfg.dynamicSmemBytes = kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = ncta;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      ok = cudaOccupancyMaxActiveClusters(&n, k_ns_cluster, &cfg) == cudaSuccess && n > 0;
    }
    cudaGetLastError();  // a refused query leaves no error behind
    fits[dev][ncta] = ok ? 1 : 2;
  }
  return fits[dev][ncta] == 1;
}

// ---- tensor maps (the driver's encoder is looked up once through the
// runtime, so the library does not link the driver) ----
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// nmat row-major m x m matrices at p, rows holding K contiguously: 3-D view
// {m k, m rows, nmat} read in {16, rows, 1} boxes, one 64-byte row per request,
// with the 64-byte swizzle (piece k4 of row r lands in slot k4 ^ ((r / 2) % 4))
bool map_kc(CUtensorMap* t, const float* p, int m, int nmat, int rows) {
  const cuuint64_t dim[3] = {(cuuint64_t)m, (cuuint64_t)m, (cuuint64_t)nmat};
  const cuuint64_t stride[2] = {(cuuint64_t)m * 4, (cuuint64_t)m * m * 4};
  const cuuint32_t box[3] = {TK, (cuuint32_t)rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encoder()(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p), dim, stride, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// the same matrices read as [k][row] (row contiguous): 3-D view {m, m, nmat}
// in {rows, TK, 1} boxes
bool map_mn(CUtensorMap* t, const float* p, int m, int nmat, int rows) {
  const cuuint64_t dim[3] = {(cuuint64_t)m, (cuuint64_t)m, (cuuint64_t)nmat};
  const cuuint64_t stride[2] = {(cuuint64_t)m * 4, (cuuint64_t)m * m * 4};
  const cuuint32_t box[3] = {(cuuint32_t)rows, TK, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encoder()(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p), dim, stride, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

void* tensor_map_encoder() { return reinterpret_cast<void*>(encoder()); }

bool encode_tiled_f32(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                      const cuuint64_t* stride, const cuuint32_t* box) {
  EncodeTiled fn = encoder();
  if (fn == nullptr || rank < 1 || rank > 5) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(p), dim, stride,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_f32_sw128(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                            const cuuint64_t* stride, const cuuint32_t* box) {
  EncodeTiled fn = encoder();
  if (fn == nullptr || rank < 1 || rank > 5) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(p), dim, stride,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_bf16_sw128(CUtensorMap* t, int rank, const void* p, const cuuint64_t* dim,
                             const cuuint64_t* stride, const cuuint32_t* box) {
  EncodeTiled fn = encoder();
  if (fn == nullptr || rank < 1 || rank > 5) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(p), dim,
            stride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ns_cluster_ok(int m) {
  return m > 64 && m <= 2 * TM && m % 4 == 0 && encoder() != nullptr &&
         cluster_fits((m + TM - 1) / TM);
}

cudaError_t run_ns_cluster(const Prob& p, bool reverse, const float* A, float* X, float* Y, int nx,
                           int ny, float* G, float* XG, float* Tm, float* dA, cudaStream_t st) {
  if (!ns_cluster_ok(p.m)) return cudaErrorInvalidValue;
  if (p.iters == 0) return cudaSuccess;
  NsArgs a;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidValue;
  a.X = X; a.Y = Y; a.G = G; a.XG = XG; a.Tm = Tm; a.dA = dA;
  a.m = p.m; a.iters = p.iters; a.nx = nx; a.ny = ny; a.reverse = reverse ? 1 : 0;
  const int m = p.m, BH = p.BH;
  // every map, also those the program does not use (the reverse buffers of a
  // forward point at A: valid memory, never read)
  const float* g = G ? G : A;
  const float* xg = XG ? XG : A;
  NsMaps mp;
  memset(&mp, 0, sizeof(mp));
  const bool ok = map_kc(&mp.a_kc, A, m, BH, TM) && map_mn(&mp.a_mn, A, m, BH, TM) &&
                  map_kc(&mp.x_akc, X, m, BH * nx, TM) && map_mn(&mp.x_amn, X, m, BH * nx, TM) &&
                  map_mn(&mp.x_bmn, X, m, BH * nx, TNMAX) && map_kc(&mp.x_bkc, X, m, BH * nx, TNMAX) &&
                  map_mn(&mp.y_bmn, Y, m, BH * ny, TNMAX) && map_kc(&mp.y_bkc, Y, m, BH * ny, TNMAX) &&
                  map_kc(&mp.g_akc, g, m, BH, TM) && map_mn(&mp.g_bmn, g, m, BH, TNMAX) &&
                  map_kc(&mp.xg_akc, xg, m, BH, TM) && map_mn(&mp.xg_bmn, xg, m, BH, TNMAX);
  if (!ok) return cudaErrorInvalidValue;
  const int ncta = (m + TM - 1) / TM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta, BH);
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int slot = prof_begin(reverse ? "ns_cluster_rev" : "ns_cluster", st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_ns_cluster, mp, a);
  prof_end(slot, st);
  count_launch();
  return e;
}

}  // namespace lapnys
