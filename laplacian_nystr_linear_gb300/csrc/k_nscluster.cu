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
// products; operands are read through L2 (ld.global.cg), never a stale L1
// line.  Twelve warps with fixed roles (three per SM sub-partition, so that
// each may hold up to 168 registers):
//   warps 0-7  per K-stage (16): load their rows of op(A) straight into
//           registers three stages ahead (lane = row, warp w covers TMEM lane
//           quarter w % 4 and k-step w / 4), split them into TF32 hi / lo and
//           write them into TMEM (tcgen05.st), where the MMA reads op(A); copy
//           op(B) into a 4-stage raw ring in shared memory (cp.async through
//           L2, each thread copying exactly the pieces it later splits, so its
//           own wait_group is all the ordering needed), split it and store hi /
//           lo into a 3-stage ring in the K-major core-matrix layout (8 rows x
//           16 bytes per core matrix; 8-row groups 144 bytes apart and K groups
//           32 bytes further apart than dense, which keeps the split stores free
//           of bank conflicts).  An op(B) whose rows hold K contiguously is read
//           four lanes per row (8 rows per warp copy); one stored [k][row] in
//           4-row blocks along the row, transposed at the split.  Keeping op(A)
//           out of shared memory removes its split stores and the tensor core's
//           reads of it, a third of the shared-memory traffic that bounds the
//           K loop.
//   warp 8  allocates TMEM (accumulator: columns 0-255; op(A) stages: 32
//           columns each from 256); its first lane issues each stage's six MMAs
//           (2 k-steps x 3 split products, A from TMEM, B from shared memory),
//           commits them to the stage's "free"
//           mbarrier and, after a product's last stage, to the accumulator
//           barrier.
//   all twelve warps then read the accumulator back with tcgen05.ld (warp w
//           reads TMEM lanes 32 (w % 4) .., three warps per lane quarter, each
//           taking every third 32-column piece), transpose 32 x 32 pieces
//           through a small per-warp buffer (in split stages 0-1, idle between a
//           product's last MMA and the next cluster barrier) and write
//           C = alpha acc + beta E in whole lines; E is fetched two pieces
//           ahead.
//
// Every mbarrier wait is bounded: on expiry the CTA records an error in the
// device word read by lapnys_device_status and stops working, but still takes
// part in every cluster barrier, so that the other CTA of its cluster finishes.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace lapnys {

namespace {
constexpr int TM = 128;    // rows per CTA (MMA M)
constexpr int TNMAX = 256; // largest MMA N
constexpr int TK = 16;     // K per stage
constexpr int NSPL = 3;    // split (hi / lo) stages
constexpr int NRAW = 4;    // raw stages (copies in flight per splitter thread)
constexpr int NSPW = 8;    // splitter warps
constexpr int NSPT = NSPW * 32;
constexpr int NEPW = 4;    // epilogue warps
constexpr int NTH = NSPT + NEPW * 32;  // 384
constexpr int kMmaWarp = NSPW;         // first epilogue warp
constexpr uint32_t kSbo = 144;                       // bytes between 8-row groups
constexpr uint32_t kLboB = (TNMAX / 8) * kSbo + 32;  // same, B tile
constexpr uint32_t kTileB = (TK / 4) * kLboB;
constexpr uint32_t kStage = 2 * kTileB;              // B hi, B lo
constexpr uint32_t kAcol = TNMAX;                     // first TMEM column of the op(A) stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRawStage = TNMAX * TK * 4;       // raw B pieces per stage (bytes)
constexpr uint32_t kEpiPitch = 36 * 4;               // staged row: 32 floats + 16-byte pad
constexpr uint32_t kEpiWarp = 32 * kEpiPitch;
static_assert(NTH / 32 * kEpiWarp <= 2 * kStage, "epilogue staging fits in two split stages");
static_assert(kAcol + NSPL * 32 <= kTmemCols, "op(A) stages fit in TMEM");
constexpr size_t kSmem = (size_t)NSPL * kStage + (size_t)NRAW * kRawStage + 128;
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

// one product of the program, slice-local m x m row-major matrices
struct Prod {
  const float* A;  // op(A) = A (ka) or A^T
  const float* B;  // op(B) = B^T (kb) or B
  float* C;
  const float* E;  // null when beta == 0
  bool ka, kb;     // the operand's rows hold K contiguously
  float alpha, beta;
};
}  // namespace

struct NsArgs {
  const float* A;  // [BH][m][m]
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
__device__ __forceinline__ Prod prod_of(const NsArgs& a, int s, int bh) {
  const long mm = (long)a.m * a.m;
  const float* Ab = a.A + bh * mm;
  auto Xs = [&](int t) { return a.X + ((long)bh * a.nx + t % a.nx) * mm; };
  auto Ys = [&](int t) { return a.Y + ((long)bh * a.ny + t % a.ny) * mm; };
  Prod p;
  if (!a.reverse) {
    const int t = s >> 1;
    if ((s & 1) == 0) {  // Y_t = A X_t
      p = Prod{Ab, Xs(t), Ys(t), nullptr, true, false, 1.f, 0.f};
    } else {             // X_{t+1} = -X_t Y_t + 2 X_t
      p = Prod{Xs(t), Ys(t), Xs(t + 1), Xs(t), true, false, -1.f, 2.f};
    }
  } else {
    const int t = a.iters - 1 - (s >> 2);
    float* G = a.G + bh * mm;
    float* XG = a.XG + bh * mm;
    float* Tm = a.Tm + bh * mm;
    float* dA = a.dA + bh * mm;
    switch (s & 3) {
      case 0: p = Prod{Xs(t), G, XG, nullptr, false, false, 1.f, 0.f}; break;       // X_t^T G
      case 1: p = Prod{XG, Xs(t), dA, t == a.iters - 1 ? nullptr : dA, true, true, -1.f,
                       t == a.iters - 1 ? 0.f : 1.f}; break;                         // -XG X_t^T + dA
      case 2: p = Prod{G, Ys(t), Tm, G, true, true, -1.f, 2.f}; break;               // -G Y_t^T + 2G
      default: p = Prod{Ab, XG, G, Tm, false, false, -1.f, 1.f}; break;              // -A^T XG + Tm
    }
  }
  return p;
}

// op(A) for one splitter lane: row `row`, the 8 k values kb .. kb + 7 (zero
// outside the matrix), through L2.
struct ARegs {
  float v[8];
};
__device__ __forceinline__ void load_a(ARegs& r, const Prod& p, int m, int row, int kb) {
  if (p.ka) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float4 x = row < m && kb + 4 * j < m ? ldcg4(p.A + (size_t)row * m + kb + 4 * j)
                                                 : make_float4(0, 0, 0, 0);
      r.v[4 * j] = x.x; r.v[4 * j + 1] = x.y; r.v[4 * j + 2] = x.z; r.v[4 * j + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      r.v[j] = row < m && kb + j < m ? __ldcg(p.A + (size_t)(kb + j) * m + row) : 0.f;
  }
}
// split into TF32 hi / lo and write them to TMEM columns colh .. + 7 and
// coll .. + 7 of this warp's lane quarter (warp-collective)
__device__ __forceinline__ void store_a(const ARegs& r, uint32_t colh, uint32_t coll) {
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float h = tf32_hi(r.v[j]);
    hi[j] = __float_as_uint(h);
    lo[j] = __float_as_uint(r.v[j] - h);
  }
  tmem_st8(colh, hi);
  tmem_st8(coll, lo);
}

// One splitter thread's share of one stage (16 k) of op(B)^T (up to 256 rows:
// the result columns), as 16-byte pieces.  Rows holding K contiguously: unit
// u = (row u / 4, k4 = u % 4), units ts + 256 h.  Stored [k][row]: unit
// (4-row block, k4), four pieces (k = 4 k4 + j) taken along the rows and
// transposed at the split.  Piece i of thread ts sits at raw + 16 (i * NSPT +
// ts), so a warp's copies and reads touch consecutive 16-byte words.
__device__ __forceinline__ void issue_stage(uint8_t* rb, const Prod& p, int m, int k0, int ts) {
  if (p.kb) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int u = ts + h * NSPT, row = u >> 2, kk = k0 + 4 * (u & 3);
      const bool ok = row < m && kk < m;
      cp_async16(smem_addr(rb + 16 * (h * NSPT + ts)), p.B + (ok ? (size_t)row * m + kk : 0), ok);
    }
  } else {
    const int row = 4 * (ts % (TNMAX / 4)), kk = k0 + 4 * (ts / (TNMAX / 4));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = row < m && kk + j < m;
      cp_async16(smem_addr(rb + 16 * (j * NSPT + ts)), p.B + (ok ? (size_t)(kk + j) * m + row : 0), ok);
    }
  }
}

__device__ __forceinline__ float4 raw_piece(const uint8_t* base, int i, int ts) {
  return *reinterpret_cast<const float4*>(base + 16 * (i * NSPT + ts));
}

__device__ __forceinline__ void store_transposed(uint8_t* hi, uint8_t* lo, uint32_t lbo, int rb,
                                                 int k4, const float4 (&x)[4]) {
  store_split(hi, lo, kmaj_off(4 * rb + 0, k4, lbo), make_float4(x[0].x, x[1].x, x[2].x, x[3].x));
  store_split(hi, lo, kmaj_off(4 * rb + 1, k4, lbo), make_float4(x[0].y, x[1].y, x[2].y, x[3].y));
  store_split(hi, lo, kmaj_off(4 * rb + 2, k4, lbo), make_float4(x[0].z, x[1].z, x[2].z, x[3].z));
  store_split(hi, lo, kmaj_off(4 * rb + 3, k4, lbo), make_float4(x[0].w, x[1].w, x[2].w, x[3].w));
}

__device__ __forceinline__ void split_stage(const uint8_t* rb, const Prod& p, uint8_t* sp, int ts) {
  uint8_t* bhi = sp;
  uint8_t* blo = sp + kTileB;
  if (p.kb) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int u = ts + h * NSPT;
      store_split(bhi, blo, kmaj_off(u >> 2, u & 3, kLboB), raw_piece(rb, h, ts));
    }
  } else {
    const float4 x[4] = {raw_piece(rb, 0, ts), raw_piece(rb, 1, ts), raw_piece(rb, 2, ts),
                         raw_piece(rb, 3, ts)};
    store_transposed(bhi, blo, kLboB, ts % (TNMAX / 4), ts / (TNMAX / 4), x);
  }
}
}  // namespace

__global__ void __launch_bounds__(NTH, 1) k_ns_cluster(NsArgs a) {
  extern __shared__ uint8_t tsm_raw[];
  __shared__ __align__(8) uint64_t spl_full[NSPL], spl_free[NSPL], acc_full, mma_done;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, i0 = TM * blockIdx.x;
  const int m = a.m;
  const int np = (m + 15) & ~15;  // MMA N
  uint8_t* tsm = tsm_raw + ((128u - (smem_u32(tsm_raw) & 127u)) & 127u);
  uint8_t* stage_base = tsm;
  uint8_t* raw_base = tsm + NSPL * kStage;
  uint8_t* epi_base = stage_base;  // split stage 0 (see the header)
  const int nchunks = (m + TK - 1) / TK;
  const int nprod = a.reverse ? 4 * a.iters : 2 * a.iters;

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
    mbar_init(smem_u32(&acc_full), 1);
    mbar_init(smem_u32(&mma_done), 1);
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base_s;
  auto fail = [&]() {
    atomicExch(a.err, 1);
    abort_s = 1;
  };

  int q = 0;  // stages of all earlier products (the same count in every role)
  for (int s = 0; s < nprod; ++s, q += nchunks) {
    const Prod p = prod_of(a, s, bh);
    if (warp < NSPW) {
      // ---- splitters ----
      const int ts = tid;
      constexpr unsigned kFull = 0xffffffffu;
      // op(A): lane = row 32 (warp % 4) + lane of the CTA's panel, k-step warp / 4
      const int aq = warp & 3, ah = warp >> 2;
      const int arow = i0 + 32 * aq + lane;
      const uint32_t alane = (uint32_t)(32 * aq) << 16;
      if (!__any_sync(kFull, abort_s)) {
        cp_wait_all();  // nothing of an earlier product is still in flight
#pragma unroll
        for (int c = 0; c < NRAW; ++c) {
          if (c < nchunks) issue_stage(raw_base + c * kRawStage, p, m, c * TK, ts);
          cp_commit();
        }
        ARegs ra0, ra1, ra2;
        load_a(ra0, p, m, arow, 0 * TK + 8 * ah);
        if (nchunks > 1) load_a(ra1, p, m, arow, 1 * TK + 8 * ah);
        if (nchunks > 2) load_a(ra2, p, m, arow, 2 * TK + 8 * ah);
        auto step = [&](int c, ARegs& ra) -> bool {
          const int qq = q + c, u = qq % NSPL;
          if (__any_sync(kFull, abort_s)) return false;
          const bool free_ok =
              qq < NSPL || mbar_wait(smem_u32(&spl_free[u]), (uint32_t)((qq / NSPL - 1) & 1));
          if (!__all_sync(kFull, free_ok)) {
            fail();
            return false;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          // op(A) of stage c into TMEM (this warp's lanes and k-step)
          const uint32_t col = tmem + alane + kAcol + 32u * u + 8u * ah;
          store_a(ra, col, col + 16u);
          if (c + 3 < nchunks) load_a(ra, p, m, arow, (c + 3) * TK + 8 * ah);
          // op(B) of stage c: raw copy landed -> hi / lo tiles
          asm volatile("cp.async.wait_group %0;" ::"n"(NRAW - 1) : "memory");
          uint8_t* raw = raw_base + (c % NRAW) * kRawStage;
          split_stage(raw, p, stage_base + u * kStage, ts);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          // generic-proxy stores visible to the tensor core's async proxy;
          // TMEM stores ordered before the MMA warp's thread sync
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&spl_full[u]));
          // this thread's pieces of stage c are read: refill the slot
          if (c + NRAW < nchunks) issue_stage(raw, p, m, (c + NRAW) * TK, ts);
          cp_commit();
          return true;
        };
        for (int c = 0; c < nchunks; c += 3) {
          if (!step(c, ra0)) break;
          if (c + 1 < nchunks && !step(c + 1, ra1)) break;
          if (c + 2 < nchunks && !step(c + 2, ra2)) break;
        }
      }
    } else if (warp == kMmaWarp) {
      // ---- MMA issuer (first lane) ----
      {
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
      if (__all_sync(0xffffffffu, ok && !abort_s)) {
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
    // the product is complete in global memory for the whole cluster before
    // the next one reads it; the accumulator is free again
    cluster_sync();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
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
}  // namespace

bool ns_cluster_ok(int m) {
  return m > 64 && m <= 2 * TM && m % 4 == 0 && cluster_fits((m + TM - 1) / TM);
}

cudaError_t run_ns_cluster(const Prob& p, bool reverse, const float* A, float* X, float* Y, int nx,
                           int ny, float* G, float* XG, float* Tm, float* dA, cudaStream_t st) {
  if (!ns_cluster_ok(p.m)) return cudaErrorInvalidValue;
  if (p.iters == 0) return cudaSuccess;
  NsArgs a;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidValue;
  a.A = A; a.X = X; a.Y = Y; a.G = G; a.XG = XG; a.Tm = Tm; a.dA = dA;
  a.m = p.m; a.iters = p.iters; a.nx = nx; a.ny = ny; a.reverse = reverse ? 1 : 0;
  const int ncta = (p.m + TM - 1) / TM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta, p.BH);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_ns_cluster, a);
  prof_end(slot, st);
  count_launch();
  return e;
}

}  // namespace lapnys
