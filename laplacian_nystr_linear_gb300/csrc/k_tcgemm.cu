// Batched fp32-accurate matrix products on the 5th-generation tensor cores
// (tcgen05, kind::tf32) for the Newton-Schulz iteration A_{k+1} = 2 A_k -
// A_k A A_k of the "SOFT" review (Proposed method) and its reverse.
//
// The iteration runs far from convergence on ill-conditioned landmark
// matrices, where single-pass TF32 products are not accurate enough, so every
// operand is split x = hi + lo (hi = x rounded to TF32, lo = x - hi exactly)
// and the product is accumulated in fp32 as hi*hi + hi*lo + lo*hi; the missing
// lo*lo term and the TF32 truncation of lo are O(2^-21) relative.
//
// CTA = 128 x 128 output tile, 256 threads (8 warps; warps w and w + 4 read
// TMEM lanes 32 (w % 4) .. + 31, one half of the columns each).
// K advances 16 at a time: cp.async copies the raw fp32 tiles of op(A) and
// op(B) one chunk ahead into shared memory; all threads then split a landed
// chunk into hi / lo tiles in the canonical K-major, no-swizzle layout (8-row x
// 16-byte core matrices, double buffered); one thread issues the 6 MMAs of the
// chunk (2 k-steps x 3 split products) and commits them to the buffer's
// mbarrier, which is waited on before that buffer is refilled.  The accumulator lives in TMEM (64 columns) and is read
// back with tcgen05.ld for the epilogue C = alpha acc + beta E.
//
// Every wait is bounded: on expiry the kernel records an error in a device
// word (read by lapnys_device_status), stops issuing work, waits a bounded
// time for its MMAs, frees its TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

__device__ int g_lapnys_wait_error;  // nonzero once a bounded wait expired

namespace lapnys {

namespace {
constexpr int TM = 128;   // rows per CTA (MMA M)
constexpr int TN = 128;   // columns per CTA (MMA N)
constexpr int TK = 16;    // K per stage
constexpr int NRAW = 2;   // raw (unsplit) stages in flight
constexpr int NTH = 256;  // threads: 8 warps, two per 32-lane TMEM quarter
constexpr uint32_t kLboA = (TM / 8) * 128;  // bytes between 4-wide K groups of the A tile
constexpr uint32_t kLboB = (TN / 8) * 128;  // same for the B tile
constexpr uint32_t kSbo = 128;              // bytes between 8-row groups
constexpr uint32_t kTileA = TM * TK * 4;    // bytes of one A matrix (hi or lo) per stage
constexpr uint32_t kTileB = TN * TK * 4;
constexpr uint32_t kStage = 2 * kTileA + 2 * kTileB;  // A hi, A lo, B hi, B lo
// raw stage: the larger of the two layouts of each operand
constexpr int kRawA = (TM * (TK + 4) > TK * (TM + 8) ? TM * (TK + 4) : TK * (TM + 8));
constexpr int kRawB = (TN * (TK + 4) > TK * (TN + 8) ? TN * (TK + 4) : TK * (TN + 8));
constexpr uint32_t kRawStage = (uint32_t)(kRawA + kRawB) * 4u;
constexpr int kWaitLimit = 1 << 22;

// instruction descriptor: D f32, A/B tf32, both K-major, N = TN, M = TM
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(TN >> 3) << 17) |
                            ((uint32_t)(TM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// shared-memory matrix descriptor, K-major without swizzle
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for this architecture
  return d;
}

// byte offset of element (row, k) of a K-major tile with `lbo` bytes per K group
__device__ __forceinline__ uint32_t kmaj_off(int row, int k, uint32_t lbo) {
  return (uint32_t)(k >> 2) * lbo + (uint32_t)(row >> 3) * kSbo + (uint32_t)(row & 7) * 16u +
         (uint32_t)(k & 3) * 4u;
}

// x = hi + lo with hi rounded to the nearest TF32 value (halfway cases away
// from zero: half an ulp added to the magnitude bits, 13 low bits cleared)
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
  lo = x - hi;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count));
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

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}

struct TcArgs {
  const float* A; const float* B; float* C; const float* E;
  int lda, ldb, ldc, lde;
  long sA, sB, sC, sE;
  int M, N, K;
  float alpha, beta;
};

// cp.async helpers (cp_async16, cp_commit) come from common.cuh
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Raw (unsplit) tile of one K chunk of an operand with ROWS output rows.
// KCONT: the source holds each row's k values contiguously, raw layout
// [ROWS][TK + 4]; otherwise the source is [k][row], raw layout [TK][ROWS + 8].
// The paddings make the split pass below bank-conflict free.
template <int ROWS, bool KCONT>
struct Raw {
  static constexpr int LD = KCONT ? TK + 4 : ROWS + 8;

  // issue the 16-byte copies of chunk k0 (zero-filled outside the matrix)
  __device__ __forceinline__ static void copy(float* raw, const float* src, int ld, int row0,
                                              int nrows, int k0, int K) {
    if (KCONT) {
      for (int e = threadIdx.x; e < ROWS * (TK / 4); e += NTH) {
        const int r = e / (TK / 4), kq = e % (TK / 4);
        const int row = row0 + r, k = k0 + 4 * kq;
        const bool ok = row < nrows && k < K;
        cp_async16(smem_u32(raw + r * LD + 4 * kq), ok ? src + (size_t)row * ld + k : src, ok);
      }
    } else {
      for (int e = threadIdx.x; e < TK * (ROWS / 4); e += NTH) {
        const int kk = e / (ROWS / 4), rq = e % (ROWS / 4);
        const int row = row0 + 4 * rq, k = k0 + kk;
        const bool ok = row < nrows && k < K;
        cp_async16(smem_u32(raw + kk * LD + 4 * rq), ok ? src + (size_t)k * ld + row : src, ok);
      }
    }
  }

  // split the raw chunk into hi / lo K-major tiles, 4 k values of a row per
  // 16-byte chunk; a source stored [k][row] is transposed in registers in
  // 4 x 4 blocks
  __device__ __forceinline__ static void split(const float* raw, uint8_t* hi, uint8_t* lo,
                                               uint32_t lbo) {
    if (KCONT) {
#pragma unroll
      for (int i = 0; i < ROWS * (TK / 4) / NTH; ++i) {
        const int e = threadIdx.x + i * NTH;
        const int r = e % ROWS, kq = e / ROWS;
        const float4 v = *reinterpret_cast<const float4*>(raw + r * LD + 4 * kq);
        float4 h, l;
        split_tf32(v.x, h.x, l.x);
        split_tf32(v.y, h.y, l.y);
        split_tf32(v.z, h.z, l.z);
        split_tf32(v.w, h.w, l.w);
        const uint32_t off = kmaj_off(r, 4 * kq, lbo);
        *reinterpret_cast<float4*>(hi + off) = h;
        *reinterpret_cast<float4*>(lo + off) = l;
      }
    } else {
#pragma unroll
      for (int i = 0; i < (ROWS / 4) * (TK / 4) / NTH + ((ROWS / 4) * (TK / 4) % NTH ? 1 : 0); ++i) {
        const int e = threadIdx.x + i * NTH;
        if (e >= (ROWS / 4) * (TK / 4)) break;
        // rows rq + (ROWS / 4) rr: lanes take consecutive rows, so both the
        // scalar loads and the 16-byte stores are bank-conflict free
        const int rq = e % (ROWS / 4), kq = e / (ROWS / 4);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int row = rq + (ROWS / 4) * rr;
          float4 h, l;
          split_tf32(raw[(4 * kq + 0) * LD + row], h.x, l.x);
          split_tf32(raw[(4 * kq + 1) * LD + row], h.y, l.y);
          split_tf32(raw[(4 * kq + 2) * LD + row], h.z, l.z);
          split_tf32(raw[(4 * kq + 3) * LD + row], h.w, l.w);
          const uint32_t off = kmaj_off(row, 4 * kq, lbo);
          *reinterpret_cast<float4*>(hi + off) = h;
          *reinterpret_cast<float4*>(lo + off) = l;
        }
      }
    }
  }
};
}  // namespace

// C[b] = alpha op(A[b]) op(B[b]) + beta E[b]; requires M, N, K, leading
// dimensions and strides to be multiples of 4 and 16-byte aligned bases.
template <bool TA, bool TB>
__global__ void __launch_bounds__(NTH, 1) k_tcgemm(TcArgs g) {
  extern __shared__ __align__(1024) uint8_t tsm[];
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bz = blockIdx.z;
  const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TN;
  const float* A = g.A + bz * g.sA;
  const float* B = g.B + bz * g.sB;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(TN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(smem_u32(&mbar[0]), 1);
    mbar_init(smem_u32(&mbar[1]), 1);
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base_s;

  const int nchunks = (g.K + TK - 1) / TK;
  uint32_t phase[2] = {0u, 0u};
  int last_st = -1;  // buffer of the most recent commit
  bool ok = true;
  using RA = Raw<TM, !TA>;  // op(A) rows i: TA ? A[k][i] : A[i][k]
  using RB = Raw<TN, TB>;   // op(B)^T rows j: TB ? B[j][k] : B[k][j]
  float* raw0 = reinterpret_cast<float*>(tsm + 2 * kStage);
  auto raw_a = [&](int c) { return raw0 + (c % NRAW) * (kRawA + kRawB); };
  auto raw_b = [&](int c) { return raw0 + (c % NRAW) * (kRawA + kRawB) + kRawA; };
#pragma unroll
  for (int c = 0; c < NRAW - 1; ++c) {
    if (c < nchunks) {
      RA::copy(raw_a(c), A, g.lda, i0, g.M, c * TK, g.K);
      RB::copy(raw_b(c), B, g.ldb, j0, g.N, c * TK, g.K);
    }
    cp_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    const int st = c & 1;
    {
      const int cn = c + NRAW - 1;  // chunk whose copies go out now
      if (cn < nchunks) {
        RA::copy(raw_a(cn), A, g.lda, i0, g.M, cn * TK, g.K);
        RB::copy(raw_b(cn), B, g.ldb, j0, g.N, cn * TK, g.K);
      }
      cp_commit();
    }
    cp_wait<NRAW - 1>();  // this thread's copies of chunk c have landed
    uint8_t* base = tsm + st * kStage;
    uint8_t* ahi = base;
    uint8_t* alo = base + kTileA;
    uint8_t* bhi = base + 2 * kTileA;
    uint8_t* blo = base + 2 * kTileA + kTileB;
    if (c >= 2) {
      // the MMAs that read this buffer two chunks ago must be done
      if (!mbar_wait(smem_u32(&mbar[st]), phase[st])) {
        atomicExch(&g_lapnys_wait_error, 1);
        abort_s = 1;
      }
      phase[st] ^= 1u;
    }
    __syncthreads();  // every thread's copies of chunk c are visible
    if (abort_s) {
      ok = false;
      break;
    }
    RA::split(raw_a(c), ahi, alo, kLboA);
    RB::split(raw_b(c), bhi, blo, kLboB);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t sa_hi = smem_u32(ahi), sa_lo = smem_u32(alo);
      const uint32_t sb_hi = smem_u32(bhi), sb_lo = smem_u32(blo);
#pragma unroll
      for (int s = 0; s < TK / 8; ++s) {
        const uint32_t oa = (uint32_t)(2 * s) * kLboA, ob = (uint32_t)(2 * s) * kLboB;
        const uint64_t dah = make_desc(sa_hi + oa, kLboA, kSbo);
        const uint64_t dal = make_desc(sa_lo + oa, kLboA, kSbo);
        const uint64_t dbh = make_desc(sb_hi + ob, kLboB, kSbo);
        const uint64_t dbl = make_desc(sb_lo + ob, kLboB, kSbo);
        mma_tf32(tmem, dah, dbh, (c > 0 || s > 0) ? 1u : 0u);
        mma_tf32(tmem, dah, dbl, 1u);
        mma_tf32(tmem, dal, dbh, 1u);
      }
      mma_commit(smem_u32(&mbar[st]));
    }
    last_st = st;
  }
  cp_wait<0>();
  // the last commit tracks every MMA issued before it; wait for it (bounded)
  // also after an abort, so that no MMA still writes TMEM when it is freed
  if (last_st >= 0) {
    if (!mbar_wait(smem_u32(&mbar[last_st]), phase[last_st])) {
      atomicExch(&g_lapnys_wait_error, 1);
      ok = false;
    }
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  __syncthreads();

  if (ok) {
    float* C = g.C + bz * g.sC;
    const float* E = g.E ? g.E + bz * g.sE : nullptr;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = i0 + 32 * quarter + lane;
#pragma unroll
    for (int cb = half * (TN / 2); cb < (half + 1) * (TN / 2); cb += 16) {
      uint32_t r[16];
      const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)cb;
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
          "%11, %12, %13, %14, %15}, [%16];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
            "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
            "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
          : "r"(taddr));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (row < g.M) {
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
          const int col = j0 + cb + q;
          if (col < g.N) {
            float4 v = make_float4(g.alpha * __uint_as_float(r[q]), g.alpha * __uint_as_float(r[q + 1]),
                                   g.alpha * __uint_as_float(r[q + 2]), g.alpha * __uint_as_float(r[q + 3]));
            if (E) {
              const float4 e = *reinterpret_cast<const float4*>(E + (size_t)row * g.lde + col);
              v.x += g.beta * e.x; v.y += g.beta * e.y; v.z += g.beta * e.z; v.w += g.beta * e.w;
            }
            *reinterpret_cast<float4*>(C + (size_t)row * g.ldc + col) = v;
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TN)
                 : "memory");
}

bool tc_gemm_ok(int M, int N, int K, int lda, int ldb, int ldc, int lde, long sA, long sB, long sC,
                long sE, const void* A, const void* B, const void* C, const void* E) {
  auto al = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  bool ok = M % 4 == 0 && N % 4 == 0 && K % 4 == 0 && lda % 4 == 0 && ldb % 4 == 0 &&
            ldc % 4 == 0 && sA % 4 == 0 && sB % 4 == 0 && sC % 4 == 0 && al(A) && al(B) && al(C);
  if (E) ok = ok && lde % 4 == 0 && sE % 4 == 0 && al(E);
  return ok;
}

cudaError_t run_tcgemm(bool ta, bool tb, int batch, int M, int N, int K, const float* A, int lda,
                       long sA, const float* B, int ldb, long sB, float* C, int ldc, long sC,
                       const float* E, int lde, long sE, float alpha, float beta, cudaStream_t st) {
  TcArgs g;
  g.A = A; g.B = B; g.C = C; g.E = beta == 0.f ? nullptr : E;
  g.lda = lda; g.ldb = ldb; g.ldc = ldc; g.lde = lde;
  g.sA = sA; g.sB = sB; g.sC = sC; g.sE = sE;
  g.M = M; g.N = N; g.K = K; g.alpha = alpha; g.beta = beta;
  const size_t smem = 2 * (size_t)kStage + NRAW * (size_t)kRawStage;
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM, batch);
#define TC(TA_, TB_)                                                                   \
  if (ta == TA_ && tb == TB_) {                                                        \
    static bool once = (allow_smem(k_tcgemm<TA_, TB_>, smem), true);                   \
    (void)once;                                                                        \
    return launch("tcgemm", k_tcgemm<TA_, TB_>, grid, dim3(NTH), smem, st, g);         \
  }
  TC(false, false) TC(false, true) TC(true, false) TC(true, true)
#undef TC
  return cudaErrorInvalidValue;
}

// Self-test of the bounded waits: one thread initialises an mbarrier that
// expects one arrival, which nothing makes, and waits on its first phase with
// the same bounded wait the tensor-core kernels use (at most `polls` polls).  The
// wait expires, the error word is set, and the kernel returns: nothing is in
// flight (no copy, no MMA, no TMEM), so the context stays usable.
__global__ void k_wait_selftest(int polls) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t a = tc::smem_u32(&bar);
  tc::mbar_init(a, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!tc::mbar_wait(a, 0u, polls)) atomicExch(&g_lapnys_wait_error, 1);
}

int tc_wait_limit() { return tc::kWaitLimit; }

cudaError_t run_wait_selftest(int polls, cudaStream_t st) {
  return launch("wait_selftest", k_wait_selftest, dim3(1), dim3(32), 0, st, polls);
}

// The address of the error word in the current context, looked up on every
// call: a symbol's device address belongs to a context (a reset device or a
// second context on the same device has its own copy), so caching it per
// device ordinal could hand a kernel a dead address.
int* wait_error_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_lapnys_wait_error) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

int read_wait_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_lapnys_wait_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_lapnys_wait_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace lapnys
