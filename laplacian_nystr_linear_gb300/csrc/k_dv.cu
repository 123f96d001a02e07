// dV of Laplacian-kernel Nystrom attention for bf16 tokens:
//     dV_j = sum_a C_ja dW_a      (W = C V, "SOFT" review, Proposed method,
//                                  S-hat = P^T A^+ P read with C = k(L, K))
// with the kernel values C the forward kept (token-major [BH][N][mp], fp32) and
// dW = X_T^T dW-hat ([BH][m][d], fp32).  The product streams C once from HBM,
// so it is bound by that read (4 mp bytes per token).  The same product is the
// forward's query pass when Q = K and no feature map applies: P = k(Q, L) is
// then C^T, stored token-major exactly like P, and O = P W-hat = C W-hat (the
// symmetric kernel of the "SOFT" review, S-hat = P^T A^+ P).
//
// C enters the tensor cores as stored: kind::tf32 MMAs read the fp32 values
// (their TF32 part) straight from the TMA stages, so no pass touches C on the
// SMs.  The result is rounded once to bf16, 2^-9 relative, well above the
// TF32 truncation of C and the TF32 rounding of R (2^-11 .. 2^-10).
//
// k_dv_pack first writes R^T as the B operand's shared-memory image (per
// slice: blocks of 32 landmarks, D rows of 128 bytes, 128-byte swizzle, TF32
// rounded), so that the product kernel fetches a slice's operand with one bulk
// copy.  k_dv: persistent CTAs over contiguous ranges of (slice, 128-token
// tile) items, warp-specialised:
//   warp 0, one lane   TMA: each 64-landmark chunk of an item's C rows as two
//                      [128 tokens][32 landmarks] boxes (128-byte swizzle) into
//                      a 3-stage ring; a new slice's R^T image into one of two
//                      buffers;
//   warp 1, one lane   eight M = 128, N = d, K = 8 MMAs per chunk into one of
//                      two TMEM accumulators (an item's epilogue overlaps the
//                      next item's products);
//   warps 2-5          epilogue: tcgen05.ld, bf16 rows to global.
// Every wait is bounded; after an expired wait the CTA stops, waits (bounded)
// for its copies and products in flight, frees its tensor memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int TM = 128;                       // tokens per item (MMA M)
constexpr int KC = 64;                        // landmarks per chunk
constexpr int NTH = 192;                      // producer, MMA, four epilogue warps
constexpr int NST = 3;                        // C stages
constexpr uint32_t BOX = TM * 32 * 4;         // [128 tokens][32 landmarks] fp32
constexpr uint32_t STAGE = 2 * BOX;           // one chunk
constexpr uint32_t SW_SBO = 1024;             // 8 rows x 128 bytes
constexpr uint64_t SW128 = 2;                 // descriptor layout type: 128-byte swizzle

template <int D>
struct DvSmem {
  __host__ __device__ static constexpr uint32_t wbytes(int mp) { return (uint32_t)mp * D * 4; }
  static constexpr uint32_t Stages = 0;
  static constexpr uint32_t Wb = NST * STAGE;  // two R^T images
  __host__ __device__ static constexpr uint32_t total(int mp) { return Wb + 2 * wbytes(mp) + 1024; }
};

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return tc::desc(saddr, 16, SW_SBO) | (SW128 << 61);
}

__device__ __forceinline__ bool wait_or_flag(int* err, uint32_t bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  if (!ok) atomicOr(err, 1);
  return ok;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
}  // namespace

// R^T image: img[bh][kb][n][32] (swizzled) = tf32(R[bh][32 kb + k][n]), zero past m.
// Grid (mp / 32, BH), 256 threads.
template <int D>
__global__ void __launch_bounds__(256) k_dv_pack(const float* __restrict__ R, float* __restrict__ img,
                                                 int m, int mp) {
  const int kb = blockIdx.x, bh = blockIdx.y;
  const float* Rb = R + (size_t)bh * m * D;
  uint8_t* blk = reinterpret_cast<uint8_t*>(img + ((size_t)bh * mp + 32 * kb) * D);
  constexpr int kPer = 32 * D / 256;  // elements a thread: all loads first, then the stores
  float v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = threadIdx.x + 256 * i, k = e / D, n = e - k * D, a = 32 * kb + k;
    v[i] = a < m ? __ldg(Rb + (size_t)a * D + n) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = threadIdx.x + 256 * i, k = e / D, n = e - k * D;
    const float t = __uint_as_float((__float_as_uint(v[i]) + 0x1000u) & 0xffffe000u);  // nearest TF32
    const uint32_t off = (uint32_t)n * 128u + ((uint32_t)((k >> 2) ^ (n & 7)) << 4) + (uint32_t)(k & 3) * 4u;
    *reinterpret_cast<float*>(blk + off) = t;
  }
}

struct DvArgs {
  const float* img;         // [BH][mp][D] R^T images (k_dv_pack)
  __nv_bfloat16* dv;        // [BH][N][D]
  int* err;
  int N, mp, BH, ntile;
};

template <int D>
__global__ void __launch_bounds__(NTH, 1) k_dv(const __grid_constant__ CUtensorMap cmap, DvArgs a) {
  using S = DvSmem<D>;
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[NST], empty[NST];   // C stages
  __shared__ __align__(8) uint64_t wfull[2], wempty[2];     // R^T images
  __shared__ __align__(8) uint64_t accf[2], acce[2];        // accumulators
  __shared__ uint32_t tmem_s;
  __shared__ int issued_s, consumed_s, wissued_s, wconsumed_s, bad_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw_u32 = tc::smem_u32(sm_raw);
  uint8_t* sm = sm_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // swizzle atoms: 1024-aligned
  const int nck = a.mp / KC;
  const long long items = (long long)a.BH * a.ntile;
  const long long i0 = items * blockIdx.x / gridDim.x, i1 = items * (blockIdx.x + 1) / gridDim.x;
  const uint32_t wbytes = S::wbytes(a.mp);
  constexpr uint32_t kCols = 2 * D < 32 ? 32 : 2 * D;

  if (warp == 1) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(tc::smem_u32(&full[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(&wfull[i]), 1);
      tc::mbar_init(tc::smem_u32(&wempty[i]), 1);
      tc::mbar_init(tc::smem_u32(&accf[i]), 1);
      tc::mbar_init(tc::smem_u32(&acce[i]), 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&cmap)) : "memory");
    issued_s = consumed_s = wissued_s = wconsumed_s = bad_s = 0;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int st = 0, issued = 0, ns = 0, cur = -1;
      uint32_t ph = 0;
      bool bad = false;
      for (long long it = i0; it < i1 && !bad; ++it) {
        const int bh = (int)(it / a.ntile), tile = (int)(it % a.ntile);
        if (bh != cur) {  // the slice's R^T image into buffer ns & 1
          const int wb = ns & 1;
          if (ns >= 2 && !wait_or_flag(a.err, tc::smem_u32(&wempty[wb]), (uint32_t)((ns - 2) >> 1) & 1u)) {
            bad = true;
            break;
          }
          const uint32_t bar = tc::smem_u32(&wfull[wb]);
          tc::mbar_expect_tx(bar, wbytes);
          tc::bulk_g2s(tc::smem_u32(sm + S::Wb + wb * wbytes), a.img + (size_t)bh * a.mp * D, wbytes, bar);
          cur = bh;
          ++ns;
        }
        for (int ck = 0; ck < nck; ++ck) {
          if (!wait_or_flag(a.err, tc::smem_u32(&empty[st]), ph ^ 1u)) { bad = true; break; }
          const uint32_t bar = tc::smem_u32(&full[st]);
          const uint32_t dst = tc::smem_u32(sm + S::Stages + st * STAGE);
          tc::mbar_expect_tx(bar, STAGE);
          tma_load_3d(dst, &cmap, ck * KC, tile * TM, bh, bar);
          tma_load_3d(dst + BOX, &cmap, ck * KC + 32, tile * TM, bh, bar);
          ++issued;
          if (++st == NST) { st = 0; ph ^= 1u; }
        }
      }
      issued_s = issued;
      wissued_s = ns;
      if (bad) atomicOr(&bad_s, 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      int st = 0, consumed = 0, ns = 0, cur = -1;
      uint32_t ph = 0;
      long long li = 0;
      bool bad = false;
      const uint32_t id = tc::idesc_tf32(TM, D);
      uint32_t wb_addr = 0;
      for (long long it = i0; it < i1 && !bad; ++it, ++li) {
        const int bh = (int)(it / a.ntile);
        if (bh != cur) {
          if (cur >= 0) tc::commit(tc::smem_u32(&wempty[(ns - 1) & 1]));  // the last slice's image is free
          if (!wait_or_flag(a.err, tc::smem_u32(&wfull[ns & 1]), (uint32_t)(ns >> 1) & 1u)) {
            bad = true;
            break;
          }
          wb_addr = tc::smem_u32(sm + S::Wb + (ns & 1) * wbytes);
          cur = bh;
          ++ns;
        }
        const int acc = (int)(li & 1);
        if (!wait_or_flag(a.err, tc::smem_u32(&acce[acc]), (uint32_t)((li >> 1) & 1) ^ 1u)) {
          bad = true;
          break;
        }
        tc::fence_after();
        const uint32_t dt = tmem + (uint32_t)(acc * D);
        for (int ck = 0; ck < nck; ++ck) {
          if (!wait_or_flag(a.err, tc::smem_u32(&full[st]), ph)) { bad = true; break; }
          tc::fence_after();
          const uint32_t sa = tc::smem_u32(sm + S::Stages + st * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ss(dt, sdesc(sa + b * BOX + kk * 32),
                         sdesc(wb_addr + (uint32_t)(2 * ck + b) * (D * 128) + kk * 32), id,
                         (ck > 0 || b > 0 || kk > 0) ? 1u : 0u);
          tc::commit(tc::smem_u32(&empty[st]));
          ++consumed;
          if (++st == NST) { st = 0; ph ^= 1u; }
        }
        if (bad) break;
        tc::commit(tc::smem_u32(&accf[acc]));
      }
      consumed_s = consumed;
      wconsumed_s = ns;
      if (bad) atomicOr(&bad_s, 1);
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                       // TMEM lane quarter
    long long li = 0;
    bool bad = false;
    for (long long it = i0; it < i1; ++it, ++li) {
      const int bh = (int)(it / a.ntile), tile = (int)(it % a.ntile);
      const int acc = (int)(li & 1);
      if (!wait_or_flag(a.err, tc::smem_u32(&accf[acc]), (uint32_t)(li >> 1) & 1u)) {
        bad = true;
        break;
      }
      tc::fence_after();
      const int j = tile * TM + 32 * q + lane;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tc::tmem_ld<32>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * D + 32 * ch), v);
        if (j < a.N) {
          uint4* o = reinterpret_cast<uint4*>(a.dv + ((size_t)bh * a.N + j) * D + 32 * ch);
#pragma unroll
          for (int p = 0; p < 4; ++p)
            o[p] = make_uint4(pack_bf16(__uint_as_float(v[8 * p]), __uint_as_float(v[8 * p + 1])),
                              pack_bf16(__uint_as_float(v[8 * p + 2]), __uint_as_float(v[8 * p + 3])),
                              pack_bf16(__uint_as_float(v[8 * p + 4]), __uint_as_float(v[8 * p + 5])),
                              pack_bf16(__uint_as_float(v[8 * p + 6]), __uint_as_float(v[8 * p + 7])));
        }
      }
      tc::fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&acce[acc])) : "memory");
    }
    if (bad) atomicOr(&bad_s, 1);
  }

  // ---- drain and free the tensor memory ----
  // On a healthy run the epilogue waited for the last products and the products
  // for every copy.  After an expired wait: the last MMA commit (it covers every
  // earlier MMA), then every copy issued but not consumed.
  __syncthreads();
  if (bad_s && warp == 1 && lane == 0) {
    const int c = consumed_s, n = issued_s;
    if (c > 0) wait_or_flag(a.err, tc::smem_u32(&empty[(c - 1) % NST]), (uint32_t)((c - 1) / NST) & 1u);
    for (int k = c; k < n; ++k)
      wait_or_flag(a.err, tc::smem_u32(&full[k % NST]), (uint32_t)(k / NST) & 1u);
    for (int k = wconsumed_s; k < wissued_s; ++k)
      wait_or_flag(a.err, tc::smem_u32(&wfull[k & 1]), (uint32_t)(k >> 1) & 1u);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool dv_tc_ok(const Prob& p) {
  if (p.dtype != 1 || (p.d != 32 && p.d != 64) || tensor_map_encoder() == nullptr) return false;
  const size_t smem = p.d == 64 ? DvSmem<64>::total(p.mp) : DvSmem<32>::total(p.mp);
  return smem <= 227u * 1024u;
}

size_t dv_image_floats(const Prob& p) { return (size_t)p.BH * p.mp * p.d; }

template <int D>
static cudaError_t dv_t(const Prob& p, const float* C, const float* R, float* img, void* dv,
                        const char* name, cudaStream_t st) {
  using S = DvSmem<D>;
  const size_t smem = S::total(p.mp);
  cudaError_t e = allow_smem(k_dv<D>, smem);
  if (e != cudaSuccess) return e;
  // C as a 3-D tensor {mp landmarks, N tokens, BH slices}, boxes of 32 x 128
  // (128-byte rows: the swizzle's span); chunk offsets are multiples of 32
  // landmarks (128 bytes), so every box starts 16-byte aligned
  CUtensorMap map;
  const cuuint64_t dim[3] = {(cuuint64_t)p.mp, (cuuint64_t)p.N, (cuuint64_t)p.BH};
  const cuuint64_t stride[2] = {(cuuint64_t)p.mp * 4, (cuuint64_t)p.N * p.mp * 4};
  const cuuint32_t box[3] = {32, TM, 1};
  if (!encode_tiled_f32_sw128(&map, 3, C, dim, stride, box)) return cudaErrorInvalidValue;
  if ((e = launch("dv_pack", k_dv_pack<D>, dim3(p.mp / 32, p.BH), dim3(256), 0, st, R, img, p.m,
                  p.mp)) != cudaSuccess)
    return e;
  DvArgs a;
  a.img = img; a.dv = (__nv_bfloat16*)dv;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidSymbol;
  a.N = p.N; a.mp = p.mp; a.BH = p.BH; a.ntile = (p.N + TM - 1) / TM;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long items = (long long)a.BH * a.ntile;
  const int grid = (int)(items < sms ? items : sms);
  return launch(name, k_dv<D>, dim3(grid), dim3(NTH), smem, st, map, a);
}

cudaError_t run_dv(const Prob& p, const float* C, const float* R, float* img, void* out,
                   const char* name, cudaStream_t st) {
  if (!dv_tc_ok(p)) return cudaErrorInvalidValue;
  if (p.d == 64) return dv_t<64>(p, C, R, img, out, name, st);
  return dv_t<32>(p, C, R, img, out, name, st);
}

}  // namespace lapnys
