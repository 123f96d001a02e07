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
// Persistent CTAs, one per SM, walk (slice, 128-token tile) items.  Per item
// the 64-landmark chunks of its C rows arrive by TMA (four stages, so three
// chunks are in flight while one is split: the read needs ~70 KB in flight per
// SM to cover the memory latency at the bandwidth's per-SM share); all threads
// split each chunk into bf16 planes c_hi + c_lo (the A operand, K-major), and one
// thread issues the tcgen05 kind::f16 products c_hi w_hi + c_hi w_lo + c_lo w_hi
// against dW^T held in shared memory as bf16 planes w_hi + w_lo (loaded once per
// slice), accumulating in tensor memory (two accumulators, so an item's
// epilogue overlaps the next item's products).  The epilogue rounds once to bf16.
// Every wait is bounded; an expired wait stops the CTA (uniformly) and drains.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lapnys {

namespace {
constexpr int TM = 128;                       // tokens per item (MMA M)
constexpr int KC = 64;                        // landmarks per chunk
constexpr int NTH = 512;                      // 16 warps: enough to hide the split's latencies
constexpr uint32_t SBO = 128;
constexpr uint32_t LBO_C = (TM / 8) * SBO + 16;   // A planes: 8-landmark K groups (padded)
constexpr uint32_t PLANE_C = (KC / 8) * LBO_C;
constexpr uint32_t RAW = TM * KC * 4;         // one TMA box: [128 tokens][64 landmarks] fp32
constexpr int NST = 4;                        // raw stages

template <int D>
struct DvSmem {
  static constexpr uint32_t LBO_W = (D / 8) * SBO;  // B planes (dW^T): 8-landmark K groups
  static constexpr uint32_t Raw = 0;                // NST stages
  static constexpr uint32_t Ca = Raw + NST * RAW;   // (hi, lo) of the chunk being multiplied
  static constexpr uint32_t Wb = Ca + 2 * PLANE_C;  // (hi, lo) x mp landmarks
  __host__ __device__ static constexpr uint32_t plane_w(int mp) { return (uint32_t)(mp / 8) * LBO_W; }
  __host__ __device__ static constexpr uint32_t total(int mp) { return Wb + 2 * plane_w(mp); }
};

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

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}
}  // namespace

struct DvArgs {
  const float* dW;          // [BH][m][D]
  __nv_bfloat16* dv;        // [BH][N][D]
  int* err;
  int N, m, mp, BH, ntile;
};

template <int D>
__global__ void __launch_bounds__(NTH, 1) k_dv(const __grid_constant__ CUtensorMap cmap, DvArgs a) {
  using S = DvSmem<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[NST];   // a raw stage landed
  __shared__ __align__(8) uint64_t mdone;       // a step's MMAs (which read the A planes) done
  __shared__ __align__(8) uint64_t adone[2];    // accumulator t finished (its last chunk's MMAs)
  __shared__ uint32_t tmem_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nck = a.mp / KC;                    // chunks per item
  const long long items = (long long)a.BH * a.ntile;
  const long long i0 = items * blockIdx.x / gridDim.x, i1 = items * (blockIdx.x + 1) / gridDim.x;
  const int nsteps = (int)(i1 - i0) * nck;      // (item, chunk) steps of this CTA
  const uint32_t id = tc::idesc_bf16(TM, D);
  constexpr uint32_t kCols = 2 * D < 32 ? 32 : 2 * D;

  if (warp == 0) tc::tmem_alloc(&tmem_s, kCols);
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) tc::mbar_init(tc::smem_u32(&full[i]), 1);
    tc::mbar_init(tc::smem_u32(&mdone), 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(tc::smem_u32(&adone[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&cmap)) : "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_s;

  // the copy of step s (item i0 + s / nck, chunk s % nck) into raw stage s % NST (thread 0)
  auto issue = [&](int s) {
    const long long it = i0 + s / nck;
    const int bh = (int)(it / a.ntile), tile = (int)(it % a.ntile), ck = s % nck;
    const uint32_t bar = tc::smem_u32(&full[s % NST]);
    tc::mbar_expect_tx(bar, RAW);
    tma_load_3d(tc::smem_u32(sm + S::Raw + (s % NST) * RAW), &cmap, ck * KC, tile * TM, bh, bar);
  };
  if (tid == 0)
    for (int s = 0; s < NST && s < nsteps; ++s) issue(s);

  // epilogue of item ni (its accumulator ni & 1): bf16 rows; lane quarter w % 4
  // holds tokens 32 (w % 4) .., warps w, w + 4, w + 8, w + 12 split the columns
  auto epilogue = [&](int ni) {
    const long long it = i0 + ni;
    const int bh = (int)(it / a.ntile), tile = (int)(it % a.ntile), t = ni & 1;
    const bool ok = wait_or_flag(a.err, tc::smem_u32(&adone[t]), (uint32_t)(ni >> 1) & 1u);
    tc::fence_after();
    constexpr int HC = D / (NTH / 128);
    uint32_t v[HC];
    tc::tmem_ld<HC>(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(t * D + (warp >> 2) * HC), v);
    const int j = tile * TM + 32 * (warp & 3) + lane;
    if (j < a.N && ok) {
      uint4* o = reinterpret_cast<uint4*>(a.dv + ((size_t)bh * a.N + j) * D + (warp >> 2) * HC);
#pragma unroll
      for (int c = 0; c < HC; c += 8)
        o[c / 8] = make_uint4(bf16_bits(__uint_as_float(v[c])) | (bf16_bits(__uint_as_float(v[c + 1])) << 16),
                              bf16_bits(__uint_as_float(v[c + 2])) | (bf16_bits(__uint_as_float(v[c + 3])) << 16),
                              bf16_bits(__uint_as_float(v[c + 4])) | (bf16_bits(__uint_as_float(v[c + 5])) << 16),
                              bf16_bits(__uint_as_float(v[c + 6])) | (bf16_bits(__uint_as_float(v[c + 7])) << 16));
    }
    tc::fence_before();
    return ok;
  };

  bool bad = false, abort = false;
  int wslice = -1;                              // slice whose dW^T planes are loaded
  int nmma = 0;                                 // MMA commits issued (chunk steps)
  for (int s = 0; s < nsteps; ++s) {
    const long long it = i0 + s / nck;
    const int bh = (int)(it / a.ntile), ck = s % nck;
    const int t = (s / nck) & 1;                // accumulator of this item
    if (bh != wslice) {
      // dW^T of a new slice as two bf16 planes (row = feature, k = landmark); the
      // previous products that read the planes are done first
      if (nmma > 0) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone), (uint32_t)(nmma - 1) & 1u);
      __syncthreads();
      const float* W = a.dW + (size_t)bh * a.m * D;
      for (int e = tid; e < (a.mp / 2) * (D / 8); e += NTH) {
        const int cg = e % (D / 8), ap = 2 * (e / (D / 8));
        float w0[8], w1[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          w0[q] = ap < a.m ? __ldg(W + (size_t)ap * D + 8 * cg + q) : 0.f;
          w1[q] = ap + 1 < a.m ? __ldg(W + (size_t)(ap + 1) * D + 8 * cg + q) : 0.f;
        }
        uint8_t* dst = sm + S::Wb + (uint32_t)(ap >> 3) * S::LBO_W + (uint32_t)cg * SBO + (ap & 7) * 2;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t h0 = bf16_bits(w0[q]), h1 = bf16_bits(w1[q]);
          const uint32_t l0 = bf16_bits(w0[q] - __uint_as_float(h0 << 16));
          const uint32_t l1 = bf16_bits(w1[q] - __uint_as_float(h1 << 16));
          *reinterpret_cast<uint32_t*>(dst + q * 16) = h0 | (h1 << 16);
          *reinterpret_cast<uint32_t*>(dst + S::plane_w(a.mp) + q * 16) = l0 | (l1 << 16);
        }
      }
      wslice = bh;
    }
    // raw chunk -> A planes (row = token, k = landmark), after the previous step's
    // products that read them
    bad |= !wait_or_flag(a.err, tc::smem_u32(&full[s % NST]), (uint32_t)(s / NST) & 1u);
    if (nmma > 0) bad |= !wait_or_flag(a.err, tc::smem_u32(&mdone), (uint32_t)(nmma - 1) & 1u);
    {
      const float* raw = reinterpret_cast<const float*>(sm + S::Raw + (s % NST) * RAW);
      uint8_t* ca = sm + S::Ca;
      for (int e = tid; e < TM * (KC / 4); e += NTH) {
        const int j = e / (KC / 4), a4 = 4 * (e % (KC / 4));
        const float4 v = *reinterpret_cast<const float4*>(raw + j * KC + a4);
        const float f[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          h[q] = bf16_bits(f[q]);
          l[q] = bf16_bits(f[q] - __uint_as_float(h[q] << 16));
        }
        const uint32_t off = (uint32_t)(a4 >> 3) * LBO_C + (uint32_t)(j >> 3) * SBO + (j & 7) * 16 + (a4 & 7) * 2;
        *reinterpret_cast<uint2*>(ca + off) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        *reinterpret_cast<uint2*>(ca + PLANE_C + off) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(bad)) {
      abort = true;
      break;
    }
    if (tid == 0) {
      if (s + NST < nsteps) issue(s + NST);   // raw stage s % NST is free (split above)
      tc::fence_after();
      // the accumulator of this item: its previous user (item - 2) was read out
      // during item - 1's first step
      const uint32_t acc = tmem + (uint32_t)(t * D);
      const uint32_t ca = tc::smem_u32(sm + S::Ca);
      const uint32_t wb = tc::smem_u32(sm + S::Wb) + (uint32_t)(ck * (KC / 8)) * S::LBO_W;
#pragma unroll
      for (int k16 = 0; k16 < KC / 16; ++k16) {
        const uint32_t ka = k16 * 2 * LBO_C, kb = k16 * 2 * S::LBO_W;
        tc::mma_bf16(acc, tc::desc(ca + ka, LBO_C, SBO), tc::desc(wb + kb, S::LBO_W, SBO), id,
                     (ck > 0 || k16 > 0) ? 1u : 0u);
        tc::mma_bf16(acc, tc::desc(ca + ka, LBO_C, SBO),
                     tc::desc(wb + S::plane_w(a.mp) + kb, S::LBO_W, SBO), id, 1u);
        tc::mma_bf16(acc, tc::desc(ca + PLANE_C + ka, LBO_C, SBO), tc::desc(wb + kb, S::LBO_W, SBO),
                     id, 1u);
      }
      tc::commit(tc::smem_u32(&mdone));
      if (ck == nck - 1) tc::commit(tc::smem_u32(&adone[t]));
    }
    ++nmma;
    // the previous item's epilogue once this item's first products are queued (the
    // two accumulators alternate, so they overlap)
    if (ck == 0 && s > 0) bad |= !epilogue(s / nck - 1);
  }
  if (!abort && nsteps > 0) epilogue(nsteps / nck - 1);
  if (abort) {
    // drain: the last MMAs (their commit covers the earlier ones) and the copies in flight
    if (nmma > 0) wait_or_flag(a.err, tc::smem_u32(&mdone), (uint32_t)(nmma - 1) & 1u);
    if (tid == 0)
      for (int k = nmma; k < min(nsteps, nmma + NST); ++k)
        wait_or_flag(a.err, tc::smem_u32(&full[k % NST]), (uint32_t)(k / NST) & 1u);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool dv_tc_ok(const Prob& p) {
  return p.dtype == 1 && (p.d == 32 || p.d == 64) && tensor_map_encoder() != nullptr &&
         DvSmem<64>::total(p.mp) <= 227u * 1024u;
}

template <int D>
static cudaError_t dv_t(const Prob& p, const float* C, const float* dW, void* dv, const char* name,
                        cudaStream_t st) {
  using S = DvSmem<D>;
  const size_t smem = S::total(p.mp);
  cudaError_t e = allow_smem(k_dv<D>, smem);
  if (e != cudaSuccess) return e;
  // C as a 3-D tensor {mp landmarks, N tokens, BH slices}, boxes of 64 x 128
  CUtensorMap map;
  const cuuint64_t dim[3] = {(cuuint64_t)p.mp, (cuuint64_t)p.N, (cuuint64_t)p.BH};
  const cuuint64_t stride[2] = {(cuuint64_t)p.mp * 4, (cuuint64_t)p.N * p.mp * 4};
  const cuuint32_t box[3] = {KC, TM, 1};
  if (!encode_tiled_f32(&map, 3, C, dim, stride, box)) return cudaErrorInvalidValue;
  DvArgs a;
  a.dW = dW; a.dv = (__nv_bfloat16*)dv;
  a.err = wait_error_address();
  if (a.err == nullptr) return cudaErrorInvalidSymbol;
  a.N = p.N; a.m = p.m; a.mp = p.mp; a.BH = p.BH; a.ntile = (p.N + TM - 1) / TM;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long items = (long long)a.BH * a.ntile;
  const int grid = (int)(items < sms ? items : sms);
  return launch(name, k_dv<D>, dim3(grid), dim3(NTH), smem, st, map, a);
}

cudaError_t run_dv(const Prob& p, const float* C, const float* dW, void* dv, const char* name,
                   cudaStream_t st) {
  if (!dv_tc_ok(p)) return cudaErrorInvalidValue;
  if (p.d == 64) return dv_t<64>(p, C, dW, dv, name, st);
  return dv_t<32>(p, C, dW, dv, name, st);
}

}  // namespace lapnys
