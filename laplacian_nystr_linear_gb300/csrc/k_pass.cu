// Token-side passes of Laplacian-kernel Nystrom attention: fused L1-distance
// + exp tiles.  The N x m kernel matrices are only written out (once, for the
// backward) when the caller keeps a ctx; the inference forward never stores them.
//
//   key pass      W   = C V,     C_aj = k(L_a, K_j)                (forward)
//   stats pass    mu, var of P_ia = k(Q_i, L_a) per landmark column (forward, norm)
//   query pass    O   = Z W-hat, Z = P or (P - mu) / sqrt(var + eta)   (forward)
//   tile backward dQ, dK, dV, dL, dW-hat through sgn(x - l)          (backward)
//
// Passages: the Laplacian kernel k(x, y) = exp(-|x - y|_1 / lambda) and its
// non-vanishing L1 gradient ("LaplacianFormer", Dutch summary Methodology 1;
// Arabic summary 2a); the Nystrom product S-hat = P^T A^+ P ("SOFT" review,
// Proposed method) read as O = k(Q, L) A^+ (k(L, K) V); the normalised query
// feature map with a diagonal variance estimate (Arabic summary 2b).
//
// The distance is not a dot product, so it runs on the FP32 pipe: each thread
// holds a 4 x 4 (token x landmark) block of distances and streams the feature
// dimension through shared memory in float4 steps (32 ALU ops per 2 LDS.128).
#include "common.cuh"
#include "internal.h"

namespace lapnys {

template <typename T>
struct TypeOf;
template <>
struct TypeOf<float> { static constexpr int id = 0; };
template <>
struct TypeOf<__nv_bfloat16> { static constexpr int id = 1; };

__device__ __forceinline__ void split_range(int nblk, int S, int s, int& b0, int& b1) {
  b0 = (int)((long long)nblk * s / S);
  b1 = (int)((long long)nblk * (s + 1) / S);
}


// ===========================================================================
// key pass: grid (landmark tile, split, slice).  Each CTA keeps its 64
// landmarks in shared memory, streams its share of the key/value tokens in
// blocks of 64 (the raw rows of the next block are copied in with cp.async
// while the current one computes) and accumulates W[a][c] = sum_j C_aj V_jc.
// ===========================================================================
template <int D, typename T, bool GAUSS>
__global__ void __launch_bounds__(kThreads, 2)
    k_key_fwd(const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ L,
              float* __restrict__ part, float* __restrict__ kvout, int N, int m, int mp, int S,
              int nblk, float ns) {
  constexpr int CPT = D / 16;
  // bf16 inputs: the contraction runs on the tensor cores (TF32 kernel values)
  constexpr bool kTC = TypeOf<T>::id == 1 && D >= 32;
  constexpr int NCT = D / 16;  // 8-wide column tiles per warp (tensor-core path)
  extern __shared__ float4 sm4[];
  float* Ls = reinterpret_cast<float*>(sm4);
  float* Xs = Ls + tile_floats(D);
  float* Vs = Xs + tile_floats(D);
  float* Cs = Vs + tile_floats(D);  // [64 tokens][68]
  constexpr int RP = D * (int)sizeof(T) + 16;  // bytes per raw row
  uint8_t* raw = reinterpret_cast<uint8_t*>(Cs + 64 * 68);  // next block: K rows, then V rows
  // tensor-core fragment coordinates: warp -> landmark rows wa .. wa + 15, columns wc .. wc + D/2 - 1
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tg = lane & 3;
  const int wa = (warp & 3) * 16, wc = (warp >> 2) * (D / 2);
  float acc[NCT][4];
#pragma unroll
  for (int n = 0; n < NCT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * kTile;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const T* Kb = K + (size_t)bh * N * D;
  const T* Vb = V + (size_t)bh * N * D;
  load_tile<D>(Ls, L + (size_t)bh * m * D, a0, m);
  float w[4][CPT];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int c = 0; c < CPT; ++c) w[s][c] = 0.f;
  int b0, b1;
  split_range(nblk, S, sp, b0, b1);
  // raw K and V rows of block b into shared memory, zero past N
  auto prefetch = [&](int b) {
    if (b >= b1) return;
    const int n0 = b * kTile;
    constexpr int CH = D * (int)sizeof(T) / 16;  // 16-byte pieces per row
    for (int id = threadIdx.x; id < 2 * kTile * CH; id += kThreads) {
      const int which = id / (kTile * CH), rem = id % (kTile * CH), j = rem / CH, ch = rem % CH;
      const bool ok = n0 + j < N;
      const T* src = (which ? Vb : Kb) + (size_t)(ok ? n0 + j : 0) * D;
      cp_async16(smem_addr(raw + (which * kTile + j) * RP + 16 * ch),
                 reinterpret_cast<const uint8_t*>(src) + 16 * ch, ok);
    }
    cp_commit();
  };
  prefetch(b0);
  for (int b = b0; b < b1; ++b) {
    cp_wait_all();
    __syncthreads();
    for (int id = threadIdx.x; id < kTile * (D / 4); id += kThreads) {
      const int r = id / (D / 4), c4 = id % (D / 4);
      st4(Xs + r * row_stride(D) + 4 * c4, raw4(raw + r * RP, c4, Kb));
      st4(Vs + r * row_stride(D) + 4 * c4, raw4(raw + (kTile + r) * RP, c4, Vb));
    }
    __syncthreads();
    prefetch(b + 1);
    float dist[4][4];
    dist_tile<D, GAUSS>(Xs, Ls, dist);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int j = b * kTile + 4 * ty + r, a = a0 + tx + 16 * s;
        Cs[(4 * ty + r) * 68 + tx + 16 * s] = (j < N && a < m) ? exp2_ftz(dist[r][s] * ns) : 0.f;
      }
    __syncthreads();
    if (kvout) {
      // keep the tile for the backward: kvout[bh][j][a0 .. a0 + 63], whole rows
      float* base = kvout + (size_t)bh * N * mp + a0;
      for (int id = threadIdx.x; id < kTile * (kTile / 4); id += kThreads) {
        const int r = id / (kTile / 4), c4 = id % (kTile / 4);
        const int j = b * kTile + r;
        if (j < N) st4(base + (size_t)j * mp + 4 * c4, lds4(Cs + r * 68 + 4 * c4));
      }
    }
    if constexpr (kTC) {
      // W[a][c] += sum_j C[j][a] V[j][c] on the tensor cores as (C_hi + C_lo) V with
      // the TF32 split of C (V is bf16, exact in TF32): W enters W-hat = X_T W, whose
      // unconverged directions amplify a single TF32 rounding of C about a hundredfold
#pragma unroll 2
      for (int k0 = 0; k0 < kTile; k0 += 8) {
        const float cv[4] = {Cs[(k0 + tg) * 68 + wa + gq], Cs[(k0 + tg) * 68 + wa + gq + 8],
                             Cs[(k0 + tg + 4) * 68 + wa + gq], Cs[(k0 + tg + 4) * 68 + wa + gq + 8]};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ah[i] = to_tf32(cv[i]);
          al[i] = to_tf32(cv[i] - __uint_as_float(ah[i]));
        }
#pragma unroll
        for (int n = 0; n < NCT; ++n) {
          uint32_t bf[2];
          bf[0] = __float_as_uint(Vs[(k0 + tg) * row_stride(D) + wc + 8 * n + gq]);
          bf[1] = __float_as_uint(Vs[(k0 + tg + 4) * row_stride(D) + wc + 8 * n + gq]);
          mma_16x8x8(acc[n], ah, bf);
          mma_16x8x8(acc[n], al, bf);
        }
      }
    } else {
#pragma unroll 4
      for (int j = 0; j < kTile; ++j) {
        const float4 c4 = lds4(Cs + j * 68 + 4 * ty);
        float v[CPT];
        lds_cpt<CPT>(Vs + j * row_stride(D) + tx * CPT, v);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          w[0][c] = fmaf(c4.x, v[c], w[0][c]);
          w[1][c] = fmaf(c4.y, v[c], w[1][c]);
          w[2][c] = fmaf(c4.z, v[c], w[2][c]);
          w[3][c] = fmaf(c4.w, v[c], w[3][c]);
        }
      }
    }
  }
  if constexpr (kTC) {
    float* P = part + ((size_t)bh * S + sp) * mp * D;
#pragma unroll
    for (int n = 0; n < NCT; ++n) {
      const int c = wc + 8 * n + 2 * tg;
      *reinterpret_cast<float2*>(P + (size_t)(a0 + wa + gq) * D + c) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(P + (size_t)(a0 + wa + gq + 8) * D + c) = make_float2(acc[n][2], acc[n][3]);
    }
  } else {
    float* P = part + (((size_t)bh * S + sp) * mp + a0 + 4 * ty) * D + tx * CPT;
#pragma unroll
    for (int s = 0; s < 4; ++s) st_cpt<CPT>(P + s * D, w[s]);
  }
}

template <int D, typename T>
static cudaError_t key_fwd_t(const Prob& p, const void* k, const void* v, const float* L, float* part,
                             float* kvout, cudaStream_t st) {
  const size_t smem = (3 * (size_t)tile_floats(D) + 64 * 68) * sizeof(float) +
                      2 * (size_t)kTile * (D * sizeof(T) + 16);
  if (p.gauss()) {
    static bool once = (allow_smem(k_key_fwd<D, T, true>, smem), true);
    (void)once;
    return launch("key_fwd", k_key_fwd<D, T, true>, dim3(p.nt, p.Sk, p.BH), dim3(kThreads), smem,
                  st, (const T*)k, (const T*)v, L, part, kvout, p.N, p.m, p.mp, p.Sk, p.nblk, p.ns);
  }
  static bool once = (allow_smem(k_key_fwd<D, T, false>, smem), true);
  (void)once;
  return launch("key_fwd", k_key_fwd<D, T, false>, dim3(p.nt, p.Sk, p.BH), dim3(kThreads), smem, st,
                (const T*)k, (const T*)v, L, part, kvout, p.N, p.m, p.mp, p.Sk, p.nblk, p.ns);
}

#define DISPATCH_DT(FN, ...)                                                        \
  do {                                                                              \
    if (p.dtype == 1) {                                                             \
      switch (p.d) {                                                                \
        case 16: return FN<16, __nv_bfloat16>(__VA_ARGS__);                         \
        case 32: return FN<32, __nv_bfloat16>(__VA_ARGS__);                         \
        case 64: return FN<64, __nv_bfloat16>(__VA_ARGS__);                         \
        case 128: return FN<128, __nv_bfloat16>(__VA_ARGS__);                       \
      }                                                                             \
    } else {                                                                        \
      switch (p.d) {                                                                \
        case 16: return FN<16, float>(__VA_ARGS__);                                 \
        case 32: return FN<32, float>(__VA_ARGS__);                                 \
        case 64: return FN<64, float>(__VA_ARGS__);                                 \
        case 128: return FN<128, float>(__VA_ARGS__);                               \
      }                                                                             \
    }                                                                               \
    return cudaErrorInvalidValue;                                                   \
  } while (0)

cudaError_t run_key_fwd(const Prob& p, const void* k, const void* v, const float* L, float* part,
                        float* kvout, cudaStream_t st) {
  DISPATCH_DT(key_fwd_t, p, k, v, L, part, kvout, st);
}

// ===========================================================================
// out[bh][a][c] = sum_s part[bh][s][a][c]  (a < m; fixed order over s)
// ===========================================================================
__global__ void k_reduce_parts(const float* __restrict__ part, float* __restrict__ out, int BH, int S,
                               int m, int mp, int d) {
  const size_t total = (size_t)BH * m * d;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = e / ((size_t)m * d);
    const size_t ac = e % ((size_t)m * d);
    const float* p = part + bh * S * mp * d + ac;
    float s = 0.f;
    for (int q = 0; q < S; ++q) s += p[(size_t)q * mp * d];
    out[e] = s;
  }
}

static int grid_for(size_t n) {
  size_t g = (n + kThreads - 1) / kThreads;
  return (int)(g < 4096 ? (g < 1 ? 1 : g) : 4096);
}

cudaError_t run_reduce_parts(int BH, int S, int m, int mp, int d, const float* part, float* out,
                             cudaStream_t st) {
  const size_t n = (size_t)BH * m * d;
  return launch("reduce_parts", k_reduce_parts, dim3(grid_for(n)), dim3(kThreads), 0, st, part, out,
                BH, S, m, mp, d);
}

// ===========================================================================
// statistics pass (normalised feature map): per landmark column, the mean and
// centred second moment of P_ia over the slice's queries.  Each 64-token block
// gives an exact two-pass (count, mean, M2) that is merged into the running
// triple with the pairwise update of Chan, Golub and LeVeque.
// grid (landmark tile, split, slice); spart [BH][S][3][mp]
// ===========================================================================
__device__ __forceinline__ void chan_merge(float& n, float& mean, float& M2, float nb, float meanb,
                                           float M2b) {
  if (nb == 0.f) return;
  const float nn = n + nb;
  const float delta = meanb - mean;
  mean += delta * (nb / nn);
  M2 += M2b + delta * delta * (n * nb / nn);
  n = nn;
}

template <int D, typename T, bool GAUSS>
__global__ void __launch_bounds__(kThreads, 2)
    k_qstats(const T* __restrict__ Q, const float* __restrict__ L, float* __restrict__ spart, int N,
             int m, int mp, int S, int nblk, float ns) {
  extern __shared__ float4 sm4[];
  float* Ls = reinterpret_cast<float*>(sm4);
  float* Xs = Ls + tile_floats(D);
  float* Ps = Xs + tile_floats(D);  // [64 tokens][68]
  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * kTile;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const T* Qb = Q + (size_t)bh * N * D;
  load_tile<D>(Ls, L + (size_t)bh * m * D, a0, m);
  float n = 0.f, mean = 0.f, M2 = 0.f;  // meaningful for threads 0..63 (landmark a0 + tid)
  int b0, b1;
  split_range(nblk, S, sp, b0, b1);
  for (int b = b0; b < b1; ++b) {
    __syncthreads();
    load_tile<D>(Xs, Qb, b * kTile, N);
    __syncthreads();
    float dist[4][4];
    dist_tile<D, GAUSS>(Xs, Ls, dist);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) Ps[(4 * ty + r) * 68 + tx + 16 * s] = exp2_ftz(dist[r][s] * ns);
    __syncthreads();
    if (threadIdx.x < kTile) {
      const int nb = min(kTile, N - b * kTile);
      float sum = 0.f;
      for (int j = 0; j < nb; ++j) sum += Ps[j * 68 + threadIdx.x];
      const float mb = sum / (float)nb;
      float m2b = 0.f;
      for (int j = 0; j < nb; ++j) {
        const float dv = Ps[j * 68 + threadIdx.x] - mb;
        m2b = fmaf(dv, dv, m2b);
      }
      chan_merge(n, mean, M2, (float)nb, mb, m2b);
    }
  }
  if (threadIdx.x < kTile) {
    float* o = spart + ((size_t)bh * S + sp) * 3 * mp + a0 + threadIdx.x;
    o[0] = n;
    o[mp] = mean;
    o[2 * mp] = M2;
  }
}

template <int D, typename T>
static cudaError_t qstats_t(const Prob& p, const void* q, const float* L, float* spart,
                            cudaStream_t st) {
  const size_t smem = (2 * (size_t)tile_floats(D) + 64 * 68) * sizeof(float);
  if (p.gauss()) {
    static bool once = (allow_smem(k_qstats<D, T, true>, smem), true);
    (void)once;
    return launch("qstats", k_qstats<D, T, true>, dim3(p.nt, p.Sq, p.BH), dim3(kThreads), smem,
                  st, (const T*)q, L, spart, p.N, p.m, p.mp, p.Sq, p.nblk, p.ns);
  }
  static bool once = (allow_smem(k_qstats<D, T, false>, smem), true);
  (void)once;
  return launch("qstats", k_qstats<D, T, false>, dim3(p.nt, p.Sq, p.BH), dim3(kThreads), smem, st,
                (const T*)q, L, spart, p.N, p.m, p.mp, p.Sq, p.nblk, p.ns);
}

cudaError_t run_qstats(const Prob& p, const void* q, const float* L, float* spart, cudaStream_t st) {
  DISPATCH_DT(qstats_t, p, q, L, spart, st);
}

// The same partial triples from kernel values P already in memory ([BH][N][mp],
// as the query pass stores them for the backward): per 64-token block, the
// block's 64 x 64 tile is staged in shared memory and reduced exactly as above,
// so the partials are bit-identical to the pass that forms P itself.
// grid (landmark tile, split, slice)
__global__ void __launch_bounds__(kThreads) k_pstats(const float* __restrict__ P,
                                                     float* __restrict__ spart, int N, int mp,
                                                     int S, int nblk) {
  __shared__ float Ps[kTile * 68];
  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * kTile;
  const float* Pb = P + (size_t)bh * N * mp + a0;
  float n = 0.f, mean = 0.f, M2 = 0.f;
  int b0, b1;
  split_range(nblk, S, sp, b0, b1);
  for (int b = b0; b < b1; ++b) {
    const int nb = min(kTile, N - b * kTile);
    __syncthreads();
    for (int id = threadIdx.x; id < nb * (kTile / 4); id += kThreads) {
      const int j = id / (kTile / 4), c4 = id % (kTile / 4);
      st4(Ps + j * 68 + 4 * c4, ld4(Pb + (size_t)(b * kTile + j) * mp + 4 * c4));
    }
    __syncthreads();
    if (threadIdx.x < kTile) {
      float sum = 0.f;
      for (int j = 0; j < nb; ++j) sum += Ps[j * 68 + threadIdx.x];
      const float mb = sum / (float)nb;
      float m2b = 0.f;
      for (int j = 0; j < nb; ++j) {
        const float dv = Ps[j * 68 + threadIdx.x] - mb;
        m2b = fmaf(dv, dv, m2b);
      }
      chan_merge(n, mean, M2, (float)nb, mb, m2b);
    }
  }
  if (threadIdx.x < kTile) {
    float* o = spart + ((size_t)bh * S + sp) * 3 * mp + a0 + threadIdx.x;
    o[0] = n;
    o[mp] = mean;
    o[2 * mp] = M2;
  }
}

cudaError_t run_pstats(const Prob& p, const float* P, float* spart, cudaStream_t st) {
  return launch("pstats", k_pstats, dim3(p.nt, p.Sq, p.BH), dim3(kThreads), 0, st, P, spart, p.N,
                p.mp, p.Sq, p.nblk);
}

// Z = (P - mu) / sqrt(var + eta) per landmark column (the normalised feature map),
// 0 past m; P and Z [BH][N][mp], stats [BH][3][m].  Four columns a thread.
__global__ void k_zmap(const float* __restrict__ P, const float* __restrict__ stats,
                       float* __restrict__ Z, int N, int m, int mp, long long n4) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n4) return;
  const int per = mp / 4;
  const long long row = e / per;
  const int a = 4 * (int)(e - row * per);
  const int bh = (int)(row / N);
  const float* sb = stats + (size_t)bh * 3 * m;
  const float4 pv = ld4(P + 4 * e);
  const float in[4] = {pv.x, pv.y, pv.z, pv.w};
  float out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) out[q] = a + q < m ? (in[q] - sb[a + q]) * sb[2 * m + a + q] : 0.f;
  st4(Z + 4 * e, make_float4(out[0], out[1], out[2], out[3]));
}

cudaError_t run_zmap(const Prob& p, const float* P, const float* stats, float* Z, cudaStream_t st) {
  const long long n4 = (long long)p.BH * p.N * p.mp / 4;
  return launch("zmap", k_zmap, dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, st, P, stats, Z,
                p.N, p.m, p.mp, n4);
}

// Statistics are taken per slice, or (batch-pooled) over the B slices of a
// head: group g < H, member r < B is slice r H + g.
//
// stats [BH][3][m]: mu, var (biased), 1 / sqrt(var + 1e-5).  Per slice: one
// thread per (slice, landmark) merges its splits in order.
__global__ void k_stats_final(const float* __restrict__ spart, float* __restrict__ stats, int BH,
                              int S, int m, int mp, int N) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= BH * m) return;
  const int bh = e / m, a = e % m;
  float n = 0.f, mean = 0.f, M2 = 0.f;
  for (int s = 0; s < S; ++s) {
    const float* o = spart + ((size_t)bh * S + s) * 3 * mp + a;
    chan_merge(n, mean, M2, o[0], o[mp], o[2 * mp]);
  }
  const float var = M2 / (float)N;
  float* st = stats + (size_t)bh * 3 * m;
  st[a] = mean;
  st[m + a] = var;
  st[2 * m + a] = 1.0f / sqrtf(var + 1e-5f);
}

// Batch-pooled: CTA (head g, 32 landmarks), 32 rows of 32 lanes; row y merges
// the (member, split) partials y, y + 32, ... in order, then row 0 merges the
// 32 row results in order (a fixed tree: deterministic), and all rows write the
// result to every member.
constexpr int kGrpRows = 32;
__global__ void __launch_bounds__(32 * kGrpRows)
    k_stats_final_grouped(const float* __restrict__ spart, float* __restrict__ stats, int H, int R,
                          int S, int m, int mp, int N) {
  __shared__ float sn[kGrpRows][32], smean[kGrpRows][32], sM2[kGrpRows][32];
  const int g = blockIdx.x, a = blockIdx.y * 32 + threadIdx.x, y = threadIdx.y;
  float n = 0.f, mean = 0.f, M2 = 0.f;
  if (a < m) {
    for (int i = y; i < R * S; i += kGrpRows) {
      const int r = i / S, s = i - r * S;
      const float* o = spart + ((size_t)(r * H + g) * S + s) * 3 * mp + a;
      chan_merge(n, mean, M2, o[0], o[mp], o[2 * mp]);
    }
  }
  sn[y][threadIdx.x] = n;
  smean[y][threadIdx.x] = mean;
  sM2[y][threadIdx.x] = M2;
  __syncthreads();
  if (y == 0) {
    for (int j = 1; j < kGrpRows; ++j)
      chan_merge(n, mean, M2, sn[j][threadIdx.x], smean[j][threadIdx.x], sM2[j][threadIdx.x]);
    smean[0][threadIdx.x] = mean;
    sM2[0][threadIdx.x] = M2 / ((float)N * (float)R);
  }
  __syncthreads();
  if (a >= m) return;
  mean = smean[0][threadIdx.x];
  const float var = sM2[0][threadIdx.x];
  const float rs = 1.0f / sqrtf(var + 1e-5f);
  for (int r = y; r < R; r += kGrpRows) {
    float* st = stats + (size_t)(r * H + g) * 3 * m;
    st[a] = mean;
    st[m + a] = var;
    st[2 * m + a] = rs;
  }
}

cudaError_t run_stats_final(const Prob& p, const float* spart, float* stats, cudaStream_t st) {
  if (p.norm_batch() && p.B > 1)
    return launch("stats_final", k_stats_final_grouped, dim3(p.H, (p.m + 31) / 32),
                  dim3(32, kGrpRows), 0, st, spart, stats, p.H, p.B, p.Sq, p.m, p.mp, p.N);
  const int n = p.BH * p.m;
  return launch("stats_final", k_stats_final, dim3((n + 255) / 256), dim3(256), 0, st, spart, stats,
                p.BH, p.Sq, p.m, p.mp, p.N);
}

// ===========================================================================
// query pass: grid (token block, slice).  Each CTA keeps 64 queries in shared
// memory and walks the landmark tiles (the next landmark and W-hat tiles are
// copied in with cp.async, double buffered): P tile on the fly, optional
// centring/whitening, then O += Z_tile W-hat_tile.
// ===========================================================================
template <int D, typename T, bool NORM, bool GAUSS>
__global__ void __launch_bounds__(kThreads, 2)
    k_query_fwd(const T* __restrict__ Q, const float* __restrict__ L, const float* __restrict__ What,
                const float* __restrict__ stats, T* __restrict__ O, float* __restrict__ kvout,
                int N, int m, int nt, float ns) {
  constexpr int CPT = D / 16;
  // bf16 inputs: O += Z W-hat runs on the tensor cores (TF32)
  constexpr bool kTC = TypeOf<T>::id == 1 && D >= 32;
  constexpr int NCT = D / 16;
  extern __shared__ float4 sm4[];
  float* Xs = reinterpret_cast<float*>(sm4);
  float* LW = Xs + tile_floats(D);          // two buffers of (landmark tile, W-hat tile)
  float* Pt = LW + 4 * tile_floats(D);      // [64 landmarks][68 tokens] (tensor-core path: [64 tokens][68 landmarks])
  __shared__ float mu_s[kTile], rs_s[kTile];
  const int b = blockIdx.x, bh = blockIdx.y;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tg = lane & 3;
  const int wj = (warp & 3) * 16, wc = (warp >> 2) * (D / 2);  // tensor-core fragment origin
  const T* Qb = Q + (size_t)bh * N * D;
  // O null: only the kernel values P go out (to kvout), no contraction
  const bool ponly = O == nullptr;
  load_tile<D>(Xs, Qb, b * kTile, N);
  float o[4][CPT];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < CPT; ++c) o[r][c] = 0.f;
  float acc[NCT][4];
#pragma unroll
  for (int n = 0; n < NCT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  // landmark and W-hat rows of tile lt into buffer lt % 2 (fp32 rows land in
  // the padded tiles directly), zero past m
  auto prefetch = [&](int lt) {
    if (lt >= nt) return;
    float* Lsb = LW + (lt & 1) * 2 * tile_floats(D);
    float* Wsb = Lsb + tile_floats(D);
    const int a0 = lt * kTile;
    for (int id = threadIdx.x; id < (ponly ? 1 : 2) * kTile * (D / 4); id += kThreads) {
      const int which = id / (kTile * (D / 4)), rem = id % (kTile * (D / 4));
      const int r = rem / (D / 4), c4 = rem % (D / 4);
      const bool ok = a0 + r < m;
      const float* src = (which ? What : L) + ((size_t)bh * m + (ok ? a0 + r : 0)) * D + 4 * c4;
      cp_async16(smem_addr((which ? Wsb : Lsb) + r * row_stride(D) + 4 * c4), src, ok);
    }
    cp_commit();
  };
  prefetch(0);
  for (int lt = 0; lt < nt; ++lt) {
    const int a0 = lt * kTile;
    const float* Ls = LW + (lt & 1) * 2 * tile_floats(D);
    const float* Ws = Ls + tile_floats(D);
    cp_wait_all();
    __syncthreads();  // tile lt has landed; every reader of the other buffer is done
    prefetch(lt + 1);
    if (NORM && threadIdx.x < kTile) {
      const int a = a0 + threadIdx.x;
      mu_s[threadIdx.x] = a < m ? stats[(size_t)bh * 3 * m + a] : 0.f;
      rs_s[threadIdx.x] = a < m ? stats[(size_t)bh * 3 * m + 2 * m + a] : 0.f;
    }
    __syncthreads();
    float dist[4][4];
    dist_tile<D, GAUSS>(Xs, Ls, dist);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int a = tx + 16 * s;
        float pv = 0.f;
        if (a0 + a < m) pv = exp2_ftz(dist[r][s] * ns);
        // keep the kernel value (before normalisation) for the backward
        const int j = b * kTile + 4 * ty + r;
        if (kvout && j < N) kvout[((size_t)bh * N + j) * (nt * kTile) + a0 + a] = pv;
        if (ponly) continue;
        if (NORM && a0 + a < m) pv = (pv - mu_s[a]) * rs_s[a];
        if (kTC)
          Pt[(4 * ty + r) * 68 + a] = pv;
        else
          Pt[a * 68 + 4 * ty + r] = pv;
      }
    if (ponly) continue;  // uniform over the CTA
    __syncthreads();
    if constexpr (kTC) {
      // O += Z W-hat on the tensor cores with both factors split into TF32 hi + lo
      // (Z_hi W_hi + Z_hi W_lo + Z_lo W_hi): fp32-level accuracy
#pragma unroll 2
      for (int k0 = 0; k0 < kTile; k0 += 8) {
        const float zv[4] = {Pt[(wj + gq) * 68 + k0 + tg], Pt[(wj + gq + 8) * 68 + k0 + tg],
                             Pt[(wj + gq) * 68 + k0 + tg + 4], Pt[(wj + gq + 8) * 68 + k0 + tg + 4]};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ah[i] = to_tf32(zv[i]);
          al[i] = to_tf32(zv[i] - __uint_as_float(ah[i]));
        }
#pragma unroll
        for (int n = 0; n < NCT; ++n) {
          const float w0 = Ws[(k0 + tg) * row_stride(D) + wc + 8 * n + gq];
          const float w1 = Ws[(k0 + tg + 4) * row_stride(D) + wc + 8 * n + gq];
          uint32_t bh[2], bl[2];
          bh[0] = to_tf32(w0);
          bh[1] = to_tf32(w1);
          bl[0] = to_tf32(w0 - __uint_as_float(bh[0]));
          bl[1] = to_tf32(w1 - __uint_as_float(bh[1]));
          mma_16x8x8(acc[n], ah, bh);
          mma_16x8x8(acc[n], ah, bl);
          mma_16x8x8(acc[n], al, bh);
        }
      }
    } else {
#pragma unroll 4
      for (int a = 0; a < kTile; ++a) {
        const float4 p4 = lds4(Pt + a * 68 + 4 * ty);
        float wv[CPT];
        lds_cpt<CPT>(Ws + a * row_stride(D) + tx * CPT, wv);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          o[0][c] = fmaf(p4.x, wv[c], o[0][c]);
          o[1][c] = fmaf(p4.y, wv[c], o[1][c]);
          o[2][c] = fmaf(p4.z, wv[c], o[2][c]);
          o[3][c] = fmaf(p4.w, wv[c], o[3][c]);
        }
      }
    }
  }
  if (ponly) return;
  if constexpr (kTC) {
    const int j1 = b * kTile + wj + gq, j2 = j1 + 8;
#pragma unroll
    for (int n = 0; n < NCT; ++n) {
      const int c = wc + 8 * n + 2 * tg;
      if (j1 < N) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(acc[n][0], acc[n][1]);
        *reinterpret_cast<__nv_bfloat162*>(O + ((size_t)bh * N + j1) * D + c) = v;
      }
      if (j2 < N) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(acc[n][2], acc[n][3]);
        *reinterpret_cast<__nv_bfloat162*>(O + ((size_t)bh * N + j2) * D + c) = v;
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = b * kTile + 4 * ty + r;
      if (j < N) st_cpt<CPT>(O + ((size_t)bh * N + j) * D + tx * CPT, o[r]);
    }
  }
}

template <int D, typename T>
static cudaError_t query_fwd_t(const Prob& p, const void* q, const float* L, const float* What,
                               const float* stats, void* out, float* kvout, cudaStream_t st) {
  const size_t smem = (5 * (size_t)tile_floats(D) + 64 * 68) * sizeof(float);
  dim3 grid(p.nblk, p.BH);
#define QF_LAUNCH(NN, GG)                                                                      \
  do {                                                                                         \
    static bool once = (allow_smem(k_query_fwd<D, T, NN, GG>, smem), true);                    \
    (void)once;                                                                                \
    return launch(out ? "query_fwd" : "query_p", k_query_fwd<D, T, NN, GG>, grid, dim3(kThreads), \
                  smem, st, (const T*)q, L, What, stats, (T*)out, kvout, p.N, p.m, p.nt, p.ns); \
  } while (0)
  if (p.norm()) {
    if (p.gauss()) QF_LAUNCH(true, true);
    QF_LAUNCH(true, false);
  }
  if (p.gauss()) QF_LAUNCH(false, true);
  QF_LAUNCH(false, false);
#undef QF_LAUNCH
}

cudaError_t run_query_fwd(const Prob& p, const void* q, const float* L, const float* What,
                          const float* stats, void* out, float* kvout, cudaStream_t st) {
  DISPATCH_DT(query_fwd_t, p, q, L, What, stats, out, kvout, st);
}

// ===========================================================================
// backward tile kernel, grid (landmark tile, split, slice).
//
// For a token block X (queries or keys, 64 rows) against the CTA's 64
// landmarks, with kv_ja = k(X_j, L_a) recomputed on the fly and
// dot_ja = U_j . R_a (U = dO, R = W-hat on the query side; U = V, R = dW on
// the key side), the upstream weight g_ja is
//   query side: g = dP * P / lambda, dP = dZ (no norm) or the centring/whitening
//               reverse (dZ - mean dZ - Z mean(dZ Z)) / sqrt(var + eta), dZ = dot
//   key side:   g = dC * C / lambda, dC = dot
// and, since dk(x, l)/dx_c = -(k / lambda) sgn(x_c - l_c),
//   token side    dX_jc = -sum_a g_ja sgn(X_jc - L_ac)   (per landmark tile)
//   landmark side dL_ac += sum_j g_ja sgn(X_jc - L_ac)   (accumulated over the split)
// plus dW-hat_a = sum_j Z_ja dO_j (query side) and dV_j = sum_a C_ja dW_a
// (key side, per landmark tile).  MODE 0 is the query-side statistics pass of
// the normalised map (sum dZ, sum dZ Z and dW-hat only).
// ===========================================================================
template <int D, typename T, int MODE, bool NORM, bool GAUSS>
__global__ void __launch_bounds__(kThreads, 2)
    k_bwd_tile(const T* __restrict__ X, const T* __restrict__ U, const float* __restrict__ L,
               const float* __restrict__ R, const float* __restrict__ stats,
               const float* __restrict__ mdz, float* __restrict__ tok_part,
               float* __restrict__ tok_part2, float* __restrict__ lm_part,
               float* __restrict__ lm_part2, float* __restrict__ ns_part, int N, int m, int mp,
               int S, int nblk, int BH, float ns, float inv_lam) {
  constexpr int CPT = D / 16;
  constexpr bool kTokenSide = MODE != 0;
  constexpr bool kDWhat = (MODE == 0) || (MODE == 1 && !NORM);
  extern __shared__ float4 sm4[];
  float* Ls = reinterpret_cast<float*>(sm4);
  float* Rs = Ls + tile_floats(D);
  float* Xs = Rs + tile_floats(D);
  float* Us = Xs + tile_floats(D);
  float* Gs = Us + tile_floats(D);  // [64 tokens][68]: g
  float* Zs = Gs + 64 * 68;         // [64 tokens][68]: Z (query side) or C (key side)
  __shared__ float mu_s[kTile], rs_s[kTile], m0_s[kTile], m1_s[kTile];

  const int lt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
  const int a0 = lt * kTile;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const T* Xb = X + (size_t)bh * N * D;
  const T* Ub = U + (size_t)bh * N * D;
  load_tile<D>(Ls, L + (size_t)bh * m * D, a0, m);
  load_tile<D>(Rs, R + (size_t)bh * m * D, a0, m);
  if (NORM && threadIdx.x < kTile) {
    const int a = a0 + threadIdx.x;
    const float* stb = stats + (size_t)bh * 3 * m;
    mu_s[threadIdx.x] = a < m ? stb[a] : 0.f;
    rs_s[threadIdx.x] = a < m ? stb[2 * m + a] : 0.f;
    if (MODE == 1) {
      m0_s[threadIdx.x] = mdz[(size_t)bh * 2 * mp + a0 + threadIdx.x];
      m1_s[threadIdx.x] = mdz[(size_t)bh * 2 * mp + mp + a0 + threadIdx.x];
    }
  }
  __syncthreads();

  // landmark-side registers: thread owns landmarks 4 ty + s, columns tx * CPT + c
  float lreg[4][CPT], dl[4][CPT], dw[4][CPT];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    lds_cpt<CPT>(Ls + (4 * ty + s) * row_stride(D) + tx * CPT, lreg[s]);
#pragma unroll
    for (int c = 0; c < CPT; ++c) dl[s][c] = dw[s][c] = 0.f;
  }
  float sdz[4] = {0.f, 0.f, 0.f, 0.f}, sdzz[4] = {0.f, 0.f, 0.f, 0.f};

  int b0, b1;
  split_range(nblk, S, sp, b0, b1);
  for (int b = b0; b < b1; ++b) {
    __syncthreads();
    load_tile<D>(Xs, Xb, b * kTile, N);
    load_tile<D>(Us, Ub, b * kTile, N);
    __syncthreads();

    // ---- phase 1: distances and dots, thread = 4 tokens x 4 landmarks ----
    float dist[4][4], dot[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) dist[r][s] = dot[r][s] = 0.f;
#pragma unroll 2
    for (int c = 0; c < D; c += 4) {
      float4 x[4], l[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) x[r] = lds4(Xs + (4 * ty + r) * row_stride(D) + c);
#pragma unroll
      for (int s = 0; s < 4; ++s) l[s] = lds4(Ls + (tx + 16 * s) * row_stride(D) + c);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) dist4_add<GAUSS>(dist[r][s], x[r], l[s]);
#pragma unroll
      for (int r = 0; r < 4; ++r) x[r] = lds4(Us + (4 * ty + r) * row_stride(D) + c);
#pragma unroll
      for (int s = 0; s < 4; ++s) l[s] = lds4(Rs + (tx + 16 * s) * row_stride(D) + c);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          dot[r][s] = fmaf(x[r].x, l[s].x, dot[r][s]);
          dot[r][s] = fmaf(x[r].y, l[s].y, dot[r][s]);
          dot[r][s] = fmaf(x[r].z, l[s].z, dot[r][s]);
          dot[r][s] = fmaf(x[r].w, l[s].w, dot[r][s]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int jl = 4 * ty + r, al = tx + 16 * s;
        const bool valid = (b * kTile + jl < N) && (a0 + al < m);
        const float kv = exp2_ftz(dist[r][s] * ns);
        float g = 0.f, zc = 0.f;
        if (MODE == 2) {
          g = dot[r][s] * kv * inv_lam;
          zc = kv;
        } else {
          const float z = NORM ? (kv - mu_s[al]) * rs_s[al] : kv;
          zc = z;
          if (MODE == 0) {
            if (valid) {
              sdz[s] += dot[r][s];
              sdzz[s] = fmaf(dot[r][s], z, sdzz[s]);
            }
          } else {
            const float dp = NORM ? (dot[r][s] - m0_s[al] - z * m1_s[al]) * rs_s[al] : dot[r][s];
            g = dp * kv * inv_lam;
          }
        }
        Gs[jl * 68 + al] = valid ? g : 0.f;
        Zs[jl * 68 + al] = valid ? zc : 0.f;
      }
    __syncthreads();

    // ---- phase A: token side, thread = 4 tokens x CPT columns ----
    if (kTokenSide) {
      float xr[4][CPT], tq[4][CPT], tv[4][CPT];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        lds_cpt<CPT>(Xs + (4 * ty + r) * row_stride(D) + tx * CPT, xr[r]);
#pragma unroll
        for (int c = 0; c < CPT; ++c) tq[r][c] = tv[r][c] = 0.f;
      }
#pragma unroll 2
      for (int a = 0; a < kTile; ++a) {
        float lv[CPT], gr[4];
        lds_cpt<CPT>(Ls + a * row_stride(D) + tx * CPT, lv);
#pragma unroll
        for (int r = 0; r < 4; ++r) gr[r] = Gs[(4 * ty + r) * 68 + a];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < CPT; ++c) tq[r][c] += sgn_times(xr[r][c] - lv[c], gr[r]);
        if (MODE == 2) {
          float rv[CPT], cr[4];
          lds_cpt<CPT>(Rs + a * row_stride(D) + tx * CPT, rv);
#pragma unroll
          for (int r = 0; r < 4; ++r) cr[r] = Zs[(4 * ty + r) * 68 + a];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < CPT; ++c) tv[r][c] = fmaf(cr[r], rv[c], tv[r][c]);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = b * kTile + 4 * ty + r;
        if (j < N) {
          const size_t off = (((size_t)lt * BH + bh) * N + j) * D + tx * CPT;
#pragma unroll
          for (int c = 0; c < CPT; ++c) tq[r][c] = -tq[r][c];
          st_cpt<CPT>(tok_part + off, tq[r]);
          if (MODE == 2) st_cpt<CPT>(tok_part2 + off, tv[r]);
        }
      }
    }

    // ---- phase B: landmark side, thread = 4 landmarks x CPT columns ----
#pragma unroll 2
    for (int j = 0; j < kTile; ++j) {
      if (kTokenSide) {
        float xv[CPT];
        lds_cpt<CPT>(Xs + j * row_stride(D) + tx * CPT, xv);
        const float4 g4 = lds4(Gs + j * 68 + 4 * ty);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          dl[0][c] += sgn_times(xv[c] - lreg[0][c], g4.x);
          dl[1][c] += sgn_times(xv[c] - lreg[1][c], g4.y);
          dl[2][c] += sgn_times(xv[c] - lreg[2][c], g4.z);
          dl[3][c] += sgn_times(xv[c] - lreg[3][c], g4.w);
        }
      }
      if (kDWhat) {
        float uv[CPT];
        lds_cpt<CPT>(Us + j * row_stride(D) + tx * CPT, uv);
        const float4 z4 = lds4(Zs + j * 68 + 4 * ty);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          dw[0][c] = fmaf(z4.x, uv[c], dw[0][c]);
          dw[1][c] = fmaf(z4.y, uv[c], dw[1][c]);
          dw[2][c] = fmaf(z4.z, uv[c], dw[2][c]);
          dw[3][c] = fmaf(z4.w, uv[c], dw[3][c]);
        }
      }
    }
  }

  const size_t lo = (((size_t)bh * S + sp) * mp + a0 + 4 * ty) * D + tx * CPT;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if (kTokenSide) st_cpt<CPT>(lm_part + lo + (size_t)s * D, dl[s]);
    if (kDWhat) st_cpt<CPT>(lm_part2 + lo + (size_t)s * D, dw[s]);
  }
  if (MODE == 0) {
    // per-landmark sums over the 16 token rows of threads, through the g / Z tiles
    float* red0 = Gs;  // [16][64]
    float* red1 = Zs;  // [16][64]
    __syncthreads();
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      red0[ty * kTile + tx + 16 * s] = sdz[s];
      red1[ty * kTile + tx + 16 * s] = sdzz[s];
    }
    __syncthreads();
    if (threadIdx.x < kTile) {
      float s0 = 0.f, s1 = 0.f;
      for (int q = 0; q < 16; ++q) {
        s0 += red0[q * kTile + threadIdx.x];
        s1 += red1[q * kTile + threadIdx.x];
      }
      float* o = ns_part + ((size_t)bh * S + sp) * 2 * mp + a0 + threadIdx.x;
      o[0] = s0;
      o[mp] = s1;
    }
  }
}

template <int D, typename T, int MODE, bool NORM, bool GAUSS>
static cudaError_t bwd_tile_t2(const Prob& p, const BwdArgs& a, cudaStream_t st) {
  const size_t smem = (4 * (size_t)tile_floats(D) + 2 * 64 * 68) * sizeof(float);
  static bool once = (allow_smem(k_bwd_tile<D, T, MODE, NORM, GAUSS>, smem), true);
  (void)once;
  static const char* names[3] = {"bwd_qstats", "bwd_query", "bwd_key"};
  return launch(names[MODE], k_bwd_tile<D, T, MODE, NORM, GAUSS>, dim3(p.nt, p.Sb, p.BH), dim3(kThreads),
                smem, st, (const T*)a.X, (const T*)a.U, a.L, a.R, a.stats, a.mdz, a.tok_part,
                a.tok_part2, a.lm_part, a.lm_part2, a.ns_part, p.N, p.m, p.mp, p.Sb, p.nblk, p.BH,
                p.ns, p.inv_lam);
}

// only the statistics pass (mode 0) of this kernel is used; the token-side
// modes run in k_bwd_pair (k_bwd.cu)
template <int D, typename T>
static cudaError_t bwd_tile_t(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st) {
  if (mode != 0) return cudaErrorInvalidValue;
  if (p.gauss()) return bwd_tile_t2<D, T, 0, true, true>(p, a, st);
  return bwd_tile_t2<D, T, 0, true, false>(p, a, st);
}

cudaError_t run_bwd_tile(const Prob& p, int mode, const BwdArgs& a, cudaStream_t st) {
  DISPATCH_DT(bwd_tile_t, p, mode, a, st);
}

// mdz [BH][2][mp]: (1/N) sum dZ and (1/N) sum dZ Z per landmark, fixed order over splits
__global__ void k_mdz(const float* __restrict__ ns_part, float* __restrict__ mdz, int BH, int S, int mp,
                      int N) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= BH * mp) return;
  const int bh = e / mp, a = e % mp;
  float s0 = 0.f, s1 = 0.f;
  for (int s = 0; s < S; ++s) {
    const float* o = ns_part + ((size_t)bh * S + s) * 2 * mp + a;
    s0 += o[0];
    s1 += o[mp];
  }
  mdz[(size_t)bh * 2 * mp + a] = s0 / (float)N;
  mdz[(size_t)bh * 2 * mp + mp + a] = s1 / (float)N;
}

// Batch-pooled: the same two means over the B * N queries of head g, summed
// with the fixed tree of k_stats_final_grouped and written to every member.
__global__ void __launch_bounds__(32 * kGrpRows)
    k_mdz_grouped(const float* __restrict__ ns_part, float* __restrict__ mdz, int H, int R, int S,
                  int mp, int N) {
  __shared__ float p0[kGrpRows][32], p1[kGrpRows][32];
  const int g = blockIdx.x, a = blockIdx.y * 32 + threadIdx.x, y = threadIdx.y;
  float s0 = 0.f, s1 = 0.f;
  for (int i = y; i < R * S; i += kGrpRows) {
    const int r = i / S, s = i - r * S;
    const float* o = ns_part + ((size_t)(r * H + g) * S + s) * 2 * mp + a;
    s0 += o[0];
    s1 += o[mp];
  }
  p0[y][threadIdx.x] = s0;
  p1[y][threadIdx.x] = s1;
  __syncthreads();
  if (y == 0) {
    for (int j = 1; j < kGrpRows; ++j) {
      s0 += p0[j][threadIdx.x];
      s1 += p1[j][threadIdx.x];
    }
    const float n = (float)N * (float)R;
    p0[0][threadIdx.x] = s0 / n;
    p1[0][threadIdx.x] = s1 / n;
  }
  __syncthreads();
  s0 = p0[0][threadIdx.x];
  s1 = p1[0][threadIdx.x];
  for (int r = y; r < R; r += kGrpRows) {
    float* o = mdz + (size_t)(r * H + g) * 2 * mp;
    o[a] = s0;
    o[mp + a] = s1;
  }
}

cudaError_t run_mdz(const Prob& p, const float* ns_part, float* mdz, cudaStream_t st) {
  if (p.norm_batch() && p.B > 1)
    return launch("mdz", k_mdz_grouped, dim3(p.H, p.mp / 32), dim3(32, kGrpRows), 0, st, ns_part,
                  mdz, p.H, p.B, p.Sb, p.mp, p.N);
  const int n = p.BH * p.mp;
  return launch("mdz", k_mdz, dim3((n + 255) / 256), dim3(256), 0, st, ns_part, mdz, p.BH, p.Sb, p.mp,
                p.N);
}

// dL[bh][a][c] = sum_s dLq + sum_s dLc + dLA (fixed order)
// dL of every landmark (split partials of both sides in order, plus the gram
// path), divided by its window's token count: the share the pool backward
// gives each token of the window
__global__ void k_reduce_dl(const float* __restrict__ dLq, const float* __restrict__ dLc,
                            const float* __restrict__ dLA, float* __restrict__ dLs, int BH, int S,
                            int m, int mp, int d, int gh, int gw, int mh, int mw) {
  const size_t total = (size_t)BH * m * d;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = e / ((size_t)m * d), ac = e % ((size_t)m * d);
    const size_t base = bh * S * mp * d + ac;
    float s = 0.f;
    for (int q = 0; q < S; ++q) s += dLq[base + (size_t)q * mp * d];
    for (int q = 0; q < S; ++q) s += dLc[base + (size_t)q * mp * d];
    const int a = (int)(ac / d), wi = a / mw, wj = a - wi * mw;
    const float inv = 1.0f / (float)(((wi + 1) * gh / mh - wi * gh / mh) *
                                     ((wj + 1) * gw / mw - wj * gw / mw));
    dLs[e] = (s + dLA[e]) * inv;
  }
}

cudaError_t run_reduce_dl(const Prob& p, int S, const float* dLq, const float* dLc, const float* dLA,
                          float* dLs, cudaStream_t st) {
  const size_t n = (size_t)p.BH * p.m * p.d;
  return launch("reduce_dl", k_reduce_dl, dim3(grid_for(n)), dim3(kThreads), 0, st, dLq, dLc, dLA,
                dLs, p.BH, S, p.m, p.mp, p.d, p.gh, p.gw, p.mh, p.mw);
}

// token gradients: sum the per-landmark-tile partials in tile order, add the
// pooling path dLs[a(n)] (dL / window size) to dK, convert to the tensor type.
template <typename T>
__global__ void k_finalize(const float* __restrict__ dQp, const float* __restrict__ dKp,
                           const float* __restrict__ dVp, const float* __restrict__ dLs,
                           const int32_t* __restrict__ idx, T* __restrict__ dq, T* __restrict__ dk,
                           T* __restrict__ dv, int BH, int N, int d, int nt, int m, int tied) {
  const size_t total4 = (size_t)BH * N * d / 4;
  const size_t plane = (size_t)BH * N * d;
  for (size_t e4 = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e4 < total4;
       e4 += (size_t)gridDim.x * blockDim.x) {
    const size_t e = e4 * 4;
    const size_t row = e / d;
    const int c = (int)(e % d);
    const int n = (int)(row % N);
    const size_t bh = row / N;
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4, v4 = q4;
    for (int t = 0; t < nt; ++t) {
      const float4 a = *reinterpret_cast<const float4*>(dQp + t * plane + e);
      const float4 b = *reinterpret_cast<const float4*>(dKp + t * plane + e);
      const float4 v = *reinterpret_cast<const float4*>(dVp + t * plane + e);
      q4.x += a.x; q4.y += a.y; q4.z += a.z; q4.w += a.w;
      k4.x += b.x; k4.y += b.y; k4.z += b.z; k4.w += b.w;
      v4.x += v.x; v4.y += v.y; v4.z += v.z; v4.w += v.w;
    }
    // the token's pooling window: its landmark's dL, already divided by the
    // window's size
    const float4 l4 = __ldg(reinterpret_cast<const float4*>(dLs + (bh * m + __ldg(idx + n)) * d + c));
    k4.x += l4.x; k4.y += l4.y; k4.z += l4.z; k4.w += l4.w;
    if (tied) {
      q4.x += k4.x; q4.y += k4.y; q4.z += k4.z; q4.w += k4.w;
      st4(dq + e, q4);
    } else {
      st4(dq + e, q4);
      st4(dk + e, k4);
    }
    st4(dv + e, v4);
  }
}

// token gradients of the tensor-core backward: dK = the sum of its nk partial
// planes (landmark groups, in order) plus the pooling path dL[a(n)] / window size;
// dQ the sum of its nq planes (nq = 0: dq was written by the tile kernel); dV
// one fp32 plane (null: dv was written already); tied: dq = dQ + dK; all
// converted to the tensor type.
// 8 consecutive values of T from two float4 (one 16-byte store for bf16)
__device__ __forceinline__ void st8(float* p, float4 a, float4 b) {
  st4(p, a);
  st4(p + 4, b);
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, float4 a, float4 b) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
  *reinterpret_cast<uint4*>(p) =
      make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                 *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_finalize_tc(
    const float* __restrict__ dQp, const float* __restrict__ dKp, const float* __restrict__ dVp,
    const float* __restrict__ dLs, const int32_t* __restrict__ idx, T* __restrict__ dq,
    T* __restrict__ dk, T* __restrict__ dv, int BH, int N, int d, int c8shift, int nq, int nk,
    int m, int tied) {
  // thread = (token n, 8 consecutive features), 32-bit index arithmetic; the
  // token's landmark from the pool's index map, its share of dL pre-divided
  const int C8 = d >> 3;
  const int per = N * C8;
  const size_t plane = (size_t)BH * N * d;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    for (int id = blockIdx.x * blockDim.x + threadIdx.x; id < per; id += gridDim.x * blockDim.x) {
      const int n = id >> c8shift, c = (id & (C8 - 1)) * 8;
      const size_t e = ((size_t)bh * N + n) * d + c;
      const int a = __ldg(idx + n);
      const float* lp = dLs + ((size_t)bh * m + a) * d + c;
      float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0;
      float4 k0 = __ldg(reinterpret_cast<const float4*>(lp));
      float4 k1 = __ldg(reinterpret_cast<const float4*>(lp + 4));
      for (int t = 0; t < nk; ++t) {
        k0 = add4(k0, __ldcs(reinterpret_cast<const float4*>(dKp + t * plane + e)));
        k1 = add4(k1, __ldcs(reinterpret_cast<const float4*>(dKp + t * plane + e + 4)));
      }
      for (int t = 0; t < nq; ++t) {
        q0 = add4(q0, __ldcs(reinterpret_cast<const float4*>(dQp + t * plane + e)));
        q1 = add4(q1, __ldcs(reinterpret_cast<const float4*>(dQp + t * plane + e + 4)));
      }
      if (tied) {
        st8(dq + e, add4(q0, k0), add4(q1, k1));
      } else {
        if (nq > 0) st8(dq + e, q0, q1);
        st8(dk + e, k0, k1);
      }
      if (dVp != nullptr)
        st8(dv + e, __ldcs(reinterpret_cast<const float4*>(dVp + e)),
            __ldcs(reinterpret_cast<const float4*>(dVp + e + 4)));
    }
  }
}

cudaError_t run_finalize_tc(const Prob& p, int nq, const float* dQp, int nk, const float* dKp,
                            const float* dVp, const float* dLs, const int32_t* idx, void* dq,
                            void* dk, void* dv, cudaStream_t st) {
  const int C8 = p.d / 8;
  int c8shift = 0;
  while ((1 << c8shift) < C8) ++c8shift;
  const long long per = (long long)p.N * C8;
  const int bx = (int)((per + kThreads - 1) / kThreads);
  dim3 grid(bx < 1024 ? bx : 1024, p.BH < 65535 ? p.BH : 65535);
  if (p.dtype == 1)
    return launch("finalize", k_finalize_tc<__nv_bfloat16>, grid, dim3(kThreads), 0, st, dQp, dKp,
                  dVp, dLs, idx, (__nv_bfloat16*)dq, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, p.BH,
                  p.N, p.d, c8shift, nq, nk, p.m, p.tied);
  return launch("finalize", k_finalize_tc<float>, grid, dim3(kThreads), 0, st, dQp, dKp, dVp, dLs,
                idx, (float*)dq, (float*)dk, (float*)dv, p.BH, p.N, p.d, c8shift, nq, nk, p.m,
                p.tied);
}

cudaError_t run_finalize(const Prob& p, const float* dQp, const float* dKp, const float* dVp,
                         const float* dLs, const int32_t* idx, void* dq, void* dk, void* dv,
                         cudaStream_t st) {
  const size_t n4 = (size_t)p.BH * p.N * p.d / 4;
  if (p.dtype == 1)
    return launch("finalize", k_finalize<__nv_bfloat16>, dim3(grid_for(n4)), dim3(kThreads), 0, st,
                  dQp, dKp, dVp, dLs, idx, (__nv_bfloat16*)dq, (__nv_bfloat16*)dk,
                  (__nv_bfloat16*)dv, p.BH, p.N, p.d, p.nt, p.m, p.tied);
  return launch("finalize", k_finalize<float>, dim3(grid_for(n4)), dim3(kThreads), 0, st, dQp, dKp,
                dVp, dLs, idx, (float*)dq, (float*)dk, (float*)dv, p.BH, p.N, p.d, p.nt, p.m,
                p.tied);
}

// zero-fill (used when the Newton-Schulz backward has no step to initialise dA)
__global__ void k_zero(float* __restrict__ x, size_t n) {
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x)
    x[e] = 0.f;
}

cudaError_t run_zero(float* x, size_t n, cudaStream_t st) {
  return launch("zero", k_zero, dim3(grid_for(n)), dim3(kThreads), 0, st, x, n);
}

}  // namespace lapnys
