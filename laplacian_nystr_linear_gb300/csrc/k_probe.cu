// FP32 FMA-rate probe (instrumentation, no part of the method): the measured
// counterpart of the ALU peak that the benchmark's roofline divides by.
#include "common.cuh"
#include "internal.h"

//
// Every thread runs 8 independent FMA chains x <- x * a + b (|a| < 1, so values
// stay bounded), scalar or as packed pairs (fma.rn.f32x2); the result is written
// only if it takes an impossible value, which keeps the chains live without
// memory traffic.
namespace lapnys {
namespace {
constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 8;

template <bool PAIRED>
__global__ void __launch_bounds__(kProbeThreads) k_fma_probe(int iters, float* sink) {
  const float a = 0.999f, b = 1e-3f * (float)(threadIdx.x & 7);
  if constexpr (PAIRED) {
    f32x2 x[8];
    const f32x2 av = pack2(a, a), bv = pack2(b, -b);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = pack2((float)k, (float)threadIdx.x);
    for (int i = 0; i < iters; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = fma2(x[k], av, bv);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 v = unpack2(x[k]);
      s += v.x + v.y;
    }
    if (s == -1234.5f) sink[0] = s;
  } else {
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (float)(k + threadIdx.x);
    for (int i = 0; i < iters; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = fmaf(x[k], a, b);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += x[k];
    if (s == -1234.5f) sink[0] = s;
  }
}
}  // namespace

cudaError_t run_fma_probe(bool paired, int iters, float* sink, unsigned long long* lane_ops,
                          cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = sms * kProbeCtasPerSm;
  *lane_ops = (unsigned long long)grid * kProbeThreads * (unsigned long long)iters * 8ull *
              (paired ? 2ull : 1ull);
  if (paired)
    return launch("fma_probe", k_fma_probe<true>, dim3(grid), dim3(kProbeThreads), 0, st, iters, sink);
  return launch("fma_probe", k_fma_probe<false>, dim3(grid), dim3(kProbeThreads), 0, st, iters, sink);
}

}  // namespace lapnys
