// C ABI of liblapnys: argument checks, ctx / workspace layout, and the launch
// sequences of the forward and backward passes of Laplacian-kernel Nystrom
// attention (see include/lapnys.h for the contract).
#include <math.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/lapnys.h"
#include "common.cuh"
#include "internal.h"

namespace lapnys {

// ---------------------------------------------------------------------------
// instrumentation
// ---------------------------------------------------------------------------
namespace {
constexpr int kMaxRec = 4096;
struct Rec {
  const char* name;
  cudaEvent_t a, b;
};
bool g_prof = false;
bool g_serial = false;  // profile mode 2: everything on the caller's stream
std::vector<Rec> g_rec;
int g_used = 0;
uint64_t g_launches = 0;
}  // namespace

int prof_begin(const char* name, cudaStream_t s) {
  if (!g_prof || g_used >= kMaxRec) return -1;
  if ((int)g_rec.size() <= g_used) {
    Rec r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return -1;
    g_rec.push_back(r);
  }
  Rec& r = g_rec[g_used];
  r.name = name;
  if (cudaEventRecord(r.a, s) != cudaSuccess) return -1;
  return g_used++;
}

void prof_end(int slot, cudaStream_t s) {
  if (slot >= 0) cudaEventRecord(g_rec[slot].b, s);
}

void count_launch() { ++g_launches; }

// ---------------------------------------------------------------------------
// problem description and memory layout
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int isqrt_exact(int m) {
  int r = (int)lrint(sqrt((double)m));
  while (r * r > m) --r;
  while ((r + 1) * (r + 1) <= m) ++r;
  return r * r == m ? r : -1;
}

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

// The mh x mw landmark grid of m landmarks on a gh x gw token grid (average
// pooling: "LaplacianFormer", Arabic summary 2c.1; "SOFT" review, Proposed
// method).  Reading: a square m keeps mh = mw = sqrt(m); any other m takes the
// factor pair shaped most like the token grid (smallest |log(mh / mw) -
// log(gh / gw)|, ties to the smaller mh).  Window row i spans token rows
// [floor(i gh / mh), floor((i + 1) gh / mh)), columns alike: a partition of the
// grid (adaptive pooling without overlap when the grid is not divisible).
// False when the grid has fewer rows or columns than the landmark grid.
static bool landmark_grid(int gh, int gw, int m, int* mh, int* mw) {
  if (gh <= 0 || gw <= 0 || m <= 0) return false;
  int a = isqrt_exact(m), b = a;
  if (a < 0) {
    double best = 0.0;
    a = -1;
    const double target = log((double)gh / (double)gw);
    for (int f = 1; f <= m; ++f) {
      if (m % f) continue;
      const double key = fabs(log((double)f / (double)(m / f)) - target);
      if (a < 0 || key < best - 1e-12) {
        best = key;
        a = f;
        b = m / f;
      }
    }
  }
  if (a > gh || b > gw) return false;
  *mh = a;
  *mw = b;
  return true;
}

// token splits so that each pass has roughly 8 CTAs per SM of a 152-SM part;
// depends on the dimensions only, so results do not depend on the device.
static int splits_for(int nblk, int nt, int BH) {
  const int target = 1216;
  int s = ceil_div(target, nt * BH);
  if (s > nblk) s = nblk;
  if (s < 1) s = 1;
  return s;
}

static bool dims_ok(int B, int H, int N, int d, int m, int iters) {
  if (B <= 0 || H <= 0 || N <= 0 || m <= 0 || m > N || iters < 0 || iters > 64) return false;
  if (d <= 0) return false;
  if (m > 1024) return false;
  if ((long long)B * H * N * d >= (1LL << 31)) return false;
  return true;
}

static bool d_supported(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

static Prob make_prob(int B, int H, int N, int d, int gh, int gw, int m, float lam, float eps,
                      int iters, int tied, int dtype, unsigned flags) {
  Prob p;
  memset(&p, 0, sizeof(p));
  p.B = B; p.H = H; p.BH = B * H; p.N = N; p.d = d; p.gh = gh; p.gw = gw; p.m = m;
  if (!landmark_grid(gh, gw, m, &p.mh, &p.mw)) p.mh = p.mw = 0;
  p.iters = iters; p.tied = tied; p.dtype = dtype; p.flags = flags;
  p.lam = lam; p.eps = eps;
  p.ns = (float)(-1.4426950408889634 / (double)lam);
  p.inv_lam = (float)(1.0 / (double)lam);
  p.nt = ceil_div(m, kTile);
  p.mp = p.nt * kTile;
  p.nblk = ceil_div(N, kTile);
  p.Sk = splits_for(p.nblk, p.nt, p.BH);
  p.Sq = p.Sk;
  p.Sb = p.Sk;
  // sized from the shape alone (the workspace query takes no dtype); used for bf16
  p.Skt = fwd_tc_shape(d, m) ? key_tc_splits(p.BH, m, p.nblk) : 0;
  // splits of the tensor-core backward (bf16, d = 64); sized from the shape alone
  p.Stc = bwd_tc_splits(p.BH, m, N);
  return p;
}

struct CtxLayout {
  size_t L, Llo, A, alpha, X, Y, W, What, stats, idx, P, C, total;
  int nx, ny;
};

static CtxLayout ctx_layout(int BH, int N, int d, int m, int iters, bool full) {
  CtxLayout c;
  c.nx = full ? iters + 1 : 2;
  c.ny = full ? (iters > 0 ? iters : 1) : 1;
  const size_t f = sizeof(float);
  size_t o = 0;
  c.L = o; o = align256(o + (size_t)BH * m * d * f);
  c.Llo = o; o = align256(o + (size_t)BH * m * d * f);
  c.A = o; o = align256(o + (size_t)BH * m * m * f);
  c.alpha = o; o = align256(o + (size_t)BH * 4 * f);
  c.X = o; o = align256(o + (size_t)BH * c.nx * m * m * f);
  c.Y = o; o = align256(o + (size_t)BH * c.ny * m * m * f);
  c.W = o; o = align256(o + (size_t)BH * m * d * f);
  c.What = o; o = align256(o + (size_t)BH * m * d * f);
  c.stats = o; o = align256(o + (size_t)BH * 3 * m * f);
  c.idx = o; o = align256(o + (size_t)N * sizeof(int32_t));
  // kernel values of both passes, kept for the backward (full layout only)
  const size_t mp = (size_t)(m + kTile - 1) / kTile * kTile;
  c.P = o; o = align256(o + (full ? (size_t)BH * N * mp * f : 0));
  c.C = o; o = align256(o + (full ? (size_t)BH * N * mp * f : 0));
  c.total = o;
  return c;
}

struct WsLayout {
  size_t lite;                                 // ctx stand-in when the forward gets no ctx
  size_t kpart, spart, fpack;                  // forward partials, packed query-pass tiles
  size_t dWhp, dLqp, dLcp, nsp, mdz;           // backward landmark-side partials
  size_t dQp, dKp, dVp;                        // backward token-side partials
  size_t dWh, dW, dLA, dL, G, XG, Tm, dA;      // backward landmark-side results
  size_t ties, tie_scratch;                    // tie records (query, key) and their scratch
  size_t dvimg;                                // R^T operand image of the streaming C R product
  size_t zmap;                                 // normalised feature map Z (m <= 64, ctx kept)
  size_t total;
};

static WsLayout ws_layout(const Prob& p) {
  WsLayout w;
  const size_t f = sizeof(float);
  const size_t BH = p.BH, m = p.m, d = p.d, mp = p.mp;
  const size_t Sb = (size_t)(p.Stc > p.Sb ? p.Stc : p.Sb);  // either backward's splits
  size_t o = 0;
  w.lite = o; o = align256(o + ctx_layout(p.BH, p.N, p.d, p.m, p.iters, false).total);
  w.kpart = o; o = align256(o + BH * (p.Skt > p.Sk ? p.Skt : p.Sk) * mp * d * f);
  w.spart = o; o = align256(o + BH * p.Sq * 3 * mp * f);
  w.fpack = o; o = align256(o + (p.Skt > 0 ? pack_q_floats(p) * f : 0));
  w.dWhp = o; o = align256(o + BH * Sb * mp * d * f);
  w.dLqp = o; o = align256(o + BH * Sb * mp * d * f);
  w.dLcp = o; o = align256(o + BH * Sb * mp * d * f);
  w.nsp = o; o = align256(o + BH * Sb * 2 * mp * f);
  w.mdz = o; o = align256(o + BH * 2 * mp * f);
  const size_t tok = (size_t)p.nt * BH * p.N * d * f;
  w.dQp = o; o = align256(o + tok);
  w.dKp = o; o = align256(o + tok);
  w.dVp = o; o = align256(o + tok);
  w.dWh = o; o = align256(o + BH * m * d * f);
  w.dW = o; o = align256(o + BH * m * d * f);
  w.dLA = o; o = align256(o + BH * m * d * f);
  w.dL = o; o = align256(o + BH * m * d * f);
  w.G = o; o = align256(o + BH * m * m * f);
  w.XG = o; o = align256(o + BH * m * m * f);
  w.Tm = o; o = align256(o + BH * m * m * f);
  w.dA = o; o = align256(o + BH * m * m * f);
  w.ties = o; o = align256(o + 2 * BH * (size_t)((p.N + 31) / 32) * kTieRec * 4);
  w.tie_scratch = o; o = align256(o + ties_scratch_bytes(p.BH, p.m, p.d));
  // sized from the shape alone (the size queries know no element type)
  w.dvimg = o; o = align256(o + (d == 32 || d == 64 ? dv_image_floats(p) * f : 0));
  w.zmap = o;
  o = align256(o + ((d == 32 || d == 64) && p.norm() && m <= kTile ? BH * p.N * mp * f : 0));
  w.total = o;
  return w;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static int check_common(int B, int H, int N, int d, int gh, int gw, int m, float lam, float eps,
                        int iters, int dtype, unsigned flags) {
  if (!dims_ok(B, H, N, d, m, iters)) return LAPNYS_EINVAL;
  if (gh <= 0 || gw <= 0 || (long long)gh * gw != N) return LAPNYS_EINVAL;
  int mh = 0, mw = 0;
  if (!landmark_grid(gh, gw, m, &mh, &mw)) return LAPNYS_EINVAL;
  if (!(lam > 0.f) || !isfinite(lam)) return LAPNYS_EINVAL;
  if (!(eps >= 0.f) || !isfinite(eps)) return LAPNYS_EINVAL;
  if (dtype != LAPNYS_F32 && dtype != LAPNYS_BF16) return LAPNYS_EINVAL;
  if ((flags & ~(unsigned)(LAPNYS_NORM | LAPNYS_GAUSS | LAPNYS_NORM_BATCH)) != 0)
    return LAPNYS_EINVAL;
  if ((flags & LAPNYS_NORM_BATCH) && !(flags & LAPNYS_NORM)) return LAPNYS_EINVAL;
  if (!d_supported(d)) return LAPNYS_ENOTSUP;
  return LAPNYS_OK;
}

int check_attention(int B, int H, int N, int d, int gh, int gw, int m, float lam, float eps,
                    int iters, int dtype, unsigned flags) {
  return check_common(B, H, N, d, gh, gw, m, lam, eps, iters, dtype, flags);
}

#define CK(x)                                  \
  do {                                         \
    if ((x) != cudaSuccess) return LAPNYS_ECUDA; \
  } while (0)

// ---------------------------------------------------------------------------
// Newton-Schulz for m > 64 via batched products (X slots: nx, Y slots: ny)
// ---------------------------------------------------------------------------
// One batched product of the Newton-Schulz solver: on the tensor cores
// (three-term TF32 split, fp32-level accuracy) when the shapes and pointers are
// 4-element aligned, otherwise on the FP32 FMA kernel.
static cudaError_t ns_mm(const Prob& p, bool ta, bool tb, int M, int N, int K, const float* A,
                         int lda, long sA, const float* B, int ldb, long sB, float* C, int ldc,
                         long sC, const float* E, int lde, long sE, float alpha, float beta,
                         cudaStream_t st) {
  if (tc_gemm_ok(M, N, K, lda, ldb, ldc, lde, sA, sB, sC, sE, A, B, C, beta != 0.f ? E : nullptr))
    return run_tcgemm(ta, tb, p.BH, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, E, lde, sE, alpha,
                      beta, st);
  return run_gemm2(ta, tb, false, p.BH, M, N, A, lda, sA, B, ldb, sB, K, nullptr, 0, 0, nullptr, 0,
                   0, 0, C, ldc, sC, E, lde, sE, alpha, beta, st);
}

static int ns_forward_large(const Prob& p, const float* A, float* X, float* Y, int nx, int ny,
                            cudaStream_t st) {
  const int m = p.m;
  const long mm = (long)m * m;
  if (ns_cluster_ok(m)) {
    // every iteration of every slice in one launch (a cluster per slice)
    CK(run_ns_cluster(p, false, A, X, Y, nx, ny, nullptr, nullptr, nullptr, nullptr, st));
    return LAPNYS_OK;
  }
  for (int t = 0; t < p.iters; ++t) {
    float* Xt = X + (long)(t % nx) * mm;
    float* Xn = X + (long)((t + 1) % nx) * mm;
    float* Yt = Y + (long)(t % ny) * mm;
    // Y_t = A X_t, computed in full: forcing this product to be exactly
    // symmetric makes the fp32 iteration diverge in its unconverged directions
    CK(ns_mm(p, false, false, m, m, m, A, m, mm, Xt, m, nx * mm, Yt, m, ny * mm, nullptr, m, 0, 1.f,
             0.f, st));
    // X_{t+1} = 2 X_t - X_t Y_t.  The FMA kernel writes it symmetric (upper
    // tiles mirrored; stable: the residual I - A X_{t+1} = (I - A X_t)^2 keeps
    // contracting); the tensor-core kernel computes it in full.
    if (tc_gemm_ok(m, m, m, m, m, m, m, nx * mm, ny * mm, nx * mm, nx * mm, Xt, Yt, Xn, Xt)) {
      CK(run_tcgemm(false, false, p.BH, m, m, m, Xt, m, nx * mm, Yt, m, ny * mm, Xn, m, nx * mm, Xt,
                    m, nx * mm, -1.f, 2.f, st));
    } else {
      CK(run_gemm2(false, false, true, p.BH, m, m, Xt, m, nx * mm, Yt, m, ny * mm, m, nullptr, 0, 0,
                   nullptr, 0, 0, 0, Xn, m, nx * mm, Xt, m, nx * mm, -1.f, 2.f, st));
    }
  }
  return LAPNYS_OK;
}

}  // namespace lapnys

using namespace lapnys;

// ---------------------------------------------------------------------------
// Side stream: the Newton-Schulz kernels of a slice set fill one cluster of
// 1-2 SMs per slice (64 of 152 SMs for the benchmark), while the key-side
// backward does not depend on their reverse (it needs dW, not dA).  lapnys_bwd
// therefore runs the solver's reverse and the gram backward on a per-device
// stream of the highest priority (its clusters get their SMs first) and the
// key-side tile kernel on the caller's stream, joined by events.  (The
// forward's key pass could run beside the forward iteration the same way, but
// measured no faster: both slow each other down by about what the overlap
// saves.)  Enqueueing is serialised per device so the shared events stay
// consistent.
// ---------------------------------------------------------------------------
namespace {
constexpr int kMaxSideDevices = 256;
struct Side {
  cudaStream_t hi = nullptr;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  std::mutex mu;
};
Side g_side[kMaxSideDevices];
std::mutex g_side_init_mu;

// the current device's side stream and events, created on first use; null if
// they cannot be created (the caller then stays on one stream)
Side* side() {
  if (g_serial) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
  Side& sd = g_side[dev];
  std::lock_guard<std::mutex> lock(g_side_init_mu);
  if (sd.hi == nullptr) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    for (int i = 0; i < 2; ++i)
      if (sd.ev[i] == nullptr && cudaEventCreateWithFlags(&sd.ev[i], cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return nullptr;
    sd.hi = s;
  }
  return &sd;
}

// make `to` wait for everything enqueued on `from` so far
cudaError_t join(cudaStream_t to, cudaStream_t from, cudaEvent_t ev) {
  cudaError_t e = cudaEventRecord(ev, from);
  if (e != cudaSuccess) return e;
  return cudaStreamWaitEvent(to, ev, 0);
}
}  // namespace

// ---------------------------------------------------------------------------
// Built-in forward scratch for callers that cannot allocate device memory.
// 32 MiB of device memory per GPU that loads this library, held until exit.
// Host code must not hand the array's name to a kernel (on the host it is a
// stand-in, not a device address): lapnys_fwd_static looks the device address
// up with cudaGetSymbolAddress on every call, with the caller's device and
// context current.  The address belongs to a context, not to a device ordinal
// (a reset device or another context on the same device has its own copy), so
// nothing is cached; the lookup is a host-side query that allocates nothing.
// ---------------------------------------------------------------------------
static constexpr size_t kStaticScratchBytes = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_fwd_scratch[kStaticScratchBytes];

namespace {
// address of g_fwd_scratch in the current context
cudaError_t static_scratch(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_fwd_scratch);
  if (e != cudaSuccess) return e;
  *out = ptr;
  return cudaSuccess;
}
}  // namespace

extern "C" {

const char* lapnys_strerror(int status) {
  switch (status) {
    case LAPNYS_OK: return "ok";
    case LAPNYS_EINVAL: return "invalid argument (dimension, pointer, alignment or parameter)";
    case LAPNYS_ECUDA: return "CUDA launch failed";
    case LAPNYS_ETIMEOUT: return "bounded device wait expired";
    case LAPNYS_ENOSPC: return "ctx or workspace buffer too small";
    case LAPNYS_ENOTSUP: return "unsupported configuration (d must be 16, 32, 64 or 128)";
    case LAPNYS_ESCRATCH:
      return "problem needs more scratch than the 32 MiB built into lapnys_fwd_static; "
             "call lapnys_fwd with a caller-owned workspace";
  }
  return "unknown status";
}

size_t lapnys_ctx_bytes(int B, int H, int N, int d, int m, int iters, unsigned flags) {
  (void)flags;
  if (!dims_ok(B, H, N, d, m, iters)) return 0;
  return ctx_layout(B * H, N, d, m, iters, true).total;
}

size_t lapnys_workspace_bytes(int B, int H, int N, int d, int m, int iters, unsigned flags) {
  if (!dims_ok(B, H, N, d, m, iters)) return 0;
  // the workspace depends on the sizes only, not on the grid's shape
  Prob p = make_prob(B, H, N, d, 1, N, m, 1.f, 0.f, iters, 0, 0, flags);
  return ws_layout(p).total;
}

int lapnys_ctx_offsets(int B, int H, int N, int d, int m, int iters, unsigned flags,
                       lapnys_ctx_layout* out) {
  (void)flags;
  if (out == nullptr || !dims_ok(B, H, N, d, m, iters)) return LAPNYS_EINVAL;
  const CtxLayout c = ctx_layout(B * H, N, d, m, iters, true);
  out->L = c.L; out->Llo = c.Llo; out->A = c.A; out->alpha = c.alpha; out->X = c.X; out->Y = c.Y;
  out->W = c.W; out->What = c.What; out->stats = c.stats; out->idx = c.idx; out->P = c.P;
  out->C = c.C; out->total = c.total;
  return LAPNYS_OK;
}

int lapnys_pool(const void* k, float* L, int32_t* idx, int B, int H, int N, int d, int grid_h,
                int grid_w, int m, int dtype, cudaStream_t stream) {
  NvtxScope nvtx_scope("lapnys_pool");
  int rc = check_common(B, H, N, d, grid_h, grid_w, m, 1.f, 0.f, 0, dtype, 0);
  if (rc != LAPNYS_OK) return rc;
  if (k == nullptr || L == nullptr || !aligned16(k) || !aligned16(L)) return LAPNYS_EINVAL;
  Prob p = make_prob(B, H, N, d, grid_h, grid_w, m, 1.f, 0.f, 0, 0, dtype, 0);
  CK(run_pool(p, k, L, nullptr, idx, stream));
  return LAPNYS_OK;
}

int lapnys_fwd(const void* q, const void* k, const void* v, void* out, int B, int H, int N, int d,
               int grid_h, int grid_w, int m, float lambda, float eps, int iters, int tied_qk,
               cudaStream_t stream, int dtype, unsigned flags, void* ctx, size_t ctx_bytes,
               void* ws, size_t ws_bytes) {
  NvtxScope nvtx_scope("lapnys_fwd");
  int rc = check_common(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, dtype, flags);
  if (rc != LAPNYS_OK) return rc;
  if (tied_qk != 0 && tied_qk != 1) return LAPNYS_EINVAL;
  if (tied_qk) {
    if (k != nullptr && k != q) return LAPNYS_EINVAL;
    k = q;
  }
  if (!q || !k || !v || !out || !ws) return LAPNYS_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws))
    return LAPNYS_EINVAL;
  if (ctx != nullptr && !aligned16(ctx)) return LAPNYS_EINVAL;
  Prob p = make_prob(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, tied_qk, dtype, flags);
  const WsLayout w = ws_layout(p);
  if (ws_bytes < w.total) return LAPNYS_ENOSPC;
  const bool full = ctx != nullptr;
  const CtxLayout c = ctx_layout(p.BH, N, d, m, iters, full);
  if (full && ctx_bytes < c.total) return LAPNYS_ENOSPC;

  char* cb = full ? (char*)ctx : (char*)ws + w.lite;
  char* wb = (char*)ws;
  float* L = (float*)(cb + c.L);
  float* Llo = (float*)(cb + c.Llo);
  float* A = (float*)(cb + c.A);
  float* alpha = (float*)(cb + c.alpha);
  float* X = (float*)(cb + c.X);
  float* Y = (float*)(cb + c.Y);
  float* W = (float*)(cb + c.W);
  float* What = (float*)(cb + c.What);
  float* stats = (float*)(cb + c.stats);
  int32_t* idx = (int32_t*)(cb + c.idx);
  const long mm = (long)m * m;

  CK(run_pool(p, k, L, Llo, idx, stream));
  // the solver (landmark matrix, alpha, Newton-Schulz) on the side stream,
  // queued first so that its CTAs take their SMs at once; the key pass on this
  // stream meanwhile; both end before W-hat = X_T W
  Side* sd = side();
  std::unique_lock<std::mutex> lock;
  if (sd) lock = std::unique_lock<std::mutex>(sd->mu);
  const cudaStream_t ss = sd ? sd->hi : stream;
  if (sd) CK(join(ss, stream, sd->ev[0]));
  if (m <= kTile) {
    CK(run_ns_small(p, L, A, alpha, X, Y, c.nx, c.ny, ss));
  } else {
    CK(run_gram(p, L, A, ss));
    CK(run_alpha(p, A, alpha, X, c.nx * mm, ss));
    rc = ns_forward_large(p, A, X, Y, c.nx, c.ny, ss);
    if (rc != LAPNYS_OK) return rc;
  }
  float* kpart = (float*)(wb + w.kpart);
  const bool tc = fwd_tc_ok(p);
  if (tc) {
    if (p.gauss())
      CK(run_key_gtc(p, k, v, L, kpart, full ? (float*)(cb + c.C) : nullptr, stream));
    else
      CK(run_key_tc(p, k, v, L, kpart, full ? (float*)(cb + c.C) : nullptr, stream));
    CK(run_reduce_parts(p.BH, p.Skt, m, p.mp, d, kpart, W, stream));
  } else {
    CK(run_key_fwd(p, k, v, L, kpart, full ? (float*)(cb + c.C) : nullptr, stream));
    CK(run_reduce_parts(p.BH, p.Sk, m, p.mp, d, kpart, W, stream));
  }
  // With a ctx kept, the query pass's kernel values P = k(Q, L) (which the ctx
  // keeps for the backward) and the feature map's statistics do not depend on
  // the solver: on the FMA path they are formed here, beside it (the statistics
  // from the stored P, Z = (P - mu) / sqrt(var + eta) into the workspace), and
  // O = Z W-hat is the streaming product once W-hat exists.
  const bool split_q = full && !tied_qk && !tc && dv_tc_ok(p);
  const float* Zq = (const float*)(cb + c.P);
  if (split_q) {
    CK(run_query_fwd(p, q, L, nullptr, stats, nullptr, (float*)(cb + c.P), stream));
    if (p.norm()) {
      float* spart = (float*)(wb + w.spart);
      float* Z = (float*)(wb + w.zmap);
      CK(run_pstats(p, (const float*)(cb + c.P), spart, stream));
      CK(run_stats_final(p, spart, stats, stream));
      CK(run_zmap(p, (const float*)(cb + c.P), stats, Z, stream));
      Zq = Z;
    }
  }
  if (sd) CK(join(stream, ss, sd->ev[1]));
  const float* XT = X + (long)(iters % c.nx) * mm;
  // W-hat = X_T W
  CK(ns_mm(p, false, false, m, d, m, XT, m, c.nx * mm, W, d, (long)m * d, What, d, (long)m * d,
           nullptr, d, 0, 1.f, 0.f, stream));
  if (split_q) {
    CK(run_dv(p, Zq, What, (float*)(wb + w.dvimg), out, "query_product", stream));
    return LAPNYS_OK;
  }
  // Q = K: P = k(Q, L) is C^T, and the key pass has just stored C token-major
  // (the layout of P).  Without a feature map the query pass is then the product
  // O = C W-hat, read once from ctx instead of recomputing the distances; the
  // backward reads C as P (a tied forward stores no separate P).
  if (full && tied_qk && !p.norm() && dv_tc_ok(p)) {
    CK(run_dv(p, (const float*)(cb + c.C), What, (float*)(wb + w.dvimg), out, "query_shared",
              stream));
    return LAPNYS_OK;
  }
  float* Pout = full && !tied_qk ? (float*)(cb + c.P) : nullptr;
  if (p.norm()) {
    float* spart = (float*)(wb + w.spart);
    CK(run_qstats(p, q, L, spart, stream));
    CK(run_stats_final(p, spart, stats, stream));
  }
  if (tc) {
    float* fpack = (float*)(wb + w.fpack);
    if (p.gauss()) {
      float* packW = fpack + (size_t)p.BH * p.nt * (64 * d + 64);
      CK(run_pack_qg(p, L, What, fpack, packW, stream));
      CK(run_query_gtc(p, q, fpack, packW, stats, out, Pout, stream));
    } else {
      CK(run_pack_q(p, L, What, fpack, stream));
      CK(run_query_tc(p, q, fpack, stats, out, Pout, stream));
    }
  } else {
    CK(run_query_fwd(p, q, L, What, stats, out, Pout, stream));
  }
  return LAPNYS_OK;
}

int lapnys_fwd_static(const void* q, const void* k, const void* v, void* out, int B, int H, int N,
                      int d, int grid_h, int grid_w, int m, float lambda, float eps, int iters,
                      int tied_qk, cudaStream_t stream, int dtype, unsigned flags) {
  int rc = check_common(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, dtype, flags);
  if (rc != LAPNYS_OK) return rc;
  if (tied_qk != 0 && tied_qk != 1) return LAPNYS_EINVAL;
  if (tied_qk) {
    if (k != nullptr && k != q) return LAPNYS_EINVAL;
    k = q;
  }
  if (!q || !k || !v || !out) return LAPNYS_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LAPNYS_EINVAL;
  Prob p = make_prob(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, tied_qk, dtype, flags);
  const WsLayout w = ws_layout(p);
  // the forward uses the leading part of the workspace layout: the stand-in
  // for the saved state and the key-pass / statistics partials
  if (w.dWhp > kStaticScratchBytes) return LAPNYS_ESCRATCH;
  void* ws = nullptr;
  CK(static_scratch(&ws));
  const CtxLayout c = ctx_layout(p.BH, N, d, m, iters, false);
  char* cb = (char*)ws + w.lite;
  char* wb = (char*)ws;
  float* L = (float*)(cb + c.L);
  float* Llo = (float*)(cb + c.Llo);
  float* A = (float*)(cb + c.A);
  float* alpha = (float*)(cb + c.alpha);
  float* X = (float*)(cb + c.X);
  float* Y = (float*)(cb + c.Y);
  float* W = (float*)(cb + c.W);
  float* What = (float*)(cb + c.What);
  float* stats = (float*)(cb + c.stats);
  int32_t* idx = (int32_t*)(cb + c.idx);
  const long mm = (long)m * m;
  // every scratch region below is fully written before it is read, so nothing
  // left over from an earlier call needs clearing
  CK(run_pool(p, k, L, Llo, idx, stream));
  if (m <= kTile) {
    CK(run_ns_small(p, L, A, alpha, X, Y, c.nx, c.ny, stream));
  } else {
    CK(run_gram(p, L, A, stream));
    CK(run_alpha(p, A, alpha, X, c.nx * mm, stream));
    rc = ns_forward_large(p, A, X, Y, c.nx, c.ny, stream);
    if (rc != LAPNYS_OK) return rc;
  }
  float* kpart = (float*)(wb + w.kpart);
  const bool tc = fwd_tc_ok(p);
  if (tc) {
    if (p.gauss())
      CK(run_key_gtc(p, k, v, L, kpart, nullptr, stream));
    else
      CK(run_key_tc(p, k, v, L, kpart, nullptr, stream));
    CK(run_reduce_parts(p.BH, p.Skt, m, p.mp, d, kpart, W, stream));
  } else {
    CK(run_key_fwd(p, k, v, L, kpart, nullptr, stream));
    CK(run_reduce_parts(p.BH, p.Sk, m, p.mp, d, kpart, W, stream));
  }
  const float* XT = X + (long)(iters % c.nx) * mm;
  CK(ns_mm(p, false, false, m, d, m, XT, m, c.nx * mm, W, d, (long)m * d, What, d, (long)m * d,
           nullptr, d, 0, 1.f, 0.f, stream));
  if (p.norm()) {
    float* spart = (float*)(wb + w.spart);
    CK(run_qstats(p, q, L, spart, stream));
    CK(run_stats_final(p, spart, stats, stream));
  }
  if (tc) {
    float* fpack = (float*)(wb + w.fpack);
    if (p.gauss()) {
      float* packW = fpack + (size_t)p.BH * p.nt * (64 * d + 64);
      CK(run_pack_qg(p, L, What, fpack, packW, stream));
      CK(run_query_gtc(p, q, fpack, packW, stats, out, nullptr, stream));
    } else {
      CK(run_pack_q(p, L, What, fpack, stream));
      CK(run_query_tc(p, q, fpack, stats, out, nullptr, stream));
    }
  } else {
    CK(run_query_fwd(p, q, L, What, stats, out, nullptr, stream));
  }
  return LAPNYS_OK;
}

int lapnys_bwd(const void* q, const void* k, const void* v, const void* dout, const void* ctx,
               void* dq, void* dk, void* dv, int B, int H, int N, int d, int grid_h, int grid_w,
               int m, float lambda, float eps, int iters, int tied_qk, cudaStream_t stream,
               int dtype, unsigned flags, void* ws, size_t ws_bytes) {
  NvtxScope nvtx_scope("lapnys_bwd");
  int rc = check_common(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, dtype, flags);
  if (rc != LAPNYS_OK) return rc;
  if (tied_qk != 0 && tied_qk != 1) return LAPNYS_EINVAL;
  if (tied_qk) {
    if (k != nullptr && k != q) return LAPNYS_EINVAL;
    if (dk != nullptr) return LAPNYS_EINVAL;
    k = q;
  } else if (dk == nullptr || !aligned16(dk)) {
    return LAPNYS_EINVAL;
  }
  if (!q || !k || !v || !dout || !ctx || !dq || !dv || !ws) return LAPNYS_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(ctx) ||
      !aligned16(dq) || !aligned16(dv) || !aligned16(ws))
    return LAPNYS_EINVAL;
  Prob p = make_prob(B, H, N, d, grid_h, grid_w, m, lambda, eps, iters, tied_qk, dtype, flags);
  const WsLayout w = ws_layout(p);
  if (ws_bytes < w.total) return LAPNYS_ENOSPC;
  const CtxLayout c = ctx_layout(p.BH, N, d, m, iters, true);

  const char* cb = (const char*)ctx;
  char* wb = (char*)ws;
  const float* L = (const float*)(cb + c.L);
  const float* Llo = (const float*)(cb + c.Llo);
  const float* A = (const float*)(cb + c.A);
  const float* alpha = (const float*)(cb + c.alpha);
  const float* X = (const float*)(cb + c.X);
  const float* Y = (const float*)(cb + c.Y);
  const float* W = (const float*)(cb + c.W);
  const float* What = (const float*)(cb + c.What);
  const float* stats = (const float*)(cb + c.stats);
  const int32_t* idx = (const int32_t*)(cb + c.idx);
  float* dWhp = (float*)(wb + w.dWhp);
  float* dLqp = (float*)(wb + w.dLqp);
  float* dLcp = (float*)(wb + w.dLcp);
  float* nsp = (float*)(wb + w.nsp);
  float* mdz = (float*)(wb + w.mdz);
  float* dQp = (float*)(wb + w.dQp);
  float* dKp = (float*)(wb + w.dKp);
  float* dVp = (float*)(wb + w.dVp);
  float* dWh = (float*)(wb + w.dWh);
  float* dW = (float*)(wb + w.dW);
  float* dLA = (float*)(wb + w.dLA);
  float* dL = (float*)(wb + w.dL);
  float* G = (float*)(wb + w.G);
  float* XG = (float*)(wb + w.XG);
  float* Tm = (float*)(wb + w.Tm);
  float* dA = (float*)(wb + w.dA);
  const long mm = (long)m * m;
  const long md = (long)m * d;

  // the query side's kernel values P: a tied forward stores none, C^T is P then
  const float* Pm = (const float*)(cb + (tied_qk ? c.C : c.P));

  // which 32-token blocks need the exact sign path (a value tied with a
  // landmark value, or out of the fast path's range)
  uint32_t* ties_q = (uint32_t*)(wb + w.ties);
  uint32_t* ties_k = tied_qk ? ties_q : ties_q + (size_t)p.BH * ((N + 31) / 32) * kTieRec;
  if (!p.gauss()) {  // the Gaussian kernel's gradient has no sign term, hence no ties
    CK(run_tie_prep(p, L, wb + w.tie_scratch, stream));
    CK(run_ties(p, q, wb + w.tie_scratch, ties_q, stream));
    if (!tied_qk) CK(run_ties(p, k, wb + w.tie_scratch, ties_k, stream));
  }

  // the bf16, d = 64 backward finishes each token's gradient in one CTA per
  // group of 256 landmarks (tensor-core dot products, no per-tile partials)
  const bool tcb = bwd_tc_shape(p.dtype, d);
  const int ng = bwd_tc_groups(m);
  const int Sl = tcb ? p.Stc : p.Sb;  // splits of the landmark-side partials
  const bool dq_direct = tcb && !tied_qk && ng == 1;

  // ---- query side ----
  BwdArgs qa;
  memset(&qa, 0, sizeof(qa));
  qa.X = q; qa.U = dout; qa.L = L; qa.Llo = Llo; qa.R = What; qa.stats = stats; qa.mdz = mdz;
  qa.tok_part = dQp; qa.lm_part = dLqp; qa.lm_part2 = dWhp; qa.ns_part = nsp; qa.ties = ties_q;
  qa.kv = Pm;
  if (p.norm()) {
    CK(run_bwd_tile(p, 0, qa, stream));
    CK(run_mdz(p, nsp, mdz, stream));
    CK(run_reduce_parts(p.BH, p.Sb, m, p.mp, d, dWhp, dWh, stream));
  }
  if (tcb) {
    BwdTcArgs qt;
    memset(&qt, 0, sizeof(qt));
    qt.X = q; qt.U = dout; qt.L = L; qt.Llo = Llo; qt.R = What; qt.stats = stats; qt.mdz = mdz;
    qt.kv = Pm; qt.ties = ties_q; qt.out = dq_direct ? dq : nullptr;
    qt.tok_part = dQp; qt.lm_part = dLqp; qt.lm_part2 = dWhp; qt.S = p.Stc;
    CK(run_bwd_tc(p, 1, qt, stream));
    if (!p.norm()) CK(run_reduce_parts(p.BH, p.Stc, m, p.mp, d, dWhp, dWh, stream));
  } else {
    CK(run_bwd_pair(p, 1, qa, stream));
    if (!p.norm()) CK(run_reduce_parts(p.BH, p.Sb, m, p.mp, d, dWhp, dWh, stream));
  }

  // ---- G = dLoss/dX_T = dW-hat W^T and dW = X_T^T dW-hat ----
  const float* XT = X + (long)iters * mm;
  const long xs = (long)(iters + 1) * mm;
  const long ys = (long)c.ny * mm;
  // ---- G, the Newton-Schulz reverse and the gram backward on the side stream
  // (they need G); dW and the key side below on this stream (they need dW) ----
  Side* sd = side();
  std::unique_lock<std::mutex> lock;
  if (sd) lock = std::unique_lock<std::mutex>(sd->mu);
  const cudaStream_t ss = sd ? sd->hi : stream;
  if (sd) CK(join(ss, stream, sd->ev[0]));
  if (m <= kTile) {
    CK(run_bgemm(false, true, p.BH, m, m, d, dWh, d, md, W, d, md, G, m, mm, nullptr, m, 0, 1.f,
                 0.f, ss));
    CK(run_bgemm(true, false, p.BH, m, d, m, XT, m, xs, dWh, d, md, dW, d, md, nullptr, d, 0, 1.f,
                 0.f, stream));
  } else {
    CK(ns_mm(p, false, true, m, m, d, dWh, d, md, W, d, md, G, m, mm, nullptr, m, 0, 1.f, 0.f,
             ss));
    CK(ns_mm(p, true, false, m, d, m, XT, m, xs, dWh, d, md, dW, d, md, nullptr, d, 0, 1.f, 0.f,
             stream));
  }
  if (m <= kTile) {
    CK(run_ns_bwd_small(p, A, alpha, X, Y, G, dA, ss));
  } else {
    // Exact reverse of the forward's own products (Y_t = A X_t, then X_t Y_t).
    // The unconverged directions grow by about 2 per step in this recursion, so
    // it must not lean on X_t commuting with A: in fp32 that shortcut diverges.
    if (iters == 0) CK(run_zero(dA, (size_t)p.BH * mm, ss));
    float* Sc = G;
    if (ns_cluster_ok(m))  // the whole reverse in one launch; G ends as dLoss/dX_0
      CK(run_ns_cluster(p, true, A, const_cast<float*>(X), const_cast<float*>(Y), c.nx, c.ny, G,
                        XG, Tm, dA, ss));
    for (int t = ns_cluster_ok(m) ? -1 : iters - 1; t >= 0; --t) {
      const float* Xt = X + (long)t * mm;
      const float* Yt = Y + (long)t * mm;
      // XG = X_t^T G
      CK(ns_mm(p, true, false, m, m, m, Xt, m, xs, Sc, m, mm, XG, m, mm, nullptr, m, 0, 1.f, 0.f,
               ss));
      // dA = dA - XG X_t^T   (the first step initialises dA)
      CK(ns_mm(p, false, true, m, m, m, XG, m, mm, Xt, m, xs, dA, m, mm, dA, m, mm, -1.f,
               t == iters - 1 ? 0.f : 1.f, ss));
      // Tm = 2 G - G Y_t^T
      CK(ns_mm(p, false, true, m, m, m, Sc, m, mm, Yt, m, ys, Tm, m, mm, Sc, m, mm, -1.f, 2.f,
               ss));
      // G = Tm - A^T XG
      CK(ns_mm(p, true, false, m, m, m, A, m, mm, XG, m, mm, Sc, m, mm, Tm, m, mm, -1.f, 1.f,
               ss));
    }
    CK(run_alpha_bwd(p, A, alpha, Sc, dA, ss));
  }
  CK(run_gram_bwd(p, L, Llo, A, dA, dLA, ss));

  // ---- key side ----
  if (tcb) {
    BwdTcArgs kt;
    memset(&kt, 0, sizeof(kt));
    kt.X = k; kt.U = v; kt.L = L; kt.Llo = Llo; kt.R = dW;
    kt.kv = (const float*)(cb + c.C); kt.ties = ties_k; kt.out = nullptr;
    kt.tok_part = dKp; kt.lm_part = dLcp; kt.S = p.Stc;
    // dV = C dW, with the kernel values C the forward kept (token-major [N][mp]):
    // bf16 directly when the streaming kernel applies, else through fp32 partials.
    // Queued before the key-side tile kernel: while the solver's reverse holds
    // its SMs, the streaming product fills the others (measured 0.05 ms less per
    // hires16k step than the other order)
    const float* Cm = (const float*)(cb + c.C);
    if (dv_tc_ok(p))
      CK(run_dv(p, Cm, dW, (float*)(wb + w.dvimg), dv, "dv", stream));
    else
      CK(ns_mm(p, false, false, N, d, m, Cm, p.mp, (long)N * p.mp, dW, d, md, dVp, d, (long)N * d,
               nullptr, d, 0, 1.f, 0.f, stream));
    CK(run_bwd_tc(p, 2, kt, stream));
  } else {
    BwdArgs ka;
    memset(&ka, 0, sizeof(ka));
    ka.X = k; ka.U = v; ka.L = L; ka.Llo = Llo; ka.R = dW;
    ka.tok_part = dKp; ka.tok_part2 = dVp; ka.lm_part = dLcp; ka.ties = ties_k;
    ka.kv = (const float*)(cb + c.C);
    CK(run_bwd_pair(p, 2, ka, stream));
  }
  if (sd) CK(join(stream, ss, sd->ev[1]));
  CK(run_reduce_dl(p, Sl, dLqp, dLcp, dLA, dL, stream));
  if (tcb)
    CK(run_finalize_tc(p, dq_direct ? 0 : ng, dQp, ng, dKp, dv_tc_ok(p) ? nullptr : dVp, dL, idx,
                       dq, dk, dv, stream));
  else
    CK(run_finalize(p, dQp, dKp, dVp, dL, idx, dq, dk, dv, stream));
  return LAPNYS_OK;
}

int lapnys_matmul(const float* A, const float* B, const float* E, float* C, int batch, int M, int N,
                  int K, int trans_a, int trans_b, int lda, int ldb, int lde, int ldc,
                  long long stride_a, long long stride_b, long long stride_e, long long stride_c,
                  float alpha, float beta, int engine, cudaStream_t stream) {
  if (!A || !B || !C || batch <= 0 || M <= 0 || N <= 0 || K <= 0) return LAPNYS_EINVAL;
  if (beta != 0.f && !E) return LAPNYS_EINVAL;
  if (lda <= 0 || ldb <= 0 || ldc <= 0 || (E && lde <= 0)) return LAPNYS_EINVAL;
  if (engine == 1) {
    if (!tc_gemm_ok(M, N, K, lda, ldb, ldc, lde, (long)stride_a, (long)stride_b, (long)stride_c,
                    (long)stride_e, A, B, C, beta != 0.f ? E : nullptr))
      return LAPNYS_ENOTSUP;
    CK(run_tcgemm(trans_a != 0, trans_b != 0, batch, M, N, K, A, lda, (long)stride_a, B, ldb,
                  (long)stride_b, C, ldc, (long)stride_c, E, lde, (long)stride_e, alpha, beta,
                  stream));
    return LAPNYS_OK;
  }
  if (engine != 0) return LAPNYS_EINVAL;
  CK(run_gemm2(trans_a != 0, trans_b != 0, false, batch, M, N, A, lda, (long)stride_a, B, ldb,
               (long)stride_b, K, nullptr, 0, 0, nullptr, 0, 0, 0, C, ldc, (long)stride_c, E, lde,
               (long)stride_e, alpha, beta, stream));
  return LAPNYS_OK;
}

int lapnys_wait_selftest(int polls, cudaStream_t stream) {
  if (polls < 1 || polls > tc_wait_limit()) return LAPNYS_EINVAL;
  CK(run_wait_selftest(polls, stream));
  return LAPNYS_OK;
}

int lapnys_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return LAPNYS_ECUDA;
  const int v = read_wait_error(clear != 0);
  if (v < 0) return LAPNYS_ECUDA;
  return v ? LAPNYS_ETIMEOUT : LAPNYS_OK;
}

uint64_t lapnys_launch_count(void) { return g_launches; }

int lapnys_profile_enable(int on) {
  if (on < 0 || on > 2) return LAPNYS_EINVAL;
  g_prof = on != 0;
  g_serial = on == 2;
  g_used = 0;
  return LAPNYS_OK;
}

int lapnys_fma_probe(int paired, int iters, float* sink, unsigned long long* lane_ops,
                     cudaStream_t stream) {
  if ((paired != 0 && paired != 1) || iters < 1 || iters > (1 << 24) || !sink || !lane_ops)
    return LAPNYS_EINVAL;
  unsigned long long n = 0;
  CK(run_fma_probe(paired != 0, iters, sink, &n, stream));
  *lane_ops = n;
  return LAPNYS_OK;
}

int lapnys_profile_read(const char** names, int* launches, double* total_ms, int max_kernels) {
  int n = 0;
  int bad = 0;
  for (int i = 0; i < g_used; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_rec[i].a, g_rec[i].b) != cudaSuccess) {
      bad = 1;
      continue;
    }
    int j = 0;
    while (j < n && strcmp(names[j], g_rec[i].name) != 0) ++j;
    if (j == n) {
      if (n >= max_kernels) continue;
      names[n] = g_rec[i].name;
      launches[n] = 0;
      total_ms[n] = 0.0;
      ++n;
    }
    launches[j] += 1;
    total_ms[j] += ms;
  }
  g_used = 0;
  return bad ? -1 : n;
}

}  // extern "C"
