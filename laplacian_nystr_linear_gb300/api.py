"""PyTorch-facing wrappers over the C ABI (marshalling only: PyTorch supplies
device memory and the current stream; every step runs in liblapnys kernels)."""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import check, load

_DT = {torch.float32: _lib.LAPNYS_F32, torch.bfloat16: _lib.LAPNYS_BF16}


@dataclasses.dataclass(frozen=True)
class Params:
    """Shape and method parameters of one call ([B, H, N, d] tensors on a grid)."""
    B: int
    H: int
    grid_h: int
    grid_w: int
    d: int
    m: int
    lam: float
    eps: float = 1e-3
    iters: int = 20
    tied: bool = False
    norm: bool = False
    kernel: str = "laplace"  # or "gauss"
    norm_batch: bool = False  # with norm: statistics over the B slices of a head

    @property
    def N(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def flags(self) -> int:
        if self.kernel not in ("laplace", "gauss"):
            raise ValueError(f"unknown kernel {self.kernel!r}")
        return ((_lib.LAPNYS_NORM if self.norm else 0)
                | (_lib.LAPNYS_GAUSS if self.kernel == "gauss" else 0)
                | (_lib.LAPNYS_NORM_BATCH if self.norm_batch else 0))

    def dims(self):
        return (self.B, self.H, self.N, self.d, self.grid_h, self.grid_w, self.m)

    @staticmethod
    def of(q: torch.Tensor, grid, m: int, lam=None, eps=1e-3, iters=20, tied=False, norm=False,
           kernel="laplace", norm_batch=False):
        B, H, N, d = q.shape
        gh, gw = grid
        return Params(B, H, gh, gw, d, m, float(d if lam is None else lam), float(eps), int(iters),
                      bool(tied), bool(norm), str(kernel), bool(norm_batch))


def ctx_bytes(p: Params) -> int:
    return load().lapnys_ctx_bytes(p.B, p.H, p.N, p.d, p.m, p.iters, p.flags)


def workspace_bytes(p: Params) -> int:
    return load().lapnys_workspace_bytes(p.B, p.H, p.N, p.d, p.m, p.iters, p.flags)


def ctx_offsets(p: Params) -> dict:
    lay = _lib.CtxLayout()
    check(load().lapnys_ctx_offsets(p.B, p.H, p.N, p.d, p.m, p.iters, p.flags, ctypes.byref(lay)),
          "lapnys_ctx_offsets")
    return {n: getattr(lay, n) for n, _ in _lib.CtxLayout._fields_}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DT[t.dtype]


def _check_tensor(t: torch.Tensor, name: str, like: torch.Tensor) -> None:
    if not t.is_cuda or not t.is_contiguous() or t.dtype != like.dtype or t.shape != like.shape:
        raise ValueError(f"{name} must be a contiguous CUDA tensor like q ({like.shape}, {like.dtype})")


def alloc_ctx(p: Params, device) -> torch.Tensor:
    return torch.empty(ctx_bytes(p), dtype=torch.uint8, device=device)


def alloc_workspace(p: Params, device) -> torch.Tensor:
    return torch.empty(workspace_bytes(p), dtype=torch.uint8, device=device)


def fwd(q, k, v, p: Params, out=None, ctx=None, ws=None, need_ctx=True):
    """lapnys_fwd: returns (out, ctx); ctx is None when need_ctx is False."""
    _check_tensor(q, "q", q)
    _check_tensor(v, "v", q)
    if not p.tied:
        _check_tensor(k, "k", q)
    dev = q.device
    out = torch.empty_like(q) if out is None else out
    if need_ctx and ctx is None:
        ctx = alloc_ctx(p, dev)
    ws = alloc_workspace(p, dev) if ws is None else ws
    rc = load().lapnys_fwd(
        _ptr(q), None if p.tied else _ptr(k), _ptr(v), _ptr(out), *p.dims(), p.lam, p.eps,
        p.iters, int(p.tied), _stream(dev), _dtype(q), p.flags,
        _ptr(ctx) if need_ctx else None, ctx.numel() if need_ctx else 0, _ptr(ws), ws.numel())
    check(rc, "lapnys_fwd")
    return out, (ctx if need_ctx else None)


def bwd(q, k, v, dout, ctx, p: Params, dq=None, dk=None, dv=None, ws=None):
    """lapnys_bwd: returns (dq, dk, dv); dk is None in tied mode (dq holds it all)."""
    _check_tensor(dout, "dout", q)
    dev = q.device
    dq = torch.empty_like(q) if dq is None else dq
    dv = torch.empty_like(q) if dv is None else dv
    if not p.tied and dk is None:
        dk = torch.empty_like(q)
    ws = alloc_workspace(p, dev) if ws is None else ws
    rc = load().lapnys_bwd(
        _ptr(q), None if p.tied else _ptr(k), _ptr(v), _ptr(dout), _ptr(ctx), _ptr(dq),
        None if p.tied else _ptr(dk), _ptr(dv), *p.dims(), p.lam, p.eps, p.iters, int(p.tied),
        _stream(dev), _dtype(q), p.flags, _ptr(ws), ws.numel())
    check(rc, "lapnys_bwd")
    return dq, (None if p.tied else dk), dv


def pool(k, grid, m):
    """lapnys_pool: landmarks [B, H, m, d] float32 and the token -> landmark index [N] int32."""
    B, H, N, d = k.shape
    L = torch.empty((B, H, m, d), dtype=torch.float32, device=k.device)
    idx = torch.empty((N,), dtype=torch.int32, device=k.device)
    rc = load().lapnys_pool(_ptr(k), _ptr(L), _ptr(idx), B, H, N, d, grid[0], grid[1], m,
                            _dtype(k), _stream(k.device))
    check(rc, "lapnys_pool")
    return L, idx


def ctx_views(ctx: torch.Tensor, p: Params) -> dict:
    """Float32 / int32 views of the intermediates saved in ctx (see lapnys_ctx_layout)."""
    off = ctx_offsets(p)
    BH, m, d, T = p.B * p.H, p.m, p.d, p.iters

    def f32(name, shape):
        n = 1
        for s in shape:
            n *= s
        return ctx[off[name]:off[name] + 4 * n].view(torch.float32).view(shape)

    views = {
        "L": f32("L", (p.B, p.H, m, d)),
        "Llo": f32("Llo", (p.B, p.H, m, d)),
        "A": f32("A", (p.B, p.H, m, m)),
        "alpha": f32("alpha", (p.B, p.H, 4)),
        "X": f32("X", (p.B, p.H, T + 1, m, m)),
        "W": f32("W", (p.B, p.H, m, d)),
        "What": f32("What", (p.B, p.H, m, d)),
        "stats": f32("stats", (p.B, p.H, 3, m)),
        "idx": ctx[off["idx"]:off["idx"] + 4 * p.N].view(torch.int32),
    }
    if T > 0:
        views["Y"] = f32("Y", (p.B, p.H, T, m, m))
    mp = (m + 63) // 64 * 64
    views["P"] = f32("P", (p.B, p.H, p.N, mp))[..., :m]
    views["C"] = f32("C", (p.B, p.H, p.N, mp))[..., :m]
    return views


def device_status(clear: bool = False) -> int:
    """lapnys_device_status: synchronises the current device; LAPNYS_ETIMEOUT if a
    bounded device wait expired since the last clear."""
    return int(load().lapnys_device_status(1 if clear else 0))


def wait_selftest(polls: int, device=None) -> None:
    """lapnys_wait_selftest on the current stream: a bounded wait that expires."""
    check(load().lapnys_wait_selftest(int(polls), _stream(device)), "lapnys_wait_selftest")


def launch_count() -> int:
    return int(load().lapnys_launch_count())


def profile_enable(on, serial: bool = False) -> None:
    """Per-launch CUDA-event timing on (on) or off; serial=True also runs each
    call on the caller's stream alone, so each kernel's time is its own."""
    check(load().lapnys_profile_enable((2 if serial else 1) if on else 0), "lapnys_profile_enable")


def fma_probe(paired: bool, iters: int, sink: torch.Tensor) -> int:
    """Enqueue the FP32 FMA-rate probe on the current stream; returns its lane-ops."""
    n = ctypes.c_ulonglong(0)
    check(load().lapnys_fma_probe(int(paired), int(iters), _ptr(sink), ctypes.byref(n),
                                  _stream(sink.device)), "lapnys_fma_probe")
    return int(n.value)


def profile_read(max_kernels: int = 64) -> dict:
    """{kernel name: (launches, total ms)} since the last read; call after a synchronize."""
    names = (ctypes.c_char_p * max_kernels)()
    launches = (ctypes.c_int * max_kernels)()
    total = (ctypes.c_double * max_kernels)()
    n = load().lapnys_profile_read(names, launches, total, max_kernels)
    if n < 0:
        raise RuntimeError("lapnys_profile_read: an event query failed")
    return {names[i].decode(): (launches[i], total[i]) for i in range(n)}


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(fctx, q, k, v, p: Params):
        out, ctx = fwd(q, k, v, p, need_ctx=True)
        fctx.p = p
        fctx.save_for_backward(q, k if not p.tied else q, v, ctx)
        return out

    @staticmethod
    def backward(fctx, dout):
        q, k, v, ctx = fctx.saved_tensors
        p = fctx.p
        dq, dk, dv = bwd(q, k, v, dout.contiguous(), ctx, p)
        if p.tied:
            return dq, None, dv, None
        return dq, dk, dv, None


def attention(q, k, v, grid, m, lam=None, eps=1e-3, iters=20, tied=False, norm=False,
              kernel="laplace", norm_batch=False):
    """Kernel Nystrom attention O = Z . X_T . (k(L, K) . V) with autograd, for the
    Laplacian kernel (kernel="laplace") or the Gaussian kernel (kernel="gauss").

    q, k, v: [B, H, N, d] CUDA tensors (float32 or bfloat16), N = grid[0] * grid[1].
    In tied mode pass k=None (or k=q); the gradient of the shared tensor goes to q.
    With norm=True, norm_batch=True takes the feature-map statistics over the B
    slices of each head instead of per slice.
    """
    p = Params.of(q, grid, m, lam, eps, iters, tied, norm, kernel, norm_batch)
    if tied:
        k = q
    return _Attention.apply(q, k, v, p)


# ---------------------------------------------------------------------------
# the attention block: [Q | K | V] = X W_qkv + b_qkv, per-head attention,
# Y = concat_h(O_h) W_o + b_o  (lapnys_block_fwd / lapnys_block_bwd)
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class BlockParams:
    """The attention's parameters plus the embedding width C of x [B, N, C]."""
    attn: Params
    C: int

    @property
    def S(self) -> int:
        return 2 if self.attn.tied else 3

    def dims(self):
        a = self.attn
        return (a.B, a.N, self.C, a.H, a.d, a.grid_h, a.grid_w, a.m)

    def sizes(self):
        a = self.attn
        return (a.B, a.N, self.C, a.H, a.d, a.m, a.iters, int(a.tied))


def block_ctx_bytes(bp: BlockParams, dtype: torch.dtype) -> int:
    return load().lapnys_block_ctx_bytes(*bp.sizes(), _DT[dtype], bp.attn.flags)


def block_workspace_bytes(bp: BlockParams, dtype: torch.dtype) -> int:
    return load().lapnys_block_workspace_bytes(*bp.sizes(), _DT[dtype], bp.attn.flags)


def _check_param(t, name, shape, like):
    if t is None:
        return
    if not t.is_cuda or not t.is_contiguous() or t.dtype != like.dtype or tuple(t.shape) != shape:
        raise ValueError(f"{name} must be a contiguous CUDA tensor of shape {shape} and {like.dtype}")


def _check_block(x, w_qkv, b_qkv, w_o, b_o, bp: BlockParams):
    a = bp.attn
    HD = a.H * a.d
    _check_param(x, "x", (a.B, a.N, bp.C), x)
    _check_param(w_qkv, "w_qkv", (bp.C, bp.S * HD), x)
    _check_param(b_qkv, "b_qkv", (bp.S * HD,), x)
    _check_param(w_o, "w_o", (HD, bp.C), x)
    _check_param(b_o, "b_o", (bp.C,), x)


def block_fwd(x, w_qkv, b_qkv, w_o, b_o, bp: BlockParams, y=None, ctx=None, ws=None,
              need_ctx=True):
    """lapnys_block_fwd: returns (y, ctx); ctx is None when need_ctx is False."""
    _check_block(x, w_qkv, b_qkv, w_o, b_o, bp)
    a = bp.attn
    dev = x.device
    y = torch.empty_like(x) if y is None else y
    _check_param(y, "y", tuple(x.shape), x)
    if need_ctx and ctx is None:
        ctx = torch.empty(block_ctx_bytes(bp, x.dtype), dtype=torch.uint8, device=dev)
    if ws is None:
        ws = torch.empty(block_workspace_bytes(bp, x.dtype), dtype=torch.uint8, device=dev)
    rc = load().lapnys_block_fwd(
        _ptr(x), _ptr(w_qkv), _ptr(b_qkv), _ptr(w_o), _ptr(b_o), _ptr(y), *bp.dims(), a.lam, a.eps,
        a.iters, int(a.tied), _stream(dev), _dtype(x), a.flags,
        _ptr(ctx) if need_ctx else None, ctx.numel() if need_ctx else 0, _ptr(ws), ws.numel())
    check(rc, "lapnys_block_fwd")
    return y, (ctx if need_ctx else None)


def block_bwd(x, w_qkv, w_o, dy, ctx, bp: BlockParams, bias_grads=True, dx=None, dw_qkv=None,
              db_qkv=None, dw_o=None, db_o=None, ws=None):
    """lapnys_block_bwd: returns (dx, dw_qkv, db_qkv, dw_o, db_o); the bias
    gradients are None when bias_grads is False."""
    _check_block(x, w_qkv, None, w_o, None, bp)
    _check_param(dy, "dy", tuple(x.shape), x)
    a = bp.attn
    dev = x.device
    HD = a.H * a.d
    dx = torch.empty_like(x) if dx is None else dx
    dw_qkv = torch.empty_like(w_qkv) if dw_qkv is None else dw_qkv
    dw_o = torch.empty_like(w_o) if dw_o is None else dw_o
    if bias_grads:
        db_qkv = x.new_empty((bp.S * HD,)) if db_qkv is None else db_qkv
        db_o = x.new_empty((bp.C,)) if db_o is None else db_o
    else:
        db_qkv = db_o = None
    if ws is None:
        ws = torch.empty(block_workspace_bytes(bp, x.dtype), dtype=torch.uint8, device=dev)
    rc = load().lapnys_block_bwd(
        _ptr(x), _ptr(w_qkv), _ptr(w_o), _ptr(dy), _ptr(ctx), _ptr(dx), _ptr(dw_qkv), _ptr(db_qkv),
        _ptr(dw_o), _ptr(db_o), *bp.dims(), a.lam, a.eps, a.iters, int(a.tied), _stream(dev),
        _dtype(x), a.flags, _ptr(ws), ws.numel())
    check(rc, "lapnys_block_bwd")
    return dx, dw_qkv, db_qkv, dw_o, db_o


class _Block(torch.autograd.Function):
    @staticmethod
    def forward(fctx, x, w_qkv, b_qkv, w_o, b_o, bp: BlockParams):
        y, ctx = block_fwd(x, w_qkv, b_qkv, w_o, b_o, bp, need_ctx=True)
        fctx.bp = bp
        fctx.has_bias = (b_qkv is not None, b_o is not None)
        fctx.save_for_backward(x, w_qkv, w_o, ctx)
        return y

    @staticmethod
    def backward(fctx, dy):
        x, w_qkv, w_o, ctx = fctx.saved_tensors
        dx, dw, db, dwo, dbo = block_bwd(x, w_qkv, w_o, dy.contiguous(), ctx, fctx.bp,
                                         bias_grads=any(fctx.has_bias))
        return (dx, dw, db if fctx.has_bias[0] else None, dwo, dbo if fctx.has_bias[1] else None,
                None)


def attention_block(x, w_qkv, b_qkv, w_o, b_o, grid, heads, m, lam=None, eps=1e-3, iters=20,
                    tied=False, norm=False, kernel="laplace", norm_batch=False):
    """One multi-head layer with autograd: [Q | K | V] = x w_qkv + b_qkv, the
    Nystrom attention per head, y = concat(heads) w_o + b_o.

    x: [B, N, C] CUDA tensor (float32 or bfloat16), N = grid[0] * grid[1];
    w_qkv: [C, S * heads * d] with column blocks (Q | K | V) (S = 3) or, tied,
    (Q = K | V) (S = 2); w_o: [heads * d, C]; biases [S * heads * d] and [C] or None.
    lam defaults to d.
    """
    B, N, C = x.shape
    d = w_o.shape[0] // heads
    a = Params(B, heads, grid[0], grid[1], d, m, float(d if lam is None else lam), float(eps),
               int(iters), bool(tied), bool(norm), str(kernel), bool(norm_batch))
    return _Block.apply(x, w_qkv, b_qkv, w_o, b_o, BlockParams(a, C))
