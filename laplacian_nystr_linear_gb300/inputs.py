"""Seeded synthetic inputs for Laplacian-kernel Nystrom attention.

This module only draws random numbers and names workload shapes; it holds none
of the method's arithmetic, so both the CUDA path and the CPU oracle can be fed
the same bytes from it.

Workloads are vision-shaped token grids (a PVT-style pyramid and a
high-resolution grid), standing in for the ImageNet/COCO feature maps the
LaplacianFormer pages evaluate on (LaplacianFormer, Results: ImageNet-1K and
COCO); no dataset is read.  Values are N(0, 1); the high-resolution workload
adds heavy-tailed tokens (Student-t, nu = 3) to Q and K, echoing the pages'
observation that query-key distances in vision transformers are heavy-tailed
(LaplacianFormer, Problem statement, point 2).

Seeds: q = 1000 + c, k = 2000 + c, v = 3000 + c, dO = 4000 + c,
outliers = 5000 + c, where c is the workload's config number (1..5).
Draws are float32; bf16 workloads round them to bf16 (round to nearest even),
so the returned float32 arrays hold exactly the bf16 values both sides use.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg: int            # config number, fixes the seeds
    B: int
    H: int
    grid_h: int
    grid_w: int
    d: int
    m: int
    dtype: str          # "f32" or "bf16"
    iters: int
    eps: float = 1e-3
    tied: bool = False
    norm: bool = False
    outliers: bool = False
    backward: bool = False
    kernel: str = "laplace"   # "laplace" or "gauss" (a name only; no arithmetic here)
    norm_batch: bool = False  # with norm: statistics over the B slices of a head

    @property
    def N(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def lam(self) -> float:
        return float(self.d)

    @property
    def tokens(self) -> int:
        return self.B * self.N

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny fp32 forward, 14x14 grid, 7x7 landmarks
    "tiny": Workload("tiny", 1, 1, 1, 14, 14, 32, 49, "f32", 20),
    # the same grid with one landmark per token (m = N)
    "tiny_mN": Workload("tiny_mN", 1, 1, 1, 14, 14, 32, 196, "f32", 20),
    # PVT stage-1 shape: 56x56 tokens, 49 landmarks, separate Q and K
    "pvt1": Workload("pvt1", 2, 32, 1, 56, 56, 64, 49, "bf16", 20),
    # PVT stage-2 / stage-3 shapes, forward + backward, normalised query map
    "pvt2": Workload("pvt2", 3, 32, 2, 28, 28, 64, 49, "bf16", 20, norm=True, backward=True),
    "pvt3": Workload("pvt3", 3, 32, 5, 14, 14, 64, 49, "bf16", 20, norm=True, backward=True),
    # high-resolution 128x128 grid, 256 landmarks, heavy-tailed Q/K tokens
    "hires16k": Workload("hires16k", 4, 8, 8, 128, 128, 64, 256, "bf16", 24,
                         outliers=True, backward=True),
    # long sequence, tied Q = K (symmetric SOFT-style), 64 landmarks
    "tied64k": Workload("tied64k", 5, 1, 16, 256, 256, 64, 64, "bf16", 20, tied=True),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32)


def _student_t3(rng: np.random.Generator, shape) -> np.ndarray:
    # Z / sqrt(chi2_3 / 3) with one chi-square draw per element (i.i.d. components)
    z = rng.standard_normal(shape)
    chi2 = rng.chisquare(3.0, size=shape)
    return (z / np.sqrt(chi2 / 3.0)).astype(np.float32)


def _normal(seed: int, shape) -> np.ndarray:
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)


def _outlier_draws(w: Workload):
    """(mask [B, H, N], heavy-tailed rows) for Q, then K unless tied, in draw order."""
    shape = (w.B, w.H, w.N, w.d)
    rng = np.random.default_rng(5000 + w.cfg)
    for _ in range(1 if w.tied else 2):
        mask = rng.random(shape[:-1]) < 0.01
        yield mask, _student_t3(rng, (int(mask.sum()), w.d))


def outlier_counts(w: Workload) -> np.ndarray:
    """Heavy-tailed tokens per (b, h) slice, Q and K together ([B, H] int; zeros
    when the workload has none)."""
    n = np.zeros((w.B, w.H), np.int64)
    if w.outliers:
        for mask, _ in _outlier_draws(w):
            n += mask.sum(axis=-1)
    return n


def make_inputs(w: Workload, with_grad: bool | None = None) -> dict:
    """Return {"q","k","v"[,"dout"]} as float32 arrays of shape [B, H, N, d].

    In tied workloads "k" is the same array object as "q".
    """
    shape = (w.B, w.H, w.N, w.d)
    c = w.cfg
    q = _normal(1000 + c, shape)
    k = q if w.tied else _normal(2000 + c, shape)
    v = _normal(3000 + c, shape)
    if w.outliers:
        for t, (mask, heavy) in zip((q,) if w.tied else (q, k), _outlier_draws(w)):
            t[mask] = heavy
    out = {"q": q, "k": k, "v": v}
    if with_grad if with_grad is not None else w.backward:
        out["dout"] = _normal(4000 + c, shape)
    if w.dtype == "bf16":
        for key in list(out):
            if key == "k" and w.tied:
                continue
            out[key] = round_bf16(out[key])
        if w.tied:
            out["k"] = out["q"]
    return out


def random_inputs(seed: int, B: int, H: int, N: int, d: int, dtype: str = "f32",
                  tied: bool = False, scale: float = 1.0) -> dict:
    """Small seeded inputs for parity sweeps over shapes not in WORKLOADS."""
    rng = np.random.default_rng(seed)
    shape = (B, H, N, d)
    q = (rng.standard_normal(shape, dtype=np.float32) * scale).astype(np.float32)
    k = q if tied else (rng.standard_normal(shape, dtype=np.float32) * scale).astype(np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    dout = rng.standard_normal(shape, dtype=np.float32)
    out = {"q": q, "k": k, "v": v, "dout": dout}
    if dtype == "bf16":
        for key in ("q", "k", "v", "dout"):
            if key == "k" and tied:
                continue
            out[key] = round_bf16(out[key])
        if tied:
            out["k"] = out["q"]
    return out


def isqrt_exact(m: int) -> int:
    r = math.isqrt(m)
    return r if r * r == m else -1


def block_inputs(seed: int, B: int, N: int, C: int, H: int, d: int, dtype: str = "f32",
                 tied: bool = False, bias: bool = True) -> dict:
    """Seeded inputs of the attention block: x and dy [B, N, C] ~ N(0, 1), the
    projection weights ~ N(0, 1 / fan_in) (so Q, K, V come out ~ N(0, 1)) and
    biases ~ N(0, 0.1^2) (None when bias is False); float32 arrays, rounded to
    bf16 values when dtype is "bf16"."""
    rng = np.random.default_rng(seed)
    S = 2 if tied else 3
    f32 = np.float32
    out = {
        "x": rng.standard_normal((B, N, C), dtype=f32),
        "w_qkv": (rng.standard_normal((C, S * H * d), dtype=f32) / np.sqrt(C)).astype(f32),
        "b_qkv": (rng.standard_normal(S * H * d, dtype=f32) * 0.1).astype(f32) if bias else None,
        "w_o": (rng.standard_normal((H * d, C), dtype=f32) / np.sqrt(H * d)).astype(f32),
        "b_o": (rng.standard_normal(C, dtype=f32) * 0.1).astype(f32) if bias else None,
        "dy": rng.standard_normal((B, N, C), dtype=f32),
    }
    if dtype == "bf16":
        out = {n: (None if a is None else round_bf16(a)) for n, a in out.items()}
    return out
