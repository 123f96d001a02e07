"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the fp64 oracle on the same seeded inputs, and compare.

Two bounds hold for every compared tensor of every sampled (b, h) slice:
  - per slice   |gpu - oracle|_F / |oracle|_F <= TOL (1e-4 fp32, 2e-2 bf16 with
    fp32 accumulation: the tolerances the method's parity target states);
  - per element |gpu - oracle| <= R |oracle| + A rms(oracle slice), so that one
    wrong row, a wrong ragged tail or a missed tie correction, which move a
    Frobenius ratio of a large slice by little, still fail.  R covers rounding
    the result to the element type (bf16: at most 2^-9 relative, R = 2^-7);
    A covers the fp32 / TF32 accumulation error, which scales with the size of
    the slice's values rather than of each element (see the tables EW below).
Set LAPNYS_PARITY_LOG=<file> to append the measured errors of every comparison
as JSON lines.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from laplacian_nystr_linear_gb300 import api
from laplacian_nystr_linear_gb300.inputs import Workload, outlier_counts
from oracle import lapnys_oracle as orc

TOL = {"f32": 1e-4, "bf16": 2e-2}
# (R, A) of the element-wise bound |gpu - oracle| <= R |oracle| + A rms(oracle slice)
EW = {"f32": (1e-4, 1e-4), "bf16": (2.0 ** -7, 2e-2)}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def params_of(w: Workload) -> api.Params:
    return api.Params(w.B, w.H, w.grid_h, w.grid_w, w.d, w.m, w.lam, w.eps, w.iters, w.tied, w.norm,
                      w.kernel, w.norm_batch)


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(TDT[dtype]).contiguous()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_run(w: Workload, inp: dict, backward: bool = False):
    p = params_of(w)
    q = to_dev(inp["q"], w.dtype)
    k = q if w.tied else to_dev(inp["k"], w.dtype)
    v = to_dev(inp["v"], w.dtype)
    out, ctx = api.fwd(q, k, v, p, need_ctx=True)
    res = {"out": out}
    if backward:
        dout = to_dev(inp["dout"], w.dtype)
        dq, dk, dv = api.bwd(q, k, v, dout, ctx, p)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    res = {n: (to_np(t) if t is not None else None) for n, t in res.items()}
    res["ctx"] = {n: t.cpu().numpy() for n, t in api.ctx_views(ctx, p).items()}
    return res


def oracle_run(w: Workload, inp: dict, slices=None, backward: bool = False):
    O, saved = orc.forward(inp["q"], inp["k"], inp["v"], w.grid_h, w.grid_w, w.m, w.lam, w.eps,
                           w.iters, w.norm, slices=slices, kernel=w.kernel,
                           norm_batch=w.norm_batch)
    res = {"out": O, "saved": saved}
    if backward:
        res["grads"] = orc.backward(saved, inp["dout"], tied=w.tied)
    return res


def rel(a: np.ndarray, b: np.ndarray) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def elementwise_excess(got: np.ndarray, ref: np.ndarray, r: float) -> tuple[float, float]:
    """(smallest A with |got - ref| <= r |ref| + A rms(ref) everywhere,
    max |got - ref| / rms(ref))."""
    rms = float(np.sqrt(np.mean(ref * ref)))
    rms = rms if rms > 0 else 1.0
    diff = np.abs(got - ref)
    return (float(np.max(np.maximum(diff - r * np.abs(ref), 0.0))) / rms,
            float(np.max(diff)) / rms)


def top_outlier_slices(w: Workload, n: int) -> set:
    """The n (b, h) slices with the most heavy-tailed tokens (ties: lowest index)."""
    c = outlier_counts(w).ravel()
    order = np.argsort(-c, kind="stable")[:n]
    return {(int(i) // w.H, int(i) % w.H) for i in order}


def _log(rec: dict) -> None:
    path = os.environ.get("LAPNYS_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def compare(w: Workload, g: dict, o: dict, backward: bool, tol: float | None = None,
            ew: tuple[float, float] | None = None):
    """Per-slice relative Frobenius errors and the element-wise bound (see the
    module docstring) on every sampled slice; returns the worst per tensor."""
    tol = TOL[w.dtype] if tol is None else tol
    r, a = EW[w.dtype] if ew is None else ew
    worst, worst_ew, worst_abs = {}, {}, {}
    for (b, h), s in o["saved"].items():
        pairs = {"out": (g["out"][b, h], o["out"][b, h])}
        if backward:
            dq, dk, dv = o["grads"][(b, h)]
            pairs["dq"] = (g["dq"][b, h], dq)
            pairs["dv"] = (g["dv"][b, h], dv)
            if not w.tied:
                pairs["dk"] = (g["dk"][b, h], dk)
        for n, (got, ref) in pairs.items():
            worst[n] = max(worst.get(n, 0.0), rel(got, ref))
            ex, ab = elementwise_excess(got, ref, r)
            worst_ew[n] = max(worst_ew.get(n, 0.0), ex)
            worst_abs[n] = max(worst_abs.get(n, 0.0), ab)
    _log({"workload": w.name, "dtype": w.dtype, "kernel": w.kernel, "fro": worst,
          "ew_excess": worst_ew, "ew_abs": worst_abs, "R": r, "A": a,
          "slices": len(o["saved"])})
    bad = {n: e for n, e in worst.items() if not e <= tol}
    assert not bad, f"{w.name}: relative error above {tol}: {bad} (all: {worst})"
    bad = {n: e for n, e in worst_ew.items() if not e <= a}
    assert not bad, (f"{w.name}: element-wise error above {r:.3g} |ref| + {a:.3g} rms: "
                     f"excess/rms {bad} (all: {worst_ew})")
    return worst
