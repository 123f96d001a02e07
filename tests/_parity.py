"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

from laplacian_nystr_linear_gb300 import api
from laplacian_nystr_linear_gb300.inputs import Workload
from oracle import lapnys_oracle as orc

TOL = {"f32": 1e-4, "bf16": 2e-2}
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


def compare(w: Workload, g: dict, o: dict, backward: bool, tol: float | None = None):
    """Per-slice relative Frobenius errors; returns the worst per tensor."""
    tol = TOL[w.dtype] if tol is None else tol
    worst = {}
    for (b, h), s in o["saved"].items():
        errs = {"out": rel(g["out"][b, h], o["out"][b, h])}
        if backward:
            dq, dk, dv = o["grads"][(b, h)]
            errs["dq"] = rel(g["dq"][b, h], dq)
            errs["dv"] = rel(g["dv"][b, h], dv)
            if not w.tied:
                errs["dk"] = rel(g["dk"][b, h], dk)
        for n, e in errs.items():
            worst[n] = max(worst.get(n, 0.0), e)
    bad = {n: e for n, e in worst.items() if not e <= tol}
    assert not bad, f"{w.name}: relative error above {tol}: {bad} (all: {worst})"
    return worst
