"""The fp64 oracle on sampled (b, h) slices of a named workload, spread over
host processes (test infrastructure).

The workers are started with `spawn` and import neither torch nor the CUDA
library: each regenerates the workload's seeded inputs and runs the oracle on
its share of the slices, so nothing but the slices' results crosses processes.
Workloads with batch-pooled statistics couple the slices of a head and are not
split here (use tests._parity.oracle_run)."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from laplacian_nystr_linear_gb300.inputs import Workload, make_inputs
from oracle import lapnys_oracle as orc


def _job(task):
    w, key, backward = task
    inp = make_inputs(w, with_grad=backward)
    O, saved = orc.forward(inp["q"], inp["k"], inp["v"], w.grid_h, w.grid_w, w.m, w.lam, w.eps,
                           w.iters, w.norm, slices={key}, kernel=w.kernel)
    grads = orc.backward(saved, inp["dout"], tied=w.tied)[key] if backward else None
    return key, O[key], grads


def oracle_slices(w: Workload, slices, backward: bool = False, procs: int | None = None) -> dict:
    """{"out": {(b, h): O}, "saved": {(b, h): None}, ["grads": {(b, h): (dq, dk, dv)}]}
    for the given slices, one process per slice up to `procs` (default: the host's
    cores).  The result indexes like oracle_run's: res["out"][b, h]."""
    assert not w.norm_batch, "batch-pooled statistics couple the slices of a head"
    keys = sorted(slices)
    n = max(1, min(len(keys), procs or os.cpu_count() or 1))
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved_env = {k: os.environ.get(k) for k in env_keys}
    os.environ.update({k: "1" for k in env_keys})  # one BLAS thread per worker
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_job, [(w, k, backward) for k in keys])
    finally:
        for k, v in saved_env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    out = {"out": {k: o for k, o, _ in res}, "saved": {k: None for k, _, _ in res}}
    if backward:
        out["grads"] = {k: g for k, _, g in res}
    return out


def _check_matches_serial():
    """Self-check on a small workload (used by the CPU tests)."""
    w = Workload("pool_check", 9, 2, 2, 8, 8, 16, 4, "f32", 3)
    par = oracle_slices(w, {(0, 1), (1, 0)}, backward=True, procs=2)
    inp = make_inputs(w, with_grad=True)
    O, saved = orc.forward(inp["q"], inp["k"], inp["v"], w.grid_h, w.grid_w, w.m, w.lam, w.eps,
                           w.iters, w.norm, slices={(0, 1), (1, 0)})
    grads = orc.backward(saved, inp["dout"])
    for key in ((0, 1), (1, 0)):
        np.testing.assert_array_equal(par["out"][key], O[key])
        for a, b in zip(par["grads"][key], grads[key]):
            np.testing.assert_array_equal(a, b)
