#!/usr/bin/env python
"""Benchmark: tokens/s of Laplacian-kernel Nystrom attention, forward + backward.

One step = one pass of the whole path (landmark pooling, landmark matrix,
Newton-Schulz, key pass, W-hat, query pass, and the full backward) over one
batch of the high-resolution workload: B=8, H=8, 128x128 token grid
(N=16384), d=64, m=256 landmarks (8x8 pooling windows), bf16 inputs with fp32
accumulation, lambda=d, eps=1e-3, 24 Newton-Schulz iterations, 1% heavy-tailed
tokens in Q and K.  Inputs are synthetic and seeded; Q, K, V and dO are 134 MB
each, so every step streams inputs larger than the 129 MB L2.

Under torchrun each rank runs its own copy of the workload on its own GPU
(independent (b, h) slices: weak scaling, no collective on the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/sec Laplacian-Nyström attn fwd & fwd+bwd; % of ALU/HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "hires16k"

# FP32 lanes per SM of the part (sm_100 family: 4 sub-partitions x 32); the ALU
# peak is SMs x lanes x maximum SM clock, with the SM count and the clock read
# from the device.  One lane-op = one FADD / FMUL / FFMA / select result.
FP32_LANES_PER_SM = 128


def max_sm_clock_mhz(gpu_index: int):
    """Maximum SM clock (MHz) as nvidia-smi reports it, or None."""
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                            "-i", str(gpu_index)], capture_output=True, text=True, timeout=30)
        return float(r.stdout.strip().splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None


def fma_probe_rates(api, torch, dev):
    """Measured FP32 FMA rate (Tlane-op/s), scalar and paired: best of five
    launches of the library's FMA probe, CUDA events on the current stream."""
    sink = torch.zeros(4, dtype=torch.float32, device=dev)
    out = {}
    for paired in (False, True):
        best = 0.0
        for _ in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            n = api.fma_probe(paired, 1 << 16, sink)
            b.record()
            b.synchronize()
            best = max(best, n / (a.elapsed_time(b) / 1e3) / 1e12)
        out["paired" if paired else "scalar"] = best
    return out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--kernel", choices=["laplace", "gauss"], default="laplace",
                    help="Laplacian kernel (the method) or its Gaussian-kernel variant")
    ap.add_argument("--block", action="store_true",
                    help="the whole attention layer: QKV projection, attention, output projection "
                         "(C = H * d)")
    ap.add_argument("--norm-batch", action="store_true",
                    help="normalised workloads: feature-map statistics over the B slices of a head")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller profiling cases)")
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller profiling cases)")
    ap.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def algorithmic_ops(w):
    """Algorithmic FP32 lane-ops per step, per kernel, from the method's
    formulas (the per-unit figures of the hot-path table: an L1 step = 2
    lane-ops, an FMA = 1).  Per (token, landmark) pair and feature: key and
    query passes 3 (distance 2, contraction 1), each backward side 7 (kernel
    value 2, dot 1, contraction 1, sign term 3); Newton-Schulz 2 m^3 per forward
    step and 6 m^3 per reverse step (all products of a step); norm statistics
    2 per element.  With Q = K the query pass's kernel values are the key
    pass's (P = C^T), so its distances are not counted again (contraction 1).
    The work is fixed by the method, not by where it runs: contractions on the
    tensor cores and kernel values read back from the forward still count."""
    BH, N, m, d, T = w.B * w.H, w.N, w.m, w.d, w.iters
    nmd = BH * N * m * d
    # Gaussian kernel: the gradient term is two FMAs (sum g l, sum g x), not the 3-op sign term
    side = 6 if w.kernel == "gauss" else 7
    return {
        "key_fwd": 3 * nmd,
        "query_fwd": (1 if w.tied else 3) * nmd,
        "qstats": 2 * nmd if w.norm else 0,
        "bwd_query": side * nmd,
        "bwd_key": side * nmd,
        "bwd_qstats": 2 * nmd if w.norm else 0,
        "ns_cluster": 2 * T * BH * m ** 3,
        "ns_cluster_rev": 6 * T * BH * m ** 3,
    }


def fp32_pipe_ops(w):
    """The part of algorithmic_ops that this build executes on the FP32 pipes
    with bf16 inputs: the distances of the forward passes (2) and the sign term
    of the backward sides (4); dots, contractions and the Newton-Schulz
    products run on the tensor cores and the backward reads the forward's
    kernel values."""
    BH, N, m, d = w.B * w.H, w.N, w.m, w.d
    nmd = BH * N * m * d
    tc = w.dtype == "bf16"
    grad = 2 if w.kernel == "gauss" else 4   # Gaussian term: two FMAs; sign term: indicator + two FMAs
    shared = w.tied and tc and not w.norm and w.d in (32, 64)   # O = C W-hat on the tensor cores
    return {"key_fwd": (2 if tc else 3) * nmd, "query_fwd": 0 if shared else (2 if tc else 3) * nmd,
            "bwd_query": (grad if tc else grad + 2) * nmd, "bwd_key": (grad if tc else grad + 2) * nmd}


def measured_traffic(workload: str, method_kernel: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the ncu capture recorded in
    profiles/traffic_<workload>.json ("bytes_per_launch": {kernel: bytes}), or
    None when there is no record for it (this GPU kernel, this attention kernel)
    or its source file has changed since the counters were taken."""
    import hashlib
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles",
                        f"traffic_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("method_kernel", "laplace") != method_kernel:
            return None
        per = rec["bytes_per_launch"]
        if kernel not in per:
            return None
        src = os.path.join(os.path.dirname(os.path.abspath(__file__)), rec["source"])
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return float(per[kernel])
    except (OSError, KeyError, ValueError, TypeError):
        return None


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest value over all ranks (step times: the slowest rank sets the pace)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch of the workload."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def clock_sampler(gpu_index: int):
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                              "-i", str(gpu_index), "-lms", "200"], stdout=f,
                             stderr=subprocess.DEVNULL)
    except OSError:
        p = None
    return p, f.name


def clock_summary(proc, path):
    if proc is not None:
        proc.terminate()
        try:
            proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            proc.kill()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    try:
        for line in open(path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(path)
    except OSError:
        pass
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
            "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm): one (b, h) slice, forward + backward
# ---------------------------------------------------------------------------
def _oracle_slice(wname: str, kernel: str = "laplace", norm_batch: bool = False,
                  block: bool = False):
    """One unit of oracle work: a (b, h) slice, or with batch-pooled statistics
    (which couple them) the B slices of one head; for the whole layer, one
    head's share of it for one batch element (its Q, K, V columns of the
    projection, the attention slice, its rows of the output projection),
    credited with N / H tokens."""
    import dataclasses

    from laplacian_nystr_linear_gb300.inputs import WORKLOADS, block_inputs, make_inputs
    from oracle import lapnys_oracle as orc
    w0 = WORKLOADS[wname]
    if block:
        import numpy as np
        C, d, S = w0.H * w0.d, w0.d, 2 if w0.tied else 3
        b = block_inputs(6000 + w0.cfg, 1, w0.N, C, w0.H, d, w0.dtype, w0.tied, True)
        cols = np.concatenate([np.arange(s * C, s * C + d) for s in range(S)])
        t0 = time.perf_counter()
        _, st = orc.block_forward(b["x"], b["w_qkv"][:, cols], b["b_qkv"][cols], b["w_o"][:d],
                                  b["b_o"], 1, d, w0.grid_h, w0.grid_w, w0.m, w0.lam, w0.eps,
                                  w0.iters, w0.norm, kernel, False, w0.tied)
        orc.block_backward(st, b["dy"])
        return time.perf_counter() - t0, w0.N / w0.H
    nb = bool(norm_batch and w0.norm)
    w = dataclasses.replace(w0, B=w0.B if nb else 1, H=1, kernel=kernel, norm_batch=nb)
    inp = make_inputs(w, with_grad=True)
    t0 = time.perf_counter()
    _, saved = orc.forward(inp["q"], inp["k"], inp["v"], w.grid_h, w.grid_w, w.m, w.lam, w.eps,
                           w.iters, w.norm, kernel=kernel, norm_batch=nb)
    orc.backward(saved, inp["dout"], tied=w.tied)
    return time.perf_counter() - t0, w.B * w.N


def _single_thread_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    return env


def cpu_baseline(wname: str, kernel: str = "laplace", norm_batch: bool = False,
                 block: bool = False):
    """The oracle as it stands, one process, one thread, on whole (b, h) slices
    of the workload (at least 10 s of work)."""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker",
                        "--workload", wname, "--kernel", kernel]
                       + (["--norm-batch"] if norm_batch else []) + (["--block"] if block else []),
                       capture_output=True, text=True, env=_single_thread_env(), timeout=1800)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1:]}
    sec, tokens, n = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": tokens / sec, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{n} head(s) x all B slices (batch-pooled statistics)" if norm_batch
                       else f"{n} (b,h) share(s) of the layer (projections + attention)" if block
                       else f"{n} (b,h) slice(s)")
                      + f" of {wname} ({tokens} tokens), fwd+bwd, fp64, {sec:.1f} s single-threaded"}


def _pool_task(task):
    os.environ.update({k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                         "MKL_NUM_THREADS")})
    return _oracle_slice(*task)


def run_reference(args, rank, world):
    """Reference arm: the fp64 oracle, each step one slice fwd+bwd, steps spread over host cores."""
    if rank != 0:
        return
    import multiprocessing as mp
    cores = max(1, min(os.cpu_count() or 1, max(args.steps, args.warmup)))
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        task = (args.workload, args.kernel, args.norm_batch, args.block)
        pool.map(_pool_task, [task] * max(args.warmup, 1))
        t0 = time.perf_counter()
        res = pool.map(_pool_task, [task] * args.steps)
        wall = time.perf_counter() - t0
    tokens = sum(t for _, t in res)
    value = tokens / wall
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "kernel": args.kernel,
                                        "norm_batch": args.norm_batch, "block": args.block,
                                        "sample": "one (b,h) slice per step (one head's B slices "
                                                  "with batch-pooled statistics)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x one (b,h) slice of {args.workload}, "
                                   f"fwd+bwd, fp64, {cores} processes x 1 thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    from laplacian_nystr_linear_gb300 import api
    from laplacian_nystr_linear_gb300.inputs import WORKLOADS, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import dataclasses
    w = dataclasses.replace(WORKLOADS[args.workload], kernel=args.kernel)
    if args.block and args.norm_batch:
        raise SystemExit("--block times per-slice statistics; drop --norm-batch")
    if args.norm_batch:
        if not w.norm:
            raise SystemExit(f"--norm-batch needs a normalised workload; {w.name} has norm=False")
        w = dataclasses.replace(w, norm_batch=True)
    if args.batch or args.heads:
        w = dataclasses.replace(w, B=args.batch or w.B, H=args.heads or w.H)
    p = api.Params(w.B, w.H, w.grid_h, w.grid_w, w.d, w.m, w.lam, w.eps, w.iters, w.tied, w.norm,
                   w.kernel, w.norm_batch)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = make_inputs(w, with_grad=True)
    host = {n: torch.from_numpy(np.ascontiguousarray(inp[n])).to(tdt) for n in ("q", "k", "v", "dout")}
    q, k, v, dout = (host[n].to(dev) for n in ("q", "k", "v", "dout"))
    if w.tied:
        k = q
    out = torch.empty_like(q)
    dq, dv = torch.empty_like(q), torch.empty_like(q)
    dk = None if w.tied else torch.empty_like(q)
    ctx = api.alloc_ctx(p, dev)
    ws = api.alloc_workspace(p, dev)

    def step():
        api.fwd(q, k, v, p, out=out, ctx=ctx, ws=ws)
        api.bwd(q, k, v, dout, ctx, p, dq=dq, dk=dk, dv=dv, ws=ws)

    def fwd_only():
        api.fwd(q, k, v, p, out=out, ctx=ctx, ws=ws)

    if args.block:
        # the layer around the attention: x [B, N, C] with C = H * d, seeded weights
        from laplacian_nystr_linear_gb300.inputs import block_inputs
        del q, k, v, dout, out, dq, dk, dv, ctx, ws
        C = w.H * w.d
        bp = api.BlockParams(p, C)
        binp = block_inputs(6000 + w.cfg, w.B, w.N, C, w.H, w.d, w.dtype, w.tied, True)
        host = {n: torch.from_numpy(binp[n]).to(tdt) for n in ("x", "dy")}
        x, dy = host["x"].to(dev), host["dy"].to(dev)
        wq, bq, wo, bo = (torch.from_numpy(binp[n]).to(tdt).to(dev)
                          for n in ("w_qkv", "b_qkv", "w_o", "b_o"))
        y, dx = torch.empty_like(x), torch.empty_like(x)
        gw_q, gb_q, gw_o, gb_o = (torch.empty_like(t) for t in (wq, bq, wo, bo))
        ctx = torch.empty(api.block_ctx_bytes(bp, tdt), dtype=torch.uint8, device=dev)
        ws = torch.empty(api.block_workspace_bytes(bp, tdt), dtype=torch.uint8, device=dev)
        q = x  # for the input-size and e2e byte counts below

        def step():
            api.block_fwd(x, wq, bq, wo, bo, bp, y=y, ctx=ctx, ws=ws)
            api.block_bwd(x, wq, wo, dy, ctx, bp, dx=dx, dw_qkv=gw_q, db_qkv=gb_q, dw_o=gw_o,
                          db_o=gb_o, ws=ws)

        def fwd_only():
            api.block_fwd(x, wq, bq, wo, bo, bp, y=y, ctx=ctx, ws=ws)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # inputs smaller than L2 (Q, K, V, dO together): flush L2 between timed
    # steps by writing a buffer of twice its size, outside the timed intervals
    L2_BYTES = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129e6)
    in_bytes = (2 if args.block else 4) * q.numel() * q.element_size()
    flush = None if in_bytes > L2_BYTES else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32,
                                                          device=dev)

    def timed(fn, n):
        """Device milliseconds per call of fn over n calls on this stream."""
        if flush is None:
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            barrier()
            return e0.elapsed_time(e1) / n
        evs = []
        for _ in range(n):
            flush.fill_(float(len(evs)))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        barrier()
        return sum(a.elapsed_time(b) for a, b in evs) / n

    for _ in range(args.warmup):
        step()
    barrier()
    sampler, cpath = clock_sampler(local_rank)
    time.sleep(0.3)
    launches0 = api.launch_count()
    ms_local = timed(step, args.steps)          # no per-launch events in this pass
    clocks = clock_summary(sampler, cpath)
    launches = api.launch_count() - launches0
    ms = max_over_ranks(ms_local, world, dev)
    value = weak_scaling_value(w.tokens, world, ms)

    # per-kernel CUDA-event times, in two more passes of the same steps: as the
    # step runs them (the solver overlapping the key side on a side stream), and
    # serialised on one stream (each kernel's time its own)
    api.profile_enable(True)
    timed(step, args.steps)
    prof = api.profile_read()
    api.profile_enable(True, serial=True)
    timed(step, args.steps)
    prof_alone = api.profile_read()
    api.profile_enable(False)

    # forward alone (same buffers)
    for _ in range(2):
        fwd_only()
    barrier()
    ms_fwd = max_over_ranks(timed(fwd_only, args.steps), world, dev)

    # roofline of the dominant kernel (FP32 lane-ops; the path is ALU-bound)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_max_mhz") or max_sm_clock_mhz(local_rank)
    if not mhz:
        raise SystemExit("bench: the maximum SM clock could not be read (nvidia-smi)")
    peak = sms * FP32_LANES_PER_SM * mhz * 1e6 / 1e12
    probe = fma_probe_rates(api, torch, dev)
    ops = algorithmic_ops(w)
    per_launch_ops = {"bwd_key": ops["bwd_key"], "bwd_query": ops["bwd_query"],
                      "key_fwd": ops["key_fwd"], "query_fwd": ops["query_fwd"]}
    kernel_ms = {n: (c, t / c) for n, (c, t) in prof.items() if c}
    kernel_ms_alone = {n: (c, t / c) for n, (c, t) in prof_alone.items() if c}
    step_ms_sum = sum(t for _, t in prof.values()) / args.steps
    dom = max(per_launch_ops, key=lambda n: prof.get(n, (0, 0.0))[1])
    dom_ms = kernel_ms[dom][1]
    dom_ms_alone = kernel_ms_alone[dom][1]
    achieved = per_launch_ops[dom] / (dom_ms / 1e3) / 1e12
    achieved_alone = per_launch_ops[dom] / (dom_ms_alone / 1e3) / 1e12
    total_ops = sum(ops.values())
    fwd_ops = ops["key_fwd"] + ops["query_fwd"] + ops["qstats"] + ops["ns_cluster"]
    pipe = fp32_pipe_ops(w)
    traffic = measured_traffic(w.name, w.kernel, dom)
    roofline = {
        "bound": "alu", "kernel": dom, "achieved": achieved, "peak": peak,
        "unit": "Tlaneop/s", "frac": achieved / peak,
        "traffic": traffic,
        "peak_source": (f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x {mhz:.0f} MHz (SM count "
                        "from the device, maximum SM clock from nvidia-smi); measured by the "
                        f"library's FMA probe: {probe['scalar']:.1f} (scalar FFMA) and "
                        f"{probe['paired']:.1f} (paired f32x2) Tlane-op/s "
                        "(profiles/fma_probe_gb300.md)"),
        "peak_measured": probe,
        "ms_per_launch": dom_ms, "ms_per_launch_alone": dom_ms_alone,
        "achieved_alone": achieved_alone, "frac_alone": achieved_alone / peak,
        "step_frac": total_ops / (ms / 1e3) / 1e12 / peak,
        "fwd_frac": fwd_ops / (ms_fwd / 1e3) / 1e12 / peak,
        "fp32_pipe_frac": pipe[dom] / (dom_ms / 1e3) / 1e12 / peak,
        "fp32_pipe_frac_alone": pipe[dom] / (dom_ms_alone / 1e3) / 1e12 / peak,
    }

    # end to end through the public API: pinned host inputs in, results back to host
    e2e = None
    if not args.no_e2e and args.block:
        # per step: x and dy in, y and dx out (the weights and their gradients stay
        # resident), overlapped across steps as in the attention's end-to-end loop below:
        # step i + 1's x and dy come in and step i's dx goes out while step i + 1
        # computes, y goes out during its own backward
        pin = {n: host[n].pin_memory() for n in host}
        back = {n: torch.empty(x.shape, dtype=tdt).pin_memory() for n in ("y", "dx")}
        ne = max(3, args.steps)
        dbuf = [{n: torch.empty_like(x) for n in ("x", "dy")} for _ in range(2)]
        obuf = [{n: torch.empty_like(x) for n in ("y", "dx")} for _ in range(2)]
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in, ev_fwd, ev_bwd, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))

        def copy_in(b):
            for n in ("x", "dy"):
                dbuf[b][n].copy_(pin[n], non_blocking=True)
            ev_in[b].record(cin)

        def run_e2e(n):
            with torch.cuda.stream(cin):
                cin.wait_stream(stream)
                copy_in(0)
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    with torch.cuda.stream(cin):
                        if i >= 1:
                            cin.wait_event(ev_bwd[1 - b])
                        copy_in(1 - b)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])
                d, o_ = dbuf[b], obuf[b]
                yo, c = api.block_fwd(d["x"], wq, bq, wo, bo, bp, y=o_["y"], ctx=ctx, ws=ws)
                ev_fwd[b].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_fwd[b])
                    back["y"].copy_(yo, non_blocking=True)
                g = api.block_bwd(d["x"], wq, wo, d["dy"], c, bp, dx=o_["dx"], dw_qkv=gw_q,
                                  db_qkv=gb_q, dw_o=gw_o, db_o=gb_o, ws=ws)
                ev_bwd[b].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_bwd[b])
                    back["dx"].copy_(g[0], non_blocking=True)
                    ev_out[b].record(cout)
            stream.wait_stream(cout)

        run_e2e(3)
        barrier()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        run_e2e(ne)
        eb.record(stream)
        barrier()
        ms_e2e = max_over_ranks(ea.elapsed_time(eb) / ne, world, dev)
        nbytes = x.numel() * x.element_size()
        e2e = {"value": world * w.tokens / (ms_e2e / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": 2 * nbytes, "d2h_bytes_per_step": 2 * nbytes,
               "ms_per_step": ms_e2e}
    elif not args.no_e2e:
        # Every step copies its inputs (Q, K, V, dO) in from pinned host memory and its
        # results (O, dQ, dK, dV) back, through the public API, as a training loop that
        # overlaps its transfers would: two copy streams beside the compute stream and
        # two device buffer sets, so that step i + 1's inputs come in and step i's
        # gradients go out while step i + 1 computes; O goes out during its own
        # backward.  The first step's inputs and the last step's gradients are not
        # overlapped; the timed region holds every copy of every step.
        pin = {n: host[n].pin_memory() for n in host}
        back = {n: torch.empty(q.shape, dtype=tdt).pin_memory() for n in ("out", "dq", "dk", "dv")}
        ne = max(3, args.steps)
        names_in = ["q", "v", "dout"] + ([] if w.tied else ["k"])
        dbuf = [{n: torch.empty_like(q) for n in names_in} for _ in range(2)]
        obuf = [{n: torch.empty_like(q) for n in ("out", "dq", "dk", "dv")} for _ in range(2)]
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in, ev_fwd, ev_bwd, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))

        def copy_in(b):
            for n in names_in:
                dbuf[b][n].copy_(pin[n], non_blocking=True)
            ev_in[b].record(cin)

        def run_e2e(n):
            with torch.cuda.stream(cin):
                cin.wait_stream(stream)
                copy_in(0)
            for i in range(n):
                b = i % 2
                if i + 1 < n:  # the next step's inputs, into the buffer step i - 1 used
                    with torch.cuda.stream(cin):
                        if i >= 1:
                            cin.wait_event(ev_bwd[1 - b])
                        copy_in(1 - b)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # step i - 2's results are on the host
                d, o_ = dbuf[b], obuf[b]
                kd = d["q"] if w.tied else d["k"]
                o, c = api.fwd(d["q"], kd, d["v"], p, out=o_["out"], ctx=ctx, ws=ws)
                ev_fwd[b].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_fwd[b])
                    back["out"].copy_(o, non_blocking=True)
                gq, gk, gv = api.bwd(d["q"], kd, d["v"], d["dout"], c, p, dq=o_["dq"],
                                     dk=None if w.tied else o_["dk"], dv=o_["dv"], ws=ws)
                ev_bwd[b].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_bwd[b])
                    back["dq"].copy_(gq, non_blocking=True)
                    if gk is not None:
                        back["dk"].copy_(gk, non_blocking=True)
                    back["dv"].copy_(gv, non_blocking=True)
                    ev_out[b].record(cout)
            stream.wait_stream(cout)  # the last step's results are on the host

        run_e2e(3)
        barrier()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        run_e2e(ne)
        eb.record(stream)
        barrier()
        ms_e2e = max_over_ranks(ea.elapsed_time(eb) / ne, world, dev)
        nbytes = q.numel() * q.element_size()
        n_in = 3 if w.tied else 4
        n_out = 3 if w.tied else 4
        e2e = {"value": world * w.tokens / (ms_e2e / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": n_in * nbytes, "d2h_bytes_per_step": n_out * nbytes,
               "ms_per_step": ms_e2e}

    if rank != 0:
        return
    base = None
    if world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(args.workload, args.kernel, w.norm_batch, args.block)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) plus 1% Student-t tokens in Q and K)",
        "config": {"workload": args.workload, "kernel": w.kernel, "B": w.B, "H": w.H, "N": w.N,
                   "grid": [w.grid_h, w.grid_w],
                   "d": w.d, "m": w.m, "iters": w.iters, "lambda": w.lam, "eps": w.eps,
                   "norm": w.norm, "norm_batch": w.norm_batch, "tied": w.tied,
                   "pass": "fwd+bwd",
                   "block": ({"C": w.H * w.d, "projections": "tcgen05 bf16 GEMMs of this library, fp32 "
                              "accumulation, head split and bias fused", "e2e": "x, dy in; y, dx out"} if args.block else None),
                   "l2": (f"inputs larger than L2 (Q, K, V, dO {in_bytes / 4e6:.0f} MB each, "
                          f"{L2_BYTES / 1e6:.0f} MB L2); no flush" if flush is None else
                          f"inputs {in_bytes / 1e6:.0f} MB < L2: {2 * L2_BYTES / 1e6:.0f} MB "
                          "written between timed steps, outside the timed intervals"),
                   "parallelism": f"replicas x{world}"},
        "fwd_tokens_per_s": world * w.tokens / (ms_fwd / 1e3), "ms_fwd": ms_fwd,
        "roofline": roofline,
        "kernels_ms_per_step": {n: t / args.steps for n, (c, t) in sorted(prof.items(), key=lambda x: -x[1][1])},
        "kernels_ms_per_step_alone": {n: t / args.steps for n, (c, t)
                                      in sorted(prof_alone.items(), key=lambda x: -x[1][1])},
        "kernel_sum_ms_per_step": step_ms_sum,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": base,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.oracle_worker:
        # whole slices until at least 10 s of CPU work (a bounded sample)
        sec = tokens = n = 0
        while sec < 10.0 or n == 0:
            s1, t1 = _oracle_slice(args.workload, args.kernel, args.norm_batch, args.block)
            sec, tokens, n = sec + s1, tokens + t1, n + 1
        print(json.dumps([sec, tokens, n]))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
