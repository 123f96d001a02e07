"""lapnys_fwd_static: the inference forward for callers that cannot allocate
device memory (it runs on scratch compiled into the library instead of a
caller-owned workspace).  Its output must match lapnys_fwd's on the same
inputs, on two calls in a row, within the parity tolerances of the other GPU
tests.  This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import _lib, api
from laplacian_nystr_linear_gb300.inputs import Workload, random_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}

CASES = [
    Workload("tiny_f32", 9, 1, 1, 14, 14, 32, 49, "f32", 20),
    Workload("norm_bf16", 9, 4, 5, 14, 14, 64, 49, "bf16", 20, norm=True),
    Workload("tied_bf16", 9, 2, 2, 32, 32, 64, 64, "bf16", 20, tied=True),
    Workload("large_m_f32", 9, 1, 2, 12, 12, 16, 144, "f32", 10),
]


def _static_fwd(q, k, v, out, w):
    lib = _lib.load()
    return lib.lapnys_fwd_static(
        ctypes.c_void_p(q.data_ptr()), None if w.tied else ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), w.B, w.H, w.N, w.d,
        w.grid_h, w.grid_w, w.m, w.lam, w.eps, w.iters, int(w.tied),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
        _lib.LAPNYS_BF16 if w.dtype == "bf16" else _lib.LAPNYS_F32,
        _lib.LAPNYS_NORM if w.norm else 0)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_scratch_forward_matches_workspace_forward(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = random_inputs(77 + w.m, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    q, k, v = (torch.from_numpy(inp[n]).cuda().to(dt).contiguous() for n in ("q", "k", "v"))
    if w.tied:
        k = q
    p = api.Params(w.B, w.H, w.grid_h, w.grid_w, w.d, w.m, w.lam, w.eps, w.iters, w.tied, w.norm)
    ref, _ = api.fwd(q, k, v, p, need_ctx=False)
    ref = ref.double().cpu().numpy()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _static_fwd(q, k, v, out, w)
        assert rc == _lib.LAPNYS_OK, _lib.load().lapnys_strerror(rc)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        for b in range(w.B):
            for h in range(w.H):
                err = np.linalg.norm(got[b, h] - ref[b, h]) / np.linalg.norm(ref[b, h])
                assert err <= TOL[w.dtype], (call, b, h, err)


def test_static_scratch_rejects_problems_beyond_its_size():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # 256 slices of a 64 x 64 grid with 256 landmarks need far more than 32 MiB
    w = Workload("big", 9, 16, 16, 64, 64, 64, 256, "bf16", 4)
    q = torch.zeros((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    before = api.launch_count()
    assert _static_fwd(q, q, q, out, w) == _lib.LAPNYS_ESCRATCH
    assert api.launch_count() == before
