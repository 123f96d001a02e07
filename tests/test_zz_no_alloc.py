"""lapnys_fwd_static: the inference forward for callers that cannot allocate
device memory (code inside another framework's memory pool, allocator-free
runtimes, code that must not allocate between steps); it runs on scratch
compiled into the library instead of a caller-owned workspace.

It launches the same kernels as lapnys_fwd, with every reduction in the same
fixed order, so its output must be bit-identical to lapnys_fwd's on the same
inputs, on two calls in a row (the second reuses the array the first left
behind), and it must match the oracle within the parity bounds of the other GPU
tests.  This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import _lib, api
from laplacian_nystr_linear_gb300.inputs import Workload, random_inputs

from tests._parity import compare, oracle_run, params_of

pytestmark = pytest.mark.gpu

CASES = [
    # m <= 64: the one-CTA solver; FMA forward passes
    Workload("tiny_f32", 9, 1, 1, 14, 14, 32, 49, "f32", 20),
    Workload("norm_bf16", 9, 4, 5, 14, 14, 64, 49, "bf16", 20, norm=True),
    Workload("tied_bf16", 9, 2, 2, 32, 32, 64, 64, "bf16", 20, tied=True),
    # 64 < m <= 256: the cluster solver
    Workload("large_m_f32", 9, 1, 2, 12, 12, 16, 144, "f32", 10),
    # bf16, d = 64, m > 64: the tensor-core forward passes, a ragged landmark tile
    Workload("tc_bf16", 9, 2, 2, 24, 24, 64, 144, "bf16", 10),
    Workload("tc_gauss_bf16", 9, 2, 2, 24, 24, 64, 144, "bf16", 10, kernel="gauss"),
    # m > 256: the per-product solver, adaptive windows
    Workload("m324_f32", 9, 1, 1, 24, 24, 32, 324, "f32", 6),
    # statistics over the B slices of a head
    Workload("norm_batch_f32", 9, 3, 2, 16, 16, 32, 16, "f32", 8, norm=True, norm_batch=True),
]


def _static_fwd(q, k, v, out, w):
    lib = _lib.load()
    return lib.lapnys_fwd_static(
        ctypes.c_void_p(q.data_ptr()), None if w.tied else ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), w.B, w.H, w.N, w.d,
        w.grid_h, w.grid_w, w.m, w.lam, w.eps, w.iters, int(w.tied),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
        _lib.LAPNYS_BF16 if w.dtype == "bf16" else _lib.LAPNYS_F32, params_of(w).flags)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_scratch_forward_matches_workspace_forward(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = random_inputs(77 + w.m, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    q, k, v = (torch.from_numpy(inp[n]).cuda().to(dt).contiguous() for n in ("q", "k", "v"))
    if w.tied:
        k = q
    ref, _ = api.fwd(q, k, v, params_of(w), need_ctx=False)
    torch.cuda.synchronize()
    ref_bits = ref.view(torch.int16 if w.dtype == "bf16" else torch.int32).cpu().numpy()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _static_fwd(q, k, v, out, w)
        assert rc == _lib.LAPNYS_OK, _lib.load().lapnys_strerror(rc)
        torch.cuda.synchronize()
        got_bits = out.view(torch.int16 if w.dtype == "bf16" else torch.int32).cpu().numpy()
        np.testing.assert_array_equal(got_bits, ref_bits, err_msg=f"call {call}")
    got = out.double().cpu().numpy()
    print(w.name, compare(w, {"out": got}, oracle_run(w, inp), backward=False))


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
