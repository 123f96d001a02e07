"""The batched fp32 product behind the Newton-Schulz solver (lapnys_matmul),
both engines, against fp64 products of the same inputs (needs a GPU).

The tensor-core engine splits every operand into TF32 hi + lo parts and
accumulates hi*hi + hi*lo + lo*hi in fp32, so it must match fp64 to fp32-level
accuracy: relative Frobenius error below 1e-5 for K <= 512 (measured: about
1e-6 at K = 256 and 3.6e-6 at K = 512)."""
import ctypes

import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(engine, A, B, E, M, N, K, ta, tb, alpha, beta, batch):
    C = torch.full((batch, M, N), float("nan"), device="cuda", dtype=torch.float32)
    lda = A.shape[-1]
    ldb = B.shape[-1]
    rc = _lib.load().lapnys_matmul(
        ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
        ctypes.c_void_p(E.data_ptr()) if E is not None else None, ctypes.c_void_p(C.data_ptr()),
        batch, M, N, K, int(ta), int(tb), lda, ldb, N, N, A[0].numel(), B[0].numel(), M * N, M * N,
        alpha, beta, engine, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, C


CASES = [(256, 256, 256), (196, 196, 196), (256, 64, 256), (128, 128, 64), (144, 144, 144),
         (256, 256, 512)]


@pytest.mark.parametrize("engine", [0, 1])
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("M,N,K", CASES)
def test_matmul_matches_fp64(engine, ta, tb, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + 2 * ta + tb)
    batch = 3
    A = torch.randn((batch, K, M) if ta else (batch, M, K), generator=g, dtype=torch.float64)
    B = torch.randn((batch, N, K) if tb else (batch, K, N), generator=g, dtype=torch.float64)
    E = torch.randn((batch, M, N), generator=g, dtype=torch.float64)
    opA = A.transpose(1, 2) if ta else A
    opB = B.transpose(1, 2) if tb else B
    ref = -0.75 * torch.bmm(opA.float().double(), opB.float().double()) + 2.0 * E.float().double()
    rc, C = _run(engine, A.float().cuda().contiguous(), B.float().cuda().contiguous(),
                 E.float().cuda().contiguous(), M, N, K, ta, tb, -0.75, 2.0, batch)
    assert rc == 0, _lib.load().lapnys_strerror(rc)
    assert _lib.load().lapnys_device_status(1) == 0
    got = C.double().cpu()
    err = float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref))
    assert err < 1e-5, err


def test_matmul_in_place_accumulate():
    # C = C - A B (E aliases C), the form of the landmark-gradient update
    g = torch.Generator().manual_seed(5)
    A = torch.randn((2, 256, 256), generator=g)
    B = torch.randn((2, 256, 256), generator=g)
    C0 = torch.randn((2, 256, 256), generator=g)
    ref = C0.double() - torch.bmm(A.double(), B.double())
    for engine in (0, 1):
        C = C0.clone().cuda()
        Ad, Bd = A.cuda(), B.cuda()
        rc = _lib.load().lapnys_matmul(
            ctypes.c_void_p(Ad.data_ptr()), ctypes.c_void_p(Bd.data_ptr()),
            ctypes.c_void_p(C.data_ptr()), ctypes.c_void_p(C.data_ptr()), 2, 256, 256, 256, 0, 0,
            256, 256, 256, 256, 65536, 65536, 65536, 65536, -1.0, 1.0, engine,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        err = float(torch.linalg.norm(C.double().cpu() - ref) / torch.linalg.norm(ref))
        assert err < 1e-5, (engine, err)


def test_tensor_core_engine_rejects_unaligned_shapes():
    A = torch.zeros((1, 81, 81), device="cuda")
    rc, _ = _run(1, A, A, None, 81, 81, 81, False, False, 1.0, 0.0, 1)
    assert rc == _lib.LAPNYS_ENOTSUP
