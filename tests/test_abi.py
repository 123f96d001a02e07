"""C ABI checks that need no GPU: the library builds and loads, exports every
symbol the header declares, sizes buffers, and rejects bad arguments on the
host before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from laplacian_nystr_linear_gb300 import build as b
    from laplacian_nystr_linear_gb300 import _lib
    b.build()
    return _lib.load()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "lapnys.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lapnys_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    from laplacian_nystr_linear_gb300 import _lib
    assert _header_functions() == sorted(_lib.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_sizes(lib):
    # hires workload: 8 x 8 slices, N = 16384, d = 64, m = 256, 24 iterations
    c = lib.lapnys_ctx_bytes(8, 8, 16384, 64, 256, 24, 0)
    # iterates dominate: 64 slices x (25 X + 24 Y) x 256^2 floats
    assert c >= 64 * 49 * 256 * 256 * 4
    assert lib.lapnys_workspace_bytes(8, 8, 16384, 64, 256, 24, 0) > 0
    # invalid dimensions give 0
    assert lib.lapnys_ctx_bytes(1, 1, 196, 32, 48, 20, 0) > 0       # a non-square m is fine
    assert lib.lapnys_ctx_bytes(1, 1, 2048, 32, 1089, 20, 0) == 0   # m > 1024
    assert lib.lapnys_ctx_bytes(1, 1, 16, 32, 25, 20, 0) == 0       # m > N
    assert lib.lapnys_ctx_bytes(1, 1, 196, 32, 49, -1, 0) == 0      # iters < 0
    assert lib.lapnys_workspace_bytes(0, 1, 196, 32, 49, 20, 0) == 0


def test_ctx_offsets_are_ordered_and_aligned(lib):
    from laplacian_nystr_linear_gb300 import _lib
    lay = _lib.CtxLayout()
    assert lib.lapnys_ctx_offsets(2, 3, 784, 64, 49, 20, 1, ctypes.byref(lay)) == 0
    offs = [getattr(lay, n) for n, _ in _lib.CtxLayout._fields_]
    assert offs == sorted(offs)
    assert all(o % 256 == 0 for o in offs)
    assert lay.total == lib.lapnys_ctx_bytes(2, 3, 784, 64, 49, 20, 1)


def test_strerror(lib):
    for code in range(7):
        assert lib.lapnys_strerror(code)
    assert b"unknown" in lib.lapnys_strerror(99)


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: every call below fails validation


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=1, N=196, d=32, gh=14, gw=14, m=49,
             lam=32.0, eps=1e-3, iters=20, tied=0, stream=None, dtype=0, flags=0, ctx=None,
             ctx_bytes=0, ws=FAKE, ws_bytes=0)
    a.update(kw)
    return lib.lapnys_fwd(a["q"], a["k"], a["v"], a["out"], a["B"], a["H"], a["N"], a["d"], a["gh"],
                          a["gw"], a["m"], a["lam"], a["eps"], a["iters"], a["tied"], a["stream"],
                          a["dtype"], a["flags"], a["ctx"], a["ctx_bytes"], a["ws"], a["ws_bytes"])


def test_fwd_rejects_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ENOSPC, LAPNYS_ENOTSUP
    assert _fwd(lib, N=195) == LAPNYS_EINVAL                       # N != grid_h * grid_w
    assert _fwd(lib, m=225) == LAPNYS_EINVAL                       # a 15 x 15 landmark grid on 14 x 14 tokens
    assert _fwd(lib, m=58) == LAPNYS_EINVAL                        # 58 = 2 x 29: 29 > 14 columns
    assert _fwd(lib, m=0) == LAPNYS_EINVAL
    # adaptive windows (6 does not divide 14) and non-square m pass validation (then fail on ws)
    assert _fwd(lib, m=36) == LAPNYS_ENOSPC
    assert _fwd(lib, m=48) == LAPNYS_ENOSPC
    assert _fwd(lib, lam=0.0) == LAPNYS_EINVAL
    assert _fwd(lib, lam=float("nan")) == LAPNYS_EINVAL
    assert _fwd(lib, eps=-1.0) == LAPNYS_EINVAL
    assert _fwd(lib, iters=-1) == LAPNYS_EINVAL
    assert _fwd(lib, dtype=7) == LAPNYS_EINVAL
    assert _fwd(lib, flags=8) == LAPNYS_EINVAL  # unknown bit (1: norm, 2: Gaussian, 4: batch stats)
    assert _fwd(lib, flags=4) == LAPNYS_EINVAL  # batch-pooled statistics without the norm
    assert _fwd(lib, flags=5) == LAPNYS_ENOSPC  # with it: valid (then fails on ws)
    assert _fwd(lib, flags=7) == LAPNYS_ENOSPC
    assert _fwd(lib, q=None) == LAPNYS_EINVAL
    assert _fwd(lib, out=ctypes.c_void_p((1 << 20) + 4)) == LAPNYS_EINVAL   # misaligned
    assert _fwd(lib, tied=1, k=ctypes.c_void_p(2 << 20)) == LAPNYS_EINVAL  # tied but k != q
    assert _fwd(lib, d=24) == LAPNYS_ENOTSUP
    assert _fwd(lib, ws_bytes=16) == LAPNYS_ENOSPC
    need = lib.lapnys_workspace_bytes(1, 1, 196, 32, 49, 20, 0)
    assert _fwd(lib, ws_bytes=need, ctx=FAKE, ctx_bytes=16) == LAPNYS_ENOSPC


def test_bwd_rejects_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ENOSPC

    def bwd(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dout=FAKE, ctx=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, tied=0,
                 ws_bytes=0)
        a.update(kw)
        return lib.lapnys_bwd(a["q"], a["k"], a["v"], a["dout"], a["ctx"], a["dq"], a["dk"],
                              a["dv"], 1, 1, 196, 32, 14, 14, 49, 32.0, 1e-3, 20, a["tied"], None,
                              0, 0, FAKE, a["ws_bytes"])

    assert bwd(ctx=None) == LAPNYS_EINVAL
    assert bwd(dk=None) == LAPNYS_EINVAL                  # untied needs dk
    assert bwd(tied=1, k=None) == LAPNYS_EINVAL           # tied forbids dk
    assert bwd() == LAPNYS_ENOSPC


def test_launch_counter_starts_at_zero_without_gpu(lib):
    assert lib.lapnys_launch_count() == 0


# ---- the attention block -------------------------------------------------------
def test_block_sizes(lib):
    # PVT-like layer: 8 x 16384 tokens, C = 512, 8 heads of 64, m = 256
    c = lib.lapnys_block_ctx_bytes(8, 16384, 512, 8, 64, 256, 24, 0, 1, 0)
    attn = lib.lapnys_ctx_bytes(8, 8, 16384, 64, 256, 24, 0)
    assert c >= attn + 4 * 8 * 16384 * 512 * 2       # + saved Q, K, V, concatenated heads (bf16)
    assert lib.lapnys_block_ctx_bytes(8, 16384, 512, 8, 64, 256, 24, 1, 1, 0) < c   # tied: no K
    assert lib.lapnys_block_workspace_bytes(8, 16384, 512, 8, 64, 256, 24, 0, 1, 0) > 0
    assert lib.lapnys_block_ctx_bytes(1, 196, 12, 1, 32, 49, 20, 0, 0, 0) == 0    # C % 8 != 0
    assert lib.lapnys_block_ctx_bytes(1, 196, 64, 1, 32, 49, 20, 2, 0, 0) == 0    # tied not 0/1
    assert lib.lapnys_block_ctx_bytes(1, 196, 64, 1, 32, 49, 20, 0, 7, 0) == 0    # dtype
    assert lib.lapnys_block_workspace_bytes(1, 16, 64, 1, 32, 25, 20, 0, 0, 0) == 0  # m > N


def _block_fwd(lib, **kw):
    a = dict(x=FAKE, w=FAKE, b=None, wo=FAKE, bo=None, y=FAKE, B=1, N=196, C=64, H=2, d=32, gh=14,
             gw=14, m=49, lam=32.0, eps=1e-3, iters=20, tied=0, dtype=0, flags=0, ctx=None,
             ctx_bytes=0, ws=FAKE, ws_bytes=0)
    a.update(kw)
    return lib.lapnys_block_fwd(a["x"], a["w"], a["b"], a["wo"], a["bo"], a["y"], a["B"], a["N"],
                                a["C"], a["H"], a["d"], a["gh"], a["gw"], a["m"], a["lam"], a["eps"],
                                a["iters"], a["tied"], None, a["dtype"], a["flags"], a["ctx"],
                                a["ctx_bytes"], a["ws"], a["ws_bytes"])


def test_block_fwd_rejects_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ENOSPC, LAPNYS_ENOTSUP
    assert _block_fwd(lib, C=12) == LAPNYS_EINVAL                  # C not a multiple of 8
    assert _block_fwd(lib, N=195) == LAPNYS_EINVAL                 # N != grid_h * grid_w
    assert _block_fwd(lib, tied=2) == LAPNYS_EINVAL
    assert _block_fwd(lib, flags=4) == LAPNYS_EINVAL               # batch statistics without norm
    assert _block_fwd(lib, x=None) == LAPNYS_EINVAL
    assert _block_fwd(lib, y=ctypes.c_void_p((1 << 20) + 8)) == LAPNYS_EINVAL   # misaligned
    assert _block_fwd(lib, b=ctypes.c_void_p((1 << 20) + 4)) == LAPNYS_EINVAL   # misaligned bias
    assert _block_fwd(lib, d=24) == LAPNYS_ENOTSUP
    assert _block_fwd(lib, ws_bytes=16) == LAPNYS_ENOSPC
    need = lib.lapnys_block_workspace_bytes(1, 196, 64, 2, 32, 49, 20, 0, 0, 0)
    assert _block_fwd(lib, ws_bytes=need, ctx=FAKE, ctx_bytes=16) == LAPNYS_ENOSPC


def test_block_bwd_rejects_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ENOSPC

    def bwd(**kw):
        a = dict(ctx=FAKE, dx=FAKE, dw=FAKE, db=None, dwo=FAKE, dbo=None, ws_bytes=0)
        a.update(kw)
        return lib.lapnys_block_bwd(FAKE, FAKE, FAKE, FAKE, a["ctx"], a["dx"], a["dw"], a["db"],
                                    a["dwo"], a["dbo"], 1, 196, 64, 2, 32, 14, 14, 49, 32.0, 1e-3, 20,
                                    0, None, 0, 0, FAKE, a["ws_bytes"])

    assert bwd(ctx=None) == LAPNYS_EINVAL
    assert bwd(dx=None) == LAPNYS_EINVAL
    assert bwd(dwo=None) == LAPNYS_EINVAL
    assert bwd(db=ctypes.c_void_p((1 << 20) + 4)) == LAPNYS_EINVAL
    assert bwd() == LAPNYS_ENOSPC


def test_matmul_rejects_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ENOTSUP

    def mm(**kw):
        a = dict(A=FAKE, B=FAKE, E=None, C=FAKE, batch=1, M=64, N=64, K=64, lda=64, ldb=64, lde=0,
                 ldc=64, beta=0.0, engine=0)
        a.update(kw)
        return lib.lapnys_matmul(a["A"], a["B"], a["E"], a["C"], a["batch"], a["M"], a["N"], a["K"],
                                 0, 0, a["lda"], a["ldb"], a["lde"], a["ldc"], 0, 0, 0, 0, 1.0,
                                 a["beta"], a["engine"], None)

    assert mm(A=None) == LAPNYS_EINVAL
    assert mm(batch=0) == LAPNYS_EINVAL
    assert mm(K=0) == LAPNYS_EINVAL
    assert mm(beta=1.0) == LAPNYS_EINVAL            # beta != 0 needs E
    assert mm(lda=0) == LAPNYS_EINVAL
    assert mm(engine=2) == LAPNYS_EINVAL            # no such engine
    assert mm(engine=1, M=62, lda=62) == LAPNYS_ENOTSUP   # tensor cores want multiples of 4


def test_static_forward_and_pool_reject_bad_arguments(lib):
    from laplacian_nystr_linear_gb300._lib import LAPNYS_EINVAL, LAPNYS_ESCRATCH

    def fs(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=1, N=196, d=32, gh=14, gw=14, m=49,
                 tied=0, flags=0)
        a.update(kw)
        return lib.lapnys_fwd_static(a["q"], a["k"], a["v"], a["out"], a["B"], a["H"], a["N"],
                                     a["d"], a["gh"], a["gw"], a["m"], 32.0, 1e-3, 20, a["tied"],
                                     None, 0, a["flags"])

    assert fs(N=195) == LAPNYS_EINVAL
    assert fs(q=None) == LAPNYS_EINVAL
    assert fs(tied=1, k=ctypes.c_void_p(2 << 20)) == LAPNYS_EINVAL
    assert fs(out=ctypes.c_void_p((1 << 20) + 4)) == LAPNYS_EINVAL
    # the 16K-token workload needs far more forward scratch than the built-in 32 MiB
    assert fs(B=8, H=8, N=16384, d=64, gh=128, gw=128, m=256) == LAPNYS_ESCRATCH
    assert lib.lapnys_pool(FAKE, FAKE, None, 1, 1, 195, 32, 14, 14, 49, 0, None) == LAPNYS_EINVAL
    assert lib.lapnys_pool(None, FAKE, None, 1, 1, 196, 32, 14, 14, 49, 0, None) == LAPNYS_EINVAL
    assert lib.lapnys_pool(FAKE, FAKE, None, 1, 1, 196, 32, 14, 14, 225, 0, None) == LAPNYS_EINVAL


def test_wait_selftest_rejects_poll_counts_out_of_range(lib):
    from laplacian_nystr_linear_gb300 import _lib
    before = lib.lapnys_launch_count()
    assert lib.lapnys_wait_selftest(0, None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_wait_selftest(-5, None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_wait_selftest((1 << 22) + 1, None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_launch_count() == before


def test_instrumentation_rejects_bad_arguments(lib):
    import ctypes as ct
    from laplacian_nystr_linear_gb300 import _lib
    assert lib.lapnys_profile_enable(3) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_profile_enable(-1) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_profile_enable(0) == _lib.LAPNYS_OK
    n = ct.c_ulonglong(0)
    before = lib.lapnys_launch_count()
    assert lib.lapnys_fma_probe(2, 10, ct.c_void_p(16), ct.byref(n), None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_fma_probe(0, 0, ct.c_void_p(16), ct.byref(n), None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_fma_probe(0, 10, None, ct.byref(n), None) == _lib.LAPNYS_EINVAL
    assert lib.lapnys_launch_count() == before
