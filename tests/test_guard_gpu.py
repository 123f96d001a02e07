"""Guard regions around every caller-owned buffer (needs a GPU).

Each output, ctx and workspace buffer handed to the C ABI sits in the middle of
a larger allocation: GUARD bytes of a fixed pattern before it and after it, and
its own bytes set to 0xFF (NaN in float32 and bf16) before the call.  After
each call the test checks that
  - every guard byte still holds the pattern (no kernel wrote outside the
    buffer it was given, for ragged token tiles, odd d and m, tied, norm,
    Gaussian, and the block's projections);
  - no output element is still NaN (every element was written);
  - the outputs equal, bit for bit, those of the same call on plain buffers
    (the results do not depend on the buffers' addresses or prior contents).
The arithmetic itself is checked against the oracle by the parity tests.
"""
from __future__ import annotations

import pytest
import torch

from laplacian_nystr_linear_gb300 import api
from laplacian_nystr_linear_gb300.inputs import block_inputs, random_inputs

from tests._parity import TDT, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096     # bytes on each side; a multiple of 256 keeps the body's alignment
PATTERN = 0xA5   # guard bytes
FILL = 0xFF      # body bytes before the call


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


class Guarded:
    """A buffer of nbytes with GUARD pattern bytes on either side."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.raw = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.raw[GUARD:GUARD + self.nbytes].fill_(FILL)

    @property
    def body(self) -> torch.Tensor:
        return self.raw[GUARD:GUARD + self.nbytes]

    def view(self, dtype: torch.dtype, shape) -> torch.Tensor:
        return self.body.view(dtype).view(shape)

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all().item()) and bool((tail == PATTERN).all().item())


def _guarded_tensor(shape, dtype) -> tuple[Guarded, torch.Tensor]:
    n = 1
    for s in shape:
        n *= s
    g = Guarded(n * torch.empty((), dtype=dtype).element_size())
    return g, g.view(dtype, shape)


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return bool(torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                            b.view(torch.uint8) if b.dtype != torch.uint8 else b))


ATTN = [
    # (name, Params(B, H, grid_h, grid_w, d, m, lam, eps, iters, tied, norm, kernel, norm_batch))
    ("f32_ragged_m4_d16", api.Params(1, 2, 10, 12, 16, 4, 16.0, 1e-3, 6)),
    ("f32_m1_d16", api.Params(1, 1, 8, 8, 16, 1, 16.0, 1e-3, 3)),
    ("f32_iters0", api.Params(1, 1, 8, 8, 32, 16, 32.0, 1e-3, 0)),
    ("f32_norm_batch_d32_m64", api.Params(2, 2, 16, 16, 32, 64, 32.0, 1e-3, 8, False, True, "laplace", True)),
    ("bf16_tied_norm_m49_d64", api.Params(1, 2, 14, 14, 64, 49, 64.0, 1e-3, 8, True, True)),
    ("bf16_tc_m256_d64", api.Params(1, 2, 32, 32, 64, 256, 64.0, 1e-3, 10)),
    ("bf16_tc_gauss_m100_d32", api.Params(1, 1, 18, 22, 32, 100, 32.0, 1e-3, 8, False, False, "gauss")),
    ("bf16_d128_m64", api.Params(1, 1, 16, 16, 128, 64, 128.0, 1e-3, 6)),
    # m <= 64, Q != K with a ctx: kernel values beside the solver, the streaming
    # product (and, with the feature map, statistics from the stored values, Z)
    ("bf16_split_norm_m49_d64", api.Params(2, 2, 14, 14, 64, 49, 64.0, 1e-3, 8, False, True)),
    ("bf16_split_ragged_m16_d32", api.Params(1, 3, 10, 12, 32, 16, 32.0, 1e-3, 6)),
]


@pytest.mark.parametrize("name,p", ATTN, ids=[c[0] for c in ATTN])
def test_attention_buffers_guarded(name, p):
    dtype = "bf16" if name.startswith("bf16") else "f32"
    tdt = TDT[dtype]
    inp = random_inputs(71, p.B, p.H, p.N, p.d, dtype, tied=p.tied)
    q = to_dev(inp["q"], dtype)
    k = q if p.tied else to_dev(inp["k"], dtype)
    v = to_dev(inp["v"], dtype)
    dout = to_dev(inp["dout"], dtype)
    shape = tuple(q.shape)

    # plain buffers (the forward with and without a ctx may take different paths)
    out0, ctx0 = api.fwd(q, k, v, p, need_ctx=True)
    dq0, dk0, dv0 = api.bwd(q, k, v, dout, ctx0, p)
    out0n, _ = api.fwd(q, k, v, p, need_ctx=False)

    # guarded buffers
    g_out, out = _guarded_tensor(shape, tdt)
    g_ctx = Guarded(api.ctx_bytes(p))
    g_ws = Guarded(api.workspace_bytes(p))
    api.fwd(q, k, v, p, out=out, ctx=g_ctx.body, ws=g_ws.body, need_ctx=True)
    torch.cuda.synchronize()
    assert g_out.intact() and g_ctx.intact() and g_ws.intact(), "forward wrote outside a buffer"

    g_dq, dq = _guarded_tensor(shape, tdt)
    g_dv, dv = _guarded_tensor(shape, tdt)
    g_dk, dk = (None, None) if p.tied else _guarded_tensor(shape, tdt)
    g_ws2 = Guarded(api.workspace_bytes(p))
    api.bwd(q, k, v, dout, g_ctx.body, p, dq=dq, dk=dk, dv=dv, ws=g_ws2.body)
    torch.cuda.synchronize()
    for g in (g_dq, g_dv, g_dk, g_ctx, g_ws2):
        if g is not None:
            assert g.intact(), "backward wrote outside a buffer"

    # the output-only forward (no ctx) into a guarded buffer
    g_out2, out2 = _guarded_tensor(shape, tdt)
    g_ws3 = Guarded(api.workspace_bytes(p))
    api.fwd(q, k, v, p, out=out2, ws=g_ws3.body, need_ctx=False)
    torch.cuda.synchronize()
    assert g_out2.intact() and g_ws3.intact()

    for got, ref in ((out, out0), (out2, out0n), (dq, dq0), (dv, dv0), (dk, dk0)):
        if ref is None:
            continue
        assert not torch.isnan(got.float()).any(), "an output element was not written"
        assert _same(got, ref), "guarded and plain buffers gave different results"


BLOCK = [
    # (name, B, grid_h, grid_w, C, H, d, m, dtype, iters, tied, norm, kernel, bias)
    ("f32_tied_norm_ragged", 2, 10, 12, 48, 3, 16, 9, "f32", 6, True, True, "laplace", False),
    ("bf16_heads_ragged", 2, 10, 12, 72, 2, 64, 9, "bf16", 6, False, False, "laplace", True),
    ("bf16_rows_h3d16", 2, 8, 8, 48, 3, 16, 16, "bf16", 6, False, False, "laplace", True),
    ("bf16_tc_gauss", 1, 16, 16, 256, 4, 64, 128, "bf16", 8, False, False, "gauss", True),
]


@pytest.mark.parametrize("case", BLOCK, ids=[c[0] for c in BLOCK])
def test_block_buffers_guarded(case):
    name, B, gh, gw, C, H, d, m, dtype, iters, tied, norm, kernel, bias = case
    tdt = TDT[dtype]
    a = api.Params(B, H, gh, gw, d, m, float(d), 1e-3, iters, tied, norm, kernel)
    bp = api.BlockParams(a, C)
    raw = block_inputs(81, B, a.N, C, H, d, dtype, tied=tied, bias=bias)
    t = {n: (None if x is None else to_dev(x, dtype)) for n, x in raw.items()}
    x, w_qkv, b_qkv, w_o, b_o, dy = (t[n] for n in ("x", "w_qkv", "b_qkv", "w_o", "b_o", "dy"))

    y0, ctx0 = api.block_fwd(x, w_qkv, b_qkv, w_o, b_o, bp)
    ref = api.block_bwd(x, w_qkv, w_o, dy, ctx0, bp, bias_grads=bias)

    g_y, y = _guarded_tensor(tuple(x.shape), tdt)
    g_ctx = Guarded(api.block_ctx_bytes(bp, tdt))
    g_ws = Guarded(api.block_workspace_bytes(bp, tdt))
    api.block_fwd(x, w_qkv, b_qkv, w_o, b_o, bp, y=y, ctx=g_ctx.body, ws=g_ws.body)
    torch.cuda.synchronize()
    assert g_y.intact() and g_ctx.intact() and g_ws.intact(), "block forward wrote outside a buffer"

    g_dx, dx = _guarded_tensor(tuple(x.shape), tdt)
    g_dw, dw = _guarded_tensor(tuple(w_qkv.shape), tdt)
    g_dwo, dwo = _guarded_tensor(tuple(w_o.shape), tdt)
    g_db, db = (_guarded_tensor((w_qkv.shape[1],), tdt) if bias else (None, None))
    g_dbo, dbo = (_guarded_tensor((C,), tdt) if bias else (None, None))
    g_ws2 = Guarded(api.block_workspace_bytes(bp, tdt))
    got = api.block_bwd(x, w_qkv, w_o, dy, g_ctx.body, bp, bias_grads=bias, dx=dx, dw_qkv=dw,
                        db_qkv=db, dw_o=dwo, db_o=dbo, ws=g_ws2.body)
    torch.cuda.synchronize()
    for g in (g_dx, g_dw, g_dwo, g_db, g_dbo, g_ctx, g_ws2):
        if g is not None:
            assert g.intact(), "block backward wrote outside a buffer"

    for a_, b_ in zip((y,) + tuple(got), (y0,) + tuple(ref)):
        if b_ is None:
            continue
        assert not torch.isnan(a_.float()).any(), "an output element was not written"
        assert _same(a_, b_), "guarded and plain buffers gave different results"
