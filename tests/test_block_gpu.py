"""The attention block (QKV projection, per-head attention, output projection)
through the C ABI against the fp64 oracle's block on seeded inputs (needs a GPU).

Tolerance: relative Frobenius error <= 1e-4 (float32) and <= 2e-2 (bf16) for y
and for every gradient (dx, dW_qkv, db_qkv, dW_o, db_o), and per element
|gpu - oracle| <= R |oracle| + A rms(oracle tensor) with the attention's (R, A)
(tests/_parity.py); Q, K, V and the gradients are rounded once to the element
type, as the attention's own tolerance already allows.
"""
import dataclasses

import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import api
from laplacian_nystr_linear_gb300.inputs import block_inputs
from oracle import lapnys_oracle as orc

from tests._parity import EW, TOL, _log, elementwise_excess, rel, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@dataclasses.dataclass(frozen=True)
class Case:
    name: str
    B: int
    grid_h: int
    grid_w: int
    C: int
    H: int
    d: int
    m: int
    dtype: str = "f32"
    iters: int = 8
    tied: bool = False
    norm: bool = False
    norm_batch: bool = False
    kernel: str = "laplace"
    bias: bool = True

    @property
    def N(self):
        return self.grid_h * self.grid_w

    def params(self):
        a = api.Params(self.B, self.H, self.grid_h, self.grid_w, self.d, self.m, float(self.d),
                       1e-3, self.iters, self.tied, self.norm, self.kernel, self.norm_batch)
        return api.BlockParams(a, self.C)


CASES = [
    Case("f32", 2, 8, 8, 64, 2, 32, 16),
    Case("f32_tied_norm_ragged_nobias", 2, 10, 12, 48, 3, 16, 9, tied=True, norm=True, bias=False),
    Case("bf16_norm_batch", 2, 14, 14, 128, 2, 64, 49, dtype="bf16", norm=True, norm_batch=True),
    Case("bf16_tc", 2, 16, 16, 256, 4, 64, 128, dtype="bf16", iters=10),
    Case("bf16_tc_gauss_tied", 1, 16, 16, 64, 2, 32, 100, dtype="bf16", tied=True, kernel="gauss"),
    Case("f32_d128", 1, 8, 8, 128, 1, 128, 64, iters=6),
    # bf16, per-head operands read in place: ragged token tiles (120 tokens), C = 72
    # (a ragged K step, N tile and weight-gradient M tile)
    Case("bf16_heads_ragged", 2, 10, 12, 72, 2, 64, 9, dtype="bf16"),
    # bf16 with H d = 48 (not a multiple of 64): concatenated heads through the
    # layout kernels and the same product on row-major operands
    Case("bf16_rows_h3d16", 2, 8, 8, 48, 3, 16, 16, dtype="bf16", iters=6),
    # bf16 with d = 128 (a 64-wide K step is half a head), no bias
    Case("bf16_d128_nobias", 1, 8, 8, 128, 1, 128, 16, dtype="bf16", iters=6, bias=False),
]


def _dev(a, dtype):
    return None if a is None else to_dev(a, dtype)


def run_gpu(c: Case, inp: dict):
    bp = c.params()
    x, w, b, wo, bo, dy = (_dev(inp[n], c.dtype) for n in ("x", "w_qkv", "b_qkv", "w_o", "b_o", "dy"))
    y, ctx = api.block_fwd(x, w, b, wo, bo, bp)
    grads = api.block_bwd(x, w, wo, dy, ctx, bp, bias_grads=c.bias)
    torch.cuda.synchronize()
    out = {"y": to_np(y)}
    out.update({n: (None if t is None else to_np(t))
                for n, t in zip(("dx", "dw_qkv", "db_qkv", "dw_o", "db_o"), grads)})
    return out


def run_oracle(c: Case, inp: dict):
    # a bf16 layer stores Q, K, V, the heads' outputs and the gradients in bf16
    # (the block's reading); the oracle rounds at the same points
    y, st = orc.block_forward(inp["x"], inp["w_qkv"], inp["b_qkv"], inp["w_o"], inp["b_o"], c.H,
                              c.d, c.grid_h, c.grid_w, c.m, float(c.d), 1e-3, c.iters, c.norm,
                              c.kernel, c.norm_batch, c.tied,
                              store="bf16" if c.dtype == "bf16" else "f64")
    g = orc.block_backward(st, inp["dy"])
    return dict(zip(("y", "dx", "dw_qkv", "db_qkv", "dw_o", "db_o"), (y,) + g))


@pytest.mark.parametrize("c", CASES, ids=lambda c: c.name)
def test_block_matches_oracle(c):
    inp = block_inputs(90 + c.m, c.B, c.N, c.C, c.H, c.d, c.dtype, c.tied, c.bias)
    g = run_gpu(c, inp)
    o = run_oracle(c, inp)
    errs = {n: rel(g[n], o[n]) for n in o if g.get(n) is not None}
    r, a = EW[c.dtype]
    ew = {n: elementwise_excess(g[n], o[n], r)[0] for n in errs}
    print(c.name, errs, ew)
    _log({"workload": "block_" + c.name, "dtype": c.dtype, "fro": errs, "ew_excess": ew,
          "R": r, "A": a})
    assert not c.bias or len(errs) == 6
    bad = {n: e for n, e in errs.items() if not e <= TOL[c.dtype]}
    assert not bad, f"{c.name}: {bad}"
    bad = {n: e for n, e in ew.items() if not e <= a}
    assert not bad, f"{c.name}: element-wise excess / rms above {a}: {bad}"


def test_block_autograd_wrapper_matches_raw_calls():
    c = CASES[0]
    inp = block_inputs(3, c.B, c.N, c.C, c.H, c.d, c.dtype, c.tied, True)
    g = run_gpu(c, inp)
    leaves = {n: to_dev(inp[n], "f32").requires_grad_(True) for n in ("x", "w_qkv", "b_qkv", "w_o",
                                                                     "b_o")}
    y = api.attention_block(leaves["x"], leaves["w_qkv"], leaves["b_qkv"], leaves["w_o"],
                            leaves["b_o"], (c.grid_h, c.grid_w), c.H, c.m, iters=c.iters)
    y.backward(to_dev(inp["dy"], "f32"))
    np.testing.assert_array_equal(y.detach().cpu().numpy(), g["y"].astype(np.float32))
    for n, gn in (("x", "dx"), ("w_qkv", "dw_qkv"), ("b_qkv", "db_qkv"), ("w_o", "dw_o"),
                  ("b_o", "db_o")):
        np.testing.assert_array_equal(leaves[n].grad.cpu().numpy(), g[gn].astype(np.float32))


def test_block_deterministic_and_inference_matches_training():
    c = CASES[3]
    inp = block_inputs(5, c.B, c.N, c.C, c.H, c.d, c.dtype, c.tied, True)
    a = run_gpu(c, inp)
    b = run_gpu(c, inp)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
    bp = c.params()
    x, w, bb, wo, bo = (_dev(inp[n], c.dtype) for n in ("x", "w_qkv", "b_qkv", "w_o", "b_o"))
    y, ctx = api.block_fwd(x, w, bb, wo, bo, bp, need_ctx=False)
    assert ctx is None
    np.testing.assert_array_equal(to_np(y), a["y"])


def test_block_hires16k_layer():
    # the 128 x 128 grid with 8 heads of 64 (C = 512), m = 256, 24 iterations,
    # bf16, all 8 batch elements in one call: y of batch element 0 against the
    # oracle, and the bias gradients against their definition (column sums)
    c = Case("hires16k_layer", 8, 128, 128, 512, 8, 64, 256, dtype="bf16", iters=24)
    inp = block_inputs(7, c.B, c.N, c.C, c.H, c.d, c.dtype, c.tied, True)
    g = run_gpu(c, inp)
    y0, _ = orc.block_forward(inp["x"][:1], inp["w_qkv"], inp["b_qkv"], inp["w_o"], inp["b_o"],
                              c.H, c.d, c.grid_h, c.grid_w, c.m, float(c.d), 1e-3, c.iters,
                              store="bf16")
    e = rel(g["y"][0], y0[0])
    r, a = EW["bf16"]
    ex = elementwise_excess(g["y"][0], y0[0], r)[0]
    print("hires16k_layer y[0]", e, ex)
    _log({"workload": "block_hires16k_layer", "dtype": "bf16", "fro": {"y": e},
          "ew_excess": {"y": ex}, "R": r, "A": a})
    assert e <= TOL["bf16"] and ex <= a
    dy = inp["dy"].astype(np.float64)
    assert rel(g["db_o"], dy.sum(axis=(0, 1))) <= TOL["bf16"]
    assert np.isfinite(g["dx"]).all() and np.isfinite(g["dw_qkv"]).all()
