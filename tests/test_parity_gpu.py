"""CUDA path against the fp64 oracle on seeded inputs (needs a GPU).

Tolerance: per (b, h) slice, |gpu - oracle|_F / |oracle|_F <= 1e-4 for float32
tensors and <= 2e-2 for bf16 tensors (fp32 accumulation), and per element
|gpu - oracle| <= R |oracle| + A rms(oracle slice) (tests/_parity.py); landmark
indices bit-exact.  Full-size workloads are checked on sampled slices, computed
by the oracle one slice at a time, in the same launch configuration the
benchmark times (the same library call on the whole batch).
"""
import dataclasses

import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import api
from laplacian_nystr_linear_gb300.inputs import (WORKLOADS, Workload, make_inputs, random_inputs,
                                                 round_bf16)
from oracle import lapnys_oracle as orc

from tests._oracle_pool import oracle_slices
from tests._parity import (compare, gpu_run, oracle_run, params_of, rel, to_dev,
                           top_outlier_slices)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


def _small(name, **kw):
    base = dict(cfg=9, B=1, H=1, grid_h=8, grid_w=8, d=32, m=16, dtype="f32", iters=8)
    base.update(kw)
    return Workload(name=name, **base)


# ---------------------------------------------------------------------------
# landmarks
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("gh,gw,m,d,dtype", [(14, 14, 49, 32, "f32"), (56, 56, 49, 64, "bf16"),
                                             (128, 128, 256, 64, "bf16"), (10, 12, 4, 16, "f32"),
                                             (8, 8, 64, 128, "f32"), (6, 6, 1, 64, "bf16"),
                                             # adaptive windows (grid not divisible)
                                             (14, 14, 16, 32, "f32"), (10, 12, 9, 16, "bf16"),
                                             (18, 22, 100, 64, "bf16"),
                                             # non-square m
                                             (16, 8, 32, 64, "f32"), (20, 12, 15, 32, "f32"),
                                             (7, 9, 6, 16, "bf16"), (24, 16, 96, 32, "bf16")])
def test_pool_indices_exact_and_values(gh, gw, m, d, dtype):
    inp = random_inputs(100 + m, 2, 3, gh * gw, d, dtype)
    k = to_dev(inp["k"], dtype)
    L, idx = api.pool(k, (gh, gw), m)
    torch.cuda.synchronize()
    ref_idx = orc.pool_index(gh, gw, m)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    Lg = L.cpu().numpy()
    for b in range(2):
        for h in range(3):
            Lr = orc.pool_landmarks(inp["k"][b, h], ref_idx, m)
            assert rel(Lg[b, h], Lr) < 1e-6


# ---------------------------------------------------------------------------
# forward intermediates (landmark matrix, alpha, every Newton-Schulz iterate, W, W-hat)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wname", ["tiny", "tiny_mN"])
def test_forward_intermediates(wname):
    w = WORKLOADS[wname]
    inp = make_inputs(w)
    g = gpu_run(w, inp)
    o = oracle_run(w, inp)
    s = o["saved"][(0, 0)]
    c = g["ctx"]
    assert rel(c["L"][0, 0], s["L"]) < 1e-6
    assert rel(c["A"][0, 0], s["A"]) < 1e-6
    alpha, n1, ninf, jc, ic = orc.ns_scale(s["A"])
    np.testing.assert_allclose(c["alpha"][0, 0, :3], [alpha, n1, ninf], rtol=1e-5)
    code = int(c["alpha"][0, 0, 3:4].view(np.int32)[0])
    assert (code & 0xFFFF, code >> 16) == (jc, ic)
    for t in range(w.iters + 1):
        assert rel(c["X"][0, 0, t], s["X"][t]) < 1e-4, t
    assert rel(c["W"][0, 0], s["W"]) < 1e-5
    assert rel(c["What"][0, 0], s["What"]) < 1e-4
    np.testing.assert_array_equal(c["idx"], s["idx"])
    # kernel values kept for the backward: P = k(Q, L) and C = k(L, K), token-major
    assert rel(c["P"][0, 0], s["P"]) < 1e-6
    assert rel(c["C"][0, 0], s["C"].T) < 1e-6


# bf16 with d = 32 / 64 and m > 64 takes the tensor-core forward passes (tcgen05,
# 128-row tiles): ragged token counts, landmark counts off the 64 / 128 tiles
TC_FWD = [
    _small("tc_m100", dtype="bf16", d=64, grid_h=20, grid_w=20, m=100, iters=8),
    _small("tc_m81_norm", dtype="bf16", d=32, grid_h=18, grid_w=18, m=81, iters=8, norm=True),
    _small("tc_m144_batch", dtype="bf16", d=64, grid_h=24, grid_w=24, m=144, iters=8, B=2, H=2),
    _small("tc_mN_tied", dtype="bf16", d=64, grid_h=16, grid_w=16, m=256, iters=6, tied=True),
]


@pytest.mark.parametrize("w", TC_FWD, ids=lambda w: w.name)
def test_tensor_core_forward_intermediates(w):
    inp = random_inputs(31 + w.m, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))
    for (b, h), s in o["saved"].items():
        c = g["ctx"]
        assert rel(c["W"][b, h], s["W"]) < 1e-5          # C V with C as three bf16 planes
        assert rel(c["C"][b, h], s["C"].T) < 1e-6        # kernel values stored as computed
        if w.tied:
            # Q = K: the forward keeps C alone, which is P's transpose (the query
            # pass and the backward read it as P)
            assert rel(c["C"][b, h], s["P"]) < 1e-6
        else:
            assert rel(c["P"][b, h], s["P"]) < 1e-6


def test_norm_statistics():
    w = WORKLOADS["pvt3"]
    inp = make_inputs(w)
    g = gpu_run(w, inp)
    o = oracle_run(w, inp, slices={(0, 0), (31, 4)})
    for (b, h), s in o["saved"].items():
        mu, var, sd = s["stats"]
        st = g["ctx"]["stats"][b, h]
        assert rel(st[0], mu) < 1e-5
        assert rel(st[1], var) < 1e-4
        assert rel(st[2], 1.0 / sd) < 1e-4


# ---------------------------------------------------------------------------
# forward outputs at the workload shapes
# ---------------------------------------------------------------------------
# The full-size workloads: the four slices with the most heavy-tailed tokens
# plus the first and the last slice (hires16k), and four heads spread over the
# batch of the tied 65K-token workload; the oracle runs them in parallel.
FWD_SLICES = {
    "tiny": None, "tiny_mN": None, "pvt1": None, "pvt2": None, "pvt3": None,
    "hires16k": top_outlier_slices(WORKLOADS["hires16k"], 4) | {(0, 0), (7, 7)},
    "tied64k": {(0, 0), (0, 5), (0, 10), (0, 15)},
}
POOLED = {"hires16k", "tied64k"}


@pytest.mark.parametrize("wname", list(FWD_SLICES))
def test_forward_workloads(wname):
    w = WORKLOADS[wname]
    inp = make_inputs(w, with_grad=False)
    g = gpu_run(w, inp)
    del inp
    if wname in POOLED:
        o = oracle_slices(w, FWD_SLICES[wname])
    else:
        o = oracle_run(w, make_inputs(w, with_grad=False), slices=FWD_SLICES[wname])
    print(w.name, compare(w, g, o, backward=False))


def test_one_landmark_per_token_reaches_exact_attention():
    # m = N, eps = 0, 30 iterations: the landmark matrix of this slice has
    # condition number ~240 and the iteration has converged (residual factor
    # (1 - alpha sigma_min^2)^(2^30) underflows), so Nystrom equals k(Q, K) V up
    # to fp32 rounding: the fp32 tolerance holds against exact attention too
    w = dataclasses.replace(WORKLOADS["tiny_mN"], eps=0.0, iters=30)
    inp = make_inputs(w)
    g = gpu_run(w, inp)
    compare(w, g, oracle_run(w, inp), backward=False)
    q, k, v = (inp[n][0, 0].astype(np.float64) for n in ("q", "k", "v"))
    S = orc.laplacian_kernel(q, k, w.lam)
    assert rel(g["out"][0, 0], S @ v) < 1e-4


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------
# hires16k: the six slices with the most heavy-tailed tokens, the first and the last
BWD_SLICES = {"pvt2": {(0, 0), (17, 1), (31, 1)}, "pvt3": {(0, 0), (31, 4)},
              "hires16k": top_outlier_slices(WORKLOADS["hires16k"], 6) | {(0, 0), (7, 7)}}


@pytest.mark.parametrize("wname", list(BWD_SLICES))
def test_backward_workloads(wname):
    w = WORKLOADS[wname]
    inp = make_inputs(w)
    g = gpu_run(w, inp, backward=True)
    if wname in POOLED:
        del inp
        o = oracle_slices(w, BWD_SLICES[wname], backward=True)
    else:
        o = oracle_run(w, inp, slices=BWD_SLICES[wname], backward=True)
    print(w.name, len(BWD_SLICES[wname]), compare(w, g, o, backward=True))


SMALL = [
    _small("f32"),
    _small("f32_norm", norm=True),
    _small("f32_tied", tied=True),
    _small("f32_tied_norm", tied=True, norm=True),
    _small("bf16", dtype="bf16", d=64),
    _small("ragged", grid_h=10, grid_w=12, m=4, d=16, iters=6),
    _small("ragged_large_m", grid_h=12, grid_w=12, m=144, d=16, iters=10),
    _small("m1", m=1, iters=3),
    _small("iters0", iters=0),
    _small("d128", d=128, m=64, iters=6),
    _small("tiny_grid", grid_h=2, grid_w=2, m=4, d=16, iters=5),
    _small("m81", grid_h=18, grid_w=18, m=81, d=32, iters=12, norm=True),
    _small("batch", B=3, H=2, grid_h=16, grid_w=16, m=16, d=64, iters=10),
    # one landmark per token with Q = K: every token ties with its own landmark
    _small("bf16_tied_mN", dtype="bf16", d=64, grid_h=4, grid_w=4, m=16, iters=6, tied=True),
    _small("bf16_mN", dtype="bf16", d=32, grid_h=8, grid_w=8, m=64, iters=6),
    # bf16, m <= 64 with the feature map and a ctx: kernel values beside the solver,
    # statistics from the stored values, Z, then the streaming product
    _small("bf16_norm_ragged", dtype="bf16", d=64, grid_h=10, grid_w=12, m=9, iters=6, norm=True),
    _small("bf16_norm_d32", dtype="bf16", d=32, grid_h=12, grid_w=12, m=36, iters=8, norm=True,
           B=2, H=2),
]


# Many slices of one or two 128-token tiles: the streaming C R product (dV, and
# the tied forward's O = C W-hat) then walks several slices per CTA, reusing its
# two operand-image buffers, with ragged last tiles.
MANY_SLICES = [
    _small("many_slices", dtype="bf16", B=40, H=16, d=64, m=16, iters=6),
    _small("many_slices_tied", dtype="bf16", B=40, H=16, d=64, m=16, iters=6, tied=True),
    _small("many_slices_d32_ragged", dtype="bf16", B=20, H=8, grid_h=12, grid_w=12, d=32, m=36,
           iters=6),
]


@pytest.mark.parametrize("w", MANY_SLICES, ids=lambda w: w.name)
def test_streaming_product_many_slices(w):
    inp = random_inputs(61 + w.m, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    slices = [(b, h) for b in range(0, w.B, 7) for h in range(0, w.H, 5)] + [(w.B - 1, w.H - 1)]
    o = oracle_run(w, inp, slices=slices, backward=True)
    print(w.name, len(slices), compare(w, g, o, backward=True))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_small_cases(w):
    inp = random_inputs(7 + w.m + w.d, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))


def test_constant_inputs_use_zero_sign():
    # every token equal: all L1 distances between tokens and landmarks are 0,
    # so sgn(0) = 0 decides the kernel gradient
    w = _small("const", grid_h=4, grid_w=4, m=4, d=16, iters=4)
    inp = random_inputs(3, 1, 1, w.N, w.d, "f32")
    inp["q"] = np.full_like(inp["q"], 0.25)
    inp["k"] = np.full_like(inp["k"], 0.25)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))


def test_constant_bf16_inputs_use_zero_sign():
    w = _small("const_bf16", dtype="bf16", grid_h=8, grid_w=8, m=16, d=64, iters=4)
    inp = random_inputs(4, 2, 2, w.N, w.d, "bf16")
    inp["q"] = np.full_like(inp["q"], -1.5)
    inp["k"] = np.full_like(inp["k"], -1.5)
    w = dataclasses.replace(w, B=2, H=2)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("m", [16, 64])
def test_ties_in_a_few_columns(dtype, m):
    # In 13 feature columns every K token of a pooling window holds the same
    # bf16 value, so that window's landmark equals it exactly and the window's
    # tokens tie with it (sgn(0) = 0); half of the Q tokens copy those values
    # too, the other columns stay random.  Reading those ties as sgn = -1
    # instead moves dq or dk of the oracle by at least 8e-3 (2.6e-2 and 4.5e-2
    # at m = 16), so bf16 is held to 5e-3 here, about 3x the bf16 rounding error
    # of the outputs, and fp32 to its usual 1e-4.
    w = _small("col_ties", dtype=dtype, grid_h=16, grid_w=16, m=m, d=64, iters=6)
    inp = random_inputs(11 + m, 1, 2, w.N, w.d, dtype)
    w = dataclasses.replace(w, B=1, H=2)
    s = int(round(m ** 0.5))
    r = w.grid_h // s
    rng = np.random.default_rng(m)
    for c in range(3, 64, 5):
        vals = round_bf16(rng.standard_normal((2, s, s)))
        for h in range(2):
            win = vals[h].repeat(r, 0).repeat(r, 1).reshape(-1)   # value of each token's window
            inp["k"][0, h, :, c] = win
            pick = rng.random(w.N) < 0.5
            inp["q"][0, h, pick, c] = win[rng.permutation(w.N)[pick]]
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, dtype, m, compare(w, g, o, backward=True, tol=5e-3 if dtype == "bf16" else None))


def _tie_positions(x, L):
    """(token, feature) positions where a token value equals a landmark value,
    and the number of (token, feature, landmark) ties per 32-token block."""
    N, d = x.shape
    per = np.zeros((N, d), np.int64)
    for c in range(d):
        per[:, c] = (x[:, c][:, None] == L[:, c][None, :]).sum(1)
    blocks = np.add.reduceat(per.sum(1), np.arange(0, N, 32))
    return np.argwhere(per > 0), blocks


@pytest.mark.parametrize("m", [16, 64])
def test_sparse_ties_are_corrected(m):
    # bf16 tokens meet a landmark value exactly a few times per 32-token block:
    # the fast sign path reads those as sgn = -1 and the listed ties are then
    # corrected.  Two ties are planted per block of Q (a Q value set to a
    # bf16-exact landmark value of its column; Q does not move the landmarks);
    # at m = 64 (16-token windows) natural ties come on both sides, in about
    # 60 % of the blocks.  Missing a correction moves that dq or dk element by
    # |g| (about 1/sqrt(m) of its size), so those elements are held to bf16
    # output rounding.
    w = _small("sparse_ties", dtype="bf16", grid_h=32, grid_w=32, m=m, d=64, iters=6)
    w = dataclasses.replace(w, B=1, H=2)
    inp = random_inputs(21, 1, 2, w.N, w.d, "bf16")
    idx = orc.pool_index(w.grid_h, w.grid_w, w.m)
    rng = np.random.default_rng(21)
    Ls = []
    for h in range(2):
        L = orc.pool_landmarks(inp["k"][0, h].astype(np.float64), idx, w.m)
        exact = (L.astype(np.float32).astype(np.float64) == L) & (round_bf16(L.astype(np.float32)) == L)
        cand = np.argwhere(exact)          # (landmark, feature) with a bf16-exact value
        assert len(cand) > 0
        for b0 in range(0, w.N, 32):
            for _ in range(2):
                a, c = cand[rng.integers(len(cand))]
                inp["q"][0, h, b0 + rng.integers(32), c] = L[a, c]
        Ls.append(L)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, m, compare(w, g, o, backward=True))
    for gi, (name, x) in enumerate((("dq", "q"), ("dk", "k"))):
        n_corr = 0
        for h in range(2):
            pos, blocks = _tie_positions(inp[x][0, h], Ls[h])
            n_corr += int(((blocks > 0) & (blocks < 16)).sum())
            full = o["grads"][(0, h)][gi]
            ref = full[pos[:, 0], pos[:, 1]]
            got = g[name][0, h][pos[:, 0], pos[:, 1]]
            rms = np.sqrt(np.mean(full ** 2))
            err = np.abs(got - ref)
            assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-3 * rms), (name, h, err.max(), rms)
        # blocks whose ties went through the correction (not the exact path)
        assert n_corr >= (32 if x == "q" else (16 if m == 64 else 0)), (name, n_corr)


@pytest.mark.parametrize("m", [16, 64, 256])
def test_out_of_range_values_take_the_exact_path(m):
    # The fast sign term (a saturated FMA with 2^64 scaling) is exact only for
    # values in {0} u [2^-40, 2^60].  Head 0: three feature columns of K scaled by
    # 2^-48, so landmarks of those columns fall below the range and every block
    # of the slice takes the exact path.  Head 1: 5 % of the Q values replaced by
    # bf16 values of size about 2^-45, so the blocks holding them take the exact
    # path while the other blocks stay on the fast one.
    w = _small("oor", dtype="bf16", grid_h=32, grid_w=32, m=m, d=64, iters=6)
    w = dataclasses.replace(w, B=1, H=2)
    inp = random_inputs(31 + m, 1, 2, w.N, w.d, "bf16")
    for c in (5, 17, 40):
        inp["k"][0, 0, :, c] = round_bf16(inp["k"][0, 0, :, c] * 2.0 ** -48)
    rng = np.random.default_rng(m)
    pick = rng.random((w.N, w.d)) < 0.05
    tiny = round_bf16(rng.standard_normal((w.N, w.d)) * 2.0 ** -45)
    inp["q"][0, 1][pick] = tiny[pick]
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, m, compare(w, g, o, backward=True))


# ---------------------------------------------------------------------------
# landmark grids beyond equal square windows: adaptive windows (the grid is not
# divisible by the landmark grid) and non-square m
# ---------------------------------------------------------------------------
GRIDS = [
    _small("adaptive_f32", grid_h=14, grid_w=14, m=16, d=32, iters=8),
    _small("adaptive_bf16_norm", dtype="bf16", grid_h=10, grid_w=12, m=9, d=64, iters=8, norm=True),
    _small("adaptive_tc", dtype="bf16", grid_h=18, grid_w=22, m=100, d=64, iters=8),
    _small("nonsquare_f32", grid_h=16, grid_w=8, m=32, d=32, iters=8),
    _small("nonsquare_bf16", dtype="bf16", grid_h=20, grid_w=12, m=15, d=64, iters=8, tied=True),
    _small("nonsquare_tc_cluster", dtype="bf16", grid_h=24, grid_w=16, m=96, d=32, iters=10),
]


@pytest.mark.parametrize("w", GRIDS, ids=lambda w: w.name)
def test_landmark_grids(w):
    inp = random_inputs(51 + w.m, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))
    np.testing.assert_array_equal(g["ctx"]["idx"], orc.pool_index(w.grid_h, w.grid_w, w.m))


def test_landmark_grid_gaussian():
    w = dataclasses.replace(GRIDS[2], name="adaptive_tc_gauss", kernel="gauss")
    inp = random_inputs(61, w.B, w.H, w.N, w.d, w.dtype)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))


# ---------------------------------------------------------------------------
# the limits of the build: m = 1024 (the largest; per-product solver for m > 256),
# iters = 64 (the largest), m > 256 with adaptive windows and a ragged landmark
# tile on the tensor-core forward
# ---------------------------------------------------------------------------
LIMITS = [
    _small("m1024", grid_h=64, grid_w=64, m=1024, d=16, iters=4),
    _small("iters64_tied_norm", m=16, d=32, iters=64, tied=True, norm=True),
    _small("m324_bf16_adaptive", dtype="bf16", grid_h=24, grid_w=24, m=324, d=64, iters=8),
]


@pytest.mark.parametrize("w", LIMITS, ids=lambda w: w.name)
def test_limits(w):
    inp = random_inputs(5, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))
    np.testing.assert_array_equal(g["ctx"]["idx"], orc.pool_index(w.grid_h, w.grid_w, w.m))


# ---------------------------------------------------------------------------
# batch-pooled feature-map statistics (LAPNYS_NORM_BATCH): mean and variance of
# each landmark column over the B * N queries of a head's B slices
# ---------------------------------------------------------------------------
BATCH_STATS = [
    _small("bstats_f32", B=3, H=2, grid_h=16, grid_w=16, m=16, d=32, iters=8, norm=True,
           norm_batch=True),
    _small("bstats_f32_tied_ragged", B=4, H=1, grid_h=10, grid_w=12, m=9, d=16, iters=6,
           norm=True, norm_batch=True, tied=True),
    _small("bstats_bf16", dtype="bf16", B=2, H=3, grid_h=14, grid_w=14, m=49, d=64, iters=10,
           norm=True, norm_batch=True),
    _small("bstats_tc", dtype="bf16", B=3, H=2, grid_h=20, grid_w=20, m=100, d=64, iters=10,
           norm=True, norm_batch=True),
    _small("bstats_tc_gauss", dtype="bf16", B=2, H=2, grid_h=16, grid_w=16, m=128, d=32, iters=10,
           norm=True, norm_batch=True, kernel="gauss"),
    _small("bstats_d128", B=2, H=2, grid_h=8, grid_w=8, m=64, d=128, iters=6, norm=True,
           norm_batch=True),
]


@pytest.mark.parametrize("w", BATCH_STATS, ids=lambda w: w.name)
def test_batch_pooled_statistics(w):
    inp = random_inputs(71 + w.m + w.B, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))
    st = g["ctx"]["stats"]
    for h in range(w.H):
        for b in range(1, w.B):   # one set of statistics per head, the same bits in every slice
            np.testing.assert_array_equal(st[b, h], st[0, h])
        mu, var, _ = o["saved"][(0, h)]["stats"]
        assert rel(st[0, h, 0], mu) < 1e-5 and rel(st[0, h, 1], var) < 1e-4


def test_batch_pooled_statistics_one_slice_per_head_is_per_slice():
    # B = 1: the pooled statistics are the slice's own, bit for bit
    w = _small("bstats_b1", B=1, H=3, grid_h=12, grid_w=12, m=16, d=64, iters=8, norm=True)
    inp = random_inputs(77, w.B, w.H, w.N, w.d, w.dtype)
    a = gpu_run(w, inp, backward=True)
    b = gpu_run(dataclasses.replace(w, norm_batch=True), inp, backward=True)
    for n in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n])


def test_batch_pooled_statistics_pvt2_full_batch():
    # the PVT stage-2 workload (B = 32, H = 2, 28 x 28 tokens, m = 49), one head's
    # 32 slices against the oracle (the statistics couple all of them)
    w = dataclasses.replace(WORKLOADS["pvt2"], norm_batch=True)
    inp = make_inputs(w, with_grad=True)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, slices={(b, 1) for b in range(w.B)}, backward=True)
    print(w.name, "norm_batch", compare(w, g, o, backward=True))


# ---------------------------------------------------------------------------
# Gaussian-kernel variant (LAPNYS_GAUSS): k(x, y) = exp(-|x - y|_2^2 / lambda)
# ---------------------------------------------------------------------------
GAUSS_NAMES = ("f32", "f32_norm", "f32_tied", "bf16", "ragged", "ragged_large_m", "m1", "iters0",
               "d128", "m81", "batch", "bf16_mN", "bf16_norm_ragged")
GAUSS_SMALL = ([dataclasses.replace(w, name="gauss_" + w.name, kernel="gauss")
                for w in SMALL if w.name in GAUSS_NAMES]
               + [dataclasses.replace(w, name="gauss_" + w.name, kernel="gauss") for w in TC_FWD])


@pytest.mark.parametrize("w", GAUSS_SMALL, ids=lambda w: w.name)
def test_gaussian_backward_small_cases(w):
    inp = random_inputs(41 + w.m + w.d, w.B, w.H, w.N, w.d, w.dtype, tied=w.tied)
    g = gpu_run(w, inp, backward=True)
    o = oracle_run(w, inp, backward=True)
    print(w.name, compare(w, g, o, backward=True))
    # bf16 with d = 32 / 64 and m > 64 forms the distances on the tensor cores with the
    # landmarks rounded to TF32 (moved by at most 2^-11 relative): kernel values to 1e-4
    tc = w.dtype == "bf16" and w.d in (32, 64) and w.m > 64
    for (b, h), s in o["saved"].items():
        c = g["ctx"]
        assert rel(c["A"][b, h], s["A"]) < 1e-6            # Gaussian landmark matrix
        Pg = c["C"] if w.tied else c["P"]                    # Q = K: C is P's transpose
        assert rel(Pg[b, h], s["P"]) < (1e-4 if tc else 1e-5)
        assert rel(c["C"][b, h], s["C"].T) < (1e-4 if tc else 1e-5)


@pytest.mark.parametrize("backward", [False, True])
def test_gaussian_hires16k(backward):
    w = dataclasses.replace(WORKLOADS["hires16k"], kernel="gauss")
    inp = make_inputs(w, with_grad=backward)
    g = gpu_run(w, inp, backward=backward)
    del inp
    o = oracle_slices(w, top_outlier_slices(w, 2) | {(0, 0), (7, 7)}, backward=backward)
    print(w.name, "gauss", compare(w, g, o, backward=backward))


def test_deterministic():
    w = WORKLOADS["pvt2"]
    inp = make_inputs(w)
    a = gpu_run(w, inp, backward=True)
    b = gpu_run(w, inp, backward=True)
    for n in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n])


def test_autograd_wrapper_matches_raw_calls():
    w = _small("autograd", d=64, m=16, iters=6, norm=True)
    inp = random_inputs(5, 2, 2, w.N, w.d, "f32")
    q = to_dev(inp["q"], "f32").requires_grad_(True)
    k = to_dev(inp["k"], "f32").requires_grad_(True)
    v = to_dev(inp["v"], "f32").requires_grad_(True)
    from laplacian_nystr_linear_gb300 import attention
    out = attention(q, k, v, (w.grid_h, w.grid_w), w.m, iters=w.iters, norm=True)
    dout = to_dev(inp["dout"], "f32")
    out.backward(dout)
    w2 = dataclasses.replace(w, B=2, H=2)
    g = gpu_run(w2, inp, backward=True)
    np.testing.assert_array_equal(out.detach().cpu().numpy(), g["out"].astype(np.float32))
    np.testing.assert_array_equal(q.grad.cpu().numpy(), g["dq"].astype(np.float32))
    np.testing.assert_array_equal(k.grad.cpu().numpy(), g["dk"].astype(np.float32))
    np.testing.assert_array_equal(v.grad.cpu().numpy(), g["dv"].astype(np.float32))


def test_launch_count_and_profile():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    p = params_of(w)
    q, k, v = (to_dev(inp[n], "f32") for n in ("q", "k", "v"))
    before = api.launch_count()
    api.profile_enable(True)
    api.fwd(q, k, v, p)
    torch.cuda.synchronize()
    prof = api.profile_read()
    api.profile_enable(False)
    launched = api.launch_count() - before
    assert launched == sum(n for n, _ in prof.values()) and launched >= 5
    assert all(ms >= 0 for _, ms in prof.values())
