"""Pins for the CPU oracle: checks against facts the pages and mathematics fix,
not against the oracle's own formulas.

- Laplacian kernel values by pure-Python loops; range (0, 1], k(x, x) = 1,
  symmetry  (LaplacianFormer, Methodology 1 / Arabic summary 2a; SOFT review,
  Proposed method: the kernel is symmetric with values in [0, 1]).
- Average-pooling windows enumerated by coordinates (LaplacianFormer Arabic
  summary 2c.1; SOFT review, Proposed method: average pooling); adaptive
  windows (the reading for grids the landmark grid does not divide, and for
  non-square m) checked as a partition of the grid, by a worked example and by
  finite differences through the pooling.
- eps I makes A strictly positive definite (LaplacianFormer Methodology 2).
- Truncated Newton-Schulz against its closed form through a library eigensolver;
  the residual |I - A X_t| falls monotonically (SOFT review, Proposed method).
- With one landmark per token, eps = 0 and a converged iteration, Nystrom gives
  exact full-kernel attention S V, brute-forced.
- lambda -> infinity closed form; centring/whitening invariants.
- Backward against central finite differences of the forward.
- The Gaussian-kernel variant (SOFT review, Proposed method: a symmetric,
  [0, 1]-valued Gaussian kernel; read as exp(-|x - y|_2^2 / lambda)): kernel
  values by loops and by the factorisation exp(-|x|^2/l) exp(-|y|^2/l)
  exp(2 x.y / l); positive definiteness; exact full-kernel attention with one
  landmark per token; lambda -> infinity; finite differences; dV = M^T dO.
"""
import math

import numpy as np
import pytest

from oracle import lapnys_oracle as orc


def _loop_kernel(X, Y, lam):
    out = [[0.0] * len(Y) for _ in range(len(X))]
    for i, x in enumerate(X):
        for j, y in enumerate(Y):
            s = 0.0
            for c in range(len(x)):
                s += abs(float(x[c]) - float(y[c]))
            out[i][j] = math.exp(-s / lam)
    return np.array(out)


def test_kernel_matches_loops_and_range():
    rng = np.random.default_rng(0)
    X = rng.standard_normal((7, 5))
    Y = rng.standard_normal((6, 5)) * 3.0
    lam = 2.5
    Kx = orc.laplacian_kernel(X, Y, lam)
    np.testing.assert_allclose(Kx, _loop_kernel(X, Y, lam), rtol=1e-14, atol=0)
    assert np.all(Kx > 0) and np.all(Kx <= 1)
    Kxx = orc.laplacian_kernel(X, X, lam)
    np.testing.assert_array_equal(np.diag(Kxx), 1.0)
    np.testing.assert_array_equal(Kxx, Kxx.T)
    # heavy-tailed values still land in (0, 1]
    Xt = rng.standard_t(3, size=(9, 64)) * 50
    Kt = orc.laplacian_kernel(Xt, Xt[::-1], 64.0)
    assert np.all(Kt >= 0) and np.all(Kt <= 1)


@pytest.mark.parametrize("gh,gw,m", [(14, 14, 49), (8, 12, 4), (6, 6, 36), (28, 28, 49), (4, 4, 1)])
def test_pool_windows_by_enumeration(gh, gw, m):
    idx = orc.pool_index(gh, gw, m)
    r = math.isqrt(m)
    sh, sw = gh // r, gw // r
    expect = -np.ones(gh * gw, dtype=np.int64)
    for i in range(r):
        for j in range(r):
            for y in range(i * sh, (i + 1) * sh):
                for x in range(j * sw, (j + 1) * sw):
                    expect[y * gw + x] = i * r + j
    np.testing.assert_array_equal(idx, expect)
    # landmark values by a reshape-mean over (window row, in-window row, window col, in-window col)
    rng = np.random.default_rng(1)
    K = rng.standard_normal((gh * gw, 3))
    L = orc.pool_landmarks(K, idx, m)
    L2 = K.reshape(r, sh, r, sw, 3).mean(axis=(1, 3)).reshape(m, 3)
    np.testing.assert_allclose(L, L2, rtol=1e-13, atol=1e-15)


def test_pool_rejects_bad_geometry():
    # more landmark rows or columns than the grid has, or no landmarks
    for args in [(4, 4, 25), (2, 8, 9), (4, 4, 7), (4, 4, 0)]:
        with pytest.raises(ValueError):
            orc.pool_index(*args)


def test_landmark_grid_shapes():
    # square m keeps a square landmark grid; other m take the factor pair shaped like the grid
    assert orc.landmark_grid(14, 14, 49) == (7, 7)
    assert orc.landmark_grid(14, 14, 16) == (4, 4)       # not dividing 14: adaptive windows
    assert orc.landmark_grid(128, 64, 128) == (16, 8)
    assert orc.landmark_grid(20, 10, 50) == (10, 5)
    assert orc.landmark_grid(8, 16, 32) == (4, 8)
    assert orc.landmark_grid(14, 14, 48) == (6, 8)       # shapes 6 x 8 and 8 x 6 tie: smaller mh


@pytest.mark.parametrize("gh,gw,m", [(14, 14, 16), (10, 12, 9), (7, 9, 6), (5, 5, 4), (20, 10, 50)])
def test_adaptive_windows_partition_the_grid(gh, gw, m):
    idx = orc.pool_index(gh, gw, m)
    mh, mw = orc.landmark_grid(gh, gw, m)
    assert idx.min() == 0 and idx.max() == m - 1
    grid = idx.reshape(gh, gw)
    rows, cols = grid // mw, grid % mw
    # each window row is one band of consecutive token rows, each window column one band of columns
    for y in range(gh):
        assert len(set(rows[y])) == 1
    for x in range(gw):
        assert len(set(cols[:, x])) == 1
    rsize = np.bincount(rows[:, 0], minlength=mh)
    csize = np.bincount(cols[0], minlength=mw)
    assert set(rsize) <= {gh // mh, -(-gh // mh)} and rsize.sum() == gh
    assert set(csize) <= {gw // mw, -(-gw // mw)} and csize.sum() == gw
    assert np.all(np.diff(rows[:, 0]) >= 0) and np.all(np.diff(cols[0]) >= 0)


def test_adaptive_windows_worked_example():
    # 14 token rows into 4 window rows: starts floor(i * 14 / 4) = 0, 3, 7, 10 (sizes 3, 4, 3, 4)
    idx = orc.pool_index(14, 14, 16).reshape(14, 14)
    np.testing.assert_array_equal(idx[:, 0] // 4, [0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 3, 3, 3, 3])
    np.testing.assert_array_equal(idx[0] % 4, [0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 3, 3, 3, 3])
    # window means by loops
    rng = np.random.default_rng(9)
    K = rng.standard_normal((196, 2))
    L = orc.pool_landmarks(K, idx.reshape(-1), 16)
    for a in range(16):
        members = [n for n in range(196) if idx.reshape(-1)[n] == a]
        np.testing.assert_allclose(L[a], K[members].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_backward_through_adaptive_pooling_matches_finite_differences():
    rng = np.random.default_rng(40)
    gh, gw, m, d, T, lam, eps = 5, 5, 4, 3, 3, 3.0, 1e-3
    N = gh * gw
    q, k, v, R = (rng.standard_normal((N, d)) for _ in range(4))

    def loss(k_):
        O, _ = orc.forward_slice(q, k_, v, gh, gw, m, lam, eps, T)
        return float((O * R).sum())

    _, saved = orc.forward_slice(q, k, v, gh, gw, m, lam, eps, T)
    _, dk, _ = orc.backward_slice(saved, R)
    h = 1e-6
    fd = np.zeros_like(k)
    for i in range(N):
        for c in range(d):
            kp, km = k.copy(), k.copy()
            kp[i, c] += h
            km[i, c] -= h
            fd[i, c] = (loss(kp) - loss(km)) / (2 * h)
    assert np.linalg.norm(dk - fd) / np.linalg.norm(fd) < 1e-6


def test_one_landmark_per_token_is_identity():
    rng = np.random.default_rng(2)
    K = rng.standard_normal((16, 4))
    idx = orc.pool_index(4, 4, 16)
    np.testing.assert_array_equal(orc.pool_landmarks(K, idx, 16), K)


def test_landmark_matrix_is_spd_with_eps_diagonal():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((49, 32))
    A = orc.landmark_matrix(L, 32.0, 1e-3)
    np.testing.assert_allclose(np.diag(A), 1.0 + 1e-3, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(A, A.T)
    assert np.linalg.eigvalsh(A).min() > 0


@pytest.mark.parametrize("m,d,T", [(49, 32, 20), (64, 64, 20), (16, 4, 3), (36, 8, 0)])
def test_newton_schulz_closed_form(m, d, T):
    rng = np.random.default_rng(4 + m)
    L = rng.standard_normal((m, d))
    A = orc.landmark_matrix(L, float(d), 1e-3)
    X, Y = orc.newton_schulz(A, T)
    assert len(X) == T + 1 and len(Y) == T
    sig, U = np.linalg.eigh(A)
    alpha = 1.0 / (np.abs(A).sum(axis=0).max() * np.abs(A).sum(axis=1).max())
    assert alpha * sig.max() ** 2 <= 1.0 + 1e-12
    # X_t has eigenvalues (1 - (1 - alpha s^2)^(2^t)) / s for eigenvalue s of A
    prev = np.inf
    for t in range(T + 1):
        e = (1.0 - alpha * sig ** 2) ** (2.0 ** t)
        Xt = (U * ((1.0 - e) / sig)) @ U.T
        np.testing.assert_allclose(X[t], Xt, rtol=0, atol=1e-10 * np.abs(Xt).max())
        res = np.linalg.norm(np.eye(m) - A @ X[t])
        np.testing.assert_allclose(res, np.sqrt((e ** 2).sum()), rtol=1e-6, atol=1e-12)
        assert res <= prev + 1e-12
        prev = res


def _brute_full_attention(q, k, v, lam):
    S = _loop_kernel(q, k, lam)
    return S @ v, S


def test_one_landmark_per_token_equals_full_kernel_attention():
    rng = np.random.default_rng(5)
    N, d = 16, 4
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    lam = float(d)
    O, _ = orc.forward_slice(q, k, v, 4, 4, N, lam, 0.0, 40)
    Oref, S = _brute_full_attention(q, k, v, lam)
    np.testing.assert_allclose(O, Oref, rtol=1e-9, atol=1e-9)
    # eps > 0 with a converged iteration gives S (G + eps I)^-1 G V, G = k(K, K)
    eps = 1e-3
    O2, _ = orc.forward_slice(q, k, v, 4, 4, N, lam, eps, 40)
    G = _loop_kernel(k, k, lam)
    O2ref = S @ np.linalg.solve(G + eps * np.eye(N), G @ v)
    np.testing.assert_allclose(O2, O2ref, rtol=1e-9, atol=1e-9)


def test_large_lambda_closed_form():
    # kernel == 1 everywhere: A = J + eps I, X_T 1 = 1 / (m + eps), O_i = m / (m + eps) sum_j V_j
    rng = np.random.default_rng(6)
    N, d, m, eps = 36, 8, 9, 1e-3
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    O, _ = orc.forward_slice(q, k, v, 6, 6, m, 1e300, eps, 5)
    expect = np.broadcast_to(m / (m + eps) * v.sum(axis=0), (N, d))
    np.testing.assert_allclose(O, expect, rtol=1e-10, atol=1e-10)


def test_feature_map_invariants():
    rng = np.random.default_rng(7)
    N, d, m = 64, 8, 16
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    _, s = orc.forward_slice(q, k, v, 8, 8, m, float(d), 1e-3, 5, norm=True)
    Z, P = s["Z"], s["P"]
    np.testing.assert_allclose(Z.mean(axis=0), 0.0, atol=1e-12)
    var = P.var(axis=0)
    np.testing.assert_allclose(Z.var(axis=0), var / (var + orc.ETA), rtol=1e-10)


def _fd_check(tied, norm, seed, kernel="laplace"):
    rng = np.random.default_rng(seed)
    gh = gw = 4
    N, d, m, T, lam, eps = 16, 4, 4, 3, 4.0, 1e-3
    q = rng.standard_normal((N, d))
    k = q.copy() if tied else rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    R = rng.standard_normal((N, d))

    def loss(q_, k_, v_):
        O, _ = orc.forward_slice(q_, q_ if tied else k_, v_, gh, gw, m, lam, eps, T, norm,
                                 kernel)
        return float((O * R).sum())

    _, saved = orc.forward_slice(q, k, v, gh, gw, m, lam, eps, T, norm, kernel)
    dq, dk, dv = orc.backward_slice(saved, R, tied=tied)
    h = 1e-6
    names = ("q", "v") if tied else ("q", "k", "v")
    grads = {"q": dq, "k": dk, "v": dv}
    for name in names:
        base = {"q": q, "k": k, "v": v}
        fd = np.zeros((N, d))
        for i in range(N):
            for c in range(d):
                plus = {n: a.copy() for n, a in base.items()}
                minus = {n: a.copy() for n, a in base.items()}
                plus[name][i, c] += h
                minus[name][i, c] -= h
                fd[i, c] = (loss(plus["q"], plus["k"], plus["v"])
                            - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        g = grads[name]
        err = np.linalg.norm(g - fd) / np.linalg.norm(fd)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("tied,norm", [(False, False), (False, True), (True, False), (True, True)])
def test_backward_matches_finite_differences(tied, norm):
    _fd_check(tied, norm, seed=10 + 2 * tied + norm)


def test_dv_is_linear_map_transpose():
    # O = M V with M = Z A^+ C, so dV = M^T dO
    rng = np.random.default_rng(11)
    N, d, m = 36, 4, 9
    q, k, v, dO = (rng.standard_normal((N, d)) for _ in range(4))
    O, s = orc.forward_slice(q, k, v, 6, 6, m, float(d), 1e-3, 6, norm=True)
    M = s["Z"] @ s["X"][-1] @ s["C"]
    np.testing.assert_allclose(O, M @ v, rtol=1e-12, atol=1e-12)
    _, _, dv = orc.backward_slice(s, dO)
    np.testing.assert_allclose(dv, M.T @ dO, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Gaussian-kernel variant
# --------------------------------------------------------------------------
def _loop_gauss(X, Y, lam):
    out = [[0.0] * len(Y) for _ in range(len(X))]
    for i, x in enumerate(X):
        for j, y in enumerate(Y):
            s = 0.0
            for c in range(len(x)):
                t = float(x[c]) - float(y[c])
                s += t * t
            out[i][j] = math.exp(-s / lam)
    return np.array(out)


def test_gaussian_kernel_by_loops_factorisation_and_range():
    rng = np.random.default_rng(20)
    X = rng.standard_normal((7, 5))
    Y = rng.standard_normal((6, 5)) * 1.5
    lam = 3.5
    Kx = orc.gaussian_kernel(X, Y, lam)
    np.testing.assert_allclose(Kx, _loop_gauss(X, Y, lam), rtol=1e-13, atol=0)
    # |x - y|^2 = |x|^2 + |y|^2 - 2 x.y
    fac = (np.exp(-(X ** 2).sum(1) / lam)[:, None] * np.exp(-(Y ** 2).sum(1) / lam)[None, :]
           * np.exp(2.0 * (X @ Y.T) / lam))
    np.testing.assert_allclose(Kx, fac, rtol=1e-12, atol=0)
    assert np.all(Kx > 0) and np.all(Kx <= 1)
    Kxx = orc.kernel_matrix(X, X, lam, "gauss")
    np.testing.assert_array_equal(np.diag(Kxx), 1.0)
    np.testing.assert_array_equal(Kxx, Kxx.T)


def test_gaussian_landmark_matrix_is_spd():
    rng = np.random.default_rng(21)
    L = rng.standard_normal((49, 8))
    G = orc.kernel_matrix(L, L, 8.0, "gauss")
    assert np.linalg.eigvalsh(G).min() > -1e-12   # a Gaussian gram matrix is positive semidefinite
    A = orc.landmark_matrix(L, 8.0, 1e-3, "gauss")
    np.testing.assert_allclose(np.diag(A), 1.0 + 1e-3, rtol=0, atol=1e-15)
    assert np.linalg.eigvalsh(A).min() >= 1e-3 - 1e-12


def test_gaussian_one_landmark_per_token_equals_full_kernel_attention():
    rng = np.random.default_rng(22)
    N, d = 16, 4
    q, k, v = (rng.standard_normal((N, d)) * 0.5 for _ in range(3))
    lam = 2.0 * math.sqrt(d)
    O, _ = orc.forward_slice(q, k, v, 4, 4, N, lam, 1e-3, 60, kernel="gauss")
    S = _loop_gauss(q, k, lam)
    G = _loop_gauss(k, k, lam)
    Oref = S @ np.linalg.solve(G + 1e-3 * np.eye(N), G @ v)
    np.testing.assert_allclose(O, Oref, rtol=1e-8, atol=1e-8)


def test_gaussian_large_lambda_closed_form():
    rng = np.random.default_rng(23)
    N, d, m, eps = 36, 8, 9, 1e-3
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    O, _ = orc.forward_slice(q, k, v, 6, 6, m, 1e300, eps, 5, kernel="gauss")
    expect = np.broadcast_to(m / (m + eps) * v.sum(axis=0), (N, d))
    np.testing.assert_allclose(O, expect, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("tied,norm", [(False, False), (False, True), (True, False)])
def test_gaussian_backward_matches_finite_differences(tied, norm):
    _fd_check(tied, norm, seed=30 + 2 * tied + norm, kernel="gauss")


def test_gaussian_dv_is_linear_map_transpose():
    rng = np.random.default_rng(24)
    N, d, m = 36, 4, 9
    q, k, v, dO = (rng.standard_normal((N, d)) for _ in range(4))
    O, s = orc.forward_slice(q, k, v, 6, 6, m, float(d), 1e-3, 6, norm=True, kernel="gauss")
    M = s["Z"] @ s["X"][-1] @ s["C"]
    np.testing.assert_allclose(O, M @ v, rtol=1e-12, atol=1e-12)
    _, _, dv = orc.backward_slice(s, dO)
    np.testing.assert_allclose(dv, M.T @ dO, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# batch-pooled feature-map statistics
# --------------------------------------------------------------------------
def _batch(seed, B, H, N, d, tied=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d))
    k = q.copy() if tied else rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    return q, k, v


def test_batch_stats_invariants():
    # pooled over the B slices of a head: zero column means and the whitened
    # variance over all B * N queries, but not within one slice
    B, H, N, d, m = 3, 2, 64, 8, 16
    q, k, v = _batch(31, B, H, N, d)
    _, saved = orc.forward(q, k, v, 8, 8, m, float(d), 1e-3, 5, norm=True, norm_batch=True)
    for h in range(H):
        Z = np.concatenate([saved[(b, h)]["Z"] for b in range(B)], axis=0)
        P = np.concatenate([saved[(b, h)]["P"] for b in range(B)], axis=0)
        np.testing.assert_allclose(Z.mean(axis=0), 0.0, atol=1e-12)
        var = P.var(axis=0)
        np.testing.assert_allclose(Z.var(axis=0), var / (var + orc.ETA), rtol=1e-10)
        assert np.abs(saved[(0, h)]["Z"].mean(axis=0)).max() > 1e-3


def test_batch_stats_reduce_to_per_slice():
    # one slice per head, or every slice of a head the same: the pooled
    # statistics are the slice's own
    q, k, v = _batch(32, 1, 2, 36, 4)
    a = orc.attention(q, k, v, 6, 6, 9, 4.0, 1e-3, 6, norm=True)
    b = orc.attention(q, k, v, 6, 6, 9, 4.0, 1e-3, 6, norm=True, norm_batch=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    q2, k2, v2 = (np.concatenate([t, t, t], axis=0) for t in (q, k, v))
    c = orc.attention(q2, k2, v2, 6, 6, 9, 4.0, 1e-3, 6, norm=True, norm_batch=True)
    for bb in range(3):
        np.testing.assert_allclose(c[bb], a[0], rtol=1e-10, atol=1e-12)
    # without norm the flag changes nothing
    np.testing.assert_array_equal(orc.attention(q2, k2, v2, 6, 6, 9, 4.0, 1e-3, 6),
                                  orc.attention(q2, k2, v2, 6, 6, 9, 4.0, 1e-3, 6,
                                                norm_batch=True))


@pytest.mark.parametrize("tied,kernel", [(False, "laplace"), (True, "laplace"),
                                         (False, "gauss")])
def test_batch_stats_backward_matches_finite_differences(tied, kernel):
    # the statistics couple the B slices of a head (not the heads): the loss
    # is summed over every slice, and every input entry is perturbed
    B, H, N, d, m, T, lam, eps = 2, 2, 16, 4, 4, 3, 4.0, 1e-3
    q, k, v = _batch(33 + tied, B, H, N, d, tied)
    R = np.random.default_rng(40).standard_normal((B, H, N, d))

    def loss(q_, k_, v_):
        O = orc.attention(q_, q_ if tied else k_, v_, 4, 4, m, lam, eps, T, True, kernel, True)
        return float((O * R).sum())

    _, saved = orc.forward(q, k, v, 4, 4, m, lam, eps, T, True, kernel=kernel, norm_batch=True)
    g = orc.backward(saved, R, tied=tied)
    grads = {n: np.stack([np.stack([g[(b, hh)][i] for hh in range(H)]) for b in range(B)])
             for i, n in enumerate(("q", "k", "v"))}
    h = 1e-6
    for name in (("q", "v") if tied else ("q", "k", "v")):
        base = {"q": q, "k": k, "v": v}
        fd = np.zeros(q.shape)
        for ix in np.ndindex(q.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[name][ix] += h
            minus[name][ix] -= h
            fd[ix] = (loss(plus["q"], plus["k"], plus["v"])
                      - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(grads[name] - fd) / np.linalg.norm(fd)
        assert err < 1e-6, (name, err)


# --------------------------------------------------------------------------
# attention block (projections around the path)
# --------------------------------------------------------------------------
def _block_args(seed, B=2, N=16, C=6, H=2, d=4, tied=False, bias=True):
    rng = np.random.default_rng(seed)
    S = 2 if tied else 3
    x = rng.standard_normal((B, N, C))
    w = rng.standard_normal((C, S * H * d)) / np.sqrt(C)
    b = rng.standard_normal(S * H * d) * 0.3 if bias else None
    wo = rng.standard_normal((H * d, C)) / np.sqrt(H * d)
    bo = rng.standard_normal(C) * 0.3 if bias else None
    return x, w, b, wo, bo


BLK = dict(grid_h=4, grid_w=4, m=4, lam=4.0, eps=1e-3, iters=3)


def _blk(x, w, b, wo, bo, H, d, **kw):
    a = dict(BLK)
    a.update(kw)
    return orc.block_forward(x, w, b, wo, bo, H, d, a["grid_h"], a["grid_w"], a["m"], a["lam"],
                             a["eps"], a["iters"], a.get("norm", False), a.get("kernel", "laplace"),
                             a.get("norm_batch", False), a.get("tied", False))


def test_block_one_head_is_projected_attention():
    x, w, b, wo, bo = _block_args(50, H=1, d=4)
    y, _ = _blk(x, w, b, wo, bo, 1, 4, norm=True)
    q, k, v = (x @ w[:, 4 * s:4 * s + 4] + b[4 * s:4 * s + 4] for s in range(3))
    O = orc.attention(q[:, None], k[:, None], v[:, None], 4, 4, 4, 4.0, 1e-3, 3, norm=True)
    np.testing.assert_allclose(y, O[:, 0] @ wo + bo, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tied", [False, True])
def test_block_head_permutation_invariance(tied):
    # relabelling the heads (their column blocks in every projection, their row
    # blocks in w_o) leaves the layer unchanged
    H, d = 3, 4
    x, w, b, wo, bo = _block_args(51, C=5, H=H, d=d, tied=tied)
    perm = [2, 0, 1]
    S = 2 if tied else 3
    cols = np.concatenate([s * H * d + np.arange(h * d, h * d + d) for s in range(S) for h in perm])
    rows = np.concatenate([np.arange(h * d, h * d + d) for h in perm])
    y0, _ = _blk(x, w, b, wo, bo, H, d, tied=tied)
    y1, _ = _blk(x, w[:, cols], b[cols], wo[rows], bo, H, d, tied=tied)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-12)
    # swapping two coordinates inside a head of Q: with Q = K every distance
    # |q - l|_1 keeps its value (both sides move together); with a separate K
    # the layer changes
    wq = w.copy()
    wq[:, [0, 1]] = wq[:, [1, 0]]
    bq = b.copy()
    bq[[0, 1]] = bq[[1, 0]]
    y2, _ = _blk(x, wq, bq, wo, bo, H, d, tied=tied)
    if tied:
        np.testing.assert_allclose(y2, y0, rtol=1e-12, atol=1e-12)
    else:
        assert np.abs(y2 - y0).max() > 1e-6


def test_block_bias_is_a_constant_input_feature():
    # a bias equals one more input feature fixed at 1 whose weight row is the bias
    x, w, b, wo, bo = _block_args(52)
    y0, st0 = _blk(x, w, b, wo, bo, 2, 4, norm=True)
    xa = np.concatenate([x, np.ones(x.shape[:2] + (1,))], axis=-1)
    y1, st1 = _blk(xa, np.vstack([w, b]), None, wo, bo, 2, 4, norm=True)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-12)
    dy = np.random.default_rng(53).standard_normal(y0.shape)
    g0 = orc.block_backward(st0, dy)
    g1 = orc.block_backward(st1, dy)
    np.testing.assert_allclose(g1[1][-1], g0[2], rtol=1e-10, atol=1e-12)   # db_qkv
    np.testing.assert_allclose(g1[1][:-1], g0[1], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g1[0][..., :-1], g0[0], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("tied,norm,norm_batch,kernel", [(False, True, False, "laplace"),
                                                         (True, True, False, "laplace"),
                                                         (False, True, True, "laplace"),
                                                         (False, False, False, "gauss")])
def test_block_backward_matches_finite_differences(tied, norm, norm_batch, kernel):
    H, d = 2, 4
    x, w, b, wo, bo = _block_args(54 + tied + 2 * norm_batch, tied=tied)
    R = np.random.default_rng(57).standard_normal(x.shape)
    kw = dict(tied=tied, norm=norm, norm_batch=norm_batch, kernel=kernel)
    args = dict(x=x, w=w, b=b, wo=wo, bo=bo)

    def loss(a):
        y, _ = _blk(a["x"], a["w"], a["b"], a["wo"], a["bo"], H, d, **kw)
        return float((y * R).sum())

    _, st = _blk(x, w, b, wo, bo, H, d, **kw)
    dx, dw, db, dwo, dbo = orc.block_backward(st, R)
    grads = dict(x=dx, w=dw, b=db, wo=dwo, bo=dbo)
    h = 1e-6
    for name, base in args.items():
        fd = np.zeros(base.shape)
        for ix in np.ndindex(base.shape):
            plus = {n: a.copy() for n, a in args.items()}
            minus = {n: a.copy() for n, a in args.items()}
            plus[name][ix] += h
            minus[name][ix] -= h
            fd[ix] = (loss(plus) - loss(minus)) / (2 * h)
        err = np.linalg.norm(grads[name] - fd) / np.linalg.norm(fd)
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------------------
# bf16 storage of the attention block (reading: a bf16 layer rounds Q, K, V,
# the heads' outputs and the gradients once to bf16)
# ---------------------------------------------------------------------------
def test_round_bf16_follows_the_definition():
    # worked cases: 8 significant bits, ties to the even significand
    cases = {1.0: 1.0, 1.0 + 2 ** -8: 1.0, 1.0 + 3 * 2 ** -8: 1.0 + 2 ** -6,
             1.0 + 2 ** -7: 1.0 + 2 ** -7, 1.0 + 2 ** -8 + 2 ** -30: 1.0 + 2 ** -7,
             -3.0 - 2 ** -7: -3.0, 255.5: 256.0, 0.0: 0.0, 2.0 ** -130: 2.0 ** -130,
             3 * 2.0 ** -134: 4 * 2.0 ** -134}
    got = orc.round_bf16(np.array(list(cases)))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))
    # against the seeded inputs' independent bit-level rounding of float32 values
    from laplacian_nystr_linear_gb300.inputs import round_bf16 as round_bits
    x = np.random.default_rng(3).standard_normal(20000).astype(np.float32) * 7.0
    np.testing.assert_array_equal(orc.round_bf16(x.astype(np.float64)),
                                  round_bits(x).astype(np.float64))
    # idempotent, and every result is a bf16 value (16 low bits of its float32 zero)
    r = orc.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(orc.round_bf16(r), r)
    assert not (r.astype(np.float32).view(np.uint32) & 0xFFFF).any()


def test_block_bf16_storage_rounds_only_the_stored_values():
    a = dict(B=1, N=16, C=8, H=2, d=4, grid_h=4, grid_w=4, m=4, lam=4.0, eps=1e-3, iters=3)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((a["B"], a["N"], a["C"]))
    w = rng.standard_normal((a["C"], 3 * a["H"] * a["d"])) / 3
    wo = rng.standard_normal((a["H"] * a["d"], a["C"])) / 3
    dy = rng.standard_normal((a["B"], a["N"], a["C"]))

    def run(store):
        y, st = orc.block_forward(x, w, None, wo, None, a["H"], a["d"], a["grid_h"], a["grid_w"],
                                  a["m"], a["lam"], a["eps"], a["iters"], store=store)
        return y, st, orc.block_backward(st, dy)

    y0, st0, g0 = run("f64")
    y1, st1, g1 = run("bf16")
    # the stored Q, K, V and heads' outputs are the f64 layer's values rounded
    np.testing.assert_array_equal(st1["qkv"], orc.round_bf16(st0["qkv"]))
    assert not (st1["Ot"].astype(np.float32).view(np.uint32) & 0xFFFF).any()
    # and the results move by about bf16 rounding, not more
    assert 0 < np.linalg.norm(y1 - y0) / np.linalg.norm(y0) < 2e-2
    for a0, a1 in zip(g0, g1):
        assert np.linalg.norm(a1 - a0) / np.linalg.norm(a0) < 5e-2
    with pytest.raises(ValueError):
        orc.block_forward(x, w, None, wo, None, a["H"], a["d"], a["grid_h"], a["grid_w"], a["m"],
                          a["lam"], a["eps"], a["iters"], store="f16")
