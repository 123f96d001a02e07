"""Plain, slow, fp64 CPU oracle for Laplacian-kernel Nystrom attention, and
for its Gaussian-kernel (SOFT) variant.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import this module.  It shares no code with the CUDA library and
imports nothing from it: it takes numpy arrays and returns numpy arrays.

Sources (page title, then section / equation):
  [LF-nl]  "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel",
           Dutch summary, Methodology 1 (Laplacian kernel and injectivity) and
           Methodology 2 (efficient computation: Nystrom and Newton-Schulz).
  [LF-ar]  the same paper, Arabic summary, section 2a (the Laplacian kernel
           equation), 2b (injective feature map), 2c (Nystrom, Newton-Schulz,
           diagonal perturbation).
  [SOFT]   "[Paper review] SOFT: Softmax-free Transformer with Linear
           Complexity", Proposed method: S-hat = P^T A^+ P, A_0 = alpha A,
           A_{k+1} = 2 A_k - A_k A A_k, bottleneck tokens by average pooling,
           the kernel values enter with no normalisation step; the attention there is
           a symmetric, [0, 1]-valued Gaussian kernel exp(Q (-) K).

Every step follows those passages in their order; where they are silent the
reading taken is stated next to the step.  The method is an approximation with a
truncated iteration, so this oracle runs the same T Newton-Schulz steps as the
GPU path (it does not substitute an exact inverse).  Everything is float64.

Per (b, h) slice, with Q, K, V in R^{N x d}, m landmarks and T iterations:
  L      = average-pool of K over non-overlapping windows of the token grid
  A      = k(L, L) + eps I                       k(x, y) = exp(-|x - y|_1 / lam)
  alpha  = 1 / (|A|_1 |A|_inf)
  X_0    = alpha A;  X_{t+1} = 2 X_t - X_t A X_t;  A^+ := X_T
  C      = k(L, K)  (m x N);  W = C V;  W-hat = A^+ W
  P      = k(Q, L)  (N x m);  Z = P, or Z = (P - mu) / sqrt(sigma^2 + eta)
  O      = Z W-hat
The backward pass is reverse-mode differentiation of exactly these steps.

kernel="gauss" replaces k by the Gaussian kernel of [SOFT], read (the page
prints no scale) as k(x, y) = exp(-||x - y||_2^2 / lam) with the same lam;
everything else is unchanged.  norm_batch=True takes mu and sigma^2 over the
B slices of each head instead of per slice (forward() / backward()).
block_forward() / block_backward() put the multi-head projections around the
attention: [Q | K | V] = X W_qkv + b_qkv, Y = concat_h(O_h) W_o + b_o.
"""
from __future__ import annotations

import math

import numpy as np

ETA = 1e-5  # variance floor inside the whitening square root (reading: not on the pages)


# --------------------------------------------------------------------------
# kernel  [LF-nl Methodology 1; LF-ar 2a: k(x, y) = exp(-||x - y||_1 / lambda)]
# --------------------------------------------------------------------------
def l1_distances(X: np.ndarray, Y: np.ndarray) -> np.ndarray:
    """D[i, j] = sum_c |X[i, c] - Y[j, c]|, by direct broadcasting (chunked)."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    out = np.empty((X.shape[0], Y.shape[0]))
    rows = max(1, (1 << 22) // max(1, Y.shape[0] * X.shape[1]))
    for s in range(0, X.shape[0], rows):
        out[s:s + rows] = np.abs(X[s:s + rows, None, :] - Y[None, :, :]).sum(axis=-1)
    return out


def laplacian_kernel(X: np.ndarray, Y: np.ndarray, lam: float) -> np.ndarray:
    return np.exp(-l1_distances(X, Y) / lam)


# --------------------------------------------------------------------------
# Gaussian kernel  [SOFT Proposed method: symmetric, [0, 1]-valued Gaussian
#  kernel attention; reading: k(x, y) = exp(-||x - y||_2^2 / lam)]
# --------------------------------------------------------------------------
def sq_distances(X: np.ndarray, Y: np.ndarray) -> np.ndarray:
    """D[i, j] = sum_c (X[i, c] - Y[j, c])^2, by direct broadcasting (chunked)."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    out = np.empty((X.shape[0], Y.shape[0]))
    rows = max(1, (1 << 22) // max(1, Y.shape[0] * X.shape[1]))
    for s in range(0, X.shape[0], rows):
        out[s:s + rows] = ((X[s:s + rows, None, :] - Y[None, :, :]) ** 2).sum(axis=-1)
    return out


def gaussian_kernel(X: np.ndarray, Y: np.ndarray, lam: float) -> np.ndarray:
    return np.exp(-sq_distances(X, Y) / lam)


KERNELS = ("laplace", "gauss")


def kernel_matrix(X: np.ndarray, Y: np.ndarray, lam: float, kernel: str = "laplace") -> np.ndarray:
    if kernel == "laplace":
        return laplacian_kernel(X, Y, lam)
    if kernel == "gauss":
        return gaussian_kernel(X, Y, lam)
    raise ValueError(f"unknown kernel {kernel!r}")


# --------------------------------------------------------------------------
# landmarks  [LF-ar 2c.1: the landmarks are average-pooled keys;
#             SOFT Proposed method: average pooling preferred]
# Readings: a grid of mh x mw landmarks, m = mh mw, in row-major order.  A
# square m takes mh = mw = sqrt(m); any other m the factor pair whose shape is
# closest to the token grid's (|log(mh / mw) - log(H / W)| smallest, ties to the
# smaller mh).  Window row i spans token rows [floor(i H / mh), floor((i+1) H / mh))
# and window column j token columns [floor(j W / mw), floor((j+1) W / mw)): the
# windows partition the grid, all of one size when mh | H and mw | W, otherwise
# of sizes floor and ceil of H / mh (adaptive pooling without overlap).
# --------------------------------------------------------------------------
def landmark_grid(grid_h: int, grid_w: int, m: int):
    """(mh, mw) for m landmarks on a grid_h x grid_w token grid."""
    if m < 1:
        raise ValueError("m must be positive")
    r = math.isqrt(m)
    if r * r == m:
        mh, mw = r, r
    else:
        best = None
        for a in range(1, m + 1):
            if m % a:
                continue
            key = abs(math.log(a / (m // a)) - math.log(grid_h / grid_w))
            if best is None or key < best[0] - 1e-12:
                best = (key, a, m // a)
        mh, mw = best[1], best[2]
    if mh > grid_h or mw > grid_w:
        raise ValueError("more landmark rows or columns than token rows or columns")
    return mh, mw


def pool_index(grid_h: int, grid_w: int, m: int) -> np.ndarray:
    """token n = y * grid_w + x  ->  landmark of the window containing (y, x)."""
    mh, mw = landmark_grid(grid_h, grid_w, m)
    idx = np.empty(grid_h * grid_w, dtype=np.int64)
    for i in range(mh):
        y0, y1 = (i * grid_h) // mh, ((i + 1) * grid_h) // mh
        for j in range(mw):
            x0, x1 = (j * grid_w) // mw, ((j + 1) * grid_w) // mw
            for y in range(y0, y1):
                for x in range(x0, x1):
                    idx[y * grid_w + x] = i * mw + j
    return idx


def pool_landmarks(K: np.ndarray, idx: np.ndarray, m: int) -> np.ndarray:
    K = np.asarray(K, dtype=np.float64)
    L = np.zeros((m, K.shape[1]))
    np.add.at(L, idx, K)
    return L / np.bincount(idx, minlength=m)[:, None]


# --------------------------------------------------------------------------
# landmark matrix and Newton-Schulz inverse
#  [LF-nl Methodology 2, LF-ar 2c.2: small diagonal perturbation eps I;
#   SOFT Proposed method: A_0 = alpha A, A_{k+1} = 2 A_k - A_k A A_k]
# Readings: eps only on A's diagonal; alpha = 1 / (|A|_1 |A|_inf) on A including
# eps I; "iters" = T updates after X_0, returning X_T.
# --------------------------------------------------------------------------
def landmark_matrix(L: np.ndarray, lam: float, eps: float, kernel: str = "laplace") -> np.ndarray:
    return kernel_matrix(L, L, lam, kernel) + eps * np.eye(L.shape[0])


def ns_scale(A: np.ndarray):
    """alpha and the two norms with their maximising column / row (lowest index on ties)."""
    colsum = A.sum(axis=0)
    rowsum = A.sum(axis=1)
    jstar = int(np.argmax(colsum))
    istar = int(np.argmax(rowsum))
    n1, ninf = colsum[jstar], rowsum[istar]
    return 1.0 / (n1 * ninf), n1, ninf, jstar, istar


def newton_schulz(A: np.ndarray, iters: int):
    """Return ([X_0 .. X_T], [Y_0 .. Y_{T-1}]) with Y_t = A X_t."""
    alpha = ns_scale(A)[0]
    X = [alpha * A]
    Y = []
    for _ in range(iters):
        Yt = A @ X[-1]
        Y.append(Yt)
        X.append(2.0 * X[-1] - X[-1] @ Yt)
    return X, Y


# --------------------------------------------------------------------------
# query-side feature map  [LF-nl Methodology 1: normalised injective feature
#  map; LF-ar 2b: centre and whiten each query's similarity vector with a
#  diagonal (per-feature) variance estimate instead of a full inverse square root]
# Readings: statistics per (b, h) and per landmark column over the slice's N
# queries; biased variance; eta inside the square root; gradients flow
# through mean and variance; applied to P only, never to C.
# --------------------------------------------------------------------------
def feature_map(P: np.ndarray, norm: bool, stats=None):
    """Z from P; `stats` = (mu, var) taken over a larger set of queries (the
    batch-pooled variant) instead of this slice's."""
    if not norm:
        return P, None
    if stats is None:
        mu = P.mean(axis=0)
        var = ((P - mu) ** 2).mean(axis=0)
    else:
        mu, var = stats
    s = np.sqrt(var + ETA)
    return (P - mu) / s, (mu, var, s)


# --------------------------------------------------------------------------
# forward  [SOFT Proposed method: S-hat = P^T A^+ P, read for separate Q and K as
#  O = k(Q, L) A^+ (k(L, K) V), no row normalisation]
# --------------------------------------------------------------------------
def forward_slice(q, k, v, grid_h, grid_w, m, lam, eps, iters, norm=False, kernel="laplace",
                  stats=None):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    idx = pool_index(grid_h, grid_w, m)
    L = pool_landmarks(k, idx, m)
    A = landmark_matrix(L, lam, eps, kernel)
    X, Y = newton_schulz(A, iters)
    C = kernel_matrix(L, k, lam, kernel)
    W = C @ v
    What = X[-1] @ W
    P = kernel_matrix(q, L, lam, kernel)
    Z, stats = feature_map(P, norm, stats)
    O = Z @ What
    saved = dict(q=q, k=k, v=v, idx=idx, L=L, A=A, X=X, Y=Y, C=C, W=W, What=What,
                 P=P, Z=Z, stats=stats, lam=lam, eps=eps, m=m, norm=norm, kernel=kernel)
    return O, saved


# --------------------------------------------------------------------------
# backward: reverse mode of forward_slice, step by step.
#  The Laplacian kernel's gradient is -(k/lam) sgn(x - y) per coordinate
#  [LF-nl Methodology 1 and LF-ar 2a: the L1 norm keeps a non-vanishing
#  gradient]; reading: sgn(0) = 0.
# --------------------------------------------------------------------------
def _sgn(x):
    return np.sign(x)


def _kernel_grad_x(G, X, Y, lam, kernel="laplace"):
    """For K = k(X, Y) and upstream G_ij = dLoss/dK_ij * K_ij, return dLoss/dX.

    Laplacian: dK_ij/dX_ic = -(K_ij / lam) sgn(X_ic - Y_jc).
    Gaussian:  dK_ij/dX_ic = -(2 K_ij / lam) (X_ic - Y_jc).
    """
    dX = np.zeros_like(X)
    for c in range(X.shape[1]):
        Dc = X[:, c][:, None] - Y[:, c][None, :]
        if kernel == "gauss":
            dX[:, c] = -2.0 * (G * Dc).sum(axis=1) / lam
        else:
            dX[:, c] = -(G * _sgn(Dc)).sum(axis=1) / lam
    return dX


def _kernel_grad_y(G, X, Y, lam, kernel="laplace"):
    """Same as _kernel_grad_x but with respect to the second argument Y."""
    dY = np.zeros_like(Y)
    for c in range(Y.shape[1]):
        Dc = X[:, c][:, None] - Y[:, c][None, :]
        if kernel == "gauss":
            dY[:, c] = 2.0 * (G * Dc).sum(axis=0) / lam
        else:
            dY[:, c] = (G * _sgn(Dc)).sum(axis=0) / lam
    return dY


def backward_slice(saved, dO, tied=False, dz_means=None):
    """Return (dq, dk, dv); with tied=True, dq holds the whole gradient of the shared tensor.

    dz_means = (mean dZ, mean dZ*Z) over the queries the statistics were taken
    over (the batch-pooled variant); by default this slice's."""
    dO = np.asarray(dO, dtype=np.float64)
    lam = saved["lam"]
    L, A, X, Y, C, W, What = (saved[n] for n in ("L", "A", "X", "Y", "C", "W", "What"))
    P, Z, q, k, v = saved["P"], saved["Z"], saved["q"], saved["k"], saved["v"]
    m = saved["m"]
    kern = saved.get("kernel", "laplace")

    # O = Z W-hat
    dWhat = Z.T @ dO
    dZ = dO @ What.T
    # feature map (batch-norm style reverse of centring and diagonal whitening)
    if saved["norm"]:
        _, _, s = saved["stats"]
        m0, m1 = (dZ.mean(axis=0), (dZ * Z).mean(axis=0)) if dz_means is None else dz_means
        dP = (dZ - m0 - Z * m1) / s
    else:
        dP = dZ
    # P = k(q, L)
    dq = _kernel_grad_x(dP * P, q, L, lam, kern)
    dL = _kernel_grad_y(dP * P, q, L, lam, kern)

    # W-hat = X_T W
    T = len(Y)
    G = dWhat @ W.T
    dW = X[T].T @ dWhat
    # unrolled Newton-Schulz: X_{t+1} = 2 X_t - X_t A X_t
    dA = np.zeros_like(A)
    for t in range(T - 1, -1, -1):
        XtG = X[t].T @ G
        dA -= XtG @ X[t].T
        G = 2.0 * G - G @ Y[t].T - A.T @ XtG
    # X_0 = alpha A, alpha = 1 / (n1 ninf)
    alpha, n1, ninf, jstar, istar = ns_scale(A)
    dA += alpha * G
    dalpha = float((G * A).sum())
    dA[:, jstar] += dalpha * (-alpha / n1)
    dA[istar, :] += dalpha * (-alpha / ninf)
    # A = k(L, L) + eps I: both arguments are L; the eps I term has no gradient
    Akern = A - saved["eps"] * np.eye(m)
    GA = dA * Akern
    dL += _kernel_grad_x(GA, L, L, lam, kern) + _kernel_grad_y(GA, L, L, lam, kern)

    # W = C V, C = k(L, k)
    dv = C.T @ dW
    dC = dW @ v.T
    GC = dC * C
    dL += _kernel_grad_x(GC, L, k, lam, kern)
    dk = _kernel_grad_y(GC, L, k, lam, kern)

    # L = window mean of k
    idx = saved["idx"]
    counts = np.bincount(idx, minlength=m)
    dk += dL[idx] / counts[idx][:, None]

    if tied:
        return dq + dk, None, dv
    return dq, dk, dv


# --------------------------------------------------------------------------
# batched drivers over [B, H, N, d]
# --------------------------------------------------------------------------
# Batch-pooled statistics (norm_batch), the other reading of the feature-map
#  statistics  [LF-ar 2b: the diagonal estimate normalises each feature
#  dimension on its own, taken over the batch]: mean and variance per head and
#  landmark column over the B * N queries of all B slices of that head, instead
#  of over one slice's N queries.  The backward's column means of dZ and dZ * Z
#  are then taken over the same B * N queries.
def _batch_stats(q, k, grid_h, grid_w, m, lam, kernel, h):
    """(mu, var) of P over the B * N queries of head h."""
    idx = pool_index(grid_h, grid_w, m)
    Ps = [kernel_matrix(np.asarray(q[b, h], np.float64),
                        pool_landmarks(k[b, h], idx, m), lam, kernel) for b in range(q.shape[0])]
    P = np.concatenate(Ps, axis=0)
    mu = P.mean(axis=0)
    return mu, ((P - mu) ** 2).mean(axis=0)


def forward(q, k, v, grid_h, grid_w, m, lam, eps, iters, norm=False, slices=None,
            kernel="laplace", norm_batch=False):
    """O [B, H, N, d] and the per-slice saved state (list)."""
    B, H, N, d = q.shape
    O = np.zeros((B, H, N, d))
    saved = {}
    for h in range(H):
        if slices is not None and not any((b, h) in slices for b in range(B)):
            continue
        st = _batch_stats(q, k, grid_h, grid_w, m, lam, kernel, h) if norm and norm_batch else None
        for b in range(B):
            if slices is not None and (b, h) not in slices:
                continue
            O[b, h], saved[(b, h)] = forward_slice(q[b, h], k[b, h], v[b, h], grid_h, grid_w,
                                                   m, lam, eps, iters, norm, kernel, st)
            saved[(b, h)]["norm_batch"] = bool(norm and norm_batch)
    return O, saved


def backward(saved, dO, tied=False):
    """Gradients for every slice in `saved`; returns dicts keyed by (b, h).

    With batch-pooled statistics every slice of a head must be in `saved`."""
    means = {}
    for (b, h), s in saved.items():
        if s.get("norm_batch") and h not in means:
            keys = [kk for kk in saved if kk[1] == h]
            dZ = [dO[kk[0], kk[1]] @ saved[kk]["What"].T for kk in keys]
            Zs = [saved[kk]["Z"] for kk in keys]
            dz = np.concatenate(dZ, axis=0)
            zz = np.concatenate([a * z for a, z in zip(dZ, Zs)], axis=0)
            means[h] = (dz.mean(axis=0), zz.mean(axis=0))
    out = {}
    for key, s in saved.items():
        out[key] = backward_slice(s, dO[key[0], key[1]], tied, means.get(key[1]))
    return out


def attention(q, k, v, grid_h, grid_w, m, lam, eps, iters, norm=False, kernel="laplace",
              norm_batch=False):
    return forward(q, k, v, grid_h, grid_w, m, lam, eps, iters, norm, kernel=kernel,
                   norm_batch=norm_batch)[0]


# --------------------------------------------------------------------------
# attention block: projections around the path
#  [SOFT Proposed method: the attention is instantiated as one layer of a
#   pyramid vision-transformer backbone with embedding width d_e and h heads]
# Readings: the plain multi-head layer — Q, K, V = X W + b from one weight
# w_qkv [C, S*H*d] whose column blocks are (Q | K | V), each H heads of d
# columns, head h at columns h*d .. h*d + d - 1 of its block (S = 2 with the
# (Q = K | V) blocks in tied mode); the heads' outputs concatenated in the same
# order and projected by w_o [H*d, C] plus b_o.  Biases may be None (zero).
# --------------------------------------------------------------------------
# A bf16 layer stores its activations and gradients in bf16 (reading): Q, K, V
# after the bias, the heads' outputs, the upstream gradient of the heads and
# the attention's gradients are rounded once to bf16, everything else is exact.
# store="f64" keeps every value exact (the float32 layer, whose rounding is at
# the level of fp32 arithmetic).
def round_bf16(x):
    """Each value rounded to the nearest bf16 number (8 significant bits, the
    float32 exponent range), ties to the even significand; from the definition:
    scale by the power of two that puts the last kept bit at 1, round half to
    even (numpy's rint), scale back.  Zeros, infinities and NaNs pass through."""
    x = np.asarray(x, np.float64)
    out = x.copy()
    nz = np.isfinite(x) & (x != 0)
    e = np.floor(np.log2(np.abs(x[nz])))
    e = np.maximum(e, -126.0)                # subnormal bf16 numbers share 2^-126's spacing
    q = np.ldexp(1.0, (e - 7).astype(np.int64))   # spacing of bf16 numbers at |x|
    out[nz] = np.rint(x[nz] / q) * q
    return out


def _store(a, store):
    return round_bf16(a) if store == "bf16" else a


def _heads(Y, B, N, H, d):
    """[B, N, H*d] -> [B, H, N, d]"""
    return Y.reshape(B, N, H, d).transpose(0, 2, 1, 3)


def _unheads(Y):
    """[B, H, N, d] -> [B, N, H*d]"""
    B, H, N, d = Y.shape
    return Y.transpose(0, 2, 1, 3).reshape(B, N, H * d)


def block_forward(x, w_qkv, b_qkv, w_o, b_o, H, d, grid_h, grid_w, m, lam, eps, iters,
                  norm=False, kernel="laplace", norm_batch=False, tied=False, store="f64"):
    """y [B, N, C] and the saved state of the block; store="bf16" rounds the
    stored activations as a bf16 layer does (see round_bf16)."""
    if store not in ("f64", "bf16"):
        raise ValueError(f"unknown store {store!r}")
    x = np.asarray(x, np.float64)
    B, N, C = x.shape
    S = 2 if tied else 3
    w_qkv = np.asarray(w_qkv, np.float64)
    assert w_qkv.shape == (C, S * H * d)
    qkv = _store(x @ w_qkv + (0.0 if b_qkv is None else np.asarray(b_qkv, np.float64)), store)
    blocks = [_heads(qkv[..., s * H * d:(s + 1) * H * d], B, N, H, d) for s in range(S)]
    q, v = blocks[0], blocks[-1]
    k = q if tied else blocks[1]
    O, saved = forward(q, k, v, grid_h, grid_w, m, lam, eps, iters, norm, kernel=kernel,
                       norm_batch=norm_batch)
    Ot = _store(_unheads(O), store)
    y = Ot @ np.asarray(w_o, np.float64) + (0.0 if b_o is None else np.asarray(b_o, np.float64))
    st = dict(x=x, w_qkv=w_qkv, w_o=np.asarray(w_o, np.float64), Ot=Ot, attn=saved, H=H, d=d,
              tied=tied, qkv=qkv, store=store)
    return y, st


def block_backward(st, dy):
    """(dx, dw_qkv, db_qkv, dw_o, db_o) for the block."""
    dy = np.asarray(dy, np.float64)
    B, N, C = dy.shape
    H, d = st["H"], st["d"]
    dw_o = np.einsum("bnk,bnc->kc", st["Ot"], dy)
    db_o = dy.sum(axis=(0, 1))
    store = st.get("store", "f64")
    dO = _store(_heads(dy @ st["w_o"].T, B, N, H, d), store)
    g = backward(st["attn"], dO, tied=st["tied"])
    grad = {n: _store(np.stack([np.stack([g[(b, h)][i] for h in range(H)]) for b in range(B)]),
                      store)
            for i, n in enumerate(("q", "k", "v")) if n != "k" or not st["tied"]}
    parts = [grad["q"], grad["v"]] if st["tied"] else [grad["q"], grad["k"], grad["v"]]
    dqkv = np.concatenate([_unheads(t) for t in parts], axis=-1)
    dw_qkv = np.einsum("bnc,bnk->ck", st["x"], dqkv)
    db_qkv = dqkv.sum(axis=(0, 1))
    dx = dqkv @ st["w_qkv"].T
    return dx, dw_qkv, db_qkv, dw_o, db_o
