"""Update flavours around the orthogonalization, in float64 (oracle; test infrastructure only).

Sources (restated, nothing copied):
  * Dion3: Full-Stack Orthogonal Updates, appendix B.2.2 "Safety Factors": every polynomial
    p_t(x) is run as p_t(x / s); s = 1.02 is the usual Polar Express setting, 1.05 the
    conservative one the page recommends.
  * Dion3 sec. 2.1 eq. (2) (NorMuon): M <- mu M + G; O = polar(M);
    v_i <- beta2 v_i + (1 - beta2) mean_j O_ij^2; O_ij <- O_ij / (sqrt(v_i) + eps);
    W <- W - eta (||O||_F / ||O_hat||_F) O_hat, with O the orthogonalized update before the
    row scaling. Algorithm 4 applies the same three steps to the selected rows of the
    fractional update (only v_i, i in S, change), then decay, update and error feedback as in
    the Muon flavour.
  * Scaling Muon for Diffusion Transformers, sec. 3.1 eq. (5) (RowNorm):
    R_eps(X)_i = X_i / max(||X_i||_2, eps) on the oriented momentum (rows = the smaller
    dimension); sec. 3.2 eq. (7) (Periodic Row-wise Muon): rho_t = [t mod K = 0]; the update
    direction is NS5 of the oriented momentum when rho_t = 1 and gamma R_eps of it otherwise;
    W <- (1 - eta lambda) W - eta s(W) O^{-1}(D); appendix C, Algorithm 1 (K = 3,
    gamma = 0.15 in sec. 4).
  * ibid. sec. 3.3 eq. (8): the column norms of a row-sharded tall matrix are the square
    roots of the sums over shards of the per-shard column sums of squares, floored at eps.

Readings where the pages leave a step open (each listed in the design notes):
  * NorMuon's denominator is sqrt(v_i) + eps: v is a second moment (a mean of squares) as
    in Adam; the extracted formula lost its square-root sign.
  * NorMuon's rows are the rows of the oriented matrix (the smaller dimension), the
    dimension Algorithm 4 selects along, so frac = 1 gives eq. (2) on the oriented rows.
  * The safety factor applies to every iteration t.
"""
from __future__ import annotations

import numpy as np

from .muon import bf16_decode, decay_rows_bf16, l1_keys_exact, momentum_update_bf16, orient, top_k_rows
from .newton_schulz import EPS, QUINTIC_FIXED, gram_ns_stabilized


def safety_adjust(coeffs, s):
    """Coefficients of p_t(x / s) for every (a_t, b_t, c_t): (a / s, b / s^3, c / s^5)."""
    s = float(s)
    return [(a / s, b / s ** 3, c / s ** 5) for (a, b, c) in coeffs]


def normuon(O, v, beta2, eps, rows=None):
    """Eq. (2) / the NorMuon steps of Algorithm 4 on O (k x m, row i of O is row rows[i] of v).

    Returns (D, v_new) with D = (||O||_F / ||O_hat||_F) O_hat the update that replaces O.
    """
    O = np.asarray(O, dtype=np.float64)
    v_new = np.array(v, dtype=np.float64, copy=True)
    idx = np.arange(O.shape[0]) if rows is None else np.asarray(rows)
    ms = np.mean(O * O, axis=1)                                  # second moments
    v_new[idx] = beta2 * v_new[idx] + (1.0 - beta2) * ms
    O_hat = O / (np.sqrt(v_new[idx]) + eps)[:, None]             # row scaling
    nh = np.linalg.norm(O_hat)
    D = O_hat * (np.linalg.norm(O) / nh) if nh > 0 else np.zeros_like(O)   # Frobenius rescale
    return D, v_new


def rownorm(X, eps):
    """R_eps(X): every row divided by max(its Euclidean norm, eps) (eq. (5))."""
    X = np.asarray(X, dtype=np.float64)
    nrm = np.sqrt(np.sum(X * X, axis=1))
    return X / np.maximum(nrm, eps)[:, None]


def refresh(t, K):
    """rho_t of eq. (7): a Newton-Schulz (refresh) step when t mod K = 0."""
    return int(t) % int(K) == 0


def normuon_step(W_bits, G_bits, M_bits, v, lr, mu, beta2, eps, weight_decay=0.0, scale=1.0,
                 coeffs=QUINTIC_FIXED, restarts=(2,), ns_eps=EPS):
    """Dense NorMuon step (eq. (2)) on the oriented matrix, mapped back.

    Returns (W_new float64, M_new bf16 bits, v_new, D oriented).
    """
    M_new = momentum_update_bf16(M_bits, G_bits, mu)
    X, tr = orient(bf16_decode(M_new))
    O = gram_ns_stabilized(X, coeffs, restarts=restarts, eps=ns_eps)
    D, v_new = normuon(O, v, beta2, eps)
    W = bf16_decode(W_bits)
    W_new = (1.0 - lr * weight_decay) * W - lr * scale * (D.T if tr else D)
    return W_new, M_new, v_new, D


def normuon_frac_step(W_bits, G_bits, M_bits, v, frac, lr, mu, beta2, eps, weight_decay=0.0, scale=1.0,
                      coeffs=QUINTIC_FIXED, restarts=(2,), ns_eps=EPS):
    """Algorithm 4 with the NorMuon steps on the selected oriented rows.

    Returns (W_new float64, M_new bf16 bits, v_new, S, D k x m).
    """
    M_bits = np.asarray(M_bits, dtype=np.uint16)
    Msum = momentum_update_bf16(M_bits, G_bits, 1.0)                 # M <- M + G
    Xb, tr = orient(Msum)
    n = Xb.shape[0]
    k = max(1, min(n, int(np.ceil(frac * n - 1e-12))))
    S = top_k_rows(l1_keys_exact(Xb), k)                             # selection
    O = gram_ns_stabilized(bf16_decode(Xb[S, :]), coeffs, restarts=restarts, eps=ns_eps)  # O = polar(M[S])
    D, v_new = normuon(O, v, beta2, eps, rows=S)                     # NorMuon steps
    W = (1.0 - lr * weight_decay) * bf16_decode(W_bits)              # weight decay
    Wo, _ = orient(W)
    Wo = Wo.copy()
    Wo[S, :] -= lr * scale * D                                       # update of the selected rows
    Xn = decay_rows_bf16(np.ascontiguousarray(Xb), S, mu)            # error feedback
    M_new = np.ascontiguousarray(Xn.T) if tr else Xn
    return (Wo.T if tr else Wo), M_new, v_new, S, D


def rownorm_step(W_bits, G_bits, M_bits, lr, mu, gamma, eps, weight_decay=0.0, scale=1.0):
    """An off-refresh step of Periodic Row-wise Muon (eq. (7), rho_t = 0).

    Returns (W_new float64, M_new bf16 bits, D = gamma R_eps of the oriented M, oriented).
    """
    M_new = momentum_update_bf16(M_bits, G_bits, mu)
    X, tr = orient(bf16_decode(M_new))
    D = gamma * rownorm(X, eps)
    W = bf16_decode(W_bits)
    W_new = (1.0 - lr * weight_decay) * W - lr * scale * (D.T if tr else D)
    return W_new, M_new, D


def column_norms_sharded(M, shards, eps):
    """Eq. (8): nu_j = max(sqrt(sum over shards of the shard's column sums of squares), eps),
    with `shards` a list of row-index arrays partitioning the rows of M."""
    M = np.asarray(M, dtype=np.float64)
    q = [np.sum(M[rows] ** 2, axis=0) for rows in shards]
    return np.maximum(np.sqrt(np.sum(q, axis=0)), eps)
