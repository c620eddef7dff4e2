"""Spectrum experiments of Dion3 appendix B in float64 (oracle; test infrastructure only).

* ``spectrum_trace``: eigen-tracking of appendix B.1.1: with X_0 = U S V^T, the diagonal
  of U^T R_t U and U^T Q_t U, and the off-diagonal fraction (the "diagonalization error"
  of B.1.3).
* ``restart_sweep``: the restart-location sweep of appendix B.2.1, run on the scalar
  recurrence of Theorem 2. Every eigen-direction has a true x_0 in [0, 1]; whenever a Gram
  matrix is formed its eigenvalue is lowered by delta (4e-4 on the pages) to model the
  spurious negative eigenvalue rounding introduces. For each restart location the sweep
  records max_t cond(Q_t) (largest |q_t| over smallest |q_t| across directions),
  min_t min r_t and max_t max |q_t|.

Pins (tests/test_oracle_pins.py): the traced diagonals equal the composition of the
printed polynomials in the singular basis with a zero off-diagonal fraction in exact
arithmetic; the sweep's figures equal those of the matrix Algorithm 3 run with the same
planted eigenvalue.
"""
from __future__ import annotations

import numpy as np

from .newton_schulz import h_poly


def spectrum_trace(X0, trace):
    """Per traced step: (t, diag(U^T R U), diag(U^T Q U), offdiag fraction of U^T Q U)."""
    U, _, _ = np.linalg.svd(np.asarray(X0, dtype=np.float64), full_matrices=False)
    out = []
    for (t, R, Q) in trace:
        if not isinstance(t, int):
            continue
        dr = None if R is None else np.diag(U.T @ R @ U)
        UQU = U.T @ Q @ U
        off = UQU - np.diag(np.diag(UQU))
        out.append((t, dr, np.diag(UQU), np.linalg.norm(off) / max(np.linalg.norm(UQU), 1e-300)))
    return out


def simulate_scalar(x0, coeffs, restart_after=None, delta=4e-4):
    """Scalar Gram iteration with a planted -delta at every Gram formation.

    Returns arrays r[t], q[t] (t = 0..T, shape (T+1, len(x0))), where q[t] is the Q_t
    eigenvalue in the current Gram "epoch" (reset to 1 by a restart).
    """
    x0 = np.asarray(x0, dtype=np.float64)
    base = x0.copy()
    r = base * base - delta
    q = np.ones_like(base)
    rs, qs = [r.copy()], [q.copy()]
    for t, (a, b, c) in enumerate(coeffs, start=1):
        if restart_after is not None and t - 1 == restart_after and t > 1:
            base = q * base
            r = base * base - delta
            q = np.ones_like(base)
        z = h_poly(r, a, b, c)
        r = r * z * z
        q = q * z
        rs.append(r.copy())
        qs.append(q.copy())
    return np.array(rs), np.array(qs)


def restart_sweep(coeffs, delta=4e-4, grid=None):
    """{restart location or None: (max_t cond(Q_t), min_t min r_t, max_t max|q_t|)}."""
    if grid is None:
        grid = np.concatenate([[0.0], np.logspace(-6, 0, 2001)])
    res = {}
    T = len(coeffs)
    for loc in [None] + list(range(1, T)):
        rs, qs = simulate_scalar(grid, coeffs, loc, delta)
        aq = np.abs(qs[1:])
        cond = np.max(aq.max(axis=1) / np.maximum(aq.min(axis=1), 1e-300))
        res[loc] = (float(cond), float(rs.min()), float(aq.max()))
    return res

