"""Newton-Schulz iterations in float64 (oracle; test infrastructure only).

Sources (the pages' text; equations restated, nothing copied):
  * Dion3: Full-Stack Orthogonal Updates, sec. 2.1 Definition 1 (polar = U V^T),
    sec. 2.2 Algorithm 1 (standard Newton-Schulz) and its FLOP count,
    sec. 2.3 (symmetric products), sec. 4 Theorem 2 (scalar recurrence),
    Algorithm 2 (naive Gram Newton-Schulz), sec. 4.1 (its FLOP count),
    sec. 4.2 and Algorithm 3 (stabilized Gram Newton-Schulz with a restart),
    appendix B.2.3 (the a_t I term is distributed, never added to Z).
  * Scaling Muon for Diffusion Transformers, appendix D.3: the fixed quintic
    coefficients (a, b, c) = (3.4445, -4.7750, 2.0315) used for all five iterations.
  * Dion3 appendix B.1.1: the classic coefficients (15/8, -10/8, 3/8).

Conventions. X is n x m with n <= m (the caller orients it). A coefficient schedule is a
list of (a_t, b_t, c_t), t = 1..T. ``restarts`` is a set of iteration counts i: a restart
happens after iteration i, i.e. at the start of iteration i+1 (Algorithm 3 restarts at
the start of t = 3, i.e. restarts = {2}).

FLOP accounting (FlopCounter): a product of an r x K by a K x c matrix counts 2 r c K; a
product whose result is symmetric counts half of that (sec. 2.3: only one triangle is
computed). Products that Algorithm 2/3 would form but whose value is never used (R after
the last iteration, R before a restart) or that multiply by Q = I are not formed, as sec.
4.1 and 4.2 count them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

EPS = 1e-7  # Algorithms 1-3, normalisation step: X <- X / (||X||_F + eps), eps = 1e-7

# Scaling Muon for Diffusion Transformers, appendix D.3: fixed quintic, five iterations.
QUINTIC_FIXED = [(3.4445, -4.7750, 2.0315)] * 5
# Dion3 appendix B.1.1: classic cubic-quintic coefficients (15/8, -10/8, 3/8).
CLASSIC = [(15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)] * 5


@dataclass
class FlopCounter:
    """Algorithmic FLOPs of the matrix products an algorithm forms (see module docstring)."""
    flops: float = 0.0
    log: list = field(default_factory=list)

    def product(self, rows: int, cols: int, inner: int, symmetric: bool, name: str = "") -> None:
        f = 2.0 * rows * cols * inner
        if symmetric:
            f /= 2.0
        self.flops += f
        self.log.append((name, rows, cols, inner, symmetric, f))


def _mm(A, B, counter, symmetric, name):
    if counter is not None:
        counter.product(A.shape[0], B.shape[1], A.shape[1], symmetric, name)
    return A @ B


def frobenius_normalize(X: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Algorithms 1-3, normalisation step: divide by the Frobenius norm plus eps (eps added, not a max)."""
    return X / (np.linalg.norm(X) + eps)


def polar(X: np.ndarray) -> np.ndarray:
    """Definition 1: polar(X) = U V^T from the thin SVD X = U S V^T."""
    U, _, Vt = np.linalg.svd(X, full_matrices=False)
    return U @ Vt


def odd_poly(x, a, b, c):
    """p(x) = a x + b x^3 + c x^5 (sec. 2.2)."""
    return a * x + b * x ** 3 + c * x ** 5


def h_poly(y, a, b, c):
    """h(y) = a + b y + c y^2, so that p(x) = x h(x^2) (sec. 4)."""
    return a + b * y + c * y * y


def compose(x, coeffs):
    """(p_T o ... o p_1)(x) elementwise: the map standard Newton-Schulz applies to each singular value."""
    x = np.asarray(x, dtype=np.float64)
    for (a, b, c) in coeffs:
        x = odd_poly(x, a, b, c)
    return x


def scalar_recurrence(x, coeffs, restarts=()):
    """Theorem 2 on scalars: r_0 = x^2, q_0 = 1; z_t = h_t(r_{t-1}), r_t = r_{t-1} z_t^2,
    q_t = q_{t-1} z_t; result q_T x.

    A restart after iteration i (sec. 4.2) replaces x by x_i = q_i x, r by x_i^2 and q by 1;
    in exact arithmetic this leaves the result unchanged. Returns (q_T * x, history) with
    history a list of (t, r_t, q_t) arrays.
    """
    x0 = np.asarray(x, dtype=np.float64)
    base = x0.copy()
    r = base * base
    q = np.ones_like(base)
    hist = [(0, r.copy(), q.copy())]
    for t, (a, b, c) in enumerate(coeffs, start=1):
        if (t - 1) in restarts and t > 1:
            base = q * base
            r = base * base
            q = np.ones_like(base)
        z = h_poly(r, a, b, c)
        r = r * z * z
        q = q * z
        hist.append((t, r.copy(), q.copy()))
    return q * base, hist


def ns_standard(X, coeffs, eps=EPS, counter=None, symmetric_products=True, normalize=True):
    """Algorithm 1 in float64 (the bfloat16 cast after the normalisation is left out: the oracle is exact).

    Each iteration: A = X X^T; B = b A + c A^2; X = a X + B X. With symmetric_products the
    counter charges A and A^2 as symmetric (sec. 2.3: T(3 alpha + 1) n^3 in total); without,
    as full products (sec. 2.2: 2T(2 alpha + 1) n^3).
    """
    X = np.asarray(X, dtype=np.float64)
    if normalize:
        X = frobenius_normalize(X, eps)
    for (a, b, c) in coeffs:
        A = _mm(X, X.T, counter, symmetric_products, "XXt")
        B = b * A + c * _mm(A, A, counter, symmetric_products, "A2")
        X = a * X + _mm(B, X, counter, False, "BX")
    return X


def gram_ns_naive(X, coeffs, eps=EPS, counter=None, trace=None, gram_perturb=None):
    """Algorithm 2 (naive Gram Newton-Schulz) in float64.

    R_0 = X X^T, Q_0 = I; for each t: Z_t = a_t I + b_t R_{t-1} + c_t R_{t-1}^2,
    Q_t = Q_{t-1} Z_t, R_t = Z_t R_{t-1} Z_t; return Q_T X.
    Q_1 = Z_1 is taken without a product (Q_0 = I) and R_T is not formed (sec. 4.1).
    ``trace`` (optional list) receives (t, R_t, Q_t) after every iteration;
    ``gram_perturb(R_0)`` (optional) is applied to R_0 right after it is formed (appendix
    B.1.2 rounds it through bfloat16).
    """
    X = frobenius_normalize(np.asarray(X, dtype=np.float64), eps)
    n = X.shape[0]
    I = np.eye(n)
    R = _mm(X, X.T, counter, True, "R0=XXt")
    if gram_perturb is not None:
        R = gram_perturb(R)
    Q = I.copy()
    q_is_identity = True
    T = len(coeffs)
    if trace is not None:
        trace.append((0, R.copy(), Q.copy()))
    for t, (a, b, c) in enumerate(coeffs, start=1):
        Z = a * I + b * R + c * _mm(R, R, counter, True, f"R{t-1}^2")
        Q = Z.copy() if q_is_identity else _mm(Q, Z, counter, True, f"Q{t}")
        q_is_identity = False
        if t < T:
            R = _mm(_mm(Z, R, counter, True, f"ZR{t}"), Z, counter, True, f"R{t}")
        if trace is not None:
            trace.append((t, R.copy(), Q.copy()))
    return _mm(Q, X, counter, False, "QX")


def gram_ns_stabilized(X, coeffs, restarts=(2,), eps=EPS, counter=None, trace=None,
                       gram_perturb=None):
    """Algorithm 3 (stabilized Gram Newton-Schulz) in float64.

    Step order per iteration t (the a_t I term is distributed, appendix B.2.3):
        if a restart falls after iteration t-1:  X <- Q_{t-1} X;  R_{t-1} <- X X^T;  Q_{t-1} <- I
        Z_t    = b_t R_{t-1} + c_t R_{t-1}^2
        Q_t    = Q_{t-1} Z_t + a_t Q_{t-1}
        (RZ)_t = R_{t-1} Z_t + a_t R_{t-1}
        R_t    = Z_t (RZ)_t + a_t (RZ)_t
    and the result is Q_T X.

    Not formed, as sec. 4.1/4.2 count them: the product Q_{t-1} Z_t when Q_{t-1} = I
    (then Q_t = Z_t + a_t I), and R_t (with its RZ) when R_t is never read, i.e. after the
    last iteration or right before a restart.

    ``gram_perturb(R)`` (optional) is applied to every Gram matrix X X^T right after it is
    formed; appendix B.2.1 uses it to plant a spurious eigenvalue. ``trace`` receives
    (t, R_t or None, Q_t) after every iteration and ("restart", R, X) at a restart.
    """
    X = frobenius_normalize(np.asarray(X, dtype=np.float64), eps)
    n = X.shape[0]
    I = np.eye(n)
    T = len(coeffs)
    restarts = set(int(r) for r in restarts)

    def gram(Y, name):
        R_ = _mm(Y, Y.T, counter, True, name)
        return gram_perturb(R_) if gram_perturb is not None else R_

    R = gram(X, "R0=XXt")
    Q = I.copy()
    q_is_identity = True
    if trace is not None:
        trace.append((0, R.copy(), Q.copy()))
    for t, (a, b, c) in enumerate(coeffs, start=1):
        if (t - 1) in restarts and t > 1:
            X = _mm(Q, X, counter, False, f"X{t-1}=QX")
            R = gram(X, f"R{t-1}=XXt")
            Q = I.copy()
            q_is_identity = True
            if trace is not None:
                trace.append(("restart", R.copy(), X.copy()))
        Z = b * R + c * _mm(R, R, counter, True, f"R{t-1}^2")
        if q_is_identity:
            Qn = Z + a * I
        else:
            Qn = _mm(Q, Z, counter, True, f"Q{t}") + a * Q
        r_needed = t < T and t not in restarts
        if r_needed:
            RZ = _mm(R, Z, counter, True, f"RZ{t}") + a * R
            R = _mm(Z, RZ, counter, True, f"R{t}") + a * RZ
        else:
            R = None
        Q = Qn
        q_is_identity = False
        if trace is not None:
            trace.append((t, None if R is None else R.copy(), Q.copy()))
    return _mm(Q, X, counter, False, "QX")


# ----------------------------------------------------------------------------------------
# FLOP formulas printed on the pages (used to pin the counter, not by the algorithms).

def flops_standard_formula(n, m, T, symmetric):
    """sec. 2.2: 2T(2 alpha + 1) n^3 without symmetric products; sec. 2.3: T(3 alpha + 1) n^3 with."""
    alpha = m / n
    return (T * (3 * alpha + 1) if symmetric else 2 * T * (2 * alpha + 1)) * n ** 3


def flops_gram_naive_formula(n, m, T):
    """sec. 4.1: (4T + 3 alpha - 3) n^3."""
    return (4 * T + 3 * (m / n) - 3) * n ** 3


def flops_restart_extra_formula(n, m):
    """sec. 4.2: a restart costs 3(alpha - 1) n^3 more."""
    return 3 * ((m / n) - 1) * n ** 3
