"""Muon step and Dion3 fractional update in float64 (oracle; test infrastructure only).

Sources (restated, nothing copied):
  * Dion3 sec. 2.1 eq. (1): M <- mu M + G;  W <- W - eta polar(M).
  * Dion3 Algorithm 1 (n <= m): a matrix with more rows than columns is orthogonalized
    through its transpose and mapped back (polar(M^T) = polar(M)^T).
  * Dion3 sec. 6 and Algorithm 4 (Muon flavour): M <- M + G; S = the k = ceil(f n) rows of
    largest l1 norm; O = polar(M[S, :]); W <- (1 - eta wd) W (all rows); W[S, :] -= eta O;
    M[S, :] <- mu M[S, :] (error feedback: only the selected rows decay). Rows are the
    smaller dimension when the matrix is not sharded (sec. 6, "Selection").

Precision contract with the GPU path. The Muon step's momentum and weight are stored in
bfloat16 there, so a value that the GPU stores and later reads back is, in the oracle too,
the same bf16 value: ``momentum_update_bf16`` and ``decay_rows_bf16`` round
float32(mu * m + g) and float32(mu * m) to bf16 exactly as one correctly rounded float32
operation followed by one round-to-nearest-even to bf16. Selection is an integer decision
taken from the stored bf16 momentum, with exact l1 sums (``l1_keys_exact``), so indices are
bit-exact whatever order the sums are formed in. The orthogonalization and the weight
update are float64.
"""
from __future__ import annotations

import math

import numpy as np

from .newton_schulz import EPS, QUINTIC_FIXED, gram_ns_stabilized


# ---------------------------------------------------------------------------------------
# bf16 storage helpers (own implementation: the oracle shares no code with the GPU path)

def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """float64 values of uint16 bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_encode_from_f32(x32: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits of float32 values, round to nearest even (NaN -> canonical NaN)."""
    x32 = np.ascontiguousarray(np.asarray(x32, dtype=np.float32))
    u = x32.view(np.uint32).astype(np.uint64)
    out = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    out[np.isnan(x32)] = 0x7FC0
    return out


def momentum_update_bf16(M_bits, G_bits, mu):
    """bf16 bits of float32(mu * M + G) (mu = 1 gives the M + G of Algorithm 4)."""
    m = bf16_decode(M_bits).astype(np.float32)
    g = bf16_decode(G_bits).astype(np.float32)
    if mu == 1.0:
        s = m + g
    else:
        s = np.float32(mu) * m + g  # float32 product then float32 sum: two roundings
    return bf16_encode_from_f32(s)


def decay_rows_bf16(M_bits, rows, mu):
    """bf16 bits of M with the given rows replaced by float32(mu * M[row])."""
    out = np.array(M_bits, dtype=np.uint16, copy=True)
    m = bf16_decode(out[rows]).astype(np.float32)
    out[rows] = bf16_encode_from_f32(np.float32(mu) * m)
    return out


# ---------------------------------------------------------------------------------------
# Exact l1 keys and top-k (the selection step of Algorithm 4)

NONFINITE_KEY = 1 << 400  # above every finite key (a finite bf16 row sum is < 2^290)


def l1_keys_exact(rows_bits: np.ndarray) -> list:
    """Exact l1 norm of every row of a bf16 matrix, as a Python int in units of 2^-133.

    A finite bf16 value with exponent field E and fraction f has magnitude
    (E > 0 ? 128 + f : f) * 2^(max(E, 1) - 134), i.e. an integer mantissa times 2^(e - 1)
    units of 2^-133 with e = max(E, 1). A row's key is the exact sum of these integers
    (histogram over e of the summed mantissas, then shifted and added). Rows holding an
    Inf or NaN get NONFINITE_KEY.
    """
    b = np.asarray(rows_bits, dtype=np.uint16)
    E = ((b >> 7) & 0xFF).astype(np.int64)
    frac = (b & 0x7F).astype(np.int64)
    mant = np.where(E > 0, frac + 128, frac)
    e = np.maximum(E, 1)
    keys = []
    for i in range(b.shape[0]):
        if np.any(E[i] == 255):
            keys.append(NONFINITE_KEY)
            continue
        hist = np.bincount(e[i], weights=mant[i], minlength=256)  # exact: < 2^53
        k = 0
        for ee in np.nonzero(hist)[0]:
            k += int(hist[ee]) << (int(ee) - 1)
        keys.append(k)
    return keys


def top_k_rows(keys: list, k: int) -> np.ndarray:
    """Indices of the k largest keys; equal keys go to the lower index; returned ascending."""
    order = sorted(range(len(keys)), key=lambda i: (-keys[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


# ---------------------------------------------------------------------------------------
# Steps

def orient(A):
    """(A or A^T, transposed?) so that the working matrix has rows <= cols."""
    return (A.T, True) if A.shape[0] > A.shape[1] else (A, False)


def orthogonalize(M, coeffs=QUINTIC_FIXED, restarts=(2,), eps=EPS):
    """Gram Newton-Schulz (Algorithm 3) applied to M of any shape, mapped back to M's shape."""
    X, tr = orient(np.asarray(M, dtype=np.float64))
    O = gram_ns_stabilized(X, coeffs, restarts=restarts, eps=eps)
    return O.T if tr else O


def muon_step(W_bits, G_bits, M_bits, lr, mu, weight_decay=0.0, scale=1.0,
              coeffs=QUINTIC_FIXED, restarts=(2,), eps=EPS):
    """One Muon step, eq. (1), with the weight update W <- (1 - lr wd) W - lr scale O.

    Returns (W_new float64, M_new bf16 bits, O float64). M_new is what the GPU stores; the
    orthogonalization runs on its decoded value.
    """
    M_new = momentum_update_bf16(M_bits, G_bits, mu)
    O = orthogonalize(bf16_decode(M_new), coeffs, restarts, eps)
    W = bf16_decode(W_bits)
    W_new = (1.0 - lr * weight_decay) * W - lr * scale * O
    return W_new, M_new, O


def frac_step(W_bits, G_bits, M_bits, frac, lr, mu, weight_decay=0.0, scale=1.0,
              coeffs=QUINTIC_FIXED, restarts=(2,), eps=EPS):
    """One Dion3 update (Algorithm 4, Muon flavour) on rows, or on columns of a tall matrix.

    Returns (W_new float64, M_new bf16 bits, S int64 ascending, O float64 k x m).
    """
    M_bits = np.asarray(M_bits, dtype=np.uint16)
    Msum = momentum_update_bf16(M_bits, G_bits, 1.0)         # M <- M + G
    Xb, tr = orient(Msum)
    n = Xb.shape[0]
    k = int(math.ceil(frac * n - 1e-12))
    k = max(1, min(k, n))
    S = top_k_rows(l1_keys_exact(Xb), k)                     # selection
    O = gram_ns_stabilized(bf16_decode(Xb[S, :]), coeffs, restarts=restarts, eps=eps)  # O = polar(M[S])
    W = bf16_decode(W_bits)
    W = (1.0 - lr * weight_decay) * W                        # weight decay (all rows)
    Wo, _ = orient(W)
    Wo = Wo.copy()
    Wo[S, :] -= lr * scale * O                               # update (selected rows)
    W_new = Wo.T if tr else Wo
    Xn = decay_rows_bf16(np.ascontiguousarray(Xb), S, mu)    # error feedback
    M_new = np.ascontiguousarray(Xn.T) if tr else Xn
    return W_new, M_new, S, O
