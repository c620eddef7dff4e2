"""Algorithm 3 (and Algorithm 1) with every stored matrix rounded to a 16-bit storage type:
a model of the error ANY implementation that stores its iterates in that type must show,
whatever its kernels do. Products are exact (fp64) and each stored result is rounded once,
as the library's epilogues do (fp32 accumulation is far finer than 16-bit storage); the
a_t I term enters as in Algorithm 3 (never added into a stored Z, Dion3 appendix B.2.3).

Test infrastructure only. It is not the oracle (the oracle is exact) and shares no code with
the CUDA library: the GPU precision tests use it to show that where the bf16 path misses the
stated tolerance, the miss is the cost of bf16 storage itself.
"""
import numpy as np

from matrix_orthogonalizing_optimizer_gb300 import inputs


def round_bf16(x):
    return inputs.bf16_bits_to_f32(inputs.round_to_bf16_bits(x)).astype(np.float64)


def round_fp16(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


def _upper_mirrored(A):
    """A symmetric product formed from its upper triangle, as the library's triangle tiles do."""
    return np.triu(A) + np.triu(A, 1).T


def gram_ns_stored(X, coeffs, rnd, restarts=(2,), eps=1e-7):
    """Dion3 Algorithm 3 with R, Z, Q, RZ and the restart's X rounded by `rnd` when stored."""
    X = np.asarray(X, dtype=np.float64)
    s = 1.0 / (np.linalg.norm(X) + eps)
    n = X.shape[0]
    I = np.eye(n)
    R = rnd(_upper_mirrored(s * s * (X @ X.T)))
    Q = None
    Xc, xs = X, s
    T = len(coeffs)
    for t, (a, b, c) in enumerate(coeffs, start=1):
        if (t - 1) in restarts and t > 1:
            Xc = rnd(xs * (Q @ Xc))
            xs = 1.0
            R = rnd(_upper_mirrored(Xc @ Xc.T))
            Q = None
        Zf = b * R + c * _upper_mirrored(R @ R)
        Z = rnd(Zf)
        Qn = rnd(Zf + a * I) if Q is None else rnd(_upper_mirrored(Q @ Z) + a * Q)
        if t < T and t not in restarts:
            RZ = rnd(_upper_mirrored(R @ Z) + a * R)
            R = rnd(_upper_mirrored(Z @ RZ) + a * RZ)
        Q = Qn
    return xs * (Q @ Xc)


def ns_standard_stored(X, coeffs, rnd, eps=1e-7):
    """Dion3 Algorithm 1 with A, B and every X_t rounded by `rnd` when stored."""
    X = np.asarray(X, dtype=np.float64)
    xs = 1.0 / (np.linalg.norm(X) + eps)
    Xc = X
    for (a, b, c) in coeffs:
        A = rnd(_upper_mirrored(xs * xs * (Xc @ Xc.T)))
        B = rnd(b * A + c * _upper_mirrored(A @ A))
        Xc = rnd(a * xs * Xc + xs * (B @ Xc))
        xs = 1.0
    return Xc
