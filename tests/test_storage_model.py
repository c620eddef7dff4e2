"""CPU checks of the 16-bit storage model used by the GPU precision tests: without rounding
it is Algorithm 3 / Algorithm 1 exactly (so it models nothing but storage), and with bf16
storage it reproduces the effect the GPU tests attribute to it (errors well above the
tolerance on effectively rank-one spectra, about 8x smaller with fp16 storage)."""
import numpy as np

from matrix_orthogonalizing_optimizer_gb300 import inputs
from oracle import muon as omuon
from oracle import newton_schulz as ons
from storage_model import gram_ns_stored, ns_standard_stored, round_bf16, round_fp16


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def test_without_rounding_the_model_is_the_algorithm():
    X = inputs.gaussian(3, (24, 96), 0.1)
    ident = lambda A: A
    assert _rel(gram_ns_stored(X, ons.QUINTIC_FIXED, ident), ons.gram_ns_stabilized(X, ons.QUINTIC_FIXED)) < 1e-12
    assert _rel(gram_ns_stored(X, ons.CLASSIC * 6, ident, restarts=(2, 4)),
                ons.gram_ns_stabilized(X, ons.CLASSIC * 6, restarts=(2, 4))) < 1e-12
    assert _rel(ns_standard_stored(X, ons.QUINTIC_FIXED, ident), ons.ns_standard(X, ons.QUINTIC_FIXED)) < 1e-12


def test_bf16_storage_loses_effectively_rank_one_spectra():
    g = np.random.default_rng(0)
    n, m = 8, 256
    U, _ = np.linalg.qr(g.standard_normal((n, n)))
    V, _ = np.linalg.qr(g.standard_normal((m, n)))
    s = np.full(n, 1e-3)
    s[0] = 1.0
    X = round_bf16((U * s) @ V.T / np.sqrt(m))
    want = omuon.orthogonalize(X)
    e_bf = _rel(gram_ns_stored(X, ons.QUINTIC_FIXED, round_bf16), want)
    e_16 = _rel(gram_ns_stored(X, ons.QUINTIC_FIXED, round_fp16), want)
    assert e_bf > 5e-2 and e_16 < e_bf / 3
