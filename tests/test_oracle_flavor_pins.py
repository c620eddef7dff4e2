"""Pins of the oracle's update flavours (oracle/flavors.py) to facts the pages and the
mathematics fix (no GPU): a library routine (numpy polynomial composition), closed forms,
invariants the definitions imply, brute force on tiny inputs and the numbers the pages print
(tests/golden/pages_numbers.json)."""
import json
import os

import numpy as np
import pytest
from numpy.polynomial import Polynomial

from matrix_orthogonalizing_optimizer_gb300 import inputs
from oracle import flavors as fl, muon, newton_schulz as ns

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def bits(seed, shape, scale=0.1):
    return inputs.round_to_bf16_bits(inputs.gaussian(seed, shape, scale))


# ---------------------------------------------------------------------------------------
# safety factor (Dion3 appendix B.2.2)

def test_safety_factor_values_are_the_printed_ones():
    assert GOLD["safety_factor_usual"]["value"] == 1.02
    assert GOLD["safety_factor_conservative"]["value"] == 1.05


@pytest.mark.parametrize("s", [1.02, 1.05, 1.3])
def test_safety_adjust_is_composition_with_x_over_s(s):
    """numpy's polynomial composition p(q) with q(x) = x / s gives the coefficients of
    p_t(x / s) independently of the oracle's formula."""
    for (a, b, c), (a2, b2, c2) in zip(ns.QUINTIC_FIXED + ns.CLASSIC, fl.safety_adjust(ns.QUINTIC_FIXED + ns.CLASSIC, s)):
        p = Polynomial([0, a, 0, b, 0, c])
        comp = p(Polynomial([0, 1.0 / s]))
        want = np.zeros(6)
        want[: len(comp.coef)] = comp.coef
        assert np.allclose([0, a2, 0, b2, 0, c2], want, rtol=1e-14, atol=1e-15)


def test_safety_factor_keeps_values_up_to_s_inside_the_unit_interval():
    """Appendix B.2.2: run as p(x / s), singular values as large as s still converge. The
    classic cubic-quintic maps [0, 1] into [0, 1] with p(1) = 1 (appendix B.1.1); adjusted,
    it maps all of [0, s] into [0, 1], while unadjusted it pushes values just above 1
    further above 1, and the iteration then drifts away instead of settling near 1."""
    s = 1.05
    x = np.linspace(0.0, s, 2001)
    (a, b, c), = fl.safety_adjust(ns.CLASSIC[:1], s)
    assert ns.odd_poly(s, a, b, c) == pytest.approx(1.0, abs=1e-14)  # p(s / s) = p(1) = 1
    assert ns.odd_poly(x, a, b, c).max() <= 1.0 + 1e-14
    assert ns.odd_poly(x, *ns.CLASSIC[0]).max() > 1.0
    y = ns.compose(x[x > 0.3], fl.safety_adjust(ns.CLASSIC, s) * 4)
    assert np.all(np.abs(y - 1.0) < 0.05)


def test_safety_one_is_identity_and_gram_ns_runs_adjusted_table():
    assert fl.safety_adjust(ns.QUINTIC_FIXED, 1.0) == list(ns.QUINTIC_FIXED)
    X = inputs.gaussian(1, (16, 48))
    adj = fl.safety_adjust(ns.QUINTIC_FIXED, 1.05)
    O = ns.gram_ns_stabilized(X, adj)
    # Theorem 2 on the singular values: the adjusted polynomials act on each sigma
    U, S, Vt = np.linalg.svd(ns.frobenius_normalize(X), full_matrices=False)
    assert rel(O, (U * ns.compose(S, adj)) @ Vt) < 1e-10


# ---------------------------------------------------------------------------------------
# NorMuon (Dion3 eq. (2), the NorMuon steps of Algorithm 4)

def test_normuon_keeps_the_frobenius_norm():
    O = inputs.gaussian(2, (12, 40))
    D, v = fl.normuon(O, np.full(12, 0.3), beta2=0.9, eps=1e-8)
    assert np.linalg.norm(D) == pytest.approx(np.linalg.norm(O), rel=1e-14)


def test_normuon_with_beta2_zero_equalises_row_norms():
    """beta2 = 0, eps -> 0: v_i = mean_j O_ij^2, so O_i / sqrt(v_i) has norm sqrt(m) for
    every row; after the Frobenius rescale every row norm is ||O||_F / sqrt(n). A divisor
    v_i instead of sqrt(v_i), or a missing mean, breaks this."""
    O = inputs.gaussian(3, (10, 32)) * np.linspace(0.1, 3.0, 10)[:, None]
    D, v = fl.normuon(O, np.zeros(10), beta2=0.0, eps=0.0)
    rn = np.linalg.norm(D, axis=1)
    assert np.allclose(rn, np.linalg.norm(O) / np.sqrt(10), rtol=1e-12)
    assert np.allclose(v, np.mean(O ** 2, axis=1), rtol=1e-14)


def test_normuon_uniform_rows_reduce_to_muon():
    """Rows of equal norm with equal second moments are scaled alike, and the rescale
    restores O exactly: NorMuon = Muon."""
    Q, _ = np.linalg.qr(inputs.gaussian(4, (48, 8)))
    O = Q.T  # 8 x 48, orthonormal rows (all of norm 1)
    D, v = fl.normuon(O, np.full(8, 0.02), beta2=0.95, eps=1e-8)
    assert rel(D, O) < 1e-13


def test_normuon_second_moment_recursion_by_hand():
    O = np.array([[1.0, -1.0, 1.0, -1.0], [2.0, 0.0, 0.0, 0.0]])
    D, v = fl.normuon(O, np.array([0.5, 4.0]), beta2=0.75, eps=0.0)
    # v_0 = 0.75*0.5 + 0.25*1 = 0.625; v_1 = 0.75*4 + 0.25*(4/4) = 3.25
    assert v == pytest.approx([0.625, 3.25], abs=1e-15)
    rows = [O[0] / np.sqrt(0.625), O[1] / np.sqrt(3.25)]
    hat = np.array(rows)
    assert rel(D, hat * np.linalg.norm(O) / np.linalg.norm(hat)) < 1e-15
    # selected rows only (Algorithm 4): rows 1 and 3 of a 4-row buffer
    D2, v2 = fl.normuon(O, np.array([9.0, 0.5, 9.0, 4.0]), beta2=0.75, eps=0.0, rows=[1, 3])
    assert v2 == pytest.approx([9.0, 0.625, 9.0, 3.25], abs=1e-15)
    assert rel(D2, D) < 1e-15


def test_normuon_step_dense_and_fractional_agree_at_full_fraction():
    W, G = bits(5, (16, 64)), bits(6, (16, 64))
    M = np.zeros_like(G)
    v = np.full(16, 0.01)
    Wd, Md, vd, Dd = fl.normuon_step(W, G, M, v, lr=0.02, mu=0.95, beta2=0.95, eps=1e-8)
    Wf, Mf, vf, S, Df = fl.normuon_frac_step(W, G, M, v, 1.0, lr=0.02, mu=0.95, beta2=0.95, eps=1e-8)
    assert list(S) == list(range(16))
    assert rel(Wf, Wd) < 1e-12 and rel(vf, vd) < 1e-14
    # tall matrix: the oriented rows are the columns
    Wt, Mt, vt, Dt = fl.normuon_step(W.T.copy(), G.T.copy(), M.T.copy(), v, lr=0.02, mu=0.95, beta2=0.95, eps=1e-8)
    assert rel(Wt, Wd.T) < 1e-12 and rel(vt, vd) < 1e-14


def test_normuon_frac_updates_only_selected_moments():
    W, G, M = bits(7, (24, 80)), bits(8, (24, 80)), bits(9, (24, 80))
    v = np.linspace(0.01, 0.05, 24)
    Wn, Mn, vn, S, D = fl.normuon_frac_step(W, G, M, v, 0.25, lr=0.02, mu=0.95, beta2=0.9, eps=1e-8)
    Wm, Mm, Sm, O = muon.frac_step(W, G, M, 0.25, lr=0.02, mu=0.95)
    assert list(S) == list(Sm) and np.array_equal(Mn, Mm)         # selection and EF as Muon's
    unsel = np.setdiff1d(np.arange(24), S)
    assert np.array_equal(vn[unsel], v[unsel])
    assert np.linalg.norm(D) == pytest.approx(np.linalg.norm(O), rel=1e-13)


# ---------------------------------------------------------------------------------------
# RowNorm and Periodic Row-wise Muon (Scaling Muon for DiTs eq. (5), (7), (8))

def test_rownorm_unit_rows_and_floor():
    X = inputs.gaussian(10, (6, 9))
    X[2] *= 1e-9
    X[4] = 0.0
    R = fl.rownorm(X, eps=1e-6)
    n = np.linalg.norm(R, axis=1)
    assert np.allclose(n[[0, 1, 3, 5]], 1.0, rtol=1e-14)
    assert np.allclose(R[2], X[2] / 1e-6) and np.all(R[4] == 0.0)


def test_rownorm_maximises_inner_product_under_row_norm_bound():
    """Lemma 1 of the page: among U with every row norm <= 1, R(X) maximises <X, U>, whose
    maximum is the sum of the row norms. Brute force over random feasible U."""
    X = inputs.gaussian(11, (5, 7))
    R = fl.rownorm(X, eps=1e-12)
    best = np.sum(X * R)
    assert best == pytest.approx(np.sum(np.linalg.norm(X, axis=1)), rel=1e-13)
    g = inputs.rng(12)
    for _ in range(2000):
        U = g.standard_normal((5, 7))
        U /= np.maximum(np.linalg.norm(U, axis=1), 1.0)[:, None] * g.uniform(1.0, 2.0, size=(5, 1))
        assert np.sum(X * U) <= best + 1e-12


def test_rownorm_of_tall_matrix_normalises_columns_and_matches_sharded_statistics():
    """Eq. (8): the column norms from per-shard sums of squares equal the dense ones, so
    RowNorm of the oriented (transposed) tall matrix divides each column by them."""
    M = inputs.gaussian(13, (40, 12))
    shards = [np.arange(0, 7), np.arange(7, 25), np.arange(25, 40)]
    nu = fl.column_norms_sharded(M, shards, eps=1e-8)
    X, tr = muon.orient(M)
    assert tr
    D = fl.rownorm(X, 1e-8).T
    assert rel(D, M / nu[None, :]) < 1e-14


def test_periodic_schedule_and_printed_defaults():
    K = GOLD["periodic_K"]["value"]
    assert K == 3 and GOLD["rownorm_gamma"]["value"] == 0.15
    assert [fl.refresh(t, K) for t in range(7)] == [True, False, False, True, False, False, True]
    # sec. 3.3: one momentum all-gather every K steps -> payload ratio 1/K
    assert sum(fl.refresh(t, K) for t in range(3000)) / 3000 == pytest.approx(GOLD["periodic_payload_ratio_K3"]["value"])


def test_rownorm_step_update_by_hand():
    W, G, M = bits(14, (8, 24)), bits(15, (8, 24)), bits(16, (8, 24))
    Wn, Mn, D = fl.rownorm_step(W, G, M, lr=0.02, mu=0.95, gamma=0.15, eps=1e-8, weight_decay=0.1, scale=1.5)
    Mv = muon.bf16_decode(muon.momentum_update_bf16(M, G, 0.95))
    want = 0.15 * Mv / np.linalg.norm(Mv, axis=1, keepdims=True)
    assert rel(D, want) < 1e-14
    assert rel(Wn, (1 - 0.002) * muon.bf16_decode(W) - 0.03 * want) < 1e-14
    # the direction's rows all have norm gamma, the polar factor's Frobenius norm is sqrt(r)
    # times gamma (sec. 3.2: both maps have Frobenius norm sqrt(r) before gamma)
    assert np.linalg.norm(D) == pytest.approx(0.15 * np.sqrt(8), rel=1e-13)
