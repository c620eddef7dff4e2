"""Pins of the CPU oracle to facts the pages and the mathematics fix (no GPU).

Each test ties an oracle function to something other than itself: a closed form from the
SVD, a library routine, brute force on tiny inputs, or a number the pages print
(tests/golden/pages_numbers.json, each entry with its citation).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from matrix_orthogonalizing_optimizer_gb300 import inputs
from oracle import muon, newton_schulz as ns, stability as st

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def test_coefficients_are_the_printed_ones():
    assert list(ns.QUINTIC_FIXED[0]) == GOLD["quintic_fixed"]["value"] and len(ns.QUINTIC_FIXED) == 5
    assert list(ns.CLASSIC[0]) == GOLD["classic"]["value"]
    assert ns.EPS == GOLD["eps"]["value"]


def test_odd_polynomial_values():
    # classic polynomial fixes 1 with zero slope: p(1) = 1, p'(1) = 15/8 - 30/8 + 15/8 = 0
    a, b, c = ns.CLASSIC[0]
    assert ns.odd_poly(1.0, a, b, c) == pytest.approx(1.0, abs=1e-15)
    d = 1e-6
    assert (ns.odd_poly(1 + d, a, b, c) - ns.odd_poly(1 - d, a, b, c)) / (2 * d) == pytest.approx(0.0, abs=1e-8)
    # p(1/2) = 15/16 - 10/64 + 3/256 by hand
    assert ns.odd_poly(0.5, a, b, c) == pytest.approx(15 / 16 - 10 / 64 + 3 / 256, abs=1e-15)
    # fixed quintic at 1: sum of the printed coefficients
    assert ns.odd_poly(1.0, *ns.QUINTIC_FIXED[0]) == pytest.approx(3.4445 - 4.7750 + 2.0315, abs=1e-12)
    # odd: p(-x) = -p(x); h relates as p(x) = x h(x^2) checked at a non-trivial point
    x = 0.37
    assert ns.odd_poly(-x, *ns.QUINTIC_FIXED[0]) == -ns.odd_poly(x, *ns.QUINTIC_FIXED[0])
    assert ns.h_poly(x * x, *ns.QUINTIC_FIXED[0]) * x == pytest.approx(ns.odd_poly(x, *ns.QUINTIC_FIXED[0]), rel=1e-14)


@pytest.mark.parametrize("coeffs", [ns.QUINTIC_FIXED, ns.CLASSIC, [(3.0, -2.0, 0.5), (1.5, -0.6, 0.1), (2.0, -1.0, 0.2)]])
@pytest.mark.parametrize("restarts", [(), (1,), (2,), (1, 2)])
def test_theorem2_scalar_recurrence_equals_composition(coeffs, restarts):
    x = np.concatenate([[0.0, 1e-4], np.linspace(0.01, 1.0, 200)])
    got, _ = ns.scalar_recurrence(x, coeffs, restarts=restarts)
    want = ns.compose(x, coeffs)
    assert np.max(np.abs(got - want)) <= 1e-13 * max(1.0, np.max(np.abs(want)))


def _svd_closed_form(X, coeffs, eps=ns.EPS):
    """Standard NS acts on singular values only: U phi(S/(||X||+eps)) V^T (Dion3 sec. 2.2)."""
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    s = S / (np.linalg.norm(X) + eps)
    return (U * ns.compose(s, coeffs)) @ Vt


@pytest.mark.parametrize("shape", [(128, 512), (17, 40), (32, 32), (1, 9)])
@pytest.mark.parametrize("coeffs", [ns.QUINTIC_FIXED, ns.CLASSIC])
def test_standard_ns_matches_svd_closed_form(shape, coeffs):
    X = inputs.gaussian(1, shape)
    assert rel(ns.ns_standard(X, coeffs), _svd_closed_form(X, coeffs)) < 1e-10


@pytest.mark.parametrize("shape", [(128, 512), (17, 40), (32, 32), (5, 64)])
@pytest.mark.parametrize("coeffs", [ns.QUINTIC_FIXED, ns.CLASSIC])
def test_gram_variants_match_svd_closed_form(shape, coeffs):
    """Theorem 2 lifted to matrices: naive and stabilized Gram NS give standard NS's result."""
    X = inputs.gaussian(2, shape)
    want = _svd_closed_form(X, coeffs)
    assert rel(ns.gram_ns_naive(X, coeffs), want) < 1e-10
    for r in [(2,), (1,), (3,), (1, 3)]:
        assert rel(ns.gram_ns_stabilized(X, coeffs, restarts=r), want) < 1e-10


def test_c1_gram_equals_standard():
    X = inputs.gaussian(1, (128, 512))
    a = ns.gram_ns_stabilized(X, ns.QUINTIC_FIXED, restarts=(2,))
    b = ns.ns_standard(X, ns.QUINTIC_FIXED)
    assert rel(a, b) < 1e-10


def test_polar_definition():
    X = inputs.gaussian(3, (20, 50))
    P = ns.polar(X)
    assert np.allclose(P @ P.T, np.eye(20), atol=1e-12)
    # polar of U diag(s) V^T with known factors
    U, _ = np.linalg.qr(inputs.gaussian(4, (6, 6)))
    V, _ = np.linalg.qr(inputs.gaussian(5, (15, 6)))
    Y = (U * np.array([3.0, 2.0, 1.0, 0.5, 0.2, 0.1])) @ V.T
    assert np.allclose(ns.polar(Y), U @ V.T, atol=1e-12)


def test_converges_toward_polar():
    """Enough classic iterations on a well-conditioned input reach polar(X) (Dion3 sec. 2.2)."""
    Y = inputs.exp_spectrum(2, 16, 64, decades=1.0)       # sigma in [0.1, 1]
    C = ns.CLASSIC[:1] * 25
    P = ns.polar(Y)
    assert np.linalg.norm(ns.ns_standard(Y, C) - P) < 1e-10
    assert np.linalg.norm(ns.gram_ns_stabilized(Y, C, restarts=(5, 10, 15, 20)) - P) < 1e-10


def test_fixed_quintic_band():
    """The fixed quintic maps [0.01, 1] into a band around 1 (it does not fix 1): the
    output's singular values lie in that band."""
    xs = np.logspace(-2, 0, 5001)
    phi = ns.compose(xs, ns.QUINTIC_FIXED)
    lo, hi = phi.min(), phi.max()
    assert 0.6 < lo < 0.7 and 1.1 < hi < 1.2
    X = inputs.exp_spectrum(6, 64, 256, decades=1.0)   # normalised sigma within [0.01, 1]
    s0 = np.linalg.svd(X, compute_uv=False) / np.linalg.norm(X)
    assert s0.min() > 0.01
    s = np.linalg.svd(ns.gram_ns_stabilized(X, ns.QUINTIC_FIXED), compute_uv=False)
    assert s.min() >= lo - 1e-9 and s.max() <= hi + 1e-9


@pytest.mark.parametrize("alpha", [1, 2, 4, 8])
@pytest.mark.parametrize("T", [3, 5, 6])
def test_flop_counter_matches_page_formulas(alpha, T):
    n = 16
    m = alpha * n
    X = inputs.gaussian(7, (n, m))
    C = ns.QUINTIC_FIXED[:1] * T
    c = ns.FlopCounter(); ns.ns_standard(X, C, counter=c, symmetric_products=False)
    assert c.flops == pytest.approx(ns.flops_standard_formula(n, m, T, symmetric=False))
    c = ns.FlopCounter(); ns.ns_standard(X, C, counter=c)
    assert c.flops == pytest.approx(ns.flops_standard_formula(n, m, T, symmetric=True))
    c = ns.FlopCounter(); ns.gram_ns_naive(X, C, counter=c)
    assert c.flops == pytest.approx(ns.flops_gram_naive_formula(n, m, T))
    c = ns.FlopCounter(); ns.gram_ns_stabilized(X, C, restarts=(2,), counter=c)
    assert c.flops == pytest.approx(ns.flops_gram_naive_formula(n, m, T) + ns.flops_restart_extra_formula(n, m))


def test_flop_formulas_match_printed_numbers():
    n, m, T = 10, 40, 5
    std_nosym = ns.flops_standard_formula(n, m, T, symmetric=False) / n ** 3
    a, b = GOLD["flops_std_nosym_T5"]["coef"]
    assert std_nosym == pytest.approx(a * 4 + b)                        # (20a+10) at a=4
    std_sym = ns.flops_standard_formula(n, m, T, symmetric=True) / n ** 3
    gram = ns.flops_gram_naive_formula(n, m, T) / n ** 3
    assert round(1 - gram / std_sym, 2) == GOLD["saving_vs_sym_T5_a4"]["value"]
    assert round(1 - gram / std_nosym, 2) == GOLD["saving_vs_nosym_T5_a4"]["value"]
    # alpha = 1: Gram and standard (symmetric) cost the same (sec. 4.1)
    assert ns.flops_gram_naive_formula(8, 8, 5) == ns.flops_standard_formula(8, 8, 5, True)
    # with restart at alpha=4: 38 n^3 = (14 + 6 alpha) n^3
    assert gram + ns.flops_restart_extra_formula(n, m) / n ** 3 == pytest.approx(38.0)


def test_negative_eigenvalue_growth_classic():
    """Appendix B.1.2 eq. (4): r_t < (15/8)^2 r_{t-1} for r_{t-1} < 0 (classic)."""
    g = GOLD["classic_negative_growth"]["value"]
    r0 = -np.logspace(-6, 0, 200)
    rs, _ = st.simulate_scalar(np.zeros(1), ns.CLASSIC[:1], None, delta=0.0)
    a, b, c = ns.CLASSIC[0]
    r1 = r0 * ns.h_poly(r0, a, b, c) ** 2
    assert np.all(r1 < g * r0)
    # simulate_scalar reproduces the step on a planted -delta
    rs, qs = st.simulate_scalar(np.zeros(1), ns.CLASSIC[:2], None, delta=4e-4)
    assert rs[1][0] < g * rs[0][0] and rs[2][0] < g * rs[1][0]


def test_restart_sweep_invariance_and_ranking():
    # with no planted error a restart changes nothing (sec. 4.2): same q_T x everywhere
    x = np.linspace(0.0, 1.0, 101)
    outs = []
    for loc in [None, 1, 2, 3, 4]:
        rs, qs = st.simulate_scalar(x, ns.QUINTIC_FIXED, loc, delta=0.0)
        base, _ = ns.scalar_recurrence(x, ns.QUINTIC_FIXED[:loc] if loc else ns.QUINTIC_FIXED)
        outs.append(qs[-1] * (base if loc else x) if loc else qs[-1] * x)
    want = ns.compose(x, ns.QUINTIC_FIXED)
    for o in outs:
        assert np.max(np.abs(o - want)) < 1e-12
    sweep = st.restart_sweep(ns.QUINTIC_FIXED, delta=GOLD["spurious_eigenvalue"]["value"] * -1)
    # no restart blows up; one restart in the middle bounds Q far better than at the ends
    assert sweep[None][0] > 1e6
    assert max(sweep[2][0], sweep[3][0]) < min(sweep[1][0], sweep[4][0])


def test_b1_naive_bf16_gram_diverges_fp64_converges():
    """B.1.1/B.1.2 on the 128x512 exponential-spectrum matrix, classic coefficients: exact
    naive Gram NS converges; with R_0 rounded through bf16 it blows up by iteration 10."""
    X = inputs.exp_spectrum(1, 128, 512)
    C = ns.CLASSIC[:1] * 16
    out = ns.gram_ns_naive(X, C)
    s = np.linalg.svd(out, compute_uv=False)
    assert np.allclose(s, 1.0, atol=1e-6)
    with np.errstate(all="ignore"):
        bad = ns.gram_ns_naive(X, ns.CLASSIC[:1] * 10, gram_perturb=inputs.bf16_round)
    assert not np.all(np.isfinite(bad)) or np.abs(bad).max() > 10.0


def test_b2_restart_bounds():
    """B.2 / B.2.1: with bf16-rounded Gram matrices, restart after 2 (fixed quintic) keeps
    eig(R_t) above -0.4 and eig(Q_t) below 100; restarting every 5 (classic, 25 its.) keeps
    Q bounded and the output's singular values near 1."""
    X = inputs.exp_spectrum(1, 128, 512)
    b = GOLD["restart2_bounds"]
    tr = []
    ns.gram_ns_stabilized(X, ns.QUINTIC_FIXED, restarts=(2,), trace=tr, gram_perturb=inputs.bf16_round)
    ev_r = min(np.linalg.eigvalsh(R).min() for (t, R, Q) in tr if isinstance(t, int) and R is not None)
    ev_q = max(np.abs(np.linalg.eigvalsh(Q)).max() for (t, R, Q) in tr if isinstance(t, int))
    assert ev_r > b["min_eig_R_above"] and ev_q < b["max_eig_Q_below"]
    with np.errstate(all="ignore"):
        trn = []
        ns.gram_ns_naive(X, ns.QUINTIC_FIXED, trace=trn, gram_perturb=inputs.bf16_round)
    assert max(np.abs(np.linalg.eigvalsh(Q)).max() for (t, R, Q) in trn) > b["max_eig_Q_below"]
    tr = []
    out = ns.gram_ns_stabilized(X, ns.CLASSIC[:1] * 25, restarts=(5, 10, 15, 20), trace=tr,
                                gram_perturb=inputs.bf16_round)
    s = np.linalg.svd(out, compute_uv=False)
    assert s.max() < 1.01 and s.min() > 0.99


def test_special_cases():
    # one row: output = phi(sigma) x/|x| with sigma = |x|/(|x|+eps)
    x = inputs.gaussian(8, (1, 33))
    sig = np.linalg.norm(x) / (np.linalg.norm(x) + ns.EPS)
    want = ns.compose(sig, ns.QUINTIC_FIXED) * x / np.linalg.norm(x)
    assert rel(ns.gram_ns_stabilized(x, ns.QUINTIC_FIXED), want) < 1e-12
    # orthonormal rows: all singular values equal 1/sqrt(n) after normalisation
    V, _ = np.linalg.qr(inputs.gaussian(9, (40, 8)))
    Y = V.T
    s = 1 / np.sqrt(8) * (np.sqrt(8) / (np.sqrt(8) + ns.EPS))
    assert rel(ns.gram_ns_stabilized(Y, ns.QUINTIC_FIXED), ns.compose(s, ns.QUINTIC_FIXED) * Y) < 1e-12
    # zero matrix: eps keeps it finite, output 0
    Z = np.zeros((4, 12))
    assert np.all(ns.gram_ns_stabilized(Z, ns.QUINTIC_FIXED) == 0)
    assert np.all(ns.ns_standard(Z, ns.QUINTIC_FIXED) == 0)


def test_bf16_rounding_against_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([inputs.gaussian(10, 5000), [0.0, -0.0, 1e-40, 3e38, -1e-30, 65504.0, 1.00390625, 1.01171875]])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(inputs.round_to_bf16_bits(x32), want)
    assert np.array_equal(muon.bf16_encode_from_f32(x32), want)
    assert np.array_equal(muon.bf16_decode(want), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_momentum_update_against_torch():
    torch = pytest.importorskip("torch")
    M = inputs.round_to_bf16_bits(inputs.gaussian(11, (8, 64)))
    G = inputs.round_to_bf16_bits(inputs.gaussian(12, (8, 64), 0.01))
    tM = torch.from_numpy(M.view(np.int16)).view(torch.bfloat16).float()
    tG = torch.from_numpy(G.view(np.int16)).view(torch.bfloat16).float()
    want = (torch.tensor(0.95, dtype=torch.float32) * tM + tG).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(muon.momentum_update_bf16(M, G, 0.95), want)
    want1 = (tM + tG).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(muon.momentum_update_bf16(M, G, 1.0), want1)


def _bits_to_fraction(b):
    b = int(b)
    E = (b >> 7) & 0xFF
    f = b & 0x7F
    if E == 0:
        return Fraction(f, 1) * Fraction(2) ** (-133)
    return Fraction(128 + f, 1) * Fraction(2) ** (E - 134)


def test_l1_keys_exact_brute_force():
    g = inputs.rng(13)
    bits = g.integers(0, 0x7F80, size=(12, 9), dtype=np.int64).astype(np.uint16)  # finite, all exponents
    bits[3] |= 0x8000                                                           # negatives
    bits[5, :] = 0                                                               # zero row
    bits[6, :4] = [1, 2, 0x0080, 0x7F7F]                                         # subnormals + max
    keys = muon.l1_keys_exact(bits)
    for i in range(bits.shape[0]):
        exact = sum((_bits_to_fraction(v & 0x7FFF) for v in bits[i]), Fraction(0))
        assert Fraction(keys[i]) * Fraction(2) ** (-133) == exact
    nf = bits.copy(); nf[2, 1] = 0x7F80
    assert muon.l1_keys_exact(nf)[2] == muon.NONFINITE_KEY


def test_top_k_ties_lowest_index():
    keys = [5, 9, 9, 1, 9, 7, 5]
    # brute force: every k-subset ranked lexicographically by (sum of key ranks), ties by index
    order = sorted(range(len(keys)), key=lambda i: (-keys[i], i))
    for k in range(1, len(keys) + 1):
        assert list(muon.top_k_rows(keys, k)) == sorted(order[:k])
    assert list(muon.top_k_rows(keys, 2)) == [1, 2]
    assert list(muon.top_k_rows(keys, 4)) == [1, 2, 4, 5]
    assert list(muon.top_k_rows(keys, 5)) == [0, 1, 2, 4, 5]


def test_duplicate_rows_select_lowest_index():
    row = inputs.round_to_bf16_bits(inputs.gaussian(14, (1, 32)))
    M = np.repeat(row, 6, axis=0)
    M[4] = inputs.round_to_bf16_bits(inputs.gaussian(15, (1, 32)) * 0.1)
    S = muon.top_k_rows(muon.l1_keys_exact(M), 3)
    assert list(S) == [0, 1, 2]


def test_muon_step_orientation_roundtrip_and_update():
    W = inputs.round_to_bf16_bits(inputs.gaussian(16, (48, 20), 0.1))
    G = inputs.round_to_bf16_bits(inputs.gaussian(17, (48, 20), 0.1))
    M = inputs.round_to_bf16_bits(inputs.gaussian(18, (48, 20), 0.1))
    W1, M1, O1 = muon.muon_step(W, G, M, lr=0.02, mu=0.95, weight_decay=0.1, scale=1.5)
    W2, M2, O2 = muon.muon_step(W.T.copy(), G.T.copy(), M.T.copy(), lr=0.02, mu=0.95, weight_decay=0.1, scale=1.5)
    assert rel(W1, W2.T) < 1e-12 and np.array_equal(M1, M2.T) and rel(O1, O2.T) < 1e-12
    # update formula written out directly
    Mn = muon.bf16_decode(M1)
    O = ns.gram_ns_stabilized(Mn.T, ns.QUINTIC_FIXED).T
    want = (1 - 0.02 * 0.1) * muon.bf16_decode(W) - 0.02 * 1.5 * O
    assert rel(W1, want) < 1e-12
    # and the orthogonalized factor is close to polar of the momentum (fixed quintic band)
    s = np.linalg.svd(O1, compute_uv=False)
    assert s.min() > 0.6 and s.max() < 1.2


def test_frac_full_fraction_equals_muon():
    """Dion3 sec. 6 'Finite Precision': f = 1 selects every row and reduces to Muon (with
    M = 0 the mu factor of footnote 4 does not enter); only M's decay differs."""
    W = inputs.round_to_bf16_bits(inputs.gaussian(19, (24, 64), 0.1))
    G = inputs.round_to_bf16_bits(inputs.gaussian(20, (24, 64), 0.1))
    M = np.zeros_like(G)
    Wf, Mf, S, O = muon.frac_step(W, G, M, 1.0, lr=0.02, mu=0.95)
    Wm, Mm, Om = muon.muon_step(W, G, M, lr=0.02, mu=0.95)
    assert list(S) == list(range(24))
    assert rel(Wf, Wm) < 1e-12
    assert np.array_equal(Mf, muon.decay_rows_bf16(G, np.arange(24), 0.95))


def test_frac_step_rows_and_error_feedback():
    W = inputs.round_to_bf16_bits(inputs.gaussian(21, (32, 96), 0.1))
    G = inputs.round_to_bf16_bits(inputs.gaussian(22, (32, 96), 0.1))
    M = inputs.round_to_bf16_bits(inputs.gaussian(23, (32, 96), 0.1))
    Wn, Mn, S, O = muon.frac_step(W, G, M, 0.25, lr=0.02, mu=0.95)
    assert len(S) == 8 and list(S) == sorted(S)
    Msum = muon.momentum_update_bf16(M, G, 1.0)
    l1 = np.abs(muon.bf16_decode(Msum)).sum(axis=1)
    assert set(S) == set(np.argsort(-l1, kind="stable")[:8])        # no ties in this draw
    unsel = np.setdiff1d(np.arange(32), S)
    assert np.array_equal(Mn[unsel], Msum[unsel])                    # untouched rows keep M + G
    assert np.array_equal(Wn[unsel], muon.bf16_decode(W)[unsel])
    assert rel(O, ns.gram_ns_stabilized(muon.bf16_decode(Msum[S]), ns.QUINTIC_FIXED)) < 1e-14
    # tall matrix: selection runs along the columns
    Wt, Mt, St, Ot = muon.frac_step(W.T.copy(), G.T.copy(), M.T.copy(), 0.25, lr=0.02, mu=0.95)
    assert list(St) == list(S) and rel(Wt, Wn.T) < 1e-12 and np.array_equal(Mt, Mn.T)
    assert math.ceil(0.25 * 4096) == 1024


def test_spectrum_trace_follows_the_polynomial_map_in_the_singular_basis():
    """Appendix B.1.1 eigen-tracking: in exact arithmetic every R_t and Q_t of Gram NS is
    diagonal in the basis U of X's left singular vectors, with R_t's eigenvalue along u_i
    equal to phi_t(s_i)^2 and Q_t's equal to phi_t(s_i) / s_i (Theorem 2: q_t x_0 is the
    composition of the first t polynomials; s_i the normalised singular values). Checked
    against the composition of the printed polynomials, and the off-diagonal fraction of
    U^T Q U (B.1.3's diagonalisation error) must be zero up to fp64 rounding; with R_0
    rounded through bf16 (B.1.2) it must not be."""
    X = inputs.exp_spectrum(3, 24, 96, decades=2.0)
    C = ns.QUINTIC_FIXED
    tr = []
    ns.gram_ns_naive(X, C, trace=tr)
    rows = st.spectrum_trace(X, tr)
    assert [r[0] for r in rows] == list(range(len(C) + 1))
    s = np.linalg.svd(X, compute_uv=False) / (np.linalg.norm(X) + ns.EPS)   # descending, as U's columns
    for (t, dr, dq, off) in rows:
        phi = ns.compose(s, C[:t])
        if t < len(C):          # R_T is not formed (sec. 4.1): the trace repeats R_{T-1}
            assert np.max(np.abs(dr - phi ** 2)) < 1e-11 * max(1.0, np.max(phi ** 2)), t
        assert np.max(np.abs(dq - phi / s)) < 1e-10 * np.max(np.abs(phi / s)), t
        assert off < 1e-12, (t, off)
    # a rounded R_0 leaves the basis: the off-diagonal fraction becomes visible
    trp = []
    with np.errstate(all="ignore"):
        ns.gram_ns_naive(X, C, trace=trp, gram_perturb=inputs.bf16_round)
    offs = [r[3] for r in st.spectrum_trace(X, trp)]
    assert offs[0] < 1e-12 and max(offs[1:]) > 1e-4   # Q_0 = I


@pytest.mark.parametrize("loc", [None, 1, 2, 3, 4])
def test_restart_sweep_matches_algorithm3_with_a_planted_eigenvalue(loc):
    """Appendix B.2.1's sweep on the scalar recurrence against the matrix algorithm: with
    X = U diag(x) V^T and -delta I planted into every Gram matrix Algorithm 3 forms (R_0
    and the restart's R), the eigenvalues of every Q_t are the scalar q_t of each direction,
    so the sweep's max_t cond(Q_t) and max_t max|q_t| must equal those of the matrix run."""
    delta = -GOLD["spurious_eigenvalue"]["value"]
    x = np.array([1.0, 0.8, 0.5, 0.2, 0.05, 0.01, 1e-3])
    n, m = len(x), 20
    g = np.random.default_rng(11)
    U, _ = np.linalg.qr(g.standard_normal((n, n)))
    V, _ = np.linalg.qr(g.standard_normal((m, n)))
    X = (U * x) @ V.T
    grid = x / (np.linalg.norm(x) + ns.EPS)   # singular values after the normalisation
    cond_s, _, qmax_s = st.restart_sweep(ns.QUINTIC_FIXED, delta=delta, grid=grid)[loc]
    tr = []
    ns.gram_ns_stabilized(X, ns.QUINTIC_FIXED, restarts=() if loc is None else (loc,), trace=tr,
                          gram_perturb=lambda R: R - delta * np.eye(R.shape[0]))
    qs = [np.linalg.eigvalsh(0.5 * (Q + Q.T)) for (t, R, Q) in tr if isinstance(t, int) and t >= 1]
    assert len(qs) == len(ns.QUINTIC_FIXED)
    cond_m = max(np.abs(q).max() / np.abs(q).min() for q in qs)
    qmax_m = max(np.abs(q).max() for q in qs)
    assert cond_s == pytest.approx(cond_m, rel=1e-8)
    assert qmax_s == pytest.approx(qmax_m, rel=1e-8)
