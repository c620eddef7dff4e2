"""Full-size parity on the benchmark-scale configurations (GPU), with inputs generated on the
device by a seeded torch generator and sampled matrices copied to the host for the fp64
oracle. Matrices the oracle cannot afford at this size are checked through properties that
hold at any size:

  * X O^T is symmetric (O = U phi(S) V^T for X = U S V^T, so X O^T = U S phi(S) U^T), tested
    with random vectors: |u^T X O^T w - w^T X O^T u| within the bound a relative error of
    2e-2 in O allows;
  * ||O^T w|| / ||w|| lies in the band the fixed quintic maps singular values into.

Configurations (synthetic stand-ins for the pages' dense-transformer and MoE shapes):
  * 32 layers x {4096 x 4096, 2 x 4096 x 11008, 11008 x 4096}: full Muon step;
  * 256 x 2048 x 8192 experts (Student-t nu = 4, normalised) + 64 x 7168 x 7168: Gram NS and
    standard NS on the same kernels;
  * 32 x 4096 x 16384, f = 1/4: Dion3 fractional update, selection bit-exact.
"""
import numpy as np
import pytest

from oracle import muon as omuon
from oracle import newton_schulz as ons
from util import bf16_ulp, rel_fro, torch_to_bits, torch_to_f64

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _randn(g, shape, scale):
    return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * scale).to(torch.bfloat16)


def _student_t_normalised(g, shape):
    z = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32)
    chi2 = torch.zeros(shape, device="cuda", dtype=torch.float32)
    for _ in range(4):
        chi2 += torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) ** 2
    t = z / torch.sqrt(chi2 / 4)
    t /= torch.linalg.vector_norm(t, dim=(-2, -1), keepdim=True)
    return t.to(torch.bfloat16)


def _w_ok(W_gpu, W_or, dW_or):
    half_ulp = 0.5 * bf16_ulp(np.maximum(np.abs(W_or), np.abs(W_gpu)))
    excess = np.maximum(np.abs(W_gpu - W_or) - half_ulp, 0.0)
    return np.linalg.norm(excess) / np.linalg.norm(dW_or)


def _properties(X, O, seed, band=(0.5, 1.2)):
    """X, O float64 (n x m, same orientation)."""
    rng = np.random.default_rng(seed)
    n = X.shape[0] if X.shape[0] <= X.shape[1] else X.shape[1]
    if X.shape[0] > X.shape[1]:
        X, O = X.T, O.T
    fro = np.linalg.norm(O)
    for _ in range(3):
        u, w = rng.standard_normal(n), rng.standard_normal(n)
        xu, xw = X.T @ u, X.T @ w
        a = xu @ (O.T @ w)
        b = xw @ (O.T @ u)
        # if O = O* + E with ||E||_F <= eps ||O||_F and X O*^T symmetric, then
        # |a - b| <= eps ||O||_F (||X^T u|| ||w|| + ||X^T w|| ||u||)
        bound = TOL_BF16 * fro * (np.linalg.norm(xu) * np.linalg.norm(w) + np.linalg.norm(xw) * np.linalg.norm(u))
        assert abs(a - b) <= bound, (abs(a - b), bound)
        r = np.linalg.norm(O.T @ w) / np.linalg.norm(w)
        assert band[0] < r < band[1], r


def test_fullsize_dense_layers_muon_step():
    g = _gen(301)
    shapes = [(32, 4096, 4096), (64, 4096, 11008), (32, 11008, 4096)]
    W = [_randn(g, s, 1.0 / np.sqrt(s[2])) for s in shapes]
    G = [_randn(g, s, 1.0) for s in shapes]
    M = [_randn(g, s, 1.0) for s in shapes]
    W0 = [w[[0, -1]].clone() for w in W]
    G0 = [x[[0, -1]].clone() for x in G]
    M0 = [x[[0, -1]].clone() for x in M]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gns.muon_step(W, G, M, lr=0.02, momentum=0.95, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for gi, s in enumerate(shapes):
        b = 0  # the first matrix of each group against the oracle, the last through properties
        Wb, Gb, Mb = torch_to_bits(W0[gi][b]), torch_to_bits(G0[gi][b]), torch_to_bits(M0[gi][b])
        W_or, M_or, O = omuon.muon_step(Wb, Gb, Mb, lr=0.02, mu=0.95)
        if s[1] == s[2]:
            O = ons.ns_standard(omuon.bf16_decode(M_or), ons.QUINTIC_FIXED)
            W_or = omuon.bf16_decode(Wb) - 0.02 * O
        assert np.array_equal(torch_to_bits(M[gi][0]), M_or)
        err = _w_ok(torch_to_f64(W[gi][0]), W_or, 0.02 * O)
        assert err < TOL_BF16, (s, err)
        # the last matrix of the group: momentum bit-exact
        M_last = omuon.momentum_update_bf16(torch_to_bits(M0[gi][1]), torch_to_bits(G0[gi][1]), 0.95)
        assert np.array_equal(torch_to_bits(M[gi][-1]), M_last)


def test_fullsize_moe_experts_and_squares_gram_vs_standard():
    g = _gen(302)
    ex = _student_t_normalised(g, (256, 2048, 8192))
    sq = _student_t_normalised(g, (64, 7168, 7168))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_g = gns.gram_ns_batched([ex, sq], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out_s = gns.ns_standard_batched(ex, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in (0, 255):
        X = torch_to_f64(ex[b])
        want = omuon.orthogonalize(X)
        assert rel_fro(torch_to_f64(out_g[0][b]), want) < TOL_BF16
        assert rel_fro(torch_to_f64(out_s[b]), want) < TOL_BF16
    # Gram and standard NS agree on every expert (Theorem 2), on the GPU
    d = torch.linalg.vector_norm((out_g[0].float() - out_s.float()), dim=(-2, -1))
    n = torch.linalg.vector_norm(out_s.float(), dim=(-2, -1))
    assert float((d / n).max()) < 2 * TOL_BF16
    for b in (0, 63):
        _properties(torch_to_f64(sq[b]), torch_to_f64(out_g[1][b]), seed=10 + b)


@pytest.mark.parametrize("shape", [(32, 4096, 16384), (32, 16384, 4096)])
def test_fullsize_fractional_quarter(shape):
    """f = 1/4 at full size, wide (rows selected; the update in the last product's epilogue)
    and tall (columns selected; O written transposed for the column scatter)."""
    g = _gen(303)
    s = shape
    W = _randn(g, s, 1.0 / np.sqrt(s[2]))
    G = _randn(g, s, 1.0 / np.sqrt(s[2]))
    M = _randn(g, s, 1.0 / np.sqrt(s[2]))
    samples = (0, 31)
    W0, G0, M0 = (torch_to_bits(x[list(samples)]) for x in (W, G, M))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gns.muon_step(W, G, M, lr=0.02, momentum=0.95, frac=0.25, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, b in enumerate(samples):
        W_or, M_or, S, O = omuon.frac_step(W0[i], G0[i], M0[i], 0.25, lr=0.02, mu=0.95)
        assert len(S) == 1024
        assert np.array_equal(torch_to_bits(M[b]), M_or), "selection and error feedback bit-exact"
        dW = np.zeros_like(W_or)
        if s[1] <= s[2]:
            dW[S] = 0.02 * O
        else:
            dW[:, S] = 0.02 * O.T
        assert _w_ok(torch_to_f64(W[b]), W_or, dW) < TOL_BF16
