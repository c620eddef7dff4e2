"""GPU parity of the widened rows: fp16 Newton-Schulz products, the safety factor, NorMuon,
RowNorm and Periodic Row-wise Muon, each against the CPU fp64 oracle on seeded inputs.

Tolerances (relative Frobenius error unless stated):
  * fp16 Newton-Schulz output: 5e-3. fp16 keeps 11 significant bits against bf16's 8, so
    every rounding of a stored R, Z, Q or X is 8x smaller (unit roundoff 2^-11 against
    2^-8); the bf16 bound of 2e-2 scaled by 1/8 is 2.5e-3, doubled for margin;
  * single fp16 products: 2e-3 (one fp16 rounding of the output, 2^-11 relative, plus fp32
    accumulation);
  * NorMuon weights: the update-relative measure of the Muon tests (2e-2), NorMuon's second
    moments 4e-2 (squares of a 2e-2-accurate O, plus bf16 storage of O);
  * RowNorm weights: 1e-3 (no Newton-Schulz: fp32 row norms and one bf16 rounding of W,
    against the fp64 oracle);
  * momentum, selection and error feedback: bit-exact, as in the Muon tests.
"""
import numpy as np
import pytest

from oracle import flavors as ofl
from oracle import muon as omuon
from oracle import newton_schulz as ons
from util import bf16_input, bf16_ulp, bits_to_torch, empty_like_padded, f16_input, f16_to_torch, rel_fro, \
    torch_to_bits, torch_to_f64

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F16 = 5e-3
TOL_F16_PRODUCT = 2e-3
TOL_V = 4e-2
TOL_ROWNORM = 1e-3


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _oracle_orth(X, coeffs=ons.QUINTIC_FIXED):
    """Algorithm 3, or Algorithm 1 for a square matrix (the library's alpha = 1 rule)."""
    if X.shape[0] == X.shape[1]:
        return ons.ns_standard(X, coeffs)
    return omuon.orthogonalize(X, coeffs)


def _w_excess(W_gpu, W_or, dW_or):
    """Frobenius norm of |W_gpu - W_or| beyond half a bf16 ulp, relative to the update."""
    half_ulp = 0.5 * bf16_ulp(np.maximum(np.abs(W_or), np.abs(W_gpu)))
    excess = np.maximum(np.abs(W_gpu - W_or) - half_ulp, 0.0)
    return np.linalg.norm(excess) / max(np.linalg.norm(dW_or), 1e-300)


# ---------------------------------------------------------------------------------------
# fp16 products (the float16 cast of Dion3 Algorithm 3, appendix B.2.2)

@pytest.mark.parametrize("count,rows,cols", [(2, 128, 512), (3, 100, 300), (1, 300, 100), (2, 256, 256),
                                             (1, 257, 1000)])
def test_gram_ns_f16(count, rows, cols):
    x16, x = f16_input(31, (count, rows, cols), 1.0 / np.sqrt(cols))
    st = _status()
    out = gns.gram_ns_batched(f16_to_torch(x16), status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and out.dtype == torch.float16
    got = torch_to_f64(out)
    for b in range(count):
        e = rel_fro(got[b], _oracle_orth(x[b]))
        assert e < TOL_F16, e


@pytest.mark.parametrize("count,rows,cols", [(2, 128, 384), (1, 200, 136)])
def test_ns_standard_f16(count, rows, cols):
    x16, x = f16_input(32, (count, rows, cols), 1.0 / np.sqrt(cols))
    out = gns.ns_standard_batched(f16_to_torch(x16))[0]
    torch.cuda.synchronize()
    got = torch_to_f64(out)
    for b in range(count):
        e = rel_fro(got[b], ons.ns_standard(x[b], ons.QUINTIC_FIXED))
        assert e < TOL_F16, e


@pytest.mark.parametrize("count,n,K", [(2, 200, 320), (1, 384, 512)])
def test_sym_gemm_xxt_f16(count, n, K):
    x16, x = f16_input(33, (count, n, K), 1.0 / np.sqrt(K))
    c = empty_like_padded(torch.empty((count, n, n), dtype=torch.float16, device="cuda"), fill=float("nan"))
    gns.sym_gemm_xxt(f16_to_torch(x16), c, alpha=1.5)
    torch.cuda.synchronize()
    got = torch_to_f64(c)
    for b in range(count):
        assert rel_fro(got[b], 1.5 * x[b] @ x[b].T) < TOL_F16_PRODUCT


def test_sym_poly_update_f16_matches_bf16_structure():
    """One Algorithm 3 iteration on fp16 buffers against the same iteration in fp64."""
    n = 192
    x16, x = f16_input(34, (1, n, 3 * n), 1.0 / np.sqrt(3 * n))
    X = x[0] / np.linalg.norm(x[0])
    R0 = X @ X.T
    R = f16_to_torch(R0.astype(np.float16)[None])
    Q = empty_like_padded(torch.empty((1, n, n), dtype=torch.float16, device="cuda"))
    Z = empty_like_padded(torch.empty((1, n, n), dtype=torch.float16, device="cuda"))
    RZ = empty_like_padded(torch.empty((1, n, n), dtype=torch.float16, device="cuda"))
    a, b, c = ons.QUINTIC_FIXED[0]
    gns.sym_poly_update(R, Q, Z, RZ, None, a, b, c, q_is_identity=True, skip_r=False)
    torch.cuda.synchronize()
    Rf = R0.astype(np.float16).astype(np.float64)
    Zw = b * Rf + c * Rf @ Rf
    assert rel_fro(torch_to_f64(Z)[0], Zw) < TOL_F16_PRODUCT
    assert rel_fro(torch_to_f64(Q)[0], Zw + a * np.eye(n)) < TOL_F16_PRODUCT
    RZw = Rf @ Zw + a * Rf
    assert rel_fro(torch_to_f64(R)[0], Zw @ RZw + a * RZw) < 4 * TOL_F16_PRODUCT


# ---------------------------------------------------------------------------------------
# safety factor (Dion3 appendix B.2.2)

@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_safety_factor_runs_the_adjusted_table(dtype):
    count, rows, cols = 2, 128, 512
    if dtype == "bf16":
        bits, x = bf16_input(35, (count, rows, cols), 1.0 / np.sqrt(cols))
        xt = bits_to_torch(bits)
        tol = TOL_BF16
    else:
        x16, x = f16_input(35, (count, rows, cols), 1.0 / np.sqrt(cols))
        xt = f16_to_torch(x16)
        tol = TOL_F16
    out = gns.gram_ns_batched(xt, ns=gns.NsParams(safety=1.05))[0]
    torch.cuda.synchronize()
    got = torch_to_f64(out)
    adj = ofl.safety_adjust(ons.QUINTIC_FIXED, 1.05)
    for b in range(count):
        want = omuon.orthogonalize(x[b], adj)
        assert rel_fro(got[b], want) < tol
        # the unadjusted table gives a different result (about 20% away on this input)
        assert rel_fro(got[b], omuon.orthogonalize(x[b])) > 5 * tol


# ---------------------------------------------------------------------------------------
# Muon step with fp16 Newton-Schulz

# (1, 2048, 8192): tiles of 32 to 128 K slices, the GEMM's shallow shared-memory plan
@pytest.mark.parametrize("count,rows,cols,frac", [(2, 256, 1024, 1.0), (2, 384, 384, 1.0), (2, 700, 200, 1.0),
                                                  (2, 256, 1024, 0.25), (1, 2048, 8192, 1.0)])
def test_muon_step_f16_products(count, rows, cols, frac):
    Wb, W = bf16_input(36, (count, rows, cols), 1.0 / np.sqrt(cols))
    Gb, _ = bf16_input(37, (count, rows, cols), 1.0 / np.sqrt(cols))
    Mb, _ = bf16_input(38, (count, rows, cols), 1.0 / np.sqrt(cols))
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    st = _status()
    p = gns.MuonParams(lr=0.02, momentum=0.95, weight_decay=0.1, scale=1.5, frac=frac, ns_dtype=torch.float16)
    gns.muon_step(Wt, Gt, Mt, params=p, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(count):
        if frac == 1.0:
            M_or = omuon.momentum_update_bf16(Mb[b], Gb[b], 0.95)
            O = _oracle_orth(omuon.bf16_decode(M_or))
            W_or = (1 - 0.02 * 0.1) * W[b] - 0.02 * 1.5 * O
            dW = 0.02 * 1.5 * O
        else:
            W_or, M_or, S, O = omuon.frac_step(Wb[b], Gb[b], Mb[b], frac, lr=0.02, mu=0.95, weight_decay=0.1,
                                               scale=1.5)
            dW = np.zeros_like(W_or)
            dW[S] = 0.02 * 1.5 * O
        assert np.array_equal(Mg[b], M_or)
        e = _w_excess(Wg[b], W_or, dW)
        assert e < TOL_F16, e


# ---------------------------------------------------------------------------------------
# NorMuon (Dion3 eq. (2), the NorMuon steps of Algorithm 4)

def _v0(count, n, seed):
    g = np.random.default_rng(seed)
    return (g.uniform(0.5, 1.5, size=(count, 1, n)) / 1024.0).astype(np.float32)


@pytest.mark.parametrize("count,rows,cols,ns_dtype", [(2, 128, 512, "bf16"), (1, 384, 128, "bf16"),
                                                      (2, 256, 256, "bf16"), (2, 128, 512, "f16"),
                                                      (1, 2048, 8192, "bf16"), (1, 8192, 2048, "f16")])
def test_normuon_dense(count, rows, cols, ns_dtype):
    Wb, W = bf16_input(40, (count, rows, cols), 1.0 / np.sqrt(cols))
    Gb, _ = bf16_input(41, (count, rows, cols), 1.0 / np.sqrt(cols))
    Mb, _ = bf16_input(42, (count, rows, cols), 1.0 / np.sqrt(cols))
    n = min(rows, cols)
    v0 = _v0(count, n, 43)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    Vt = torch.from_numpy(v0).cuda()
    st = _status()
    p = gns.MuonParams(lr=0.02, momentum=0.95, weight_decay=0.1, scale=1.5, flavor="normuon", beta2=0.95,
                       norm_eps=1e-8, ns_dtype=torch.float16 if ns_dtype == "f16" else torch.bfloat16)
    gns.muon_step(Wt, Gt, Mt, V=Vt, params=p, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Mg, Wg, Vg = torch_to_bits(Mt), torch_to_f64(Wt), Vt.double().cpu().numpy()
    for b in range(count):
        M_or = omuon.momentum_update_bf16(Mb[b], Gb[b], 0.95)
        X, tr = omuon.orient(omuon.bf16_decode(M_or))
        O = _oracle_orth(X)
        D, v_or = ofl.normuon(O, v0[b, 0].astype(np.float64), 0.95, 1e-8)
        W_or = (1 - 0.02 * 0.1) * W[b] - 0.02 * 1.5 * (D.T if tr else D)
        assert np.array_equal(Mg[b], M_or)
        e = _w_excess(Wg[b], W_or, 0.02 * 1.5 * D)
        assert e < TOL_BF16, e
        assert rel_fro(Vg[b, 0], v_or) < TOL_V


@pytest.mark.parametrize("count,rows,cols,frac", [(2, 256, 1024, 0.25), (2, 640, 192, 0.25)])
def test_normuon_fractional(count, rows, cols, frac):
    Wb, W = bf16_input(44, (count, rows, cols), 1.0 / np.sqrt(cols))
    Gb, _ = bf16_input(45, (count, rows, cols), 1.0 / np.sqrt(cols))
    Mb, _ = bf16_input(46, (count, rows, cols), 1.0 / np.sqrt(cols))
    n = min(rows, cols)
    v0 = _v0(count, n, 47)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    Vt = torch.from_numpy(v0).cuda()
    p = gns.MuonParams(lr=0.02, momentum=0.95, frac=frac, flavor="normuon", beta2=0.9, norm_eps=1e-8)
    gns.muon_step(Wt, Gt, Mt, V=Vt, params=p)
    torch.cuda.synchronize()
    Mg, Wg, Vg = torch_to_bits(Mt), torch_to_f64(Wt), Vt.double().cpu().numpy()
    for b in range(count):
        W_or, M_or, v_or, S, D = ofl.normuon_frac_step(Wb[b], Gb[b], Mb[b], v0[b, 0].astype(np.float64), frac,
                                                       lr=0.02, mu=0.95, beta2=0.9, eps=1e-8)
        assert np.array_equal(Mg[b], M_or), "selection and error feedback must match bit for bit"
        unsel = np.setdiff1d(np.arange(n), S)
        assert np.array_equal(Vg[b, 0][unsel], v0[b, 0][unsel].astype(np.float64))
        assert rel_fro(Vg[b, 0][S], v_or[S]) < TOL_V
        dW = np.zeros((n, max(rows, cols)))
        dW[S] = 0.02 * D
        e = _w_excess(Wg[b], W_or, dW.T if rows > cols else dW)
        assert e < TOL_BF16, e


# ---------------------------------------------------------------------------------------
# RowNorm and Periodic Row-wise Muon (Scaling Muon for DiTs eq. (5), (7))

@pytest.mark.parametrize("count,rows,cols", [(2, 128, 512), (2, 640, 192), (3, 100, 100)])
def test_rownorm_step(count, rows, cols):
    Wb, W = bf16_input(50, (count, rows, cols), 1.0 / np.sqrt(cols))
    Gb, _ = bf16_input(51, (count, rows, cols), 1.0 / np.sqrt(cols))
    Mb, _ = bf16_input(52, (count, rows, cols), 1.0 / np.sqrt(cols))
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    p = gns.MuonParams(lr=0.02, momentum=0.95, weight_decay=0.1, scale=1.5, flavor="rownorm", rownorm_gamma=0.15,
                       norm_eps=1e-8)
    gns.muon_step(Wt, Gt, Mt, params=p)
    torch.cuda.synchronize()
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(count):
        W_or, M_or, D = ofl.rownorm_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95, gamma=0.15, eps=1e-8,
                                         weight_decay=0.1, scale=1.5)
        assert np.array_equal(Mg[b], M_or)
        tr = rows > cols
        e = _w_excess(Wg[b], W_or, 0.02 * 1.5 * (D.T if tr else D))
        assert e < TOL_ROWNORM, e


def test_periodic_takes_newton_schulz_on_refresh_steps_only():
    count, rows, cols = 2, 128, 512
    Wb, _ = bf16_input(53, (count, rows, cols), 1.0 / np.sqrt(cols))
    Gb, _ = bf16_input(54, (count, rows, cols), 1.0 / np.sqrt(cols))
    Mb, _ = bf16_input(55, (count, rows, cols), 1.0 / np.sqrt(cols))

    def run(**kw):
        Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
        gns.muon_step(Wt, Gt, Mt, params=gns.MuonParams(lr=0.02, momentum=0.95, **kw))
        torch.cuda.synchronize()
        return torch_to_bits(Wt), torch_to_bits(Mt)

    muon_w, muon_m = run(flavor="muon")
    rn_w, rn_m = run(flavor="rownorm", rownorm_gamma=0.15, norm_eps=1e-8)
    for t in range(5):
        w, m = run(flavor="periodic", period=3, step=t, rownorm_gamma=0.15, norm_eps=1e-8)
        want = (muon_w, muon_m) if ofl.refresh(t, 3) else (rn_w, rn_m)
        assert np.array_equal(w, want[0]) and np.array_equal(m, want[1]), t
    assert not np.array_equal(muon_w, rn_w)


# ---------------------------------------------------------------------------------------
# the benchmark's workload (24 x 1024 x 4096 bf16, the configuration bench.py times for each
# flavour), checked on sampled matrices of the batch

FULL = (24, 1024, 4096)
SAMPLES = (0, 11, 23)


def _full_inputs(seed):
    from matrix_orthogonalizing_optimizer_gb300 import inputs
    count, rows, cols = FULL
    s = 1.0 / np.sqrt(cols)
    W = inputs.round_to_bf16_bits(inputs.gaussian(seed, FULL, s, stream=0))
    G = inputs.round_to_bf16_bits(inputs.gaussian(seed, FULL, s, stream=1))
    M = inputs.round_to_bf16_bits(inputs.gaussian(seed, FULL, s, stream=2))
    return W, G, M


def test_full_size_f16_products():
    Wb, Gb, Mb = _full_inputs(200)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    st = _status()
    gns.muon_step(Wt, Gt, Mt, params=gns.MuonParams(lr=0.02, momentum=0.95, ns_dtype=torch.float16), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in SAMPLES:
        W_or, M_or, O = omuon.muon_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95)
        assert np.array_equal(Mg[b], M_or)
        e = _w_excess(Wg[b], W_or, 0.02 * O)
        assert e < TOL_F16, (b, e)


def test_full_size_normuon():
    Wb, Gb, Mb = _full_inputs(201)
    v0 = _v0(FULL[0], FULL[1], 202)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    Vt = torch.from_numpy(v0).cuda()
    gns.muon_step(Wt, Gt, Mt, V=Vt, params=gns.MuonParams(lr=0.02, momentum=0.95, flavor="normuon", beta2=0.95,
                                                          norm_eps=1e-8))
    torch.cuda.synchronize()
    Mg, Wg, Vg = torch_to_bits(Mt), torch_to_f64(Wt), Vt.double().cpu().numpy()
    for b in SAMPLES:
        W_or, M_or, v_or, D = ofl.normuon_step(Wb[b], Gb[b], Mb[b], v0[b, 0].astype(np.float64), lr=0.02, mu=0.95,
                                               beta2=0.95, eps=1e-8)
        assert np.array_equal(Mg[b], M_or)
        assert _w_excess(Wg[b], W_or, 0.02 * D) < TOL_BF16
        assert rel_fro(Vg[b, 0], v_or) < TOL_V


def test_full_size_rownorm_every_matrix():
    Wb, Gb, Mb = _full_inputs(203)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    gns.muon_step(Wt, Gt, Mt, params=gns.MuonParams(lr=0.02, momentum=0.95, flavor="rownorm", rownorm_gamma=0.15,
                                                    norm_eps=1e-8))
    torch.cuda.synchronize()
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(FULL[0]):
        W_or, M_or, D = ofl.rownorm_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95, gamma=0.15, eps=1e-8)
        assert np.array_equal(Mg[b], M_or)
        assert _w_excess(Wg[b], W_or, 0.02 * D) < TOL_ROWNORM, b
