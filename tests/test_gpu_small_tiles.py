"""The 1-CTA 128 x 128 tile plan (chosen for products of at most 128 rows) against the fp64
oracle, and against the 2-CTA 256 x 256 plan on the same inputs: GNS_CTA_GROUP forces either
plan for any size, so both are checked on shapes whose tile grids differ (ragged edges, the
upper-triangle storage of internal symmetric buffers read across 128-blocks, diagonal
tiles with the a_t I patch, mirrored stores). Also the small-matrix shapes of the many-small-
matrices regime at their full batch sizes, sampled."""
import os

import numpy as np
import pytest

from oracle import muon as omuon
from util import bf16_input, bits_to_torch, empty_like_padded, rel_fro, torch_to_bits, torch_to_f64

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_PRODUCT = 1e-2


def _with_env(env, fn):
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return fn()
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _with_group(g, fn):
    # the tile plans themselves: groups the on-chip chain kernel would take stay on the
    # batched tile path here
    return _with_env({"GNS_CTA_GROUP": str(g), "GNS_CHAIN_SMALL": "0"}, fn)


@pytest.mark.parametrize("count,n,K", [(3, 128, 512), (2, 100, 72), (2, 200, 328), (1, 384, 256), (4, 8, 24)])
def test_sym_gemm_xxt_both_plans(count, n, K):
    bits, x = bf16_input(70, (count, n, K), 1.0 / np.sqrt(K))
    xt = bits_to_torch(bits)
    for g in (1, 2):
        c = empty_like_padded(torch.empty((count, n, n), dtype=torch.bfloat16, device="cuda"), fill=float("nan"))
        _with_group(g, lambda: gns.sym_gemm_xxt(xt, c, alpha=1.5))
        torch.cuda.synchronize()
        got = torch_to_f64(c)
        for b in range(count):
            assert rel_fro(got[b], 1.5 * x[b] @ x[b].T) < TOL_PRODUCT, (g, b)
        cb = torch_to_bits(c)
        assert np.array_equal(cb, np.swapaxes(cb, 1, 2)), g


@pytest.mark.parametrize("count,rows,cols", [(5, 128, 512), (3, 96, 2000), (2, 200, 800), (2, 384, 1024),
                                            (3, 512, 128), (2, 1, 40), (3, 136, 136)])
def test_gram_ns_both_plans(count, rows, cols):
    bits, x = bf16_input(71, (count, rows, cols))
    xt = bits_to_torch(bits)
    want = [omuon.orthogonalize(x[b]) for b in range(count)]
    for g in (1, 2):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = _with_group(g, lambda: gns.gram_ns_batched(xt, status=st)[0])
        torch.cuda.synchronize()
        assert int(st.item()) == 0, g
        got = torch_to_f64(out)
        tol = 4e-2 if min(rows, cols) == 1 else TOL_BF16
        for b in range(count):
            assert rel_fro(got[b], want[b]) < tol, (g, b)


def test_muon_step_small_matrices_plan1():
    """Full Muon step (momentum, Gram NS, update in the last epilogue) on 128 x 512 matrices
    on the 1-CTA tile plan (the chain kernel turned off)."""
    count, rows, cols = 16, 128, 512
    s = 1.0 / np.sqrt(cols)
    Wb, _ = bf16_input(72, (count, rows, cols), s, stream=0)
    Gb, _ = bf16_input(72, (count, rows, cols), s, stream=1)
    Mb, _ = bf16_input(72, (count, rows, cols), s, stream=2)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    _with_env({"GNS_CHAIN_SMALL": "0"}, lambda: gns.muon_step(Wt, Gt, Mt, lr=0.02, momentum=0.95))
    torch.cuda.synchronize()
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(count):
        W_or, M_or, O = omuon.muon_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95)
        assert np.array_equal(Mg[b], M_or)
        dW = Wg[b] - W_or
        mag = np.maximum(np.maximum(np.abs(Wg[b]), np.abs(W_or)), 2.0 ** -126)
        excess = np.maximum(np.abs(dW) - 0.5 * 2.0 ** (np.floor(np.log2(mag)) - 7), 0.0)
        assert np.linalg.norm(excess) / np.linalg.norm(0.02 * O) < TOL_BF16, b


@pytest.mark.parametrize("count,rows,cols", [(2048, 128, 512), (512, 256, 1024), (96, 512, 2048)])
def test_small_matrix_batches_full_size_sampled(count, rows, cols):
    """The many-small-matrices shapes at their full batch sizes: Gram and standard NS of the
    whole batch in one call each; every matrix finite, sampled matrices against the oracle."""
    g = torch.Generator(device="cuda")
    g.manual_seed(73)
    X = (torch.randn((count, rows, cols), generator=g, device="cuda") / cols ** 0.5).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gns.gram_ns_batched(X, status=st)[0]
    outs = gns.ns_standard_batched(X, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in sorted({0, 1, count // 2, count - 1}):
        want = omuon.orthogonalize(torch_to_f64(X[b]))
        assert rel_fro(torch_to_f64(out[b]), want) < TOL_BF16, b
        assert rel_fro(torch_to_f64(outs[b]), want) < TOL_BF16, b
