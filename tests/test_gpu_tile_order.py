"""The tile order of a persistent launch (waves of matrices and their skew, GNS_TILE_ORDER
"W,D") changes only when each output tile is computed, never how: every tile runs the same
deterministic arithmetic, so Gram Newton-Schulz and Muon-step results must be bit-identical
under every order, and every order must complete (each tile depends only on earlier tiles).
"""
import os

import pytest

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")

pytestmark = pytest.mark.gpu

ORDERS = ["1,0", "1,17", "3,5", "4,17", "8,0", "8,8", "5,2", "24,0"]


def _with_order(order, fn):
    old = os.environ.get("GNS_TILE_ORDER")
    os.environ["GNS_TILE_ORDER"] = order
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["GNS_TILE_ORDER"]
        else:
            os.environ["GNS_TILE_ORDER"] = old


def test_gram_ns_bit_identical_under_every_tile_order():
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    X = (torch.randn((10, 384, 1536), generator=g, device="cuda") / 1536 ** 0.5).to(torch.bfloat16)
    ref = _with_order("10,0", lambda: gns.gram_ns_batched(X)[0].clone())
    for order in ORDERS:
        out = _with_order(order, lambda: gns.gram_ns_batched(X)[0])
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), order


def test_muon_step_bit_identical_under_every_tile_order():
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    r = lambda: (torch.randn((12, 1024, 256), generator=g, device="cuda") / 16).to(torch.bfloat16)
    W0, G, M0 = r(), r(), r()

    def step():
        W, M = W0.clone(), M0.clone()
        gns.muon_step(W, G, M, lr=0.02, momentum=0.95, weight_decay=0.1)
        return W, M
    Wr, Mr = _with_order("12,0", step)
    for order in ORDERS:
        W, M = _with_order(order, step)
        assert torch.equal(W.view(torch.int16), Wr.view(torch.int16)), order
        assert torch.equal(M.view(torch.int16), Mr.view(torch.int16)), order
