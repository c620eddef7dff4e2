"""Stream capture: the library's calls enqueue only stream-ordered work (kernels with cluster
launches, memsets), so a step captured into a CUDA graph and replayed must give the same bits
as the same calls run eagerly from the same state. Every kernel of the path is deterministic
(fixed reduction orders, exact integer keys), which makes bit equality the right test."""
import pytest

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")
from matrix_orthogonalizing_optimizer_gb300 import _lib  # noqa: E402

pytestmark = pytest.mark.gpu

STEPS = 3


def _tensors(seed, count, rows, cols):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    r = lambda: (torch.randn((count, rows, cols), generator=g, device="cuda") / cols ** 0.5).to(torch.bfloat16)
    return r(), r(), r()


def _params(kind):
    if kind == "muon":
        return gns.MuonParams(lr=0.02, weight_decay=0.1)
    if kind == "frac":
        return gns.MuonParams(lr=0.02, frac=0.25)
    if kind == "normuon":
        return gns.MuonParams(lr=0.02, flavor="normuon")
    if kind == "fp16":
        return gns.MuonParams(lr=0.02, ns_dtype=torch.float16)
    if kind == "rownorm":
        return gns.MuonParams(lr=0.02, flavor="rownorm")
    raise ValueError(kind)


@pytest.mark.parametrize("kind,count,rows,cols", [("muon", 6, 512, 2048), ("frac", 6, 512, 2048),
                                                  ("normuon", 4, 512, 1024), ("fp16", 4, 512, 1024),
                                                  ("rownorm", 4, 384, 1024), ("frac", 4, 1024, 384),
                                                  ("muon", 4, 1024, 384)])
def test_captured_muon_step_matches_eager(kind, count, rows, cols):
    W0, G, M0 = _tensors(11, count, rows, cols)
    p = _params(kind)
    n = min(rows, cols)
    V0 = torch.zeros((count, 1, n), dtype=torch.float32, device="cuda") if kind == "normuon" else None
    ws = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_MUON_STEP, M0, muon=p), "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # eager reference
    We, Me = W0.clone(), M0.clone()
    Ve = V0.clone() if V0 is not None else None
    for _ in range(STEPS):
        gns.muon_step(We, G, Me, V=Ve, params=p, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    # captured: a first eager call on scratch state has already run above (device set-up),
    # so the capture sees only stream-ordered work
    Wg, Mg = W0.clone(), M0.clone()
    Vg = V0.clone() if V0 is not None else None
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gns.muon_step(Wg, G, Mg, V=Vg, params=p, workspace=ws, status=status)
    torch.cuda.synchronize()
    # capturing enqueues nothing: the state is still the initial one
    assert torch.equal(Wg.view(torch.int16), W0.view(torch.int16))
    for _ in range(STEPS):
        graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(Mg.view(torch.int16), Me.view(torch.int16))
    assert torch.equal(Wg.view(torch.int16), We.view(torch.int16))
    if Vg is not None:
        assert torch.equal(Vg, Ve)


def test_captured_gram_ns_matches_eager():
    X, _, _ = _tensors(12, 8, 768, 3072)
    ns = gns.NsParams()
    ws = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_GRAM_NS, X, ns), "cuda")
    out_e = torch.empty_like(X)
    gns.gram_ns_batched(X, outs=[out_e], ns=ns, workspace=ws)
    out_g = torch.zeros_like(X)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gns.gram_ns_batched(X, outs=[out_g], ns=ns, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
