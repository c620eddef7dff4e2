"""gns_gram_ns_batched_noalloc: the entry point for callers that cannot allocate device
memory where they orthogonalize (a framework memory pool that forbids allocations it does
not own, a loop that must not allocate after start-up, a plug-in given pointers but no
allocator). It takes its scratch from a fixed array inside the library instead of a
caller workspace.

Checked through the C ABI against gns_gram_ns_batched (caller workspace) on two calls in a
row: both run the same deterministic kernels (fixed reduction orders), so the outputs must
be bit-identical, which also catches scratch the second call finds stale from the first.
The cases cover the layouts the array is carved into: wide and tall bf16 Gram groups, a
square group (standard Newton-Schulz plan), and two fp32 groups in one call (one launch
per product). This file is collected last on purpose, and passes both alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from util import bf16_input, bits_to_torch, empty_like_padded, padded_copy

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _ns_default(lib, _lib):
    p = _lib.GnsNsParams()
    lib.gns_ns_params_default(ctypes.byref(p))
    return p


def _f32_input(seed, shape):
    g = np.random.default_rng(seed)
    x = (g.standard_normal(shape) / np.sqrt(shape[-1])).astype(np.float32)
    return padded_copy(torch.from_numpy(x).cuda())


def _same_bits(a, b):
    ai = a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32)
    bi = b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32)
    return torch.equal(ai, bi)


def _cases():
    b1, _ = bf16_input(40, (3, 256, 1024))
    b2, _ = bf16_input(41, (2, 384, 200))
    b3, _ = bf16_input(42, (2, 256, 256))
    return [
        ("bf16 wide", "bf16", [bits_to_torch(b1)]),
        ("bf16 tall", "bf16", [bits_to_torch(b2)]),
        ("bf16 square (standard NS plan)", "bf16", [bits_to_torch(b3)]),
        ("fp32 two groups", "f32", [_f32_input(43, (2, 64, 256)), _f32_input(44, (3, 100, 48))]),
    ]


@pytest.mark.parametrize("which", range(4))
def test_noalloc_matches_workspace_entry_point_twice(which):
    import matrix_orthogonalizing_optimizer_gb300 as gns
    from matrix_orthogonalizing_optimizer_gb300 import _lib

    lib = _lib.load()
    ns = _ns_default(lib, _lib)
    stream = torch.cuda.current_stream().cuda_stream
    name, dt, xs = _cases()[which]
    code = _lib.GNS_BF16 if dt == "bf16" else _lib.GNS_F32
    ng = len(xs)
    xb = (_lib.GnsBatch * ng)(*[gns.batch_of(x) for x in xs])
    # reference: the entry point with a caller workspace
    refs = [empty_like_padded(x) for x in xs]
    rb = (_lib.GnsBatch * ng)(*[gns.batch_of(r) for r in refs])
    need = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, xb, ng, code, ctypes.byref(ns), None)
    assert 0 < need <= _lib.GNS_NOALLOC_SCRATCH_BYTES, name
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.gns_gram_ns_batched(xb, rb, ng, code, ctypes.byref(ns), ws.data_ptr(), need, st.data_ptr(), stream)
    assert rc == 0, _lib.last_error()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for call in range(2):
        outs = [empty_like_padded(x, fill=float("nan")) for x in xs]
        ob = (_lib.GnsBatch * ng)(*[gns.batch_of(o) for o in outs])
        rc = lib.gns_gram_ns_batched_noalloc(xb, ob, ng, code, ctypes.byref(ns), st.data_ptr(), stream)
        assert rc == 0, _lib.last_error()
        torch.cuda.synchronize()
        assert int(st.item()) == 0, (name, call)
        for o, r in zip(outs, refs):
            assert _same_bits(o, r), (name, call)


def test_noalloc_rejects_batches_above_the_fixed_scratch():
    import matrix_orthogonalizing_optimizer_gb300 as gns
    from matrix_orthogonalizing_optimizer_gb300 import _lib

    lib = _lib.load()
    ns = _ns_default(lib, _lib)
    x = torch.zeros((16, 1024, 4096), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    xb = (_lib.GnsBatch * 1)(gns.batch_of(x))
    ob = (_lib.GnsBatch * 1)(gns.batch_of(out))
    need = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, xb, 1, _lib.GNS_BF16, ctypes.byref(ns), None)
    assert need > _lib.GNS_NOALLOC_SCRATCH_BYTES
    rc = lib.gns_gram_ns_batched_noalloc(xb, ob, 1, _lib.GNS_BF16, ctypes.byref(ns), None,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.GNS_ERR_WORKSPACE
    assert "GNS_NOALLOC_SCRATCH_BYTES" in _lib.last_error()


def test_noalloc_returns_the_planners_status():
    """An unsupported request (rows not on 16-byte boundaries) returns GNS_ERR_UNSUPPORTED,
    as gns_gram_ns_batched does, not a generic argument error."""
    import matrix_orthogonalizing_optimizer_gb300 as gns
    from matrix_orthogonalizing_optimizer_gb300 import _lib

    lib = _lib.load()
    ns = _ns_default(lib, _lib)
    x = torch.zeros((2, 64, 100), dtype=torch.bfloat16, device="cuda")   # ld = 100 elements
    out = torch.zeros_like(x)
    xb = (_lib.GnsBatch * 1)(gns.batch_of(x))
    ob = (_lib.GnsBatch * 1)(gns.batch_of(out))
    rc = lib.gns_gram_ns_batched_noalloc(xb, ob, 1, _lib.GNS_BF16, ctypes.byref(ns), None,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.GNS_ERR_UNSUPPORTED and "16 bytes" in _lib.last_error()
