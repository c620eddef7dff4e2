"""gns_gram_ns_batched_noalloc: the entry point for callers that cannot allocate device
memory where they orthogonalize (a framework memory pool that forbids allocations it does
not own, a loop that must not allocate after start-up, a plug-in given pointers but no
allocator). It takes its scratch from a fixed array inside the library instead of a
caller workspace.

Checked through the C ABI against gns_gram_ns_batched (caller workspace) on two calls in a
row, within the bf16 tolerance of the other parity tests; the second call finds the array
as the first left it. This file is collected last on purpose, and passes both alone in a
fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from util import bf16_input, bits_to_torch, empty_like_padded, rel_fro, torch_to_f64

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _ns_default(lib, _lib):
    p = _lib.GnsNsParams()
    lib.gns_ns_params_default(ctypes.byref(p))
    return p


def test_noalloc_matches_workspace_entry_point_twice():
    import matrix_orthogonalizing_optimizer_gb300 as gns
    from matrix_orthogonalizing_optimizer_gb300 import _lib

    lib = _lib.load()
    ns = _ns_default(lib, _lib)
    stream = torch.cuda.current_stream().cuda_stream
    for seed, (count, rows, cols) in [(40, (3, 256, 1024)), (41, (2, 384, 200))]:
        bits, _ = bf16_input(seed, (count, rows, cols))
        xt = bits_to_torch(bits)
        xb = (_lib.GnsBatch * 1)(gns.batch_of(xt))
        # reference: the entry point with a caller workspace
        ref = empty_like_padded(xt)
        rb = (_lib.GnsBatch * 1)(gns.batch_of(ref))
        need = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, xb, 1, _lib.GNS_BF16, ctypes.byref(ns), None)
        assert 0 < need <= _lib.GNS_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        rc = lib.gns_gram_ns_batched(xb, rb, 1, _lib.GNS_BF16, ctypes.byref(ns), ws.data_ptr(), need, None, stream)
        assert rc == 0, _lib.last_error()
        torch.cuda.synchronize()
        want = torch_to_f64(ref)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        for call in range(2):
            out = empty_like_padded(xt, fill=float("nan"))
            ob = (_lib.GnsBatch * 1)(gns.batch_of(out))
            rc = lib.gns_gram_ns_batched_noalloc(xb, ob, 1, _lib.GNS_BF16, ctypes.byref(ns), st.data_ptr(), stream)
            assert rc == 0, _lib.last_error()
            torch.cuda.synchronize()
            got = torch_to_f64(out)
            assert int(st.item()) == 0
            for b in range(count):
                assert np.all(np.isfinite(got[b]))
                assert rel_fro(got[b], want[b]) < TOL_BF16, (call, b)


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
