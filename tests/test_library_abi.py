"""The C-ABI library builds, loads and exports every symbol include/gns.h declares; host-side
argument validation and workspace sizing (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

from matrix_orthogonalizing_optimizer_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gns.h")).read()
    return sorted(set(re.findall(r"GNS_API\s+[\w\s\*]+?\b(gns_\w+)\s*\(", src)))


def test_exports_match_header(lib):
    decl = declared_symbols()
    assert len(decl) >= 12
    assert sorted(_lib.EXPORTS) == decl
    for name in decl:
        assert hasattr(lib, name), name


def test_defaults_and_strings(lib):
    assert lib.gns_version() == 1
    p = _lib.GnsNsParams()
    lib.gns_ns_params_default(ctypes.byref(p))
    assert p.T == 5 and p.restart_mask == 4
    assert [round(v, 4) for v in (p.a[0], p.b[0], p.c[0])] == [3.4445, -4.775, 2.0315]
    assert abs(p.eps - 1e-7) < 1e-12
    assert lib.gns_status_string(-3) == b"GNS_ERR_WORKSPACE"


def _batch(count, rows, cols, ld=None, stride=None, ptr=1 << 20):
    b = (_lib.GnsBatch * 1)()
    b[0].ptr = ptr
    b[0].count, b[0].rows, b[0].cols = count, rows, cols
    b[0].ld = cols if ld is None else ld
    b[0].stride = rows * b[0].ld if stride is None else stride
    return b


def _ns(**kw):
    p = _lib.GnsNsParams()
    _lib.load().gns_ns_params_default(ctypes.byref(p))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_workspace_sizes(lib):
    p = _ns()
    # Gram NS of 24 x 1024 x 4096: R, Z, RZ, Q, Q' (5 n^2) and one restart buffer (n m), bf16
    b = _batch(24, 1024, 4096)
    n = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, b, 1, _lib.GNS_BF16, ctypes.byref(p), None)
    expect = 24 * (5 * 1024 * 1024 + 1024 * 4096) * 2
    assert expect <= n <= expect + 1 << 20
    # the fp32 path needs twice that
    n32 = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, b, 1, _lib.GNS_F32, ctypes.byref(p), None)
    assert abs(n32 - 2 * n) < 1 << 20
    # no restart: no restart buffer
    n0 = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, b, 1, _lib.GNS_BF16, ctypes.byref(_ns(restart_mask=0)), None)
    assert n - n0 >= 24 * 1024 * 4096 * 2
    # square groups take standard NS: A, B (n^2) and two X buffers
    sq = _batch(2, 512, 512)
    ns_ = lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, sq, 1, _lib.GNS_BF16, ctypes.byref(p), None)
    assert ns_ >= 2 * 4 * 512 * 512 * 2
    # fractional update works on k = ceil(f n) rows
    mp = _lib.GnsMuonParams(0.02, 0.95, 0.0, 1.0, 0.25)
    big = _batch(32, 4096, 16384)
    nf = lib.gns_workspace_size(_lib.GNS_OP_MUON_STEP, big, 1, _lib.GNS_BF16, ctypes.byref(p), ctypes.byref(mp))
    dense = lib.gns_workspace_size(_lib.GNS_OP_MUON_STEP, big, 1, _lib.GNS_BF16, ctypes.byref(p),
                                   ctypes.byref(_lib.GnsMuonParams(0.02, 0.95, 0.0, 1.0, 1.0)))
    assert 0 < nf < dense


@pytest.mark.parametrize("kw,msg", [
    (dict(ld=100, cols=96), b"16 bytes"),
    (dict(ld=50, cols=64), b"ld < cols"),
    (dict(ptr=(1 << 20) + 8), b"aligned"),
    (dict(rows=0), b">= 1"),
    (dict(count=2, stride=100 * 64), b"stride"),
    (dict(count=65536, stride=100 * 128), b"too large"),
    (dict(rows=65536, cols=65536, ld=65536), b"too large"),
    (dict(rows=8, cols=65535 * 64 + 8, ld=65535 * 64 + 8), b"too large"),
])
def test_invalid_batches(lib, kw, msg):
    args = dict(count=1, rows=100, cols=128)
    args.update(kw)
    b = _batch(**args)
    assert lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, b, 1, _lib.GNS_BF16, ctypes.byref(_ns()), None) == 0
    assert msg in _lib.last_error().encode()


@pytest.mark.parametrize("kw", [dict(count=65535, stride=100 * 128), dict(rows=8, cols=65535 * 64, ld=65535 * 64)])
def test_batches_at_the_grid_limits(lib, kw):
    args = dict(count=1, rows=100, cols=128)
    args.update(kw)
    assert lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, _batch(**args), 1, _lib.GNS_BF16, ctypes.byref(_ns()), None) > 0


@pytest.mark.parametrize("kw,msg", [
    (dict(T=0), b"T must"),
    (dict(T=17), b"T must"),
    (dict(restart_mask=1), b"restart_mask"),
    (dict(restart_mask=1 << 5), b"restart_mask"),
])
def test_invalid_schedules(lib, kw, msg):
    b = _batch(1, 64, 128)
    assert lib.gns_workspace_size(_lib.GNS_OP_GRAM_NS, b, 1, _lib.GNS_BF16, ctypes.byref(_ns(**kw)), None) == 0
    assert msg in _lib.last_error().encode()


def test_calls_reject_bad_arguments_before_launch(lib):
    """Validation failures return without touching the device (pointers here are fake)."""
    b = _batch(1, 64, 128)
    o = _batch(1, 64, 128, ptr=1 << 21)
    rc = lib.gns_gram_ns_batched(b, o, 1, _lib.GNS_BF16, ctypes.byref(_ns()), None, 0, None, None)
    assert rc == _lib.GNS_ERR_WORKSPACE
    rc = lib.gns_gram_ns_batched(b, b, 1, _lib.GNS_BF16, ctypes.byref(_ns()), ctypes.c_void_p(1 << 24), 1 << 30,
                                 None, None)
    assert rc == _lib.GNS_ERR_INVALID and b"alias" in _lib.last_error().encode()
    mp = _lib.GnsMuonParams(0.02, 0.95, 0.0, 1.0, 1.5)
    rc = lib.gns_muon_step(b, o, _batch(1, 64, 128, ptr=1 << 22), None, 1, ctypes.byref(mp), ctypes.byref(_ns()),
                           None, 0, None, None)
    assert rc == _lib.GNS_ERR_INVALID and b"frac" in _lib.last_error().encode()
    rc = lib.gns_frac_row_select(b, 65, ctypes.c_void_p(1 << 23), None, ctypes.c_void_p(1 << 24), 1 << 30, None)
    assert rc == _lib.GNS_ERR_INVALID
