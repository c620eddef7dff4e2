"""The on-chip chain kernel (chain_small.cu): Gram and standard Newton-Schulz of matrices
whose oriented X has at most 128 rows and 512 columns, one CTA per matrix, against the fp64
oracle. Covers ragged shapes (n < 128, m not a multiple of 64), tall matrices (X loaded
transposed), square matrices (standard NS), a single row, fp16 products, schedules with no,
one and several restarts, T = 1, the Muon step with the weight update in the last epilogue,
the in-kernel norm against a norm passed in, degenerate and non-finite inputs, and the
same groups on the batched tile path (GNS_CHAIN_SMALL=0) for comparison."""
import ctypes
import os

import numpy as np
import pytest

from oracle import muon as omuon
from oracle import newton_schulz as ons
from util import bf16_input, bits_to_torch, f16_input, rel_fro, torch_to_bits, torch_to_f64

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")
from matrix_orthogonalizing_optimizer_gb300 import _lib  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F16 = 5e-3
# a single row: every singular value is 1 after normalisation (the rank-1 precision class)
TOL_RANK1 = 4e-2


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _launches(fn):
    """(GEMM-class launches, all launches) of libgns during fn()."""
    lib = _lib.load()
    torch.cuda.synchronize()
    lib.gns_profile_set(None, 0)
    r = fn()
    torch.cuda.synchronize()
    g, a = ctypes.c_int(0), ctypes.c_int(0)
    lib.gns_profile_query(ctypes.byref(g), ctypes.byref(a))
    return r, g.value, a.value


def _chain_off(fn):
    old = os.environ.get("GNS_CHAIN_SMALL")
    os.environ["GNS_CHAIN_SMALL"] = "0"
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["GNS_CHAIN_SMALL"]
        else:
            os.environ["GNS_CHAIN_SMALL"] = old


@pytest.mark.parametrize("count,rows,cols", [(5, 128, 512), (3, 100, 300), (4, 64, 200), (2, 1, 40), (3, 512, 128),
                                            (2, 300, 97), (3, 128, 64), (2, 16, 512)])
def test_chain_gram_vs_oracle(count, rows, cols):
    bits, x = bf16_input(80, (count, rows, cols))
    xt = bits_to_torch(bits)
    st = _status()
    (out, ), n_gemm, n_all = _launches(lambda: gns.gram_ns_batched(xt, status=st))
    assert int(st.item()) == 0
    # one launch: no separate norm pass (the kernel sums ||X||_F from the X it holds)
    assert (n_gemm, n_all) == (1, 1)
    got = torch_to_f64(out)
    tol = TOL_RANK1 if min(rows, cols) == 1 else TOL_BF16
    for b in range(count):
        assert rel_fro(got[b], omuon.orthogonalize(x[b])) < tol, b


@pytest.mark.parametrize("count,rows,cols", [(5, 128, 512), (3, 96, 96), (2, 100, 300), (2, 128, 128)])
def test_chain_standard_vs_oracle(count, rows, cols):
    bits, x = bf16_input(81, (count, rows, cols))
    xt = bits_to_torch(bits)
    st = _status()
    (out, ), n_gemm, n_all = _launches(lambda: gns.ns_standard_batched(xt, status=st))
    assert int(st.item()) == 0 and (n_gemm, n_all) == (1, 1)
    got = torch_to_f64(out)
    for b in range(count):
        want = ons.ns_standard(x[b], ons.QUINTIC_FIXED)
        assert rel_fro(got[b], want) < TOL_BF16, b


@pytest.mark.parametrize("coeffs,restarts", [
    (ons.QUINTIC_FIXED, ()),
    (ons.QUINTIC_FIXED, (1, 3)),
    (ons.QUINTIC_FIXED[:1], ()),
    (ons.QUINTIC_FIXED * 2, (2, 5, 8)),
    (ons.CLASSIC, (2,)),
])
@pytest.mark.parametrize("rows,cols", [(128, 448), (400, 72)])
def test_chain_schedules(coeffs, restarts, rows, cols):
    """Any schedule and restart set, against the oracle and against the tile path. Ten
    iterations accumulate bf16 storage rounding beyond 2e-2 on both paths alike (measured
    2.2-3.4 %; fp16 products 0.3-0.4 %): that class is held to 4e-2."""
    count = 3
    bits, x = bf16_input(82, (count, rows, cols))
    xt = bits_to_torch(bits)
    ns = gns.NsParams(coeffs=coeffs, restarts=restarts)
    got = torch_to_f64(gns.gram_ns_batched(xt, ns=ns)[0])
    tile = torch_to_f64(_chain_off(lambda: gns.gram_ns_batched(xt, ns=ns))[0])
    tol = TOL_BF16 if len(coeffs) <= 5 else 4e-2
    for b in range(count):
        want = omuon.orthogonalize(x[b], coeffs=coeffs, restarts=restarts)
        assert rel_fro(got[b], want) < tol, b
        # the two paths sum ||X||_F differently: their bf16 roundings part at noise level
        # (up to 1.7 % over ten iterations)
        assert rel_fro(got[b], tile[b]) < 2.5e-2, b


@pytest.mark.parametrize("rows,cols", [(128, 512), (320, 96)])
def test_chain_fp16(rows, cols):
    count = 3
    x16, x = f16_input(83, (count, rows, cols))
    xt = torch.from_numpy(x16).cuda()
    st = _status()
    out = gns.gram_ns_batched(xt, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and out.dtype == torch.float16
    got = torch_to_f64(out)
    for b in range(count):
        assert rel_fro(got[b], omuon.orthogonalize(x[b])) < TOL_F16, b


@pytest.mark.parametrize("rows,cols", [(128, 512), (384, 96), (128, 128)])
def test_chain_muon_step(rows, cols):
    """Momentum, the norm from the momentum pass, the chain and the weight update fused into
    the last epilogue (wide, tall: written transposed; square: standard NS)."""
    count = 6
    s = 1.0 / np.sqrt(cols)
    Wb, _ = bf16_input(84, (count, rows, cols), s, stream=0)
    Gb, _ = bf16_input(84, (count, rows, cols), s, stream=1)
    Mb, _ = bf16_input(84, (count, rows, cols), s, stream=2)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    _, n_gemm, _ = _launches(lambda: gns.muon_step(Wt, Gt, Mt, lr=0.02, momentum=0.95, weight_decay=0.1))
    assert n_gemm == 1
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(count):
        W_or, M_or, O = omuon.muon_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95, weight_decay=0.1)
        if rows == cols:
            O = ons.ns_standard(omuon.bf16_decode(M_or), ons.QUINTIC_FIXED)
            W_or = (1 - 0.02 * 0.1) * omuon.bf16_decode(Wb[b]) - 0.02 * O
        assert np.array_equal(Mg[b], M_or)
        dW = Wg[b] - W_or
        mag = np.maximum(np.maximum(np.abs(Wg[b]), np.abs(W_or)), 2.0 ** -126)
        excess = np.maximum(np.abs(dW) - 0.5 * 2.0 ** (np.floor(np.log2(mag)) - 7), 0.0)
        assert np.linalg.norm(excess) / np.linalg.norm(0.02 * O) < TOL_BF16, b


@pytest.mark.parametrize("rows,cols", [(128, 512), (96, 200), (500, 100)])
def test_chain_matches_tile_path(rows, cols):
    """The same group on the chain kernel and on the batched tile path (both near the oracle,
    and near each other: they round the same products in the same type)."""
    count = 4
    bits, x = bf16_input(85, (count, rows, cols))
    xt = bits_to_torch(bits)
    a = torch_to_f64(gns.gram_ns_batched(xt)[0])
    (b_out, ), _, n_all = _launches(lambda: _chain_off(lambda: gns.gram_ns_batched(xt)))
    assert n_all == 3  # norm pass, norm finalisation, one GEMM launch (n < 512: the scale as an array)
    b = torch_to_f64(b_out)
    for i in range(count):
        want = omuon.orthogonalize(x[i])
        assert rel_fro(a[i], want) < TOL_BF16 and rel_fro(b[i], want) < TOL_BF16
        assert rel_fro(a[i], b[i]) < TOL_BF16


@pytest.mark.parametrize("count,rows,cols", [(4, 64, 72), (4, 100, 112), (3, 128, 144)])
def test_chain_near_square(count, rows, cols):
    """Near-square Gaussian matrices (m / n <= 1.25): the smallest singular values sit near
    1 - sqrt(n / m) of the largest, where bf16 storage of R and Q costs 2-4 % on either path
    (measured on the tile path too, to the same digits). Both paths against the oracle at the
    class bound, and against each other closely."""
    bits, x = bf16_input(80, (count, rows, cols))
    xt = bits_to_torch(bits)
    a = torch_to_f64(gns.gram_ns_batched(xt)[0])
    b = torch_to_f64(_chain_off(lambda: gns.gram_ns_batched(xt))[0])
    for i in range(count):
        want = omuon.orthogonalize(x[i])
        assert rel_fro(a[i], want) < 5e-2 and rel_fro(b[i], want) < 5e-2, i
        assert rel_fro(a[i], b[i]) < 4e-2, i  # each path carries 2-4 % of its own rounding noise


def test_chain_degenerate_and_nonfinite():
    # zero matrices: eps keeps the result finite and zero
    z = torch.zeros((3, 128, 256), dtype=torch.bfloat16, device="cuda")
    st = _status()
    out = gns.gram_ns_batched(z, status=st)[0]
    outs = gns.ns_standard_batched(z, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.count_nonzero(out).item() == 0 and torch.count_nonzero(outs).item() == 0
    # a non-finite entry in one matrix is reported; the other matrices are unaffected
    bits, x = bf16_input(86, (3, 96, 320))
    bad = bits_to_torch(bits).clone()
    bad[1, 7, 11] = float("inf")
    st = _status()
    out = gns.gram_ns_batched(bad, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    got = torch_to_f64(out)
    for b in (0, 2):
        assert rel_fro(got[b], omuon.orthogonalize(x[b])) < TOL_BF16
    with pytest.raises(gns.GnsDeviceError, match="non-finite"):
        gns.gram_ns_batched(bad)
    gns.check_status()


def test_chain_many_matrices_per_cta():
    """More matrices than SMs: each CTA runs several matrices in turn (the X reload waits for
    the previous matrix's last product; parities of every barrier alternate)."""
    count, rows, cols = 700, 112, 448
    g = torch.Generator(device="cuda")
    g.manual_seed(87)
    X = (torch.randn((count, rows, cols), generator=g, device="cuda") / cols ** 0.5).to(torch.bfloat16)
    st = _status()
    out = gns.gram_ns_batched(X, status=st)[0]
    outs = gns.ns_standard_batched(X, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in sorted({0, 1, 151, 152, 153, 303, 304, 455, count - 1}):
        want = omuon.orthogonalize(torch_to_f64(X[b]))
        assert rel_fro(torch_to_f64(out[b]), want) < TOL_BF16, b
        want_s = ons.ns_standard(torch_to_f64(X[b]), ons.QUINTIC_FIXED)
        assert rel_fro(torch_to_f64(outs[b]), want_s) < TOL_BF16, b


def test_chain_several_groups_one_launch():
    """Several shape groups in one call: the chain kernel carries all Gram groups in one launch
    (wide, ragged, tall, a single-row group), square groups (standard NS) in a second, and
    more than eight groups in further launches of eight."""
    shapes = [(40, 128, 512), (17, 96, 300), (33, 400, 72), (5, 1, 64), (9, 64, 64)]
    xs, refs = [], []
    for i, (c, r, k) in enumerate(shapes):
        bits, x = bf16_input(88, (c, r, k), stream=i)
        xs.append(bits_to_torch(bits))
        refs.append(x)
    st = _status()
    outs, n_gemm, n_all = _launches(lambda: gns.gram_ns_batched(xs, status=st))
    assert int(st.item()) == 0
    assert (n_gemm, n_all) == (2, 2)  # the four Gram groups, then the square group
    for (c, r, k), out, x in zip(shapes, outs, refs):
        got = torch_to_f64(out)
        for b in sorted({0, c // 2, c - 1}):
            want = (ons.ns_standard(x[b], ons.QUINTIC_FIXED) if r == k else omuon.orthogonalize(x[b]))
            tol = TOL_RANK1 if min(r, k) == 1 else TOL_BF16
            assert rel_fro(got[b], want) < tol, (r, k, b)
    # ten groups: two launches (eight, then two)
    xs10 = [xs[0][:3].clone() for _ in range(10)]
    outs10, n_gemm, _ = _launches(lambda: gns.gram_ns_batched(xs10))
    assert n_gemm == 2
    for o in outs10:
        assert torch.equal(o, outs10[0])


def test_chain_muon_step_several_groups():
    """A Muon step over small groups (chain kernel, one launch after their momentum passes)
    and a larger group (batched tile path), each against the oracle."""
    shapes = [(12, 128, 512), (7, 384, 96), (5, 256, 1024)]
    Ws, Gs, Ms, raw = [], [], [], []
    for i, (c, r, k) in enumerate(shapes):
        s = 1.0 / np.sqrt(k)
        Wb, _ = bf16_input(89, (c, r, k), s, stream=3 * i)
        Gb, _ = bf16_input(89, (c, r, k), s, stream=3 * i + 1)
        Mb, _ = bf16_input(89, (c, r, k), s, stream=3 * i + 2)
        Ws.append(bits_to_torch(Wb))
        Gs.append(bits_to_torch(Gb))
        Ms.append(bits_to_torch(Mb))
        raw.append((Wb, Gb, Mb))
    _, n_gemm, _ = _launches(lambda: gns.muon_step(Ws, Gs, Ms, lr=0.02, momentum=0.95))
    assert n_gemm == 2  # one chain launch for the two small groups, one tile-path launch
    for (c, r, k), Wt, Mt, (Wb, Gb, Mb) in zip(shapes, Ws, Ms, raw):
        Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
        for b in sorted({0, c - 1}):
            W_or, M_or, O = omuon.muon_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95)
            assert np.array_equal(Mg[b], M_or)
            dW = Wg[b] - W_or
            mag = np.maximum(np.maximum(np.abs(Wg[b]), np.abs(W_or)), 2.0 ** -126)
            excess = np.maximum(np.abs(dW) - 0.5 * 2.0 ** (np.floor(np.log2(mag)) - 7), 0.0)
            assert np.linalg.norm(excess) / np.linalg.norm(0.02 * O) < TOL_BF16, (r, k, b)


def _pack_off(fn):
    old = os.environ.get("GNS_CHAIN_PACK")
    os.environ["GNS_CHAIN_PACK"] = "0"
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["GNS_CHAIN_PACK"]
        else:
            os.environ["GNS_CHAIN_PACK"] = old


# Gaussian matrices of at most 64 rows: bf16 storage costs 1.3-3.2 % on every path (the
# packed and unpacked chains and the batched tile path give the same errors to three digits)
TOL_SMALL_N = 4e-2


@pytest.mark.parametrize("count,rows,cols", [(5, 64, 200), (7, 32, 96), (6, 48, 320), (9, 20, 64), (3, 1, 24),
                                            (6, 64, 64), (4, 33, 512)])
def test_chain_packed(count, rows, cols):
    """Wide matrices of at most 64 (32) rows packed two (four) to a 128-row chain in diagonal
    blocks: bit-identical to the same group unpacked (GNS_CHAIN_PACK=0), each matrix against
    the oracle (standard NS for a square group), groups whose last chain is partly empty."""
    bits, x = bf16_input(92, (count, rows, cols))
    xt = bits_to_torch(bits)
    fn = gns.ns_standard_batched if rows == cols else gns.gram_ns_batched
    st = _status()
    got = fn(xt, status=st)[0]
    unpacked = _pack_off(lambda: fn(xt))[0]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got, unpacked)
    got = torch_to_f64(got)
    tol = TOL_RANK1 if rows == 1 else TOL_SMALL_N
    for b in range(count):
        want = ons.ns_standard(x[b], ons.QUINTIC_FIXED) if rows == cols else omuon.orthogonalize(x[b])
        assert rel_fro(got[b], want) < tol, b


def test_chain_packed_muon_step():
    """A Muon step over packed chains: momentum bit-exact, the weight update against the oracle."""
    count, rows, cols = 11, 64, 256
    s = 1.0 / np.sqrt(cols)
    Wb, _ = bf16_input(93, (count, rows, cols), s, stream=0)
    Gb, _ = bf16_input(93, (count, rows, cols), s, stream=1)
    Mb, _ = bf16_input(93, (count, rows, cols), s, stream=2)
    Wt, Gt, Mt = bits_to_torch(Wb), bits_to_torch(Gb), bits_to_torch(Mb)
    gns.muon_step(Wt, Gt, Mt, lr=0.02, momentum=0.95, weight_decay=0.1)
    torch.cuda.synchronize()
    Mg, Wg = torch_to_bits(Mt), torch_to_f64(Wt)
    for b in range(count):
        W_or, M_or, O = omuon.muon_step(Wb[b], Gb[b], Mb[b], lr=0.02, mu=0.95, weight_decay=0.1)
        assert np.array_equal(Mg[b], M_or)
        dW = Wg[b] - W_or
        mag = np.maximum(np.maximum(np.abs(Wg[b]), np.abs(W_or)), 2.0 ** -126)
        excess = np.maximum(np.abs(dW) - 0.5 * 2.0 ** (np.floor(np.log2(mag)) - 7), 0.0)
        assert np.linalg.norm(excess) / np.linalg.norm(0.02 * O) < TOL_BF16, b


@pytest.mark.parametrize("rows,cols,bad", [(64, 200, 2), (32, 96, 5), (64, 64, 1)])
def test_chain_packed_nonfinite_isolated(rows, cols, bad):
    """A non-finite entry in one matrix of a packed chain: reported, that matrix's result not
    finite, and the matrices packed with it bit-identical to the same call without it (their
    rows never meet its values)."""
    count = 8
    bits, x = bf16_input(94, (count, rows, cols))
    clean = bits_to_torch(bits)
    dirty = clean.clone()
    dirty[bad, 3, 7] = float("inf")
    fn = gns.ns_standard_batched if rows == cols else gns.gram_ns_batched
    ref = fn(clean)[0]
    st = _status()
    out = fn(dirty, status=st)[0]
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    assert not torch.isfinite(out[bad]).all()
    for b in range(count):
        if b != bad:
            assert torch.equal(out[b], ref[b]), b
