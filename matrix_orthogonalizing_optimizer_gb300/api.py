"""Python API over libgns with the C ABI's names. PyTorch supplies device memory and the
stream; every step of the computation runs in the library's CUDA kernels.

Tensors are CUDA tensors of dtype bfloat16 (hot path), float16 (Dion3 Algorithm 3's
float16 products) or float32 (validation path), 2-D (one matrix) or 3-D (a batch of
same-shape matrices, the megabatch of Dion3 sec. 7), with a contiguous last dimension,
16-byte aligned rows (ld a multiple of 16 bytes) and 16-byte aligned storage.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass
from typing import Iterable, List, Optional, Sequence

import torch

from . import _lib
from ._lib import GnsBatch, GnsMuonParams, GnsNsParams, load
from ._lib import check as check_rc

# Fixed quintic of "Scaling Muon for Diffusion Transformers", appendix D.3.
QUINTIC_FIXED = ((3.4445, -4.7750, 2.0315),) * 5


@dataclass
class NsParams:
    """Newton-Schulz schedule (T = len(coeffs)); restarts = iterations after which Gram NS
    restarts (Dion3 Algorithm 3: after iteration 2); safety = s runs every polynomial as
    p_t(x / s) (Dion3 appendix B.2.2; 1.05 is the pages' conservative choice for a Polar
    Express table, 1 leaves the coefficients as given)."""
    coeffs: Sequence = QUINTIC_FIXED
    restarts: Sequence[int] = (2,)
    eps: float = 1e-7
    safety: float = 1.0

    def c_struct(self) -> GnsNsParams:
        p = GnsNsParams()
        p.T = len(self.coeffs)
        if not 1 <= p.T <= _lib.GNS_MAX_T:
            raise ValueError("T must be in [1, 16]")
        for t, (a, b, c) in enumerate(self.coeffs):
            p.a[t], p.b[t], p.c[t] = float(a), float(b), float(c)
        mask = 0
        for r in self.restarts:
            mask |= 1 << int(r)
        p.restart_mask = mask
        p.eps = float(self.eps)
        p.safety = float(self.safety)
        return p


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.GNS_BF16
    if t.dtype == torch.float16:
        return _lib.GNS_F16
    if t.dtype == torch.float32:
        return _lib.GNS_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16, float16 or float32")


_FLAVORS = {"muon": _lib.GNS_FLAVOR_MUON, "normuon": _lib.GNS_FLAVOR_NORMUON, "rownorm": _lib.GNS_FLAVOR_ROWNORM,
            "periodic": _lib.GNS_FLAVOR_PERIODIC}


@dataclass
class MuonParams:
    """Hyper-parameters of one optimizer step (gns_muon_params). flavor: "muon" (Dion3 eq.
    (1)), "normuon" (eq. (2)), "rownorm" (Scaling Muon for DiTs eq. (5)) or "periodic"
    (ibid. eq. (7): Newton-Schulz when step % period == 0, RowNorm otherwise). ns_dtype:
    torch.bfloat16 or torch.float16, the storage type of the Newton-Schulz products."""
    lr: float
    momentum: float = 0.95
    weight_decay: float = 0.0
    scale: float = 1.0
    frac: float = 1.0
    flavor: str = "muon"
    ns_dtype: torch.dtype = torch.bfloat16
    beta2: float = 0.95
    norm_eps: float = 1e-8
    rownorm_gamma: float = 0.15
    period: int = 3
    step: int = 0

    def c_struct(self) -> GnsMuonParams:
        if self.flavor not in _FLAVORS:
            raise ValueError(f"flavor must be one of {sorted(_FLAVORS)}")
        if self.ns_dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("ns_dtype must be torch.bfloat16 or torch.float16")
        return GnsMuonParams(float(self.lr), float(self.momentum), float(self.weight_decay), float(self.scale),
                             float(self.frac), _FLAVORS[self.flavor],
                             _lib.GNS_F16 if self.ns_dtype == torch.float16 else _lib.GNS_BF16, float(self.beta2),
                             float(self.norm_eps), float(self.rownorm_gamma), int(self.period), int(self.step))


def batch_of(t: torch.Tensor) -> GnsBatch:
    """gns_batch describing a 2-D or 3-D CUDA tensor (no copy)."""
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if t.dim() == 2:
        t3 = t.unsqueeze(0)
    elif t.dim() == 3:
        t3 = t
    else:
        raise ValueError("tensors must be 2-D or 3-D")
    if t3.stride(2) != 1:
        raise ValueError("the last dimension must be contiguous")
    b = GnsBatch()
    b.ptr = t3.data_ptr()
    b.count, b.rows, b.cols = t3.shape
    # a single row has no row stride of its own: any ld >= cols that keeps rows aligned
    b.ld = t3.stride(1) if t3.shape[1] > 1 else ((b.cols + 7) // 8) * 8
    b.stride = t3.stride(0) if t3.shape[0] > 1 else b.rows * b.ld
    return b


def empty_padded(shape, dtype, device) -> torch.Tensor:
    """Uninitialised tensor of `shape` whose rows start on 16-byte boundaries (the last
    dimension is padded in storage, the returned view has the requested shape)."""
    *lead, cols = shape
    al = 16 // torch.empty((), dtype=dtype).element_size()
    ld = (cols + al - 1) // al * al
    return torch.empty((*lead, ld), dtype=dtype, device=device)[..., :cols]


def _batches(ts: Iterable[torch.Tensor]):
    ts = list(ts)
    arr = (GnsBatch * len(ts))(*[batch_of(t) for t in ts])
    return arr, ts


def _stream_ptr(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _as_list(x) -> List[torch.Tensor]:
    return [x] if isinstance(x, torch.Tensor) else list(x)


def workspace_size(op: int, xs, ns: Optional[NsParams] = None, frac: float = 1.0, dtype=None,
                   muon: Optional[MuonParams] = None) -> int:
    xs = _as_list(xs)
    arr, _ = _batches(xs)
    dt = _dtype_code(xs[0]) if dtype is None else dtype
    nsp = (ns or NsParams()).c_struct()
    mp = muon.c_struct() if muon is not None else GnsMuonParams(0.0, 0.0, 0.0, 1.0, float(frac))
    n = load().gns_workspace_size(op, arr, len(xs), dt, ctypes.byref(nsp), ctypes.byref(mp))
    if n == 0:
        raise _lib.GnsError(f"workspace_size: {_lib.last_error()}")
    return int(n)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned device buffer of at least nbytes (torch allocations are)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _status_ptr(status: Optional[torch.Tensor]) -> Optional[int]:
    if status is None:
        return None
    if status.dtype != torch.int32 or not status.is_cuda:
        raise ValueError("status must be a CUDA int32 tensor")
    return status.data_ptr()


# Device status words (include/gns.h: bit 0 non-finite output, bit 1 a bounded wait timed
# out) owned by this module, one per device, for calls made without `status=`. The kernels OR
# into them; a word is only cleared when its bits are reported, so nothing the GPU detects is
# lost: a call that cannot check (check=False, or stream capture) leaves its bits for the next
# checked call on the device, or for check_status().
_OWNED_STATUS = {}


def _device_index(device) -> int:
    d = torch.device(device) if device is not None else torch.device("cuda")
    return d.index if d.index is not None else torch.cuda.current_device()


def _capturing(stream: Optional[torch.cuda.Stream]) -> bool:
    if torch.cuda.is_current_stream_capturing():
        return True
    if stream is not None:
        with torch.cuda.stream(stream):
            return torch.cuda.is_current_stream_capturing()
    return False


def _owned_status(device) -> torch.Tensor:
    idx = _device_index(device)
    t = _OWNED_STATUS.get(idx)
    if t is None:
        if torch.cuda.is_current_stream_capturing():
            raise ValueError("the first call on a device must run outside stream capture (or pass status=)")
        t = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda", idx))
        _OWNED_STATUS[idx] = t
    return t


def _report(what: str, st: torch.Tensor) -> None:
    v = int(st.cpu()[0])
    if v:
        st.zero_()
        raise _lib.GnsDeviceError(what, v)


class _CallStatus:
    """The status word one call passes to the library: the caller's own (`status=`, read by
    the caller, or by check_status(status)), else this module's word of the device, which is
    checked after the call when `check` is set by synchronising the call's stream."""

    def __init__(self, status: Optional[torch.Tensor], device, check: bool, stream):
        self.owned = status is None
        self.word = _owned_status(device) if self.owned else status
        self.check = check
        self.stream = stream
        self.device = device

    def ptr(self) -> int:
        return _status_ptr(self.word)

    def done(self, what: str) -> None:
        if not self.owned or not self.check or _capturing(self.stream):
            return
        s = self.stream if self.stream is not None else torch.cuda.current_stream(self.device)
        s.synchronize()
        _report(what, self.word)


def check_status(status: Optional[torch.Tensor] = None, device=None, what: str = "libgns") -> None:
    """Synchronises the device and raises GnsDeviceError when the status word has bits set
    (then clears it): the caller's `status` tensor, or, when None, this module's word for the
    device, which collects the bits of every call made without `status=` (including calls
    recorded into CUDA graphs and replayed)."""
    if status is None:
        idx = _device_index(device)
        if idx not in _OWNED_STATUS:
            return
        status = _OWNED_STATUS[idx]
    torch.cuda.synchronize(status.device)
    _report(what, status)


def _ns_common(fn_name: str, op: int, xs, outs, ns, workspace, status, stream, check_dev):
    xs = _as_list(xs)
    outs = [empty_padded(x.shape, x.dtype, x.device) for x in xs] if outs is None else _as_list(outs)
    ns = ns or NsParams()
    need = workspace_size(op, xs, ns)
    ws = workspace if workspace is not None else alloc_workspace(need, xs[0].device)
    xa, _ = _batches(xs)
    oa, _ = _batches(outs)
    nsp = ns.c_struct()
    fn = getattr(load(), fn_name)
    cs = _CallStatus(status, xs[0].device, check_dev, stream)
    rc = fn(xa, oa, len(xs), _dtype_code(xs[0]), ctypes.byref(nsp), ws.data_ptr(), ws.numel(),
            cs.ptr(), _stream_ptr(stream, xs[0].device))
    check_rc(rc, fn_name)
    cs.done(fn_name)
    return outs


# Device status of every call below: with `status=` (a CUDA int32 tensor) the library ORs its
# bits into that tensor and the call returns without synchronising (read it, or pass it to
# check_status(), after the stream is done). Without it the call uses this module's status
# word of the device and, when `check` is set (the default), synchronises the call's stream
# and raises GnsDeviceError if the GPU flagged a non-finite output or a timed-out wait.


def gram_ns_batched(xs, outs=None, ns: Optional[NsParams] = None, workspace=None, status=None, stream=None,
                    check: bool = True):
    """Gram Newton-Schulz (Dion3 Algorithm 3) of every matrix in xs (tensor or list of
    tensors, one per shape group); returns the list of outputs."""
    return _ns_common("gns_gram_ns_batched", _lib.GNS_OP_GRAM_NS, xs, outs, ns, workspace, status, stream, check)


def ns_standard_batched(xs, outs=None, ns: Optional[NsParams] = None, workspace=None, status=None, stream=None,
                        check: bool = True):
    """Standard Newton-Schulz (Dion3 Algorithm 1 with symmetric products)."""
    return _ns_common("gns_ns_standard_batched", _lib.GNS_OP_NS_STANDARD, xs, outs, ns, workspace, status, stream,
                      check)


def sym_gemm_xxt(x: torch.Tensor, c: torch.Tensor, alpha: float = 1.0, beta: float = 0.0, status=None, stream=None,
                 check: bool = True):
    xb, cb = batch_of(x), batch_of(c)
    cs = _CallStatus(status, x.device, check, stream)
    rc = load().gns_sym_gemm_xxt(ctypes.byref(xb), ctypes.byref(cb), float(alpha), float(beta), _dtype_code(x),
                                 cs.ptr(), _stream_ptr(stream, x.device))
    check_rc(rc, "gns_sym_gemm_xxt")
    cs.done("gns_sym_gemm_xxt")
    return c


def sym_gemm(a: torch.Tensor, b: torch.Tensor, c: Optional[torch.Tensor], d: torch.Tensor, alpha: float = 1.0,
             beta: float = 0.0, status=None, stream=None, check: bool = True):
    ab, bb, db = batch_of(a), batch_of(b), batch_of(d)
    cb = batch_of(c) if c is not None else None
    cs = _CallStatus(status, a.device, check, stream)
    rc = load().gns_sym_gemm(ctypes.byref(ab), ctypes.byref(bb), ctypes.byref(cb) if cb is not None else None,
                             ctypes.byref(db), float(alpha), float(beta), _dtype_code(a), cs.ptr(),
                             _stream_ptr(stream, a.device))
    check_rc(rc, "gns_sym_gemm")
    cs.done("gns_sym_gemm")
    return d


def sym_poly_update(R, Q, Z, RZ, q_scratch, a: float, b: float, c: float, q_is_identity: bool, skip_r: bool,
                    status=None, stream=None, check: bool = True):
    bs = [batch_of(t) for t in (R, Q, Z, RZ)]
    qs = batch_of(q_scratch) if q_scratch is not None else None
    cs = _CallStatus(status, R.device, check, stream)
    rc = load().gns_sym_poly_update(*[ctypes.byref(x) for x in bs], ctypes.byref(qs) if qs is not None else None,
                                    float(a), float(b), float(c), int(bool(q_is_identity)), int(bool(skip_r)),
                                    _dtype_code(R), cs.ptr(), _stream_ptr(stream, R.device))
    check_rc(rc, "gns_sym_poly_update")
    cs.done("gns_sym_poly_update")


def muon_step(W, G, M, lr: Optional[float] = None, momentum: float = 0.95, weight_decay: float = 0.0, scale: float = 1.0,
              frac: float = 1.0, ns: Optional[NsParams] = None, workspace=None, status=None, stream=None,
              V=None, params: Optional[MuonParams] = None, check: bool = True):
    """One optimizer step in place on W and M (and V): Muon (frac = 1), the Dion3 fractional
    update (frac < 1), or the flavour named in `params` (which then supplies every
    hyper-parameter). V: NorMuon second moments, fp32 tensors (count, 1, min(rows, cols)) or
    (1, min(rows, cols)) per group."""
    Ws, Gs, Ms = _as_list(W), _as_list(G), _as_list(M)
    ns = ns or NsParams()
    if params is None:
        if lr is None:
            raise ValueError("muon_step needs lr (or params)")
        params = MuonParams(lr=lr, momentum=momentum, weight_decay=weight_decay, scale=scale, frac=frac)
    need = workspace_size(_lib.GNS_OP_MUON_STEP, Ms, ns, muon=params)
    ws = workspace if workspace is not None else alloc_workspace(need, Ms[0].device)
    wa, _ = _batches(Ws)
    ga, _ = _batches(Gs)
    ma, _ = _batches(Ms)
    va = None
    if V is not None:
        va, _ = _batches(_as_list(V))
    nsp = ns.c_struct()
    mp = params.c_struct()
    cs = _CallStatus(status, Ms[0].device, check, stream)
    rc = load().gns_muon_step(wa, ga, ma, va, len(Ms), ctypes.byref(mp), ctypes.byref(nsp), ws.data_ptr(),
                              ws.numel(), cs.ptr(), _stream_ptr(stream, Ms[0].device))
    check_rc(rc, "gns_muon_step")
    cs.done("gns_muon_step")


def frac_row_select(m: torch.Tensor, k: int, idx: Optional[torch.Tensor] = None, gathered=None, workspace=None,
                    stream=None):
    """Exact-l1 top-k rows (columns of a tall matrix) of every matrix of m; returns idx."""
    mb = batch_of(m)
    count = mb.count
    if idx is None:
        idx = torch.empty((count, k), dtype=torch.int32, device=m.device)
    if idx.dtype != torch.int32 or not idx.is_contiguous() or idx.numel() < count * k:
        raise ValueError("idx must be a contiguous int32 tensor of count * k entries")
    need = workspace_size(_lib.GNS_OP_FRAC_SELECT, [m])
    ws = workspace if workspace is not None else alloc_workspace(need, m.device)
    gb = batch_of(gathered) if gathered is not None else None
    rc = load().gns_frac_row_select(ctypes.byref(mb), int(k), idx.data_ptr(),
                                    ctypes.byref(gb) if gb is not None else None, ws.data_ptr(), ws.numel(),
                                    _stream_ptr(stream, m.device))
    check_rc(rc, "gns_frac_row_select")
    return idx


def frac_k(frac: float, n: int) -> int:
    """k = ceil(f n) of Dion3 Algorithm 4, clamped to [1, n]."""
    return max(1, min(n, int(math.ceil(frac * n - 1e-9))))
