"""ctypes view of libgns (include/gns.h). Marshalling only: no arithmetic happens here."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgns.so")

GNS_OK = 0
GNS_ERR_INVALID = -1
GNS_ERR_UNSUPPORTED = -2
GNS_ERR_WORKSPACE = -3
GNS_ERR_CUDA = -4
GNS_DEVST_NONFINITE = 1
GNS_DEVST_TIMEOUT = 2
GNS_BF16 = 0
GNS_F32 = 1
GNS_F16 = 2
GNS_FLAVOR_MUON = 0
GNS_FLAVOR_NORMUON = 1
GNS_FLAVOR_ROWNORM = 2
GNS_FLAVOR_PERIODIC = 3
GNS_OP_GRAM_NS = 0
GNS_OP_NS_STANDARD = 1
GNS_OP_MUON_STEP = 2
GNS_OP_FRAC_SELECT = 3
GNS_MAX_T = 16
GNS_NOALLOC_SCRATCH_BYTES = 64 << 20

# Every symbol include/gns.h declares.
EXPORTS = [
    "gns_version", "gns_status_string", "gns_last_error", "gns_ns_params_default", "gns_workspace_size",
    "gns_gram_ns_batched", "gns_ns_standard_batched", "gns_sym_gemm_xxt", "gns_sym_gemm",
    "gns_sym_poly_update", "gns_muon_step", "gns_frac_row_select", "gns_profile_set", "gns_profile_query", "gns_gram_ns_batched_noalloc",
    "gns_selftest_bounded_wait",
]


class GnsBatch(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("count", ctypes.c_int64), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64), ("stride", ctypes.c_int64)]


class GnsNsParams(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("a", ctypes.c_float * GNS_MAX_T), ("b", ctypes.c_float * GNS_MAX_T),
                ("c", ctypes.c_float * GNS_MAX_T), ("restart_mask", ctypes.c_uint32), ("eps", ctypes.c_float),
                ("safety", ctypes.c_float)]


class GnsMuonParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("momentum", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("scale", ctypes.c_float), ("frac", ctypes.c_float), ("flavor", ctypes.c_int32),
                ("ns_dtype", ctypes.c_int32), ("beta2", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("rownorm_gamma", ctypes.c_float), ("period", ctypes.c_int32), ("step", ctypes.c_int32)]


_lib = None


class GnsError(RuntimeError):
    pass


class GnsDeviceError(GnsError):
    """A condition the GPU detected during a call (bits of the device status word)."""

    def __init__(self, what: str, bits: int):
        names = [n for b, n in ((GNS_DEVST_NONFINITE, "non-finite output"),
                                (GNS_DEVST_TIMEOUT, "a bounded wait timed out (results are incomplete)"))
                 if bits & b]
        super().__init__(f"{what}: device status {bits}: {', '.join(names) or 'unknown bits'}")
        self.bits = bits


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise GnsError(f"libgns.so not found at {path}: build it with "
                       f"`python -m matrix_orthogonalizing_optimizer_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    B = P(GnsBatch)
    lib.gns_version.restype = i32
    lib.gns_status_string.restype = ctypes.c_char_p
    lib.gns_status_string.argtypes = [i32]
    lib.gns_last_error.restype = i32
    lib.gns_last_error.argtypes = [ctypes.c_char_p, sz]
    lib.gns_ns_params_default.restype = None
    lib.gns_ns_params_default.argtypes = [P(GnsNsParams)]
    lib.gns_workspace_size.restype = sz
    lib.gns_workspace_size.argtypes = [i32, B, i32, i32, P(GnsNsParams), P(GnsMuonParams)]
    for name in ("gns_gram_ns_batched", "gns_ns_standard_batched"):
        fn = getattr(lib, name)
        fn.restype = i32
        fn.argtypes = [B, B, i32, i32, P(GnsNsParams), vp, sz, vp, vp]
    lib.gns_sym_gemm_xxt.restype = i32
    lib.gns_sym_gemm_xxt.argtypes = [B, B, f32, f32, i32, vp, vp]
    lib.gns_sym_gemm.restype = i32
    lib.gns_sym_gemm.argtypes = [B, B, B, B, f32, f32, i32, vp, vp]
    lib.gns_sym_poly_update.restype = i32
    lib.gns_sym_poly_update.argtypes = [B, B, B, B, B, f32, f32, f32, i32, i32, i32, vp, vp]
    lib.gns_muon_step.restype = i32
    lib.gns_muon_step.argtypes = [B, B, B, B, i32, P(GnsMuonParams), P(GnsNsParams), vp, sz, vp, vp]
    lib.gns_frac_row_select.restype = i32
    lib.gns_frac_row_select.argtypes = [B, i32, vp, B, vp, sz, vp]
    lib.gns_gram_ns_batched_noalloc.restype = i32
    lib.gns_gram_ns_batched_noalloc.argtypes = [B, B, i32, i32, P(GnsNsParams), vp, vp]
    lib.gns_selftest_bounded_wait.restype = i32
    lib.gns_selftest_bounded_wait.argtypes = [vp, i32, ctypes.c_uint32, vp, vp, vp]
    lib.gns_profile_set.restype = i32
    lib.gns_profile_set.argtypes = [P(vp), i32]
    lib.gns_profile_query.restype = i32
    lib.gns_profile_query.argtypes = [P(i32), P(i32)]
    _lib = lib
    return lib


def last_error() -> str:
    lib = load()
    buf = ctypes.create_string_buffer(1024)
    lib.gns_last_error(buf, 1024)
    return buf.value.decode(errors="replace")


def check(rc: int, what: str) -> None:
    if rc != GNS_OK:
        lib = load()
        raise GnsError(f"{what}: {lib.gns_status_string(rc).decode()}: {last_error()}")
