"""Batched Gram Newton-Schulz orthogonalization and the Muon step for NVIDIA GB300.

The computation lives in libgns (CUDA, sm_103a) behind the C ABI of include/gns.h; this
package holds its build step (``build``), the ctypes binding (``_lib``), the Python API
with the C ABI's names (``api``) and the seeded synthetic inputs (``inputs``).
Importing the package does not load the library: the first API call does, and fails
loudly when it has not been built.
"""
from .api import (  # noqa: F401
    MuonParams,
    NsParams,
    QUINTIC_FIXED,
    alloc_workspace,
    batch_of,
    check_status,
    empty_padded,
    frac_k,
    frac_row_select,
    gram_ns_batched,
    muon_step,
    ns_standard_batched,
    sym_gemm,
    sym_gemm_xxt,
    sym_poly_update,
    workspace_size,
)
from ._lib import GnsDeviceError, GnsError  # noqa: F401

__all__ = [
    "MuonParams", "NsParams", "QUINTIC_FIXED", "alloc_workspace", "batch_of", "check_status", "empty_padded", "frac_k", "frac_row_select", "gram_ns_batched",
    "muon_step", "ns_standard_batched", "sym_gemm", "sym_gemm_xxt", "sym_poly_update", "workspace_size",
    "GnsDeviceError", "GnsError",
]
