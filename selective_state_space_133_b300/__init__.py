"""Selective state-space (Mamba S6) scan for B300 (sm_103a).

The compute path is the C-ABI library ``libmambascan.so`` (hand-written CUDA
kernels); ``ops`` is its thin Python binding and ``synthetic`` the seeded
input generators. Importing this package does not load the library; the ops
load it on first use and raise if it has not been built.
"""
from .build import build_library  # noqa: F401

__all__ = ["build_library", "mamba_scan_fwd", "mamba_conv_scan_fwd", "mamba_scan_bwd", "mamba_state_update",
           "mamba_ssd_fwd", "mamba_ssd_update", "check_device_error"]


def __getattr__(name):
    if name in ("mamba_scan_fwd", "mamba_conv_scan_fwd", "mamba_scan_bwd", "mamba_state_update", "mamba_ssd_fwd",
                "mamba_ssd_update",
                "check_device_error"):
        from . import ops
        return getattr(ops, name)
    raise AttributeError(name)
