"""ctypes handle on libmambascan.so (the C ABI in include/mamba_scan.h).

There is no fallback: if the library is missing the import of an op raises.
``using(path)`` points every op at another build of the same ABI for a while
(the checked-bounds build, libmambascan_checked.so, in its tests).
"""
from __future__ import annotations

import contextlib
import ctypes
import os

from .build import CHECKED_LIBRARY, LIBRARY  # noqa: F401

MAMBA_F32 = 0
MAMBA_BF16 = 1
MAMBA_FLAG_SOFTPLUS = 1
MAMBA_FLAG_ZOH = 2
STATUS = {0: "MAMBA_OK", -1: "MAMBA_ERR_NULL", -2: "MAMBA_ERR_SHAPE", -3: "MAMBA_ERR_DTYPE",
          -4: "MAMBA_ERR_ALIGN", -5: "MAMBA_ERR_CUDA", -6: "MAMBA_ERR_DEVICE_TIMEOUT",
          -7: "MAMBA_ERR_WORKSPACE", -8: "MAMBA_ERR_FLAGS", -9: "MAMBA_ERR_DEVICE_BOUNDS"}

# (name, restype, argtypes) of every symbol the header declares.
_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
SIGNATURES = {
    "mamba_scan_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "mamba_scan_fwd_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "mamba_scan_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "mamba_conv_scan_fwd_ws": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I,
                                    _I, _P, _Z, _P]),
    "mamba_scan_bwd_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "mamba_scan_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                            _I, _I, _I, _I, _I, _P, _Z, _P]),
    "mamba_scan_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "mamba_state_update": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P]),
    "mamba_ssd_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "mamba_ssd_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "mamba_ssd_update": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "mamba_check_device_error": (_I, [_P]),
    "mamba_status_string": (ctypes.c_char_p, [_I]),
    "mamba_version": (_I, []),
    "mamba_checked_bounds": (_I, []),
}

_lib = None
_handles = {}


class MambaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def load(path: str) -> ctypes.CDLL:
    """The library at ``path`` (loaded once, with every ABI signature set); raise if it has not been built."""
    if path not in _handles:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "selective_state_space_133_b300.build.build_library()")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _handles[path] = handle
    return _handles[path]


def lib() -> ctypes.CDLL:
    """The library every op calls: libmambascan.so unless ``using`` says otherwise."""
    global _lib
    if _lib is None:
        _lib = load(LIBRARY)
    return _lib


@contextlib.contextmanager
def using(path: str):
    """Route every op through the build at ``path`` inside the ``with`` block."""
    global _lib
    before = lib()
    _lib = load(path)
    try:
        yield _lib
    finally:
        _lib = before


def check(status: int, where: str) -> None:
    if status != 0:
        raise MambaError(status, where)
