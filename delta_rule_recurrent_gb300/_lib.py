"""ctypes loader for libdeltanet.so, the C ABI declared in include/deltanet.h.

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

from .build import INCLUDE, LIB_PATH

HEADER = INCLUDE / "deltanet.h"

DN_OK, DN_ERR_INVALID_ARG, DN_ERR_UNSUPPORTED, DN_ERR_CUDA = 0, 1, 2, 3
DN_F32, DN_BF16 = 0, 1
DN_ALGO_AUTO, DN_ALGO_SIMT, DN_ALGO_TCGEN05 = 0, 1, 2
ABI_VERSION = 9

_vp, _fp = ctypes.c_void_p, ctypes.c_void_p
_int, _size = ctypes.c_int, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)
_f32, _ll = ctypes.c_float, ctypes.c_longlong


class QkNorm(ctypes.Structure):
    """dn_qk_norm: the in-kernel preparation of q and k."""
    _fields_ = [("l2norm", ctypes.c_int), ("scale", ctypes.c_float), ("eps", ctypes.c_float)]


_np = ctypes.POINTER(QkNorm)

# Signatures of every entry point in include/deltanet.h.
SIGNATURES = {
    "dn_chunk_fwd": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _int, _int, _int, _int, _int,
                            _int, _int, _vp, _size, _vp]),
    "dn_chunk_fwd_algo": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _int, _int, _int, _int,
                                 _int, _int, _int, _vp, _size, _vp, _int]),
    "dn_chunk_fwd_workspace_bytes": (_size, [_int] * 7),
    "dn_chunk_fwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _int, _int, _int, _int,
                                    _int, _int, _int, _vp]),
    "dn_recurrent_step": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _int, _int, _int, _int, _int,
                                 _vp]),
    "dn_chunk_bwd": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _vp, _vp, _vp, _vp, _fp]
                     + [_int] * 7 + [_vp, _size, _vp]),
    "dn_chunk_bwd_workspace_bytes": (_size, [_int] * 7),
    "dn_chunk_fwd_varlen": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _ip] + [_int] * 7
                            + [_vp, _size, _vp]),
    "dn_chunk_fwd_varlen_workspace_bytes": (_size, [_ip] + [_int] * 6),
    "dn_chunk_fwd_gated": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp] + [_int] * 7
                           + [_vp, _size, _vp]),
    "dn_chunk_fwd_gated_workspace_bytes": (_size, [_int] * 7),
    "dn_recurrent_step_gated": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp] + [_int] * 5 + [_vp]),
    "dn_chunk_fwd_kda": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp] + [_int] * 7 + [_vp]),
    "dn_recurrent_step_kda": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp] + [_int] * 5 + [_vp]),
    "dn_qk_prepare": (_int, [_vp, _vp, _vp, _vp, _ll, _int, _int, _f32, _f32, _int, _vp]),
    "dn_qk_prepare_bwd": (_int, [_vp] * 6 + [_ll, _int, _int, _f32, _f32, _int, _vp]),
    "dn_chunk_fwd_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp] + [_int] * 7
                        + [_vp, _size, _vp, _int, _np]),
    "dn_chunk_fwd_gated_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp] + [_int] * 7
                              + [_vp, _size, _vp, _np]),
    "dn_chunk_fwd_varlen_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _ip] + [_int] * 7
                               + [_vp, _size, _vp, _np]),
    "dn_chunk_fwd_kda_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp] + [_int] * 7
                            + [_vp, _size, _vp, _np]),
    "dn_chunk_fwd_kda_workspace_bytes": (_size, [_int] * 7),
    "dn_recurrent_step_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _vp] + [_int] * 5 + [_vp, _np]),
    "dn_recurrent_step_gated_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp] + [_int] * 5
                                   + [_vp, _np]),
    "dn_recurrent_step_kda_qk": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp] + [_int] * 5
                                 + [_vp, _np]),
    "dn_status_string": (ctypes.c_char_p, [_int]),
    "dn_last_error": (ctypes.c_char_p, []),
    "dn_abi_version": (_int, []),
    "dn_device_error": (_int, []),
    "dn_debug_first_wait_ns": (_int, [ctypes.c_ulonglong]),
    "dn_chunk_fwd_split": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp] + [_int] * 8
                           + [_vp, _size, _vp]),
    "dn_chunk_fwd_split_workspace_bytes": (_size, [_int] * 8),
    "dn_chunk_bwd_varlen": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _vp, _vp, _vp, _vp, _fp, _ip]
                            + [_int] * 7 + [_vp, _size, _vp]),
    "dn_chunk_bwd_varlen_workspace_bytes": (_size, [_ip] + [_int] * 6),
    "dn_chunk_bwd_gated": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp, _vp, _vp, _vp, _vp, _fp,
                                  _fp] + [_int] * 7 + [_vp, _size, _vp]),
    "dn_chunk_bwd_gated_workspace_bytes": (_size, [_int] * 7),
    "dn_chunk_bwd_kda": (_int, [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp, _vp, _vp, _vp, _vp, _fp,
                                _fp] + [_int] * 7 + [_vp, _size, _vp]),
    "dn_chunk_bwd_kda_workspace_bytes": (_size, [_int] * 7),
}

_lib = None


class DeltaNetError(RuntimeError):
    """A non-OK status from the library, with its detail message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def _status_name(status: int) -> str:
    names = {0: "DN_OK", 1: "DN_ERR_INVALID_ARG", 2: "DN_ERR_UNSUPPORTED", 3: "DN_ERR_CUDA"}
    return names.get(status, f"status {status}")


def header_symbols(path: Path = HEADER) -> list[str]:
    """Names of the entry points the header declares (DN_API functions)."""
    text = path.read_text()
    return re.findall(r"DN_API\s+[\w\s\*]*?\b(dn_\w+)\s*\(", text)


def lib_path() -> Path:
    return LIB_PATH


def load(path: Path | None = None):
    """Loads the library (once) and declares every signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise RuntimeError(
            f"{p} is not built; run `python -m delta_rule_recurrent_gb300.build` "
            "(the operator has no fallback implementation)")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if lib.dn_abi_version() != ABI_VERSION:
        raise RuntimeError("libdeltanet ABI version mismatch")
    if path is None:
        _lib = lib
    return lib


def check(status: int) -> None:
    """Raises DeltaNetError for a non-OK status."""
    if status != DN_OK:
        msg = load().dn_last_error().decode(errors="replace")
        raise DeltaNetError(status, msg)
