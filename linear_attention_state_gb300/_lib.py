"""ctypes view of libhypic's C ABI (``include/hypic.h``).  Loading fails loudly if the library is missing."""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhypic.so")

HYPIC_OK, HYPIC_EINVAL, HYPIC_EUNSUPPORTED, HYPIC_ECUDA, HYPIC_ETIMEOUT, HYPIC_ENOSPACE, HYPIC_EDEVICE = (
    0, -1, -2, -3, -4, -5, -6)
FAMILY = {"scalar_const": 0, "scalar": 1, "diag": 2, "delta": 3, "gated_delta": 4, "kda": 5}
DTYPE = {"f32": 0, "bf16": 1}

# Every symbol include/hypic.h declares, with (restype, argtypes).
_vp, _fp, _i32p, _i64p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i32, _i64, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class Shape(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("family", ctypes.c_int32), ("in_dtype", ctypes.c_int32)]


_SP = ctypes.POINTER(Shape)

SIGNATURES = {
    "hypic_abi_version": (_i32, []),
    "hypic_t_size": (_i64, [_SP]),
    "hypic_strerror": (ctypes.c_char_p, [_i32]),
    "hypic_segment_build": (_i32, [_SP, _vp, _vp, _vp, _fp, _fp, _i64, _fp, _fp, _fp, _vp, _sz, _vp]),
    "hypic_segment_build_batched": (_i32, [_SP, _i32, _i64p, _i64, _i64, _vp, _vp, _vp, _fp, _fp, _fp, _fp,
                                           _fp, _vp, _sz, _vp]),
    "hypic_segment_build_batched_host": (_i32, [_SP, _i32, _i64p, _i64, _i64, _vp, _vp, _fp, _fp, _vp, _vp, _fp,
                                                _fp, _i64p, _fp, _fp, _vp, _sz, _vp, _vp, _vp]),
    "hypic_build_workspace_bytes": (_sz, [_SP, _i32, _i64]),
    "hypic_build_workspace_bytes_outputs": (_sz, [_SP, _i32, _i64]),
    "hypic_segment_build_batched_noalloc": (_i32, [_SP, _i32, _i64p, _i64, _i64, _vp, _vp, _vp, _fp, _fp, _fp,
                                                   _fp, _fp, _vp]),
    "hypic_compose": (_i32, [_SP, _i32, _i32, _i32p, _i64, _fp, _fp, _fp, _fp, _vp]),
    "hypic_affine_scan": (_i32, [_SP, _i32, _fp, _fp, _fp, _fp, _vp, _sz, _vp]),
    "hypic_scan_workspace_bytes": (_sz, [_SP, _i32]),
    "hypic_seam_advance": (_i32, [_SP, _i32, _fp, _vp, _vp, _vp, _fp, _fp, _i32, _fp, _vp]),
    "hypic_assemble": (_i32, [_SP, _i32, _i32, _i32, _i32p, _i64, _fp, _fp, _vp, _vp, _vp, _fp, _fp, _fp,
                              _fp, _fp, _vp]),
    "hypic_pairs_to_bf16": (_i32, [_SP, _i64, _fp, _fp, _vp, _vp, _vp]),
    "hypic_compose_bf16": (_i32, [_SP, _i32, _i32, _i32p, _i64, _vp, _vp, _fp, _fp, _vp]),
    "hypic_assemble_bf16": (_i32, [_SP, _i32, _i32, _i32, _i32p, _i64, _vp, _vp, _vp, _vp, _vp, _fp, _fp, _fp,
                                   _fp, _fp, _vp]),
    "hypic_rope_shift": (_i32, [_i64, _i32, _i32, ctypes.c_double, _i64, _i32, _vp, _vp, _vp]),
    "hypic_state_rerotate": (_i32, [_SP, _i64, _fp, _i32, ctypes.c_double, _i64, _vp]),
    "hypic_conv_tail": (_i32, [_i32, _i32, _i32, _i64p, _i64, _i32, _vp, _vp, _vp]),
    "hypic_conv_seam": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _fp, _fp, _i32, _fp, _vp]),
    "hypic_stream_status": (_i32, [_vp]),
    "hypic_selftest_bounded_wait": (_i32, [_i64, _vp]),
}

_lock = threading.Lock()
_lib = None


class HypicError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


def load(path: str | None = None) -> ctypes.CDLL:
    """The loaded libhypic.  Raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libhypic.so not found at {p}: build it first "
                                   "(python -m linear_attention_state_gb300.build)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return lib
            _lib = lib
    return _lib


def strerror(status: int) -> str:
    try:
        return load().hypic_strerror(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {status}"


def check(status: int, where: str) -> None:
    if status != HYPIC_OK:
        raise HypicError(status, where)


def shape(H: int, d: int, family: str, in_dtype: str) -> Shape:
    return Shape(int(H), int(d), int(d), FAMILY[family], DTYPE[in_dtype])
