"""Float64 CPU oracle for the linear-attention segment transition cache.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may.  The oracle shares no code with the CUDA path: the C
file ``hypic_oracle.c`` holds the arithmetic, this module only marshals numpy
float64 arrays into it.

What it computes (all from the HYPIC reading notes, see ``hypic_oracle.c``):
the token-by-token recurrence S_i = T_i S_{i-1} + u_i with o_i = q_i^T S_i
(paper Eq. (2), variants of Table 1), the segment pair (T_C, S_{C|0})
(Method 2 and the two-pass build of paper Sec. 5), composition of pairs and the
n-segment form of paper Eq. (6), and the inclusive scan over affine maps.

Every function works on ONE head with contiguous float64 arrays:
k, q: [len, d_k]; v: [len, d_v]; alpha: [1] (scalar_const), [len] (scalar,
gated_delta), [len, d_k] (diag), unused for delta; beta: [len].

Parity: every function is pinned by ``tests/test_oracle_pins.py`` against
closed forms, brute-force dense products, special cases and the page's worked
example and Table 2 values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

FAMILIES = {"scalar_const": 0, "scalar": 1, "diag": 2, "delta": 3, "gated_delta": 4, "kda": 5}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hypic_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libhypic_oracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no machine-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return ctypes.cast(None, _dp)
    return x.ctypes.data_as(_dp)


def _gates(family, alpha, beta, n, dk):
    fam = FAMILIES[family]
    if fam == 0:
        alpha = _f64(np.reshape(np.asarray(alpha, dtype=np.float64), (-1,))[:1])
    elif fam == 3:
        alpha = np.ones(1)
    elif fam in (2, 5):
        alpha = _f64(alpha).reshape(n, dk)
    else:
        alpha = _f64(alpha).reshape(n)
    if fam in (3, 4, 5):
        beta = _f64(beta).reshape(n)
    else:
        beta = np.zeros(1)
    return fam, alpha, beta


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.orc_t_size.argtypes = [i32, i32]
        lib.orc_run.argtypes = [i32, i32, i32, i64, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
        lib.orc_transition.argtypes = [i32, i32, i64, _dp, _dp, _dp, _dp]
        lib.orc_segment_pair.argtypes = [i32, i32, i32, i64, _dp, _dp, _dp, _dp, _dp, _dp]
        lib.orc_affine_combine.argtypes = [i32, i32, i32, _dp, _dp, _dp, _dp, _dp, _dp]
        lib.orc_compose.argtypes = [i32, i32, i32, i32, _dp, _dp, _dp]
        lib.orc_affine_scan.argtypes = [i32, i32, i32, i32, _dp, _dp, _dp, _dp]
        for f in ("orc_run", "orc_transition", "orc_segment_pair", "orc_affine_combine",
                  "orc_compose", "orc_affine_scan", "orc_t_size"):
            getattr(lib, f).restype = i32
        self.lib = lib

    def t_size(self, family: str, dk: int) -> int:
        return int(self.lib.orc_t_size(FAMILIES[family], dk))

    def run(self, family, k, v, alpha, beta=None, q=None, S0=None):
        """Token-by-token recurrence of one head.  Returns (S_end, o or None)."""
        k, v = _f64(k), _f64(v)
        n, dk = k.shape
        dv = v.shape[1]
        fam, alpha, beta = _gates(family, alpha, beta, n, dk)
        S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
        qq = _f64(q) if q is not None else None
        o = np.zeros((n, dv)) if q is not None else None
        rc = self.lib.orc_run(fam, dk, dv, n, _ptr(k), _ptr(v), _ptr(qq), _ptr(alpha), _ptr(beta),
                              _ptr(S), _ptr(o))
        assert rc == 0
        return S, o

    def transition(self, family, k, alpha, beta=None):
        """T_C of one head in storage form: shape [1], [d_k] or [d_k, d_k]."""
        k = _f64(k)
        n, dk = k.shape
        fam, alpha, beta = _gates(family, alpha, beta, n, dk)
        ts = self.lib.orc_t_size(fam, dk)
        T = np.zeros(ts)
        rc = self.lib.orc_transition(fam, dk, n, _ptr(k), _ptr(alpha), _ptr(beta), _ptr(T))
        assert rc == 0
        return T.reshape((dk, dk)) if ts == dk * dk else T

    def segment_pair(self, family, k, v, alpha, beta=None):
        """(T_C, S_{C|0}) of one segment body of one head."""
        k, v = _f64(k), _f64(v)
        n, dk = k.shape
        dv = v.shape[1]
        fam, alpha, beta = _gates(family, alpha, beta, n, dk)
        ts = self.lib.orc_t_size(fam, dk)
        T = np.zeros(ts)
        S = np.zeros((dk, dv))
        rc = self.lib.orc_segment_pair(fam, dk, dv, n, _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                       _ptr(T), _ptr(S))
        assert rc == 0
        return (T.reshape((dk, dk)) if ts == dk * dk else T), S

    def affine_combine(self, family, T2, S2, T1, S1):
        """(T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2): segment 1 first, then 2."""
        S1, S2 = _f64(S1), _f64(S2)
        dk, dv = S1.shape
        T1, T2 = _f64(T1).reshape(-1), _f64(T2).reshape(-1)
        T3 = np.zeros_like(T1)
        S3 = np.zeros_like(S1)
        rc = self.lib.orc_affine_combine(FAMILIES[family], dk, dv, _ptr(T2), _ptr(S2), _ptr(T1), _ptr(S1),
                                         _ptr(T3), _ptr(S3))
        assert rc == 0
        return (T3.reshape((dk, dk)) if T3.size == dk * dk else T3), S3

    def compose(self, family, T, S0, S_init=None):
        """S <- T_j S + S0_j for j = 0..n-1 (paper Eq. (6)).  T: [n, ...], S0: [n, dk, dv]."""
        S0 = _f64(S0)
        n, dk, dv = S0.shape
        T = _f64(T).reshape(n, -1)
        S = np.zeros((dk, dv)) if S_init is None else _f64(S_init).copy()
        rc = self.lib.orc_compose(FAMILIES[family], dk, dv, n, _ptr(T), _ptr(S0), _ptr(S))
        assert rc == 0
        return S

    def affine_scan(self, family, T, S):
        """Inclusive prefix scan of n affine maps; returns (T_prefix, S_prefix)."""
        S = _f64(S)
        n, dk, dv = S.shape
        T = _f64(T).reshape(n, -1)
        Tp = np.zeros_like(T)
        Sp = np.zeros_like(S)
        rc = self.lib.orc_affine_scan(FAMILIES[family], dk, dv, n, _ptr(T), _ptr(S), _ptr(Tp), _ptr(Sp))
        assert rc == 0
        shape = (n, dk, dk) if T.shape[1] == dk * dk else T.shape
        return Tp.reshape(shape), Sp


def default() -> Oracle:
    """The oracle built from ``hypic_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def t_size(family, dk):
    return default().t_size(family, dk)


def run(*a, **kw):
    return default().run(*a, **kw)


def transition(*a, **kw):
    return default().transition(*a, **kw)


def segment_pair(*a, **kw):
    return default().segment_pair(*a, **kw)


def affine_combine(*a, **kw):
    return default().affine_combine(*a, **kw)


def compose(*a, **kw):
    return default().compose(*a, **kw)


def affine_scan(*a, **kw):
    return default().affine_scan(*a, **kw)


def parallel_map(fn, items, threads: int | None = None):
    """Map fn over items on host threads (the C calls release the GIL)."""
    threads = threads or os.cpu_count() or 1
    items = list(items)
    if threads <= 1 or len(items) <= 1:
        return [fn(x) for x in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))
