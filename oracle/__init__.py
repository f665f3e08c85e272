"""fp64 CPU oracle for the late-interaction MaxSim operator.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition that the CUDA
library is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the library itself never
does, and the two share no code.

The arithmetic lives in ``maxsim_oracle.c`` (plain C, fp64, OpenMP over
independent (query, document) pairs).  This module only compiles it with gcc
and marshals numpy arrays through ctypes.

Inputs are numpy arrays in their storage type: float64, float32, float16, or
bfloat16 bit patterns held in a uint16 array (pass ``dtype="bf16"``).  Masks
are bool/uint8 arrays, 1 = valid token, or None (every token valid).

Every forward returns ``(scores, argmax, gap)``: fp64 scores, int32 argmax
(-1 for a masked query token or an empty document) and the fp64 distance
between the best and second-best similarity of each query token.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "maxsim_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, F16, BF16, F64 = 0, 1, 2, 3
EMPTY_DOC_SCORE = -1e9

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _declare(lib):
    i64, ptr, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
    fwd_common = [ptr, ptr, ctypes.c_int]
    lib.oracle_pair.restype = dbl
    lib.oracle_pair.argtypes = [ptr, ptr, i64, ptr, ptr, i64, i64, ptr, ptr]
    lib.oracle_allpairs_fwd.restype = None
    lib.oracle_allpairs_fwd.argtypes = fwd_common + [i64] * 5 + [ptr] * 5
    lib.oracle_pairwise_fwd.restype = None
    lib.oracle_pairwise_fwd.argtypes = fwd_common + [i64] * 4 + [ptr] * 5
    lib.oracle_kd_fwd.restype = None
    lib.oracle_kd_fwd.argtypes = fwd_common + [i64] * 5 + [ptr] * 5
    lib.oracle_allpairs_bwd.restype = None
    lib.oracle_allpairs_bwd.argtypes = fwd_common + [i64] * 5 + [ptr] * 4
    lib.oracle_pairwise_bwd.restype = None
    lib.oracle_pairwise_bwd.argtypes = fwd_common + [i64] * 4 + [ptr] * 4
    lib.oracle_kd_bwd.restype = None
    lib.oracle_kd_bwd.argtypes = fwd_common + [i64] * 5 + [ptr] * 4
    lib.oracle_ce_rows.restype = None
    lib.oracle_ce_rows.argtypes = [ptr, i64, i64, ptr, dbl, ptr, ptr, ptr]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def load_library(path: str | None = None):
    """Load (compiling first if needed) the oracle library.

    With an explicit ``path`` the library at that path is loaded as is and not
    cached; this is how tests load deliberately broken copies of the oracle.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                compile_oracle()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _dtype_code(a: np.ndarray, dtype: str | None) -> int:
    if dtype == "bf16":
        if a.dtype != np.uint16:
            raise TypeError("bf16 inputs are passed as uint16 bit patterns")
        return BF16
    if dtype not in (None, "f16", "f32", "f64"):
        raise ValueError(f"unknown dtype {dtype!r}")
    codes = {np.dtype(np.float64): F64, np.dtype(np.float32): F32, np.dtype(np.float16): F16}
    if a.dtype not in codes:
        raise TypeError(f"unsupported oracle input dtype {a.dtype}")
    return codes[a.dtype]


def _c(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _mask(m, shape):
    if m is None:
        return None
    m = np.ascontiguousarray(np.asarray(m).astype(np.uint8))
    if m.shape != tuple(shape):
        raise ValueError(f"mask shape {m.shape} != {tuple(shape)}")
    return m


class Oracle:
    """Thin ctypes front end; one instance may wrap a deliberately broken copy."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load_library()

    # -- threads ----------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    # -- one pair ---------------------------------------------------------
    def pair(self, q, d, qmask=None, dmask=None):
        """Score one query [Lq,dim] against one document [Ld,dim] (fp64 inputs)."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        d = np.ascontiguousarray(d, dtype=np.float64)
        Lq, dim = q.shape
        Ld = d.shape[0]
        qm, dm = _mask(qmask, (Lq,)), _mask(dmask, (Ld,))
        am = np.empty(Lq, np.int32)
        gap = np.empty(Lq, np.float64)
        s = self.lib.oracle_pair(_c(q), _c(qm), Lq, _c(d), _c(dm), Ld, dim, _c(am), _c(gap))
        return float(s), am, gap

    # -- forward ----------------------------------------------------------
    def allpairs_fwd(self, Q, D, qmask=None, dmask=None, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        assert _dtype_code(D, dtype) == code, "Q and D must share one dtype"
        Nq, Lq, dim = Q.shape
        Nd, Ld, dim2 = D.shape
        assert dim == dim2
        qm, dm = _mask(qmask, (Nq, Lq)), _mask(dmask, (Nd, Ld))
        s = np.empty((Nq, Nd), np.float64)
        am = np.empty((Nq, Nd, Lq), np.int32)
        gap = np.empty((Nq, Nd, Lq), np.float64)
        self.lib.oracle_allpairs_fwd(_c(Q), _c(D), code, Nq, Nd, Lq, Ld, dim,
                                     _c(qm), _c(dm), _c(s), _c(am), _c(gap))
        return s, am, gap

    def pairwise_fwd(self, Q, D, qmask=None, dmask=None, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        assert _dtype_code(D, dtype) == code
        B, Lq, dim = Q.shape
        B2, Ld, dim2 = D.shape
        assert B == B2 and dim == dim2
        qm, dm = _mask(qmask, (B, Lq)), _mask(dmask, (B, Ld))
        s = np.empty(B, np.float64)
        am = np.empty((B, Lq), np.int32)
        gap = np.empty((B, Lq), np.float64)
        self.lib.oracle_pairwise_fwd(_c(Q), _c(D), code, B, Lq, Ld, dim,
                                     _c(qm), _c(dm), _c(s), _c(am), _c(gap))
        return s, am, gap

    def kd_fwd(self, Q, D, qmask=None, dmask=None, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        assert _dtype_code(D, dtype) == code
        B, Lq, dim = Q.shape
        B2, N, Ld, dim2 = D.shape
        assert B == B2 and dim == dim2
        qm, dm = _mask(qmask, (B, Lq)), _mask(dmask, (B, N, Ld))
        s = np.empty((B, N), np.float64)
        am = np.empty((B, N, Lq), np.int32)
        gap = np.empty((B, N, Lq), np.float64)
        self.lib.oracle_kd_fwd(_c(Q), _c(D), code, B, N, Lq, Ld, dim,
                               _c(qm), _c(dm), _c(s), _c(am), _c(gap))
        return s, am, gap

    # -- backward ---------------------------------------------------------
    def allpairs_bwd(self, Q, D, grad_out, argmax, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        Nq, Lq, dim = Q.shape
        Nd, Ld, _ = D.shape
        g = np.ascontiguousarray(grad_out, dtype=np.float64).reshape(Nq, Nd)
        am = np.ascontiguousarray(argmax, dtype=np.int32).reshape(Nq, Nd, Lq)
        gQ = np.empty((Nq, Lq, dim), np.float64)
        gD = np.empty((Nd, Ld, dim), np.float64)
        self.lib.oracle_allpairs_bwd(_c(Q), _c(D), code, Nq, Nd, Lq, Ld, dim,
                                     _c(g), _c(am), _c(gQ), _c(gD))
        return gQ, gD

    def pairwise_bwd(self, Q, D, grad_out, argmax, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        B, Lq, dim = Q.shape
        _, Ld, _ = D.shape
        g = np.ascontiguousarray(grad_out, dtype=np.float64).reshape(B)
        am = np.ascontiguousarray(argmax, dtype=np.int32).reshape(B, Lq)
        gQ = np.empty((B, Lq, dim), np.float64)
        gD = np.empty((B, Ld, dim), np.float64)
        self.lib.oracle_pairwise_bwd(_c(Q), _c(D), code, B, Lq, Ld, dim,
                                     _c(g), _c(am), _c(gQ), _c(gD))
        return gQ, gD

    def kd_bwd(self, Q, D, grad_out, argmax, dtype=None):
        Q, D = np.ascontiguousarray(Q), np.ascontiguousarray(D)
        code = _dtype_code(Q, dtype)
        B, Lq, dim = Q.shape
        _, N, Ld, _ = D.shape
        g = np.ascontiguousarray(grad_out, dtype=np.float64).reshape(B, N)
        am = np.ascontiguousarray(argmax, dtype=np.int32).reshape(B, N, Lq)
        gQ = np.empty((B, Lq, dim), np.float64)
        gD = np.empty((B, N, Ld, dim), np.float64)
        self.lib.oracle_kd_bwd(_c(Q), _c(D), code, B, N, Lq, Ld, dim,
                               _c(g), _c(am), _c(gQ), _c(gD))
        return gQ, gD


    def ce_rows(self, scores, target, scale=1.0):
        """Mean softmax cross-entropy over score rows: (loss, row_loss, grad)."""
        S = np.ascontiguousarray(scores, dtype=np.float64)
        rows, cols = S.shape
        t = np.ascontiguousarray(target, dtype=np.int32).reshape(rows)
        row_loss = np.empty(rows, np.float64)
        grad = np.empty((rows, cols), np.float64)
        loss = np.empty(1, np.float64)
        self.lib.oracle_ce_rows(_c(S), rows, cols, _c(t), float(scale), _c(row_loss), _c(grad), _c(loss))
        return float(loss[0]), row_loss, grad


_default = None


def get() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
