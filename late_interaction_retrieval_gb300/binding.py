"""Thin ctypes binding of liblik (C ABI: include/lik.h).

Argument marshalling only: each function checks that the torch tensors have
the shapes, dtypes and device the C ABI expects, passes their device
pointers and the current CUDA stream, and raises :class:`LIKError` on a
non-OK status.  Every step of the operator runs in liblik's kernels; there
is no other backend and no CPU fallback.  If liblik cannot be loaded (not
built, or built for another machine) the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LIK_F32, LIK_F16, LIK_BF16 = 0, 1, 2
STATUS = {0: "LIK_OK", 1: "LIK_ERR_INVALID_ARG", 2: "LIK_ERR_UNSUPPORTED", 3: "LIK_ERR_CUDA",
          4: "LIK_ERR_TIMEOUT"}

# Every entry point include/lik.h declares, with its ctypes signature.
_P, _I64, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
SIGNATURES = {
    "lik_status_string": (ctypes.c_char_p, [_I32]),
    "lik_last_error_message": (ctypes.c_char_p, []),
    "lik_version": (ctypes.c_char_p, []),
    "lik_check_device_error": (_I32, [_P]),
    "lik_selftest_bounded_wait": (_I32, [_I64, _P]),
    "lik_maxsim_allpairs_fwd": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_allpairs_bwd": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_pairwise_fwd": (_I32, [_P, _P, _I32] + [_I64] * 4 + [_P] * 5),
    "lik_maxsim_pairwise_bwd": (_I32, [_P, _P, _I32] + [_I64] * 4 + [_P] * 5),
    "lik_maxsim_kd_fwd": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_pairwise_fwd_workspace_bytes": (_I32, [_I32] + [_I64] * 4 + [_I32, _P]),
    "lik_maxsim_kd_fwd_workspace_bytes": (_I32, [_I32] + [_I64] * 5 + [_I32, _P]),
    "lik_maxsim_pairwise_fwd_ws": (_I32, [_P, _P, _I32] + [_I64] * 4 + [_P] * 5 + [ctypes.c_size_t, _P]),
    "lik_maxsim_kd_fwd_ws": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5 + [ctypes.c_size_t, _P]),
    "lik_maxsim_kd_bwd": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_allpairs_bwd_same_dtype": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_pairwise_bwd_same_dtype": (_I32, [_P, _P, _I32] + [_I64] * 4 + [_P] * 5),
    "lik_maxsim_kd_bwd_same_dtype": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 5),
    "lik_maxsim_allpairs_bwd_recompute": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 7),
    "lik_maxsim_pairwise_bwd_recompute": (_I32, [_P, _P, _I32] + [_I64] * 4 + [_P] * 7),
    "lik_maxsim_kd_bwd_recompute": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 7),
    "lik_maxsim_allpairs_bwd_recompute_noalloc": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 6),
    "lik_ce_rows": (_I32, [_P, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _P]),
    "lik_maxsim_allpairs_ce_step": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 3 + [ctypes.c_float]
                                    + [_P] * 7 + [_I32, _P]),
    "lik_maxsim_kd_ce_step": (_I32, [_P, _P, _I32] + [_I64] * 5 + [_P] * 3 + [ctypes.c_float]
                              + [_P] * 7 + [_I32, _P]),
}

_DTYPES = {torch.float32: LIK_F32, torch.float16: LIK_F16, torch.bfloat16: LIK_BF16}

_lock = threading.Lock()
_lib = None


class LIKError(RuntimeError):
    """A liblik call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.status_name}: {message}")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load liblik (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if path is None and not _build.up_to_date():
            try:
                _build.build()
            except Exception as e:  # the CUDA path is the only path: say so loudly
                raise RuntimeError(f"liblik is not built and the build failed: {e}") from e
        if not os.path.exists(p):
            raise RuntimeError(f"liblik not found at {p}; run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        msg = load().lik_last_error_message().decode()
        raise LIKError(status, msg)


def _stream(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor | None, name: str, shape, dtype, device, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _embeddings(Q: torch.Tensor, D: torch.Tensor, q_rank: int, d_rank: int):
    if Q.dim() != q_rank or D.dim() != d_rank:
        raise ValueError(f"expected Q of rank {q_rank} and D of rank {d_rank}")
    if Q.dtype != D.dtype or Q.dtype not in _DTYPES:
        raise ValueError(f"Q and D must share one dtype of float32/float16/bfloat16 "
                         f"(got {Q.dtype}, {D.dtype})")
    if Q.device != D.device or Q.device.type != "cuda":
        raise ValueError("Q and D must be CUDA tensors on one device")
    if Q.shape[-1] != D.shape[-1]:
        raise ValueError("Q and D must share the embedding dimension")
    if not (Q.is_contiguous() and D.is_contiguous()):
        raise ValueError("Q and D must be contiguous")
    return _DTYPES[Q.dtype], Q.device


# ----------------------------------------------------------- all-pairs --

def lik_maxsim_allpairs_fwd(Q, D, qmask, dmask, scores, argmax=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    _need(qmask, "qmask", (Nq, Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", (Nd, Ld), torch.bool, dev, optional=True)
    _need(scores, "scores", (Nq, Nd), torch.float32, dev)
    _need(argmax, "argmax", (Nq, Nd, Lq), torch.int32, dev, optional=True)
    _check(load().lik_maxsim_allpairs_fwd(
        _ptr(Q), _ptr(D), dt, Nq, Nd, Lq, Ld, dim, _ptr(qmask), _ptr(dmask),
        _ptr(scores), _ptr(argmax), _stream(dev, stream)))


def lik_maxsim_allpairs_bwd(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    _need(grad_out, "grad_out", (Nq, Nd), torch.float32, dev)
    _need(argmax, "argmax", (Nq, Nd, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (Nq, Lq, dim), torch.float32, dev, optional=True)
    _need(grad_D, "grad_D", (Nd, Ld, dim), torch.float32, dev, optional=True)
    _check(load().lik_maxsim_allpairs_bwd(
        _ptr(Q), _ptr(D), dt, Nq, Nd, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


# ------------------------------------------------------------ pairwise --

def lik_maxsim_pairwise_fwd(Q, D, qmask, dmask, scores, argmax=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    B, Lq, dim = Q.shape
    if D.shape[0] != B:
        raise ValueError("pairwise: Q and D must have the same batch size")
    Ld = D.shape[1]
    _need(qmask, "qmask", (B, Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", (B, Ld), torch.bool, dev, optional=True)
    _need(scores, "scores", (B,), torch.float32, dev)
    _need(argmax, "argmax", (B, Lq), torch.int32, dev, optional=True)
    _check(load().lik_maxsim_pairwise_fwd(
        _ptr(Q), _ptr(D), dt, B, Lq, Ld, dim, _ptr(qmask), _ptr(dmask),
        _ptr(scores), _ptr(argmax), _stream(dev, stream)))


def lik_maxsim_pairwise_bwd(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    B, Lq, dim = Q.shape
    Ld = D.shape[1]
    _need(grad_out, "grad_out", (B,), torch.float32, dev)
    _need(argmax, "argmax", (B, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (B, Lq, dim), torch.float32, dev, optional=True)
    _need(grad_D, "grad_D", (B, Ld, dim), torch.float32, dev, optional=True)
    _check(load().lik_maxsim_pairwise_bwd(
        _ptr(Q), _ptr(D), dt, B, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


# ------------------------------------------------- per-query candidates --

def lik_maxsim_kd_fwd(Q, D, qmask, dmask, scores, argmax=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 4)
    B, Lq, dim = Q.shape
    if D.shape[0] != B:
        raise ValueError("kd: Q and D must have the same batch size")
    N, Ld = D.shape[1], D.shape[2]
    _need(qmask, "qmask", (B, Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", (B, N, Ld), torch.bool, dev, optional=True)
    _need(scores, "scores", (B, N), torch.float32, dev)
    _need(argmax, "argmax", (B, N, Lq), torch.int32, dev, optional=True)
    _check(load().lik_maxsim_kd_fwd(
        _ptr(Q), _ptr(D), dt, B, N, Lq, Ld, dim, _ptr(qmask), _ptr(dmask),
        _ptr(scores), _ptr(argmax), _stream(dev, stream)))


def lik_maxsim_kd_bwd(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 4)
    B, Lq, dim = Q.shape
    N, Ld = D.shape[1], D.shape[2]
    _need(grad_out, "grad_out", (B, N), torch.float32, dev)
    _need(argmax, "argmax", (B, N, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (B, Lq, dim), torch.float32, dev, optional=True)
    _need(grad_D, "grad_D", (B, N, Ld, dim), torch.float32, dev, optional=True)
    _check(load().lik_maxsim_kd_bwd(
        _ptr(Q), _ptr(D), dt, B, N, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


# ------------------------------------- caller-provided forward workspace --

def _stream_sizes(kind, Q, D):
    if kind == "kd":
        dt, dev = _embeddings(Q, D, 3, 4)
        B, Lq, dim = Q.shape
        if D.shape[0] != B:
            raise ValueError("kd: Q and D must have the same batch size")
        N, Ld = D.shape[1], D.shape[2]
        return dt, dev, (B, N, Lq, Ld, dim), (B, N), (B, N, Ld)
    dt, dev = _embeddings(Q, D, 3, 3)
    B, Lq, dim = Q.shape
    if D.shape[0] != B:
        raise ValueError("pairwise: Q and D must have the same batch size")
    Ld = D.shape[1]
    return dt, dev, (B, Lq, Ld, dim), (B,), (B, Ld)


def _workspace_bytes(kind, Q, D, has_dmask):
    dt, dev, sizes, _, _ = _stream_sizes(kind, Q, D)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(dev):
        _check(getattr(load(), f"lik_maxsim_{kind}_fwd_workspace_bytes")(dt, *sizes, 1 if has_dmask else 0,
                                                                        ctypes.byref(out)))
    return int(out.value)


def lik_maxsim_pairwise_fwd_workspace_bytes(Q, D, has_dmask=True) -> int:
    """Bytes of device workspace lik_maxsim_pairwise_fwd_ws needs for these inputs."""
    return _workspace_bytes("pairwise", Q, D, has_dmask)


def lik_maxsim_kd_fwd_workspace_bytes(Q, D, has_dmask=True) -> int:
    """Bytes of device workspace lik_maxsim_kd_fwd_ws needs for these inputs."""
    return _workspace_bytes("kd", Q, D, has_dmask)


def _fwd_ws(kind, Q, D, qmask, dmask, scores, argmax, workspace, stream):
    dt, dev, sizes, pairs, dshape = _stream_sizes(kind, Q, D)
    Lq = Q.shape[1]
    _need(qmask, "qmask", (Q.shape[0], Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", dshape, torch.bool, dev, optional=True)
    _need(scores, "scores", pairs, torch.float32, dev)
    _need(argmax, "argmax", (*pairs, Lq), torch.int32, dev, optional=True)
    if workspace is not None and (workspace.device != dev or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(getattr(load(), f"lik_maxsim_{kind}_fwd_ws")(
        _ptr(Q), _ptr(D), dt, *sizes, _ptr(qmask), _ptr(dmask), _ptr(scores), _ptr(argmax),
        _ptr(workspace), nbytes, _stream(dev, stream)))


def lik_maxsim_pairwise_fwd_ws(Q, D, qmask, dmask, scores, argmax=None, workspace=None, stream=None):
    """Pairwise forward with a caller-provided workspace (any dtype tensor of at
    least lik_maxsim_pairwise_fwd_workspace_bytes bytes); allocates nothing."""
    _fwd_ws("pairwise", Q, D, qmask, dmask, scores, argmax, workspace, stream)


def lik_maxsim_kd_fwd_ws(Q, D, qmask, dmask, scores, argmax=None, workspace=None, stream=None):
    """Per-query-candidate forward with a caller-provided workspace; allocates nothing."""
    _fwd_ws("kd", Q, D, qmask, dmask, scores, argmax, workspace, stream)


# ------------------------------------------- gradients in the inputs' dtype --

def lik_maxsim_allpairs_bwd_same_dtype(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    _need(grad_out, "grad_out", (Nq, Nd), torch.float32, dev)
    _need(argmax, "argmax", (Nq, Nd, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (Nq, Lq, dim), Q.dtype, dev, optional=True)
    _need(grad_D, "grad_D", (Nd, Ld, dim), Q.dtype, dev, optional=True)
    _check(load().lik_maxsim_allpairs_bwd_same_dtype(
        _ptr(Q), _ptr(D), dt, Nq, Nd, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


def lik_maxsim_pairwise_bwd_same_dtype(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 3)
    B, Lq, dim = Q.shape
    Ld = D.shape[1]
    _need(grad_out, "grad_out", (B,), torch.float32, dev)
    _need(argmax, "argmax", (B, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (B, Lq, dim), Q.dtype, dev, optional=True)
    _need(grad_D, "grad_D", (B, Ld, dim), Q.dtype, dev, optional=True)
    _check(load().lik_maxsim_pairwise_bwd_same_dtype(
        _ptr(Q), _ptr(D), dt, B, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


def lik_maxsim_kd_bwd_same_dtype(Q, D, grad_out, argmax, grad_Q=None, grad_D=None, stream=None):
    dt, dev = _embeddings(Q, D, 3, 4)
    B, Lq, dim = Q.shape
    N, Ld = D.shape[1], D.shape[2]
    _need(grad_out, "grad_out", (B, N), torch.float32, dev)
    _need(argmax, "argmax", (B, N, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", (B, Lq, dim), Q.dtype, dev, optional=True)
    _need(grad_D, "grad_D", (B, N, Ld, dim), Q.dtype, dev, optional=True)
    _check(load().lik_maxsim_kd_bwd_same_dtype(
        _ptr(Q), _ptr(D), dt, B, N, Lq, Ld, dim, _ptr(grad_out), _ptr(argmax),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


# ------------------------------------------ backward that recomputes argmax --

def _recompute(kind, Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q, grad_D, stream):
    if kind == "kd":
        dt, dev = _embeddings(Q, D, 3, 4)
        B, Lq, dim = Q.shape
        N, Ld = D.shape[1], D.shape[2]
        sizes, pairs, dshape = (B, N, Lq, Ld, dim), (B, N), (B, N, Ld)
    else:
        dt, dev = _embeddings(Q, D, 3, 3)
        nq, Lq, dim = Q.shape
        nd, Ld = D.shape[0], D.shape[1]
        if kind == "allpairs":
            sizes, pairs = (nq, nd, Lq, Ld, dim), (nq, nd)
        else:
            sizes, pairs = (nq, Lq, Ld, dim), (nq,)
        dshape = (nd, Ld)
    _need(qmask, "qmask", (Q.shape[0], Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", dshape, torch.bool, dev, optional=True)
    _need(grad_out, "grad_out", pairs, torch.float32, dev)
    _need(argmax_workspace, "argmax_workspace", (*pairs, Lq), torch.int32, dev)
    _need(grad_Q, "grad_Q", tuple(Q.shape), torch.float32, dev, optional=True)
    _need(grad_D, "grad_D", tuple(D.shape), torch.float32, dev, optional=True)
    _check(getattr(load(), f"lik_maxsim_{kind}_bwd_recompute")(
        _ptr(Q), _ptr(D), dt, *sizes, _ptr(qmask), _ptr(dmask), _ptr(grad_out), _ptr(argmax_workspace),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


def lik_maxsim_allpairs_bwd_recompute(Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q=None, grad_D=None,
                                      stream=None):
    _recompute("allpairs", Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q, grad_D, stream)


def lik_maxsim_pairwise_bwd_recompute(Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q=None, grad_D=None,
                                      stream=None):
    _recompute("pairwise", Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q, grad_D, stream)


def lik_maxsim_kd_bwd_recompute(Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q=None, grad_D=None,
                                stream=None):
    _recompute("kd", Q, D, qmask, dmask, grad_out, argmax_workspace, grad_Q, grad_D, stream)


def lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, qmask, dmask, grad_out, grad_Q=None, grad_D=None,
                                              stream=None):
    """The all-pairs recompute backward with the library's built-in argmax
    workspace (no device memory is allocated; Nq * Nd * Lq <= 2**21)."""
    dt, dev = _embeddings(Q, D, 3, 3)
    nq, Lq, dim = Q.shape
    nd, Ld = D.shape[0], D.shape[1]
    _need(qmask, "qmask", (nq, Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", (nd, Ld), torch.bool, dev, optional=True)
    _need(grad_out, "grad_out", (nq, nd), torch.float32, dev)
    _need(grad_Q, "grad_Q", tuple(Q.shape), torch.float32, dev, optional=True)
    _need(grad_D, "grad_D", tuple(D.shape), torch.float32, dev, optional=True)
    _check(load().lik_maxsim_allpairs_bwd_recompute_noalloc(
        _ptr(Q), _ptr(D), dt, nq, nd, Lq, Ld, dim, _ptr(qmask), _ptr(dmask), _ptr(grad_out),
        _ptr(grad_Q), _ptr(grad_D), _stream(dev, stream)))


# --------------------------------------------------- cross-entropy head --

def lik_ce_rows(scores, target, loss, row_loss, grad_scores=None, scale=1.0, stream=None):
    """Mean softmax cross-entropy over the rows of scores [rows, cols]."""
    if scores.dim() != 2:
        raise ValueError("scores must be [rows, cols]")
    dev = scores.device
    rows, cols = scores.shape
    _need(scores, "scores", (rows, cols), torch.float32, dev)
    _need(target, "target", (rows,), torch.int32, dev)
    _need(loss, "loss", (1,), torch.float32, dev)
    _need(row_loss, "row_loss", (rows,), torch.float32, dev)
    _need(grad_scores, "grad_scores", (rows, cols), torch.float32, dev, optional=True)
    _check(load().lik_ce_rows(_ptr(scores), rows, cols, _ptr(target), float(scale), _ptr(loss),
                              _ptr(row_loss), _ptr(grad_scores), _stream(dev, stream)))


def _ce_step(kind, Q, D, qmask, dmask, target, scale, scores, argmax, loss, row_loss, grad_scores,
             grad_Q, grad_D, stream):
    if kind == "allpairs":
        dt, dev = _embeddings(Q, D, 3, 3)
        Nq, Lq, dim = Q.shape
        Nd, Ld, _ = D.shape
        sizes, rows, cols = (Nq, Nd, Lq, Ld, dim), Nq, Nd
        dshape = (Nd, Ld)
    else:
        dt, dev = _embeddings(Q, D, 3, 4)
        B, Lq, dim = Q.shape
        N, Ld = D.shape[1], D.shape[2]
        sizes, rows, cols = (B, N, Lq, Ld, dim), B, N
        dshape = (B, N, Ld)
    same = grad_Q is not None and grad_Q.dtype != torch.float32 or grad_D is not None and grad_D.dtype != torch.float32
    gdt = Q.dtype if same else torch.float32
    _need(qmask, "qmask", (Q.shape[0], Lq), torch.bool, dev, optional=True)
    _need(dmask, "dmask", dshape, torch.bool, dev, optional=True)
    _need(target, "target", (rows,), torch.int32, dev)
    _need(scores, "scores", (rows, cols), torch.float32, dev)
    _need(argmax, "argmax", (rows, cols, Lq), torch.int32, dev)
    _need(loss, "loss", (1,), torch.float32, dev)
    _need(row_loss, "row_loss", (rows,), torch.float32, dev)
    _need(grad_scores, "grad_scores", (rows, cols), torch.float32, dev)
    _need(grad_Q, "grad_Q", tuple(Q.shape), gdt, dev, optional=True)
    _need(grad_D, "grad_D", tuple(D.shape), gdt, dev, optional=True)
    _check(getattr(load(), f"lik_maxsim_{kind}_ce_step")(
        _ptr(Q), _ptr(D), dt, *sizes, _ptr(qmask), _ptr(dmask), _ptr(target), float(scale),
        _ptr(scores), _ptr(argmax), _ptr(loss), _ptr(row_loss), _ptr(grad_scores),
        _ptr(grad_Q), _ptr(grad_D), 1 if same else 0, _stream(dev, stream)))


def lik_maxsim_allpairs_ce_step(Q, D, qmask, dmask, target, scores, argmax, loss, row_loss, grad_scores,
                                grad_Q=None, grad_D=None, scale=1.0, stream=None):
    """In-batch cross-entropy head in one call: forward, loss, backward.
    Gradients in fp32, or in the inputs' dtype when grad_Q/grad_D have it."""
    _ce_step("allpairs", Q, D, qmask, dmask, target, scale, scores, argmax, loss, row_loss,
             grad_scores, grad_Q, grad_D, stream)


def lik_maxsim_kd_ce_step(Q, D, qmask, dmask, target, scores, argmax, loss, row_loss, grad_scores,
                          grad_Q=None, grad_D=None, scale=1.0, stream=None):
    """Per-query-candidate cross-entropy head in one call: forward, loss, backward."""
    _ce_step("kd", Q, D, qmask, dmask, target, scale, scores, argmax, loss, row_loss,
             grad_scores, grad_Q, grad_D, stream)


def lik_check_device_error(stream=None, device=None):
    """Synchronise the stream and raise if a kernel flagged an error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(load().lik_check_device_error(_stream(dev, stream)))


def lik_selftest_bounded_wait(timeout_us: int, stream=None, device=None):
    """Make one bounded device wait run out (see include/lik.h); the next
    lik_check_device_error on the stream then raises LIK_ERR_TIMEOUT."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(load().lik_selftest_bounded_wait(int(timeout_us), _stream(dev, stream)))


def version() -> str:
    return load().lik_version().decode()
