"""Python front of the double-precision CPU oracle (``flce_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing here imports the
CUDA package, and the CUDA package never imports this.

Every function takes CPU torch tensors or numpy arrays (float64, float32 or
bfloat16) and returns float64 numpy arrays.  bfloat16 inputs are passed to C
as their raw 16-bit patterns and widened exactly there.

What is computed (the plain definition; the loss call ``loss_fn(weight,
input, target)`` of the Liger-Kernel project overview, "Método de API de
Baixo Nível", computed exactly as "Cálculo Preciso" states):
    loss  = mean over valid rows of (logsumexp(S_i) - S_{i,t_i}),  S = X W^T
    dX    = G W,  dW = G^T X,  G_ij = valid_i (softmax(S_i)_j - [j = t_i]) / n_valid
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flce_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_flce.argtypes = [p, p, i32, p, i64, i64, i64, i64, i64,
                                        p, p, p, p, p, p]
            lib.oracle_flce.restype = i32
            lib.oracle_flce_rows.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                             p, i64, p, p, p, p]
            lib.oracle_flce_rows.restype = i32
            lib.oracle_flce_dw_rows.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                                p, i64, p]
            lib.oracle_flce_dw_rows.restype = i32
            lib.oracle_ce.argtypes = [p, i32, p, i64, i64, i64, p, p, p, p, p]
            lib.oracle_ce.restype = i32
            lib.oracle_count_valid.argtypes = [p, i64, i64]
            lib.oracle_count_valid.restype = i64
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _as_matrix(a):
    """(contiguous numpy array, type code) for a float64/float32/bf16 input."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16), BF16
            if a.dtype == torch.float32:
                return a.numpy(), F32
            if a.dtype == torch.float64:
                return a.numpy(), F64
            raise TypeError(f"unsupported dtype {a.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _as_targets(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().to(torch.int64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t, dtype=np.int64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc == 1:
        raise OracleError("bad arguments")
    if rc == 2:
        raise OracleError("target outside [0, V) that is not the ignore index")


def flce(X, W, t, ignore_index: int = -100, grads: bool = True,
         norm_count: int = 0) -> dict:
    """Full problem: loss, n_valid, lse [N], loss_rows [N], dX [N,H], dW [V,H].

    ``norm_count > 0`` makes this call one data-parallel shard of a larger
    batch: the mean and G are divided by that count (the whole batch's valid
    rows) instead of by this call's own ``n_valid``."""
    x, tx = _as_matrix(X)
    w, tw = _as_matrix(W)
    if tx != tw:
        raise TypeError("X and W must share one element type")
    tt = _as_targets(t)
    N, H = x.shape
    V = w.shape[0]
    assert w.shape[1] == H and tt.shape == (N,)
    loss = np.zeros(1)
    nv = np.zeros(1, dtype=np.int64)
    lse = np.zeros(N)
    lrows = np.zeros(N)
    dX = np.zeros((N, H)) if grads else None
    dW = np.zeros((V, H)) if grads else None
    rc = _load().oracle_flce(_ptr(x), _ptr(w), tx, _ptr(tt), N, H, V, int(ignore_index),
                             int(norm_count), _ptr(loss), _ptr(nv), _ptr(lse), _ptr(lrows),
                             _ptr(dX), _ptr(dW))
    _check(rc)
    return {"loss": float(loss[0]), "n_valid": int(nv[0]), "lse": lse,
            "loss_rows": lrows, "dX": dX, "dW": dW}


def flce_rows(X, W, t, rows, ignore_index: int = -100, grads: bool = True) -> dict:
    """Selected token rows of the full problem: lse, loss_rows, dX rows."""
    x, tx = _as_matrix(X)
    w, tw = _as_matrix(W)
    if tx != tw:
        raise TypeError("X and W must share one element type")
    tt = _as_targets(t)
    N, H = x.shape
    V = w.shape[0]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    lse = np.zeros(len(r))
    lrows = np.zeros(len(r))
    dX = np.zeros((len(r), H)) if grads else None
    nv = np.zeros(1, dtype=np.int64)
    rc = _load().oracle_flce_rows(_ptr(x), _ptr(w), tx, _ptr(tt), N, H, V,
                                  int(ignore_index), _ptr(r), len(r), _ptr(lse),
                                  _ptr(lrows), _ptr(dX), _ptr(nv))
    _check(rc)
    return {"lse": lse, "loss_rows": lrows, "dX": dX, "n_valid": int(nv[0])}


def flce_dw_rows(X, W, t, vocab_rows, ignore_index: int = -100) -> np.ndarray:
    """Selected vocabulary rows of dW for the full problem."""
    x, tx = _as_matrix(X)
    w, tw = _as_matrix(W)
    if tx != tw:
        raise TypeError("X and W must share one element type")
    tt = _as_targets(t)
    N, H = x.shape
    V = w.shape[0]
    r = np.ascontiguousarray(vocab_rows, dtype=np.int64)
    out = np.zeros((len(r), H))
    rc = _load().oracle_flce_dw_rows(_ptr(x), _ptr(w), tx, _ptr(tt), N, H, V,
                                     int(ignore_index), _ptr(r), len(r), _ptr(out))
    _check(rc)
    return out


def ce(S, t, ignore_index: int = -100, grads: bool = True) -> dict:
    """Cross-entropy on materialised logits S [N, V]: loss, n_valid, lse,
    loss_rows, dS [N, V] (the gradient of the mean loss)."""
    s, ts = _as_matrix(S)
    tt = _as_targets(t)
    N, V = s.shape
    assert tt.shape == (N,)
    loss = np.zeros(1)
    nv = np.zeros(1, dtype=np.int64)
    lse = np.zeros(N)
    lrows = np.zeros(N)
    dS = np.zeros((N, V)) if grads else None
    rc = _load().oracle_ce(_ptr(s), ts, _ptr(tt), N, V, int(ignore_index), _ptr(loss),
                           _ptr(nv), _ptr(lse), _ptr(lrows), _ptr(dS))
    _check(rc)
    return {"loss": float(loss[0]), "n_valid": int(nv[0]), "lse": lse, "loss_rows": lrows,
            "dS": dS}


def count_valid(t, ignore_index: int = -100) -> int:
    tt = _as_targets(t)
    return int(_load().oracle_count_valid(_ptr(tt), len(tt), int(ignore_index)))
