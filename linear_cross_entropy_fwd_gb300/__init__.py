"""Python binding of libflce, the GB300 (sm_103a) fused linear cross-entropy
engine.  Argument marshalling only: every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and every call
fails loudly when the library is missing or the device is not sm_103.

The operation is the one of the Liger-Kernel project overview's low-level API
("Método de API de Baixo Nível"): ``loss = loss_fn(weight, input, target)``
then ``loss.backward()``, i.e. softmax cross-entropy on the LM-head logits
``input @ weight.T`` averaged over rows whose target is not ``ignore_index``,
with the exact gradients ("Cálculo Preciso").

C names are kept: ``flce_fwd_bwd``, ``flce_fwd_bwd_ex``, ``flce_fwd``,
``flce_fwd_bwd_host``, ``flce_fwd_noalloc``, ``flce_ce_fwd_bwd``,
``flce_workspace_bytes``; ``scale_convert`` wraps ``flce_scale_convert``.
``LinearCrossEntropyLoss`` is the autograd front with the overview's
(weight, input, target) order.  Every output buffer handed to the library
is checked for shape, dtype, device and contiguity first, and each call runs
with its input's device current.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libflce.so")

FLCE_OK, FLCE_ERR_ARG, FLCE_ERR_ALIGN, FLCE_ERR_ARCH, FLCE_ERR_TARGET, \
    FLCE_ERR_WORKSPACE, FLCE_ERR_CUDA, FLCE_ERR_TIMEOUT = range(8)
FLCE_BF16, FLCE_FP32 = 0, 1
TRACE_KINDS = {1: "logits_lse", 2: "combine", 3: "logits_grad", 4: "dw", 5: "dx",
               6: "convert", 7: "ce_count", 8: "ce_rows"}

EXPORTED = ["flce_opts_init", "flce_fwd_bwd", "flce_fwd_bwd_ex", "flce_fwd",
            "flce_fwd_bwd_host", "flce_workspace_bytes", "flce_status_str",
            "flce_last_error", "flce_version", "flce_opts_sizeof", "flce_fwd_noalloc",
            "flce_ce_fwd_bwd", "flce_selftest_wait_expiry", "flce_scale_convert"]


class FlceOpts(ctypes.Structure):
    """Mirror of ``struct flce_opts`` (include/flce.h)."""
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("sync", ctypes.c_int32),
        ("stream", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("workspace_budget", ctypes.c_size_t),
        ("vocab_chunk", ctypes.c_int64),
        ("grad_scale", ctypes.c_float),
        ("target_is_int32", ctypes.c_int32),
        ("norm_count", ctypes.c_int64),
        ("loss_dev", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("loss_rows_out", ctypes.c_void_p),
        ("n_valid_dev", ctypes.c_void_p),
        ("status_dev", ctypes.c_void_p),
        ("workspace_used", ctypes.POINTER(ctypes.c_size_t)),
        ("vocab_chunk_used", ctypes.POINTER(ctypes.c_int64)),
        ("trace_events", ctypes.POINTER(ctypes.c_void_p)),
        ("trace_kinds", ctypes.POINTER(ctypes.c_int32)),
        ("trace_capacity", ctypes.c_int32),
        ("trace_count", ctypes.POINTER(ctypes.c_int32)),
    ]


class FlceError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libflce status {status}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load libflce (built in-tree by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libflce is not built ({p} missing): run "
                "`python -m linear_cross_entropy_fwd_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i64, i32, fp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        po = ctypes.POINTER(FlceOpts)
        lib.flce_opts_init.argtypes = [po]
        lib.flce_opts_init.restype = None
        lib.flce_fwd_bwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, fp, vp, vp]
        lib.flce_fwd_bwd.restype = i32
        lib.flce_fwd_bwd_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, fp, vp, vp, po]
        lib.flce_fwd_bwd_ex.restype = i32
        lib.flce_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, fp, po]
        lib.flce_fwd.restype = i32
        lib.flce_fwd_bwd_host.argtypes = [vp, vp, vp, i64, i64, i64, i64, fp, vp, vp, po]
        lib.flce_fwd_bwd_host.restype = i32
        lib.flce_workspace_bytes.argtypes = [i64, i64, i64, i32, po]
        lib.flce_workspace_bytes.restype = ctypes.c_size_t
        lib.flce_status_str.argtypes = [i32]
        lib.flce_status_str.restype = ctypes.c_char_p
        lib.flce_last_error.argtypes = []
        lib.flce_last_error.restype = ctypes.c_char_p
        lib.flce_version.argtypes = []
        lib.flce_version.restype = i32
        lib.flce_opts_sizeof.argtypes = []
        lib.flce_opts_sizeof.restype = ctypes.c_size_t
        lib.flce_fwd_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp]
        lib.flce_fwd_noalloc.restype = i32
        lib.flce_ce_fwd_bwd.argtypes = [vp, vp, i64, i64, i64, fp, vp, po]
        lib.flce_ce_fwd_bwd.restype = i32
        lib.flce_selftest_wait_expiry.argtypes = [i64]
        lib.flce_selftest_wait_expiry.restype = i32
        lib.flce_scale_convert.argtypes = [vp, i32, vp, i32, i64, vp, vp]
        lib.flce_scale_convert.restype = i32
        if lib.flce_opts_sizeof() != ctypes.sizeof(FlceOpts):
            raise RuntimeError("flce_opts layout mismatch between libflce and the binding")
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != FLCE_OK:
        lib = load_library()
        msg = lib.flce_last_error().decode() or lib.flce_status_str(status).decode()
        raise FlceError(status, msg)


def make_opts(dtype: torch.dtype = torch.bfloat16, stream=None, **kw) -> FlceOpts:
    """An initialised options struct; keyword arguments set fields by name."""
    lib = load_library()
    o = FlceOpts()
    lib.flce_opts_init(ctypes.byref(o))
    o.dtype = FLCE_FP32 if dtype == torch.float32 else FLCE_BF16
    if stream is not None:
        o.stream = stream
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FLCE_BF16
    if t.dtype == torch.float32:
        return FLCE_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _check_inputs(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor, device_needed=True):
    if X.dim() != 2 or W.dim() != 2 or target.dim() != 1:
        raise ValueError("X [N, H], W [V, H], target [N]")
    if X.shape[1] != W.shape[1] or X.shape[0] != target.shape[0]:
        raise ValueError(f"shape mismatch X{tuple(X.shape)} W{tuple(W.shape)} "
                         f"target{tuple(target.shape)}")
    if X.dtype != W.dtype:
        raise TypeError("X and W must share one dtype")
    if target.dtype not in (torch.int64, torch.int32):
        raise TypeError("target must be int64 or int32")
    for name, t in (("X", X), ("W", W), ("target", target)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if device_needed and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _is32(target: torch.Tensor) -> int:
    return 1 if target.dtype == torch.int32 else 0


def _check_out(t: torch.Tensor, shape, dtype: torch.dtype, device, name: str) -> None:
    """An output buffer the library writes: exact shape, dtype, device, and
    contiguous (the library is given only its address)."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{name} must be a {dtype} tensor of shape {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_row_outs(N: int, device, lse_out, loss_rows_out) -> None:
    if lse_out is not None:
        _check_out(lse_out, (N,), torch.float32, device, "lse_out")
    if loss_rows_out is not None:
        _check_out(loss_rows_out, (N,), torch.float32, device, "loss_rows_out")


def flce_fwd_bwd_ex(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor,
                    ignore_index: int = -100, *, dX: torch.Tensor | None = None,
                    dW: torch.Tensor | None = None, sync: bool = False,
                    grad_scale: float = 1.0, norm_count: int = 0,
                    lse_out: torch.Tensor | None = None,
                    loss_rows_out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, workspace_budget: int = 0,
                    vocab_chunk: int = 0, trace=None, info: dict | None = None):
    """Loss and gradients on the current CUDA stream.

    Returns (loss [0-d fp32 tensor on the device], n_valid [0-d int64], dX, dW).
    With ``sync=True`` the call blocks and kernel-side errors (bad targets,
    expired waits) raise ``FlceError``; otherwise check ``status`` afterwards
    through ``info['status']`` (a 0-d int32 device tensor)."""
    lib = load_library()
    _check_inputs(X, W, target)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if dX is None:
        dX = torch.empty_like(X)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    _check_out(dX, (N, H), X.dtype, dev, "dX")
    _check_out(dW, (V, H), torch.float32, dev, "dW")
    _check_row_outs(N, dev, lse_out, loss_rows_out)
    if workspace is not None:
        _check_out(workspace, (workspace.numel(),), workspace.dtype, dev, "workspace")
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nval = torch.empty((), dtype=torch.int64, device=dev)
    status = torch.zeros((), dtype=torch.int32, device=dev)
    o = make_opts(X.dtype, torch.cuda.current_stream(dev).cuda_stream,
                  sync=1 if sync else 0, grad_scale=float(grad_scale),
                  norm_count=int(norm_count), workspace_budget=int(workspace_budget),
                  vocab_chunk=int(vocab_chunk), target_is_int32=_is32(target))
    o.dtype = _dtype_code(X)
    o.loss_dev = loss.data_ptr()
    o.n_valid_dev = nval.data_ptr()
    o.status_dev = status.data_ptr()
    if lse_out is not None:
        o.lse_out = lse_out.data_ptr()
    if loss_rows_out is not None:
        o.loss_rows_out = loss_rows_out.data_ptr()
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    used = ctypes.c_size_t(0)
    vcu = ctypes.c_int64(0)
    o.workspace_used = ctypes.pointer(used)
    o.vocab_chunk_used = ctypes.pointer(vcu)
    keep = _attach_trace(o, trace)
    with torch.cuda.device(dev):
        st = lib.flce_fwd_bwd_ex(X.data_ptr(), W.data_ptr(), target.data_ptr(), N, H, V,
                                 int(ignore_index), None, dX.data_ptr(), dW.data_ptr(),
                                 ctypes.byref(o))
    del keep
    _check(st)
    if info is not None:
        info.update(workspace_bytes=used.value, vocab_chunk=vcu.value, status=status)
    return loss, nval, dX, dW


def flce_fwd_bwd(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor,
                 ignore_index: int = -100):
    """Synchronous loss and gradients through the simple C entry point.
    Returns (loss: float, dX, dW)."""
    lib = load_library()
    _check_inputs(X, W, target)
    if X.dtype != torch.bfloat16 or target.dtype != torch.int64:
        raise TypeError("flce_fwd_bwd takes bf16 inputs and int64 targets; use "
                        "flce_fwd_bwd_ex for fp32 inputs or int32 targets")
    N, H = X.shape
    V = W.shape[0]
    dX = torch.empty_like(X)
    dW = torch.empty((V, H), dtype=torch.float32, device=X.device)
    loss = ctypes.c_float(0.0)
    torch.cuda.current_stream(X.device).synchronize()  # the C call uses the default stream
    with torch.cuda.device(X.device):
        st = lib.flce_fwd_bwd(X.data_ptr(), W.data_ptr(), target.data_ptr(), N, H, V,
                              int(ignore_index), ctypes.byref(loss), dX.data_ptr(),
                              dW.data_ptr())
    _check(st)
    return loss.value, dX, dW


def flce_fwd(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor, ignore_index: int = -100,
             *, sync: bool = False, lse_out: torch.Tensor | None = None,
             loss_rows_out: torch.Tensor | None = None, norm_count: int = 0, trace=None,
             info: dict | None = None):
    """Loss only (no gradients).  Returns (loss 0-d device tensor, n_valid)."""
    lib = load_library()
    _check_inputs(X, W, target)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    _check_row_outs(N, dev, lse_out, loss_rows_out)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nval = torch.empty((), dtype=torch.int64, device=dev)
    status = torch.zeros((), dtype=torch.int32, device=dev)
    o = make_opts(X.dtype, torch.cuda.current_stream(dev).cuda_stream, sync=1 if sync else 0,
                  norm_count=int(norm_count), target_is_int32=_is32(target))
    o.dtype = _dtype_code(X)
    o.loss_dev = loss.data_ptr()
    o.n_valid_dev = nval.data_ptr()
    o.status_dev = status.data_ptr()
    if lse_out is not None:
        o.lse_out = lse_out.data_ptr()
    if loss_rows_out is not None:
        o.loss_rows_out = loss_rows_out.data_ptr()
    used = ctypes.c_size_t(0)
    o.workspace_used = ctypes.pointer(used)
    keep = _attach_trace(o, trace)
    with torch.cuda.device(dev):
        st = lib.flce_fwd(X.data_ptr(), W.data_ptr(), target.data_ptr(), N, H, V,
                          int(ignore_index), None, ctypes.byref(o))
    del keep
    _check(st)
    if info is not None:
        info.update(workspace_bytes=used.value, status=status)
    return loss, nval


def flce_fwd_noalloc(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor,
                     ignore_index: int = -100, *, loss: torch.Tensor | None = None,
                     lse_out: torch.Tensor | None = None, n_valid: torch.Tensor | None = None,
                     status: torch.Tensor | None = None):
    """Loss only, through the entry point that allocates no device memory
    inside the library (its scratch is a fixed 32 MiB static array; larger
    problems raise FlceError with FLCE_ERR_WORKSPACE).  For callers that plan
    device memory up front and cannot allocate at this point; pass
    preallocated ``loss`` (0-d fp32), ``n_valid`` (0-d int64) and ``status``
    (0-d int32) to keep the call itself allocation-free.  Calls share the
    library's scratch, so calls that may overlap on the GPU must be
    serialised.  Returns (loss, n_valid, status) device tensors."""
    lib = load_library()
    _check_inputs(X, W, target)
    if target.dtype != torch.int64:
        raise TypeError("flce_fwd_noalloc takes int64 targets")
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if loss is None:
        loss = torch.empty((), dtype=torch.float32, device=dev)
    if n_valid is None:
        n_valid = torch.empty((), dtype=torch.int64, device=dev)
    if status is None:
        status = torch.empty((), dtype=torch.int32, device=dev)
    _check_out(loss, (), torch.float32, dev, "loss")
    _check_out(n_valid, (), torch.int64, dev, "n_valid")
    _check_out(status, (), torch.int32, dev, "status")
    if lse_out is not None:
        _check_out(lse_out, (N,), torch.float32, dev, "lse_out")
    # the library picks its static scratch by the current device
    with torch.cuda.device(dev):
        st = lib.flce_fwd_noalloc(X.data_ptr(), W.data_ptr(), target.data_ptr(), N, H, V,
                                  int(ignore_index), _dtype_code(X), loss.data_ptr(),
                                  None if lse_out is None else lse_out.data_ptr(),
                                  n_valid.data_ptr(), status.data_ptr(),
                                  torch.cuda.current_stream(dev).cuda_stream)
    _check(st)
    return loss, n_valid, status


def flce_ce_fwd_bwd(logits: torch.Tensor, target: torch.Tensor, ignore_index: int = -100, *,
                    grad: bool = True, inplace: bool = False,
                    dlogits: torch.Tensor | None = None, sync: bool = False,
                    grad_scale: float = 1.0, norm_count: int = 0,
                    lse_out: torch.Tensor | None = None,
                    loss_rows_out: torch.Tensor | None = None, trace=None,
                    info: dict | None = None):
    """Cross-entropy on logits already in device memory [N, V] (bf16 or fp32).

    Returns (loss 0-d device tensor, n_valid 0-d int64, dlogits or None).
    ``inplace=True`` writes the gradient over ``logits``."""
    lib = load_library()
    if logits.dim() != 2 or target.dim() != 1 or logits.shape[0] != target.shape[0]:
        raise ValueError("logits [N, V], target [N]")
    if not (logits.is_cuda and target.is_cuda and logits.is_contiguous()
            and target.is_contiguous()):
        raise ValueError("contiguous CUDA tensors expected")
    if target.dtype not in (torch.int64, torch.int32):
        raise TypeError("target must be int64 or int32")
    N, V = logits.shape
    dev = logits.device
    if grad:
        if inplace:
            dlogits = logits
        elif dlogits is None:
            dlogits = torch.empty_like(logits)
    else:
        dlogits = None
    if dlogits is not None:
        _check_out(dlogits, (N, V), logits.dtype, dev, "dlogits")
    _check_row_outs(N, dev, lse_out, loss_rows_out)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    nval = torch.empty((), dtype=torch.int64, device=dev)
    status = torch.zeros((), dtype=torch.int32, device=dev)
    o = make_opts(logits.dtype, torch.cuda.current_stream(dev).cuda_stream,
                  sync=1 if sync else 0, grad_scale=float(grad_scale),
                  norm_count=int(norm_count), target_is_int32=_is32(target))
    o.dtype = _dtype_code(logits)
    o.loss_dev = loss.data_ptr()
    o.n_valid_dev = nval.data_ptr()
    o.status_dev = status.data_ptr()
    if lse_out is not None:
        o.lse_out = lse_out.data_ptr()
    if loss_rows_out is not None:
        o.loss_rows_out = loss_rows_out.data_ptr()
    used = ctypes.c_size_t(0)
    o.workspace_used = ctypes.pointer(used)
    keep = _attach_trace(o, trace)
    with torch.cuda.device(dev):
        st = lib.flce_ce_fwd_bwd(logits.data_ptr(), target.data_ptr(), N, V,
                                 int(ignore_index), None,
                                 None if dlogits is None else dlogits.data_ptr(),
                                 ctypes.byref(o))
    del keep
    _check(st)
    if info is not None:
        info.update(workspace_bytes=used.value, status=status)
    return loss, nval, dlogits


def flce_fwd_bwd_host(X: torch.Tensor, W: torch.Tensor, target: torch.Tensor,
                      ignore_index: int = -100, *, dX: torch.Tensor | None = None,
                      dW: torch.Tensor | None = None, stream=None, vocab_chunk: int = 0):
    """End to end on CPU tensors: the library copies the inputs in, runs, and
    copies loss, dX, dW out, overlapping the W upload with pass 1 and each
    chunk's dW download with the later chunks (pinned memory makes the copies
    asynchronous; pageable memory works but serialises them)."""
    lib = load_library()
    _check_inputs(X, W, target, device_needed=False)
    N, H = X.shape
    V = W.shape[0]
    if dX is None:
        dX = torch.empty_like(X)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32)
    loss = ctypes.c_float(0.0)
    o = make_opts(X.dtype, stream, vocab_chunk=int(vocab_chunk), target_is_int32=_is32(target))
    o.dtype = _dtype_code(X)
    st = lib.flce_fwd_bwd_host(X.data_ptr(), W.data_ptr(), target.data_ptr(), N, H, V,
                               int(ignore_index), ctypes.byref(loss), dX.data_ptr(),
                               dW.data_ptr(), ctypes.byref(o))
    _check(st)
    return loss.value, dX, dW


def flce_workspace_bytes(N: int, H: int, V: int, with_grads: bool = True,
                         dtype: torch.dtype = torch.bfloat16, workspace_budget: int = 0,
                         vocab_chunk: int = 0) -> int:
    lib = load_library()
    o = make_opts(dtype, workspace_budget=int(workspace_budget), vocab_chunk=int(vocab_chunk))
    return int(lib.flce_workspace_bytes(N, H, V, 1 if with_grads else 0, ctypes.byref(o)))


def scale_convert(src: torch.Tensor, dst: torch.Tensor,
                  scale: torch.Tensor | None = None) -> torch.Tensor:
    """dst = (dst.dtype)(src * scale) on the device in one pass (bf16 or
    fp32 each; ``scale`` a one-element fp32 device tensor, None for 1).
    ``dst`` may be ``src`` itself when the dtypes are equal.  Returns dst."""
    lib = load_library()
    if src.numel() != dst.numel() or not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous with the same number of elements")
    if src.device != dst.device or not src.is_cuda:
        raise ValueError("src and dst must be CUDA tensors on one device")
    if scale is not None:
        _check_out(scale, tuple(scale.shape), torch.float32, src.device, "scale")
        if scale.numel() != 1:
            raise ValueError("scale must hold one element")
    with torch.cuda.device(src.device):
        st = lib.flce_scale_convert(src.data_ptr(), _dtype_code(src), dst.data_ptr(),
                                    _dtype_code(dst), src.numel(),
                                    None if scale is None else scale.data_ptr(),
                                    torch.cuda.current_stream(src.device).cuda_stream)
    _check(st)
    return dst


class Trace:
    """Per-launch CUDA events recorded by the library on its stream."""

    def __init__(self, capacity: int = 1024):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        stream = torch.cuda.current_stream()
        for e in self.events:  # torch creates the CUDA event on first record
            e.record(stream)
        self.count = ctypes.c_int32(0)
        self.kinds = (ctypes.c_int32 * capacity)()
        self._ev = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.events])

    def launches(self):
        """[(kind name, milliseconds)] of the last traced call (after sync)."""
        out = []
        for k in range(1, self.count.value):
            out.append((TRACE_KINDS.get(self.kinds[k - 1], "?"),
                        self.events[k - 1].elapsed_time(self.events[k])))
        return out


def _attach_trace(o: FlceOpts, trace: Trace | None):
    if trace is None:
        return None
    o.trace_events = ctypes.cast(trace._ev, ctypes.POINTER(ctypes.c_void_p))
    o.trace_kinds = ctypes.cast(trace.kinds, ctypes.POINTER(ctypes.c_int32))
    o.trace_capacity = len(trace.events)
    o.trace_count = ctypes.pointer(trace.count)
    return (trace,)


def _grad_scale(grad_out: torch.Tensor) -> torch.Tensor:
    return grad_out.detach().to(torch.float32).reshape(1).contiguous()


class _FLCEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, weight, inp, target, ignore_index):
        loss, _, dX, dW = flce_fwd_bwd_ex(inp.contiguous(), weight.contiguous(),
                                          target.contiguous(), ignore_index)
        ctx.save_for_backward(dX, dW)
        ctx.w_dtype = weight.dtype
        return loss

    @staticmethod
    def backward(ctx, grad_out):
        # the gradients were computed in forward: scale them by grad_output
        # (and cast dW to the weight's dtype) in the library, one pass each
        dX, dW = ctx.saved_tensors
        g = _grad_scale(grad_out)
        gW = scale_convert(dW, torch.empty(dW.shape, dtype=ctx.w_dtype, device=dW.device), g)
        gX = scale_convert(dX, torch.empty_like(dX), g)
        return gW, gX, None, None


class _CEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, target, ignore_index):
        loss, _, dS = flce_ce_fwd_bwd(logits.contiguous(), target.contiguous(), ignore_index)
        ctx.save_for_backward(dS)
        return loss

    @staticmethod
    def backward(ctx, grad_out):
        (dS,) = ctx.saved_tensors
        return scale_convert(dS, torch.empty_like(dS), _grad_scale(grad_out)), None, None


class CrossEntropyLoss(torch.nn.Module):
    """loss_fn(logits, target) on logits already materialised (mean over
    non-ignored rows); forward computes the gradient as well."""

    def __init__(self, ignore_index: int = -100):
        super().__init__()
        self.ignore_index = ignore_index

    def forward(self, logits, target):
        return _CEFunction.apply(logits, target, self.ignore_index)


class LinearCrossEntropyLoss(torch.nn.Module):
    """loss_fn(weight, input, target) -> mean loss over non-ignored rows.

    Forward runs the whole fused path (loss and both gradients) in one call;
    backward scales the stored gradients by the incoming gradient."""

    def __init__(self, ignore_index: int = -100):
        super().__init__()
        self.ignore_index = ignore_index

    def forward(self, weight, inp, target):
        return _FLCEFunction.apply(weight, inp, target, self.ignore_index)
