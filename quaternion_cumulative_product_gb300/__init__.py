"""Quaternion cumulative-product scan on GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/quat_cumprod.h`` (library
``libquatscan.so`` next to this file).  The binding only checks and marshals
arguments: every step of the scan runs in the library's CUDA kernels.  PyTorch
provides device memory and the current stream.  There is no CPU fallback: if
the library is missing or the device is not sm_103, calls raise.

Operation (burn-mamba ``mamba3/quat_scan/backward.rs``, "Gradient math"):
``cum[t] = q_t (x) cum[t-1]`` with ``cum[-1] = init`` over ``[B,S,H,J,4]``
fp32 tensors, and its vector-Jacobian product ``(d_q, d_init)`` recomputed
from ``(q, init, d_cum)``.

Calls: ``quat_cumprod_fwd`` / ``quat_cumprod_bwd`` (the page's operation),
``quat_cumprod_fwd_carries`` / ``quat_cumprod_bwd_carries`` (keep the 64-step
chunk carries between the two), ``quat_cumprod_fwd_bf16`` /
``quat_cumprod_bwd_bf16`` (bfloat16 tensors), ``quat_cumprod_bwd_noalloc``
(no allocation), ``quat_cumprod_fwd_bwd_host`` (a whole step on host
tensors, copies overlapped with the kernels), ``quat_cumprod_plan`` and
``quat_cumprod_status``.  The
autograd wrapper is in :mod:`quaternion_cumulative_product_gb300.autograd`.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

__all__ = [
    "QS_OK", "QS_ERR_NULL", "QS_ERR_DIMS", "QS_ERR_MISALIGNED", "QS_ERR_ALIAS",
    "QS_ERR_CUDA", "QS_ERR_TIMEOUT", "QS_ERR_NOMEM", "QS_ERR_DEVICE", "QS_ERR_SCRATCH",
    "QS_NOALLOC_MAX_TILES", "QS_CARRY_STEPS", "QuatScanError", "library_path", "load_library",
    "quat_cumprod_fwd", "quat_cumprod_bwd", "quat_cumprod_fwd_carries", "quat_cumprod_bwd_carries",
    "quat_cumprod_fwd_bf16", "quat_cumprod_bwd_bf16",
    "quat_cumprod_bwd_noalloc", "quat_cumprod_fwd_bwd_host", "quat_cumprod_plan", "quat_cumprod_status",
    "quat_cumprod_strerror",
]

QS_OK = 0
QS_ERR_NULL = -1
QS_ERR_DIMS = -2
QS_ERR_MISALIGNED = -3
QS_ERR_ALIAS = -4
QS_ERR_CUDA = -5
QS_ERR_TIMEOUT = -6
QS_ERR_NOMEM = -7
QS_ERR_DEVICE = -8
QS_ERR_SCRATCH = -9

# Steps per chunk of the carries written by quat_cumprod_fwd_carries.
QS_CARRY_STEPS = 64

# Work tiles (B * ceil(H*J/32) * ceil(S/64)) that quat_cumprod_bwd_noalloc's
# fixed scratch array holds.
QS_NOALLOC_MAX_TILES = 8192

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libquatscan.so"
_lock = threading.Lock()
_lib = None


class QuatScanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {quat_cumprod_strerror(status)} (status {status})")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library():
    """Loads ``libquatscan.so`` (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:   # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.quat_cumprod_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_fwd.restype = ctypes.c_int
        lib.quat_cumprod_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_bwd.restype = ctypes.c_int
        lib.quat_cumprod_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_bwd_noalloc.restype = ctypes.c_int
        lib.quat_cumprod_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_fwd_bwd_host.restype = ctypes.c_int
        lib.quat_cumprod_fwd_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_fwd_bf16.restype = ctypes.c_int
        lib.quat_cumprod_bwd_bf16.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_bwd_bf16.restype = ctypes.c_int
        lib.quat_cumprod_fwd_carries.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_fwd_carries.restype = ctypes.c_int
        lib.quat_cumprod_bwd_carries.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.quat_cumprod_bwd_carries.restype = ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        lib.quat_cumprod_plan.argtypes = [ctypes.c_int, i64, i64, i64, i64, ip, ip]
        lib.quat_cumprod_plan.restype = ctypes.c_int
        lib.quat_cumprod_status.argtypes = [vp]
        lib.quat_cumprod_status.restype = ctypes.c_int
        lib.quat_cumprod_strerror.argtypes = [ctypes.c_int]
        lib.quat_cumprod_strerror.restype = ctypes.c_char_p
        lib.quat_cumprod_debug_set_timeout_ns.argtypes = [i64]
        lib.quat_cumprod_debug_set_timeout_ns.restype = ctypes.c_int
        lib.quat_cumprod_debug_stall_tile.argtypes = [i64]
        lib.quat_cumprod_debug_stall_tile.restype = ctypes.c_int
        lib.quat_cumprod_debug_set_variant.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.quat_cumprod_debug_set_variant.restype = ctypes.c_int
        lib.quat_cumprod_debug_set_walk_cap.argtypes = [ctypes.c_int64]
        lib.quat_cumprod_debug_set_walk_cap.restype = ctypes.c_int
        lib.quat_cumprod_debug_set_variant_bf16.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.quat_cumprod_debug_set_variant_bf16.restype = ctypes.c_int
        _lib = lib
        return lib


def quat_cumprod_strerror(status: int) -> str:
    return load_library().quat_cumprod_strerror(int(status)).decode()


_torch_mod = None
_NULL_CONTEXT = contextlib.nullcontext()


def _torch():
    global _torch_mod
    if _torch_mod is None:
        import torch
        _torch_mod = torch
    return _torch_mod


def _on_device(device):
    """The CUDA device context for a call on ``device``; none when it is already current."""
    torch = _torch()
    if device.index is None or torch.cuda.current_device() == device.index:
        return _NULL_CONTEXT
    return torch.cuda.device(device)


def _stream_handle(stream, device):
    """The cudaStream_t of ``stream``, else of the current torch stream on ``device``."""
    torch = _torch()
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)   # no Stream object per call
    if raw is not None:
        index = device.index if device.index is not None else torch.cuda.current_device()
        return ctypes.c_void_p(raw(index))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_tensor(name, t, shape, device=None, dtype=None):
    torch = _torch()
    dtype = torch.float32 if dtype is None else dtype
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q, init, dtype=None):
    if q.dim() != 5 or q.shape[-1] != 4:
        raise ValueError(f"q must be [B,S,H,J,4], got {tuple(q.shape)}")
    B, S, H, J, _ = q.shape
    _check_tensor("q", q, (B, S, H, J, 4), dtype=dtype)
    _check_tensor("init", init, (B, H, J, 4), q.device, dtype)
    return B, S, H, J


def quat_cumprod_fwd(q, init, cum=None, stream=None):
    """cum[b,t,h,j] = q[b,t,h,j] (x) cum[b,t-1,h,j], cum[b,-1,h,j] = init[b,h,j].

    ``q``: [B,S,H,J,4] float32 CUDA, ``init``: [B,H,J,4]; ``cum`` (optional
    output) has the shape of ``q``.  Enqueued on ``stream`` (default: the
    current torch stream).  Returns ``cum``.
    """
    torch = _torch()
    B, S, H, J = _dims(q, init)
    if cum is None:
        cum = torch.empty_like(q)
    else:
        _check_tensor("cum", cum, q.shape, q.device)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_fwd(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()),
            ctypes.c_void_p(cum.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_fwd")
    return cum


def quat_cumprod_bwd(q, init, d_cum, d_q=None, d_init=None, stream=None):
    """(d_q, d_init): vector-Jacobian product of the scan for the cotangent ``d_cum``.

    Recomputed from the leaves ``q``, ``init`` (nothing is saved by the forward).
    Returns ``(d_q, d_init)`` with the shapes of ``q`` and ``init``.
    """
    torch = _torch()
    B, S, H, J = _dims(q, init)
    _check_tensor("d_cum", d_cum, q.shape, q.device)
    if d_q is None:
        d_q = torch.empty_like(q)
    else:
        _check_tensor("d_q", d_q, q.shape, q.device)
    if d_init is None:
        d_init = torch.empty_like(init)
    else:
        _check_tensor("d_init", d_init, init.shape, q.device)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_bwd(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()),
            ctypes.c_void_p(d_cum.data_ptr()), ctypes.c_void_p(d_q.data_ptr()),
            ctypes.c_void_p(d_init.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_bwd")
    return d_q, d_init


def quat_cumprod_fwd_bf16(q, init, cum=None, stream=None):
    """``quat_cumprod_fwd`` on bfloat16 tensors (fp32 arithmetic, outputs rounded once)."""
    torch = _torch()
    B, S, H, J = _dims(q, init, torch.bfloat16)
    if cum is None:
        cum = torch.empty_like(q)
    else:
        _check_tensor("cum", cum, q.shape, q.device, torch.bfloat16)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_fwd_bf16(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()),
            ctypes.c_void_p(cum.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_fwd_bf16")
    return cum


def quat_cumprod_bwd_bf16(q, init, d_cum, d_q=None, d_init=None, stream=None):
    """``quat_cumprod_bwd`` on bfloat16 tensors.  Returns ``(d_q, d_init)`` (bfloat16)."""
    torch = _torch()
    B, S, H, J = _dims(q, init, torch.bfloat16)
    _check_tensor("d_cum", d_cum, q.shape, q.device, torch.bfloat16)
    if d_q is None:
        d_q = torch.empty_like(q)
    else:
        _check_tensor("d_q", d_q, q.shape, q.device, torch.bfloat16)
    if d_init is None:
        d_init = torch.empty_like(init)
    else:
        _check_tensor("d_init", d_init, init.shape, q.device, torch.bfloat16)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_bwd_bf16(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()),
            ctypes.c_void_p(d_cum.data_ptr()), ctypes.c_void_p(d_q.data_ptr()),
            ctypes.c_void_p(d_init.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_bwd_bf16")
    return d_q, d_init


def _carries_shape(q):
    B, S, H, J, _ = q.shape
    return (B, (S + QS_CARRY_STEPS - 1) // QS_CARRY_STEPS, H, J, 4)


def quat_cumprod_fwd_carries(q, init, cum=None, carries=None, stream=None):
    """``quat_cumprod_fwd`` that also returns the chunk carries.

    ``carries[b, c] = cum[b, c*QS_CARRY_STEPS - 1]`` (``init`` for ``c = 0``),
    shape ``[B, ceil(S/64), H, J, 4]``.  Returns ``(cum, carries)``.
    """
    torch = _torch()
    B, S, H, J = _dims(q, init)
    if cum is None:
        cum = torch.empty_like(q)
    else:
        _check_tensor("cum", cum, q.shape, q.device)
    if carries is None:
        carries = torch.empty(_carries_shape(q), dtype=q.dtype, device=q.device)
    else:
        _check_tensor("carries", carries, _carries_shape(q), q.device)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_fwd_carries(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()), ctypes.c_void_p(cum.data_ptr()),
            ctypes.c_void_p(carries.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_fwd_carries")
    return cum, carries


def quat_cumprod_bwd_carries(q, carries, d_cum, d_q=None, d_init=None, stream=None):
    """``quat_cumprod_bwd`` from the carries of ``quat_cumprod_fwd_carries``.

    Returns ``(d_q, d_init)``; ``d_init`` has the shape ``[B, H, J, 4]``.
    """
    torch = _torch()
    if q.dim() != 5 or q.shape[-1] != 4:
        raise ValueError(f"q must be [B,S,H,J,4], got {tuple(q.shape)}")
    B, S, H, J, _ = q.shape
    _check_tensor("q", q, q.shape)
    _check_tensor("carries", carries, _carries_shape(q), q.device)
    _check_tensor("d_cum", d_cum, q.shape, q.device)
    if d_q is None:
        d_q = torch.empty_like(q)
    else:
        _check_tensor("d_q", d_q, q.shape, q.device)
    if d_init is None:
        d_init = torch.empty((B, H, J, 4), dtype=q.dtype, device=q.device)
    else:
        _check_tensor("d_init", d_init, (B, H, J, 4), q.device)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_bwd_carries(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(carries.data_ptr()),
            ctypes.c_void_p(d_cum.data_ptr()), ctypes.c_void_p(d_q.data_ptr()),
            ctypes.c_void_p(d_init.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_bwd_carries")
    return d_q, d_init


def quat_cumprod_bwd_noalloc(q, init, d_cum, d_q, d_init, stream=None):
    """``quat_cumprod_bwd`` into caller-owned ``d_q`` and ``d_init``, with no allocation.

    For callers that must not allocate device memory at this point: the
    library call uses a fixed scratch array of the library instead of a
    cudaMalloc'ed workspace, and this wrapper allocates no tensor either.  The
    sizes must satisfy ``B * ceil(H*J/32) * ceil(S/64) <= QS_NOALLOC_MAX_TILES``.
    All calls on one device share the scratch: calls whose work can overlap on
    the GPU (unordered streams) race.  Returns ``(d_q, d_init)``.
    """
    torch = _torch()
    B, S, H, J = _dims(q, init)
    _check_tensor("d_cum", d_cum, q.shape, q.device)
    _check_tensor("d_q", d_q, q.shape, q.device)
    _check_tensor("d_init", d_init, init.shape, q.device)
    with _on_device(q.device):
        rc = load_library().quat_cumprod_bwd_noalloc(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()),
            ctypes.c_void_p(d_cum.data_ptr()), ctypes.c_void_p(d_q.data_ptr()),
            ctypes.c_void_p(d_init.data_ptr()), B, S, H, J, _stream_handle(stream, q.device))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_bwd_noalloc")
    return d_q, d_init


def _check_host(name, t, shape):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def quat_cumprod_fwd_bwd_host(q, init, d_cum, cum=None, d_q=None, d_init=None, device=None, stream=None,
                              synchronize=True):
    """One forward + backward step on host tensors: ``(cum, d_q, d_init)``.

    ``q``, ``init``, ``d_cum``: CPU float32 tensors ([B,S,H,J,4], [B,H,J,4],
    [B,S,H,J,4]); page-locked (``pin_memory()``) tensors let the copies to
    and from the GPU overlap the kernels.  Outputs are allocated page-locked
    when not given.  The step runs on ``device`` (default: the current CUDA
    device) and is enqueued on ``stream``; with ``synchronize`` (default) the
    call returns once the outputs are complete, otherwise the caller
    synchronizes ``stream`` before touching any of the six tensors.
    """
    torch = _torch()
    if q.dim() != 5 or q.shape[-1] != 4:
        raise ValueError(f"q must be [B,S,H,J,4], got {tuple(q.shape)}")
    B, S, H, J, _ = q.shape
    _check_host("q", q, q.shape)
    _check_host("init", init, (B, H, J, 4))
    _check_host("d_cum", d_cum, q.shape)
    cum = torch.empty(q.shape, dtype=torch.float32).pin_memory() if cum is None else cum
    d_q = torch.empty(q.shape, dtype=torch.float32).pin_memory() if d_q is None else d_q
    d_init = torch.empty(init.shape, dtype=torch.float32).pin_memory() if d_init is None else d_init
    _check_host("cum", cum, q.shape)
    _check_host("d_q", d_q, q.shape)
    _check_host("d_init", d_init, init.shape)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        handle = _stream_handle(stream, device)
        rc = load_library().quat_cumprod_fwd_bwd_host(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(init.data_ptr()), ctypes.c_void_p(d_cum.data_ptr()),
            ctypes.c_void_p(cum.data_ptr()), ctypes.c_void_p(d_q.data_ptr()), ctypes.c_void_p(d_init.data_ptr()),
            B, S, H, J, handle)
        if rc != QS_OK:
            raise QuatScanError(rc, "quat_cumprod_fwd_bwd_host")
        if synchronize:
            (torch.cuda.current_stream(device) if stream is None else stream).synchronize()
    return cum, d_q, d_init


_PLAN_CALLS = {"fwd": 0, "bwd": 1, "fwd_carries": 2, "bwd_carries": 3, "fwd_bf16": 4, "bwd_bf16": 5}


def quat_cumprod_plan(call, B, S, H, J, device=None):
    """(variant, kernels) a call with these sizes would use on ``device`` (launches nothing).

    ``call``: ``"fwd"``, ``"bwd"``, ``"fwd_carries"``, ``"bwd_carries"`` (or
    False / True for the first two).
    """
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    code = _PLAN_CALLS[call] if isinstance(call, str) else int(bool(call))
    v, k = ctypes.c_int(0), ctypes.c_int(0)
    with torch.cuda.device(device):
        rc = load_library().quat_cumprod_plan(code, B, S, H, J, ctypes.byref(v), ctypes.byref(k))
    if rc != QS_OK:
        raise QuatScanError(rc, "quat_cumprod_plan")
    return v.value, k.value


def quat_cumprod_status(stream=None, device=None):
    """Synchronizes the stream and returns its recorded status (QS_OK or an error code)."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return load_library().quat_cumprod_status(_stream_handle(stream, device))
