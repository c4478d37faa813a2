"""Thin Python binding of libmsa.so (C ABI in include/msa.h).

Argument marshalling only: every step of the method runs in the CUDA library.  PyTorch supplies
device memory (tensors and the workspace) and the current stream.  There is no fallback: if the
library is missing or fails to load, every call raises.

Entry points (same names as the C ABI):
  msa_forward, msa_backward, msa_warmup_forward, msa_warmup_backward, msa_device_status,
  msa_workspace_size.
And the autograd pair mirroring the package API of Flash-MSA (``flash_msa_func`` /
``flash_msa_warmup_func``, PyPI page "Usage"): ``msa_func`` and ``msa_warmup_func`` return
``(attn_out, kl_loss)`` where kl_loss is a zero placeholder whose gradient drives the proxy
heads in the backward.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

OP_FORWARD, OP_BACKWARD, OP_WARMUP_FORWARD, OP_WARMUP_BACKWARD, OP_DECODE = 0, 1, 2, 3, 4
STATUS_BITS = {1: "bad block index", 2: "work list overflow", 4: "device wait timeout",
               8: "internal layout check"}
_SYMBOLS = ("msa_workspace_size", "msa_forward", "msa_backward", "msa_warmup_forward",
            "msa_warmup_backward", "msa_device_status", "msa_status_string", "msa_last_error",
            "msa_profile_begin", "msa_profile_end", "msa_launch_count", "msa_forward_noalloc",
            "msa_forward_noalloc_status", "msa_selftest_wait_timeout", "msa_decode")


class MSAError(RuntimeError):
    pass


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("Hp", ctypes.c_int32), ("D", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load libmsa.so (raises MSAError if it is missing: there is no CPU fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise MSAError(f"{path} not found: build it with block_sparse_attention_qp_gb300.build")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        SP = ctypes.POINTER(Shape)
        lib.msa_workspace_size.argtypes = [SP, I]
        lib.msa_workspace_size.restype = Z
        lib.msa_forward.argtypes = [SP, P, P, P, P, P, P, I, P, P, P, Z, P]
        lib.msa_backward.argtypes = [SP, P, P, P, P, P, P, P, P, P, F, P, P, P, P, P, P, P, P, Z,
                                     P]
        lib.msa_warmup_forward.argtypes = [SP, P, P, P, P, P, P, Z, P]
        lib.msa_warmup_backward.argtypes = [SP, P, P, P, P, P, P, P, P, F, P, P, P, P, P, P, P, P,
                                            Z, P]
        lib.msa_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint), P]
        lib.msa_decode.argtypes = [SP, P, P, P, P, P, P, P, P, P, P, Z, P]
        lib.msa_decode.restype = I
        lib.msa_status_string.argtypes = [I]
        lib.msa_status_string.restype = ctypes.c_char_p
        lib.msa_last_error.restype = ctypes.c_char_p
        for name in ("msa_forward", "msa_backward", "msa_warmup_forward", "msa_warmup_backward",
                     "msa_device_status", "msa_profile_begin", "msa_profile_end"):
            getattr(lib, name).restype = I
        lib.msa_profile_end.argtypes = [ctypes.c_char_p, Z]
        lib.msa_forward_noalloc.argtypes = [SP, P, P, P, P, P, P, I, P, P, P]
        lib.msa_forward_noalloc.restype = I
        lib.msa_forward_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_uint), P]
        lib.msa_forward_noalloc_status.restype = I
        lib.msa_launch_count.restype = ctypes.c_longlong
        lib.msa_selftest_wait_timeout.argtypes = [P, ctypes.c_uint, P]
        lib.msa_selftest_wait_timeout.restype = I
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        lib = load_library()
        raise MSAError(f"{what}: {lib.msa_status_string(rc).decode()} "
                       f"({lib.msa_last_error().decode()})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on_tensor_device(fn):
    """Runs fn with the CUDA device of its first tensor argument current, so that the library
    launches on the device that holds the data (with that device's current stream); every other
    tensor argument must be on the same device."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        tensors = [a for a in list(args) + list(kwargs.values()) if isinstance(a, torch.Tensor)]
        if not tensors or not tensors[0].is_cuda:
            return fn(*args, **kwargs)
        dev = tensors[0].device
        for t in tensors[1:]:
            if t.device != dev:
                raise MSAError(f"{fn.__name__}: tensors on {dev} and {t.device}; all arguments "
                               "must be on one device")
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return wrapper


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _req(t, name, dtype=torch.bfloat16, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise MSAError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MSAError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MSAError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise MSAError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def make_shape(q, k, qp, top_k, scale) -> Shape:
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    Hp = qp.shape[2] if qp is not None else Hkv
    return Shape(B, S, Hq, Hkv, Hp, D, int(top_k), float(scale))


def msa_workspace_size(shape: Shape, op: int) -> int:
    n = load_library().msa_workspace_size(ctypes.byref(shape), op)
    if n == 0:
        raise MSAError(f"unsupported shape for op {op}: "
                       f"{load_library().msa_last_error().decode()}")
    return int(n)


def workspace(shape: Shape, op: int, device) -> torch.Tensor:
    """Fresh workspace (uint8 tensor, 256-byte aligned by the CUDA caching allocator)."""
    return torch.empty(msa_workspace_size(shape, op), dtype=torch.uint8, device=device)


_WS_CACHE: dict = {}


def cached_workspace(shape: Shape, op: int, device) -> torch.Tensor:
    """Workspace kept per (device, current stream) and reused by later calls on that stream: the
    stream orders each call after the previous one, and no call leaves state in it that a later
    call reads.  Grows (never shrinks) to the largest size asked for; clear_workspace_cache()
    releases it."""
    device = torch.device(device)
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           torch.cuda.current_stream(device).cuda_stream)
    need = msa_workspace_size(shape, op)
    ws = _WS_CACHE.get(key)
    if ws is None or ws.numel() < need:
        _WS_CACHE.pop(key, None)
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        _WS_CACHE[key] = ws
    return ws


def clear_workspace_cache() -> None:
    _WS_CACHE.clear()


def _kl_grad_args(kl_grad, device):
    """(host value, device pointer) for the library's kl_grad / kl_grad_dev pair: a number is
    passed by value; a one-element fp32 tensor on the device is read by the kernel, so the host
    never waits for it."""
    if isinstance(kl_grad, torch.Tensor):
        if kl_grad.numel() != 1:
            raise MSAError(f"kl_grad must have one element, got shape {tuple(kl_grad.shape)}")
        if kl_grad.device != torch.device(device):
            raise MSAError(f"kl_grad is on {kl_grad.device}, the inputs on {device}")
        t = kl_grad.detach().reshape(()).to(torch.float32).contiguous()
        return 0.0, t
    return float(kl_grad), None


@_on_tensor_device
def msa_device_status(ws: torch.Tensor) -> int:
    """Read and clear the device status word of a workspace (synchronises the stream)."""
    flags = ctypes.c_uint(0)
    _check(load_library().msa_device_status(_ptr(ws), ctypes.byref(flags), _stream(ws.device)),
           "msa_device_status")
    return int(flags.value)


@_on_tensor_device
def selftest_wait_timeout(ws: torch.Tensor, limit_us: int = 1000) -> None:
    """Run the library's bounded-wait self-test on ws's device (see msa_selftest_wait_timeout);
    the timeout shows up in msa_device_status(ws)."""
    _check(load_library().msa_selftest_wait_timeout(_ptr(ws), int(limit_us), _stream(ws.device)),
           "msa_selftest_wait_timeout")


def profile_begin() -> None:
    """Start per-kernel CUDA-event timing inside the library (measurement aid)."""
    _check(load_library().msa_profile_begin(), "msa_profile_begin")


def profile_end() -> dict:
    """Stop timing; returns {kernel name: (launches, total milliseconds)}."""
    buf = ctypes.create_string_buffer(1 << 16)
    _check(load_library().msa_profile_end(buf, len(buf)), "msa_profile_end")
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        out[name] = (int(n), float(ms))
    return out


def launch_count() -> int:
    """Kernels launched by the library since it was loaded."""
    return int(load_library().msa_launch_count())


@_on_tensor_device
def msa_forward(q, k, v, qp, kp, top_k: int, scale: float, block_idx=None, ws=None):
    """Sparse forward.  Returns (o, lse, block_idx).  block_idx given -> used as the selection."""
    B, S, Hq, D = q.shape
    Hkv, Hp = k.shape[2], qp.shape[2]
    for t, n, shp in ((q, "q", None), (k, "k", (B, S, Hkv, D)), (v, "v", (B, S, Hkv, D)),
                      (qp, "qp", (B, S, Hp, D)), (kp, "kp", (B, S, 1, D))):
        _req(t, n, shape=shp)
    shape = make_shape(q, k, qp, top_k, scale)
    given = block_idx is not None
    if given:
        _req(block_idx, "block_idx", torch.int32, (B, Hp, S, top_k))
    else:
        block_idx = torch.empty((B, Hp, S, top_k), dtype=torch.int32, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, OP_FORWARD, q.device)
    _check(load_library().msa_forward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(qp),
                                      _ptr(kp), _ptr(block_idx), int(given), _ptr(o), _ptr(lse),
                                      _ptr(ws), ws.numel(), _stream(q.device)), "msa_forward")
    return o, lse, block_idx


@_on_tensor_device
def msa_forward_noalloc(q, k, v, qp, kp, top_k: int, scale: float, block_idx=None):
    """msa_forward without a workspace: the library's fixed device scratch array is used instead
    (see include/msa.h).  Returns (o, lse, block_idx)."""
    B, S, Hq, D = q.shape
    Hp = qp.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (qp, "qp"), (kp, "kp")):
        _req(t, n)
    shape = make_shape(q, k, qp, top_k, scale)
    given = block_idx is not None
    if given:
        _req(block_idx, "block_idx", torch.int32, (B, Hp, S, top_k))
    else:
        block_idx = torch.empty((B, Hp, S, top_k), dtype=torch.int32, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _check(load_library().msa_forward_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(qp), _ptr(kp), _ptr(block_idx), int(given),
                                              _ptr(o), _ptr(lse), _stream(q.device)),
           "msa_forward_noalloc")
    return o, lse, block_idx


def msa_forward_noalloc_status(device=None) -> int:
    """Read and clear the status word of the fixed scratch array msa_forward_noalloc uses on the
    current device (synchronises the current stream)."""
    flags = ctypes.c_uint(0)
    _check(load_library().msa_forward_noalloc_status(ctypes.byref(flags), _stream(device)),
           "msa_forward_noalloc_status")
    return int(flags.value)


@_on_tensor_device
def msa_backward(q, k, v, qp, kp, o, lse, dout, block_idx, top_k: int, scale: float,
                 kl_grad=1.0, ws=None, return_kl: bool = False):
    """Sparse backward.  Returns (dq, dk, dv, dqp, dkp), plus the KL value L_KL as a 0-d fp32
    CUDA tensor when return_kl (computed on the device; no host synchronisation).  kl_grad: a
    number, or a one-element tensor on the device (read by the kernel)."""
    B, S, Hq, D = q.shape
    Hp = qp.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (qp, "qp"), (kp, "kp"), (o, "o"), (dout, "dout")):
        _req(t, n)
    _req(lse, "lse", torch.float32, (B, Hq, S))
    _req(block_idx, "block_idx", torch.int32, (B, Hp, S, top_k))
    shape = make_shape(q, k, qp, top_k, scale)
    grads = [torch.empty_like(x) for x in (q, k, v, qp, kp)]
    kl = torch.empty((), dtype=torch.float32, device=q.device) if return_kl else None
    klg, klg_dev = _kl_grad_args(kl_grad, q.device)
    if ws is None:
        ws = workspace(shape, OP_BACKWARD, q.device)
    _check(load_library().msa_backward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(qp),
                                       _ptr(kp), _ptr(o), _ptr(lse), _ptr(dout), _ptr(block_idx),
                                       klg, _ptr(klg_dev), *map(_ptr, grads), _ptr(kl), _ptr(ws),
                                       ws.numel(), _stream(q.device)), "msa_backward")
    return tuple(grads) + ((kl,) if return_kl else ())


@_on_tensor_device
def msa_decode(q, qp, k_cache, v_cache, kp_cache, seq_len, top_k: int, scale: float, ws=None):
    """Decode step: q [B, Hq, D], qp [B, Hp, D] (the new tokens), caches k/v [B, S, Hkv, D] and
    kp [B, S, 1, D] (or [B, S, D]) already holding the new tokens at seq_len - 1, seq_len [B] int32
    on the device.  Returns (o [B, Hq, D], lse [B, Hq], block_idx [B, Hp, top_k])."""
    B, Hq, D = q.shape
    S, Hkv = k_cache.shape[1], k_cache.shape[2]
    Hp = qp.shape[1]
    for t, n in ((q, "q"), (qp, "qp"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (kp_cache, "kp_cache")):
        _req(t, n)
    _req(seq_len, "seq_len", torch.int32, (B,))
    shape = Shape(B, S, Hq, Hkv, Hp, D, int(top_k), float(scale))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    idx = torch.empty((B, Hp, top_k), dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(shape, OP_DECODE, q.device)
    _check(load_library().msa_decode(ctypes.byref(shape), _ptr(q), _ptr(qp), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(kp_cache), _ptr(seq_len), _ptr(idx),
                                     _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(q.device)),
           "msa_decode")
    return o, lse, idx


@_on_tensor_device
def msa_warmup_forward(q, k, v, scale: float, ws=None):
    """Dense causal forward (warmup).  Returns (o, lse)."""
    B, S, Hq, D = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _req(t, n)
    shape = make_shape(q, k, None, 0, scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, OP_WARMUP_FORWARD, q.device)
    _check(load_library().msa_warmup_forward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                             _stream(q.device)), "msa_warmup_forward")
    return o, lse


@_on_tensor_device
def msa_warmup_backward(q, k, v, qp, kp, o, lse, dout, scale: float, kl_grad=1.0,
                        ws=None, return_kl: bool = False):
    """Dense warmup backward (proxy KL over the full causal prefix).  Returns grads (and the KL
    value as a 0-d fp32 CUDA tensor when return_kl).  kl_grad as in msa_backward."""
    B, S, Hq, D = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (qp, "qp"), (kp, "kp"), (o, "o"), (dout, "dout")):
        _req(t, n)
    _req(lse, "lse", torch.float32, (B, Hq, S))
    shape = make_shape(q, k, qp, 0, scale)
    grads = [torch.empty_like(x) for x in (q, k, v, qp, kp)]
    kl = torch.empty((), dtype=torch.float32, device=q.device) if return_kl else None
    klg, klg_dev = _kl_grad_args(kl_grad, q.device)
    if ws is None:
        ws = workspace(shape, OP_WARMUP_BACKWARD, q.device)
    _check(load_library().msa_warmup_backward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(qp), _ptr(kp), _ptr(o), _ptr(lse), _ptr(dout),
                                              klg, _ptr(klg_dev), *map(_ptr, grads), _ptr(kl),
                                              _ptr(ws), ws.numel(), _stream(q.device)),
           "msa_warmup_backward")
    return tuple(grads) + ((kl,) if return_kl else ())


class _MSAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qp, kp, q, k, v, top_k, scale, warmup):
        qp, kp, q, k, v = (x.contiguous() for x in (qp, kp, q, k, v))
        if warmup:
            o, lse = msa_warmup_forward(
                q, k, v, scale,
                ws=cached_workspace(make_shape(q, k, None, 0, scale), OP_WARMUP_FORWARD, q.device))
            idx = None
        else:
            o, lse, idx = msa_forward(
                q, k, v, qp, kp, top_k, scale,
                ws=cached_workspace(make_shape(q, k, qp, top_k, scale), OP_FORWARD, q.device))
        ctx.save_for_backward(qp, kp, q, k, v, o, lse, *(() if idx is None else (idx,)))
        ctx.top_k, ctx.scale, ctx.warmup = top_k, scale, warmup
        kl = torch.zeros((), dtype=torch.float32, device=q.device)
        return o, kl

    @staticmethod
    def backward(ctx, do, dkl):
        saved = ctx.saved_tensors
        qp, kp, q, k, v, o, lse = saved[:7]
        kl_grad = 0.0 if dkl is None else dkl  # a device tensor: read by the kernel, no sync
        do = torch.zeros_like(o) if do is None else do.contiguous()
        if ctx.warmup:
            ws = cached_workspace(make_shape(q, k, qp, 0, ctx.scale), OP_WARMUP_BACKWARD, q.device)
            dq, dk, dv, dqp, dkp = msa_warmup_backward(q, k, v, qp, kp, o, lse, do, ctx.scale,
                                                       kl_grad, ws=ws)
        else:
            ws = cached_workspace(make_shape(q, k, qp, ctx.top_k, ctx.scale), OP_BACKWARD,
                                  q.device)
            dq, dk, dv, dqp, dkp = msa_backward(q, k, v, qp, kp, o, lse, do, saved[7], ctx.top_k,
                                                ctx.scale, kl_grad, ws=ws)
        return dqp, dkp, dq, dk, dv, None, None, None


def msa_func(Q_proxy, K_proxy, Q, K, V, top_k: int, scale: float):
    """Sparse MSA attention with the Flash-MSA call convention.  Returns (attn_out, kl_loss);
    add kl_loss to the training loss so that backward() trains the proxy heads."""
    return _MSAFunction.apply(Q_proxy, K_proxy, Q, K, V, int(top_k), float(scale), False)


def msa_warmup_func(Q_proxy, K_proxy, Q, K, V, top_k: int, scale: float):
    """Warmup mode: dense main attention, proxy trained over the full causal prefix."""
    return _MSAFunction.apply(Q_proxy, K_proxy, Q, K, V, int(top_k), float(scale), True)
