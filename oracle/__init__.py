"""fp64 CPU oracle for MiniMax Sparse Attention (MSA) training -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product library never loads it; it shares no code with the CUDA path.

The arithmetic lives in ``msa_oracle.c`` (plain loops, fp64).  This module compiles it with gcc,
loads it with ctypes and converts numpy / torch arrays to the float64 layouts it expects.  Each
wrapper names the steps of the method it runs; the step list and its sources (the Flash-MSA blog
and the MSA forum summary) are at the top of ``msa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128  # key-block size fixed by the method ("blocks of 128")


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmsa_oracle.so`` (portable: no -march flags)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            Dd = ctypes.c_double
            lib.msa_oracle_select.argtypes = [I, I, I, I, I, Dd, P, P, I, P, P, P]
            lib.msa_oracle_forward.argtypes = [I, I, I, I, I, I, I, Dd, P, P, P, P, I, P, P, P]
            lib.msa_oracle_backward.argtypes = [I, I, I, I, I, I, I, Dd, Dd, P, P, P, P, P, P, P,
                                                P, I, I, I, P, P, P, P, P, P]
            lib.msa_oracle_threads.restype = I
            lib.msa_oracle_set_threads.argtypes = [I]
            _lib = lib
    return _lib


class use_library:
    """Temporarily route every wrapper through another build of the oracle source (used by the
    tests that plant mistakes in a copy of ``msa_oracle.c`` to show that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("msa_oracle_select", "msa_oracle_forward", "msa_oracle_backward"):
            getattr(lib, name).argtypes = getattr(self.saved, name).argtypes
        _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (test use only)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o",
                           out_path, src, "-lm"])
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return _load().msa_oracle_threads()


def set_threads(n: int) -> None:
    _load().msa_oracle_set_threads(int(n))


def f64(x) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype, e.g. bf16) or array to contiguous fp64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only needed for tensors
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def select(qp, kp, top_k: int, scale: float, rows=None):
    """Steps 1-3 (proxy scores, causal block max-pool with the local block forced, top-k).

    qp: [B,S,Hp,D], kp: [B,S,1,D] or [B,S,D].  rows: optional int array [n,3] of (b, g, t).
    Returns (idx, gap): idx int32 [B,Hp,S,top_k] (or [n,top_k]), ascending and -1 padded;
    gap float64 [B,Hp,S] (or [n]): relative gap between the lowest selected and the highest
    unselected non-local block score (inf when nothing could flip).
    """
    qp = f64(qp)
    kp = f64(kp)
    B, S, Hp, D = qp.shape
    kp = kp.reshape(B, S, D)
    if rows is None:
        idx = np.empty((B, Hp, S, top_k), np.int32)
        gap = np.empty((B, Hp, S), np.float64)
        n, r = 0, None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        n = r.shape[0]
        idx = np.empty((n, top_k), np.int32)
        gap = np.empty((n,), np.float64)
    rc = _load().msa_oracle_select(B, S, Hp, D, top_k, float(scale), _p(qp), _p(kp), n, _p(r),
                                   _p(idx), _p(gap))
    if rc:
        raise ValueError(f"oracle select rejected the shape (code {rc})")
    return idx, gap


def forward(q, k, v, idx, top_k: int, scale: float, rows=None, Hp=None):
    """Steps 4-5 (key set and main attention).  idx=None: warmup (dense causal).

    q [B,S,Hq,D], k/v [B,S,Hkv,D], idx int32 [B,Hp,S,top_k] (query head h uses the selection of
    proxy head h / (Hq/Hp) and the keys of KV head h / (Hq/Hkv)).  rows: optional [n,3] (b, t, h).
    Returns (o, lse): o [B,S,Hq,D], lse [B,Hq,S] (or [n,D], [n]).
    """
    q, k, v = f64(q), f64(k), f64(v)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if idx is not None:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        top_k = idx.shape[-1]
        if Hp is None:
            Hp = idx.shape[1]  # the map's proxy heads
    Hp = Hkv if Hp is None else Hp
    if rows is None:
        o = np.empty((B, S, Hq, D), np.float64)
        lse = np.empty((B, Hq, S), np.float64)
        n, r = 0, None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        n = r.shape[0]
        o = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
    rc = _load().msa_oracle_forward(B, S, Hq, Hkv, Hp, D, top_k, float(scale), _p(q), _p(k),
                                    _p(v), _p(idx), n, _p(r), _p(o), _p(lse))
    if rc:
        raise ValueError(f"oracle forward rejected the shape (code {rc})")
    return o, lse


def backward(q, k, v, qp, kp, dout, idx, top_k: int, scale: float, kl_grad: float = 1.0,
             tok_mask=None, key_window=None, only_masked=False):
    """Steps 4-10: gradients of  sum(O*dO) + kl_grad * L_KL  and the KL value.

    idx=None: warmup (dense causal key sets).  tok_mask: optional bool [B,S] -- dq/dqp are only
    produced for flagged tokens.  key_window: optional (j0, j1) -- dk/dv/dkp only for keys in
    [j0, j1).  only_masked: tokens outside tok_mask contribute nothing at all (exact share of
    the flagged tokens in every gradient).  Entries outside the sample are zero.
    Returns dict(dq, dk, dv, dqp, dkp, kl) in the input layouts (dkp [B,S,1,D]).
    """
    q, k, v, qp, kp, dout = f64(q), f64(k), f64(v), f64(qp), f64(kp), f64(dout)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    Hp = qp.shape[2]
    kp = kp.reshape(B, S, D)
    if idx is not None:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        top_k = idx.shape[-1]
    dq = np.zeros(q.shape, np.float64)  # np.zeros maps lazily-zeroed pages: sampled runs on long
    dk = np.zeros(k.shape, np.float64)  # sequences only touch the rows they write
    dv = np.zeros(v.shape, np.float64)
    dqp = np.zeros(qp.shape, np.float64)
    dkp = np.zeros((B, S, D), np.float64)
    kl = np.zeros((1,), np.float64)
    tm = None if tok_mask is None else np.ascontiguousarray(tok_mask, dtype=np.uint8)
    j0, j1 = (0, S) if key_window is None else (int(key_window[0]), int(key_window[1]))
    rc = _load().msa_oracle_backward(B, S, Hq, Hkv, Hp, D, top_k, float(scale), float(kl_grad),
                                     _p(q), _p(k), _p(v), _p(qp), _p(kp), _p(dout), _p(idx),
                                     _p(tm), int(bool(only_masked)), j0, j1, _p(dq), _p(dk), _p(dv), _p(dqp), _p(dkp),
                                     _p(kl))
    if rc:
        raise ValueError(f"oracle backward rejected the shape (code {rc})")
    return dict(dq=dq, dk=dk, dv=dv, dqp=dqp, dkp=dkp.reshape(B, S, 1, D), kl=float(kl[0]))
