"""The allocation-free forward entry point (msa_forward_noalloc), called through the C ABI.

Some callers cannot allocate device memory where they call the forward (a C layer whose host
framework owns the allocator, or code recording launches for later replay, where allocation is
not allowed).  msa_forward_noalloc serves them from a fixed 64 MiB device array instead of a
workspace.  This file runs last so that, if it fails, every other test has already run.
"""
import ctypes

import pytest
import torch

from block_sparse_attention_qp_gb300 import binding as msa
from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs
from tests.parity import close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _call_noalloc(lib, shape, g, top_k, block_idx, given, o, lse):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.msa_forward_noalloc(ctypes.byref(shape), p(g["q"]), p(g["k"]), p(g["v"]), p(g["qp"]),
                                   p(g["kp"]), p(block_idx), int(given), p(o), p(lse),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_forward_matches_workspace_forward():
    lib = msa.load_library()
    w = Workload("noalloc", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4)
    x = make_inputs(w, 4242)
    g = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o_ref, lse_ref, idx_ref = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k,
                                              w.scale)
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    for _ in range(2):  # two calls in a row share the fixed scratch array
        idx = torch.full_like(idx_ref, -7)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(lse_ref)
        rc = _call_noalloc(lib, shape, g, w.top_k, idx, 0, o, lse)
        assert rc == 0, lib.msa_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref)
        close("O", o, o_ref.float(), rel=1e-5, atol=2e-3, ulps=1.0)
        close("LSE", lse, lse_ref, rel=1e-6, atol=1e-5, ulps=0.0)
    # with the selection given as input
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    assert _call_noalloc(lib, shape, g, w.top_k, idx_ref, 1, o, lse) == 0
    torch.cuda.synchronize()
    close("O", o, o_ref.float(), rel=1e-5, atol=2e-3, ulps=1.0)


def test_noalloc_rejects_shapes_beyond_the_fixed_array():
    lib = msa.load_library()
    big = msa.Shape(2, 8192, 32, 8, 8, 128, 16, 128 ** -0.5)  # needs ~2 GB of scratch
    null = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    rc = lib.msa_forward_noalloc(ctypes.byref(big), null, null, null, null, null, null, 0, null,
                                 null, None)
    assert rc == 3  # MSA_ERR_WORKSPACE
    assert b"scratch" in lib.msa_last_error()
