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


def _fresh_forward(w, g, idx=None):
    """msa_forward on a workspace of its own (the comparison for the fixed-array calls)."""
    return msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                           block_idx=idx)


def test_noalloc_shapes_in_turn_leave_no_stale_state():
    """A larger call, then a smaller one with other head counts and top_k, then the first shape
    again: each must match msa_forward on a fresh workspace, so nothing a call leaves in the
    shared array (longer lists, more work items) leaks into the next."""
    lib = msa.load_library()
    cases = [Workload("big", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4),
             Workload("small", B=1, S=512, Hq=16, Hkv=4, Hp=4, top_k=2),
             Workload("big", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4)]
    for n, w in enumerate(cases):
        x = make_inputs(w, 900 + n)
        g = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
        o_ref, lse_ref, idx_ref = _fresh_forward(w, g)
        shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
        idx = torch.full_like(idx_ref, -7)
        o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
        assert _call_noalloc(lib, shape, g, w.top_k, idx, 0, o, lse) == 0, lib.msa_last_error()
        assert msa.msa_forward_noalloc_status() == 0
        assert torch.equal(idx, idx_ref), w.name
        close("O " + w.name, o, o_ref.float(), rel=1e-5, atol=2e-3, ulps=1.0)
        close("LSE " + w.name, lse, lse_ref, rel=1e-6, atol=1e-5, ulps=0.0)


def test_noalloc_reports_bad_given_indices():
    """Given indices that are out of range are skipped and flagged; callers of the fixed-array
    forward read the flag with msa_forward_noalloc_status (they have no workspace pointer)."""
    lib = msa.load_library()
    w = Workload("badidx", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    g = {k: v.to(DEV) for k, v in make_inputs(w, 77).items() if isinstance(v, torch.Tensor)}
    _, _, idx = _fresh_forward(w, g)
    bad = idx.clone()
    bad[0, 0, 300, 0] = 99  # beyond the token's local block
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    o = torch.empty(g["q"].shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((1, 8, 512), dtype=torch.float32, device=DEV)
    assert _call_noalloc(lib, shape, g, w.top_k, bad, 1, o, lse) == 0
    assert msa.msa_forward_noalloc_status() & 1
    assert torch.isfinite(o.float()).all()
    assert msa.msa_forward_noalloc_status() == 0  # the read clears the word
    # a clean call after the bad one reports nothing
    assert _call_noalloc(lib, shape, g, w.top_k, idx.clone(), 1, o, lse) == 0
    assert msa.msa_forward_noalloc_status() == 0
