"""The C ABI library loads, exports every entry point include/msa.h declares, and rejects bad
arguments on the host (no GPU work is issued by any call in this file)."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_qp_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^MSA_API\s+[\w\s\*]+?\b(msa_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return binding.load_library(path)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding._SYMBOLS) <= set(names)


def test_workspace_size_is_host_only(lib):
    s = binding.Shape(1, 1024, 8, 2, 2, 128, 4, 128 ** -0.5)
    for op in range(4):
        assert binding.msa_workspace_size(s, op) > 0
    bad = binding.Shape(1, 1000, 8, 2, 2, 128, 4, 0.1)  # S not a multiple of 128
    assert lib.msa_workspace_size(ctypes.byref(bad), 0) == 0
    assert b"multiple of 128" in lib.msa_last_error()
    # proxy heads that do not divide the query heads, or that neither divide nor are divided by
    # the KV heads, are rejected; Hp < Hkv and Hp > Hkv mappings are accepted
    assert lib.msa_workspace_size(ctypes.byref(binding.Shape(1, 256, 8, 2, 3, 128, 4, 0.1)), 0) == 0
    assert b"proxy heads" in lib.msa_last_error()
    assert lib.msa_workspace_size(ctypes.byref(binding.Shape(1, 256, 24, 6, 4, 128, 4, 0.1)), 0) == 0
    assert binding.msa_workspace_size(binding.Shape(1, 256, 16, 4, 2, 128, 4, 0.1), 1) > 0
    assert binding.msa_workspace_size(binding.Shape(1, 256, 16, 2, 4, 128, 4, 0.1), 1) > 0
    # heads per attention group Hq / max(Hp, Hkv) = 2: forward only
    assert binding.msa_workspace_size(binding.Shape(1, 256, 8, 2, 4, 128, 4, 0.1), 0) > 0
    assert lib.msa_workspace_size(ctypes.byref(binding.Shape(1, 256, 8, 2, 4, 128, 4, 0.1)), 1) == 0
    assert lib.msa_workspace_size(ctypes.byref(binding.Shape(1, 256, 8, 2, 2, 64, 4, 0.1)), 0) == 0
    assert lib.msa_workspace_size(ctypes.byref(binding.Shape(1, 256, 8, 2, 2, 128, 65, 0.1)), 0) == 0


def test_workspace_is_bounded_by_passes(lib):
    """The forward's partial outputs and the backwards' teacher rows are held one pass at a time
    (8 GiB of each by default), so beyond them the workspace grows linearly with S: in the warmup
    backward as well, whose lists grow with S^2 (B Hp S^2 / 256 entries)."""
    gib = 2 ** 30
    budget = 8 * gib

    def linear_bwd(B, S, Hq, Hkv, Hp):  # fp32 accumulators and per-row data, bytes
        return B * S * (Hq * 512 + 2 * Hkv * 512 + Hp * 512 + 512 + Hq * 8 + Hp * 8)

    for S in (32768, 65536, 131072):
        s = binding.Shape(1, S, 32, 8, 8, 128, 0, 128 ** -0.5)
        ws = binding.msa_workspace_size(s, binding.OP_WARMUP_BACKWARD)
        entries = 8 * S * S // 256
        assert entries * 256 > ws or S == 32768  # all the teacher rows would not fit
        # teacher pass + linear part + work items and list offsets (a few bytes per 64 entries)
        assert ws <= budget + linear_bwd(1, S, 32, 8, 8) + entries // 8 + (64 << 20), (S, ws)
    for S in (1 << 20, 1 << 21):
        s = binding.Shape(1, S, 16, 4, 4, 128, 16, 128 ** -0.5)
        fwd = binding.msa_workspace_size(s, binding.OP_FORWARD)
        assert fwd <= budget + S * 4 * 16 * 12 + (256 << 20), (S, fwd)  # partials + lists
        bwd = binding.msa_workspace_size(s, binding.OP_BACKWARD)
        per_entry = 4 + 4 + 4 * 8 + 4  # entry, proxy normaliser, row data copy, partial normaliser
        assert bwd <= budget + linear_bwd(1, S, 16, 4, 4) + S * 4 * 16 * per_entry + (256 << 20), (S, bwd)


def test_argument_errors_before_any_launch(lib):
    s = binding.Shape(1, 256, 8, 2, 2, 128, 2, 0.1)
    P = ctypes.c_void_p
    null = P(0)
    rc = lib.msa_forward(ctypes.byref(s), null, null, null, null, null, null, 0, null, null,
                         null, 0, null)
    assert rc == 1 and lib.msa_status_string(rc) == b"invalid argument"
    odd = P(0x1008)  # not 16-byte aligned; rejected before it is ever dereferenced
    rc = lib.msa_warmup_forward(ctypes.byref(s), odd, odd, odd, odd, odd, null, 0, null)
    assert rc == 1 and b"aligned" in lib.msa_last_error()
    s_bad = binding.Shape(1, 256, 8, 2, 2, 128, 2, -1.0)
    rc = lib.msa_warmup_forward(ctypes.byref(s_bad), null, null, null, null, null, null, 0, null)
    assert rc == 1
    assert lib.msa_status_string(3) == b"workspace too small"


def test_decode_host_checks(lib):
    s = binding.Shape(128, 65536, 64, 8, 8, 128, 16, 128 ** -0.5)
    assert binding.msa_workspace_size(s, binding.OP_DECODE) > 0
    P = ctypes.c_void_p
    null = P(0)
    rc = lib.msa_decode(ctypes.byref(s), null, null, null, null, null, null, null, null, null,
                        null, 0, null)
    assert rc == 1  # null pointers, before any launch
    many = binding.Shape(1, 256, 64, 1, 64, 128, 4, 0.1)  # 64 proxy heads: too many for decode
    assert lib.msa_workspace_size(ctypes.byref(many), binding.OP_DECODE) == 0
    assert b"32 proxy heads" in lib.msa_last_error()


def test_selftest_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    assert lib.msa_selftest_wait_timeout(P(0), 1000, P(0)) == 1
    assert lib.msa_selftest_wait_timeout(P(0x1008), 1000, P(0)) == 1  # misaligned, never touched
    assert b"aligned" in lib.msa_last_error()
    assert lib.msa_selftest_wait_timeout(P(0x1000), 0, P(0)) == 1  # limit out of range
    assert lib.msa_selftest_wait_timeout(P(0x1000), 2_000_000, P(0)) == 1
    assert b"limit_us" in lib.msa_last_error()


def declared_arity():
    """Parameter count of every msa_* prototype in include/."""
    out = {}
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            for name, params in re.findall(r"^MSA_API\s+[\w\s\*]+?\b(msa_\w+)\s*\(([^)]*)\)",
                                           text, flags=re.M):
                params = params.strip()
                out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header(lib):
    for name, n in declared_arity().items():
        argtypes = getattr(lib, name).argtypes
        if argtypes is not None:
            assert len(argtypes) == n, f"{name}: header has {n} parameters, binding {len(argtypes)}"


def test_backward_rejects_a_misaligned_kl_grad_pointer(lib):
    s = binding.Shape(1, 256, 8, 2, 2, 128, 2, 0.1)
    P = ctypes.c_void_p
    a = P(0x10000)  # aligned and never dereferenced: the call fails on the host first
    odd = P(0x10002)
    rc = lib.msa_backward(ctypes.byref(s), a, a, a, a, a, a, a, a, a, 1.0, odd, a, a, a, a, a,
                          P(0), a, 1 << 30, P(0))
    assert rc == 1 and b"kl_grad_dev" in lib.msa_last_error()
    rc = lib.msa_warmup_backward(ctypes.byref(s), a, a, a, a, a, a, a, a, 1.0, odd, a, a, a, a, a,
                                 P(0), a, 1 << 30, P(0))
    assert rc == 1 and b"kl_grad_dev" in lib.msa_last_error()


def test_kl_grad_argument_marshalling():
    """kl_grad goes to the library by value when it is a number and as a device pointer (read by
    the kernel, no host synchronisation) when it is a one-element tensor on the inputs' device."""
    import torch

    assert binding._kl_grad_args(0.5, "cpu") == (0.5, None)
    v, t = binding._kl_grad_args(torch.tensor([2.0], dtype=torch.float64), "cpu")
    assert v == 0.0 and t.dtype == torch.float32 and t.shape == () and float(t) == 2.0
    with pytest.raises(binding.MSAError, match="one element"):
        binding._kl_grad_args(torch.ones(2), "cpu")
    with pytest.raises(binding.MSAError, match="is on"):
        binding._kl_grad_args(torch.ones(()), "meta")
