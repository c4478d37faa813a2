"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Small shapes that span several tiles and ragged tails are compared in full; the workload sizes
of the benchmark are compared on sampled rows (see test_gpu_fullsize.py).
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_qp_gb300 import binding as msa
from block_sparse_attention_qp_gb300.inputs import WORKLOADS, Workload, make_inputs, workload_seed
from tests.parity import close, compare_selection

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_sparse(w: Workload, seed: int, kl_grad=1.0):
    x = make_inputs(w, seed)
    g = to_dev(x)
    # 1. selection on the GPU vs the oracle
    _, _, gidx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale)
    oidx, gap = oracle.select(x["qp"], x["kp"], w.top_k, w.scale)
    n_bad, n_exc = compare_selection(gidx, oidx, gap)
    # 2. forward and backward from the oracle's indices
    idx_t = torch.from_numpy(oidx).to(DEV)
    ws = msa.workspace(msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale), msa.OP_FORWARD, DEV)
    o, lse, _ = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                                block_idx=idx_t, ws=ws)
    assert msa.msa_device_status(ws) == 0
    if w.Hq // max(w.Hp, w.Hkv) < 4:  # the backward supports 4, 8 and 16 heads per attention group
        o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], oidx, w.top_k, w.scale)
        close("O", o, o_ref)
        close("LSE", lse, lse_ref)
        with pytest.raises(msa.MSAError, match="unsupported"):
            msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx_t,
                             w.top_k, w.scale)
        return n_bad, n_exc
    wsb = msa.workspace(msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale), msa.OP_BACKWARD, DEV)
    *grads, kl = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"],
                                  idx_t, w.top_k, w.scale, kl_grad=kl_grad, ws=wsb, return_kl=True)
    assert msa.msa_device_status(wsb) == 0, "a bounded device wait gave up"
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], oidx, w.top_k, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], oidx, w.top_k,
                          w.scale, kl_grad=kl_grad)
    close("O", o, o_ref)
    close("LSE", lse, lse_ref)
    for name, gt in zip(("dq", "dk", "dv", "dqp", "dkp"), grads):
        close(name, gt, ref[name])
    check_kl(kl, ref["kl"])
    return n_bad, n_exc


def check_kl(kl, want, rel=5e-3):
    """The KL value the backward materialises on request, against the oracle's L_KL."""
    got = float(kl)
    assert want > 0 and abs(got - want) <= rel * want, f"KL {got:.6e} vs oracle {want:.6e}"


SMALL = [
    # name, B, S, Hq, Hkv, top_k, planted
    ("cfg1", 1, 1024, 8, 2, 4, 0),
    ("g4_b2_k6", 2, 1280, 16, 4, 6, 0),
    ("ragged_g4", 2, 640, 8, 2, 3, 0),
    ("g2_k5", 1, 896, 4, 2, 5, 0),
    ("g8_planted", 1, 1536, 16, 2, 6, 4),
    ("g16", 1, 768, 16, 1, 3, 0),
    ("g16_b2_k5", 2, 1024, 32, 2, 5, 0),
    ("k1_local_only", 2, 512, 8, 2, 1, 0),
    ("k_covers_all", 1, 640, 8, 2, 8, 0),
    ("single_block", 3, 128, 8, 2, 4, 0),
]


@pytest.mark.parametrize("name,B,S,Hq,Hkv,k,planted", SMALL, ids=[c[0] for c in SMALL])
def test_sparse_small(name, B, S, Hq, Hkv, k, planted):
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hkv, top_k=k, planted=planted)
    run_sparse(w, seed=100 + S + Hq)


MAPPINGS = [
    # name, B, S, Hq, Hkv, Hp, top_k: one proxy head selecting for several GQA groups (Hp < Hkv,
    # the inverted mapping), and GQA groups split among proxy heads (Hp > Hkv)
    ("hp_lt_hkv_r2", 1, 1024, 16, 4, 2, 4),
    ("hp_lt_hkv_r4_b2", 2, 640, 16, 4, 1, 3),
    ("hp_gt_hkv", 1, 1024, 16, 2, 4, 4),
    ("hp_gt_hkv_fwd_only", 1, 768, 8, 2, 4, 3),
]


@pytest.mark.parametrize("name,B,S,Hq,Hkv,Hp,k", MAPPINGS, ids=[c[0] for c in MAPPINGS])
def test_sparse_proxy_kv_head_mappings(name, B, S, Hq, Hkv, Hp, k):
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hp, top_k=k)
    run_sparse(w, seed=700 + S + Hq + Hp)


@pytest.mark.parametrize("B,S,Hq,Hkv,Hp", [(1, 768, 16, 4, 2), (1, 640, 16, 2, 4)])
def test_warmup_proxy_kv_head_mappings(B, S, Hq, Hkv, Hp):
    """Dense warmup backward with a proxy head over two attention groups (its teacher rows summed
    from both) and with two proxy heads over one, in one pass and in about three teacher passes
    over runs of lists (ending inside the 512-token chunks), each against the oracle."""
    w = Workload("wmap", B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hp, top_k=0)
    x = make_inputs(w, 800 + S + Hp)
    g = to_dev(x)
    o, lse = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], None, 1, w.scale)
    shape = msa.make_shape(g["q"], g["k"], g["qp"], 0, w.scale)
    full = msa.msa_workspace_size(shape, msa.OP_WARMUP_BACKWARD)
    nblk = S // 128
    teacher = B * Hp * (S * nblk - 128 * nblk * (nblk - 1) // 2) * 128 * 2  # all teacher rows
    for nbytes in (full, full - teacher * 2 // 3):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        *grads, kl = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse,
                                             g["dout"], w.scale, ws=ws, return_kl=True)
        torch.cuda.synchronize()
        assert msa.msa_device_status(ws) == 0
        for name_, gt in zip(("dq", "dk", "dv", "dqp", "dkp"), grads):
            close(name_, gt, ref[name_])
        check_kl(kl, ref["kl"])


def test_sparse_kl_grad_scales_proxy_only():
    w = Workload("klg", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    run_sparse(w, seed=5, kl_grad=2.5)


WARM = [("w_g4", 1, 768, 8, 2), ("w_g4_b2", 2, 640, 8, 2), ("w_g8", 1, 512, 16, 2),
        ("w_g16", 1, 384, 16, 1), ("w_g4_long", 1, 1536, 8, 2)]


@pytest.mark.parametrize("case", WARM, ids=[c[0] for c in WARM])
def test_warmup_small(case):
    name, B, S, Hq, Hkv = case
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hkv, top_k=0)
    x = make_inputs(w, 300 + S)
    g = to_dev(x)
    o, lse = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    *grads, kl = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse,
                                         g["dout"], w.scale, kl_grad=1.0, return_kl=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], None, 1, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], None, 1, w.scale)
    close("O", o, o_ref)
    close("LSE", lse, lse_ref)
    for name_, gt in zip(("dq", "dk", "dv", "dqp", "dkp"), grads):
        close(name_, gt, ref[name_])
    check_kl(kl, ref["kl"])


def test_dense_forward_group_one():
    """Hq == Hkv (one query head per group) is supported by the forward ops."""
    w = Workload("g1", B=1, S=512, Hq=2, Hkv=2, Hp=2, top_k=2)
    x = make_inputs(w, 9)
    g = to_dev(x)
    o, lse = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], None, 1, w.scale)
    close("O", o, o_ref)
    close("LSE", lse, lse_ref)
    oidx, _ = oracle.select(x["qp"], x["kp"], 2, w.scale)
    o2, lse2, _ = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 2, w.scale,
                                  block_idx=torch.from_numpy(oidx).to(DEV))
    o_ref2, lse_ref2 = oracle.forward(x["q"], x["k"], x["v"], oidx, 2, w.scale)
    close("O", o2, o_ref2)
    close("LSE", lse2, lse_ref2)


def test_full_selection_equals_warmup_on_gpu():
    """With top_k >= number of blocks the sparse path computes dense causal attention."""
    w = Workload("all", B=1, S=640, Hq=8, Hkv=2, Hp=2, top_k=5)
    g = to_dev(make_inputs(w, 77))
    o1, l1, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 5, w.scale)
    o2, l2 = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    close("O", o1, o2.float(), rel=2e-3, ulps=1.5)
    close("LSE", l1, l2, rel=1e-5, atol=1e-4)
    g1 = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o1, l1, g["dout"], idx, 5, w.scale)
    g2 = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o2, l2, g["dout"], w.scale)
    for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), g1, g2):
        close(name, a, b.float(), rel=5e-3, ulps=1.5)


def test_cfg2_full_parity():
    """Workload 2 (B=2, S=8192, 32/8/8 heads, top_k=16, planted blocks), every output."""
    w = WORKLOADS[1]
    n_bad, n_exc = run_sparse(w, workload_seed(2))
    print(f"workload 2: {n_bad} selection rows differ, all near ties ({n_exc})")


def test_forward_is_bitwise_repeatable():
    """The list building places tokens with atomic cursors, so a token's tile partners differ from
    run to run; the forward's per-row arithmetic must not depend on them (same summation order on
    the masked and the unmasked softmax path), so two runs give identical bits."""
    w = Workload("det", B=2, S=1536, Hq=16, Hkv=4, Hp=4, top_k=5)
    g = to_dev(make_inputs(w, 77))
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    runs = []
    for _ in range(3):
        ws = msa.workspace(shape, msa.OP_FORWARD, DEV)
        runs.append(msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                                    ws=ws))
        assert msa.msa_device_status(ws) == 0  # no bounded wait gave up
    for o, lse, idx in runs[1:]:
        assert torch.equal(idx, runs[0][2])
        assert torch.equal(o, runs[0][0])
        assert torch.equal(lse, runs[0][1])


def test_kl_value_does_not_change_the_gradients():
    """Asking for the KL value leaves every gradient unchanged up to fp32 summation order, since
    the value is computed beside the proxy gradients, not from them.  The gradient accumulators
    take reductions in whatever order blocks finish and the gradients come out in bf16, so an
    fp32 sum that lands on the other side of a rounding boundary moves that entry by one bf16
    unit: every entry must agree within one bf16 ulp, and few may differ at all (measured on
    GB300 between two runs: rel L2 1.7e-5 to 1.4e-4, a handful of entries one ulp apart)."""
    w = Workload("klv", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4)
    g = to_dev(make_inputs(w, 61))
    o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale)
    a = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx,
                         w.top_k, w.scale)
    *b, kl = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx,
                              w.top_k, w.scale, return_kl=True)
    for name, x, y in zip(("dq", "dk", "dv", "dqp", "dkp"), a, b):
        close(name, x, y.float(), rel=1e-3, atol=2e-3, ulps=1.0)
        differ = (x.float() != y.float()).float().mean().item()
        assert differ <= 0.01, f"{name}: {differ:.2%} of the entries differ"
    assert float(kl) > 0


def test_bad_indices_are_flagged_not_faulted():
    """Out-of-range / unsorted given indices are skipped by the kernels and reported."""
    w = Workload("bad", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    g = to_dev(make_inputs(w, 3))
    oidx, _ = oracle.select(make_inputs(w, 3)["qp"], make_inputs(w, 3)["kp"], 3, w.scale)
    bad = torch.from_numpy(oidx.copy())
    bad[0, 0, 300, 0] = 99          # beyond the token's local block
    bad[0, 1, 400, :] = torch.tensor([2, 1, 3], dtype=torch.int32)  # not ascending
    bad = bad.to(DEV)
    ws = msa.workspace(msa.make_shape(g["q"], g["k"], g["qp"], 3, w.scale), msa.OP_FORWARD, DEV)
    o, lse, _ = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 3, w.scale,
                                block_idx=bad, ws=ws)
    flags = msa.msa_device_status(ws)
    assert flags & 1
    assert torch.isfinite(o.float()).all()
    assert msa.msa_device_status(ws) == 0  # cleared by the read


def test_host_validation_errors():
    w = Workload("v", B=1, S=256, Hq=8, Hkv=2, Hp=2, top_k=2)
    g = to_dev(make_inputs(w, 1))
    with pytest.raises(msa.MSAError, match="unsupported"):
        msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 0, w.scale)
    with pytest.raises(msa.MSAError):
        msa.msa_forward(g["q"][:, :200].contiguous(), g["k"][:, :200].contiguous(),
                        g["v"][:, :200].contiguous(), g["qp"][:, :200].contiguous(),
                        g["kp"][:, :200].contiguous(), 2, w.scale)
    shape = msa.make_shape(g["q"], g["k"], g["qp"], 2, w.scale)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(msa.MSAError, match="workspace"):
        msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 2, w.scale, ws=small)
    assert msa.msa_workspace_size(shape, msa.OP_FORWARD) > 0
    with pytest.raises(msa.MSAError, match="one device"):  # every argument on the data's device
        msa.msa_forward(g["q"], g["k"].cpu(), g["v"], g["qp"], g["kp"], 2, w.scale)


def test_autograd_function_matches_direct_calls():
    w = Workload("ag", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    g = to_dev(make_inputs(w, 11))
    leaves = {n: g[n].clone().requires_grad_(True) for n in ("qp", "kp", "q", "k", "v")}
    out, kl = msa.msa_func(leaves["qp"], leaves["kp"], leaves["q"], leaves["k"], leaves["v"], 3, w.scale)
    assert float(kl.detach()) == 0.0
    ((out.float() * g["dout"].float()).sum() + 1.5 * kl).backward()
    o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 3, w.scale)
    ref = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx, 3,
                           w.scale, kl_grad=1.5)
    close("O", out, o.float(), rel=1e-5, atol=2e-3, ulps=1.0)  # equal up to fp32 summation order
    for name, r in zip(("q", "k", "v", "qp", "kp"), ref):
        close("d" + name, leaves[name].grad, r.float(), rel=1e-2, ulps=1.5)


def test_kl_grad_from_a_device_tensor_matches_the_host_value():
    w = Workload("klgd", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    g = to_dev(make_inputs(w, 12))
    o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 3, w.scale)
    host = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx, 3,
                            w.scale, kl_grad=0.625)
    dev = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx, 3,
                           w.scale, kl_grad=torch.tensor(0.625, device=DEV))
    # equal up to the order of the fp32 reductions into the gradients (and 0.625/N against
    # 0.625*(1/N) in the proxy ones): a bf16 ulp apart, or 1e-4 where a sum nearly cancels
    for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), host, dev):
        close(name, b, a.float(), rel=1e-3, atol=1e-4, ulps=1.0)
    wh = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"],
                                 w.scale, kl_grad=0.0)
    wd = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"],
                                 w.scale, kl_grad=torch.zeros((), device=DEV))
    for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), wh, wd):
        close("warmup " + name, b, a.float(), rel=1e-3, atol=1e-4, ulps=1.0)
    assert float(host[3].abs().max()) > 0  # kl_grad 0.625: the proxy gradients are live
    assert float(wd[3].abs().max()) == 0 and float(wd[4].abs().max()) == 0  # kl_grad 0 on the device


def test_autograd_backward_never_waits_on_the_host_and_reuses_its_workspace():
    """The placeholder's incoming gradient stays on the device (torch raises on a synchronising
    call in sync-debug "error" mode), and a second, larger call on the same stream grows the
    cached workspace and still matches the direct calls."""
    msa.clear_workspace_cache()
    for S, seed in ((512, 21), (1024, 22), (512, 23)):
        w = Workload("agc", B=1, S=S, Hq=8, Hkv=2, Hp=2, top_k=3)
        g = to_dev(make_inputs(w, seed))
        leaves = {n: g[n].clone().requires_grad_(True) for n in ("qp", "kp", "q", "k", "v")}
        out, kl = msa.msa_func(leaves["qp"], leaves["kp"], leaves["q"], leaves["k"], leaves["v"],
                               3, w.scale)
        loss = (out.float() * g["dout"].float()).sum() + 0.5 * kl
        torch.cuda.set_sync_debug_mode("error")
        try:
            loss.backward()
        finally:
            torch.cuda.set_sync_debug_mode("default")
        o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], 3, w.scale)
        ref = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx,
                               3, w.scale, kl_grad=0.5)
        close("O", out, o.float(), rel=1e-5, atol=2e-3, ulps=1.0)
        for name, r in zip(("q", "k", "v", "qp", "kp"), ref):
            close("d" + name, leaves[name].grad, r.float(), rel=1e-2, ulps=1.5)
    assert len(msa._WS_CACHE) == 1
    msa.clear_workspace_cache()


@pytest.mark.parametrize("G,S", [(2, 768), (4, 1280), (8, 896)])
def test_warmup_forward_growing_row_maxima(G, S):
    """Dense forward on inputs whose score scale grows along the sequence (key rows scaled by
    1 + t/128, queries by 3): later key blocks keep raising the row maxima by far more than the
    kernel's lazy-rescale threshold, so O and l are rescaled many times per row."""
    Hkv = 2
    w = Workload("grow", B=1, S=S, Hq=G * Hkv, Hkv=Hkv, Hp=Hkv, top_k=0)
    x = make_inputs(w, 500 + S + G)
    ramp = (1.0 + torch.arange(S, dtype=torch.float32) / 128.0).view(1, S, 1, 1)
    x["k"] = (x["k"].float() * ramp).to(torch.bfloat16)
    x["q"] = (x["q"].float() * 3.0).to(torch.bfloat16)
    g = to_dev(x)
    o, lse = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], None, 1, w.scale)
    close("O", o, o_ref)
    close("LSE", lse, lse_ref, rel=1e-5, atol=1e-3, ulps=0.0)


def test_training_step_replays_from_a_cuda_graph():
    """One forward + backward captured in a CUDA graph (the backward forks onto the library's side
    stream and joins back inside the capture) replays to the eager results."""
    w = Workload("graph", B=1, S=1024, Hq=16, Hkv=2, Hp=2, top_k=4)
    g = to_dev(make_inputs(w, 31))
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    wsf = msa.workspace(shape, msa.OP_FORWARD, DEV)
    wsb = msa.workspace(shape, msa.OP_BACKWARD, DEV)

    def step():
        o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                                      ws=wsf)
        grads = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx,
                                 w.top_k, w.scale, ws=wsb)
        return (o, lse, idx) + tuple(grads)

    eager = step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on a non-default stream, as graph capture wants
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert msa.msa_device_status(wsf) == 0 and msa.msa_device_status(wsb) == 0
    assert torch.equal(captured[2], eager[2])                  # selection
    assert torch.equal(captured[0], eager[0]) and torch.equal(captured[1], eager[1])  # O, LSE
    for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), captured[3:], eager[3:]):
        close(name, a, b.float(), rel=1e-3, atol=1e-4, ulps=1.0)  # fp32 reduction order only


def test_forward_in_passes_equals_one_pass():
    """A workspace smaller than msa_workspace_size makes the forward produce and merge its partial
    outputs in passes over the sequence chunks (here four chunks of 8192 tokens: passes of 3 + 1
    and 1 + 1 + 1 + 1 chunks); every result equals the one-pass result bit for bit."""
    w = Workload("passes", B=2, S=32768, Hq=16, Hkv=2, Hp=2, top_k=8)  # chunks of 8192 tokens
    g = to_dev(make_inputs(w, 41))
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    full = msa.msa_workspace_size(shape, msa.OP_FORWARD)
    chunk_bytes = w.B * 8192 * w.Hq * w.top_k * (128 * 2 + 4)  # partials of one chunk
    ref = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                          ws=torch.empty(full, dtype=torch.uint8, device=DEV))
    for fewer in (1, 3):
        ws = torch.empty(full - fewer * chunk_bytes, dtype=torch.uint8, device=DEV)
        got = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale, ws=ws)
        assert msa.msa_device_status(ws) == 0
        for name, a, b in zip(("O", "LSE", "block_idx"), got, ref):
            assert torch.equal(a, b), (fewer, name)
    with pytest.raises(msa.MSAError, match="workspace"):
        msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                        ws=torch.empty(full - 4 * chunk_bytes, dtype=torch.uint8, device=DEV))


def test_backward_in_passes_equals_one_pass():
    """A smaller workspace makes the backward keep the teacher rows for fewer sequence chunks at a
    time (attn_bwd then proxy_bwd, pass by pass): 3 + 1 and 4 x 1 passes of chunks of 8192 tokens
    here, and runs of consecutive lists in the dense warmup backward.  The gradients and the KL
    value equal the one-pass results up to the order of the fp32 reductions."""
    w = Workload("bpasses", B=2, S=32768, Hq=16, Hkv=2, Hp=2, top_k=8)
    g = to_dev(make_inputs(w, 43))
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    o, lse, idx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale)
    full = msa.msa_workspace_size(shape, msa.OP_BACKWARD)
    teacher_chunk = w.B * w.Hp * 8192 * w.top_k * 128 * 2  # teacher rows of one chunk (at most)

    def run(nbytes):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        out = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse, g["dout"], idx,
                               w.top_k, w.scale, ws=ws, return_kl=True)
        assert msa.msa_device_status(ws) == 0
        return out

    ref = run(full)
    for nbytes in (full - 1, full - 3 * teacher_chunk):
        got = run(nbytes)
        for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), got[:5], ref[:5]):
            close(name, a, b.float(), rel=1e-3, atol=1e-4, ulps=1.0)
        assert abs(float(got[5]) - float(ref[5])) <= 1e-6 * abs(float(ref[5]))
    with pytest.raises(msa.MSAError, match="workspace"):
        run(full - 4 * teacher_chunk)
    # dense warmup backward (two chunks of 16384 tokens): its passes are runs of consecutive
    # lists, so with less room they end inside a chunk -- 2, 3 and about 10 passes here
    wd = Workload("wpasses", B=1, S=32768, Hq=8, Hkv=2, Hp=2, top_k=0)
    gd = to_dev(make_inputs(wd, 44))
    od, ld = msa.msa_warmup_forward(gd["q"], gd["k"], gd["v"], wd.scale)
    shd = msa.make_shape(gd["q"], gd["k"], gd["qp"], 0, wd.scale)
    fulld = msa.msa_workspace_size(shd, msa.OP_WARMUP_BACKWARD)
    nblk = wd.S // 128
    teacher = wd.B * wd.Hp * (wd.S * nblk - 128 * nblk * (nblk - 1) // 2) * 128 * 2  # all rows

    def run_dense(nbytes):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        out = msa.msa_warmup_backward(gd["q"], gd["k"], gd["v"], gd["qp"], gd["kp"], od, ld,
                                      gd["dout"], wd.scale, ws=ws, return_kl=True)
        assert msa.msa_device_status(ws) == 0
        return out

    refd = run_dense(fulld)
    for nbytes in (fulld - 1, fulld - teacher * 2 // 3, fulld - teacher * 9 // 10):
        got = run_dense(nbytes)
        for name, a, b in zip(("dq", "dk", "dv", "dqp", "dkp"), got[:5], refd[:5]):
            close("warmup " + name, a, b.float(), rel=1e-3, atol=1e-4, ulps=1.0)
        assert abs(float(got[5]) - float(refd[5])) <= 1e-6 * abs(float(refd[5]))
    for nbytes in (fulld - teacher, fulld - teacher + 10000 * 256):  # no room / less than a list
        with pytest.raises(msa.MSAError, match="workspace"):
            run_dense(nbytes)
