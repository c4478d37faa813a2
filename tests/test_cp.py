"""Head-wise context parallelism (block_sparse_attention_qp_gb300/cp.py) on two gloo ranks on CPU.

Each rank holds a sequence shard; the exchanges re-shard by heads, a local MSA computes its heads
over the whole sequence, and the gradients come back by sequence with the proxy key gradient summed
over ranks.  Here the local compute is the fp64 oracle (injected by the test; the product path
calls the CUDA library), so every output shard must equal the single-process oracle's result on
the whole problem up to fp64 summation order -- which checks the exchanges, the head mapping of
the shards and the 1/N of the KL gradient."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _oracle_forward(q, k, v, qp, kp, top_k, scale):
    import oracle

    idx, _ = oracle.select(qp, kp, top_k, scale)
    o, lse = oracle.forward(q, k, v, idx, top_k, scale)
    return torch.from_numpy(o), torch.from_numpy(lse), idx


def _oracle_backward(q, k, v, qp, kp, o, lse, dout, idx, top_k, scale, kl_grad):
    import oracle

    g = oracle.backward(q, k, v, qp, kp, dout, idx, top_k, scale, kl_grad=kl_grad)
    return tuple(torch.from_numpy(g[n]) for n in ("dq", "dk", "dv", "dqp", "dkp"))


SHAPES = {  # B, S, Hq, Hkv, Hp, top_k
    "hp_eq_hkv": (1, 512, 8, 2, 2, 3),
    "hp_lt_hkv": (1, 512, 8, 4, 2, 3),
}


def _worker(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from block_sparse_attention_qp_gb300 import cp
    from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    oracle.set_threads(2)
    B, S, Hq, Hkv, Hp, top_k = SHAPES[name]
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hp, top_k=top_k)
    x = make_inputs(w, 31)  # the same whole problem on every rank
    f = {n: x[n].to(torch.float64) for n in ("q", "k", "v", "qp", "kp", "dout")}
    Sl = S // world
    sh = {n: t[:, rank * Sl:(rank + 1) * Sl].contiguous() for n, t in f.items()}
    o, state = cp.cp_forward(sh["q"], sh["k"], sh["v"], sh["qp"], sh["kp"], top_k, w.scale,
                             local_forward=_oracle_forward)
    grads = cp.cp_backward(state, sh["dout"], kl_grad=0.75, local_backward=_oracle_backward)
    out[rank] = [t.numpy() for t in (o,) + tuple(grads)]
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_headwise_cp_matches_whole_problem(name):
    import oracle
    from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs

    oracle.build()
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, name, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(out)
    B, S, Hq, Hkv, Hp, top_k = SHAPES[name]
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hp, top_k=top_k)
    x = make_inputs(w, 31)
    idx, _ = oracle.select(x["qp"], x["kp"], top_k, w.scale)
    o_ref, _ = oracle.forward(x["q"], x["k"], x["v"], idx, top_k, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, top_k,
                          w.scale, kl_grad=0.75)
    Sl = S // world
    for r in range(world):
        sl = slice(r * Sl, (r + 1) * Sl)
        got = res[r]
        np.testing.assert_allclose(got[0], o_ref[:, sl], rtol=1e-12, atol=1e-13, err_msg="o")
        for name_, g in zip(("dq", "dk", "dv", "dqp", "dkp"), got[1:]):
            np.testing.assert_allclose(g, ref[name_][:, sl], rtol=1e-10, atol=1e-14, err_msg=name_)


def test_exchanges_are_inverse_and_reject_uneven_heads():
    """seq_to_head then head_to_seq is the identity; head counts not divisible by the ranks are
    refused before any collective (single process, world size 1 shortcut not needed)."""
    from block_sparse_attention_qp_gb300 import cp

    with pytest.raises(ValueError, match="divisible"):
        cp.check_heads(8, 2, 3, 2)
    cp.check_heads(8, 2, 2, 2)
