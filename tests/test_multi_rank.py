"""Two gloo ranks on CPU exercise the multi-rank measurement path (barrier, max over ranks,
per-rank seeds, whole-job rate)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    from block_sparse_attention_qp_gb300 import dist as d
    from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs

    w, r, _ = d.init("gloo")
    assert (w, r) == (world, rank)
    d.barrier()
    elapsed = 1.0 + rank  # rank 1 is the slow one
    slowest = d.max_over_ranks(elapsed)
    wk = Workload("t", B=1, S=256, Hq=4, Hkv=2, Hp=2, top_k=2)
    x = make_inputs(wk, d.rank_seed(10, rank))
    out[rank] = (slowest, d.whole_job_rate(256, w, slowest), float(x["q"].float().sum()))
    d.barrier()
    d.shutdown()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0  # max over ranks
    assert res[0][1] == pytest.approx(256 * 2 / 2.0)
    assert res[0][2] != res[1][2]  # each rank draws its own batch
