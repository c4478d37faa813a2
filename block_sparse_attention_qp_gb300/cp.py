"""Head-wise context parallelism for MSA training (blog, "Context parallelism", point 1: MSA groups
are independent, so a sequence-sharded layout can be re-sharded by heads with one all-to-all,
every rank runs MSA on the whole sequence for its own heads, and the only reduction is the proxy
key gradient, because the one proxy key head is shared by every group).

Layout.  N ranks; rank r holds the sequence shard [r S/N, (r+1) S/N) of every tensor:
q, dout [B, S/N, Hq, D], k, v [B, S/N, Hkv, D], qp [B, S/N, Hp, D], kp [B, S/N, 1, D].
Forward: q, k, v, qp go sequence -> heads (all-to-all): rank r gets query heads
[r Hq/N, (r+1) Hq/N), KV heads [r Hkv/N, ...) and proxy heads [r Hp/N, ...) over the whole
sequence -- the same head mapping as the full problem, since Hkv and Hp are divisible by N -- and
kp is gathered whole.  The local call computes the output of its heads, which goes back heads ->
sequence.  Backward: dout goes sequence -> heads, the local backward returns the gradients of its
heads (dkp: its proxy heads' share over the whole sequence), dq / dk / dv / dqp go heads ->
sequence, and dkp is summed over ranks and scattered by sequence (one reduce-scatter).  The KL
term is a mean over (b, t, proxy head) of the whole problem, so each rank's local backward takes
kl_grad / N (its local mean is over Hp / N heads).

The local compute is the CUDA library (binding.msa_forward / msa_backward) unless a caller passes
other functions with the same signatures.  Collectives use torch.distributed (all_to_all_single,
all_gather_into_tensor, reduce_scatter_tensor), NCCL on GPUs.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _world(group):
    return dist.get_world_size(group), dist.get_rank(group)


def seq_to_head(x: torch.Tensor, group=None) -> torch.Tensor:
    """[B, S/N, H, D] sequence shard -> [B, S, H/N, D] head shard (this rank's heads)."""
    n, _ = _world(group)
    B, Sl, H, D = x.shape
    assert H % n == 0, f"{H} heads do not split over {n} ranks"
    inp = x.reshape(B, Sl, n, H // n, D).permute(2, 0, 1, 3, 4).contiguous()  # chunk j -> rank j
    out = torch.empty_like(inp)
    dist.all_to_all_single(out, inp, group=group)  # out[i]: rank i's tokens, this rank's heads
    return out.permute(1, 0, 2, 3, 4).reshape(B, n * Sl, H // n, D)


def head_to_seq(y: torch.Tensor, group=None) -> torch.Tensor:
    """[B, S, H/N, D] head shard -> [B, S/N, H, D] sequence shard (inverse of seq_to_head)."""
    n, _ = _world(group)
    B, S, Hl, D = y.shape
    assert S % n == 0
    inp = y.reshape(B, n, S // n, Hl, D).permute(1, 0, 2, 3, 4).contiguous()  # chunk j: rank j's tokens
    out = torch.empty_like(inp)
    dist.all_to_all_single(out, inp, group=group)  # out[i]: this rank's tokens, rank i's heads
    return out.permute(1, 2, 0, 3, 4).reshape(B, S // n, n * Hl, D)


def gather_seq(x: torch.Tensor, group=None) -> torch.Tensor:
    """[B, S/N, H, D] -> [B, S, H, D]: every rank's sequence shard, in rank order."""
    n, _ = _world(group)
    B, Sl, H, D = x.shape
    out = torch.empty((n * B, Sl, H, D), dtype=x.dtype, device=x.device)  # rank-major
    dist.all_gather_into_tensor(out, x.contiguous(), group=group)
    return out.reshape(n, B, Sl, H, D).permute(1, 0, 2, 3, 4).reshape(B, n * Sl, H, D)


def reduce_scatter_seq(x: torch.Tensor, group=None) -> torch.Tensor:
    """[B, S, H, D] (a partial sum on every rank) -> [B, S/N, H, D]: the sum over ranks of this
    rank's sequence shard."""
    n, _ = _world(group)
    B, S, H, D = x.shape
    inp = x.reshape(B, n, S // n, H, D).permute(1, 0, 2, 3, 4).reshape(n * B, S // n, H, D)
    out = torch.empty((B, S // n, H, D), dtype=x.dtype, device=x.device)
    dist.reduce_scatter_tensor(out, inp.contiguous(), group=group)  # rank j gets block j
    return out


def _default_forward(q, k, v, qp, kp, top_k, scale):
    from . import binding
    return binding.msa_forward(q, k, v, qp, kp, top_k, scale)


def _default_backward(q, k, v, qp, kp, o, lse, dout, idx, top_k, scale, kl_grad):
    from . import binding
    return binding.msa_backward(q, k, v, qp, kp, o, lse, dout, idx, top_k, scale, kl_grad=kl_grad)


def check_heads(Hq: int, Hkv: int, Hp: int, n: int) -> None:
    """Head-wise sharding needs every head count divisible by the number of ranks."""
    if Hq % n or Hkv % n or Hp % n:
        raise ValueError(f"head-wise context parallelism over {n} ranks needs Hq={Hq}, Hkv={Hkv} "
                         f"and Hp={Hp} divisible by {n}")


def cp_forward(q, k, v, qp, kp, top_k: int, scale: float, group=None, local_forward=None):
    """Forward on sequence shards.  Returns (o_shard, state) where state holds the head-sharded
    tensors the backward needs."""
    n, _ = _world(group)
    check_heads(q.shape[2], k.shape[2], qp.shape[2], n)
    fwd = local_forward or _default_forward
    qh, kh, vh, qph = (seq_to_head(x, group) for x in (q, k, v, qp))
    kpf = gather_seq(kp, group)
    oh, lseh, idxh = fwd(qh, kh, vh, qph, kpf, top_k, scale)
    o = head_to_seq(oh, group)
    return o, dict(q=qh, k=kh, v=vh, qp=qph, kp=kpf, o=oh, lse=lseh, idx=idxh, top_k=top_k,
                   scale=scale)


def cp_backward(state, dout, kl_grad=1.0, group=None, local_backward=None):
    """Backward on sequence shards: dout [B, S/N, Hq, D] -> (dq, dk, dv, dqp, dkp) shards.
    kl_grad: a number or a one-element tensor (kept on its device)."""
    n, _ = _world(group)
    bwd = local_backward or _default_backward
    douth = seq_to_head(dout, group)
    dqh, dkh, dvh, dqph, dkpf = bwd(state["q"], state["k"], state["v"], state["qp"], state["kp"],
                                    state["o"], state["lse"], douth, state["idx"], state["top_k"],
                                    state["scale"], kl_grad / n)
    dq, dk, dv, dqp = (head_to_seq(x, group) for x in (dqh, dkh, dvh, dqph))
    dkp = reduce_scatter_seq(dkpf, group)
    return dq, dk, dv, dqp, dkp


class _CPFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qp, kp, q, k, v, top_k, scale, group):
        o, state = cp_forward(q.contiguous(), k.contiguous(), v.contiguous(), qp.contiguous(),
                              kp.contiguous(), top_k, scale, group)
        ctx.state, ctx.group, ctx.o_meta = state, group, (o.shape, o.dtype, o.device)
        return o, torch.zeros((), dtype=torch.float32, device=q.device)

    @staticmethod
    def backward(ctx, do, dkl):
        kl_grad = 0.0 if dkl is None else dkl  # stays on the device: no host sync
        shape, dtype, device = ctx.o_meta
        do = torch.zeros(shape, dtype=dtype, device=device) if do is None else do.contiguous()
        dq, dk, dv, dqp, dkp = cp_backward(ctx.state, do, kl_grad, ctx.group)
        return dqp, dkp, dq, dk, dv, None, None, None


def msa_func_cp(Q_proxy, K_proxy, Q, K, V, top_k: int, scale: float, group=None):
    """msa_func on sequence shards with head-wise context parallelism over `group`: returns
    (attn_out shard, kl_loss placeholder), like binding.msa_func on the whole sequence."""
    return _CPFunction.apply(Q_proxy, K_proxy, Q, K, V, int(top_k), float(scale), group)
