"""A second, independent fp64 implementation of MSA training in eager PyTorch (CPU).

Used only to pin the C oracle on tiny shapes.  It is written from the same definition but in a
different style: dense masks, a stable sort for the top-k (ties -> lower block index), the KL
loss materialised as a number, and every gradient -- including the proxy gradients -- taken by
autograd, so it does not rely on the closed-form KL gradient the oracle uses.

Definition: "Flash-MSA: Accelerating Million-Token Training with Sparse Attention Kernels",
sections "About MSA", "Proxy attention", "Main attention", "KL Divergence Loss", "Warmup kernels";
forum summary "MiniMax Sparse Attention (MSA) ...", section "Architecture: two-stage block-sparse
attention" and "Training stability" (teacher = group mean of the main softmax, stop-gradient).
"""
import torch

BLOCK = 128


def eager_select(qp, kp, top_k, scale):
    """qp [B,S,Hp,D], kp [B,S,1,D] (fp64) -> idx [B,Hp,S,top_k] (ascending, -1 padded)."""
    B, S, Hp, D = qp.shape
    nblk = S // BLOCK
    z = scale * torch.einsum("bthd,bjd->bhtj", qp, kp[:, :, 0, :])  # [B,Hp,S,S]
    zb = z.reshape(B, Hp, S, nblk, BLOCK).amax(-1)  # [B,Hp,S,nblk]
    t = torch.arange(S)
    m = t // BLOCK
    n = torch.arange(nblk)
    c = torch.where(n[None, :] < m[:, None], zb, torch.full_like(zb, float("-inf")))
    c = torch.where(n[None, :] == m[:, None], torch.full_like(c, float("inf")), c)
    order = torch.sort(c, dim=-1, descending=True, stable=True).indices
    idx = torch.full((B, Hp, S, top_k), -1, dtype=torch.int32)
    for tt in range(S):
        K = min(top_k, int(m[tt]) + 1)
        chosen = torch.sort(order[:, :, tt, :K], dim=-1).values
        idx[:, :, tt, :K] = chosen.to(torch.int32)
    return idx


def key_mask(idx, S, warmup=False, Hp=None, B=None):
    """Boolean mask [B,Hp,S(t),S(j)] of the key sets J(t,g)."""
    t = torch.arange(S)
    causal = t[None, :] <= t[:, None]
    if warmup:
        return causal[None, None].expand(B, Hp, S, S)
    B, Hp = idx.shape[0], idx.shape[1]
    blk_of_j = t // BLOCK
    blocks = torch.arange(S // BLOCK)
    sel = (idx.long()[..., None] == blocks).any(-2)  # [B,Hp,S,nblk]; -1 padding matches nothing
    return sel[..., blk_of_j] & causal[None, None]


def eager_msa(q, k, v, qp, kp, dout, idx, scale, kl_grad=1.0, warmup=False):
    """Forward + backward.  Returns dict(o, lse, kl, dq, dk, dv, dqp, dkp) (fp64)."""
    q, k, v, qp, kp = (x.detach().clone().requires_grad_(True) for x in (q, k, v, qp, kp))
    B, S, Hq, D = q.shape
    Hkv, Hp = k.shape[2], qp.shape[2]
    G, Gp = Hq // Hkv, Hq // Hp  # query heads per KV head / per proxy head (MSA group)
    mask = key_mask(idx, S, warmup=warmup, Hp=Hp, B=B)  # [B,Hp,S,S]
    kv_of = torch.arange(Hq) // G      # query head -> KV head
    proxy_of = torch.arange(Hq) // Gp  # query head -> proxy head whose selection it uses
    mask_h = mask[:, proxy_of]  # [B,Hq,S,S]
    k_h = k[:, :, kv_of, :]
    v_h = v[:, :, kv_of, :]
    s = scale * torch.einsum("bthd,bjhd->bhtj", q, k_h)
    s = s.masked_fill(~mask_h, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)  # [B,Hq,S]
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhtj,bjhd->bthd", p, v_h)
    # teacher: mean over the Gp query heads of each proxy head, stop-gradient
    pbar = p.detach().reshape(B, Hp, Gp, S, S).mean(2)
    z = scale * torch.einsum("bthd,bjd->bhtj", qp, kp[:, :, 0, :])
    z = z.masked_fill(~mask, float("-inf"))
    logp_px = torch.log_softmax(z, dim=-1)
    logp_px = torch.where(mask, logp_px, torch.zeros_like(logp_px))  # keep -inf out of autograd
    terms = torch.where(mask, pbar * (torch.log(pbar.clamp_min(1e-300)) - logp_px),
                        torch.zeros_like(pbar))
    kl = terms.sum() / (B * S * Hp)
    loss = (o * dout).sum() + kl_grad * kl
    loss.backward()
    return dict(o=o.detach(), lse=lse.detach(), kl=float(kl.detach()), dq=q.grad, dk=k.grad, dv=v.grad,
                dqp=qp.grad, dkp=kp.grad)
