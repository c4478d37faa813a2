"""Closed-form work counts of one MSA training step (used to report TFLOP/s).

Counting convention (the one behind the forum summary's "28.4x per-token attention compute
reduction at 1M context", section "Architecture"): 4d FLOPs per main-attention (query, key) pair
in the forward (QK^T and PV), 2d per proxy (query, key) pair (QK^T only); the backward counts
10d per main pair (the score recompute, dP, dV, dK, dQ) and 6d per proxy pair over the selected
tokens (score recompute, dQp, dKp).  The proxy normaliser recompute of the backward is overhead and
is not counted.
"""
from __future__ import annotations

BLOCK = 128


def n_sel(S: int, top_k: int) -> int:
    """(token, key) pairs attended by one head of one sequence: every non-local selected block is
    fully visible, the local block up to the token itself."""
    nblk = S // BLOCK
    total = 0
    for m in range(nblk):
        K = min(top_k, m + 1)
        total += BLOCK * BLOCK * (K - 1) + BLOCK * (BLOCK + 1) // 2
    return total


def n_px(S: int) -> int:
    """Proxy (token, key) pairs scored for selection by one proxy head: keys in earlier blocks."""
    nblk = S // BLOCK
    return BLOCK * BLOCK * nblk * (nblk - 1) // 2


def n_dense(S: int) -> int:
    """Causal (token, key) pairs, diagonal included."""
    return S * (S + 1) // 2


def step_flops(B: int, S: int, Hq: int, Hp: int, top_k: int, D: int = 128) -> dict:
    """FLOPs of one forward + backward step; top_k == 0 means the dense warmup step."""
    if top_k == 0:
        pairs = n_dense(S)
        f = dict(main_fwd=4 * D * pairs * Hq, main_bwd=10 * D * pairs * Hq, proxy_fwd=0,
                 proxy_bwd=6 * D * pairs * Hp)
    else:
        sel = n_sel(S, top_k)
        f = dict(main_fwd=4 * D * sel * Hq, main_bwd=10 * D * sel * Hq,
                 proxy_fwd=2 * D * n_px(S) * Hp, proxy_bwd=6 * D * sel * Hp)
    f = {k: v * B for k, v in f.items()}
    f["total"] = sum(f.values())
    return f


def per_token_reduction(N: int, Hq: int, Hp: int, top_k: int) -> float:
    """Dense causal GQA attention vs MSA, per token, at context N (causal average N/2 keys):
    Hq main heads over N/2 keys  vs  Hq heads over top_k*128 keys + Hp index heads over N/2 keys
    (QK^T only)."""
    dense = 4 * Hq * (N / 2)
    sparse = 4 * Hq * top_k * BLOCK + 2 * Hp * (N / 2)
    return dense / sparse
