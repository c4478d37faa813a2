"""Seeded synthetic inputs for MSA training workloads.

This module only draws random numbers; it holds none of the method's arithmetic, so both the
CUDA path and the fp64 oracle consume the same values from it.

Recipe (every workload):
  * torch CPU generator seeded with ``seed``; fp32 draws rounded to bf16 (round to nearest even);
  * draw order Q [B,S,Hq,D], K [B,S,Hkv,D], V [B,S,Hkv,D], Qp [B,S,Hp,D], Kp [B,S,1,D],
    dO [B,S,Hq,D], all N(0, 1);
  * with ``planted > 0`` (selection made non-uniform): per sequence b, a unit direction u (a
    normalised N(0, I) draw) and ``planted`` distinct key blocks (a random permutation of the
    blocks, first ``planted`` taken).  ``plant_amp * u`` is added to every proxy-key row of those
    blocks and to every proxy-query row of the sequence, before the bf16 rounding.
"""
from __future__ import annotations

import dataclasses

import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    Hp: int
    top_k: int  # 0 = warmup (dense causal main attention, no selection)
    planted: int = 0
    plant_amp: float = 2.0
    D: int = 128

    @property
    def scale(self) -> float:
        return self.D ** -0.5

    @property
    def warmup(self) -> bool:
        return self.top_k == 0

    @property
    def nblk(self) -> int:
        return self.S // BLOCK

    def describe(self) -> str:
        mode = "warmup (dense)" if self.warmup else f"top_k={self.top_k}"
        extra = f", {self.planted} planted blocks" if self.planted else ""
        return (f"B={self.B} S={self.S} Hq={self.Hq} Hkv={self.Hkv} Hp={self.Hp} d={self.D} "
                f"{mode}{extra}")


# The five workloads of the method's training benchmark, then a profiling case (index =
# workload number - 1).
WORKLOADS = [
    Workload("msa_s1k", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4),
    Workload("msa_s8k_planted", B=2, S=8192, Hq=32, Hkv=8, Hp=8, top_k=16, planted=4),
    Workload("msa_s64k_planted", B=1, S=65536, Hq=64, Hkv=8, Hp=8, top_k=16, planted=4),
    Workload("msa_warmup_s32k", B=1, S=32768, Hq=32, Hkv=8, Hp=8, top_k=0),
    Workload("msa_s1m", B=1, S=1048576, Hq=16, Hkv=4, Hp=4, top_k=16),
    # the 64K workload's heads at 8K tokens: the small case its kernels are profiled on
    Workload("msa_s8k_g8_planted", B=1, S=8192, Hq=64, Hkv=8, Hp=8, top_k=16, planted=4),
]


def workload_seed(i: int) -> int:
    """Seed of workload number i (1-based)."""
    return 1000 + i


def make_inputs(w: Workload, seed: int, device="cpu"):
    """Draw the bf16 inputs of workload ``w``.  Returns dict q, k, v, qp, kp, dout (+ planted)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, S, D = w.B, w.S, w.D

    def draw(*shape):
        return torch.randn(*shape, generator=g, dtype=torch.float32)

    q = draw(B, S, w.Hq, D)
    k = draw(B, S, w.Hkv, D)
    v = draw(B, S, w.Hkv, D)
    qp = draw(B, S, w.Hp, D)
    kp = draw(B, S, 1, D)
    dout = draw(B, S, w.Hq, D)
    planted = []
    if w.planted:
        nblk = S // BLOCK
        for b in range(B):
            u = torch.randn(D, generator=g, dtype=torch.float32)
            u = u / u.norm()
            blocks = torch.randperm(nblk, generator=g)[: w.planted]
            planted.append(sorted(int(x) for x in blocks))
            for n in blocks.tolist():
                kp[b, n * BLOCK:(n + 1) * BLOCK, 0, :] += w.plant_amp * u
            qp[b] += w.plant_amp * u
    out = {name: t.to(torch.bfloat16).to(device)
           for name, t in dict(q=q, k=k, v=v, qp=qp, kp=kp, dout=dout).items()}
    out["planted"] = planted
    return out


def random_selection(B: int, Hp: int, S: int, top_k: int, seed: int, exclude: int = -1):
    """A seeded random valid block map [B, Hp, S, top_k] int32 (numpy): every row holds its local
    block t // 128 plus min(top_k, m + 1) - 1 distinct earlier blocks drawn uniformly (never
    ``exclude``), ascending, padded with -1.  It stands in for a selection where a test needs the
    gradient passes driven by an index map that both sides know without running the selection
    (the map is a plain input of the backward)."""
    import numpy as np

    rng = np.random.default_rng(seed)
    nblk = S // BLOCK
    k1 = top_k - 1
    out = np.full((B, Hp, S, top_k), -1, np.int32)
    t = np.arange(S)
    m = t // BLOCK
    step = max(1, (1 << 24) // max(nblk, 1))  # rows per draw: bounded host memory
    for b in range(B):
        for g in range(Hp):
            for r0 in range(0, S, step):
                r1 = min(S, r0 + step)
                mm = m[r0:r1]
                keys = rng.random((r1 - r0, nblk), dtype=np.float32)
                blk = np.arange(nblk)
                bad = (blk[None, :] >= mm[:, None]) | (blk[None, :] == exclude)
                keys[bad] = np.inf
                if k1 > 0:
                    pick = np.argpartition(keys, min(k1, nblk - 1), axis=1)[:, :k1] if nblk > k1 \
                        else np.argsort(keys, axis=1)[:, :k1]
                    ok = np.take_along_axis(keys, pick, axis=1) < np.inf
                    pick = np.where(ok, pick, nblk + 1)  # not enough visible blocks: padding
                else:
                    pick = np.zeros((r1 - r0, 0), np.int64)
                rows = np.concatenate([pick, mm[:, None]], axis=1)
                rows.sort(axis=1)
                rows[rows > nblk] = -1
                # padding (-1) sorted first: move it to the end of the row
                valid = rows >= 0
                order = np.argsort(~valid, axis=1, kind="stable")
                out[b, g, r0:r1] = np.take_along_axis(rows, order, axis=1)
    return out


def force_block(idx, rows, n: int):
    """Put block ``n`` into the given rows (b, g, t) of a map from random_selection in place of
    the row's first non-local block (each row must have t // 128 > n and no block n yet), keeping
    the row ascending.  Returns the map (modified in place)."""
    import numpy as np

    for b, g, t in rows:
        row = idx[b, g, t]
        m = t // BLOCK
        assert m > n and n not in row, (b, g, t)
        first = int(np.nonzero((row >= 0) & (row != m))[0][0])
        row[first] = n
        valid = np.sort(row[row >= 0])
        row[:] = -1
        row[:len(valid)] = valid
    return idx
