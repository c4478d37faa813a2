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


# The five workloads of the method's training benchmark (index = workload number - 1).
WORKLOADS = [
    Workload("msa_s1k", B=1, S=1024, Hq=8, Hkv=2, Hp=2, top_k=4),
    Workload("msa_s8k_planted", B=2, S=8192, Hq=32, Hkv=8, Hp=8, top_k=16, planted=4),
    Workload("msa_s64k_planted", B=1, S=65536, Hq=64, Hkv=8, Hp=8, top_k=16, planted=4),
    Workload("msa_warmup_s32k", B=1, S=32768, Hq=32, Hkv=8, Hp=8, top_k=0),
    Workload("msa_s1m", B=1, S=1048576, Hq=16, Hkv=4, Hp=4, top_k=16),
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
