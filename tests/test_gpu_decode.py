"""The decode step (msa_decode) against the oracle's rows and against the training forward.

Decoding token t_b of sequence b is, by definition, row t_b of the whole-sequence computation:
the oracle's selection of row (b, g, t_b) and its attention output of rows (b, t_b, h) -- computed
one by one from the same caches -- are the references (forum summary, "GPU kernel co-design";
blog, "Proxy attention", "Main attention")."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_qp_gb300 import binding as msa
from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs
from tests.parity import close, compare_selection

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _decode_case(w, lens, seed):
    x = make_inputs(w, seed)
    lens = np.asarray(lens, np.int32)
    t = lens - 1
    bi = np.arange(w.B)
    q = x["q"][bi, t].contiguous()    # [B, Hq, D]: the new token of each sequence
    qp = x["qp"][bi, t].contiguous()  # [B, Hp, D]
    return x, lens, t, q, qp


def _check_against_oracle(w, lens, seed):
    x, lens, t, q, qp = _decode_case(w, lens, seed)
    o, lse, idx = msa.msa_decode(q.to(DEV), qp.to(DEV), x["k"].to(DEV), x["v"].to(DEV),
                                 x["kp"].to(DEV), torch.from_numpy(lens).to(DEV), w.top_k, w.scale)
    torch.cuda.synchronize()
    # oracle selection of rows (b, g, t_b) from the same caches
    rows = np.array([(b, g, int(t[b])) for b in range(w.B) for g in range(w.Hp)], np.int32)
    osel, gap = oracle.select(x["qp"], x["kp"], w.top_k, w.scale, rows=rows)
    gsel = idx.cpu().numpy().reshape(-1, w.top_k)
    n_bad, _ = compare_selection(gsel, osel, gap)
    full = np.full((w.B, w.Hp, w.S, w.top_k), -1, np.int32)
    full[rows[:, 0], rows[:, 1], rows[:, 2]] = osel
    frows = np.array([(b, int(t[b]), h) for b in range(w.B) for h in range(w.Hq)], np.int32)
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], full, w.top_k, w.scale, rows=frows)
    # compare the rows whose selection agrees (a near tie may flip a block; none expected here)
    same = np.array([(gsel[b * w.Hp:(b + 1) * w.Hp] == osel[b * w.Hp:(b + 1) * w.Hp]).all()
                     for b in range(w.B)])
    keep = np.repeat(same, w.Hq)
    assert same.sum() >= w.B - n_bad
    close("O", o.reshape(-1, w.D)[torch.from_numpy(keep)], o_ref[keep])
    close("LSE", lse.reshape(-1)[torch.from_numpy(keep)], lse_ref[keep])
    return n_bad


@pytest.mark.parametrize("name,B,S,Hq,Hkv,Hp,k,lens", [
    ("g8", 6, 1024, 16, 2, 2, 4, [1, 127, 128, 129, 700, 1024]),
    ("g4_k16", 4, 4096, 16, 4, 4, 16, [4096, 2000, 300, 3333]),
    ("hp_lt_hkv", 5, 1536, 16, 4, 2, 6, [1536, 1, 640, 641, 1000]),
    ("hp_gt_hkv_g2", 3, 768, 8, 2, 4, 3, [768, 129, 500]),
    ("g16", 3, 640, 32, 2, 2, 4, [640, 200, 129]),      # 16 heads per group: the MMA's full N
    ("g1", 3, 512, 4, 4, 4, 3, [512, 128, 300]),        # one head per group
    ("hp32", 2, 384, 64, 32, 32, 3, [384, 250]),        # 32 proxy heads: the N = 32 score product
])
def test_decode_matches_oracle_rows(name, B, S, Hq, Hkv, Hp, k, lens):
    w = Workload(name, B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hp, top_k=k)
    _check_against_oracle(w, lens, seed=900 + S + Hq)


def test_decode_equals_training_forward_last_row():
    """Decoding the last token of full caches gives the training forward's last row."""
    w = Workload("last", B=3, S=2048, Hq=16, Hkv=2, Hp=2, top_k=8)
    x, lens, t, q, qp = _decode_case(w, [2048] * 3, 41)
    g = {n: x[n].to(DEV) for n in ("q", "k", "v", "qp", "kp")}
    o_f, lse_f, idx_f = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale)
    o_d, lse_d, idx_d = msa.msa_decode(q.to(DEV), qp.to(DEV), g["k"], g["v"], g["kp"],
                                       torch.from_numpy(lens).to(DEV), w.top_k, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(idx_d, idx_f[:, :, -1])
    close("O", o_d, o_f[:, -1].float(), rel=5e-3, ulps=1.5)
    close("LSE", lse_d, lse_f[:, :, -1], rel=1e-5, atol=1e-4, ulps=0.0)


def test_decode_flags_bad_lengths():
    w = Workload("bad", B=3, S=512, Hq=8, Hkv=2, Hp=2, top_k=3)
    x, _, _, q, qp = _decode_case(w, [512, 512, 512], 5)
    lens = torch.tensor([512, 0, 513], dtype=torch.int32, device=DEV)  # two out of range
    shape = msa.Shape(w.B, w.S, w.Hq, w.Hkv, w.Hp, 128, w.top_k, w.scale)
    ws = msa.workspace(shape, msa.OP_DECODE, DEV)
    o, lse, idx = msa.msa_decode(q.to(DEV), qp.to(DEV), x["k"].to(DEV), x["v"].to(DEV),
                                 x["kp"].to(DEV), lens, w.top_k, w.scale, ws=ws)
    assert msa.msa_device_status(ws) & 1
    assert torch.isfinite(o[0].float()).all()
