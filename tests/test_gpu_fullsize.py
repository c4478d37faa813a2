"""The benchmark workloads at full size, on sampled outputs the oracle computes one by one.

For each workload the CUDA path runs exactly as the benchmark runs it (same entry points, own
selection).  The oracle then computes, from the same inputs:
  * the selection of sampled rows: every group of a random set of tokens plus the last block's
    tokens -- compared bit-exactly (near ties excused);
  * with those rows' selection given to both sides: O and LSE of the sampled tokens (all heads),
    dQ / dQp of the sampled tokens, and dK / dV / dKp of the last 64 keys, which only the tokens
    of the last block can reach.
The oracle's fp64 inputs are lazily zeroed arrays with only the rows it reads filled in, so the
host memory stays small even at one million tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_qp_gb300 import binding as msa
from block_sparse_attention_qp_gb300.inputs import WORKLOADS, make_inputs, workload_seed
from tests.parity import close, compare_selection

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
WINDOW = 64  # trailing keys whose dK / dV / dKp are checked


def _f64_rows(t, tokens):
    """fp64 copy of [B,S,H,D] tensor t with only the given (b, token) rows filled (others 0)."""
    out = np.zeros(tuple(t.shape), np.float64)  # lazily allocated zero pages
    for b, ts in tokens.items():
        idx = torch.as_tensor(sorted(ts), dtype=torch.long)
        out[b, idx.numpy()] = t[b, idx].to(torch.float64).numpy()
    return out


def _sampled_tokens(w, rng, n_rand):
    toks = {}
    for b in range(w.B):
        r = set(rng.choice(w.S - WINDOW, size=n_rand, replace=False).tolist())
        r |= set(range(w.S - WINDOW, w.S))  # every token that can reach the window
        r |= {0, 1, 127, 128}
        toks[b] = r
    return toks


@pytest.mark.parametrize("wname,n_rand", [("msa_s64k_planted", 24), ("msa_s1m", 8)])
def test_fullsize_sparse_sampled(wname, n_rand):
    wi, w = [(i + 1, x) for i, x in enumerate(WORKLOADS) if x.name == wname][0]
    x = make_inputs(w, workload_seed(wi))
    g = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    _, _, gidx = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale)
    rng = np.random.default_rng(wi)
    toks = _sampled_tokens(w, rng, n_rand)
    rows = np.array([(b, gg, t) for b in toks for t in sorted(toks[b]) for gg in range(w.Hp)], np.int32)
    kp64 = oracle.f64(x["kp"])
    qp64 = _f64_rows(x["qp"], toks)
    osel, gap = oracle.select(qp64, kp64, w.top_k, w.scale, rows=rows)
    gsel = gidx[rows[:, 0], rows[:, 1], rows[:, 2]].cpu().numpy()
    n_bad, n_exc = compare_selection(gsel, osel, gap)
    print(f"{wname}: {len(rows)} sampled selection rows, {n_bad} differ (all near ties)")
    # both sides use the oracle's selection for the sampled rows
    idx_mix = gidx.clone()
    idx_mix[rows[:, 0], rows[:, 1], rows[:, 2]] = torch.from_numpy(osel).to(DEV)
    wsf = msa.workspace(msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale), msa.OP_FORWARD, DEV)
    o, lse, _ = msa.msa_forward(g["q"], g["k"], g["v"], g["qp"], g["kp"], w.top_k, w.scale,
                                block_idx=idx_mix, ws=wsf)
    assert msa.msa_device_status(wsf) == 0
    del wsf
    wsb = msa.workspace(msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale), msa.OP_BACKWARD, DEV)
    dq, dk, dv, dqp, dkp = msa.msa_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse,
                                            g["dout"], idx_mix, w.top_k, w.scale, ws=wsb)
    assert msa.msa_device_status(wsb) == 0
    del wsb
    torch.cuda.synchronize()
    idx_o = np.full((w.B, w.Hp, w.S, w.top_k), -1, np.int32)
    idx_o[rows[:, 0], rows[:, 1], rows[:, 2]] = osel
    q64, do64 = _f64_rows(x["q"], toks), _f64_rows(x["dout"], toks)
    k64, v64 = oracle.f64(x["k"]), oracle.f64(x["v"])
    frows = np.array([(b, t, h) for b in toks for t in sorted(toks[b]) for h in range(w.Hq)], np.int32)
    o_ref, lse_ref = oracle.forward(q64, k64, v64, idx_o, w.top_k, w.scale, rows=frows, Hp=w.Hp)
    close("O", o[frows[:, 0], frows[:, 1], frows[:, 2]], o_ref)
    close("LSE", lse[frows[:, 0], frows[:, 2], frows[:, 1]], lse_ref)
    mask = np.zeros((w.B, w.S), bool)
    for b in toks:
        mask[b, sorted(toks[b])] = True
    ref = oracle.backward(q64, k64, v64, qp64, kp64, do64, idx_o, w.top_k, w.scale,
                          tok_mask=mask, key_window=(w.S - WINDOW, w.S))
    bi, ti = np.nonzero(mask)
    close("dq", dq[bi, ti], ref["dq"][bi, ti])
    close("dqp", dqp[bi, ti], ref["dqp"][bi, ti])
    win = slice(w.S - WINDOW, w.S)
    close("dk", dk[:, win], ref["dk"][:, win])
    close("dv", dv[:, win], ref["dv"][:, win])
    close("dkp", dkp[:, win], ref["dkp"][:, win])


def test_fullsize_warmup_sampled():
    wi, w = [(i + 1, x) for i, x in enumerate(WORKLOADS) if x.name == "msa_warmup_s32k"][0]
    x = make_inputs(w, workload_seed(wi))
    g = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o, lse = msa.msa_warmup_forward(g["q"], g["k"], g["v"], w.scale)
    dq, dk, dv, dqp, dkp = msa.msa_warmup_backward(g["q"], g["k"], g["v"], g["qp"], g["kp"], o, lse,
                                                   g["dout"], w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(wi)
    toks = _sampled_tokens(w, rng, 6)
    q64, do64, qp64 = (_f64_rows(x[n], toks) for n in ("q", "dout", "qp"))
    k64, v64, kp64 = oracle.f64(x["k"]), oracle.f64(x["v"]), oracle.f64(x["kp"])
    frows = np.array([(b, t, h) for b in toks for t in sorted(toks[b]) for h in range(w.Hq)], np.int32)
    o_ref, lse_ref = oracle.forward(q64, k64, v64, None, 1, w.scale, rows=frows, Hp=w.Hp)
    close("O", o[frows[:, 0], frows[:, 1], frows[:, 2]], o_ref)
    close("LSE", lse[frows[:, 0], frows[:, 2], frows[:, 1]], lse_ref)
    mask = np.zeros((w.B, w.S), bool)
    for b in toks:
        mask[b, sorted(toks[b])] = True
    ref = oracle.backward(q64, k64, v64, qp64, kp64, do64, None, 1, w.scale, tok_mask=mask,
                          key_window=(w.S - WINDOW, w.S))
    bi, ti = np.nonzero(mask)
    close("dq", dq[bi, ti], ref["dq"][bi, ti])
    close("dqp", dqp[bi, ti], ref["dqp"][bi, ti])
    win = slice(w.S - WINDOW, w.S)
    close("dk", dk[:, win], ref["dk"][:, win])
    close("dv", dv[:, win], ref["dv"][:, win])
    close("dkp", dkp[:, win], ref["dkp"][:, win])


def test_fullsize_multichunk_key_window():
    """dK / dV / dKp of a mid-sequence key block that tokens of every backward chunk reach, at
    the 64K workload's full size and launch configuration.

    The backward splits each key block's token list by sequence chunk (8192 tokens at 64K with
    8 heads per group: 32 MB of fp32 dQ rows per proxy head) and items of different chunks add
    their dK / dV / dKp into the same rows
    at different times.  The last-window check above cannot see that (only the last block's
    tokens reach the last keys).  Here both sides run on one seeded random index map
    (random_selection, the same input for both) in which block FOCUS is put into the selection of
    tokens from all eight chunks -- 600 of them in one chunk for group 0, so that list spans two
    work items -- and of nobody else but the block's own tokens.  The oracle then computes every
    contribution to that block exactly (it visits every row whose key set touches the window)."""
    from block_sparse_attention_qp_gb300.inputs import force_block, random_selection

    wi, w = [(i + 1, x) for i, x in enumerate(WORKLOADS) if x.name == "msa_s64k_planted"][0]
    FOCUS = 50  # keys 6400 .. 6527, in the first chunk
    x = make_inputs(w, workload_seed(wi))
    idx = random_selection(w.B, w.Hp, w.S, w.top_k, seed=4321, exclude=FOCUS)
    rng = np.random.default_rng(99)
    chunk = 8192
    forced = []
    for g in range(w.Hp):
        for c in range(w.S // chunk):
            lo = max(c * chunk, (FOCUS + 1) * 128)
            n = 600 if (g == 0 and c == 1) else 20
            for t in rng.choice(np.arange(lo, (c + 1) * chunk), size=n, replace=False):
                forced.append((0, g, int(t)))
    force_block(idx, forced, FOCUS)
    g_ = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    idx_d = torch.from_numpy(idx).to(DEV)
    o, lse, _ = msa.msa_forward(g_["q"], g_["k"], g_["v"], g_["qp"], g_["kp"], w.top_k, w.scale,
                                block_idx=idx_d)
    wsb = msa.workspace(msa.make_shape(g_["q"], g_["k"], g_["qp"], w.top_k, w.scale),
                        msa.OP_BACKWARD, DEV)
    dq, dk, dv, dqp, dkp = msa.msa_backward(g_["q"], g_["k"], g_["v"], g_["qp"], g_["kp"], o,
                                            lse, g_["dout"], idx_d, w.top_k, w.scale, ws=wsb)
    assert msa.msa_device_status(wsb) == 0
    del wsb
    torch.cuda.synchronize()
    # every token whose key set touches the block: the forced ones and the block's own tokens
    touch = {t for _, _, t in forced} | set(range(FOCUS * 128, (FOCUS + 1) * 128))
    toks = {0: touch}
    q64, do64, qp64 = (_f64_rows(x[n], toks) for n in ("q", "dout", "qp"))
    k64, v64, kp64 = oracle.f64(x["k"]), oracle.f64(x["v"]), oracle.f64(x["kp"])
    sample = sorted(rng.choice(sorted(touch), size=24, replace=False).tolist())
    mask = np.zeros((w.B, w.S), bool)
    mask[0, sample] = True
    j0, j1 = FOCUS * 128, (FOCUS + 1) * 128
    ref = oracle.backward(q64, k64, v64, qp64, kp64, do64, idx, w.top_k, w.scale,
                          tok_mask=mask, key_window=(j0, j1))
    print(f"{len(forced)} forced rows over {w.S // chunk} chunks, {len(touch)} tokens reach "
          f"keys {j0}..{j1 - 1}")
    close("dk window", dk[:, j0:j1], ref["dk"][:, j0:j1])
    close("dv window", dv[:, j0:j1], ref["dv"][:, j0:j1])
    close("dkp window", dkp[:, j0:j1], ref["dkp"][:, j0:j1])
    close("dq sample", dq[0, sample], ref["dq"][0, sample])
    close("dqp sample", dqp[0, sample], ref["dqp"][0, sample])
    frows = np.array([(0, t, h) for t in sample for h in range(w.Hq)], np.int32)
    o_ref, lse_ref = oracle.forward(q64, k64, v64, idx, w.top_k, w.scale, rows=frows, Hp=w.Hp)
    close("O sample", o[frows[:, 0], frows[:, 1], frows[:, 2]], o_ref)
    close("LSE sample", lse[frows[:, 0], frows[:, 2], frows[:, 1]], lse_ref)
