"""Pins for the fp64 oracle: checks against things other than the oracle itself.

* brute-force top-k properties on tiny inputs, hand-built ties (lower block index wins), the
  forced local block, padding when fewer blocks than k are visible;
* with k >= number of blocks, sparse MSA is dense causal GQA attention: forward against
  torch's scaled_dot_product_attention (fp64) and backward against its autograd;
* central finite differences of the total loss (frozen indices) for every gradient, which
  checks the closed-form KL gradient against the materialised KL value;
* KL >= 0, KL == 0 when the student equals the teacher, sum_j dz_j == 0;
* a second independent fp64 implementation in eager PyTorch (stable-sort top-k, autograd KL);
* the number of selected tokens per query (k * 128 = 2048 at k = 16) from the forum summary.

Sources: Flash-MSA blog sections "About MSA", "Proxy attention", "Main attention", "Backward",
"KL Divergence Loss", "Warmup kernels"; MSA forum summary, "Architecture" and "Training
stability".
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_qp_gb300.inputs import Workload, make_inputs
from tests.eager_msa import eager_msa, eager_select

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(S=512, Hq=4, Hkv=2, top_k=3, D=128, seed=7, planted=0, B=1, Hp=None):
    w = Workload("tiny", B=B, S=S, Hq=Hq, Hkv=Hkv, Hp=Hkv if Hp is None else Hp, top_k=top_k,
                 planted=planted, D=D)
    return w, make_inputs(w, seed)


def block_scores_np(qp, kp, scale):
    """Block max of the proxy scores via a library matmul: c[b,g,t,n] (all blocks, unmasked)."""
    qp = oracle.f64(qp)
    kp = oracle.f64(kp)[:, :, 0, :]
    B, S, Hp, D = qp.shape
    z = scale * np.einsum("bthd,bjd->bhtj", qp, kp)
    return z.reshape(B, Hp, S, S // 128, 128).max(-1)


# ----------------------------------------------------------------------------- top-k


@pytest.mark.parametrize("top_k", [1, 2, 3, 5, 8])
def test_selection_brute_force_properties(top_k, B=2, S=768):
    w, x = tiny(S=S, top_k=top_k, seed=11, B=B)
    idx, gap = oracle.select(x["qp"], x["kp"], top_k, w.scale)
    c = block_scores_np(x["qp"], x["kp"], w.scale)
    B, Hp, S, _ = idx.shape
    for b in range(B):
        for g in range(Hp):
            for t in range(S):
                m = t // 128
                row = idx[b, g, t]
                K = min(top_k, m + 1)
                sel = [int(n) for n in row if n >= 0]
                assert len(sel) == K and all(n == -1 for n in row[K:])
                assert sel == sorted(sel) and len(set(sel)) == K
                assert m in sel, "local block must always be selected"
                assert all(0 <= n <= m for n in sel)
                rest = [n for n in range(m) if n not in sel]
                for a in sel:
                    if a == m:
                        continue
                    for r in rest:  # every chosen block beats every other visible block
                        assert (c[b, g, t, a], -a) > (c[b, g, t, r], -r)


def test_selection_exhaustive_small():
    """Enumerate every admissible subset: the oracle's must be the best by sorted score vector."""
    import itertools

    w, x = tiny(S=768, top_k=3, seed=3)
    idx, _ = oracle.select(x["qp"], x["kp"], 3, w.scale)
    c = block_scores_np(x["qp"], x["kp"], w.scale)
    for t in range(0, 768, 37):
        m = t // 128
        for g in range(2):
            K = min(3, m + 1)
            best = None
            for comb in itertools.combinations(range(m), K - 1):
                key = sorted([(c[0, g, t, n], -n) for n in comb], reverse=True)
                if best is None or key > best[0]:
                    best = (key, comb)
            want = sorted(list(best[1]) + [m])
            got = [int(n) for n in idx[0, g, t] if n >= 0]
            assert got == want


def test_selection_ties_prefer_lower_block():
    """Identical proxy-key blocks give equal block scores; the lower block index must win."""
    w, x = tiny(S=1024, top_k=2, seed=5)
    g = torch.Generator().manual_seed(0)
    u = torch.randn(128, generator=g)
    u = 3.0 * u / u.norm()
    qp = u.expand(1, 1024, 2, 128).to(torch.bfloat16).contiguous()  # every proxy query = u
    kp = (0.05 * torch.randn(1, 1024, 1, 128, generator=g)).to(torch.bfloat16)
    kp[0, 2 * 128:3 * 128, 0, :] = u.to(torch.bfloat16)  # blocks 2 and 5: exact copies of u,
    kp[0, 5 * 128:6 * 128, 0, :] = u.to(torch.bfloat16)  # so they tie for the best score
    idx, gap = oracle.select(qp, kp, 2, w.scale)
    c = block_scores_np(qp, kp, w.scale)
    for t in range(6 * 128, 1024):  # both visible; top_k=2 -> local block + one of {2, 5}
        m = t // 128
        assert c[0, 0, t, 2] == c[0, 0, t, 5] == c[0, 0, t, :m].max()
        for gg in range(2):
            assert [int(n) for n in idx[0, gg, t]] == [2, m]
            assert gap[0, gg, t] == 0.0


def _uniform_block_keys(vecs, S):
    """Proxy keys whose 128 rows in block n all equal vecs[n]: block n's score is then exactly
    scale * qp . vecs[n] (no max over differing keys)."""
    kp = torch.zeros(1, S, 1, 128)
    for n, v in enumerate(vecs):
        kp[0, n * 128:(n + 1) * 128, 0, :] = v
    return kp.to(torch.bfloat16)


def _e(i, a=1.0):
    v = torch.zeros(128)
    v[i] = a
    return v


GAP_CASES = {
    # name: (proxy query row, block key vectors, top_k, {query block m: expected gap})
    # qp = e0 + e1 and block n = e0 + d_n e1 give block scores scale * (1 + d_n), all exact in
    # bf16 and fp64; the near-tie gap is (lowest selected - highest unselected non-local score)
    # / max(|lowest selected|, |highest unselected|).
    "positive": (_e(0) + _e(1),
                 [_e(0) + _e(1, 2.0 ** -9), _e(0), _e(0) + _e(1, 2.0 ** -11), _e(0, 0.5),
                  _e(0) + _e(1, 2.0 ** -7)],
                 3,
                 {5: (2.0 ** -9 - 2.0 ** -11) / (1 + 2.0 ** -9),   # picks 4, 0; best left out: 2
                  4: 2.0 ** -11 / (1 + 2.0 ** -11),               # picks 0, 2; best left out: 1
                  3: 2.0 ** -11 / (1 + 2.0 ** -11),
                  2: math.inf, 1: math.inf, 0: math.inf}),      # nothing visible left out
    # the same keys against -qp: every score changes sign, the order reverses
    "negative": (-(_e(0) + _e(1)),
                 [_e(0) + _e(1, 2.0 ** -9), _e(0), _e(0) + _e(1, 2.0 ** -11), _e(0, 0.5),
                  _e(0) + _e(1, 2.0 ** -7)],
                 3,
                 {5: 2.0 ** -11 / (1 + 2.0 ** -11),   # picks 3 (-0.5), 1 (-1); left out: 2
                  4: 2.0 ** -11 / (1 + 2.0 ** -11),   # visible 0-3: same picks and left-out
                  3: (2.0 ** -9 - 2.0 ** -11) / (1 + 2.0 ** -9)}),  # picks 1, 2; left out: 0
    # one non-local pick: +1/4 chosen over -1/4 and -1 -> gap (1/4 + 1/4) / (1/4) = 2
    "mixed sign": (_e(0) + _e(1), [_e(0, 0.25), _e(0, -0.25), _e(0, -1.0)], 2,
                   {3: 2.0, 2: 2.0, 1: math.inf}),
}


@pytest.mark.parametrize("case", sorted(GAP_CASES))
def test_selection_gap_closed_form(case):
    """The near-tie gap the parity rule excuses mismatches by, on block scores known exactly."""
    qrow, vecs, top_k, want = GAP_CASES[case]
    S = 768
    kp = _uniform_block_keys(vecs, S)
    qp = qrow.to(torch.bfloat16).expand(1, S, 2, 128).contiguous()
    scale = 128 ** -0.5
    idx, gap = oracle.select(qp, kp, top_k, scale)
    for m, g in want.items():
        for t in (128 * m, 128 * m + 77, 128 * m + 127):
            for gg in range(2):
                if math.isinf(g):
                    assert math.isinf(gap[0, gg, t]), (case, m, gap[0, gg, t])
                else:
                    assert abs(gap[0, gg, t] - g) <= 1e-12 * abs(g), (case, m, gap[0, gg, t], g)


def test_selection_gap_brute_force_random():
    """Gap on random and planted inputs against block scores from a library matmul."""
    for seed, planted in ((31, 0), (37, 4)):
        w, x = tiny(S=1024, top_k=4, seed=seed, planted=planted)
        idx, gap = oracle.select(x["qp"], x["kp"], 4, w.scale)
        c = block_scores_np(x["qp"], x["kp"], w.scale)
        for g in range(2):
            for t in range(0, 1024, 13):
                m = t // 128
                sel = [int(n) for n in idx[0, g, t] if 0 <= n < m]
                rest = [n for n in range(m) if n not in sel]
                if not sel or not rest:
                    assert math.isinf(gap[0, g, t])
                    continue
                lo = min(c[0, g, t, n] for n in sel)
                hi = max(c[0, g, t, n] for n in rest)
                want = (lo - hi) / max(abs(lo), abs(hi))
                assert want >= 0 and abs(gap[0, g, t] - want) <= 1e-9 * max(1.0, want)


def test_selection_k_covers_everything():
    w, x = tiny(S=640, top_k=5, seed=9)
    idx, gap = oracle.select(x["qp"], x["kp"], 5, w.scale)
    for t in range(640):
        m = t // 128
        assert list(idx[0, 0, t, :m + 1]) == list(range(m + 1))
        assert math.isinf(gap[0, 0, t])


def test_selected_tokens_per_query():
    """k=16, B_k=128 gives ~2048 selected tokens per query (forum summary, "Architecture")."""
    with open(os.path.join(GOLDEN, "tokens_per_query.json")) as f:
        gold = json.load(f)
    w, x = tiny(S=128 * 20, Hq=2, Hkv=1, top_k=gold["top_k"], D=16, seed=1)
    idx, _ = oracle.select(x["qp"], x["kp"], w.top_k, w.scale)
    t = 128 * 20 - 1  # last token of a block: every selected block fully visible
    sel = [int(n) for n in idx[0, 0, t] if n >= 0]
    assert len(sel) * 128 == gold["tokens_per_query"]


# ----------------------------------------------------------------------------- dense == SDPA


def sdpa_reference(q, k, v, scale):
    """torch SDPA in fp64 with the GQA heads expanded (library routine)."""
    G = q.shape[2] // k.shape[2]
    qh = q.permute(0, 2, 1, 3)
    kh = k.repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    vh = v.repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=True, scale=scale)
    return o.permute(0, 2, 1, 3)


@pytest.mark.parametrize("warmup", [False, True])
def test_full_selection_is_dense_causal_attention(warmup):
    w, x = tiny(S=512, Hq=4, Hkv=2, top_k=4, seed=21)
    q, k, v, dout = (x[n].double() for n in ("q", "k", "v", "dout"))
    idx = None
    if not warmup:
        idx, _ = oracle.select(x["qp"], x["kp"], 4, w.scale)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], idx, 4, w.scale)
    ref = sdpa_reference(q, k, v, w.scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-10, atol=1e-12)
    # LSE via torch.logsumexp of the causally masked scores
    G = 2
    s = w.scale * torch.einsum("bthd,bjhd->bhtj", q, k.repeat_interleave(G, dim=2))
    s = s.masked_fill(~torch.tril(torch.ones(512, 512, dtype=torch.bool)), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)
    # backward of the main loss against autograd of SDPA
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    (sdpa_reference(qq, kk, vv, w.scale) * dout).sum().backward()
    g = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 4, w.scale)
    for name, ref_g in (("dq", qq.grad), ("dk", kk.grad), ("dv", vv.grad)):
        np.testing.assert_allclose(g[name], ref_g.numpy(), rtol=1e-9, atol=1e-10, err_msg=name)


def test_warmup_equals_sparse_with_every_block():
    w, x = tiny(S=384, Hq=4, Hkv=2, top_k=3, seed=4)
    idx, _ = oracle.select(x["qp"], x["kp"], 3, w.scale)
    a = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 3, w.scale)
    b = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], None, 3, w.scale)
    for name in ("dq", "dk", "dv", "dqp", "dkp"):
        np.testing.assert_allclose(a[name], b[name], rtol=1e-12, atol=1e-15, err_msg=name)
    assert abs(a["kl"] - b["kl"]) < 1e-12


# ----------------------------------------------------------------------------- finite differences


def _fd_case(Hq=4, Hkv=2, Hp=None):
    w, x = tiny(S=384, Hq=Hq, Hkv=Hkv, top_k=2, D=16, seed=13, Hp=Hp)
    idx, _ = oracle.select(x["qp"], x["kp"], 2, w.scale)
    arrs = {n: oracle.f64(x[n]) for n in ("q", "k", "v", "qp", "kp", "dout")}
    return w, idx, arrs


def _main_loss(w, idx, a):
    o, _ = oracle.forward(a["q"], a["k"], a["v"], idx, w.top_k, w.scale)
    return float((o * a["dout"]).sum())


def _kl(w, idx, a, warmup=False):
    return oracle.backward(a["q"], a["k"], a["v"], a["qp"], a["kp"], a["dout"],
                           None if warmup else idx, w.top_k, w.scale)["kl"]


@pytest.mark.parametrize("warmup", [False, True])
def test_finite_differences_every_gradient(warmup, n_coords=6, heads=None):
    w, idx, a = _fd_case(*(heads or ()))
    kl_grad = 0.75
    use_idx = None if warmup else idx
    g = oracle.backward(a["q"], a["k"], a["v"], a["qp"], a["kp"], a["dout"], use_idx, w.top_k,
                        w.scale, kl_grad=kl_grad)
    rng = np.random.default_rng(0)
    eps = 1e-5
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("qp", "dqp"), ("kp", "dkp")):
        arr = a[name]
        for _ in range(n_coords):
            pos = tuple(int(rng.integers(0, s)) for s in arr.shape)
            vals = []
            for sgn in (+1, -1):
                b = dict(a)
                b[name] = arr.copy()
                b[name][pos] += sgn * eps
                if name in ("q", "k", "v"):
                    # teacher is detached: the KL term contributes nothing to dq/dk/dv
                    if warmup:
                        o, _ = oracle.forward(b["q"], b["k"], b["v"], None, w.top_k, w.scale)
                        vals.append(float((o * b["dout"]).sum()))
                    else:
                        vals.append(_main_loss(w, idx, b))
                else:
                    vals.append(kl_grad * _kl(w, idx, b, warmup))
            fd = (vals[0] - vals[1]) / (2 * eps)
            an = g[gname][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)) + 1e-9, (name, pos, fd, an)


@pytest.mark.parametrize("Hq,Hkv,Hp", [(4, 1, 2), (8, 4, 2), (8, 2, 1), (4, 2, 4)])
def test_finite_differences_general_mapping(Hq, Hkv, Hp, n_coords=4):
    """Every gradient against central differences when proxy heads and KV heads differ in
    number (teacher over the proxy head's Hq/Hp query heads; keys of each head's own KV head)."""
    for warmup in (False, True):
        test_finite_differences_every_gradient(warmup, n_coords=n_coords, heads=(Hq, Hkv, Hp))


# ----------------------------------------------------------------------------- KL properties


def test_kl_nonnegative_and_zero_gradient_sum():
    w, x = tiny(S=512, seed=17)
    idx, _ = oracle.select(x["qp"], x["kp"], 3, w.scale)
    g = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 3, w.scale)
    assert g["kl"] > 0
    # sum_j dz_j = 0 per row: with every proxy key equal, dQp = scale * (sum_j dz_j) * kp = 0
    kp = x["kp"].clone()
    kp[:] = kp[0, 0]
    g2 = oracle.backward(x["q"], x["k"], x["v"], x["qp"], kp, x["dout"], idx, 3, w.scale)
    assert np.abs(g2["dqp"]).max() < 1e-15


def test_kl_zero_when_proxy_head_spans_several_kv_heads():
    """Hp < Hkv: every query head of proxy head g equals Qp[g] and every key head equals Kp, so
    each head's softmax is the student and so is their mean over the Hkv/Hp GQA groups."""
    Hq, Hkv, Hp = 8, 4, 2
    w, x = tiny(S=512, Hq=Hq, Hkv=Hkv, Hp=Hp, seed=41)
    qp, kp = x["qp"], x["kp"]
    q = qp.repeat_interleave(Hq // Hp, dim=2)
    k = kp.expand(-1, -1, Hkv, -1).contiguous()
    idx, _ = oracle.select(qp, kp, 3, w.scale)
    g = oracle.backward(q, k, x["v"], qp, kp, x["dout"], idx, 3, w.scale)
    assert abs(g["kl"]) < 1e-13
    assert np.abs(g["dqp"]).max() < 1e-15 and np.abs(g["dkp"]).max() < 1e-15


@pytest.mark.parametrize("G", [1, 2])
def test_kl_zero_when_student_equals_teacher(G):
    Hkv = 2
    w, x = tiny(S=512, Hq=G * Hkv, Hkv=Hkv, seed=19)
    qp, kp = x["qp"], x["kp"]
    q = qp.repeat_interleave(G, dim=2)  # every query head of group g equals proxy query g
    k = kp.expand(-1, -1, Hkv, -1).contiguous()  # every key head equals the proxy key head
    idx, _ = oracle.select(qp, kp, 3, w.scale)
    g = oracle.backward(q, k, x["v"], qp, kp, x["dout"], idx, 3, w.scale)
    assert abs(g["kl"]) < 1e-13
    assert np.abs(g["dqp"]).max() < 1e-15 and np.abs(g["dkp"]).max() < 1e-15


# ----------------------------------------------------------------------------- second implementation


# (B, S, Hq, Hkv, Hp, top_k): Hp == Hkv, then proxy heads fewer than KV heads (one proxy head
# selects for several GQA groups) and more (a GQA group split among proxy heads)
EAGER_SHAPES = [(1, 384, 4, 2, 2, 2), (2, 512, 4, 1, 1, 3), (1, 640, 6, 3, 3, 4),
                (1, 384, 8, 4, 2, 2), (1, 512, 8, 4, 1, 3), (2, 384, 8, 1, 2, 2),
                (1, 512, 8, 2, 4, 3)]


@pytest.mark.parametrize("warmup", [False, True])
@pytest.mark.parametrize("shape", EAGER_SHAPES)
def test_eager_second_implementation(shape, warmup):
    B, S, Hq, Hkv, Hp, top_k = shape
    w, x = tiny(S=S, Hq=Hq, Hkv=Hkv, top_k=top_k, D=32, seed=S + Hq, B=B, planted=0, Hp=Hp)
    d = {n: x[n].double() for n in ("q", "k", "v", "qp", "kp", "dout")}
    idx, _ = oracle.select(x["qp"], x["kp"], top_k, w.scale)
    if not warmup:
        e_idx = eager_select(d["qp"], d["kp"], top_k, w.scale)
        assert np.array_equal(e_idx.numpy(), idx)
    ref = eager_msa(d["q"], d["k"], d["v"], d["qp"], d["kp"], d["dout"], torch.from_numpy(idx),
                    w.scale, kl_grad=1.3, warmup=warmup)
    use = None if warmup else idx
    o, lse = oracle.forward(x["q"], x["k"], x["v"], use, top_k, w.scale)
    g = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], use, top_k,
                        w.scale, kl_grad=1.3)
    np.testing.assert_allclose(o, ref["o"].numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref["lse"].numpy(), rtol=1e-12, atol=1e-12)
    assert abs(g["kl"] - ref["kl"]) < 1e-10
    for name in ("dq", "dk", "dv", "dqp", "dkp"):
        np.testing.assert_allclose(g[name], ref[name].numpy(), rtol=1e-8, atol=1e-12,
                                   err_msg=name)


def test_sampled_backward_matches_full():
    """The sampling options (token mask, key window) return exactly the full values."""
    w, x = tiny(S=640, Hq=4, Hkv=2, top_k=3, seed=23)
    idx, _ = oracle.select(x["qp"], x["kp"], 3, w.scale)
    full = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 3, w.scale)
    mask = np.zeros((1, 640), bool)
    mask[0, [0, 5, 200, 639]] = True
    part = oracle.backward(x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 3, w.scale,
                           tok_mask=mask, key_window=(512, 640))
    for name in ("dq", "dqp"):
        np.testing.assert_allclose(part[name][:, mask[0]], full[name][:, mask[0]], rtol=1e-13,
                                   atol=1e-16)
    for name in ("dk", "dv", "dkp"):
        np.testing.assert_allclose(part[name][:, 512:], full[name][:, 512:], rtol=1e-13,
                                   atol=1e-16)
    rows = np.array([[0, 0, 1], [0, 300, 3], [0, 639, 2]], np.int32)
    o_s, lse_s = oracle.forward(x["q"], x["k"], x["v"], idx, 3, w.scale, rows=rows)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], idx, 3, w.scale)
    for r, (b, t, h) in enumerate(rows):
        np.testing.assert_array_equal(o_s[r], o[b, t, h])
        assert lse_s[r] == lse[b, h, t]
    srows = np.array([[0, 1, 600], [0, 0, 130]], np.int32)
    i_s, _ = oracle.select(x["qp"], x["kp"], 3, w.scale, rows=srows)
    for r, (b, g_, t) in enumerate(srows):
        np.testing.assert_array_equal(i_s[r], idx[b, g_, t])


def test_token_restricted_backward_partitions_the_gradient():
    """Contributions of disjoint token sets (only_masked) add up to the full gradients."""
    w, x = tiny(S=512, Hq=4, Hkv=2, top_k=3, seed=29)
    idx, _ = oracle.select(x["qp"], x["kp"], 3, w.scale)
    args = (x["q"], x["k"], x["v"], x["qp"], x["kp"], x["dout"], idx, 3, w.scale)
    full = oracle.backward(*args)
    mask = np.zeros((1, 512), bool)
    mask[0, ::3] = True
    a = oracle.backward(*args, tok_mask=mask, only_masked=True)
    b = oracle.backward(*args, tok_mask=~mask, only_masked=True)
    for name in ("dq", "dk", "dv", "dqp", "dkp"):
        np.testing.assert_allclose(a[name] + b[name], full[name], rtol=1e-12, atol=1e-15)
    assert abs(a["kl"] + b["kl"] - full["kl"]) < 1e-12
