"""The work model used for TFLOP/s reporting, pinned to the figures the pages print."""
import json
import os

from block_sparse_attention_qp_gb300 import flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_per_token_reduction_matches_the_published_figure():
    g = json.load(open(os.path.join(GOLDEN, "compute_reduction.json")))
    r = flops.per_token_reduction(g["context"], g["query_heads"], g["index_heads"], g["top_k"])
    assert round(r, 1) == g["reduction"]


def test_pair_counts_brute_force():
    for S, k in ((512, 2), (1024, 4), (1280, 16), (384, 1)):
        sel = px = 0
        for t in range(S):
            m = t // 128
            K = min(k, m + 1)
            sel += 128 * (K - 1) + (t % 128) + 1
            px += 128 * m
        assert flops.n_sel(S, k) == sel
        assert flops.n_px(S) == px
        assert flops.n_dense(S) == sum(t + 1 for t in range(S))


def test_selected_pairs_never_exceed_dense():
    for S in (1024, 8192):
        assert flops.n_sel(S, S // 128) == flops.n_dense(S)
        assert flops.n_sel(S, 4) < flops.n_dense(S)
