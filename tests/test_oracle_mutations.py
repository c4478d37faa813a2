"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutant is compiled from ``oracle/msa_oracle.c`` with one textual change, loaded in place of
the real oracle, and run through a few pins; at least one must fail.  This is what makes the pins
worth trusting: a dropped term, a wrong sign or index, or a flipped tie rule cannot pass them.
"""
import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "dS sign": ("dS[a] = Ph[a] * (dP - Drow);", "dS[a] = Ph[a] * (dP + Drow);"),
    "local block not forced": ("c[m] = INFINITY;", "c[m] = -INFINITY;"),
    "tie rule flipped": ("return n1 < n2;", "return n1 > n2;"),
    "KL gradient sign": ("const double dz = cz * (p_px - pbar[a]);",
                         "const double dz = cz * (pbar[a] - p_px);"),
    "causal cut dropped": ("j < (n + 1) * MSA_ORACLE_BLOCK && j <= t;",
                           "j < (n + 1) * MSA_ORACLE_BLOCK;"),
    "dKp from the wrong operand": ("acc[d] += scale * dz * qprow[d];",
                                   "acc[d] += scale * dz * kprow[d];"),
    "teacher not averaged": ("pbar[a] += Ph[a] / Gp;", "pbar[a] += Ph[a];"),
    "teacher averaged over the KV group": ("pbar[a] += Ph[a] / Gp;", "pbar[a] += Ph[a] / G;"),
    "keys of the proxy head's first KV head": ("const int kvh = h / G; /* the KV head of query head h */",
                                               "const int kvh = (h / Gp) * Hkv / Hp;"),
    "scale dropped in dQ": ("dqrow[d] += scale * dS[a] * krow[d];",
                            "dqrow[d] += dS[a] * krow[d];"),
    "block max over a shifted block": ("for (int j = n * MSA_ORACLE_BLOCK; j < (n + 1) * MSA_ORACLE_BLOCK; ++j) {\n      double z",
                                       "for (int j = n * MSA_ORACLE_BLOCK + 1; j < (n + 1) * MSA_ORACLE_BLOCK; ++j) {\n      double z"),
    "dV from dS instead of P": ("dvrow[d] += Ph[a] * dorow[d];", "dvrow[d] += dS[a] * dorow[d];"),
    "scale dropped in dK": ("dkrow[d] += scale * dS[a] * qrow[d];", "dkrow[d] += dS[a] * qrow[d];"),
    "row term D dropped": ("const double Drow = dot(dorow, o, D);",
                           "const double Drow = 0.0 * dot(dorow, o, D);"),
    "student not normalised": ("const double lse_px = zmx + log(zsum);", "const double lse_px = zmx;"),
    "query head mapped to the wrong group": ("const int g = h / G;", "const int g = h % Hkv;"),
    "scale dropped in dQp": ("dqprow[d] += scale * dz * kprow[d];", "dqprow[d] += dz * kprow[d];"),
    "KL mean not over proxy heads": ("if (kl_out) *kl_out = kl / ((double)B * S * Hp);",
                                     "if (kl_out) *kl_out = kl / ((double)B * S);"),
    "padding with block 0": ("for (; w < top_k; ++w) out[w] = -1;", "for (; w < top_k; ++w) out[w] = 0;"),
    "one block too few": ("const int K = top_k < m + 1 ? top_k : m + 1;",
                          "const int K = top_k - 1 < m + 1 ? top_k - 1 : m + 1;"),
    "near-tie gap always zero": ("*gap = den > 0.0 ? (lo_sel - hi_uns) / den : 0.0;",
                                 "*gap = 0.0;"),
    "near-tie gap from the highest selected score": (
        "if (c[n] < lo_sel) lo_sel = c[n];",
        "if (lo_sel == INFINITY || c[n] > lo_sel) lo_sel = c[n];"),
    "near-tie gap not relative": ("*gap = den > 0.0 ? (lo_sel - hi_uns) / den : 0.0;",
                                  "*gap = lo_sel - hi_uns;"),
}

PINS = [
    lambda: pins.test_selection_brute_force_properties(3, B=1, S=512),
    lambda: pins.test_selection_ties_prefer_lower_block(),
    lambda: [pins.test_selection_gap_closed_form(c) for c in sorted(pins.GAP_CASES)],
    lambda: pins.test_full_selection_is_dense_causal_attention(False),
    lambda: pins.test_finite_differences_every_gradient(False, n_coords=2),
    lambda: pins.test_kl_zero_when_student_equals_teacher(2),
    lambda: pins.test_eager_second_implementation((1, 384, 8, 4, 2, 2), False),
    lambda: pins.test_finite_differences_general_mapping(4, 1, 2, n_coords=2),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    caught = []
    with oracle.use_library(lib):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin)
    assert caught, f"no pin caught the planted mistake: {name}"
