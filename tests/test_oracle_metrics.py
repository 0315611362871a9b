"""Eq. 7-10 against hand-worked cases and the blog's throughput arithmetic."""
import json
import os
from fractions import Fraction

from oracle import metrics

G = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_cases():
    with open(os.path.join(G, "metrics_eq7_10.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        m = metrics.efficiency(c["N_k"], c["C_k"])
        assert m["total_tokens"] == c["total_tokens"], c["name"]
        assert m["total_steps"] == c["total_steps"], c["name"]
        assert m["effective_steps_exact"] == Fraction(*c["effective_steps"]), c["name"]
        assert m["tpf_exact"] == Fraction(*c["tpf"]), c["name"]


def test_adaptive_off_effective_steps_is_budget():
    for N in (8, 48, 192):
        for C_k in ([256], [256, 256, 3], [1, 2, 3, 4]):
            assert metrics.efficiency([N] * len(C_k), C_k)["effective_steps_exact"] == N


def test_valid_tokens_up_to_first_eos():
    assert metrics.valid_tokens([5, 6, 7, 2, 9, 2], 2) == 3
    assert metrics.valid_tokens([5, 6, 7], 2) == 3
    assert metrics.valid_tokens([5, 6, 7], -1) == 3
    assert metrics.valid_tokens([2, 6, 7], 2) == 0


def test_blog_throughput_arithmetic():
    with open(os.path.join(G, "blog_throughput.json")) as f:
        b = json.load(f)
    tps = metrics.tokens_per_second(b["tpf"], b["ms_per_forward"] / 1000.0)
    assert round(tps) == b["tokens_per_second_rounded"]
