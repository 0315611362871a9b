"""Pins for the oracle's Philox4x32-10 and the draws built on it."""
import json
import os

import numpy as np
from scipy import stats

from oracle import philox, weights

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox_kat.json")


def _kat():
    with open(GOLD) as f:
        for c in json.load(f)["cases"]:
            yield ([int(x, 16) for x in c["ctr"]], [int(x, 16) for x in c["key"]],
                   [int(x, 16) for x in c["out"]])


def test_numpy_philox_known_answers():
    for ctr, key, out in _kat():
        got = [int(w) for w in philox.philox4x32_10(*ctr, *key)]
        assert got == out


def test_c_philox_known_answers():
    for ctr, key, out in _kat():
        assert [int(w) for w in weights.philox_c(ctr, key)] == out


def test_vectorised_matches_scalar_calls():
    c0 = np.arange(5, dtype=np.uint64)
    vec = philox.philox4x32_10(c0, 7, 9, 11, 0x1234, 0x5678)
    for i in range(5):
        sc = weights.philox_c([i, 7, 9, 11], [0x1234, 0x5678])
        assert [int(w[i]) for w in vec] == [int(x) for x in sc]


def test_canvas_init_is_uniform_over_vocab():
    V, C = 16, 256
    ids = np.concatenate([philox.canvas_init_ids(3, k, C, V) for k in range(64)])
    assert ids.min() >= 0 and ids.max() < V
    counts = np.bincount(ids, minlength=V)
    assert stats.chisquare(counts).pvalue > 1e-3


def test_canvas_init_full_vocab_range():
    ids = philox.canvas_init_ids(0, 0, 256, 262144)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < 262144
    assert len(np.unique(ids)) > 250          # 256 draws from 2^18: collisions are rare


def test_gumbel_uniforms_open_interval_and_layout():
    u = philox.gumbel_uniforms(5, 1, 3, [0, 7], 16)
    assert u.dtype == np.float32 and u.shape == (2, 16)
    assert (u > 0).all() and (u < 1).all()
    # vocab entry v uses word v % 4 of the call with counter v // 4
    w = philox.philox4x32_10(2, 7, (1 << 16) | 3, philox.TAG_GUMBEL, 5, 0)
    expect = (2 * (int(w[1]) >> 9) + 1) * 2.0 ** -24
    assert u[1, 9] == np.float32(expect)
