"""Pins for the synthetic weight draw: closed-form Irwin-Hall(4) statistics and bf16 rounding."""
import math

import numpy as np
import torch

from oracle import philox, weights


def test_element_formula_against_python_philox():
    # element e of tensor t: Irwin-Hall(4) over the words of Philox(ctr=(e, 0, t, 1)).
    e = np.arange(1000, dtype=np.uint64)
    w = philox.philox4x32_10(e, 0, 77, 1, 9, 0)
    s = sum((x >> np.uint32(9)).astype(np.int64) for x in w)
    scale = np.float32(float(np.float32(0.02)) * math.sqrt(3.0) / 8388608.0)
    v = (s - (1 << 24)).astype(np.float32) * scale
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()     # RNE conversion
    assert np.array_equal(weights.elements(9, 77, 0, 1000, 0.02), ref)


def test_moments_match_irwin_hall():
    x = weights.elements(0, 5, 0, 4_000_000, 0.02).astype(np.float64)
    # mean 0, variance std^2 (4 uniforms of variance 1/12, times 3*std^2)
    assert abs(x.mean()) < 3 * 0.02 / math.sqrt(len(x)) * 2
    assert abs(x.std() / 0.02 - 1.0) < 2e-3
    # support: |sum - 2| <= 2, so |w| <= 2*sqrt(3)*std (plus bf16 rounding)
    assert np.abs(x).max() <= 2 * math.sqrt(3) * 0.02 * (1 + 2 ** -8)
    # Irwin-Hall(4) excess kurtosis is -6/(5*4) = -0.3
    k = ((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3.0
    assert abs(k - (-0.3)) < 0.02


def test_offsets_and_tensor_ids_are_independent_streams():
    a = weights.elements(0, 5, 100, 50, 0.02)
    b = weights.elements(0, 5, 0, 150, 0.02)[100:]
    assert np.array_equal(a, b)
    assert not np.array_equal(weights.elements(0, 6, 0, 50, 0.02), weights.elements(0, 5, 0, 50, 0.02))
    assert not np.array_equal(weights.elements(1, 5, 0, 50, 0.02), weights.elements(0, 5, 0, 50, 0.02))


def test_values_are_bf16():
    x = weights.elements(0, 1, 0, 10000, 0.02)
    assert np.all((x.view(np.uint32) & 0xFFFF) == 0)


def test_lazy_weights_equal_the_eager_tensors():
    # The full-width tests generate weights lazily (per expert, per row range);
    # on the tiny model both forms must give the same values and the same prefill.
    from oracle import model as om
    cfg = om.TINY
    W, L = weights.Weights(cfg), weights.LazyWeights(cfg)
    ids = np.arange(0, cfg.vocab, 37)
    assert np.array_equal(om.embed_rows(W, ids), om.embed_rows(L, ids))
    for k in ("wq", "wk", "wv", "wo", "wr"):
        assert np.array_equal(W.layers[1][k], L.layers[1][k])
    for k in ("wg", "wu", "wd"):
        for e in (0, 5, cfg.n_experts - 1):
            assert np.array_equal(W.layers[1][k][e], L.layers[1][k][e])
    assert np.array_equal(W.lm_head[100:164], L.lm_head.block(100, 64))
    prompt = np.arange(64) * 13 % cfg.vocab
    a, b = om.prefill(W, cfg, prompt), om.prefill(L, cfg, prompt)
    assert all(np.array_equal(x, y) for x, y in zip(a.k + a.v, b.k + b.v))
