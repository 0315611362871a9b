"""Pins for the oracle's forward passes: library routines, hand-worked cases, invariants."""
import json
import os

import numpy as np
import pytest
import torch
from scipy import special

from oracle import model, weights

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_layers.json")
with open(GOLD) as _f:
    HAND = json.load(_f)

SMALL = model.TINY.with_(n_layers=1, d_model=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                         n_experts=4, top_k=2, d_ff=32, vocab=256)


@pytest.fixture(scope="module")
def small_weights():
    return weights.Weights(SMALL)


def test_attention_hand_worked():
    a = HAND["attention"]
    K = np.array(a["prefix_k"] + a["new_k"], float)[:, None, :]
    V = np.array(a["prefix_v"] + a["new_v"], float)[:, None, :]
    q = np.array(a["q"], float)[:, None, :]
    for mode, key in (("bidir", "bidir_out"), ("causal", "causal_out")):
        out = model.attention(q, K, V, model.visibility(1, 2, mode))
        assert np.allclose(out[:, 0, :], a[key], atol=1e-12)


@pytest.mark.parametrize("mode,P,T", [("bidir", 37, 19), ("causal", 37, 19), ("causal", 0, 23), ("bidir", 0, 5)])
def test_attention_against_torch_sdpa(mode, P, T):
    rng = np.random.default_rng(7)
    Hq, Hkv, hd = 8, 2, 16
    q = rng.standard_normal((T, Hq, hd))
    k = rng.standard_normal((P + T, Hkv, hd))
    v = rng.standard_normal((P + T, Hkv, hd))
    vis = model.visibility(P, T, mode)
    ours = model.attention(q, k, v, vis)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)[None]
    tv = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(vis))
    assert np.allclose(ours, ref[0].permute(1, 0, 2).numpy(), atol=1e-10)


def test_causal_and_bidirectional_differ_without_prefix():
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((6, 2, 8)) for _ in range(3))
    c = model.attention(q, k, v, model.visibility(0, 6, "causal"))
    b = model.attention(q, k, v, model.visibility(0, 6, "bidir"))
    assert np.allclose(c[0], v[0])                       # first causal query sees only itself
    assert np.allclose(c[-1], b[-1])                     # last causal query sees everything
    assert not np.allclose(c[:-1], b[:-1])


def test_uniform_values_pass_through():
    rng = np.random.default_rng(9)
    q, k = rng.standard_normal((5, 2, 8)), rng.standard_normal((9, 1, 8))
    v = np.broadcast_to(rng.standard_normal(8), (9, 1, 8))
    out = model.attention(q, k, v, model.visibility(4, 5, "bidir"))
    assert np.allclose(out, v[0, 0])


def test_rope_matches_complex_rotation_and_is_relative():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((7, 3, 16))
    pos = np.array([0, 1, 5, 100, 2047, 32768, 36863])
    r = model.rope(x, pos, 10000.0)
    z = x[..., :8] + 1j * x[..., 8:]
    th = 10000.0 ** (-np.arange(8) * 2.0 / 16)
    zr = z * np.exp(1j * pos[:, None, None] * th[None, None, :])
    assert np.allclose(r[..., :8], zr.real) and np.allclose(r[..., 8:], zr.imag)
    assert np.allclose(r[0], x[0])                                   # position 0 is the identity
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1))
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 1, 16))
    d1 = (model.rope(q, [50], 1e4) * model.rope(k, [20], 1e4)).sum()
    d2 = (model.rope(q, [1030], 1e4) * model.rope(k, [1000], 1e4)).sum()
    assert abs(d1 - d2) < 1e-9


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 64)) * 5
    y = model.rmsnorm(x, np.ones(64), 1e-6)
    assert np.allclose(np.sqrt((y * y).mean(axis=1)), 1.0, atol=1e-6)
    assert np.allclose(model.rmsnorm(3 * x, np.ones(64), 1e-12), model.rmsnorm(x, np.ones(64), 1e-12))


def test_swiglu_hand_worked():
    s = HAND["swiglu"]
    y = model.expert_ffn(np.array([s["x"]], float), np.array(s["w_gate"]), np.array(s["w_up"]),
                         np.array(s["w_down"]))
    assert np.allclose(y[0], s["out"], atol=1e-12)
    assert np.allclose(model.silu(np.array([-3.0, 0.0, 2.5])),
                       np.array([-3.0, 0.0, 2.5]) * special.expit([-3.0, 0.0, 2.5]))


def test_sparse_moe_equals_dense_all_experts_with_zeroed_gates(small_weights):
    W = small_weights.layers[0]
    rng = np.random.default_rng(12)
    y = rng.standard_normal((20, SMALL.d_model))
    out, ids, gates, r = model.moe(y, W, SMALL.top_k)
    dense_g = np.zeros((20, SMALL.n_experts))
    np.put_along_axis(dense_g, ids, gates, axis=1)
    dense = sum(dense_g[:, e:e + 1] * model.expert_ffn(y, W["wg"][e], W["wu"][e], W["wd"][e])
                for e in range(SMALL.n_experts))
    assert np.allclose(out, dense, atol=1e-12)
    assert np.allclose(gates.sum(axis=1), 1.0)
    # selected logits are the k largest
    srt = np.sort(r, axis=1)[:, ::-1]
    assert np.allclose(np.sort(np.take_along_axis(r, ids, 1), axis=1)[:, ::-1], srt[:, :SMALL.top_k])


def test_moe_with_k_equal_E_is_softmax_mixture(small_weights):
    W = small_weights.layers[0]
    rng = np.random.default_rng(13)
    y = rng.standard_normal((6, SMALL.d_model))
    out, ids, gates, r = model.moe(y, W, SMALL.n_experts)
    p = special.softmax(r, axis=1)
    mix = sum(p[:, e:e + 1] * model.expert_ffn(y, W["wg"][e], W["wu"][e], W["wd"][e])
              for e in range(SMALL.n_experts))
    assert np.allclose(out, mix, atol=1e-12)


def test_router_ties_go_to_lower_expert_id():
    wr = np.array([[1.0, 0], [2.0, 0], [2.0, 0], [0.5, 0]])
    ids, gates, _ = model.route(np.array([[1.0, 0.0]]), wr, 2)
    assert list(ids[0]) == [1, 2]
    ids, gates, _ = model.route(np.array([[1.0, 0.0]]), wr, 1)
    assert list(ids[0]) == [1]


def _prefix_and_canvas(W, cfg, P=8, C=12, shift=0, seed=14):
    rng = np.random.default_rng(seed)
    prompt = rng.integers(0, cfg.vocab, P)
    x = rng.integers(0, cfg.vocab, C)
    cache = model.prefill(W, cfg, prompt, p0=shift)
    return prompt, x, cache


def test_canvas_joint_permutation_invariance(small_weights):
    cfg = SMALL
    prompt, x, cache = _prefix_and_canvas(small_weights, cfg)
    pos = len(prompt) + np.arange(len(x))
    base = model.canvas_logits(small_weights, cfg, cache, x, pos)
    perm = np.random.default_rng(15).permutation(len(x))
    out = model.canvas_logits(small_weights, cfg, cache, x[perm], pos[perm])
    assert np.allclose(out, base[perm], atol=1e-10)


def test_global_position_shift_invariance(small_weights):
    cfg = SMALL
    prompt, x, cache = _prefix_and_canvas(small_weights, cfg)
    _, _, cache2 = _prefix_and_canvas(small_weights, cfg, shift=1000)
    a = model.canvas_logits(small_weights, cfg, cache, x, len(prompt))
    b = model.canvas_logits(small_weights, cfg, cache2, x, 1000 + len(prompt))
    assert np.allclose(a, b, atol=1e-9)


def test_prefill_is_causal(small_weights):
    cfg = SMALL
    rng = np.random.default_rng(16)
    p = rng.integers(0, cfg.vocab, 10)
    p2 = p.copy()
    p2[7] = (p2[7] + 1) % cfg.vocab
    c1, c2 = model.prefill(small_weights, cfg, p), model.prefill(small_weights, cfg, p2)
    assert np.allclose(c1.k[0][:7], c2.k[0][:7]) and not np.allclose(c1.k[0][7:], c2.k[0][7:])


def test_causal_commit_equals_extended_prefill():
    cfg = SMALL.with_(n_layers=2)
    W = weights.Weights(cfg)
    prompt, x, cache = _prefix_and_canvas(W, cfg)
    model.commit_forward(W, cfg, cache, x, len(prompt), "causal")
    full = model.prefill(W, cfg, np.concatenate([prompt, x]))
    for L in range(cfg.n_layers):
        assert np.allclose(cache.k[L], full.k[L], atol=1e-10)
        assert np.allclose(cache.v[L], full.v[L], atol=1e-10)


def test_zero_output_projections_make_layers_identity():
    cfg = SMALL.with_(n_layers=2)
    W = weights.Weights(cfg)
    for L in W.layers:
        L["wo"] = np.zeros_like(L["wo"])
        L["wd"] = np.zeros_like(L["wd"])
    prompt, x, cache = _prefix_and_canvas(W, cfg)
    lg = model.canvas_logits(W, cfg, cache, x, len(prompt))
    e = W.embed[x].astype(np.float64)
    ref = (e / np.sqrt((e * e).mean(axis=1, keepdims=True) + cfg.rms_eps)) @ W.lm_head.astype(np.float64).T
    assert np.allclose(lg, ref, atol=1e-10)


def test_forced_routing_accepts_valid_ties_and_rejects_others(small_weights):
    W = small_weights.layers[0]
    rng = np.random.default_rng(17)
    y = rng.standard_normal((12, SMALL.d_model))
    out, ids, gates, r = model.moe(y, W, SMALL.top_k)
    same, _, _, _ = model.moe(y, W, SMALL.top_k, forced=ids[:, ::-1])     # order is irrelevant
    assert np.allclose(same, out, atol=1e-12)
    # swap the k-th choice for the (k+1)-th: valid only when their logits are within tol
    order = np.argsort(-r, axis=1, kind="stable")
    alt = ids.copy()
    alt[:, -1] = order[:, SMALL.top_k]
    gap = np.take_along_axis(r, ids[:, -1:], 1)[:, 0] - np.take_along_axis(r, alt[:, -1:], 1)[:, 0]
    with pytest.raises(ValueError):
        model.route(y, W["wr"], SMALL.top_k, forced=alt, tol=float(gap.min()) / 2)
    ok_ids, ok_g, _ = model.route(y, W["wr"], SMALL.top_k, forced=alt, tol=float(gap.max()) + 1e-9)
    assert np.array_equal(ok_ids, alt) and np.allclose(ok_g.sum(axis=1), 1.0)
    with pytest.raises(ValueError):                                   # repeated expert
        model.route(y, W["wr"], SMALL.top_k, forced=np.repeat(ids[:, :1], SMALL.top_k, 1), tol=10.0)


def test_forced_routing_relative_allowance():
    # rel_tol scales the near-tie allowance by the row's largest |logit|:
    # with logits up to 2.0 and rel_tol 2e-2 a swap across a 0.03 gap is a
    # valid top-k, across a 0.05 gap it is not.
    wr = np.eye(4)
    y = np.array([[2.0, 1.0, 0.97, 0.0], [2.0, 1.0, 0.95, 0.0]])
    ids, _, _ = model.route(y[:1], wr, 2, forced=[[0, 2]], rel_tol=2e-2)
    assert ids.tolist() == [[0, 2]]
    with pytest.raises(ValueError):
        model.route(y[1:], wr, 2, forced=[[0, 2]], rel_tol=2e-2)
    with pytest.raises(ValueError):
        model.route(y[:1], wr, 2, forced=[[0, 2]])          # the absolute 1e-2 allowance
    m, mx = model.routing_margin(y, wr, np.array([[0, 2], [0, 2]]))
    assert np.allclose(m, [-0.03, -0.05]) and np.allclose(mx, [2.0, 2.0])
