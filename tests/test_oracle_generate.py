"""Pins for the canvas loop: Eq. 10's extra forwards, adaptive-off budget, EOS cut-off."""
import numpy as np

from oracle import generate, metrics, model, weights

CFG = model.TINY.with_(n_layers=1, d_model=64, n_q_heads=2, n_kv_heads=1, head_dim=32,
                       n_experts=4, top_k=2, d_ff=64, vocab=256)


def test_forward_counts_match_eq10():
    W = weights.Weights(CFG)
    prompt = np.arange(10) % CFG.vocab
    sc = generate.SamplerConfig(canvas_len=16, budget_N=3)
    cnt = {}
    ids, Ns, Cs, m = generate.generate(W, CFG, sc, prompt, 3, counters=cnt)
    assert cnt["denoise"] == sum(Ns)
    assert cnt["commit"] == len(Ns) - 1                        # no commit after the last canvas
    assert m["tpf_exact"] * (cnt["denoise"] + cnt["commit"]) == m["total_tokens"]


def test_adaptive_off_runs_every_canvas_to_the_budget():
    W = weights.Weights(CFG)
    sc = generate.SamplerConfig(canvas_len=16, budget_N=4, adaptive=False, conf_threshold=0.0)
    ids, Ns, Cs, m = generate.generate(W, CFG, sc, np.arange(5), 2)
    assert Ns == [4, 4] and m["effective_steps"] == 4


def test_confident_model_stops_after_one_step():
    sc = generate.SamplerConfig(canvas_len=16, budget_N=8, conf_threshold=0.0)

    def lf(x):
        return np.zeros((16, 256), np.float32)
    lf.vocab = 256
    x, n = generate.run_canvas(lf, sc, 0)
    assert n == 1 and np.all(x == 0)


def test_eos_cuts_the_canvas_and_ends_generation():
    # A stub model whose argmax is the EOS id at position 5 and i+10 elsewhere,
    # confident enough to commit at once.
    sc = generate.SamplerConfig(canvas_len=16, budget_N=8, eos_id=1, conf_threshold=0.5)

    def lf(x):
        l = np.zeros((16, 256), np.float32)
        tgt = np.arange(16) + 10
        tgt[5] = 1
        l[np.arange(16), tgt] = 40.0
        return l
    lf.vocab = 256
    x, n = generate.run_canvas(lf, sc, 0)
    assert n == 1 and metrics.valid_tokens(x, sc.eos_id) == 5
