"""Block-diffusion generation loop over canvases (oracle).

Follows the pages' statement of the procedure:
  * the prompt is encoded once with causal attention (report §1);
  * each canvas of C tokens starts fully corrupted, x_1 ~ Unif(V^C)
    (report §2.1), and is refined by up to N denoising forwards that see the
    read-only prefix and the whole canvas (blog, "Once Written, a Prefix
    Becomes History"), with adaptive stopping (report §3.3);
  * a finished canvas is encoded by one extra forward that appends its K/V to
    the prefix, after which it is read-only; no such forward follows the last
    canvas (the K-1 term of Eq. 10, report §3.4);
  * generation ends after the canvas that holds the first end-of-sequence
    token, or after K_max canvases; C_k counts the tokens before that EOS.

parity pinned by: tests/test_oracle_generate.py (forward-pass counting
against Eq. 10's K-1 term, adaptive-off runs giving N_k = N, EOS cut-off).
"""
from dataclasses import dataclass

import numpy as np

from . import metrics, model, philox, sampler


@dataclass(frozen=True)
class SamplerConfig:
    canvas_len: int = 256
    budget_N: int = 48
    stable_steps: int = 2
    adaptive: bool = True
    eos_id: int = -1
    commit_mode: str = "causal"
    conf_threshold: float = 0.9
    sample_seed: int = 0
    temp_start: float = 1.0     # re-noise temperature at step 1 ...
    temp_end: float = 1.0       # ... and at step N (linear in between)


def run_canvas(logits_fn, scfg, k, on_step=None):
    """Denoise canvas k.  logits_fn(x) -> fp32 logits [C, V].  Returns (x, N_k)."""
    x0 = philox.canvas_init_ids(scfg.sample_seed, k, scfg.canvas_len, logits_fn.vocab)
    st = sampler.CanvasState(x0)
    for n in range(1, scfg.budget_N + 1):
        x_in = st.x.copy()
        l = np.asarray(logits_fn(x_in), np.float32)
        done, a, conf, g = sampler.step(st, l, scfg.sample_seed, k, n, scfg.budget_N,
                                        scfg.stable_steps, scfg.conf_threshold, scfg.adaptive,
                                        scfg.temp_start, scfg.temp_end)
        if on_step is not None:
            on_step(k=k, n=n, x_in=x_in, logits=l, a=a, conf=conf, g=g, state=st.copy(), done=done)
        if done:
            return st.x, n
    raise AssertionError("unreachable: the budget step always finishes the canvas")


def generate(W, cfg, scfg, prompt, K_max, on_step=None, counters=None):
    """Full generation.  Returns (ids [K, C], N_k list, C_k list, Eq. 7-10 dict)."""
    cache = model.prefill(W, cfg, prompt)
    p0 = len(prompt)
    outs, Ns, Cs = [], [], []
    for k in range(K_max):
        def lf(x, p0=p0):
            if counters is not None:
                counters["denoise"] = counters.get("denoise", 0) + 1
            return model.canvas_logits(W, cfg, cache, x, p0).astype(np.float32)
        lf.vocab = cfg.vocab
        x, n_k = run_canvas(lf, scfg, k, on_step)
        outs.append(x)
        Ns.append(n_k)
        c_k = metrics.valid_tokens(x, scfg.eos_id)
        Cs.append(c_k)
        if c_k < scfg.canvas_len or k == K_max - 1:
            break
        if counters is not None:
            counters["commit"] = counters.get("commit", 0) + 1
        model.commit_forward(W, cfg, cache, x, p0, scfg.commit_mode)
        p0 += scfg.canvas_len
    return np.stack(outs), Ns, Cs, metrics.efficiency(Ns, Cs)
