"""Inference-efficiency metrics, report §3.4, Eq. 7-10.

For K canvases with N_k denoising steps and C_k valid tokens each (C_k = C,
or the count before the first end-of-sequence token):
    Total Tokens                = sum_k C_k                                (Eq. 7)
    Total Denoising Steps       = sum_k N_k                                (Eq. 8)
    Effective Denoising Steps   = (sum_k N_k C_k) / Total Tokens           (Eq. 9)
    Tokens Per Forward (TPF)    = Total Tokens / (Total Steps + K - 1)     (Eq. 10)
The K - 1 term counts the one extra forward between consecutive canvases
that encodes the finished canvas and appends its K/V.

parity pinned by: tests/golden/metrics_eq7_10.json (hand-worked cases) and
the report's own statement that without adaptive stopping Eq. 9 equals N.
"""
from fractions import Fraction


def efficiency(N_k, C_k):
    N_k, C_k = [int(n) for n in N_k], [int(c) for c in C_k]
    assert len(N_k) == len(C_k) and len(N_k) > 0
    K = len(N_k)
    total_tokens = sum(C_k)
    total_steps = sum(N_k)
    eff = Fraction(sum(n * c for n, c in zip(N_k, C_k)), total_tokens) if total_tokens else Fraction(0)
    tpf = Fraction(total_tokens, total_steps + K - 1)
    return dict(K=K, total_tokens=total_tokens, total_steps=total_steps,
                effective_steps=float(eff), tpf=float(tpf),
                effective_steps_exact=eff, tpf_exact=tpf)


def valid_tokens(ids, eos_id):
    """C_k: the whole canvas, or the tokens before the first EOS."""
    if eos_id is None or eos_id < 0:
        return len(ids)
    hits = [i for i, t in enumerate(ids) if int(t) == int(eos_id)]
    return hits[0] if hits else len(ids)


def tokens_per_second(tpf, seconds_per_forward):
    """Output tokens/s = TPF / time per forward (how the blog's 1,456 tok/s
    follows from 19.74 TPF at 13.56 ms per forward)."""
    return tpf / seconds_per_forward
