"""Seeded synthetic inputs shared by the tests and the benchmark.

Holds none of the decoder's arithmetic: only draws of prompt ids, Gaussian
tensors and logits from numpy's PCG64 generator, rounded to bf16 where the
consumer takes bf16 so that both sides of a comparison read identical values.
The pages measure on evaluation suites and PG-19 (DiffusionGemma report §3.3,
§6); none of those are used: uniform random token ids and N(0, 1) tensors of
the same shapes stand in for them.
"""
import numpy as np
import torch


def prompt_ids(n, vocab, seed=0):
    """n uniform random token ids."""
    return np.random.default_rng(seed).integers(0, vocab, n, dtype=np.int64).astype(np.int32)


def normal(shape, seed=0, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def normal_bf16(shape, seed=0, scale=1.0):
    """N(0, scale^2) values rounded to bf16: (fp32 values, torch bf16 CPU tensor)."""
    t = torch.from_numpy(normal(shape, seed, scale)).to(torch.bfloat16)
    return t.float().numpy(), t


def logits(rows, vocab, seed=0, scale=3.0):
    """fp32 logits of a peaked-but-not-degenerate shape (N(0, scale^2))."""
    return normal((rows, vocab), seed, scale)
