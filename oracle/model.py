"""fp64 forward passes of the synthetic MoE block-diffusion decoder (oracle).

What the pages fix:
  * context (prompt) encoding uses causal attention; canvas denoising uses
    bidirectional attention within the 256-token canvas while conditioning on
    the clean prefix through its KV cache (report §1; blog "Once Written, a
    Prefix Becomes History"; report §4, which also says the canvas never sees
    other denoising blocks);
  * the FFN is a top-k mixture of experts (report abstract, §6 "GPU time
    breakdown", "MoE").

Readings where the pages are silent (architecture §3 is not among them):
  * pre-norm residual blocks: h += Attn(RMSNorm(h)); h += MoE(RMSNorm(h));
    final RMSNorm before an untied LM head;
  * RMSNorm y = x / sqrt(mean(x^2) + eps) * g, eps = 1e-6, g = 1;
  * RoPE, rotate-half pairing (j, j + hd/2), theta_j = base^(-2j/hd), applied
    to q and k (k is cached after rotation);
  * softmax scale 1/sqrt(hd); grouped-query attention, query head h reads
    KV head h // (Hq/Hkv);
  * router: logits r = RMSNorm(h) W_r^T, the k largest (ties -> lower expert
    id), gates = softmax over those k logits;
  * expert e: W_down,e (silu(W_gate,e y) * W_up,e y)  (SwiGLU);
  * the commit forward that re-encodes a finished canvas uses causal attention
    inside the canvas (context encoding is causal, report §1); a flag selects
    bidirectional instead.

parity pinned by: tests/test_oracle_model.py (torch scaled_dot_product_attention
with the same mask, hand-computed attention and SwiGLU cases, RoPE's complex
form and relative-position property, sparse MoE == dense all-experts MoE with
zeroed gates, joint canvas permutation and global position-shift invariants,
zero-weight layers reduce to the identity, forced routing accepted only
within tolerance of the top-k boundary).
"""
from dataclasses import dataclass, replace

import numpy as np

from . import fp8


@dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    d_ff: int
    vocab: int
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    init_std: float = 0.02
    weight_seed: int = 0
    expert_fp8: bool = False   # gate/up weights and their input rows in e4m3 (oracle/fp8.py)

    def with_(self, **kw):
        return replace(self, **kw)


# 2 layers, d=256, 4/2 heads of 64, 8 experts top-2, FFN 512, vocab 1024.
TINY = ModelConfig(2, 256, 4, 2, 64, 8, 2, 512, 1024)
# 30 layers, d=2816, 16/8 heads of 128, 128 experts top-8, FFN 704, vocab 262144.
FULL = ModelConfig(30, 2816, 16, 8, 128, 128, 8, 704, 262144)


def rmsnorm(x, g, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x, pos, base):
    """x [T, H, hd] at integer positions pos [T] -> rotated copy (rotate-half)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    theta = float(base) ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]       # [T, half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def attention(q, k, v, visible):
    """softmax(q k^T / sqrt(hd)) v over visible keys.

    q [T, Hq, hd]; k, v [S, Hkv, hd]; visible [T, S] bool -> [T, Hq, hd].
    """
    T, Hq, hd = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((T, Hq, hd))
    for h in range(Hq):
        kh, vh = k[:, h // G, :], v[:, h // G, :]
        sc = (q[:, h, :] @ kh.T) / np.sqrt(hd)
        sc = np.where(visible, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


def visibility(n_prefix, n_new, mode):
    """Mask for n_new query tokens that follow n_prefix cached tokens.

    The prefix is always fully visible; inside the new block 'bidir' sees all
    of it and 'causal' sees positions <= the query's own.
    """
    vis = np.ones((n_new, n_prefix + n_new), dtype=bool)
    if mode == "causal":
        vis[:, n_prefix:] = np.tril(np.ones((n_new, n_new), dtype=bool))
    elif mode != "bidir":
        raise ValueError(mode)
    return vis


def silu(x):
    return x / (1.0 + np.exp(-x))


ROUTING_TOL = 1e-2


def route(y, wr, k, forced=None, tol=ROUTING_TOL, rel_tol=None):
    """Top-k experts (ties -> lower id) and softmax gates over their logits.

    `forced` [T, k] replays another implementation's expert choice: top-k is
    an integer decided by floating point, so where router logits are tied
    within rounding either side of the tie is a correct result.  A forced set
    is accepted only if it holds k distinct experts whose logits all reach
    the k-th largest logit minus the allowance; otherwise ValueError.  The
    allowance is `tol`, or with `rel_tol` that fraction of the row's largest
    |logit| (the normwise relative error of bf16 logits against fp32).
    """
    r = y @ np.asarray(wr, np.float64).T                       # [T, E]
    order = np.argsort(-r, axis=1, kind="stable")
    ids = order[:, :k]
    if forced is not None:
        forced = np.asarray(forced).astype(np.int64)
        kth = np.take_along_axis(r, ids[:, -1:], axis=1)[:, 0]
        allow = tol if rel_tol is None else rel_tol * np.abs(r).max(axis=1)
        ok = np.take_along_axis(r, forced, axis=1).min(axis=1) >= kth - allow
        ok &= np.array([len(set(row)) == k for row in forced])
        if not ok.all():
            raise ValueError(f"forced routing is not a top-{k} choice within the allowance "
                             f"(tokens {np.nonzero(~ok)[0][:8].tolist()})")
        ids = forced
    sel = np.take_along_axis(r, ids, axis=1)
    g = np.exp(sel - sel.max(axis=1, keepdims=True))
    return ids.astype(np.int32), g / g.sum(axis=1, keepdims=True), r


def routing_margin(y, wr, forced):
    """Per token: the lowest logit of the forced experts minus the k-th largest
    logit (>= 0 when the forced set is the exact top-k), and the row's largest
    |logit|; for reporting how close a replayed expert choice is to the top-k."""
    r = y @ np.asarray(wr, np.float64).T
    k = forced.shape[1]
    kth = -np.sort(-r, axis=1)[:, k - 1]
    return np.take_along_axis(r, np.asarray(forced, np.int64), axis=1).min(axis=1) - kth, np.abs(r).max(axis=1)


def expert_ffn(x, wg, wu, wd, fp8_gate_up=False, x_bf16=None):
    """SwiGLU expert on rows x [n, d].

    fp8_gate_up: the gate/up products take e4m3 operands (oracle/fp8.py):
    each weight row (output feature) and each input row, rounded to bf16 as
    the decoder hands it over, scaled by its own power of two.  x_bf16
    (optional, [n, d] bf16 values): the input rows to quantize instead of
    bf16(x) -- a replay passes the decoder's own rows so that both sides take
    the integer quantization decisions on the same values."""
    wg, wu, wd = (np.asarray(w, np.float64) for w in (wg, wu, wd))
    if fp8_gate_up:
        xb = bf16_round(x) if x_bf16 is None else np.asarray(x_bf16, np.float64)
        x = fp8.dequantize_rows(*fp8.quantize_rows(xb))
        wg = fp8.dequantize_rows(*fp8.quantize_rows(wg))
        wu = fp8.dequantize_rows(*fp8.quantize_rows(wu))
    return (silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def bf16_round(x):
    """Round to the nearest bf16 value, ties to even (float64 in and out)."""
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def moe_given_routing(y, ids, gates, W, fp8_gate_up=False, y_bf16=None):
    out = np.zeros_like(y)
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        xb = None if y_bf16 is None else y_bf16[tok]
        out[tok] += gates[tok, slot][:, None] * expert_ffn(y[tok], W["wg"][e], W["wu"][e], W["wd"][e],
                                                           fp8_gate_up, xb)
    return out


def moe(y, W, k, forced=None, rel_tol=None, fp8_gate_up=False, y_bf16=None):
    ids, gates, r = route(y, W["wr"], k, forced, rel_tol=rel_tol)
    return moe_given_routing(y, ids, gates, W, fp8_gate_up, y_bf16), ids, gates, r


def block(h, pos, W, cfg, prefix_k, prefix_v, mode, trace=None, forced_routing=None, routing_rel_tol=None,
          moe_input_bf16=None):
    """One decoder layer over new tokens h [T, d] at positions pos.

    prefix_k/v [S, Hkv, hd] are the cached (rotated) keys/values visible to
    every new token; forced_routing (optional [T, k]) and routing_rel_tol as
    in route(); moe_input_bf16 (optional) as expert_ffn's x_bf16.
    Returns (h_out, k_new, v_new).
    """
    T = h.shape[0]
    hd, Hq, Hkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    n = rmsnorm(h, W["attn_norm"], cfg.rms_eps)
    q = (n @ np.asarray(W["wq"], np.float64).T).reshape(T, Hq, hd)
    k = (n @ np.asarray(W["wk"], np.float64).T).reshape(T, Hkv, hd)
    v = (n @ np.asarray(W["wv"], np.float64).T).reshape(T, Hkv, hd)
    q = rope(q, pos, cfg.rope_base)
    k = rope(k, pos, cfg.rope_base)
    K = np.concatenate([prefix_k, k], axis=0)
    V = np.concatenate([prefix_v, v], axis=0)
    o = attention(q, K, V, visibility(prefix_k.shape[0], T, mode))
    h = h + o.reshape(T, Hq * hd) @ np.asarray(W["wo"], np.float64).T
    n2 = rmsnorm(h, W["moe_norm"], cfg.rms_eps)
    y, ids, gates, r = moe(n2, W, cfg.top_k, forced_routing, routing_rel_tol, cfg.expert_fp8, moe_input_bf16)
    if trace is not None:
        trace.append(dict(n=n, q=q, k=k, v=v, o=o, n2=n2, ids=ids, gates=gates, router=r, y=y))
    return h + y, k, v


class KVCache:
    """Per-layer rotated keys and values of the clean prefix, [S, Hkv, hd]."""

    def __init__(self, cfg):
        self.k = [np.zeros((0, cfg.n_kv_heads, cfg.head_dim)) for _ in range(cfg.n_layers)]
        self.v = [np.zeros((0, cfg.n_kv_heads, cfg.head_dim)) for _ in range(cfg.n_layers)]

    @property
    def length(self):
        return self.k[0].shape[0]

    def append(self, layer, k, v):
        self.k[layer] = np.concatenate([self.k[layer], k], axis=0)
        self.v[layer] = np.concatenate([self.v[layer], v], axis=0)


def embed_rows(W, ids):
    """Embedding rows of token ids (fp64); W.embed is an array or a table that
    generates rows on demand (oracle.weights.RowTensor)."""
    if isinstance(W.embed, np.ndarray):
        return np.asarray(W.embed, np.float64)[ids]
    return W.embed.take(ids).astype(np.float64)


def forward(W, cfg, ids, pos, cache, mode, append=False, trace=None, routing=None):
    """Run all layers over tokens `ids` at positions `pos` with `cache` as prefix.

    `pos` is an int (first position; the tokens then sit at pos, pos+1, ...)
    or an explicit array of positions.  `routing` (optional) is a per-layer
    list of forced expert choices (see route()).  Returns the final hidden
    states [T, d] (fp64).  With append=True the new tokens' K/V are added to
    the cache after the pass (prefill and commit).
    """
    ids = np.asarray(ids)
    pos = pos + np.arange(len(ids)) if np.ndim(pos) == 0 else np.asarray(pos)
    h = embed_rows(W, ids)
    new_kv = []
    for L, WL in enumerate(W.layers):
        forced = None if routing is None else routing[L]
        h, k, v = block(h, pos, WL, cfg, cache.k[L], cache.v[L], mode, trace, forced)
        new_kv.append((k, v))
    if append:
        for L, (k, v) in enumerate(new_kv):
            cache.append(L, k, v)
    return h


def logits(W, cfg, h):
    """LM head on the final-normed hidden states -> fp64 logits [T, V]."""
    n = rmsnorm(h, W.final_norm, cfg.rms_eps)
    return n @ np.asarray(W.lm_head, np.float64).T


def prefill(W, cfg, prompt, p0=0, routing=None):
    """Encode the prompt with causal attention and cache its K/V (report §1)."""
    cache = KVCache(cfg)
    if len(prompt):
        forward(W, cfg, prompt, p0, cache, "causal", append=True, routing=routing)
    return cache


def canvas_logits(W, cfg, cache, x, p0, trace=None, routing=None):
    """One denoising forward: canvas x at positions p0.. (or an explicit
    position array) sees the whole prefix and the whole canvas; nothing is
    cached.  Returns fp64 logits [C, V]."""
    return logits(W, cfg, forward(W, cfg, x, p0, cache, "bidir", trace=trace, routing=routing))


def commit_forward(W, cfg, cache, x, p0, mode="causal", routing=None):
    """The single extra forward between canvases: encodes the finished canvas
    and appends its K/V to the prefix cache (report §3.4, the K-1 term)."""
    forward(W, cfg, x, p0, cache, mode, append=True, routing=routing)
