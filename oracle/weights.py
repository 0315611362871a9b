"""Seeded synthetic weights of the random-init decoder (oracle side).

The pages release trained weights (report §1, "Open-weights release") that
are not available here; every workload runs on random-init weights, drawn
"N(0, 0.02)".  Both sides must hold bit-identical bf16 weights, so the draw is
a counter-based Irwin-Hall(4) sum (see weightgen.c), rounded to bf16; the
oracle keeps those bf16 values and computes with them in fp64.

Logical tensors and their generator ids (element index = row-major index in
the listed shape):
    1            token embedding    [V, d]
    2            LM head (untied)   [V, d]
    100+16L+0    W_q                [Hq*hd, d]
    100+16L+1    W_k                [Hkv*hd, d]
    100+16L+2    W_v                [Hkv*hd, d]
    100+16L+3    W_o                [d, Hq*hd]
    100+16L+4    router W_r         [E, d]
    100+16L+5    expert W_gate      [E, F, d]
    100+16L+6    expert W_up        [E, F, d]
    100+16L+7    expert W_down      [E, d, F]
RMSNorm gains are ones (not drawn).

parity pinned by: tests/test_oracle_weights.py (Philox KAT through this C
code, closed-form Irwin-Hall mean/variance/range, bf16 rounding against
torch's round-to-nearest-even conversion).
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "weightgen.c")
_LIB = os.path.join(_HERE, "liboracle_wg.so")
_lock = threading.Lock()
_lib = None

EMBED = 1
LM_HEAD = 2
WQ, WK, WV, WO, WR, WG, WU, WD = range(8)


def layer_tid(layer, which):
    return 100 + 16 * layer + which


def build():
    """Compile the oracle's C generator (plain gcc, OpenMP, no contraction)."""
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", _LIB, _SRC, "-lm"])


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_weights.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p]
            lib.oracle_weights.restype = None
            lib.oracle_philox4x32_10.argtypes = [ctypes.c_void_p] * 3
            lib.oracle_philox4x32_10.restype = None
            _lib = lib
    return _lib


def philox_c(ctr, key):
    """The C generator's raw Philox4x32-10 (for known-answer checks)."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def elements(seed, tid, start, count, std):
    """Weight elements [start, start+count) of tensor `tid` as fp32 (bf16-exact)."""
    out = np.empty(int(count), dtype=np.float32)
    if count:
        _load().oracle_weights(int(seed), int(tid), int(start), int(count),
                               float(np.float32(std)), out.ctypes.data)
    return out


def tensor(seed, tid, shape, std):
    n = int(np.prod(shape))
    return elements(seed, tid, 0, n, std).reshape(shape)


def rows(seed, tid, shape, row_ids, std):
    """Selected leading-axis rows of a 2-D or 3-D logical tensor."""
    inner = int(np.prod(shape[1:]))
    return np.stack([elements(seed, tid, int(r) * inner, inner, std).reshape(shape[1:])
                     for r in row_ids])


class Weights:
    """All tensors of the decoder, fp32 arrays holding bf16-rounded values."""

    def __init__(self, cfg):
        self.cfg = cfg
        s, std = cfg.weight_seed, cfg.init_std
        d, V = cfg.d_model, cfg.vocab
        qd, kd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
        E, F = cfg.n_experts, cfg.d_ff
        self.embed = tensor(s, EMBED, (V, d), std)
        self.lm_head = tensor(s, LM_HEAD, (V, d), std)
        self.layers = []
        for L in range(cfg.n_layers):
            t = lambda w: layer_tid(L, w)
            self.layers.append(dict(
                wq=tensor(s, t(WQ), (qd, d), std),
                wk=tensor(s, t(WK), (kd, d), std),
                wv=tensor(s, t(WV), (kd, d), std),
                wo=tensor(s, t(WO), (d, qd), std),
                wr=tensor(s, t(WR), (E, d), std),
                wg=tensor(s, t(WG), (E, F, d), std),
                wu=tensor(s, t(WU), (E, F, d), std),
                wd=tensor(s, t(WD), (E, d, F), std),
                attn_norm=np.ones(d, np.float32),
                moe_norm=np.ones(d, np.float32),
            ))
        self.final_norm = np.ones(d, np.float32)


class ExpertTensor:
    """Expert tensor [E, a, b] whose experts are generated when indexed (never
    stored: a full-width layer holds ~3 GB of expert weights in fp32)."""

    def __init__(self, seed, tid, shape, std):
        self.seed, self.tid, self.shape, self.std = seed, tid, tuple(shape), std

    def __getitem__(self, e):
        inner = self.shape[1] * self.shape[2]
        return elements(self.seed, self.tid, int(e) * inner, inner, self.std).reshape(self.shape[1:])

    def __len__(self):
        return self.shape[0]


class RowTensor:
    """[V, d] table (embedding, LM head) generated row range by row range."""

    def __init__(self, seed, tid, shape, std):
        self.seed, self.tid, self.shape, self.std = seed, tid, tuple(shape), std

    def take(self, row_ids):
        return rows(self.seed, self.tid, self.shape, row_ids, self.std)

    def block(self, r0, n):
        d = self.shape[1]
        return elements(self.seed, self.tid, int(r0) * d, int(n) * d, self.std).reshape(n, d)


class LazyWeights:
    """The decoder's tensors for full-width shapes: the same generator and
    values as Weights, but expert tensors are generated per expert when used
    and the embedding / LM head per row range, so that a 30-layer model of
    the full configuration fits in host memory.  Per-layer projection and
    router matrices are generated once, on the layer's first use."""

    def __init__(self, cfg):
        self.cfg = cfg
        s, std = cfg.weight_seed, cfg.init_std
        self.embed = RowTensor(s, EMBED, (cfg.vocab, cfg.d_model), std)
        self.lm_head = RowTensor(s, LM_HEAD, (cfg.vocab, cfg.d_model), std)
        self.final_norm = np.ones(cfg.d_model, np.float32)
        self.layers = _LazyLayers(cfg)


class _LazyLayers:
    def __init__(self, cfg):
        self.cfg, self._done = cfg, {}

    def __len__(self):
        return self.cfg.n_layers

    def __iter__(self):
        return (self[L] for L in range(len(self)))

    def __getitem__(self, L):
        if L not in self._done:
            cfg = self.cfg
            s, std = cfg.weight_seed, cfg.init_std
            d, E, F = cfg.d_model, cfg.n_experts, cfg.d_ff
            qd, kd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
            t = lambda w: layer_tid(L, w)
            self._done[L] = dict(
                wq=tensor(s, t(WQ), (qd, d), std), wk=tensor(s, t(WK), (kd, d), std),
                wv=tensor(s, t(WV), (kd, d), std), wo=tensor(s, t(WO), (d, qd), std),
                wr=tensor(s, t(WR), (E, d), std),
                wg=ExpertTensor(s, t(WG), (E, F, d), std), wu=ExpertTensor(s, t(WU), (E, F, d), std),
                wd=ExpertTensor(s, t(WD), (E, d, F), std),
                attn_norm=np.ones(d, np.float32), moe_norm=np.ones(d, np.float32))
        return self._done[L]
