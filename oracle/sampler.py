"""Commit / re-noise / stop sampler of one denoising step (oracle, fp32).

What the pages fix: per position a full-vocabulary softmax gives a predicted
token and its confidence; high-confidence positions lock in first while the
rest keep being revised (blog, "Once Written, a Prefix Becomes History");
re-noising is multinomial (uniform-vocabulary corruption, report §4); the
canvas stops adaptively before the budget N (report §3.3).

Reading of the rule (the report section that gives it is not among the
pages; this is the commit rule of the synthetic workload):
  * a_i = argmax_v l_iv (lowest index on ties); conf_i = max_v softmax(l_i)_v;
  * an uncommitted position commits when conf_i >= tau (fp32 compare,
    tau = 0.9) or when its argmax has been unchanged for `stable_steps`
    consecutive steps (stable counter: +1 when a_i equals the previous
    step's argmax, else reset to 0); a committed position is set to a_i and
    never changes again;
  * every other position is re-noised by a fresh sample from its softmax at
    temperature 1, drawn by Gumbel-max: g_i = argmax_v (l_iv + G_iv) with
    G = -log(-log u), u from the Philox stream of oracle.philox;
  * the canvas is done when every position is committed (adaptive stopping)
    or the step count reaches N; on reaching N the still-uncommitted
    positions take a_i.

Temperature annealing (report §5: the online teacher samples "with mild
temperature annealing"; no schedule is given).  Reading: the re-noise sample
of step n is drawn from softmax(l / tau_n), with tau_n moving linearly from
temp_start at step 1 to temp_end at step N:
    tau_n = temp_start + (temp_end - temp_start) * (n - 1) / (N - 1)   (N > 1)
in double, and inv_tau_n = fp32(1 / tau_n); the Gumbel keys become
k_v = fp32(l_v * inv_tau_n) + G_v (two roundings, no fused multiply-add),
which at tau = 1 are the keys above exactly.  The argmax and the confidence
are those of the model's own distribution (tau = 1).

Canonical reduction order (the pages give none; this one makes the sampler
reproducible bit for bit on any hardware given the same fp32 logits):
  1. vocab tiles of 256 entries, t = 0 .. V/256-1; inside tile t, ascending v:
       m_t = max, a_t = first index reaching it,
       s_t = sum of dg_exp(l_v - m_t) accumulated left to right in fp32,
       (gk_t, gi_t) = max of k_v = l_v + G_v, first index on ties;
  2. the tiles are combined by a balanced binary tree, leaves in tile order,
     left operand = lower vocab range:
       M = max(mL, mR)
       S = fp32(sL * dg_exp(mL - M)) + fp32(sR * dg_exp(mR - M))
       a = aR if mR > mL else aL;  (gk, gi) = right if gkR > gkL else left
     a right operand that covers no tile is skipped (the left passes up);
  3. conf = 1 / S (one correctly rounded division).
Every fp32 operation is a single correctly rounded IEEE operation (numpy
float32 ufuncs; no fused multiply-add).

parity pinned by: tests/test_oracle_sampler.py (closed forms: uniform logits
give conf = 1/V exactly and one-hot logits conf ~ 1; S against an fp64
softmax; argmax against numpy over the whole vocabulary; Gumbel-max
frequencies against softmax by chi-square; scripted commit, stability,
budget and adaptive-off trajectories).
"""
import numpy as np

from . import philox
from .dgmath import dg_exp, gumbel_from_uniform

TILE = 256
f32 = np.float32


def annealed_inv_tau(n, budget_N, temp_start=1.0, temp_end=1.0):
    """fp32(1 / tau_n) of step n (1-based) under the linear schedule above."""
    if budget_N > 1:
        tau = float(temp_start) + (float(temp_end) - float(temp_start)) * (n - 1) / (budget_N - 1)
    else:
        tau = float(temp_start)
    return f32(1.0 / tau)


def tile_partials(l, G, inv_tau=f32(1.0)):
    """Per-(position, tile) partials of fp32 logits l [R, V] and Gumbel noise G [R, V];
    the Gumbel keys are fp32(l * inv_tau) + G."""
    R, V = l.shape
    assert V % TILE == 0
    T = V // TILE
    lt = l.reshape(R, T, TILE).astype(f32)
    m = lt.max(axis=2)
    a = lt.argmax(axis=2).astype(np.int64) + np.arange(T)[None, :] * TILE
    s = np.zeros((R, T), f32)
    for v in range(TILE):                      # ascending, one rounding per add
        s = s + dg_exp(lt[:, :, v] - m)
    lk = (lt * f32(inv_tau)).astype(f32)       # exact when inv_tau == 1
    kap = (lk + G.reshape(R, T, TILE).astype(f32)).astype(f32)
    gk = kap.max(axis=2)
    gi = kap.argmax(axis=2).astype(np.int64) + np.arange(T)[None, :] * TILE
    return dict(m=m, a=a, s=s, gk=gk, gi=gi)


def _merge(Lp, Rp):
    present = Rp["m"] > -np.inf                 # an empty slot has m = -inf
    M = np.maximum(Lp["m"], Rp["m"])
    with np.errstate(invalid="ignore"):
        S = (Lp["s"] * dg_exp(Lp["m"] - M)) + (Rp["s"] * dg_exp(Rp["m"] - M))
    take_a = Rp["m"] > Lp["m"]
    take_g = Rp["gk"] > Lp["gk"]
    out = dict(m=M, s=S.astype(f32),
               a=np.where(take_a, Rp["a"], Lp["a"]),
               gk=np.where(take_g, Rp["gk"], Lp["gk"]),
               gi=np.where(take_g, Rp["gi"], Lp["gi"]))
    return {k: np.where(present, out[k], Lp[k]) for k in out}


def reduce_tiles(p):
    """Balanced binary tree over the tiles (see module docstring, step 2)."""
    p = {k: v.copy() for k, v in p.items()}
    T = p["m"].shape[1]
    width = 1
    while width < T:
        width *= 2
    if width != T:                              # pad with empty slots
        pad = width - T
        p["m"] = np.concatenate([p["m"], np.full((p["m"].shape[0], pad), -np.inf, f32)], 1)
        p["gk"] = np.concatenate([p["gk"], np.full((p["m"].shape[0], pad), -np.inf, f32)], 1)
        p["s"] = np.concatenate([p["s"], np.zeros((p["m"].shape[0], pad), f32)], 1)
        for k in ("a", "gi"):
            p[k] = np.concatenate([p[k], np.zeros((p[k].shape[0], pad), np.int64)], 1)
    while p["m"].shape[1] > 1:
        Lp = {k: v[:, 0::2] for k, v in p.items()}
        Rp = {k: v[:, 1::2] for k, v in p.items()}
        p = _merge(Lp, Rp)
    return {k: v[:, 0] for k, v in p.items()}


def position_outputs(l, seed, k, n, positions=None, inv_tau=f32(1.0)):
    """(argmax a, confidence conf, Gumbel sample g) for fp32 logits l [R, V].

    `positions` gives the canvas index of each row of l (default 0..R-1); the
    Gumbel stream of step n (1-based) of canvas k (0-based) is keyed by it.
    g is a sample of softmax(l * inv_tau).
    """
    l = np.asarray(l, dtype=f32)
    R, V = l.shape
    positions = np.arange(R) if positions is None else np.asarray(positions)
    G = gumbel_from_uniform(philox.gumbel_uniforms(seed, k, n, positions, V))
    r = reduce_tiles(tile_partials(l, G, inv_tau))
    conf = (f32(1.0) / r["s"]).astype(f32)
    return r["a"].astype(np.int32), conf, r["gi"].astype(np.int32), r


class CanvasState:
    """x (ids), committed flags, previous argmax and stability counters."""

    def __init__(self, x):
        C = len(x)
        self.x = np.asarray(x, np.int32).copy()
        self.committed = np.zeros(C, np.uint8)
        self.last = np.full(C, -1, np.int32)
        self.stable = np.zeros(C, np.int32)

    def copy(self):
        s = CanvasState(self.x)
        s.committed, s.last, s.stable = self.committed.copy(), self.last.copy(), self.stable.copy()
        return s


def apply_rule(state, a, conf, g, n, budget_N, stable_steps=2, conf_threshold=0.9,
               adaptive=True):
    """Commit / re-noise / stop update for step n (1-based).  Returns done."""
    free = state.committed == 0
    same = a == state.last
    state.stable = np.where(free, np.where(same, state.stable + 1, 0), state.stable).astype(np.int32)
    state.last = np.where(free, a, state.last).astype(np.int32)
    commit = free & ((conf >= f32(conf_threshold)) | (state.stable >= stable_steps))
    state.x = np.where(commit, a, np.where(free, g, state.x)).astype(np.int32)
    state.committed = (state.committed | commit).astype(np.uint8)
    all_done = bool(state.committed.all())
    if n >= budget_N:
        left = state.committed == 0
        state.x = np.where(left, a, state.x).astype(np.int32)
        state.committed[:] = 1
        return True
    return all_done and adaptive


def step(state, l, seed, k, n, budget_N, stable_steps=2, conf_threshold=0.9, adaptive=True,
         temp_start=1.0, temp_end=1.0):
    """Full sampler step on fp32 logits [C, V]: returns (done, a, conf, g)."""
    a, conf, g, _ = position_outputs(l, seed, k, n, inv_tau=annealed_inv_tau(n, budget_N, temp_start, temp_end))
    done = apply_rule(state, a, conf, g, n, budget_N, stable_steps, conf_threshold, adaptive)
    return done, a, conf, g
