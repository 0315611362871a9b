"""Kernel-level parity of the CUDA path (through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import synth
from gpu_util import bf16_to_f32, dev, new_partials, partial_planes, rel_err, tiles_dev, top2_gap
from oracle import dgmath, model as om, philox, sampler as osamp, weights as ow

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from discrete_diffusion_block_gb300 import build
    build.build()
    dgp.load()
    torch.cuda.set_device(0)


# ---- seeded weights ---------------------------------------------------------

@pytest.mark.parametrize("tid,e0,n", [(1, 0, 100_003), (2, 12345, 4096), (137, (1 << 32) - 7, 64)])
def test_weight_generator_bit_exact(tid, e0, n):
    t = torch.empty(n, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_weights(t, 7, tid, e0, 0.02)
    got = t.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = (ow.elements(7, tid, e0, n, 0.02).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(got, ref)


def untile(phys, lead, blocks, kt):
    """Operand tiles [*lead][blocks][kt][128][64] (16-byte chunk c of row r
    stored at chunk position c ^ (r % 8)) back to the row-major matrix
    [*lead][blocks * 128][kt * 64]."""
    t = phys.reshape(*lead, blocks, kt, 128, 8, 8)
    r = np.arange(128)[:, None]
    pos = np.arange(8)[None, :] ^ (r % 8)          # position of logical chunk c in row r
    t = np.take_along_axis(t, np.broadcast_to(pos[..., None], (128, 8, 8)).reshape((1,) * (t.ndim - 3) + (128, 8, 8)), axis=-2)
    t = t.reshape(*lead, blocks, kt, 128, 64)
    return np.moveaxis(t, -3, -2).reshape(*lead, blocks * 128, kt * 64)


def untile_blocks(phys, E, d):
    """Operand tiles of an [E][d] matrix (128-row blocks, the last one
    partial; per block the k-tiles [rows][64], chunk c of row r at position
    c ^ (r % 8)) back to row-major [E][d]."""
    out = np.zeros((E, d), np.float32)
    off = 0
    for b0 in range(0, E, 128):
        rows = min(128, E - b0)
        for j in range(d // 64):
            t = phys[off: off + rows * 64].reshape(rows, 8, 8)
            pos = np.arange(8)[None, :] ^ (np.arange(rows)[:, None] % 8)
            out[b0:b0 + rows, 64 * j:64 * j + 64] = np.take_along_axis(t, pos[..., None], axis=1).reshape(rows, 64)
            off += rows * 64
    return out


def test_moe_weight_layout_matches_logical_tensors():
    d, E, F, L = 256, 4, 192, 3
    wr = torch.empty(E * d, dtype=torch.bfloat16, device=dev())
    wgu = torch.empty(E * 2 * F * d, dtype=torch.bfloat16, device=dev())
    wd = torch.empty(E * d * F, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_moe_weights(wr, wgu, wd, d, E, F, L, 5, 0.02)
    base = 100 + 16 * L
    assert np.array_equal(untile_blocks(bf16_to_f32(wr), E, d), ow.tensor(5, base + 4, (E, d), 0.02))
    # gate/up: per expert the operand tiles of W_gate [F][d], then those of
    # W_up (F = 192: a full 128-row block and a 64-row one)
    phys = bf16_to_f32(wgu).reshape(E, 2, F * d)
    g = ow.tensor(5, base + 5, (E, F, d), 0.02)
    u = ow.tensor(5, base + 6, (E, F, d), 0.02)
    for e in range(E):
        assert np.array_equal(untile_blocks(phys[e, 0], F, d), g[e])
        assert np.array_equal(untile_blocks(phys[e, 1], F, d), u[e])
    wdl = untile(bf16_to_f32(wd), (E,), d // 128, F // 64)
    assert np.array_equal(wdl, ow.tensor(5, base + 7, (E, d, F), 0.02))


def test_router_layout_with_a_partial_expert_block():
    d, E, F, L = 128, 200, 64, 1
    wr = torch.empty(E * d, dtype=torch.bfloat16, device=dev())
    wgu = torch.empty(E * 2 * F * d, dtype=torch.bfloat16, device=dev())
    wd = torch.empty(E * d * F, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_moe_weights(wr, wgu, wd, d, E, F, L, 9, 0.02)
    assert np.array_equal(untile_blocks(bf16_to_f32(wr), E, d), ow.tensor(9, 100 + 16 * L + 4, (E, d), 0.02))


# ---- sampler: bit-exact given identical logits --------------------------------

def gpu_sampler(l, scfg, step, canvas, state):
    C, V = l.shape
    L = torch.from_numpy(np.ascontiguousarray(l)).to(dev())
    part = new_partials(C, V)
    dgp.dg_op_logits_partials(L, C, V, scfg.sample_seed, canvas, step, part)
    x = torch.from_numpy(state.x.copy()).to(dev())
    com = torch.from_numpy(state.committed.copy()).to(dev())
    last = torch.from_numpy(state.last.copy()).to(dev())
    stab = torch.from_numpy(state.stable.copy()).to(dev())
    a = torch.zeros(C, dtype=torch.int32, device=dev())
    conf = torch.zeros(C, dtype=torch.float32, device=dev())
    g = torch.zeros(C, dtype=torch.int32, device=dev())
    done = torch.zeros(1, dtype=torch.int32, device=dev())
    dgp.dg_op_sampler_update(part, C, V, step, scfg, x, com, last, stab, a, conf, g, done)
    torch.cuda.synchronize()
    return dict(part=partial_planes(part, C, V), a=a.cpu().numpy(), conf=conf.cpu().numpy(),
                g=g.cpu().numpy(), x=x.cpu().numpy(), committed=com.cpu().numpy(),
                last=last.cpu().numpy(), stable=stab.cpu().numpy(), done=bool(done.item()))


def oracle_partials(l, seed, canvas, step, positions=None, inv_tau=np.float32(1.0)):
    """Partials of the rows of l, row r being canvas position positions[r]."""
    positions = np.arange(l.shape[0]) if positions is None else np.asarray(positions)
    G = dgmath.gumbel_from_uniform(philox.gumbel_uniforms(seed, canvas, step, positions, l.shape[1]))
    return osamp.tile_partials(l, G, inv_tau)


@pytest.mark.parametrize("C,V,seed", [(256, 1024, 0), (40, 768, 3), (32, 262144, 9)])
def test_sampler_partials_and_outputs_bit_exact(C, V, seed):
    l = synth.logits(C, V, seed=seed)
    scfg = dgp.SamplerConfig(canvas_len=C, sample_seed=seed * 7 + 1)
    st = osamp.CanvasState(philox.canvas_init_ids(scfg.sample_seed, 2, C, V))
    got = gpu_sampler(l, scfg, 3, 2, st)
    ref = oracle_partials(l, scfg.sample_seed, 2, 3)
    for k in ("m", "a", "s", "gk", "gi"):
        assert np.array_equal(got["part"][k], ref[k]), k
    a, conf, g, _ = osamp.position_outputs(l, scfg.sample_seed, 2, 3)
    assert np.array_equal(got["a"], a)
    assert np.array_equal(got["conf"].view(np.uint32), conf.view(np.uint32))
    assert np.array_equal(got["g"], g)
    done = osamp.apply_rule(st, a, conf, g, 3, scfg.budget_N)
    for k in ("x", "committed", "last", "stable"):
        assert np.array_equal(got[k], getattr(st, k)), k
    assert got["done"] == done


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_tempered_sampler_partials_bit_exact(tau):
    C, V = 64, 65536
    l = synth.logits(C, V, seed=21)
    inv = np.float32(1.0 / tau)
    part = new_partials(C, V)
    dgp.dg_op_logits_partials(torch.from_numpy(l).to(dev()), C, V, 77, 1, 9, part, inv_tau=float(inv))
    got = partial_planes(part, C, V)
    ref = oracle_partials(l, 77, 1, 9, inv_tau=inv)
    for k in ("m", "a", "s", "gk", "gi"):
        assert np.array_equal(got[k].view(np.uint32), ref[k].astype(got[k].dtype).view(np.uint32)), k


def test_sampler_full_vocab_full_canvas_sampled_rows():
    C, V = 256, 262144
    l = synth.logits(C, V, seed=11, scale=2.0)
    scfg = dgp.SamplerConfig(sample_seed=5)
    st = osamp.CanvasState(np.zeros(C, np.int32))
    got = gpu_sampler(l, scfg, 1, 0, st)
    rows = np.array([0, 1, 77, 128, 200, 255])
    ref = oracle_partials(l[rows], 5, 0, 1, rows)
    for k in ("m", "a", "s", "gk", "gi"):
        assert np.array_equal(got["part"][k][rows], ref[k]), k
    r = osamp.reduce_tiles(ref)
    assert np.array_equal(got["a"][rows], r["a"])
    assert np.array_equal(got["g"][rows], r["gi"])
    assert np.array_equal(got["conf"][rows].view(np.uint32),
                          (np.float32(1) / r["s"]).astype(np.float32).view(np.uint32))


def test_sampler_rule_branches_over_scripted_steps():
    C, V, N = 64, 512, 5
    rng = np.random.default_rng(4)
    scfg = dgp.SamplerConfig(canvas_len=C, budget_N=N, sample_seed=21)
    st = osamp.CanvasState(rng.integers(0, V, C).astype(np.int32))
    gst = st.copy()
    target = rng.integers(0, V, C)
    done = False
    for n in range(1, N + 1):
        l = rng.standard_normal((C, V)).astype(np.float32)
        hot = np.arange(C) < 8 * n                      # more rows spike each step (stable argmax)
        l[hot, target[hot]] += 6.0
        l[:4, target[:4]] += 40.0                       # confident: commit at once
        got = gpu_sampler(l, scfg, n, 1, gst)
        a, conf, g, _ = osamp.position_outputs(l, 21, 1, n)
        done = osamp.apply_rule(st, a, conf, g, n, N)
        for k in ("x", "committed", "last", "stable"):
            assert np.array_equal(got[k], getattr(st, k)), (n, k)
        assert got["done"] == done
        gst = st.copy()
        if done:
            break
    assert done and st.committed.all()


# ---- LM head fused with the vocab reduction -------------------------------------

@pytest.mark.parametrize("rows,d,V,sample", [
    (256, 256, 1024, None),
    (200, 256, 1024, None),                  # a last row block of 72 rows
    (384, 320, 2048, None),                  # three row blocks sharing each vocab tile, five k-steps
    (512, 256, 4096, None),                  # four row blocks
    (256, 2816, 262144, [0, 63, 64, 130, 255])])
def test_lm_head_partials_against_fp64_logits(rows, d, V, sample):
    xf, xt = synth.normal_bf16((rows, d), seed=2)
    xn = tiles_dev(xt)
    w = torch.empty(V * d, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_tiled_weights(w, V, d, 0, 2, 0.02)
    part = new_partials(rows, V)
    dgp.dg_op_lm_head_partials(xn, w, rows, d, V, 3, 1, 2, part)
    got = partial_planes(part, rows, V)
    sample = np.arange(rows) if sample is None else np.asarray(sample)
    x64 = xf[sample].astype(np.float64)
    lo = np.empty((len(sample), V))
    for v0 in range(0, V, 16384):                     # oracle weights, chunk by chunk
        nv = min(16384, V - v0)
        Wc = ow.elements(0, 2, v0 * d, nv * d, 0.02).reshape(nv, d).astype(np.float64)
        lo[:, v0:v0 + nv] = x64 @ Wc.T
    ref = oracle_partials(lo.astype(np.float32), 3, 1, 2, sample)
    assert rel_err(got["m"][sample], ref["m"]) <= TOL
    tiles = lo.reshape(len(sample), V // 256, 256)
    clear = top2_gap(tiles) > 1e-2
    assert np.array_equal(got["a"][sample][clear], ref["a"][clear])
    assert np.allclose(got["s"][sample], ref["s"], rtol=TOL)


def test_gumbel_noise_matches_oracle_on_every_input():
    # All 2^23 distinct uniforms (the low 9 bits of a word are dropped; they
    # are random here).  With the transform strictly increasing (a CPU pin of
    # the oracle), this makes the LM-head epilogue's per-bucket noise bound exact.
    i = np.arange(1 << 23, dtype=np.uint32)
    low = np.random.default_rng(0).integers(0, 512, 1 << 23, dtype=np.uint32)
    words = torch.from_numpy(((i << np.uint32(9)) | low).view(np.int32)).to(dev())
    out = torch.empty(1 << 23, dtype=torch.float32, device=dev())
    dgp.dg_op_gumbel_noise(words, out)
    u = (2 * i.astype(np.int64) + 1).astype(np.float32) * np.float32(2.0 ** -24)
    ref = dgmath.gumbel_from_uniform(u)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def _lm_head_rows(C, d, seed, split):
    """Final-norm-like rows: fp32 N(0, 1), as bf16 (hi) and, with `split`, the
    bf16 rounding of the remainder (lo).  Rows 0-7 are zero (every logit is
    exactly 0: all ties, the Gumbel winner decided by the noise alone and
    every noise bucket a candidate); rows 8-15 are scaled by 1e-3 (near-flat
    logits: many keys within a few ulp of the running maximum)."""
    x = np.random.default_rng(seed).standard_normal((C, d)).astype(np.float32)
    x[:8] = 0.0
    x[8:16] *= np.float32(1e-3)
    xt = torch.from_numpy(x)
    hi = xt.to(torch.bfloat16)
    lo = (xt - hi.float()).to(torch.bfloat16) if split else None
    return tiles_dev(hi), (tiles_dev(lo) if split else None)


@pytest.mark.parametrize("split,canvas,step,seed,rows,inv_tau", [
    (True, 0, 1, 5, None, 1.0),                              # the decoder's hi/lo instantiation, every row
    (False, 3, 17, (1 << 40) + 9, [0, 5, 8, 13, 16, 100, 129, 255], 1.0 / 0.7)])   # tempered re-noise keys
def test_lm_head_epilogue_partials_bit_exact_on_its_own_logits(split, canvas, step, seed, rows, inv_tau):
    """The decoder's fused LM-head epilogue, bit for bit: one launch writes the
    fp32 logits and the partials reduced from the same accumulators; the
    oracle's canonical tile partials of those logits (with the oracle's own
    Gumbel stream) must equal them in every plane, and the partials-only
    launch the decoder runs must equal them too."""
    C, d, V = 256, 2816, 262144
    w = torch.empty(V * d, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_tiled_weights(w, V, d, 0, 2, 0.02)
    hi, lo = _lm_head_rows(C, d, 31 + step, split)
    logits = torch.empty(C, V, dtype=torch.float32, device=dev())
    inv_tau = np.float32(inv_tau)
    both = new_partials(C, V)
    dgp.dg_op_lm_head_partials(hi, w, C, d, V, seed, canvas, step, both, xn_lo=lo, logits=logits,
                               inv_tau=float(inv_tau))
    only = new_partials(C, V)
    dgp.dg_op_lm_head_partials(hi, w, C, d, V, seed, canvas, step, only, xn_lo=lo, inv_tau=float(inv_tau))
    injected = new_partials(C, V)
    dgp.dg_op_logits_partials(logits, C, V, seed, canvas, step, injected, inv_tau=float(inv_tau))
    torch.cuda.synchronize()
    assert torch.equal(both, only)          # the decoder's partials-only launch: same bits
    assert torch.equal(both, injected)      # the injected-logit entry: same code, same bits
    l = logits.cpu().numpy()
    assert np.all(l[:8] == 0.0)
    got = partial_planes(both, C, V)
    sample = np.arange(C) if rows is None else np.asarray(rows)
    ref = oracle_partials(l[sample], seed, canvas, step, sample, inv_tau)
    for k in ("m", "a", "s", "gk", "gi"):
        assert np.array_equal(got[k][sample].view(np.uint32), ref[k].astype(got[k].dtype).view(np.uint32)), k
    # merge + rule on the GPU against the oracle on the same logits
    scfg = dgp.SamplerConfig(sample_seed=seed)
    st = osamp.CanvasState(philox.canvas_init_ids(seed, canvas, C, V))
    st.last[::3] = 7                                         # some positions one step from stable
    st.stable[::3] = 1
    st.committed[::11] = 1
    x, com = torch.from_numpy(st.x.copy()).to(dev()), torch.from_numpy(st.committed.copy()).to(dev())
    last, stab = torch.from_numpy(st.last.copy()).to(dev()), torch.from_numpy(st.stable.copy()).to(dev())
    a = torch.zeros(C, dtype=torch.int32, device=dev())
    conf = torch.zeros(C, dtype=torch.float32, device=dev())
    g = torch.zeros(C, dtype=torch.int32, device=dev())
    done = torch.zeros(1, dtype=torch.int32, device=dev())
    dgp.dg_op_sampler_update(only, C, V, step, scfg, x, com, last, stab, a, conf, g, done)
    torch.cuda.synchronize()
    r = osamp.reduce_tiles(ref)
    assert np.array_equal(a.cpu().numpy()[sample], r["a"])
    assert np.array_equal(g.cpu().numpy()[sample], r["gi"])
    assert np.array_equal(conf.cpu().numpy()[sample].view(np.uint32),
                          (np.float32(1) / r["s"]).astype(np.float32).view(np.uint32))
    assert np.all(a.cpu().numpy()[:8] == 0)                  # all-equal logits: the first index
    if rows is None:
        co = (np.float32(1) / r["s"]).astype(np.float32)
        d_ref = osamp.apply_rule(st, r["a"].astype(np.int32), co, r["gi"].astype(np.int32), step, scfg.budget_N)
        for k, t in (("x", x), ("committed", com), ("last", last), ("stable", stab)):
            assert np.array_equal(t.cpu().numpy(), getattr(st, k)), k
        assert bool(done.item()) == d_ref


# ---- canvas attention -----------------------------------------------------------

def pool_layout(blocks):
    """(page, head) blocks [..., pg, hd] (slot-major) to the pool's storage
    order: hd/64 sub-blocks [pg][64] in which the 16-byte chunk c of slot s
    sits at chunk position c ^ (s % 8)."""
    *lead, pg, hd = blocks.shape
    x = blocks.reshape(*lead, pg, hd // 64, 8, 8)
    s = np.arange(pg)[:, None]
    src = np.arange(8)[None, :] ^ (s % 8)      # logical chunk stored at position c
    x = np.take_along_axis(x, np.broadcast_to(src[:, None, :, None], (pg, hd // 64, 8, 8)).reshape(
        (1,) * len(lead) + (pg, hd // 64, 8, 8)), axis=-2)
    return np.moveaxis(x, -3, -4).reshape(*lead, pg, hd)


def paged(kv, Hkv, hd, pg, n_pages, perm):
    """Scatter logical keys [S][Hkv][hd] into pages through the page table `perm`."""
    pool = np.zeros((n_pages, Hkv, pg, hd), np.float32)
    for j in range(kv.shape[0]):
        pool[perm[j // pg], :, j % pg, :] = kv[j]
    return pool_layout(pool)


@pytest.mark.parametrize("P,causal,Hq,Hkv,hd", [
    (0, False, 16, 4, 128), (1000, False, 16, 4, 128), (1024, True, 16, 4, 128),
    (8192, False, 16, 4, 128), (32768, False, 16, 4, 128),
    (64, False, 4, 2, 64), (200, True, 4, 2, 64), (2048, False, 16, 8, 128)])
def test_canvas_attention_against_fp64(P, causal, Hq, Hkv, hd):
    C, pg = 256, 128
    S = P + C
    n_pages = (S + pg - 1) // pg + 3
    perm = np.random.default_rng(P + 1).permutation(n_pages)[: (S + pg - 1) // pg]
    qf, qt = synth.normal_bf16((C, Hq, hd), seed=10)
    kf, _ = synth.normal_bf16((S, Hkv, hd), seed=11)
    vf, _ = synth.normal_bf16((S, Hkv, hd), seed=12)
    kp = torch.from_numpy(paged(kf, Hkv, hd, pg, n_pages, perm)).to(torch.bfloat16).to(dev())
    vp = torch.from_numpy(paged(vf, Hkv, hd, pg, n_pages, perm)).to(torch.bfloat16).to(dev())
    table = torch.from_numpy(perm.astype(np.int32)).to(dev())
    out = torch.empty(C, Hq, hd, dtype=torch.bfloat16, device=dev())
    ws = torch.empty(max(dgp.dg_op_attention_workspace_bytes(P, C, Hq, Hkv, hd), 1), dtype=torch.uint8, device=dev())
    dgp.dg_op_canvas_attention(qt.to(dev()), kp, vp, table, P, C, Hq, Hkv, hd, pg, causal, out, ws)
    ref = om.attention(qf.astype(np.float64), kf.astype(np.float64), vf.astype(np.float64),
                       om.visibility(P, C, "causal" if causal else "bidir"))
    assert rel_err(bf16_to_f32(out), ref) <= TOL


# ---- mixture of experts -----------------------------------------------------------

@pytest.mark.parametrize("T,d,E,k,F", [(256, 256, 8, 2, 512), (77, 256, 8, 2, 512), (256, 2816, 128, 8, 704),
                                       (64, 256, 200, 4, 128),
                                       # d = 384: a down unit with a single 128-row block of W_down;
                                       # F = 192: a gate/up unit of 64 features; a ragged token group
                                       (130, 384, 16, 3, 192),
                                       # ~150 rows per expert: experts split into several work items
                                       (300, 384, 4, 2, 128)])
def test_moe_against_fp64(T, d, E, k, F):
    wr = torch.empty(E * d, dtype=torch.bfloat16, device=dev())
    wgu = torch.empty(E * 2 * F * d, dtype=torch.bfloat16, device=dev())
    wd = torch.empty(E * d * F, dtype=torch.bfloat16, device=dev())
    dgp.dg_op_fill_moe_weights(wr, wgu, wd, d, E, F, 0, 0, 0.02)
    xf, xt = synth.normal_bf16((T, d), seed=3)
    y = torch.empty(T, d, dtype=torch.float32, device=dev())
    ids = torch.empty(T, k, dtype=torch.int32, device=dev())
    gates = torch.empty(T, k, dtype=torch.float32, device=dev())
    ws = torch.empty(dgp.dg_op_moe_workspace_bytes(T, d, E, k, F), dtype=torch.uint8, device=dev())
    dgp.dg_op_moe(xt.to(dev()), wr, wgu, wd, T, d, E, k, F, y, ids, gates, ws)
    gi = ids.cpu().numpy()
    W = dict(wr=ow.tensor(0, 104, (E, d), 0.02), wg=ow.tensor(0, 105, (E, F, d), 0.02),
             wu=ow.tensor(0, 106, (E, F, d), 0.02), wd=ow.tensor(0, 107, (E, d, F), 0.02))
    x64 = xf.astype(np.float64)
    ids_o, gates_o, r = om.route(x64, W["wr"], k)
    # routing: exact where the top-(k+1) logits are separated, valid everywhere
    srt = -np.sort(-r, axis=1)
    sep = np.all(np.diff(-srt[:, : k + 1], axis=1) > 1e-2, axis=1)
    assert np.array_equal(gi[sep], ids_o[sep])
    _, g_ref, _ = om.route(x64, W["wr"], k, forced=gi)      # raises unless a valid top-k
    assert np.abs(gates.cpu().numpy() - g_ref).max() <= TOL
    y_ref = om.moe_given_routing(x64, gi, g_ref, W)
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


@pytest.mark.parametrize("d", [512, 128])
def test_moe_split_overflow_gate_up_units_against_fp64(d):
    """Gate/up units just past a whole number of waves run split along K (the
    last part sums the parts in order): a routing whose unit count exceeds the
    SM count by at most a quarter of it, against the fp64 oracle.  At d = 128
    a unit has two k-steps, fewer than its four parts: it must run whole.
    The parts are summed in a fixed order, so a second launch on the same
    inputs must give the same bits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k, F = 8, 704
    mA = (F + 127) // 128
    found = None
    for E in (26, 28, 24, 30):
        for T in (256, 240, 272, 224, 288):
            wr = torch.empty(E * d, dtype=torch.bfloat16, device=dev())
            wgu = torch.empty(E * 2 * F * d, dtype=torch.bfloat16, device=dev())
            wd = torch.empty(E * d * F, dtype=torch.bfloat16, device=dev())
            dgp.dg_op_fill_moe_weights(wr, wgu, wd, d, E, F, 0, 0, 0.02)
            xf, xt = synth.normal_bf16((T, d), seed=5)
            y = torch.empty(T, d, dtype=torch.float32, device=dev())
            ids = torch.empty(T, k, dtype=torch.int32, device=dev())
            gates = torch.empty(T, k, dtype=torch.float32, device=dev())
            ws = torch.empty(dgp.dg_op_moe_workspace_bytes(T, d, E, k, F), dtype=torch.uint8, device=dev())
            dgp.dg_op_moe(xt.to(dev()), wr, wgu, wd, T, d, E, k, F, y, ids, gates, ws)
            gi = ids.cpu().numpy()
            items = int(sum((c + 127) // 128 for c in np.bincount(gi.ravel(), minlength=E) if c > 0))
            n_a = items * mA
            if n_a > sms and 0 < n_a % sms <= sms // 4:
                y2, ids2, gates2 = torch.empty_like(y), torch.empty_like(ids), torch.empty_like(gates)
                dgp.dg_op_moe(xt.to(dev()), wr, wgu, wd, T, d, E, k, F, y2, ids2, gates2, ws)
                assert torch.equal(ids, ids2) and torch.equal(gates, gates2)
                assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
                found = (T, E, xf, gi, gates.cpu().numpy(), y.cpu().numpy())
                break
        if found:
            break
    assert found, "no routing with a few gate/up units past a whole wave"
    T, E, xf, gi, g_gpu, y_gpu = found
    W = dict(wr=ow.tensor(0, 104, (E, d), 0.02), wg=ow.tensor(0, 105, (E, F, d), 0.02),
             wu=ow.tensor(0, 106, (E, F, d), 0.02), wd=ow.tensor(0, 107, (E, d, F), 0.02))
    x64 = xf.astype(np.float64)
    _, g_ref, _ = om.route(x64, W["wr"], k, forced=gi)      # raises unless a valid top-k
    assert np.abs(g_gpu - g_ref).max() <= TOL
    y_ref = om.moe_given_routing(x64, gi, g_ref, W)
    assert rel_err(y_gpu, y_ref) <= TOL


# ---- KV append (bit-exact indexing) ----------------------------------------------

def test_kv_append_bit_exact_with_shuffled_pages():
    L, n_pages, pg, Hkv, hd, pos0, n = 3, 8, 128, 2, 64, 200, 256
    perm = np.random.default_rng(0).permutation(n_pages).astype(np.int32)
    rng = np.random.default_rng(1)
    kn = rng.integers(0, 65535, (L, n, Hkv, hd), dtype=np.uint16)
    vn = rng.integers(0, 65535, (L, n, Hkv, hd), dtype=np.uint16)
    sentinel = 0x7FC1
    kp = torch.full((L, n_pages, Hkv, pg, hd), sentinel, dtype=torch.int16, device=dev())
    vp = torch.full((L, n_pages, Hkv, pg, hd), sentinel, dtype=torch.int16, device=dev())
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).to(dev())
    dgp.dg_op_kv_append(to_dev(kn), to_dev(vn), kp, vp, torch.from_numpy(perm).to(dev()), L, n_pages,
                        pos0, n, Hkv, hd, pg)
    kref = np.full((L, n_pages, Hkv, pg, hd), sentinel, np.uint16)
    vref = kref.copy()
    for t in range(n):
        p = pos0 + t
        kref[:, perm[p // pg], :, p % pg, :] = kn[:, t]
        vref[:, perm[p // pg], :, p % pg, :] = vn[:, t]
    assert np.array_equal(kp.cpu().numpy().view(np.uint16), pool_layout(kref))
    assert np.array_equal(vp.cpu().numpy().view(np.uint16), pool_layout(vref))


# ---- failure detection (no GPU fault: a wait that nothing completes) -------------

def test_bounded_wait_gives_up_and_reports_etimeout():
    # The bounded wait of the tensor-core kernels, on a barrier nothing
    # arrives at, must give up after its limit, record its code in the status
    # word (dg_op_status -> DG_ETIMEOUT, then cleared) and leave the context
    # usable: an attention call afterwards is still correct.
    dgp.dg_op_status()
    dgp.dg_op_wait_selftest(200_000)
    with pytest.raises(dgp.DgError) as e:
        dgp.dg_op_status()
    assert e.value.code == dgp.DG_ETIMEOUT and "code 99" in str(e.value)
    dgp.dg_op_status()
    test_canvas_attention_against_fp64(1000, False, 16, 4, 128)
    dgp.dg_op_status()
