"""The allocation-free canvas attention entry point.

Some callers cannot give the library device memory: a host framework owns
and budgets every byte of it (a serving engine's memory pool), a plugin
signature has no workspace argument, or an allocation inside a
latency-critical loop is not acceptable.  dg_op_canvas_attention_noalloc
serves them: it takes only inputs and outputs, allocates nothing, and the
only device memory it touches besides them is the library's fixed status
word.  It must give the workspace entry point's results (and the fp64
oracle's, within the tolerance of the other attention tests) on calls in a
row, and leave the device's free memory unchanged.

This file is collected last on purpose; it must pass on its own in a fresh
process and after the other tests.
"""
import numpy as np
import pytest
import torch

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import synth
from gpu_util import bf16_to_f32, dev, rel_err
from oracle import model as om

pytestmark = pytest.mark.gpu
TOL = 2e-2
PG = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from discrete_diffusion_block_gb300 import build
    build.build()
    dgp.load()
    torch.cuda.set_device(0)


def _case(P, Hq, Hkv, hd, seed, C=256):
    """Paged pools (shuffled page table, two spare pages) and the logical
    q, K, V they hold, for the oracle."""
    S = P + C
    n_used = (S + PG - 1) // PG
    n_pages = n_used + 2
    perm = np.random.default_rng(seed).permutation(n_pages)[:n_used].astype(np.int32)
    qf, qt = synth.normal_bf16((C, Hq, hd), seed=seed)
    pools, logical = [], []
    for s in (seed + 1, seed + 2):
        pf, pt = synth.normal_bf16((n_pages, Hkv, PG, hd), seed=s)
        pools.append(pt.to(dev()))
        logical.append(pf)
    return qf, qt.to(dev()), pools, logical, perm


def _logical_keys(pool_f32, perm, S, hd):
    """Keys 0..S-1 out of a pool in the swizzled (page, head) block layout:
    per block hd/64 sub-blocks [PG slots][64], the 16-byte chunk c of slot s
    stored at chunk position c ^ (s % 8); key j in page perm[j // PG]."""
    n_pages, Hkv = pool_f32.shape[:2]
    x = pool_f32.reshape(n_pages, Hkv, hd // 64, PG, 8, 8)
    slot = np.arange(PG)[:, None]
    pos = np.arange(8)[None, :] ^ (slot % 8)                 # stored position of logical chunk c
    x = np.take_along_axis(x, np.broadcast_to(pos[None, None, None, :, :, None], x.shape), axis=4)
    blocks = np.moveaxis(x, 2, 3).reshape(n_pages, Hkv, PG, hd)
    keys = blocks[perm].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)
    return keys[:S]


def _noalloc(L, q, kp, vp, table, P, Hq, Hkv, hd, causal, out):
    rc = L.dg_op_canvas_attention_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(), P,
                                          256, Hq, Hkv, hd, PG, kp.shape[0], int(causal), out.data_ptr(), None)
    assert rc == dgp.DG_OK, L.dg_last_error()


@pytest.mark.parametrize("calls", [[(2048, 16, 8, 128, False), (1000, 16, 4, 128, True)]])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls(calls):
    L = dgp.load()
    cases = []
    for i, (P, Hq, Hkv, hd, causal) in enumerate(calls):
        qf, q, (kp, vp), (kf, vf), perm = _case(P, Hq, Hkv, hd, seed=40 + i)
        table = torch.from_numpy(perm).to(dev())
        ref = torch.empty(256, Hq, hd, dtype=torch.bfloat16, device=dev())
        ws = torch.empty(max(dgp.dg_op_attention_workspace_bytes(P, 256, Hq, Hkv, hd), 1), dtype=torch.uint8,
                         device=dev())
        dgp.dg_op_canvas_attention(q, kp, vp, table, P, 256, Hq, Hkv, hd, PG, causal, ref, ws)
        cases.append((P, Hq, Hkv, hd, causal, qf, q, kp, vp, kf, vf, perm, table, ref))
    outs = [torch.empty_like(c[-1]) for c in cases]      # the caller's outputs, allocated up front
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for (P, Hq, Hkv, hd, causal, _, q, kp, vp, _, _, _, table, ref), out in zip(cases, outs):   # two calls in a row
        _noalloc(L, q, kp, vp, table, P, Hq, Hkv, hd, causal, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0                      # the calls held no device memory
    dgp.dg_op_status()                         # no wait gave up, no bad page index
    for (P, Hq, Hkv, hd, causal, qf, _, _, _, kf, vf, perm, _, ref), out in zip(cases, outs):
        assert rel_err(bf16_to_f32(out), bf16_to_f32(ref)) <= TOL
        S = P + 256
        o64 = om.attention(qf.astype(np.float64), _logical_keys(kf, perm, S, hd).astype(np.float64),
                           _logical_keys(vf, perm, S, hd).astype(np.float64),
                           om.visibility(P, 256, "causal" if causal else "bidir"))
        assert rel_err(bf16_to_f32(out), o64) <= TOL


def test_noalloc_covers_the_longest_contexts():
    # No shape needs device scratch: the split-KV partial states of up to 8
    # key splits are merged in distributed shared memory, 32k-token contexts
    # included.
    for P, Hq, Hkv, hd in [(32768, 64, 4, 128), (32768, 1, 1, 128), (32768, 16, 16, 64), (8192, 32, 8, 128)]:
        assert dgp.dg_op_attention_workspace_bytes(P, 256, Hq, Hkv, hd) == 0
    L = dgp.load()
    P, Hq, Hkv, hd = 32768, 2, 1, 128                    # few query tiles: 8 key splits per tile
    _, q, (kp, vp), _, perm = _case(P, Hq, Hkv, hd, seed=60)
    table = torch.from_numpy(perm).to(dev())
    ref = torch.empty(256, Hq, hd, dtype=torch.bfloat16, device=dev())
    ws = torch.empty(1, dtype=torch.uint8, device=dev())
    dgp.dg_op_canvas_attention(q, kp, vp, table, P, 256, Hq, Hkv, hd, PG, False, ref, ws)
    out = torch.empty_like(ref)
    _noalloc(L, q, kp, vp, table, P, Hq, Hkv, hd, False, out)
    torch.cuda.synchronize()
    dgp.dg_op_status()
    assert rel_err(bf16_to_f32(out), bf16_to_f32(ref)) <= TOL


def test_noalloc_reports_a_bad_page_index_through_the_status_word():
    # An entry outside the pools is never read (its keys are skipped) and is
    # reported by dg_op_status, which then clears the record.
    L = dgp.load()
    P, Hq, Hkv, hd = 1000, 16, 8, 128
    _, q, (kp, vp), _, perm = _case(P, Hq, Hkv, hd, seed=70)
    bad = perm.copy()
    bad[3] = kp.shape[0] + 7
    out = torch.empty(256, Hq, hd, dtype=torch.bfloat16, device=dev())
    _noalloc(L, q, kp, vp, torch.from_numpy(bad).to(dev()), P, Hq, Hkv, hd, False, out)
    with pytest.raises(dgp.DgError) as e:
        dgp.dg_op_status()
    assert e.value.code == dgp.DG_EINVAL
    assert torch.isfinite(out.float()).all()
    dgp.dg_op_status()                         # cleared
    _noalloc(L, q, kp, vp, torch.from_numpy(perm).to(dev()), P, Hq, Hkv, hd, False, out)
    dgp.dg_op_status()
