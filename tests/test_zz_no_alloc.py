"""The allocation-free attention entry point against the workspace one.

Some callers cannot give the library device memory: their framework owns and
budgets every byte, their plugin signature has no workspace argument, or an
allocation inside a latency-critical loop is not acceptable.  For them
dg_op_canvas_attention_noalloc keeps its split-KV scratch in a fixed array
inside the library.  This file is collected last on purpose; it must pass on
its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import synth
from gpu_util import bf16_to_f32, dev, rel_err

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from discrete_diffusion_block_gb300 import build
    build.build()
    dgp.load()
    torch.cuda.set_device(0)


def _case(P, Hq, Hkv, hd, seed, C=256, pg=128):
    S = P + C
    n_pages = (S + pg - 1) // pg + 2
    perm = np.random.default_rng(seed).permutation(n_pages)[: (S + pg - 1) // pg].astype(np.int32)
    _, qt = synth.normal_bf16((C, Hq, hd), seed=seed)
    pools = []
    for s in (seed + 1, seed + 2):
        _, kv = synth.normal_bf16((n_pages, Hkv, pg, hd), seed=s)
        pools.append(kv.to(dev()))
    return qt.to(dev()), pools[0], pools[1], torch.from_numpy(perm).to(dev())


@pytest.mark.parametrize("calls", [[(2048, 16, 8, 128, False), (1000, 16, 4, 128, True)]])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(calls):
    L = dgp.load()
    for i, (P, Hq, Hkv, hd, causal) in enumerate(calls):
        need = dgp.dg_op_attention_workspace_bytes(P, 256, Hq, Hkv, hd)
        assert need == 0                                 # split-KV states are merged on chip
        q, kp, vp, table = _case(P, Hq, Hkv, hd, seed=40 + i)
        ref = torch.empty(256, Hq, hd, dtype=torch.bfloat16, device=dev())
        ws = torch.empty(1, dtype=torch.uint8, device=dev())
        dgp.dg_op_canvas_attention(q, kp, vp, table, P, 256, Hq, Hkv, hd, 128, causal, ref, ws)
        out = torch.empty_like(ref)
        rc = L.dg_op_canvas_attention_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                              table.data_ptr(), P, 256, Hq, Hkv, hd, 128,
                                              int(causal), out.data_ptr(), None)
        assert rc == dgp.DG_OK, L.dg_last_error()
        torch.cuda.synchronize()
        assert rel_err(bf16_to_f32(out), bf16_to_f32(ref)) <= TOL


def test_noalloc_covers_the_longest_contexts():
    # No shape needs device scratch: the split-KV partial states of up to 8
    # key splits are merged in distributed shared memory, 32k-token contexts
    # included.
    for P, Hq, Hkv, hd in [(32768, 64, 4, 128), (32768, 1, 1, 128), (32768, 16, 16, 64), (8192, 32, 8, 128)]:
        assert dgp.dg_op_attention_workspace_bytes(P, 256, Hq, Hkv, hd) == 0
    L = dgp.load()
    P, Hq, Hkv, hd = 32768, 2, 1, 128                    # few query tiles: 8 key splits per tile
    q, kp, vp, table = _case(P, Hq, Hkv, hd, seed=60)
    ref = torch.empty(256, Hq, hd, dtype=torch.bfloat16, device=dev())
    ws = torch.empty(1, dtype=torch.uint8, device=dev())
    dgp.dg_op_canvas_attention(q, kp, vp, table, P, 256, Hq, Hkv, hd, 128, False, ref, ws)
    out = torch.empty_like(ref)
    rc = L.dg_op_canvas_attention_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(), P,
                                          256, Hq, Hkv, hd, 128, 0, out.data_ptr(), None)
    assert rc == dgp.DG_OK, L.dg_last_error()
    torch.cuda.synchronize()
    assert rel_err(bf16_to_f32(out), bf16_to_f32(ref)) <= TOL
