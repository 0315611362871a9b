"""Multi-request batching (lockstep): B requests share every denoising and
KV-append forward (B * 256 rows through the projections, the expert FFN and
the LM head).  Request b samples with sample_seed + b; its tokens, step
counts and Eq. 7-10 must be those of a single-request model with that seed,
bit for bit: every row of a forward is computed as in a single request's
forward (attention per request with the request's own key splits, the
projections and the expert FFN row by row, the sampler per request)."""
import numpy as np
import pytest
import torch

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from discrete_diffusion_block_gb300 import build
    build.build()
    dgp.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("skw", [dict(budget_N=6), dict(budget_N=5, temp_start=1.4, temp_end=0.7),
                                 dict(budget_N=6, conf_threshold=0.004)])
def test_batched_generation_equals_single_requests(skw):
    B, K = 3, 2
    prompts = [synth.prompt_ids(n, 1024, seed=50 + n) for n in (64, 100, 37)]   # different prefixes
    scfg = dgp.SamplerConfig(sample_seed=11, **skw)
    mb = dgp.dg_init_model(dgp.tiny_config(max_requests=B), scfg)
    out_b, st_b = dgp.dg_generate_batch(mb, prompts, K)
    mb.close()
    for b in range(B):
        ms = dgp.dg_init_model(dgp.tiny_config(), dgp.SamplerConfig(**{**scfg.__dict__, "sample_seed": 11 + b}))
        out_s, st_s = dgp.dg_generate(ms, prompts[b], K)
        ms.close()
        assert st_b[b]["K"] == st_s["K"] and st_b[b]["N_k"] == st_s["N_k"] and st_b[b]["C_k"] == st_s["C_k"], b
        for key in ("total_tokens", "total_steps", "effective_steps", "tpf"):
            assert st_b[b][key] == st_s[key], (b, key)
        assert np.array_equal(out_b[b][:st_s["K"]], out_s), b


def test_batch_model_rejects_single_request_calls():
    m = dgp.dg_init_model(dgp.tiny_config(max_requests=2), dgp.SamplerConfig(budget_N=2))
    for call in (lambda: dgp.dg_prefill(m, synth.prompt_ids(16, 1024)), lambda: dgp.dg_denoise_step(m),
                 lambda: dgp.dg_generate(m, synth.prompt_ids(16, 1024), 1)):
        with pytest.raises(dgp.DgError) as e:
            call()
        assert e.value.code == dgp.DG_EINVAL
    dgp.dg_prefill_batch(m, [synth.prompt_ids(16, 1024, seed=1), synth.prompt_ids(70, 1024, seed=2)])
    steps = dgp.dg_denoise_canvas_batch(m)
    assert steps == [2, 2]
    ids, valid = dgp.dg_commit_canvas_batch(m)
    assert ids.shape == (2, 256) and valid == [256, 256]
    assert dgp.dg_read_canvas(m)["prefix_len"] == 16 + 256      # request 0
    m.close()
