"""The FP8 (e4m3) expert path (dg_config.expert_fp8): the weight quantizer bit
for bit against the oracle's, and the decoder with e4m3 gate/up products
against the oracle's FP8 forward."""
import numpy as np
import pytest
import torch

import discrete_diffusion_block_gb300 as dgp
from discrete_diffusion_block_gb300 import synth
from gpu_util import bits_to_f32, dev, rel_err, tiles_dev
from oracle import fp8, model as om, weights as ow

pytestmark = pytest.mark.gpu
TOL = 2e-2
P = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from discrete_diffusion_block_gb300 import build
    build.build()
    dgp.load()
    torch.cuda.set_device(0)


def _tile_positions(rows, cols):
    """Element index in operand tiles of every (r, c) of a [rows][cols] matrix."""
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    b, rr, kt, cc = r >> 7, r & 127, c >> 6, c & 63
    rows_b = np.minimum(128, rows - 128 * b)
    return 128 * cols * b + rows_b * 64 * kt + rr * 64 + ((((cc >> 3) ^ (rr & 7)) << 3) | (cc & 7))


def _untile_e4m3(flat, rows, cols):
    """e4m3 operand tiles (the bytes of bf16 tiles of [rows][cols/2]) -> [rows][cols] codes."""
    words = np.ascontiguousarray(flat).view(np.uint16)
    return words[_tile_positions(rows, cols // 2)].copy().view(np.uint8).reshape(rows, cols)


def test_quantizer_matches_the_oracle_bit_for_bit():
    rng = np.random.default_rng(11)
    n_mat, R, C = 3, 200, 384              # a ragged second row block, three k-tiles of 128
    w = rng.standard_normal((n_mat, R, C)) * 0.02
    w[0, 5] = 0.0                                          # a zero row: exponent 0, all codes 0
    w[1, 7] = rng.standard_normal(C) * 1e-6                # tiny values: exponents far below 0
    w[2, 9] = rng.standard_normal(C)
    w[2, 9, 3] = 448.0 * 2.0 ** -3                         # the row maximum on a scale boundary
    w[2, 11] = rng.standard_normal(C) * 1e3
    bf = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
    src = torch.cat([tiles_dev(bf[i]) for i in range(n_mat)])
    dst = torch.empty(n_mat * R * C, dtype=torch.uint8, device=dev())
    exps = torch.empty(n_mat * R, dtype=torch.int32, device=dev())
    dgp.dg_op_quantize_rows_e4m3(src, n_mat, R, C, dst, exps)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().reshape(n_mat, R * C)
    k_got = exps.cpu().numpy().reshape(n_mat, R)
    wb = bf.to(torch.float64).numpy()
    for i in range(n_mat):
        q, k = fp8.quantize_rows(wb[i])
        assert np.array_equal(k_got[i], k), i
        assert np.array_equal(_untile_e4m3(got[i], R, C), fp8.e4m3_bits(q)), i
    assert k_got[0, 5] == 0 and not _untile_e4m3(got[0], R, C)[5].any()


def _fp8_model():
    cfg = dgp.tiny_config(expert_fp8=1)
    return dgp.dg_init_model(cfg, dgp.SamplerConfig(budget_N=8))


def _routing(m, skip_last):
    n = om.TINY.n_layers
    return [None if (skip_last and L == n - 1) else dgp.dg_read_routing(m, L) for L in range(n)]


def test_fp8_decoder_matches_the_fp8_oracle():
    W = ow.Weights(om.TINY)
    cfg8 = om.TINY.with_(expert_fp8=True)
    m = _fp8_model()
    prompt = synth.prompt_ids(P, 1024, seed=1)
    dgp.dg_prefill(m, prompt)
    prefill_routing = _routing(m, skip_last=True)
    cache = om.prefill(W, cfg8, prompt, routing=prefill_routing)
    for L in range(2):
        k, v = dgp.dg_read_kv(m, L, 0, P)
        assert rel_err(bits_to_f32(k), cache.k[L]) <= TOL
        assert rel_err(bits_to_f32(v), cache.v[L]) <= TOL
    # the e4m3 path is the one that ran: layer 1's keys (which follow layer 0's
    # expert output) are farther from the bf16 oracle's (same layer-0 routing,
    # valid for both: the router reads bf16) than from the FP8 oracle's
    k1 = bits_to_f32(dgp.dg_read_kv(m, 1, 0, P)[0])
    cache16 = om.prefill(W, om.TINY, prompt, routing=[prefill_routing[0], None])
    e8, e16 = rel_err(k1, cache.k[1]), rel_err(k1, cache16.k[1])
    print(f"layer-1 keys: vs FP8 oracle {e8:.2e}, vs bf16 oracle {e16:.2e}")
    assert e16 > 2 * e8
    logits = torch.empty(256, 1024, dtype=torch.float32, device=dev())
    dgp.dg_canvas_logits(m, logits)
    ids = dgp.dg_read_canvas(m)["ids"]
    routing = _routing(m, skip_last=False)
    lo8 = om.canvas_logits(W, cfg8, cache, ids, P, routing=routing)
    assert rel_err(logits.cpu().numpy(), lo8) <= TOL
    # a full canvas decodes to the end
    done, n = False, 0
    while not done:
        done = dgp.dg_denoise_step(m)
        n += 1
    assert n == 8
    dgp.dg_commit_canvas(m)
    m.close()


def test_fp8_needs_d_model_a_multiple_of_128():
    with pytest.raises(dgp.DgError) as e:
        dgp.dg_init_model(dgp.tiny_config(expert_fp8=1, d_model=192, d_ff=512), dgp.SamplerConfig(budget_N=8))
    assert e.value.code == dgp.DG_EINVAL
