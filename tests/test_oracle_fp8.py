"""Pins of oracle/fp8.py: e4m3 rounding against torch's float8 conversion, the
per-row power-of-two scale rule and the error bound of a quantized row."""
import numpy as np
import torch

from oracle import fp8


def _all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)].astype(np.float64)


def test_e4m3_rounding_equals_torch_on_every_bf16_value_in_range():
    v = _all_bf16_values()
    v = v[np.abs(v) <= fp8.E4M3_MAX]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(v), ref)


def test_e4m3_saturates_and_keeps_exact_grid_points():
    assert fp8.e4m3_round(np.array([449.0, 1e6, -500.0])).tolist() == [448.0, 448.0, -448.0]
    grid = np.array([0.0, 2.0 ** -9, 3 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 240.0, 448.0])
    assert np.array_equal(fp8.e4m3_round(grid), grid)
    # ties to even: 2^-10 lies halfway between 0 and 2^-9; 1.0625 between 1 and 1.125
    assert fp8.e4m3_round(np.array([2.0 ** -10, 1.0625, 1.1875])).tolist() == [0.0, 1.0, 1.25]


def test_e4m3_bits_round_trip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)   # 0x7F / 0xFF: NaN
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_bits(vals)
    # -0 and +0 both encode as +0 here (the kernels never produce -0 bits differently from +0 values)
    nz = vals != 0
    assert np.array_equal(got[nz], codes[nz])


def test_scale_exponent_brackets_the_row_maximum():
    rng = np.random.default_rng(5)
    a = np.abs(rng.standard_normal(20000)) * np.exp2(rng.integers(-30, 30, 20000))
    a = np.concatenate([a, [448.0, 448.0 * 2.0 ** 5, np.nextafter(448.0, 1e9), 0.875 * 2.0 ** 9, 2.0 ** 9]])
    k = fp8.scale_exponent(a)
    assert np.all(a <= 448.0 * np.exp2(k.astype(np.float64)))
    assert np.all(a > 448.0 * np.exp2(k.astype(np.float64) - 1))
    assert fp8.scale_exponent(np.array([0.0]))[0] == 0


def test_quantized_rows_are_within_half_a_step():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32).astype(np.float64)
    q, k = fp8.quantize_rows(w)
    back = fp8.dequantize_rows(q, k)
    # e4m3 normals carry 3 mantissa bits: |error| <= 2^-4 |w| (half a step); below 2^-6 the step is 2^-9
    step = np.exp2(k.astype(np.float64))[:, None] * np.maximum(
        np.exp2(np.floor(np.log2(np.maximum(np.abs(np.ldexp(w, -k[:, None])), 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(back - w) <= step / 2 + 1e-300)
    assert np.all(np.max(np.abs(q), axis=1) <= fp8.E4M3_MAX)
    assert np.all(np.max(np.abs(q), axis=1) >= fp8.E4M3_MAX / 2)   # the scale uses the range


def test_bf16_round_equals_torch():
    from oracle import model
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(100000) * np.exp2(rng.integers(-20, 20, 100000)),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 65504.0]])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(model.bf16_round(v32.astype(np.float64)), ref)


def test_fp8_gate_product_obeys_the_rounding_bound():
    # each e4m3 operand carries a relative error of at most 2^-4 (half of a
    # 3-bit mantissa step) above the subnormal range, the bf16 input rounding
    # 2^-9 more: |x_q w_q - x w| <= sum |x||w| (2^-4 + 2^-4 + 2^-9 + products),
    # plus subnormal steps (2^-10 of the row scale) -- a bound, not an average:
    # e4m3 dot products keep a few percent of relative error (no averaging
    # over d for random-sign sums)
    from oracle import model
    rng = np.random.default_rng(8)
    d, F, n = 256, 128, 16
    x = rng.standard_normal((n, d))
    wg = rng.standard_normal((F, d)) * 0.02
    xq = fp8.dequantize_rows(*fp8.quantize_rows(model.bf16_round(x)))
    wq = fp8.dequantize_rows(*fp8.quantize_rows(wg))
    exact, q = x @ wg.T, xq @ wq.T
    _, kx = fp8.quantize_rows(model.bf16_round(x))
    _, kw = fp8.quantize_rows(wg)
    rel = 2 * 2.0 ** -4 + 2.0 ** -9 + 2.0 ** -7
    sub = np.exp2(kx - 10.0)[:, None] * np.sum(np.abs(wg), axis=1)[None, :] + \
        np.sum(np.abs(x), axis=1)[:, None] * np.exp2(kw - 10.0)[None, :]
    bound = rel * (np.abs(x) @ np.abs(wg).T) + sub
    assert np.all(np.abs(q - exact) <= bound)
    assert np.max(np.abs(q - exact)) > 0       # the operands were quantized
