"""Pins for the sampler's fp32 exp/log: libm in double is the exact value."""
import math

import numpy as np

from oracle.dgmath import dg_exp, dg_log, gumbel_from_uniform


def _ulps(y, ref):
    y = np.asarray(y, np.float64)
    ulp = np.spacing(np.abs(np.asarray(ref, np.float32))).astype(np.float64)
    return np.abs(y - ref) / ulp


def test_exp_within_two_ulp():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-87, 88, 100000), rng.uniform(-30, 0, 100000)]).astype(np.float32)
    assert _ulps(dg_exp(x), np.exp(x.astype(np.float64))).max() <= 2.0


def test_log_within_two_ulp():
    rng = np.random.default_rng(2)
    x = np.concatenate([np.exp(rng.uniform(-85, 85, 100000)),
                        rng.uniform(0.5, 2.0, 100000),
                        rng.uniform(2.0 ** -24, 1.0, 100000)]).astype(np.float32)
    x = x[x != 1.0]
    assert _ulps(dg_log(x), np.log(x.astype(np.float64))).max() <= 2.0


def test_special_values():
    assert dg_exp(np.float32(0.0)) == 1.0
    assert dg_exp(np.float32(-np.inf)) == 0.0
    assert dg_exp(np.float32(-100.0)) == 0.0
    assert np.isinf(dg_exp(np.float32(100.0)))
    assert np.isnan(dg_exp(np.float32(np.nan)))
    assert dg_log(np.float32(1.0)) == 0.0
    assert dg_log(np.float32(0.0)) == -np.inf
    assert np.isnan(dg_log(np.float32(-1.0)))
    assert abs(float(dg_log(np.float32(2.0 ** -130))) - (-130 * math.log(2))) < 1e-4


def test_exp_log_round_trip():
    x = np.linspace(-20, 20, 4001).astype(np.float32)
    assert np.abs(dg_log(dg_exp(x)) - x).max() < 1e-5 * 20


def test_gumbel_moments():
    # Standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2 / 6.
    u = ((2 * np.arange(1 << 20) + 1) / float(1 << 21)).astype(np.float32)   # stratified uniforms
    g = gumbel_from_uniform(u).astype(np.float64)
    assert abs(g.mean() - 0.5772156649) < 2e-3
    assert abs(g.var() - math.pi ** 2 / 6) < 1e-2


def test_gumbel_noise_strictly_increasing_over_every_input():
    # The sampler's noise takes 2^23 distinct inputs u = (2 i + 1) 2^-24.  A
    # strictly increasing transform is what lets a kernel bound the noise of a
    # whole bucket of Philox words (those sharing their top byte) by its value
    # at the bucket's largest word; check it exhaustively, together with the
    # limits of the standard Gumbel at the two ends of the open interval.
    i = np.arange(1 << 23, dtype=np.int64)
    u = ((2 * i + 1).astype(np.float32) * np.float32(2.0 ** -24)).astype(np.float32)
    g = gumbel_from_uniform(u).astype(np.float64)
    assert np.all(np.diff(g) > 0)
    # -log(-log u) near u = 2^-24 and u = 1 - 2^-24, evaluated in double
    lo, hi = float(u[0]), float(u[-1])
    assert abs(g[0] - (-math.log(-math.log(lo)))) < 1e-5
    assert abs(g[-1] - (-math.log(-math.log(hi)))) < 1e-4
