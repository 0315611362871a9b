"""Pins for the commit / re-noise / stop sampler and its canonical reduction."""
import numpy as np
from scipy import special, stats

from oracle import sampler
from oracle.sampler import CanvasState, apply_rule, position_outputs

f32 = np.float32


def test_uniform_logits_give_conf_exactly_one_over_V():
    for V in (256, 1024, 262144 // 64):
        l = np.full((3, V), 0.37, f32)
        a, conf, g, _ = position_outputs(l, 0, 0, 1)
        assert np.all(conf == f32(1.0 / V))
        assert np.all(a == 0)                                    # tie -> lowest index


def test_one_hot_logits_give_confidence_near_one():
    V = 1024
    l = np.zeros((4, V), f32)
    hot = [3, 300, 777, 1023]
    l[np.arange(4), hot] = 30.0
    a, conf, g, _ = position_outputs(l, 0, 0, 1)
    assert list(a) == hot
    expect = 1.0 / (1.0 + (V - 1) * np.exp(-30.0))
    assert np.allclose(conf, expect, rtol=1e-6)
    assert list(g) == hot                                        # Gumbel noise cannot beat a gap of 30


def test_normaliser_and_argmax_against_fp64_softmax():
    rng = np.random.default_rng(0)
    l = (rng.standard_normal((16, 4096)) * 3).astype(f32)
    a, conf, g, r = position_outputs(l, 1, 0, 1)
    assert np.array_equal(a, np.argmax(l, axis=1))
    p = special.softmax(l.astype(np.float64), axis=1)
    assert np.allclose(conf, p.max(axis=1), rtol=2e-6)
    S = np.exp(l.astype(np.float64) - l.max(axis=1, keepdims=True)).sum(axis=1)
    assert np.allclose(r["s"], S, rtol=2e-6)


def test_tree_order_is_balanced_and_tiles_ascending():
    # A tie of the max in two different tiles must resolve to the lower tile;
    # a tie inside one tile to the lower index.
    V = 2048
    l = np.zeros((2, V), f32)
    l[0, [700, 1500]] = 5.0
    l[1, [1025, 1030]] = 5.0
    a, _, _, _ = position_outputs(l, 0, 0, 1)
    assert list(a) == [700, 1025]


def test_ragged_tile_count_pads_with_empty_slots():
    # 3 tiles (not a power of two) must give the same result as an fp64 reference
    rng = np.random.default_rng(3)
    l = rng.standard_normal((5, 768)).astype(f32)
    a, conf, g, _ = position_outputs(l, 0, 0, 1)
    assert np.array_equal(a, np.argmax(l, axis=1))
    assert np.allclose(conf, special.softmax(l.astype(np.float64), axis=1).max(axis=1), rtol=2e-6)


def test_gumbel_max_samples_the_softmax():
    # Chi-square of 1e5 Gumbel-max draws against softmax(l), V = 256, one tile.
    l = np.log(np.array([0.3, 0.2, 0.15, 0.1, 0.1, 0.05, 0.05, 0.05] + [1e-30] * 248)).astype(f32)
    draws = []
    for n in range(1, 401):
        _, _, g, _ = position_outputs(np.broadcast_to(l, (250, 256)), 11, 0, n)
        draws.append(g)
    draws = np.concatenate(draws)
    counts = np.bincount(draws, minlength=256)[:8]
    assert counts.sum() == len(draws)
    expect = special.softmax(l.astype(np.float64))[:8] * len(draws)
    assert stats.chisquare(counts, expect).pvalue > 1e-3


def test_confidence_threshold_commits_immediately():
    C = 4
    st = CanvasState(np.array([9, 9, 9, 9]))
    a = np.array([1, 2, 3, 4], np.int32)
    g = np.array([5, 6, 7, 8], np.int32)
    conf = np.array([0.95, 0.9, 0.8999999, 0.1], f32)
    done = apply_rule(st, a, conf, g, 1, 48)
    assert not done
    assert list(st.committed) == [1, 1, 0, 0]
    assert list(st.x) == [1, 2, 7, 8]                          # committed -> argmax, rest re-noised


def test_stability_commits_after_two_unchanged_steps():
    st = CanvasState(np.zeros(2, np.int32))
    conf = np.zeros(2, f32)
    seq_a = [np.array([5, 5]), np.array([5, 6]), np.array([5, 6]), np.array([7, 6])]
    g = np.array([100, 101], np.int32)
    got = []
    for n, a in enumerate(seq_a, start=1):
        apply_rule(st, a.astype(np.int32), conf, g, n, 48)
        got.append((list(st.committed), list(st.x)))
    # position 0: argmax 5 at steps 1,2,3 -> stable 2 at step 3 -> commits with 5
    # position 1: argmax 5,6,6,6 -> stable 0,0,1,2 -> commits at step 4 with 6
    assert got[0] == ([0, 0], [100, 101])
    assert got[1] == ([0, 0], [100, 101])
    assert got[2] == ([1, 0], [5, 101])
    assert got[3] == ([1, 1], [5, 6])                          # committed x never changes


def test_budget_exhaustion_takes_argmax_and_stops():
    st = CanvasState(np.zeros(3, np.int32))
    a = np.array([1, 2, 3], np.int32)
    for n in range(1, 4):
        done = apply_rule(st, (a + n).astype(np.int32), np.zeros(3, f32), np.array([7, 7, 7], np.int32), n, 3)
    assert done
    assert list(st.x) == [4, 5, 6] and st.committed.all()


def test_adaptive_stopping_and_adaptive_off():
    st = CanvasState(np.zeros(2, np.int32))
    one = np.ones(2, f32)
    assert apply_rule(st.copy(), np.array([1, 2], np.int32), one, np.zeros(2, np.int32), 1, 48)
    assert not apply_rule(st.copy(), np.array([1, 2], np.int32), one, np.zeros(2, np.int32), 1, 48,
                          adaptive=False)


def test_tile_partial_definition_matches_brute_force_in_small_case():
    # one position, one tile: s is the left-to-right fp32 sum of dg_exp(l - max)
    from oracle.dgmath import dg_exp
    rng = np.random.default_rng(5)
    l = rng.standard_normal((1, 256)).astype(f32)
    p = sampler.tile_partials(l, np.zeros_like(l))
    acc = f32(0)
    for v in range(256):
        acc = f32(acc + dg_exp(f32(l[0, v] - l.max())))
    assert p["s"][0, 0] == acc


def test_tempered_gumbel_max_samples_the_tempered_softmax():
    # Re-noise at temperature tau samples softmax(l / tau): chi-square of the
    # draws against it for a sharpening (0.5) and a flattening (2.0) tau; the
    # argmax and confidence stay those of tau = 1.
    l = np.log(np.array([0.3, 0.2, 0.15, 0.1, 0.1, 0.05, 0.05, 0.05] + [1e-30] * 248)).astype(f32)
    for tau in (0.5, 2.0):
        inv = f32(1.0 / tau)
        draws = []
        for n in range(1, 401):
            a, conf, g, _ = position_outputs(np.broadcast_to(l, (250, 256)), 13, 0, n, inv_tau=inv)
            draws.append(g)
        draws = np.concatenate(draws)
        counts = np.bincount(draws, minlength=256)[:8]
        assert counts.sum() == len(draws)
        expect = special.softmax(l.astype(np.float64) / tau)[:8] * len(draws)
        assert stats.chisquare(counts, expect).pvalue > 1e-3
        assert np.all(a == 0) and np.allclose(conf, 0.3, rtol=1e-5)


def test_temperature_one_keys_are_the_untempered_keys_and_schedule_endpoints():
    rng = np.random.default_rng(5)
    l = (rng.standard_normal((4, 1024)) * 2).astype(f32)
    a1 = position_outputs(l, 3, 1, 2)
    a2 = position_outputs(l, 3, 1, 2, inv_tau=sampler.annealed_inv_tau(5, 48))   # default schedule: tau = 1
    assert all(np.array_equal(x, y) for x, y in zip(a1[:3], a2[:3]))
    assert sampler.annealed_inv_tau(1, 48, 1.5, 0.5) == f32(1 / 1.5)
    assert sampler.annealed_inv_tau(48, 48, 1.5, 0.5) == f32(2.0)
    taus = [1 / float(sampler.annealed_inv_tau(n, 48, 1.5, 0.5)) for n in range(1, 49)]
    assert all(x > y for x, y in zip(taus, taus[1:]))
    assert sampler.annealed_inv_tau(1, 1, 0.8, 0.2) == f32(1 / 0.8)
    # a cold temperature turns the re-noise sample into the argmax where the
    # top-2 gap times 1/tau dwarfs the Gumbel range (< 20)
    l2 = l.copy()
    l2[:, 17] = l.max(axis=1) + f32(1.0)
    a, _, g, _ = position_outputs(l2, 3, 1, 2, inv_tau=f32(1000.0))
    assert np.array_equal(g, a) and np.all(a == 17)
