"""Pins of the sampling oracle (oracle/sampling.py): greedy, temperature, top-k, top-p and
repetition penalty after the tied lm_head ("Qwen3ASR ncnn多平台移植" sections 1, 2 and 6),
against published generator outputs, closed forms on small vocabularies and brute-force
frequencies."""
import math
import os

import numpy as np
import pytest

from oracle import sampling as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed0.txt")


def _golden():
    with open(GOLDEN) as f:
        return [int(l, 16) for l in f if l.strip() and not l.startswith("#")]


def test_splitmix64_published_outputs():
    assert S.splitmix64_outputs(0, 3) == _golden()


def test_counter_uniform_is_the_sequence_from_the_seed():
    for seed in (0, 1, 12345, 2**63 + 7):
        outs = S.splitmix64_outputs(seed, 5)
        for pos in range(5):
            u = S.counter_uniform(seed, pos)
            assert u == (outs[pos] >> 40) * 2.0 ** -24
            assert 0.0 <= u < 1.0
            assert np.float32(u) == u   # exact in float32


def test_counter_uniform_is_uniform():
    u = np.array([S.counter_uniform(7, pos) for pos in range(20000)])
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / u.size)
    hist, _ = np.histogram(u, bins=10, range=(0, 1))
    expect = u.size / 10
    assert np.all(np.abs(hist - expect) < 5 * math.sqrt(expect))


def test_repetition_penalty_closed_form_once_per_distinct_id():
    z = np.array([2.0, -2.0, 1.0, 0.5, 0.0])
    got = S.repetition_penalty(z, [0, 1, 1, 4, 4], 2.0)
    np.testing.assert_array_equal(got, [1.0, -4.0, 1.0, 0.5, 0.0])
    np.testing.assert_array_equal(S.repetition_penalty(z, [0, 1], 1.0), z)


def test_greedy_is_argmax_lowest_index():
    z = np.array([0.5, 3.0, 3.0, -1.0])
    for seed in range(5):
        assert S.sample_token(z, [], 0.0, 0, 1.0, 1.0, seed, seed) == 1
    # the penalty acts before the greedy pick
    assert S.sample_token(z, [1], 0.0, 0, 1.0, 4.0, 0, 0) == 2


def test_top_k_keeps_ties():
    z = np.array([1.0, 1.0, 1.0, 0.0, -1.0])
    np.testing.assert_array_equal(S.top_k_mask(z, 2), [True, True, True, False, False])
    np.testing.assert_array_equal(S.top_k_mask(z, 0), [True] * 5)
    np.testing.assert_array_equal(S.top_k_mask(z, 4), [True, True, True, True, False])


def test_top_p_closed_forms():
    z = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    allk = np.ones(4, dtype=bool)
    # sorted 0.4, 0.3, 0.2, 0.1: masses before each 0, 0.4, 0.7, 0.9
    np.testing.assert_array_equal(S.top_p_mask(z, allk, 0.5), [False, False, True, True])
    np.testing.assert_array_equal(S.top_p_mask(z, allk, 0.4), [False, False, False, True])
    np.testing.assert_array_equal(S.top_p_mask(z, allk, 0.95), [True, True, True, True])
    np.testing.assert_array_equal(S.top_p_mask(z, allk, 1e-9), [False, False, False, True])
    # equal probabilities: nothing is strictly more probable, all kept
    np.testing.assert_array_equal(S.top_p_mask(np.zeros(4), allk, 0.3), [True] * 4)


def test_top_k_one_and_tiny_top_p_are_greedy():
    rng = np.random.default_rng(3)
    for seed in range(200):
        z = rng.normal(size=50)
        best = int(np.argmax(z))
        assert S.sample_token(z, [], 0.8, 1, 1.0, 1.0, seed, 3) == best
        assert S.sample_token(z, [], 0.8, 0, 1e-9, 1.0, seed, 3) == best


def _freqs(z, n, **kw):
    counts = np.zeros(len(z))
    for seed in range(n):
        counts[S.sample_token(z, kw.get("history", []), kw.get("t", 1.0), kw.get("k", 0), kw.get("p", 1.0),
                              kw.get("r", 1.0), seed, 11)] += 1
    return counts / n


@pytest.mark.parametrize("kw,expect", [
    ({}, [0.1, 0.2, 0.3, 0.4]),
    ({"k": 2}, [0.0, 0.0, 3 / 7, 4 / 7]),
    ({"p": 0.5}, [0.0, 0.0, 3 / 7, 4 / 7]),
    ({"t": 0.5}, [0.01 / 0.30, 0.04 / 0.30, 0.09 / 0.30, 0.16 / 0.30]),   # p^2 normalised
    ({"history": [3], "r": math.exp(1.0)}, None),
])
def test_sampling_frequencies(kw, expect):
    z = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    if expect is None:
        # z3 = log 0.4 < 0: multiplied by e; probabilities proportional to the penalised exp
        z2 = z.copy()
        z2[3] *= math.e
        w = np.exp(z2)
        expect = w / w.sum()
    n = 20000
    f = _freqs(z, n, **kw)
    sd = np.sqrt(np.maximum(np.asarray(expect) * (1 - np.asarray(expect)), 1e-12) / n)
    assert np.all(np.abs(f - expect) <= 5 * sd + 1e-12), (f, expect)


def test_draw_picks_the_smallest_kept_id_for_small_u():
    z = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    seeds = [s for s in range(5000) if S.counter_uniform(s, 0) < 0.05][:20]
    assert seeds
    for s in seeds:
        assert S.sample_token(z, [], 1.0, 0, 1.0, 1.0, s, 0) == 0
        assert S.sample_token(z, [], 1.0, 2, 1.0, 1.0, s, 0) == 2
