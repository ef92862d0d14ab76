"""The adaptive draft-tree planner ("Adaptive tree MTP"): oracle pins, then the library's
planner against the oracle on seeded synthetic acceptance statistics.  Host code only."""
import itertools
import random

import numpy as np
import pytest

from oracle import tree as T

import weight_only_quantised_gb300 as woq


# --------------------------------------------------------------------------- oracle pins

def test_shapes_are_the_64_compositions_of_seven():
    comps = set()
    for k in range(7):
        for cuts in itertools.combinations(range(1, 7), k):  # stars and bars
            edges = (0,) + cuts + (7,)
            comps.add(tuple(b - a for a, b in zip(edges, edges[1:])))
    s = T.shapes()
    assert len(s) == 64 == len(set(s)) and set(s) == comps
    assert s[0] == (7,) and s[1] == (1, 6) and s[63] == (1,) * 7


def _counts_from_probs(probs, mass=1000.0):
    return [[mass * p for p in row] for row in probs]


def _random_level_probs(rng, first_bias):
    out = []
    for _ in range(7):
        w = [rng.random() ** 2 for _ in range(8)]
        w[0] += first_bias
        s = sum(w)
        out.append([x / s for x in w])
    return out


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_expected_tokens_matches_simulating_the_drafting_process(seed):
    rng = random.Random(seed)
    probs = _random_level_probs(rng, first_bias=1.5)
    counts = _counts_from_probs(probs)
    for shape in [(1,) * 7, (7,), (2, 2, 3), (3, 1, 1, 1, 1)]:
        n = 60000
        total = sum(T.simulate_step(probs, shape, rng)[0] for _ in range(n))
        mean = total / n
        e = T.expected_tokens(counts, shape)
        assert abs(mean - e) < 4 * 1.5 / n ** 0.5 + 1e-9, (shape, mean, e)


def test_extreme_statistics_pick_the_obvious_shapes():
    always_first = [[1.0] + [0.0] * 7 for _ in range(7)]
    never_first = [[0.0] + [1.0 / 7] * 6 + [1.0 / 7] for _ in range(7)]
    c1 = _counts_from_probs(always_first)
    scores = [T.score(c1, 0.01, 1.0, s) for s in T.shapes()]
    assert T.shapes()[int(np.argmax(scores))] == (1,) * 7 and T.expected_tokens(c1, (1,) * 7) == 8.0
    c2 = _counts_from_probs(never_first)
    scores = [T.score(c2, 0.5, 1.0, s) for s in T.shapes()]
    assert T.shapes()[int(np.argmax(scores))] == (7,)
    assert abs(T.expected_tokens(c2, (7,)) - (1 + 6 / 7)) < 1e-12


def test_decay_closed_form():
    p = T.Planner(decay=0.9, replan_every=10 ** 9)
    for _ in range(37):
        p.observe([1, 2])
    assert abs(p.counts[0][0] - T.decayed_mass(0.9, 37)) < 1e-12
    assert abs(p.counts[1][1] - T.decayed_mass(0.9, 37)) < 1e-12
    assert p.counts[2] == [0.0] * 8


def _planner_with(probs, draft_ms, verify_ms, hysteresis=0.03):
    p = T.Planner(hysteresis=hysteresis, replan_every=10 ** 9)
    p.counts = _counts_from_probs(probs)
    p.draft_ms, p.verify_ms, p.times_seen = draft_ms, verify_ms, True
    return p


def test_hysteresis_margin():
    # statistics for level 1 only and free drafting: every shape costs the verify time, a
    # shape's tokens are 1 + P(rank <= w_1), so (7,) is best at 2 / (1 + p1) times the chain
    for ratio, expect_switch in [(1.02, False), (1.04, True)]:
        p1 = 2.0 / ratio - 1.0
        probs = [[p1] + [(1.0 - p1) / 6] * 6 + [0.0]] + [[0.0] * 8 for _ in range(6)]
        p = _planner_with(probs, 0.0, 1.0)
        assert abs(T.score(p.counts, 0.0, 1.0, (7,)) / T.score(p.counts, 0.0, 1.0, (1,) * 7) - ratio) < 1e-12
        best, s, changed = p.replan()
        assert T.shapes()[best] == (7,)
        assert changed == expect_switch
        assert p.shape == ((7,) if expect_switch else (1,) * 7)


# --------------------------------------------------------------------------- library vs oracle

def _synthetic_run(seed, steps=1200):
    """Seeded synthetic acceptance statistics: a predictable regime (deep chains hit)
    that turns into a creative one (the first choice often misses, a runner-up hits)."""
    rng = random.Random(seed)
    regime_a = _random_level_probs(rng, first_bias=4.0)
    regime_b = _random_level_probs(rng, first_bias=0.2)
    return rng, regime_a, regime_b


@pytest.mark.parametrize("seed", [7, 8])
def test_library_planner_matches_oracle(seed):
    rng, regime_a, regime_b = _synthetic_run(seed)
    lib = woq.TreePlanner()
    ora = T.Planner()
    switches = 0
    for step in range(1200):
        probs = regime_a if step < 600 else regime_b
        assert lib.shape == ora.shape
        _, ranks = T.simulate_step(probs, ora.shape, rng)
        draft_ms = 0.08 + 0.01 * rng.random()
        verify_ms = 1.0 + 0.05 * rng.random()
        s_lib = lib.observe(ranks, draft_ms, verify_ms)
        s_ora = ora.observe(ranks, draft_ms, verify_ms)
        assert s_lib == s_ora
        switches += s_ora
        np.testing.assert_allclose(lib.counts(), np.array(ora.counts), rtol=1e-12, atol=1e-12)
        assert abs(lib.state.draft_ms - ora.draft_ms) < 1e-12 and abs(lib.state.verify_ms - ora.verify_ms) < 1e-12
    assert switches >= 2  # it adapted to both regimes
    for s in T.shapes():
        e, sc = lib.score(s)
        assert abs(e - T.expected_tokens(ora.counts, s)) < 1e-12
        assert abs(sc - T.score(ora.counts, ora.draft_ms, ora.verify_ms, s)) < 1e-12


def test_library_shapes_and_errors():
    assert [woq.woq_tree_shape(i) for i in range(64)] == T.shapes()
    with pytest.raises(woq.WoqError):
        woq.woq_tree_shape(64)
    p = woq.TreePlanner()
    with pytest.raises(woq.WoqError):
        p.score((2, 2))        # does not lay out seven rows
    with pytest.raises(woq.WoqError):
        p.observe([2, 1])      # a chain continues only past a first-choice hit
    assert p.observe([]) is False
