"""Pins of the adaptive-width oracle (oracle/adapt.py) against what does not depend on it:
exhaustive enumeration and a Monte Carlo of the acceptance chain for E(k), the closed form of
the moving average, and the corner cases of the choice."""

import itertools

import numpy as np
import pytest

from oracle import adapt


@pytest.mark.parametrize("seed", range(5))
def test_expected_tokens_equals_enumeration(seed):
    """E(k) against all 2^k accept/reject patterns: the cycle keeps drafts up to the first
    rejection and always emits one more token."""
    rng = np.random.default_rng(seed)
    rate = [0.0] + list(rng.uniform(0, 1, 7))
    for k in range(0, 8):
        exp = 0.0
        for pattern in itertools.product((0, 1), repeat=k):
            pr = 1.0
            for d, x in enumerate(pattern, start=1):
                pr *= rate[d] if x else 1.0 - rate[d]
            kept = next((i for i, x in enumerate(pattern) if not x), k)
            exp += pr * (kept + 1)
        assert adapt.expected_tokens(rate, k) == pytest.approx(exp, rel=1e-12, abs=1e-12)


def test_expected_tokens_monte_carlo():
    rng = np.random.default_rng(7)
    rate = [0.0, 0.9, 0.8, 0.7, 0.6, 0.5, 0.4, 0.3]
    n, k = 200_000, 7
    u = rng.uniform(size=(n, k))
    ok = u < np.array(rate[1:k + 1])
    kept = np.where(ok.all(axis=1), k, np.argmin(ok, axis=1))
    assert adapt.expected_tokens(rate, k) == pytest.approx((kept + 1).mean(), rel=5e-3)


def test_moving_average_closed_form():
    """From the prior 0.5, one rejection of depth 1 and then n - 1 acceptances leave
    rate[1] = 1 - (1 - 0.5 (1 - alpha)) (1 - alpha)^(n - 1)."""
    alpha = 0.1
    st = adapt.new_state()
    adapt.observe(st, 0, 0, False, 3, alpha)
    assert st["rate"][1] == pytest.approx(0.5 * (1 - alpha), rel=1e-12)
    for n in range(2, 30):
        adapt.observe(st, 0, 3, False, 3, alpha)
        want = 1 - (1 - 0.5 * (1 - alpha)) * (1 - alpha) ** (n - 1)
        assert st["rate"][1] == pytest.approx(want, rel=1e-12)
    assert st["cycles"] == 29


def test_observation_rules():
    st = adapt.new_state()
    adapt.observe(st, 0, 2, False, 5, 0.5)  # depths 1, 2 kept, 3 rejected, 4-5 unseen
    assert st["rate"][1:6] == [0.75, 0.75, 0.25, None, None]
    adapt.observe(st, 0, 1, True, 5, 0.5)  # depth 1 kept and it was EOS: nothing else seen
    # depth 1: 0.75 -> 0.875; depths 2 and 3 relax halfway to the depth above, in order:
    # 0.75 + (0.875 - 0.75)/2 = 0.8125, then 0.25 + (0.8125 - 0.25)/2 = 0.53125
    assert st["rate"][1:6] == [0.875, 0.8125, 0.53125, None, None]
    adapt.observe(st, 1, 0, False, 5, 0.5)  # a failed request changes nothing
    assert st["cycles"] == 2
    assert adapt.rates(st)[4] == st["rate"][3]  # unseen depth: the belief of the one above


def test_unseen_depths_follow_the_last_seen_one():
    """Only depth 1 observed (accepted every cycle): every deeper depth is believed as good, so
    the width grows past 1 where a fixed 0.5 for unseen depths would keep it at 1."""
    st = adapt.new_state()
    for _ in range(40):
        adapt.observe(st, 0, 1, False, 1, 0.1)
    b = adapt.rates(st)
    assert b[1] > 0.95 and b[2:] == [b[1]] * 6
    cost = [1.0 + 0.5 * k for k in range(8)]
    assert adapt.choose(st, cost, 7)[0] > 1


def test_a_depth_that_looked_poor_is_tried_again():
    """Depth 2 rejected a few times early, then only width 1 chosen: the relaxation brings
    depth 2 back towards depth 1 until width 2 pays again (with depth 1 at ~0.87 and a draft
    costing half a cycle)."""
    st = adapt.new_state()
    cost = [1.0 + 0.5 * k for k in range(8)]
    for _ in range(30):
        adapt.observe(st, 0, 1, False, 1, 0.1)   # depth 1 accepted at width 1
    for _ in range(4):
        adapt.observe(st, 0, 1, False, 2, 0.1)   # depth 2 rejected at width 2
    k, _ = adapt.choose(st, cost, 7)
    assert k == 1                                # depth 2 now looks poor
    widths = []
    for _ in range(60):
        k, _ = adapt.choose(st, cost, 7)
        widths.append(k)
        adapt.observe(st, 0, min(k, 1), False, k, 0.1) if k == 1 else \
            adapt.observe(st, 0, k, False, k, 0.1)    # deeper drafts are in fact accepted
    assert max(widths) > 1 and widths[-1] > 1


def test_choice_corner_cases():
    cost = [1.0 + 0.3 * k for k in range(8)]
    st = adapt.new_state()
    st["rate"] = [None] + [1.0] * 7
    assert adapt.choose(st, cost, 7)[0] == 7
    st["rate"] = [None] + [0.0] * 7
    assert adapt.choose(st, cost, 7)[0] == 1  # never below one draft: depth 1 stays observed
    assert adapt.choose(st, cost, 0)[0] == 0
    flat = [1.0] * 8
    st["rate"] = [None] + [0.2] * 7
    assert adapt.choose(st, flat, 7)[0] == 7  # more width never loses when it costs nothing
    assert adapt.choose(st, flat, 3)[0] == 3
