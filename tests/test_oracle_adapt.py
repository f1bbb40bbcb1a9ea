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


# ---------------------------------------------------------------- the per-request cost fit

def _feed(st, ks, cs, alpha):
    for k, c in zip(ks, cs):
        adapt.observe_cost(st, 0, k, c, alpha)


def test_cost_fit_recovers_exact_linear_costs():
    """Costs exactly a + b*k at varying widths: the moving-average regression returns a and b
    whatever the weights (the covariance is b times the variance for any weighting)."""
    st = adapt.new_state()
    ks = [1, 5, 2, 7, 3, 6, 4] * 6
    _feed(st, ks, [113.0 + 61.5 * k for k in ks], 0.1)
    a, b = adapt.fit_model(st)
    assert a == pytest.approx(113.0, rel=1e-9) and b == pytest.approx(61.5, rel=1e-9)
    assert st["ratio"] == pytest.approx(61.5 / 113.0, rel=1e-9)
    assert adapt.costs(st, [9.0] * 8, 7)[3] == pytest.approx(1 + 3 * 61.5 / 113.0, rel=1e-9)


@pytest.mark.parametrize("seed", range(3))
def test_cost_fit_equals_weighted_least_squares(seed):
    """The moving averages are least squares with weights (1 - alpha)^(n-1) on the first
    observation and alpha (1 - alpha)^(n-1-i) on observation i: numpy's weighted polyfit with
    those weights gives the same line."""
    rng = np.random.default_rng(seed)
    alpha, n = 0.1, 60
    ks = rng.integers(1, 8, n)
    cs = 120.0 + 60.0 * ks + rng.normal(0, 8.0, n)
    st = adapt.new_state()
    _feed(st, ks, cs, alpha)
    w = np.array([(1 - alpha) ** (n - 1)] + [alpha * (1 - alpha) ** (n - 1 - i)
                                             for i in range(1, n)])
    b, a = np.polyfit(ks.astype(float), cs, 1, w=np.sqrt(w))
    fa, fb = adapt.fit_model(st)
    assert fa == pytest.approx(a, rel=1e-9) and fb == pytest.approx(b, rel=1e-9)


def test_cost_fit_fallbacks():
    prior = [1.0 + 0.5 * k for k in range(8)]
    st = adapt.new_state()
    _feed(st, [3] * 20, [300.0] * 20, 0.1)  # one width only: nothing to separate a from b
    assert adapt.fit_model(st) is None and adapt.costs(st, prior, 7) == prior
    adapt.observe_cost(st, 1, 5, 500.0, 0.1)  # a failed cycle is not folded in
    adapt.observe_cost(st, 0, 5, 0.0, 0.1)    # nor a cycle without a measured cost
    assert st["fit"] == [3.0, 9.0, 300.0, 900.0]
    st = adapt.new_state()
    _feed(st, [1, 7] * 10, [100.0 + 50.0 * k for k in [1, 7] * 10], 0.2)
    assert adapt.fit_model(st) is not None
    kept = st["ratio"]
    assert kept == pytest.approx(0.5, rel=1e-9)
    _feed(st, [4] * 60, [300.0] * 60, 0.2)  # the width settles: the variance decays
    assert adapt.fit_model(st) is None
    assert adapt.costs(st, prior, 7)[2] == pytest.approx(1 + 2 * kept, rel=1e-9)


def test_cost_fit_skips_outliers():
    st = adapt.new_state()
    ks = [1, 7, 3, 5] * 5
    _feed(st, ks, [100.0 + 50.0 * k for k in ks], 0.2)
    before = list(st["fit"])
    adapt.observe_cost(st, 0, 3, 4.5 * (100.0 + 150.0), 0.2)  # a host pause between cycles
    assert st["fit"] == before
    adapt.observe_cost(st, 0, 3, 3.5 * (100.0 + 150.0), 0.2)  # slow, but within the bound
    assert st["fit"] != before


def test_choice_follows_the_fitted_cost():
    """With every depth accepted at 0.9, a prior that makes draft steps cheap picks the widest
    width; a fit saying a draft step costs as much as the rest of the cycle picks fewer."""
    st = adapt.new_state()
    for _ in range(80):
        adapt.observe(st, 0, 7, False, 7, 0.1)
    st["rate"] = [None] + [0.9] * 7
    cheap = [1.0 + 0.01 * k for k in range(8)]
    assert adapt.choose(st, cheap, 7)[0] == 7
    ks = [1, 7, 2, 6] * 10
    _feed(st, ks, [100.0 + 100.0 * k for k in ks], 0.1)
    k, vals = adapt.choose(st, cheap, 7)
    e = [adapt.expected_tokens([0.0] + [0.9] * 7, kk) / (1 + kk) for kk in range(8)]
    assert k == max(range(1, 8), key=lambda kk: (e[kk], -kk))
    assert k < 7
