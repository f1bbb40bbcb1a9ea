"""Property pins of the oracle: invariants that hold for any input, checked on many random
inputs (hypothesis). They complement the exact pins (enumerated laws, closed forms, published
vectors) by sweeping the input space for a mistake those cases could miss.

* filtered_probs: a distribution, supported on its kept set; the kept set is a prefix of the
  (logit descending, id ascending) order, at most top_k long, and cut where the top-p rule
  says; invariant under adding a constant to every logit; nested in top_k and in top_p.
* inverse_cdf: the chosen bin contains u*S and carries weight; on a dyadic grid of u each bin
  is chosen for exactly the grid points its cumulative weights enclose.
* adapt: beliefs stay in [0, 1] under any sequence of cycle results; the chosen width is in
  range; E(k) never decreases in k; all-accepting and all-rejecting histories choose the
  extreme widths.
"""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from oracle import accept, adapt  # noqa: E402

SETTINGS = settings(max_examples=150, deadline=None, derandomize=True)

logit_rows = st.lists(st.integers(-40, 40), min_size=1, max_size=48).map(
    lambda xs: np.array(xs, dtype=np.float64) / 8.0)  # multiples of 1/8: many exact ties


def _order(z):
    return sorted(range(len(z)), key=lambda t: (-z[t], t))


@SETTINGS
@given(z=logit_rows, T=st.floats(0.1, 4.0), top_k=st.integers(1, 40),
       top_p=st.floats(0.01, 1.0))
def test_filtered_probs_invariants(z, T, top_k, top_p):
    p, kept, margins = accept.filtered_probs(z, T, top_k, top_p)
    V = len(z)
    kept = [int(t) for t in kept]
    assert (p >= 0).all() and abs(p.sum() - 1.0) <= 1e-12
    assert set(np.flatnonzero(p)) == set(kept)
    assert 1 <= len(kept) <= min(top_k, V)
    order = _order(z)
    assert kept == order[:len(kept)]
    # the top-p rule on the top-k distribution: the mass ahead of the last kept token is below
    # top_p, and the mass ahead of the first dropped one (inside the top-k set) is not
    kk = min(top_k, V)
    w = np.exp((z[order[:kk]] - z[order[0]]) / T)
    pk = w / w.sum()
    ahead = np.concatenate(([0.0], np.cumsum(pk)))
    assert ahead[len(kept) - 1] < top_p
    if len(kept) < kk:
        assert ahead[len(kept)] >= top_p
    assert all(m >= 0 for _, m in margins)


@SETTINGS
@given(z=logit_rows, T=st.floats(0.1, 4.0), top_k=st.integers(1, 40),
       top_p=st.floats(0.01, 1.0), c=st.integers(-64, 64))
def test_filtered_probs_shift_invariant(z, T, top_k, top_p, c):
    p0, k0, m0 = accept.filtered_probs(z, T, top_k, top_p)
    p1, k1, _ = accept.filtered_probs(z + c / 4.0, T, top_k, top_p)  # exact shifts
    if dict(m0)["cdf"] > 1e-9:  # away from a top-p boundary the kept set cannot move
        assert list(k0) == list(k1)
        assert np.allclose(p0, p1, rtol=1e-12, atol=1e-15)


@SETTINGS
@given(z=logit_rows, T=st.floats(0.1, 4.0), top_k=st.integers(1, 39),
       top_p=st.floats(0.01, 0.99))
def test_filtered_kept_sets_nest(z, T, top_k, top_p):
    _, a, _ = accept.filtered_probs(z, T, top_k, 1.0)
    _, b, _ = accept.filtered_probs(z, T, top_k + 1, 1.0)
    assert list(a) == list(b[:len(a)])
    _, c, _ = accept.filtered_probs(z, T, top_k, top_p)
    _, d, _ = accept.filtered_probs(z, T, top_k, min(1.0, top_p + 0.01))
    assert list(c) == list(d[:len(c)]) and len(c) <= len(d)


@SETTINGS
@given(w=st.lists(st.integers(0, 9), min_size=1, max_size=20).filter(lambda v: sum(v) > 0),
       u=st.integers(0, (1 << 24) - 1))
def test_inverse_cdf_bin_contains_the_target(w, u):
    w = np.array(w, dtype=np.float64)
    j, margin = accept.inverse_cdf(w, u / 2.0**24)
    c = np.cumsum(w)
    t = u / 2.0**24 * c[-1]
    assert w[j] > 0
    assert (c[j - 1] if j else 0.0) <= t < c[j]
    assert margin >= 0


@SETTINGS
@given(w=st.lists(st.integers(0, 7), min_size=1, max_size=12).filter(lambda v: sum(v) > 0))
def test_inverse_cdf_law_on_a_grid(w):
    """On the dyadic grid u = i / 2^10 (u * S exact for these integer weights) bin j is chosen
    for exactly the i with c[j-1] <= i * S / 2^10 < c[j]: ceil(c[j] 2^10 / S) - ceil(c[j-1]
    2^10 / S) grid points, counted in integers."""
    S = sum(w)
    c = np.cumsum([0] + list(w))
    n = 1 << 10
    counts = [0] * len(w)
    for i in range(n):
        counts[accept.inverse_cdf(np.array(w, dtype=np.float64), i / n)[0]] += 1
    ceil = [-((-int(cj) * n) // S) for cj in c]
    assert counts == [ceil[j + 1] - ceil[j] for j in range(len(w))]


cycle = st.tuples(st.integers(0, 1), st.integers(0, 7), st.booleans(), st.integers(0, 7))


@SETTINGS
@given(hist=st.lists(cycle, max_size=40), alpha=st.floats(0.01, 1.0),
       k_max=st.integers(0, 7))
def test_adapt_beliefs_stay_probabilities(hist, alpha, k_max):
    s = adapt.new_state()
    for status, n_acc, eos, k in hist:
        k = min(k, 7)
        n_acc = min(n_acc, k)
        s = adapt.observe(s, status, n_acc, eos and n_acc > 0, k, alpha)
    r = adapt.rates(s)
    assert all(0.0 <= x <= 1.0 for x in r[1:])
    cost = [1.0 + 0.5 * i for i in range(8)]
    kb, vals = adapt.choose(s, cost, k_max)
    assert min(1, k_max) <= kb <= k_max
    E = [adapt.expected_tokens(r, k) for k in range(8)]
    assert all(E[i] <= E[i + 1] for i in range(7))


@pytest.mark.parametrize("x,expect", [(1, 7), (0, 1)])
def test_adapt_extreme_histories(x, expect):
    s = adapt.new_state()
    for _ in range(200):
        # x = 1: every draft of width 7 accepted; x = 0: the first draft rejected
        s = adapt.observe(s, 0, 7 if x else 0, False, 7, 0.2)
    cost = [1.0 + 0.1 * i for i in range(8)]
    assert adapt.choose(s, cost, 7)[0] == expect
