"""Adaptive verify width, chosen on the device each cycle (oracle; test infrastructure only).

lucebox-hub PR #15 "MTP speculative decoding", *What* and *Speed*: the default verify width is
adaptive -- it settles at seven drafts on a prompt the draft head predicts well and stays small
where it does not. The pages do not give the controller; this is a plain reading of it: an
exponential moving average of the acceptance rate at each draft depth plus a
cycle-cost table, choosing the width with the most expected tokens per unit of cost.

State per request (all float64 here): rate[d] for depth d = 1..7 -- the average, over the
cycles that reached depth d, of "draft d was accepted given drafts 1..d-1 were" -- and the
number of cycles observed.

Update from one cycle's acceptance result (status, n_accept, eos_hit) at width k:
    depth d = 1..n_accept: accepted (x = 1);
    depth d = n_accept + 1 <= k, unless the block ended at an accepted EOS: rejected (x = 0);
    deeper depths: not observed.
    Each observation moves the depth's belief b[d] as rate[d] = b[d] + alpha * (x - b[d]), b
    taken before the cycle's update. The belief of an observed depth is its rate; that of a
    depth never observed is the belief of the depth above it (0.5 for depth 1): a deeper draft
    is assumed to do as well as the last one seen until it is tried, so widths grow while drafts
    keep being accepted (with a fixed 0.5 for unseen depths a width of 1 never looks worth
    extending and depth 2 is never observed). A depth observed before but not in this cycle
    relaxes towards the belief of the depth above it, rate[d] += alpha * (b'[d-1] - rate[d]),
    in increasing d with b' the updated beliefs: a depth that once looked poor is tried again
    once the relaxation makes it pay, instead of never being observed again (measured: a
    width stuck at 1 after a few early rejections at depth 2). A request whose status is not OK
    leaves its state unchanged.

Choice: expected tokens at width k, with the depths independent at their beliefs,
    E(k) = 1 + sum_{j=1..k} prod_{i=1..j} rate[i]
(each accepted draft is a token, and the cycle always ends with one more: the correction or the
bonus); the next width is the k in [1, k_max] maximising E(k) / cost[k], the smallest on ties.
The width never drops to 0: at least the first draft is always tried, so depth 1 stays observed
and a request whose drafts start failing can recover (at width 0 nothing would be observed).

Per-request cycle-cost fit (same page, *What*: besides the acceptance seen at each draft depth,
the width follows a fit of what a cycle costs for that request; the fit's form is this build's
reading). A cycle at width k costs
about a + b*k: a for the verify and acceptance, b for each draft step. Each observed cycle (its
width k and its measured cost c > 0, status OK) moves the moving averages of k, k^2, c and k*c
by alpha (the first observation sets them), which is exponentially weighted least squares:
    var = E[k^2] - E[k]^2,  b = (E[k c] - E[k] E[c]) / var,  a = E[c] - b E[k].
The fit is used when the widths have varied enough to separate the two terms (var >= 1/4) and
a, b > 0; its ratio b / a is then kept, so that once the width settles (var decays) the last
fitted shape still applies. Without a usable fit, and before any, the caller's cost table is
the prior. A measured cost above four times the fitted one (a host pause between cycles) is
not folded in.

Pinned by: E(k) against exhaustive enumeration of the 2^k accept/reject patterns with those
rates, and against a Monte Carlo of the acceptance chain; the EMA against its closed form; the
choice at the corner cases (rates 1 -> k_max, rates 0 -> 1, flat cost -> the largest width);
the fit against exact linear costs (a and b recovered), against numpy's weighted least squares
with the same exponential weights, and its fallbacks (one width only -> the prior; a settled
width -> the kept ratio).
"""

import numpy as np

PRIOR = 0.5
STATUS_OK = 0


VAR_MIN = 0.25    # widths must have varied at least this much (variance of k) for a fit
OUTLIER = 4.0     # a cost above OUTLIER times the fitted one is not folded in


def new_state(k_max=7):
    return {"rate": [None] * (k_max + 1), "cycles": 0, "fit": None, "ratio": 0.0}


def fit_model(state):
    """(a, b) of the current fit, or None when it is not usable (see the module doc)."""
    fit = state["fit"]
    if fit is None:
        return None
    mk, mkk, mc, mkc = fit
    var = mkk - mk * mk
    if not var >= VAR_MIN:
        return None
    b = (mkc - mk * mc) / var
    a = mc - b * mk
    if not (a > 0 and b > 0):
        return None
    return a, b


def observe_cost(state, status, k, cost, alpha):
    """Fold one cycle's measured cost at width k into the fit (status OK and cost > 0)."""
    if status != STATUS_OK or not cost > 0:
        return state
    x = [float(k), float(k * k), float(cost), float(k * cost)]
    if state["fit"] is None:
        state["fit"] = x
    else:
        model = fit_model(state)
        if model is not None and cost > OUTLIER * (model[0] + model[1] * k):
            return state
        state["fit"] = [m + alpha * (xi - m) for m, xi in zip(state["fit"], x)]
    model = fit_model(state)
    if model is not None:
        state["ratio"] = model[1] / model[0]
    return state


def costs(state, prior, k_max):
    """The cost of a cycle at each width 0..k_max: 1 + ratio * k from the fit (its last usable
    shape), else the caller's prior table."""
    if state["ratio"] > 0:
        return [1.0 + state["ratio"] * k for k in range(k_max + 1)]
    return [float(c) for c in prior[:k_max + 1]]


def observe(state, status, n_accept, eos_hit, k, alpha):
    """Update the per-depth rates from one cycle's result (see the module doc)."""
    if status != STATUS_OK:
        return state
    rate = state["rate"]
    before = rates(state)
    seen = set()
    for d in range(1, k + 1):
        if d <= n_accept:
            x = 1.0
        elif d == n_accept + 1 and not eos_hit:
            x = 0.0
        else:
            break
        rate[d] = before[d] + alpha * (x - before[d])
        seen.add(d)
    for d in range(2, len(rate)):  # relax the depths this cycle did not observe
        if d not in seen and rate[d] is not None:
            above = rates(state)[d - 1]
            rate[d] = rate[d] + alpha * (above - rate[d])
    state["cycles"] += 1
    return state


def rates(state):
    """Beliefs b[0..k_max]: the rate of an observed depth, else the belief of the depth above
    (PRIOR for depth 1); b[0] is unused."""
    b = [PRIOR] * len(state["rate"])
    for d in range(1, len(b)):
        r = state["rate"][d]
        b[d] = float(r) if r is not None else (b[d - 1] if d > 1 else PRIOR)
    return b


def expected_tokens(rate, k):
    """E(k) = 1 + sum_j prod_{i<=j} rate[i] (rate[0] unused)."""
    total, run = 1.0, 1.0
    for j in range(1, k + 1):
        run *= rate[j]
        total += run
    return total


def choose(state, cost, k_max):
    """The width in [min(1, k_max), k_max] with the most expected tokens per unit of cost
    (smallest on ties), the cost being the fitted one when the state holds a usable fit and
    the table ``cost`` otherwise. Returns (k, values) with values[k] for every k in [0, k_max]."""
    r = rates(state)
    cost = costs(state, cost, k_max) if "ratio" in state else cost
    vals = [expected_tokens(r, k) / cost[k] for k in range(k_max + 1)]
    lo = min(1, k_max)
    best = max(range(lo, k_max + 1), key=lambda k: (vals[k], -k))
    return best, vals
