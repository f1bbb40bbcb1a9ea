"""Pins for the oracle's drafting and acceptance (CPU only).

The target these tests hold the oracle to is fixed by the pages, not by the oracle:

* DS4Server issue #98, *Completion requirements*: "MTP preserves the target distribution" --
  the emitted tokens are a sample of the trunk's own autoregressive distribution. Checked
  exactly by enumerating every draft and every cell of the 24-bit uniforms at V = 8, and
  statistically by a chi-square test at V = 4096 over 10^6 seeded cycles.
* lucebox-hub PR #15, *Exactness*: at temperature 0 the output equals, byte for byte, decoding
  without drafts
  (sequential greedy decoding, written here with numpy's argmax).
* Special cases of the ratio rule: p == q accepts every draft; a one-hot q on a token the trunk
  gives probability zero is always rejected and the residual is p itself.
"""

import itertools
import multiprocessing as mp
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import accept, lmhead, philox

GRID = 2**24


class ToyModel:
    """Trunk and draft head over a tiny vocabulary whose logits are a seeded function of the
    whole prefix, so verify row r depends on x_0, d_1..d_r like a real trunk."""

    def __init__(self, V, Vd, scale, noise, seed=0):
        self.V, self.Vd, self.scale, self.noise, self.seed = V, Vd, scale, noise, seed
        self._cache = {}

    def trunk(self, prefix):
        key = ("t",) + tuple(prefix)
        if key not in self._cache:
            rng = np.random.default_rng([self.seed, 1] + list(prefix))
            self._cache[key] = rng.standard_normal(self.V) * self.scale
        return self._cache[key]

    def draft(self, prefix):
        key = ("d",) + tuple(prefix)
        if key not in self._cache:
            rng = np.random.default_rng([self.seed, 2] + list(prefix))
            self._cache[key] = self.trunk(prefix)[: self.Vd] + \
                rng.standard_normal(self.Vd) * self.noise
        return self._cache[key]


class _Need(Exception):
    def __init__(self, slot):
        super().__init__()
        self.slot = slot


def _run(model, prefix, drafts, T, eos, fixed, pos_base, one_hot=False):
    k = len(drafts)

    def uni(pos, purpose):
        s = (pos, purpose)
        if s in fixed:
            return fixed[s] / GRID
        raise _Need(s)

    z = np.array([model.trunk(prefix + list(drafts[:r])) for r in range(k + 1)])
    y = None if one_hot else (
        np.array([model.draft(prefix + list(drafts[: i - 1])) for i in range(1, k + 1)])
        if k else np.zeros((0, model.Vd)))
    try:
        r = accept.accept_request(z, y, list(drafts), k, T, eos, uni, pos_base)
        assert r["status"] == 0
        return ("done", tuple(r["tokens"]))
    except _Need as e:
        return ("need", e.slot)


def _partition(f, lo, hi):
    """Maximal intervals of [lo, hi] where f is constant, for f taking each value on a single
    interval (true for a ratio test and for an inverse-CDF draw as functions of u)."""
    out = []
    a, fa = lo, f(lo)
    while True:
        if f(hi) == fa:
            out.append((a, hi))
            return out
        l, r = a, hi
        while r - l > 1:
            mid = (l + r) // 2
            if f(mid) == fa:
                l = mid
            else:
                r = mid
        out.append((a, l))
        a, fa = r, f(r)


def _cycle_law(model, prefix, drafts, T, eos, pos_base, one_hot=False):
    """Exact law of the emitted block for fixed drafts, over the 24-bit uniform grid."""
    memo = {}

    def run(fixed):
        key = tuple(sorted(fixed.items()))
        if key not in memo:
            memo[key] = _run(model, prefix, drafts, T, eos, fixed, pos_base, one_hot)
        return memo[key]

    def law(fixed):
        kind, val = run(fixed)
        if kind == "done":
            return {val: 1.0}
        slot = val
        out = {}
        for a, b in _partition(lambda n: run({**fixed, slot: n}), 0, GRID - 1):
            w = (b - a + 1) / GRID
            for toks, pr in law({**fixed, slot: a}).items():
                out[toks] = out.get(toks, 0.0) + w * pr
        return out

    return law({})


def _extend(model, prefix, toks, J, T):
    """Distribution over length-J sequences that continue ``toks`` with exact trunk sampling."""
    out = {}
    need = J - len(toks)
    if need <= 0:
        return {tuple(toks[:J]): 1.0}
    for cont in itertools.product(range(model.V), repeat=need):
        pr = 1.0
        seq = list(toks)
        for t in cont:
            pr *= special.softmax(model.trunk(prefix + seq) / T)[t]
            seq.append(t)
        out[tuple(seq)] = pr
    return out


def _target_law(model, prefix, J, T):
    return _extend(model, prefix, [], J, T)


def _speculative_law(model, prefix, k, T, eos, pos_base, one_hot=False):
    J = k + 1
    total = {}
    if one_hot:  # deterministic drafts: argmax of the draft head, q = one-hot
        d = []
        for i in range(k):
            d.append(int(np.argmax(model.draft(prefix + d))))
        draft_seqs = [(tuple(d), 1.0)]
    else:
        draft_seqs = []
        for d in itertools.product(range(model.Vd), repeat=k):
            w = 1.0
            for i in range(k):
                w *= special.softmax(model.draft(prefix + list(d[:i])) / T)[d[i]]
            draft_seqs.append((d, w))
    for d, w in draft_seqs:
        for toks, pr in _cycle_law(model, prefix, d, T, eos, pos_base, one_hot).items():
            for seq, pe in _extend(model, prefix, list(toks), J, T).items():
                total[seq] = total.get(seq, 0.0) + w * pr * pe
    return total


@pytest.mark.parametrize("V,Vd,k,T,eos,one_hot", [
    (8, 6, 2, 1.0, -1, False),
    (8, 4, 3, 0.7, 2, False),
    (8, 8, 2, 1.3, 5, False),
    (8, 8, 3, 1.0, -1, True),
])
def test_brute_force_law_equals_target(V, Vd, k, T, eos, one_hot):
    model = ToyModel(V, Vd, scale=1.2, noise=0.9, seed=V * 100 + Vd * 10 + k)
    prefix = [1]
    spec = _speculative_law(model, prefix, k, T, eos, pos_base=40, one_hot=one_hot)
    target = _target_law(model, prefix, k + 1, T)
    assert set(spec) <= set(target)
    assert abs(sum(spec.values()) - 1.0) < 1e-9
    err = max(abs(spec.get(s, 0.0) - p) for s, p in target.items())
    # each decision on a path is quantised to the 24-bit grid: at most (k+1) cells of 2^-24
    assert err <= (k + 1) * 2.0**-24 + 1e-12, err


def test_draft_sampler_law_is_q():
    rng = np.random.default_rng(5)
    y = rng.standard_normal(7) * 1.5
    for T in (0.5, 1.0):
        memo = {}

        def f(n):
            if n not in memo:
                memo[n] = accept.draft_token(y, T, n / GRID)[0]
            return memo[n]

        law = np.zeros(7)
        for a, b in _partition(f, 0, GRID - 1):
            law[f(a)] += (b - a + 1) / GRID
        assert np.max(np.abs(law - special.softmax(y / T))) <= 2.0**-24 + 1e-15


def test_p_equals_q_accepts_every_draft():
    rng = np.random.default_rng(6)
    V, k = 50, 5
    z = rng.standard_normal((k + 1, V))
    y = z[:k].copy()  # draft head == trunk over all rows
    for seed in range(50):
        u = philox.make_uniform_source(seed)
        d, _ = accept.draft_chain_tokens(y, 1.0, u, pos_base=10)
        r = accept.accept_request(z, y, d, k, 1.0, -1, u, pos_base=10)
        assert r["n_accept"] == k and r["n_emit"] == k + 1 and r["tokens"][:k] == d
        assert r["sample_kind"] == 2 and r["sample_row"] == k


def test_one_hot_q_on_impossible_token_rejects_and_resamples_p():
    z = np.array([[0.3, -np.inf, 1.0, 0.2, -0.5], [0.0] * 5])
    x = 1  # p(x) == 0
    memo = {}

    def f(n):
        if n not in memo:
            def uni(pos, purpose, n=n):
                return n / GRID if purpose == philox.PURPOSE_RESIDUAL else 0.0
            r = accept.accept_request(z, None, [x], 1, 1.0, -1, uni, pos_base=0)
            assert r["n_accept"] == 0 and r["sample_kind"] == 1 and r["n_emit"] == 1
            memo[n] = r["tokens"][0]
        return memo[n]

    law = np.zeros(5)
    for a, b in _partition(f, 0, GRID - 1):
        law[f(a)] += (b - a + 1) / GRID
    assert law[1] == 0.0
    assert np.max(np.abs(law - lmhead.probs(z[0], 1.0))) <= 2.0**-24


def test_greedy_identical_to_mtp_off():
    """T = 0: speculative output == sequential greedy decoding, for several k and an EOS id."""
    for k, eos in ((1, 22), (3, 6), (7, 16)):  # EOS ids first produced after ~120 tokens
        model = ToyModel(64, 48, scale=2.0, noise=0.8, seed=k)
        ref = [0]
        while len(ref) < 150:
            t = int(np.argmax(model.trunk(ref)))
            ref.append(t)
            if t == eos:
                break
        seq = [0]
        accepted = rejected = 0
        while len(seq) < len(ref):
            d = []
            for i in range(k):
                d.append(accept.draft_token(model.draft(seq + d), 0.0)[0])
            z = np.array([model.trunk(seq + d[:r]) for r in range(k + 1)])
            r = accept.accept_request(z, None, d, k, 0.0, eos, None, pos_base=len(seq))
            assert r["status"] == 0 and 1 <= r["n_emit"] <= k + 1
            accepted += r["n_accept"]
            rejected += int(r["n_accept"] < k and not r["eos_hit"])
            seq.extend(r["tokens"])
            if r["eos_hit"]:
                break
        assert seq[: len(ref)] == ref
        assert accepted > 0 and rejected > 0  # both branches exercised


def _sequential_sample(model, T, seed, n, eos):
    """Decoding without drafts, written here from the definition: at absolute position pos the
    token is the smallest j with cumsum(p)[j] > u * sum(p), p = softmax(trunk(prefix) / T),
    u = U(seed, pos, BONUS). Independent of the oracle's helpers (own softmax and search)."""
    seq = [0]
    while len(seq) < n:
        z = model.trunk(seq) / T
        w = np.exp(z - z.max())
        c = np.cumsum(w)
        u = philox.uniform(seed, len(seq), philox.PURPOSE_BONUS)
        j = int(np.searchsorted(c, u * c[-1], side="right"))
        # distance to the nearest bin edge, relative to the mass: near-ties are reported
        lo = c[j - 1] if j > 0 else 0.0
        near = min(abs(c[j] - u * c[-1]), abs(u * c[-1] - lo)) / c[-1] < 1e-12
        seq.append(j)
        if near:
            return seq, True
        if j == eos:
            break
    return seq, False


@pytest.mark.parametrize("k,T,seed", [(1, 1.0, 3), (3, 0.7, 4), (7, 1.0, 5), (7, 1.6, 6)])
def test_exact_match_at_temperature_equals_sampling_without_drafts(k, T, seed):
    """NEXT item F1 (lucebox-hub PR #15, *Exactness* / *Notes*): with exact-match acceptance the
    emitted tokens equal, token for token, decoding without drafts under the same seed -- for
    drafts from a noisy draft head, so both keeps and mismatches occur."""
    eos = 5
    model = ToyModel(32, 24, scale=3.0, noise=0.2, seed=10 + k)
    ref, near = _sequential_sample(model, T, seed, 200, eos)
    assert not near
    src = philox.make_uniform_source(seed)
    seq = [0]
    kept = mism = 0
    while len(seq) < len(ref):
        d = []
        for i in range(k):  # drafts: the draft head's own samples (DRAFT purpose)
            u = src(len(seq) + i, philox.PURPOSE_DRAFT)
            d.append(accept.draft_token(model.draft(seq + d), T, u)[0])
        z = np.array([model.trunk(seq + d[:r]) for r in range(k + 1)])
        r = accept.accept_request_exact(z, d, k, T, eos, src, pos_base=len(seq))
        assert r["status"] == 0 and 1 <= r["n_emit"] <= k + 1 and r["sample_kind"] == 3
        kept += r["n_accept"]
        mism += int(r["n_accept"] < k and not r["eos_hit"])
        seq.extend(r["tokens"])
        if r["eos_hit"]:
            break
    assert seq[: len(ref)] == ref[: len(seq)]
    assert kept > 0 and mism > 0


def test_exact_match_at_zero_temperature_is_greedy_acceptance():
    rng = np.random.default_rng(8)
    src = philox.make_uniform_source(1)
    for trial in range(50):
        k = int(rng.integers(0, 8))
        z = rng.standard_normal((k + 1, 64))
        d = [int(x) for x in rng.integers(0, 64, k)]
        for i in range(k):  # plant some agreements
            if rng.random() < 0.6:
                d[i] = int(np.argmax(z[i]))
        a = accept.accept_request(z, None, d, k, 0.0, 7, src, 100)
        b = accept.accept_request_exact(z, d, k, 0.0, 7, src, 100)
        assert a == b


def test_exact_match_validation_and_eos():
    src = philox.make_uniform_source(2)
    z = np.zeros((3, 16))
    assert accept.accept_request_exact(z, [1, 2], 9, 1.0, 0, src, 0)["status"] == 2
    assert accept.accept_request_exact(z, [1, 99], 2, 1.0, 0, src, 0)["status"] == 5
    bad = z.copy()
    bad[1, 3] = np.nan
    assert accept.accept_request_exact(bad, [1, 2], 2, 1.0, 0, src, 0)["status"] == 1
    # a row whose whole mass sits on the EOS id: the trunk samples EOS, a matching draft is
    # kept and ends the block with no bonus
    z = np.full((3, 16), -50.0)
    z[0, 4] = 50.0
    r = accept.accept_request_exact(z, [4, 9], 2, 1.0, 4, src, 0)
    assert r["tokens"] == [4] and r["eos_hit"] and r["n_accept"] == 1 and r["n_emit"] == 1


def test_eos_at_every_draft_position():
    rng = np.random.default_rng(8)
    V, k, eos = 30, 5, 3
    z = rng.standard_normal((k + 1, V))
    for pos in range(1, k + 1):
        d = [int(np.argmax(z[i])) for i in range(k)]
        d[pos - 1] = eos
        z2 = z.copy()
        z2[pos - 1, eos] = z2[pos - 1].max() + 1.0  # the trunk agrees with the EOS draft
        r = accept.accept_request(z2, None, d, k, 0.0, eos, None, pos_base=0)
        assert r["eos_hit"] and r["n_accept"] == pos and r["n_emit"] == pos
        assert r["tokens"][-1] == eos and r["sample_kind"] == 0
        # at temperature with p == one-hot-q the EOS draft is accepted too (u*1 <= p(eos)~1)
        z3 = np.full((k + 1, V), -np.inf)
        for i in range(k + 1):
            z3[i, d[i] if i < k else 0] = 0.0
        r = accept.accept_request(z3, None, d, k, 1.0, eos, philox.make_uniform_source(1), 0)
        assert r["eos_hit"] and r["n_emit"] == pos and r["tokens"] == d[:pos]


def test_status_codes_and_k_zero():
    rng = np.random.default_rng(9)
    z = rng.standard_normal((4, 20))
    u = philox.make_uniform_source(0)
    assert accept.accept_request(z, None, [1, 2, 3], 8, 0.0, -1, u, 0)["status"] == 2
    assert accept.accept_request(z, None, [1, 2, 3], -1, 0.0, -1, u, 0)["status"] == 2
    assert accept.accept_request(z, None, [1, 20, 3], 3, 0.0, -1, u, 0)["status"] == 5
    for bad in (np.nan, np.inf):
        zb = z.copy()
        zb[2, 7] = bad
        r = accept.accept_request(zb, None, [1, 2, 3], 3, 1.0, -1, u, 0)
        assert r["status"] == 1 and r["n_emit"] == 0 and r["tokens"] == []
    zb = z.copy()
    zb[1] = -np.inf
    assert accept.accept_request(zb, None, [1, 2, 3], 3, 0.0, -1, u, 0)["status"] == 1
    # k = 0 is MTP off: one token from row 0 (argmax at T=0, BONUS draw at T>0)
    r = accept.accept_request(z, None, [], 0, 0.0, -1, u, 5)
    assert r["tokens"] == [int(np.argmax(z[0]))] and r["n_accept"] == 0
    r = accept.accept_request(z, None, [], 0, 1.0, -1, u, 5)
    j, _ = accept.inverse_cdf(lmhead.probs(z[0], 1.0), u(5, philox.PURPOSE_BONUS))
    assert r["tokens"] == [j] and r["sample_kind"] == 2


def test_inverse_cdf_edges():
    w = np.array([0.0, 0.25, 0.0, 0.75])
    assert accept.inverse_cdf(w, 0.0)[0] == 1       # smallest j with cum > 0 skips zero bins
    assert accept.inverse_cdf(w, 0.25)[0] == 3      # strict '>' at a boundary
    assert accept.inverse_cdf(w, 1 - 2**-24)[0] == 3
    assert accept.inverse_cdf(w, 0.1)[1] == pytest.approx(0.1)


# ---------------------------------------------------------------- chi-square at V = 4096

def _chi_rows():
    from synth import configs, gen
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    rng = np.random.default_rng([0, 0xC41])
    H = gen.encode(rng.standard_normal((2, cfg.d), dtype=np.float32), cfg.wdtype)
    Hd = gen.noisy_rows(gen.as_f32(H[:1]), cfg.draft_noise, cfg.wdtype, rng)
    z = lmhead.logits(W, H)
    y = lmhead.logits(W, Hd, rows=cfg.Vd)
    return z, y


def _chi_worker(args):
    lo, hi = args
    z, y = _chi_rows()
    T = 1.0
    pos = np.arange(lo, hi, dtype=np.int64) * 16
    ud = philox.uniform_np(0, pos, philox.PURPOSE_DRAFT)
    ua = philox.uniform_np(0, pos, philox.PURPOSE_ACCEPT)
    ur = philox.uniform_np(0, pos, philox.PURPOSE_RESIDUAL)
    ub = philox.uniform_np(0, pos + 1, philox.PURPOSE_BONUS)
    first, second = [], []
    for n in range(hi - lo):
        table = {philox.PURPOSE_ACCEPT: ua[n], philox.PURPOSE_RESIDUAL: ur[n],
                 philox.PURPOSE_BONUS: ub[n]}
        d, _ = accept.draft_token(y[0], T, ud[n])
        r = accept.accept_request(z, y, [d], 1, T, -1, lambda p, q: table[q], int(pos[n]))
        first.append(r["tokens"][0])
        second.append(r["tokens"][1] if r["n_accept"] == 1 else -1)
    return np.array(first), np.array(second)


def _chi_test(counts, p):
    exp = p * counts.sum()
    order = np.argsort(exp)
    obs_m, exp_m, acc_o, acc_e = [], [], 0.0, 0.0
    for j in order:  # merge the smallest bins until every expected count is >= 5
        acc_o += counts[j]
        acc_e += exp[j]
        if acc_e >= 5:
            obs_m.append(acc_o)
            exp_m.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        obs_m[-1] += acc_o
        exp_m[-1] += acc_e
    return stats.chisquare(obs_m, exp_m).pvalue


@pytest.mark.slow
def test_chi_square_1e6_cycles_at_v4096():
    n = 1_000_000
    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    chunks = [(i * n // (4 * workers), (i + 1) * n // (4 * workers)) for i in range(4 * workers)]
    with mp.get_context("spawn").Pool(workers) as pool:
        parts = pool.map(_chi_worker, chunks)
    first = np.concatenate([p[0] for p in parts])
    second = np.concatenate([p[1] for p in parts])
    z, _ = _chi_rows()
    p0, p1 = lmhead.probs(z[0], 1.0), lmhead.probs(z[1], 1.0)
    assert _chi_test(np.bincount(first, minlength=p0.size), p0) > 1e-3
    sec = second[second >= 0]
    assert sec.size > 100_000
    assert _chi_test(np.bincount(sec, minlength=p1.size), p1) > 1e-3
