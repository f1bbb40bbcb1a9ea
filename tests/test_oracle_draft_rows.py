"""Pins of the draft set read as two row ranges (lucebox-hub PR #15, *What*: the draft head
covers the control and special tokens plus the lowest ids): the ids of the draft rows, the
reduction to the first-Vd case when the ranges touch, and the exact law of the emitted block
(every draft and every cell of the 24-bit uniforms at V = 8) against the target: the ratio rule
stays exact when q lives on a split subset of the vocabulary."""

import itertools

import numpy as np
import pytest
from scipy import special

from oracle import accept, philox
from test_oracle_accept import GRID, ToyModel, _Need, _extend, _partition, _target_law


def test_draft_rows_ids():
    assert list(accept.draft_rows(3, 6, 2)) == [0, 1, 2, 6, 7]
    assert list(accept.draft_rows(4, 4, 0)) == [0, 1, 2, 3]
    assert list(accept.draft_rows(0, 5, 3)) == [5, 6, 7]


def test_touching_ranges_are_the_first_vd_rows():
    rng = np.random.default_rng(0)
    V, Vd, k, T = 40, 25, 3, 0.9
    z = rng.standard_normal((k + 1, V))
    y = rng.standard_normal((k, Vd))
    rows = accept.draft_rows(10, 10, 15)
    for trial in range(30):
        uni = philox.make_uniform_source(trial)
        d1, _ = accept.draft_chain_tokens(y, T, uni, 5 * trial)
        d2, _ = accept.draft_chain_tokens(y, T, uni, 5 * trial, rows)
        assert d1 == d2
        a = accept.accept_request(z, y, d1, k, T, -1, uni, 5 * trial)
        b = accept.accept_request(z, y, d1, k, T, -1, uni, 5 * trial, rows=rows)
        assert a == b


class SplitModel(ToyModel):
    """The toy trunk, with a draft head over the vocabulary ids ``rows``."""

    def __init__(self, V, rows, scale, noise, seed):
        super().__init__(V, len(rows), scale, noise, seed)
        self.rows = np.asarray(rows)

    def draft(self, prefix):
        key = ("r",) + tuple(prefix)
        if key not in self._cache:
            rng = np.random.default_rng([self.seed, 3] + list(prefix))
            self._cache[key] = self.trunk(prefix)[self.rows] + \
                rng.standard_normal(self.Vd) * self.noise
        return self._cache[key]


def _block_law(model, prefix, drafts, T, eos, pos_base):
    k = len(drafts)
    z = np.array([model.trunk(prefix + list(drafts[:r])) for r in range(k + 1)])
    y = np.array([model.draft(prefix + list(drafts[:i])) for i in range(k)])
    memo = {}

    def run(fixed):
        key = tuple(sorted(fixed.items()))
        if key not in memo:
            def uni(pos, purpose):
                if (pos, purpose) in fixed:
                    return fixed[(pos, purpose)] / GRID
                raise _Need((pos, purpose))
            try:
                r = accept.accept_request(z, y, list(drafts), k, T, eos, uni, pos_base,
                                          rows=model.rows)
                memo[key] = ("done", tuple(r["tokens"]))
            except _Need as e:
                memo[key] = ("need", e.slot)
        return memo[key]

    def law(fixed):
        kind, val = run(fixed)
        if kind == "done":
            return {val: 1.0}
        out = {}
        for a, b in _partition(lambda n: run({**fixed, val: n}), 0, GRID - 1):
            for toks, pr in law({**fixed, val: a}).items():
                out[toks] = out.get(toks, 0.0) + (b - a + 1) / GRID * pr
        return out

    return law({})


@pytest.mark.parametrize("rows,k,T,eos", [([0, 1, 2, 6, 7], 2, 1.0, -1),
                                          ([0, 1, 5, 6, 7], 2, 0.7, 6),
                                          ([0, 7], 3, 1.2, -1)])
def test_law_with_a_split_draft_set_is_the_target(rows, k, T, eos):
    """Drafts sampled from q over the split set (draft row -> id through ``rows``)."""
    model = SplitModel(8, rows, scale=1.2, noise=0.9, seed=len(rows) * 11 + k)
    prefix = [3]
    J = k + 1
    total = {}
    for idx in itertools.product(range(len(rows)), repeat=k):
        d = [int(rows[i]) for i in idx]
        w = 1.0
        for i in range(k):
            w *= special.softmax(model.draft(prefix + d[:i]) / T)[idx[i]]
        for toks, pr in _block_law(model, prefix, d, T, eos, 50).items():
            for seq, pe in _extend(model, prefix, list(toks), J, T).items():
                total[seq] = total.get(seq, 0.0) + w * pr * pe
    target = _target_law(model, prefix, J, T)
    assert abs(sum(total.values()) - 1.0) < 1e-9
    err = max(abs(total.get(s, 0.0) - p) for s, p in target.items())
    assert err <= (k + 1) * 2.0**-24 + 1e-12, err


def test_planted_mistake_ignoring_the_map_breaks_the_law(monkeypatch):
    """q placed on the first Vd ids instead of the draft rows' ids fails the law."""
    real = accept.accept_request

    def first_vd(z, y, drafts, k, T, eos_id, uniform, pos_base, k_max=7, rows=None):
        return real(z, y, drafts, k, T, eos_id, uniform, pos_base, k_max)

    monkeypatch.setattr(accept, "accept_request", first_vd)
    with pytest.raises(AssertionError):
        test_law_with_a_split_draft_set_is_the_target([0, 1, 2, 6, 7], 2, 1.0, -1)
