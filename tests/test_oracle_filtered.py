"""Pins of the oracle's top-k / top-p filtered acceptance (``accept.filtered_probs`` and
``accept.accept_request_filtered``) against what does not depend on them: a characterisation
of the top-k set checked over every subset, hand-computed cases, the reduction to the unfiltered
ratio rule with one-hot q when nothing is filtered, greedy acceptance at T = 0, and the exact law
of the emitted block (every cell of the 24-bit uniforms) against sequential sampling from the
filtered target (llama.cpp PR #28104, *Result*: temperature 1.0, top-p 0.95, top-k 20)."""

import itertools

import numpy as np
import pytest
from scipy import special

from oracle import accept, philox
from test_oracle_accept import GRID, ToyModel, _partition, _Need


def test_hand_cases():
    z = np.array([3.0, 1.0, 2.0, 0.0])
    p, kept, _ = accept.filtered_probs(z, 1.0, 2, 1.0)
    e3, e2 = np.exp(3.0), np.exp(2.0)
    assert list(kept) == [0, 2]
    assert np.allclose(p, [e3 / (e3 + e2), 0, e2 / (e3 + e2), 0], rtol=1e-15)
    # top-p 0.5: token 0 alone carries 0.73 of the top-2 mass
    p, kept, _ = accept.filtered_probs(z, 1.0, 2, 0.5)
    assert list(kept) == [0] and p[0] == 1.0
    # top-p 0.75 needs the second token too (0.731 < 0.75)
    p, kept, _ = accept.filtered_probs(z, 1.0, 4, 0.75)
    assert list(kept) == [0, 2]
    # ties at the cut keep the lower ids
    p, kept, _ = accept.filtered_probs(np.array([1.0, 2.0, 1.0, 1.0]), 1.0, 2, 1.0)
    assert list(kept) == [1, 0]
    # top-k 1 is the argmax, whatever top-p
    p, kept, _ = accept.filtered_probs(z, 0.3, 1, 0.99)
    assert list(kept) == [0] and p[0] == 1.0


@pytest.mark.parametrize("seed", range(6))
def test_top_k_set_characterisation(seed):
    """The kept set under top_p = 1 is the unique set of size min(k, V) in which every token
    beats every token outside it (larger logit, or equal logit and lower id): checked against
    every subset of that size."""
    rng = np.random.default_rng(seed)
    V = 7
    z = rng.integers(-2, 3, V).astype(np.float64)  # small integers: many ties
    for k in range(1, V + 1):
        _, kept, _ = accept.filtered_probs(z, 1.0, k, 1.0)

        def beats(a, b):
            return z[a] > z[b] or (z[a] == z[b] and a < b)

        good = [set(S) for S in itertools.combinations(range(V), k)
                if all(beats(a, b) for a in S for b in range(V) if b not in S)]
        assert good == [set(int(x) for x in kept)]


@pytest.mark.parametrize("seed", range(5))
def test_nothing_filtered_is_the_softmax_and_the_one_hot_ratio_rule(seed):
    rng = np.random.default_rng(seed)
    V, k, T = 50, 3, 0.8
    z = rng.standard_normal((k + 1, V)) * 2
    p, _, _ = accept.filtered_probs(z[0], T, V, 1.0)
    assert np.allclose(p, special.softmax(z[0] / T), rtol=1e-12, atol=1e-15)
    for trial in range(20):
        drafts = list(rng.integers(0, V, k))
        uni = philox.make_uniform_source(100 + trial)
        a = accept.accept_request_filtered(z, drafts, k, T, V, 1.0, -1, uni, 7 * trial)
        b = accept.accept_request(z, None, drafts, k, T, -1, uni, 7 * trial)
        assert a["tokens"] == b["tokens"] and a["n_accept"] == b["n_accept"]


def test_greedy_ignores_the_filters():
    rng = np.random.default_rng(9)
    z = rng.standard_normal((4, 30))
    uni = philox.make_uniform_source(1)
    for drafts in ([3, 4, 5], [int(np.argmax(z[0])), 1, 2]):
        a = accept.accept_request_filtered(z, drafts, 3, 0.0, 2, 0.5, -1, uni, 0)
        b = accept.accept_request(z, None, drafts, 3, 0.0, -1, uni, 0)
        assert a == b


def _filtered_law_of_block(model, prefix, k, T, top_k, top_p, eos, pos_base):
    """Exact law of the emitted block over the 24-bit uniform grid, argmax drafts."""
    d = []
    for _ in range(k):
        d.append(int(np.argmax(model.draft(prefix + d))))
    z = np.array([model.trunk(prefix + d[:r]) for r in range(k + 1)])
    memo = {}

    def run(fixed):
        key = tuple(sorted(fixed.items()))
        if key not in memo:
            def uni(pos, purpose):
                if (pos, purpose) in fixed:
                    return fixed[(pos, purpose)] / GRID
                raise _Need((pos, purpose))
            try:
                r = accept.accept_request_filtered(z, d, k, T, top_k, top_p, eos, uni, pos_base)
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


def _filtered_target(model, prefix, toks, J, T, top_k, top_p, eos):
    """Sequential sampling from the filtered target: the law of the first J tokens (stopping at
    an EOS), given the tokens already emitted. The filter here is written from its definition:
    sort by (logit desc, id asc), cut at top_k, then keep while the mass ahead is below top_p."""
    if len(toks) >= J or (toks and toks[-1] == eos):
        return {tuple(toks): 1.0}
    zr = model.trunk(prefix + list(toks))
    ranked = sorted(range(model.V), key=lambda t: (-zr[t], t))[:top_k]
    w = [np.exp((zr[t] - zr[ranked[0]]) / T) for t in ranked]
    tot, ahead, keep = sum(w), 0.0, []
    for t, wt in zip(ranked, w):
        if ahead < top_p:
            keep.append((t, wt))
        ahead += wt / tot
    s = sum(wt for _, wt in keep)
    out = {}
    for t, wt in keep:
        for seq, pr in _filtered_target(model, prefix, list(toks) + [t], J, T, top_k, top_p,
                                        eos).items():
            out[seq] = out.get(seq, 0.0) + wt / s * pr
    return out


@pytest.mark.parametrize("V,k,T,top_k,top_p,eos", [
    (8, 2, 1.0, 4, 0.9, -1),
    (8, 3, 0.7, 3, 0.95, 2),
    (8, 2, 1.3, 8, 0.6, -1),
    (8, 3, 1.0, 2, 1.0, 5),
])
def test_emitted_law_is_the_filtered_target(V, k, T, top_k, top_p, eos):
    """The block the speculative cycle emits, continued by sequential filtered sampling to k+1
    tokens, has the law of k+1 tokens sampled sequentially from the filtered target."""
    model = ToyModel(V, V, scale=1.3, noise=0.8, seed=V * 7 + k + top_k)
    prefix = [2]
    J = k + 1
    spec = {}
    for toks, pr in _filtered_law_of_block(model, prefix, k, T, top_k, top_p, eos, 30).items():
        for seq, pe in _filtered_target(model, prefix, list(toks), J, T, top_k, top_p,
                                        eos).items():
            spec[seq] = spec.get(seq, 0.0) + pr * pe
    target = _filtered_target(model, prefix, [], J, T, top_k, top_p, eos)
    assert set(spec) <= set(target)
    err = max(abs(spec.get(s, 0.0) - p) for s, p in target.items())
    assert err <= (k + 1) * 2.0**-24 + 1e-12, err


def test_planted_mistakes_fail(monkeypatch):
    """A top-p cut that keeps one token too many breaks the emitted law; top-k ties broken to the
    higher id break the characterisation."""
    real = accept.filtered_probs

    def one_too_many(z, T, top_k, top_p):
        p, kept, m = real(z, T, top_k, top_p)
        order = np.lexsort((np.arange(z.shape[0]), -z))[:min(top_k, z.shape[0])]
        if len(kept) < len(order):
            kept = order[:len(kept) + 1]
            w = np.exp((z[kept] - z[kept[0]]) / T)
            p = np.zeros(z.shape[0])
            p[kept] = w / w.sum()
        return p, kept, m

    monkeypatch.setattr(accept, "filtered_probs", one_too_many)
    with pytest.raises(AssertionError):
        test_emitted_law_is_the_filtered_target(8, 2, 1.0, 4, 0.6, -1)
    monkeypatch.setattr(accept, "filtered_probs", real)

    def high_ties(z, T, top_k, top_p):
        zz = np.asarray(z, dtype=np.float64)
        V = zz.shape[0]
        flip = real(zz[::-1].copy(), T, top_k, top_p)
        return flip[0][::-1], V - 1 - flip[1], flip[2]

    monkeypatch.setattr(accept, "filtered_probs", high_ties)
    with pytest.raises(AssertionError):
        for seed in range(6):
            test_top_k_set_characterisation(seed)
