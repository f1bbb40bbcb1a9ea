"""Pins for the oracle's Philox4x32-10 and its 24-bit uniforms (CPU only)."""

import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = line.split()
            assert int(w[0]) == 10
            vals = [int(x, 16) for x in w[1:]]
            rows.append((tuple(vals[0:4]), tuple(vals[4:6]), tuple(vals[6:10])))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat_rows())
def test_known_answer_vectors(ctr, key, expect):
    assert philox.philox4x32_10(ctr, key) == expect


@pytest.mark.parametrize("ctr,key,expect", _kat_rows())
def test_vectorised_matches_kat(ctr, key, expect):
    out = philox.philox4x32_10_np(*[np.array([c]) for c in ctr], np.array([key[0]]),
                                  np.array([key[1]]))
    assert tuple(int(o[0]) for o in out) == expect


def test_vectorised_matches_scalar_on_random_counters():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 2**32, (4, 200), dtype=np.uint64)
    k = rng.integers(0, 2**32, (2, 200), dtype=np.uint64)
    out = philox.philox4x32_10_np(c[0], c[1], c[2], c[3], k[0], k[1])
    for i in range(200):
        ref = philox.philox4x32_10(tuple(int(x) for x in c[:, i]), (int(k[0, i]), int(k[1, i])))
        assert tuple(int(o[i]) for o in out) == ref


def test_uniform_layout_and_range():
    # counter = (pos lo, pos hi, 0, purpose), key = (seed lo, seed hi), u = (w0 >> 8) / 2^24
    seed, pos = 0x0123456789ABCDEF, (5 << 32) | 77
    w0 = philox.philox4x32_10((77, 5, 0, philox.PURPOSE_RESIDUAL), (0x89ABCDEF, 0x01234567))[0]
    assert philox.uniform(seed, pos, philox.PURPOSE_RESIDUAL) == (w0 >> 8) / 2**24
    u = philox.uniform_np(seed, np.arange(1000) + pos, philox.PURPOSE_RESIDUAL)
    assert u[0] == philox.uniform(seed, pos, philox.PURPOSE_RESIDUAL)
    assert np.all(u >= 0) and np.all(u <= 1 - 2**-24)
    assert np.all(u * 2**24 == np.floor(u * 2**24))  # exactly 24-bit, representable in fp32
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_purposes_and_seeds_give_distinct_streams():
    pos = np.arange(4096)
    streams = [philox.uniform_np(s, pos, p) for s in (0, 1) for p in (1, 2, 3, 4)]
    for i in range(len(streams)):
        for j in range(i + 1, len(streams)):
            assert np.mean(streams[i] == streams[j]) < 0.01


def test_uniformity_chi_square():
    u = philox.uniform_np(0, np.arange(1_000_000), philox.PURPOSE_ACCEPT)
    counts = np.bincount((u * 256).astype(np.int64), minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-3
    # serial pairs (u_n, u_n+1) on an 16x16 grid
    pairs = (u[:-1] * 16).astype(np.int64) * 16 + (u[1:] * 16).astype(np.int64)
    assert stats.chisquare(np.bincount(pairs, minlength=256)).pvalue > 1e-3
