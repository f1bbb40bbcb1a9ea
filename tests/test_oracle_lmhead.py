"""Pins for the oracle's logits and row statistics (CPU only)."""

import numpy as np
import pytest
from scipy import special

from oracle import lmhead
from synth import gen


def test_bf16_widening_is_exact():
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4049, 0x7F80, 0xFF80, 0x0001], np.uint16)
    ref = [0.0, -0.0, 1.0, -1.0, 3.140625, np.inf, -np.inf, 2.0**-133]
    out = lmhead.bf16_to_f64(bits)
    assert list(out) == ref
    assert np.signbit(out[1])


@pytest.mark.parametrize("enc", ["bf16", "f32"])
def test_logits_equal_exact_integer_dot_products(enc):
    # small integers are exact in bf16 and fp32; the exact dot product is Python-int arithmetic
    rng = np.random.default_rng(0)
    V, d, R = 37, 48, 3
    Wi = rng.integers(-8, 9, (V, d))
    Hi = rng.integers(-8, 9, (R, d))
    W = gen.encode(Wi.astype(np.float32), enc)
    H = gen.encode(Hi.astype(np.float32), enc)
    z = lmhead.logits(W, H)
    for r in range(R):
        for v in range(V):
            assert z[r, v] == sum(int(a) * int(b) for a, b in zip(Wi[v], Hi[r]))
    assert np.array_equal(lmhead.logits(W, H, rows=10), z[:, :10])
    assert lmhead.logit(W, H[1], 5) == z[1, 5]


def test_logits_scaled_powers_of_two_exact():
    # bf16 values k * 2^-e keep the products exact; the float64 sum of d such terms is exact
    rng = np.random.default_rng(1)
    V, d = 20, 64
    Wi = rng.integers(-100, 101, (V, d))
    Hi = rng.integers(-100, 101, (1, d))
    W = gen.encode((Wi * 2.0**-7).astype(np.float32), "bf16")
    H = gen.encode((Hi * 2.0**-3).astype(np.float32), "bf16")
    z = lmhead.logits(W, H)[0]
    exact = (Wi @ Hi[0]).astype(np.float64) * 2.0**-10
    assert np.array_equal(z, exact)


def test_row_stats_against_library_and_brute_force():
    rng = np.random.default_rng(2)
    for T in (0.0, 0.5, 1.0, 2.0):
        z = rng.standard_normal(1000) * 3
        st = lmhead.row_stats(z, T)
        Teff = T if T > 0 else 1.0
        assert st["max"] == z.max()
        assert st["argmax"] == int(np.argmax(z))
        assert st["gap"] == z.max() - np.sort(z)[-2]
        assert np.isclose(st["log_norm"], special.logsumexp(z / Teff) - z.max() / Teff,
                          rtol=0, atol=1e-12)
        if T > 0:
            assert np.allclose(lmhead.probs(z, T), special.softmax(z / T), rtol=1e-12, atol=0)


def test_row_stats_closed_forms():
    st = lmhead.row_stats(np.full(16, 0.25), 1.0)  # constant row
    assert st["argmax"] == 0 and st["gap"] == 0.0
    assert np.isclose(st["log_norm"], np.log(16), rtol=0, atol=1e-15)
    z = np.full(8, -np.inf)
    z[5] = 1.5  # one-hot: all other tokens impossible
    st = lmhead.row_stats(z, 0.7)
    assert st["argmax"] == 5 and st["log_norm"] == 0.0 and st["gap"] == np.inf
    assert list(lmhead.probs(z, 0.7)) == [0, 0, 0, 0, 0, 1.0, 0, 0]
    # ties: lowest index wins, gap zero
    st = lmhead.row_stats(np.array([0.0, 3.0, 1.0, 3.0]), 0.0)
    assert st["argmax"] == 1 and st["gap"] == 0.0
    # temperature scaling: log_norm at T equals log sum exp((z-max)/T)
    z = np.array([0.0, 1.0, 2.0])
    st = lmhead.row_stats(z, 2.0)
    assert np.isclose(st["log_norm"], np.log(np.exp(-1.0) + np.exp(-0.5) + 1.0), atol=1e-15)


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_nonfinite_rows_flagged(bad):
    z = np.zeros(10)
    z[3] = bad
    assert lmhead.row_stats(z, 1.0)["nonfinite"]
    assert lmhead.row_stats(np.full(4, -np.inf), 1.0)["nonfinite"]
    z = np.zeros(10)
    z[3] = -np.inf  # -inf alone is allowed: probability zero
    st = lmhead.row_stats(z, 1.0)
    assert not st["nonfinite"] and lmhead.probs(z, 1.0)[3] == 0.0


def test_fp32_bound_covers_fp32_accumulation():
    # sequential fp32 accumulation of bf16 products stays inside the stated bound
    rng = np.random.default_rng(3)
    W = gen.f32_to_bf16(rng.standard_normal((50, 2560)).astype(np.float32) * 0.02)
    H = gen.f32_to_bf16(rng.standard_normal((2, 2560)).astype(np.float32))
    z = lmhead.logits(W, H)
    bound = lmhead.fp32_abs_bound(W, H)
    Wf, Hf = gen.bf16_to_f32(W), gen.bf16_to_f32(H)
    for r in range(2):
        for v in range(50):
            acc = np.float32(0)
            for j in range(0, 2560, 1):
                acc = np.float32(acc + np.float32(Wf[v, j] * Hf[r, j]))
            assert abs(float(acc) - z[r, v]) <= bound[r, v]
