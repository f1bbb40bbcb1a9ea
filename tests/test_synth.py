"""The seeded input generators (`synth/`) shared by the oracle tests, the GPU parity tests and the
benchmark: the same seed gives the same bytes, different seeds differ, and the inputs follow
the recipe the design notes state (weights ~ N(0, 0.02^2); planted targets drawn from the draft
rows with probability pi; draft rows = verify row i-1 plus N(0, sigma^2); EOS injected in the
stated share of cycles; bf16 encoding rounds to nearest even)."""

import numpy as np
import pytest

from synth import configs, gen

C0 = configs.get(0)


def test_same_seed_same_bytes_and_seeds_differ():
    a = gen.lm_weights(C0, seed=3, cache=False)
    b = gen.lm_weights(C0, seed=3, cache=False)
    c = gen.lm_weights(C0, seed=4, cache=False)
    assert a.tobytes() == b.tobytes() and a.tobytes() != c.tobytes()
    x = gen.cycle_inputs(C0, a, 5, seed=1)
    y = gen.cycle_inputs(C0, a, 5, seed=1)
    z = gen.cycle_inputs(C0, a, 6, seed=1)
    assert x["H"].tobytes() == y["H"].tobytes() and x["Hd"].tobytes() == y["Hd"].tobytes()
    assert x["H"].tobytes() != z["H"].tobytes()
    q1 = gen.q4_weights(C0, seed=3, cache=False)
    q2 = gen.q4_weights(C0, seed=3, cache=False)
    assert q1.tobytes() == q2.tobytes()


def test_weight_distribution():
    W = gen.lm_weights(C0, cache=False).astype(np.float64)
    assert W.shape == (C0.V, C0.d)
    assert abs(W.mean()) < 1e-3 and abs(W.std() - gen.W_STD) < 2e-4


def test_bf16_encoding_rounds_to_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: ties go to the even one (1)
    x = np.array([1.0, 1 + 2.0**-8, 1 + 3 * 2.0**-8, -2.5, np.inf, np.nan], dtype=np.float32)
    bits = gen.f32_to_bf16(x)
    assert list(bits[:5]) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F80]
    assert bits[5] == 0x7FC0
    assert np.array_equal(gen.bf16_to_f32(bits[:5]), np.array([1.0, 1.0, 1 + 2.0**-6, -2.5,
                                                                np.inf], dtype=np.float32))


def test_planted_targets_follow_the_recipe():
    cfg = configs.Config(name="t", d=64, V=2000, Vd=500, wdtype="bf16", k=3, k_mode="fixed",
                         batch=1, rows_per_request=4, temps=(1.0,), cycles=1, seeds=(0,),
                         plant_scale=8.0, pi_draft=0.8, draft_noise=0.3)
    W = gen.lm_weights(cfg, cache=False)
    rng = np.random.default_rng(0)
    _, H32, t = gen.planted_rows(cfg, W, 4000, rng)
    assert ((t >= 0) & (t < cfg.V)).all()
    assert abs(np.mean(t < cfg.Vd) - cfg.pi_draft) < 0.03
    # the planted direction makes the target the row's argmax far more often than chance
    # (1/V = 0.0005; ~0.76 at this toy size, ~0.8 at the full-size greedy workload)
    z = H32.astype(np.float64) @ gen.as_f32(W).astype(np.float64).T
    assert np.mean(np.argmax(z, axis=1) == t) > 0.6


def test_draft_rows_are_noisy_verify_rows():
    W = gen.lm_weights(C0)
    inp = gen.cycle_inputs(C0, W, 0, seed=2)
    k = inp["k"]
    assert inp["H"].shape == (k + 1, C0.d) and inp["Hd"].shape == (k, C0.d)
    diff = gen.as_f32(inp["Hd"]) - gen.as_f32(inp["H"][:k])
    assert abs(diff.std() - C0.draft_noise) < 0.05


@pytest.mark.parametrize("idx", [2])
def test_eos_injection_share(idx):
    cfg = configs.get(idx)
    pos = [gen.eos_injection(cfg, c, cfg.k) for c in range(4000)]
    share = np.mean([p > 0 for p in pos])
    assert abs(share - cfg.eos_inject) < 0.015
    assert all(0 <= p <= cfg.k for p in pos)


def test_q4_generator_codes_in_range_and_groups_span_their_values():
    from oracle import quant
    d = 128
    packed = gen.q4_quantise(gen.lm_weights(configs.Config(
        name="q", d=d, V=64, Vd=64, wdtype="bf16", k=1, k_mode="fixed", batch=1,
        rows_per_request=2, temps=(0.0,), cycles=1, seeds=(0,), plant_scale=0.0, pi_draft=0.0,
        draft_noise=0.5), cache=False))
    assert packed.shape == (64, 5 * d // 8)
    q = quant.unpack_codes(packed[:, :d // 2], d)
    assert q.min() >= 0 and q.max() <= 15
    # min/max quantisation: every group uses code 0 and code 15
    g = q.reshape(q.shape[0], -1, 32)
    assert (g.min(axis=2) == 0).all() and (g.max(axis=2) == 15).all()
