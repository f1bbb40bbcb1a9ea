"""GPU parity of exact-match acceptance at temperature (spec_accept_exact, through the C ABI)
against the oracle's ``accept_request_exact`` (lucebox-hub PR #15, "Exactness" and "Notes": a
draft counts only if it is the trunk's own sample, so the output equals decoding without
drafts).

* C0 (d=256, V=4,096, fp32, k=3): 1,000 cycles at T = 1 and 500 at T = 0.05, drafts from the
  GPU draft head; emitted tokens, kept counts, EOS flags and draw kinds equal the oracle's exactly
  outside near-tie cycles (a CDF boundary within 1e-5 of u*S), which are counted separately.
* At T = 0 spec_accept_exact returns exactly what spec_accept returns.
* Full size (V = 151,936, d = 2560, bf16, k = 7): requests with planted verify rows, drafts
  partly equal to the planted targets, against the oracle on float64 logits.
"""

import numpy as np
import pytest

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, workspace, zeros_bytes  # noqa: E402
from test_gpu_accept import Cycle, _compare, _near  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


@pytest.fixture(scope="module")
def c0():
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def _accept_exact(cyc, k, temps, seeds, pos, eos):
    spec.spec_accept_exact(cyc.B, cyc.k_max, k, cyc.drafts, cyc.logits, cyc.stats, cyc.cfg.V,
                           cyc.R, temps, eos, seeds, pos, cyc.out, cyc.counters, cyc.ws)


@pytest.mark.parametrize("T,n,both", [(1.0, 1000, False), (0.05, 500, True)])
def test_c0_exact_match_cycles(c0, T, n, both):
    """At T = 1 the C0 distributions are nearly flat over 4,096 tokens and a draft is almost
    never the trunk's own sample (pure parity); at T = 0.05 drafts are kept as well."""
    cfg, W, Wd = c0
    B, k = 2, cfg.k
    cyc = Cycle(cfg, Wd, B, k + 1, k)
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    seeds = to_dev(np.full(B, 11, dtype=np.uint64))
    kk = to_dev(np.full(B, k, dtype=np.int32))
    near = compared = kept = mism = 0
    for c in range(0, n, B):
        inps = [gen.cycle_inputs(cfg, W, c + b, seed=int(T * 1000) + 7) for b in range(B)]
        pos_np = np.array([16 * (c + b) + 5 for b in range(B)], dtype=np.int64)
        pos = to_dev(pos_np)
        for i in range(1, k + 1):
            cyc.draft(i, to_dev(np.stack([inp["Hd"][i - 1] for inp in inps])), temps, seeds, pos)
        cyc.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        _accept_exact(cyc, kk, temps, seeds, pos, cfg.eos_id)
        out = cyc.result()
        drafts = to_np(cyc.drafts)
        for b in range(B):
            uni = o_ph.make_uniform_source(11)
            z = o_lm.logits(W, inps[b]["H"])
            y = o_lm.logits(W, inps[b]["Hd"], rows=cfg.Vd)
            d, dm = o_accept.draft_chain_tokens(y, T, uni, int(pos_np[b]))
            tag = f"T={T} cycle {c + b}"
            if _near(dm) and list(drafts[b, :k]) != d:
                near += 1
                continue
            assert list(drafts[b, :k]) == d, tag
            r = o_accept.accept_request_exact(z, d, k, T, cfg.eos_id, uni, int(pos_np[b]))
            if _near(r["margins"]):
                near += 1
                continue
            _compare(out[b], r, tag)
            compared += 1
            kept += r["n_accept"]
            mism += int(r["n_accept"] < k and not r["eos_hit"])
    print(f"\nC0 exact-match T={T}: {compared} cycles bit-exact, {near} near-tie cycles set "
          f"aside, {kept} drafts kept, {mism} mismatches")
    assert compared >= 0.9 * n and mism > 0
    if both:
        assert kept > 0
    cnt = to_np(cyc.counters, spec.COUNTERS_DTYPE)
    assert cnt["cycles"].sum() == n and cnt["drafted"].sum() == n * k


def test_exact_at_zero_temperature_equals_greedy_accept(c0):
    cfg, W, Wd = c0
    B, k = 2, cfg.k  # 2 requests x 4 rows: the 8-row limit of the fp32 path
    a = Cycle(cfg, Wd, B, k + 1, k)
    temps = torch.zeros(B, dtype=torch.float32, device=dev())
    seeds = to_dev(np.arange(B, dtype=np.uint64))
    for c in range(20):
        kk = to_dev(np.array([c % (k + 1), k], dtype=np.int32))
        inps = [gen.cycle_inputs(cfg, W, 500 + 4 * c + b, seed=3) for b in range(B)]
        pos = to_dev(np.arange(B, dtype=np.int64) * 8 + c)
        for i in range(1, k + 1):
            a.draft(i, to_dev(np.stack([inp["Hd"][i - 1] for inp in inps])), temps, seeds, pos)
        a.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        a.accept(kk, temps, seeds, pos, cfg.eos_id, use_q=False)
        greedy = a.result().copy()
        _accept_exact(a, kk, temps, seeds, pos, cfg.eos_id)
        exact = a.result()
        assert (greedy == exact).all(), c


@pytest.fixture(scope="module")
def c1():
    ensure_built()
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def test_full_size_exact_match_k7(c1):
    """V = 151,936 x 2560 bf16, 8 requests x 8 rows at T = 0.25 with planted targets; drafts
    follow the targets for a random prefix, so keeps, mismatches and bonus draws all occur. (At
    T = 1 about 30% of each row's mass lies in tail bins ~2e-6 wide, so most multi-draw
    requests hit a near tie; at 0.25 the planted rows are decisive.)"""
    cfg, W, Wd = c1
    B, R, k = 8, 8, 7
    rng = np.random.default_rng(41)
    H, _, targets = gen.planted_rows(cfg, W, B * R, rng)
    drafts = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        n_follow = int(rng.integers(0, k + 1))
        for i in range(k):
            drafts[b, i] = targets[b * R + i] if i < n_follow else int(rng.integers(0, cfg.V))
    ws = workspace(cfg.V, B)
    logits = torch.zeros((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    T = 0.25
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(H), B, R, temps, logits,
                            stats, ws)
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    seeds = np.arange(B, dtype=np.uint64) + 900
    pos = np.arange(B, dtype=np.int64) * 100 + 4000
    spec.spec_accept_exact(B, k, to_dev(np.full(B, k, dtype=np.int32)), to_dev(drafts), logits,
                           stats, cfg.V, R, temps, cfg.eos_id, to_dev(seeds), to_dev(pos), out,
                           None, ws)
    torch.cuda.synchronize()
    o = to_np(out, spec.ACCEPT_OUT_DTYPE)
    z = o_lm.logits(W, H)
    compared = kept = mism = 0
    for b in range(B):
        r = o_accept.accept_request_exact(z[b * R:(b + 1) * R], list(drafts[b]), k, T,
                                          cfg.eos_id, o_ph.make_uniform_source(int(seeds[b])),
                                          int(pos[b]))
        if _near(r["margins"]):
            continue
        _compare(o[b], r, f"request {b}")
        compared += 1
        kept += r["n_accept"]
        mism += int(r["n_accept"] < k)
    assert compared >= 7 and kept > 0 and mism > 0
