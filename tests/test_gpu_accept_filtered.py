"""GPU parity of acceptance against the top-k / top-p filtered target (spec_accept_filtered,
through the C ABI) against the oracle's ``accept_request_filtered`` (llama.cpp PR #28104,
*Result*: temperature 1.0, top-p 0.95, top-k 20; argmax drafts with q one-hot at the draft).

* C0 (d=256, V=4,096, fp32, k=3): several hundred cycles for each of four filter settings,
  drafts from the GPU draft head at temperature 0; emitted tokens, kept counts, EOS flags and
  draw kinds equal the oracle's exactly outside near-ties (a top-k cut, top-p cut, ratio test
  or CDF boundary within 1e-5), which are counted separately.
* At T = 0 the filtered call returns exactly what spec_accept returns.
* Invalid top_k / top_p give SPEC_REQ_BAD_FILTER for that request only.
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


def _filtered(cyc, kk, temps, top_k, top_p, seeds, pos, eos):
    spec.spec_accept_filtered(cyc.B, cyc.k_max, kk, cyc.drafts, cyc.logits, cyc.stats,
                              cyc.cfg.V, cyc.R, temps, top_k, top_p, eos, seeds, pos, cyc.out,
                              cyc.counters, cyc.ws)


@pytest.mark.parametrize("T,top_k,top_p,n", [(1.0, 20, 0.95, 600), (0.7, 5, 0.7, 300),
                                             (1.3, 32, 1.0, 300), (0.2, 1, 0.5, 200)])
def test_c0_filtered_cycles(c0, T, top_k, top_p, n):
    cfg, W, Wd = c0
    B, k = 2, cfg.k
    cyc = Cycle(cfg, Wd, B, k + 1, k)
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    zero = torch.zeros(B, dtype=torch.float32, device=dev())
    seeds = to_dev(np.full(B, 17, dtype=np.uint64))
    kk = to_dev(np.full(B, k, dtype=np.int32))
    tk = to_dev(np.full(B, top_k, dtype=np.int32))
    tp = to_dev(np.full(B, top_p, dtype=np.float32))
    tp32 = float(np.float32(top_p))  # the value the kernel reads
    near = compared = kept = 0
    kinds = {0: 0, 1: 0, 2: 0}
    for c in range(0, n, B):
        inps = [gen.cycle_inputs(cfg, W, c + b, seed=top_k * 7 + 3) for b in range(B)]
        pos_np = np.array([32 * (c + b) + 1 for b in range(B)], dtype=np.int64)
        pos = to_dev(pos_np)
        for i in range(1, k + 1):
            cyc.draft(i, to_dev(np.stack([inp["Hd"][i - 1] for inp in inps])), zero, seeds, pos)
        cyc.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        _filtered(cyc, kk, temps, tk, tp, seeds, pos, cfg.eos_id)
        out = cyc.result()
        drafts = to_np(cyc.drafts)
        for b in range(B):
            uni = o_ph.make_uniform_source(17)
            z = o_lm.logits(W, inps[b]["H"])
            y = o_lm.logits(W, inps[b]["Hd"], rows=cfg.Vd)
            d, dm = o_accept.draft_chain_tokens(y, 0.0, uni, int(pos_np[b]))
            tag = f"T={T} k={top_k} p={top_p} cycle {c + b}"
            if list(drafts[b, :k]) != d:
                assert _near(dm), tag
                near += 1
                continue
            r = o_accept.accept_request_filtered(z, d, k, T, top_k, tp32, cfg.eos_id, uni,
                                                 int(pos_np[b]))
            if _near(r["margins"]):
                near += 1
                continue
            _compare(out[b], r, tag)
            compared += 1
            kept += r["n_accept"]
            kinds[r["sample_kind"]] += 1
    print(f"\nC0 filtered T={T} top-k {top_k} top-p {top_p}: {compared} cycles bit-exact, "
          f"{near} near-tie cycles set aside, {kept} drafts kept, draws {kinds}")
    assert compared >= 0.85 * n
    assert kinds[1] > 0  # the noisy C0 draft head rarely passes all three rows: see below
    cnt = to_np(cyc.counters, spec.COUNTERS_DTYPE)
    assert cnt["cycles"].sum() == n and cnt["errors"].sum() == 0


@pytest.mark.parametrize("top_k,top_p", [(1, 0.9), (2, 0.99), (4, 0.6)])
def test_forced_argmax_drafts_reach_the_bonus_draw(c0, top_k, top_p):
    """Drafts set to each verify row's argmax: with top-k 1 every draft passes and the bonus
    draw runs; wider filters mix passes, residual and bonus draws. Against the oracle."""
    cfg, W, Wd = c0
    B, k = 2, cfg.k
    cyc = Cycle(cfg, Wd, B, k + 1, k)
    T = 0.3
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    seeds = to_dev(np.full(B, 23, dtype=np.uint64))
    kk = to_dev(np.full(B, k, dtype=np.int32))
    tk = to_dev(np.full(B, top_k, dtype=np.int32))
    tp = to_dev(np.full(B, top_p, dtype=np.float32))
    tp32 = float(np.float32(top_p))
    kinds = {0: 0, 1: 0, 2: 0}
    compared = 0
    for c in range(0, 60, B):
        inps = [gen.cycle_inputs(cfg, W, 3000 + c + b, seed=9) for b in range(B)]
        z = [o_lm.logits(W, inp["H"]) for inp in inps]
        d = np.array([[int(np.argmax(z[b][i])) for i in range(k)] for b in range(B)],
                     dtype=np.int32)
        pos_np = np.array([64 * (c + b) for b in range(B)], dtype=np.int64)
        cyc.drafts.copy_(to_dev(d))
        cyc.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        _filtered(cyc, kk, temps, tk, tp, seeds, to_dev(pos_np), cfg.eos_id)
        out = cyc.result()
        for b in range(B):
            r = o_accept.accept_request_filtered(z[b], list(d[b]), k, T, top_k, tp32,
                                                 cfg.eos_id, o_ph.make_uniform_source(23),
                                                 int(pos_np[b]))
            if _near(r["margins"]):
                continue
            _compare(out[b], r, f"top-k {top_k} cycle {c + b}")
            compared += 1
            kinds[r["sample_kind"]] += 1
    print(f"\nforced argmax drafts, top-k {top_k} top-p {top_p}: {compared} compared, "
          f"draws {kinds}")
    assert compared >= 50 and kinds[2] > 0
    if top_k == 1:
        assert kinds[2] == compared


def test_filtered_at_zero_temperature_is_greedy_accept(c0):
    cfg, W, Wd = c0
    B, k = 2, cfg.k
    cyc = Cycle(cfg, Wd, B, k + 1, k)
    temps = torch.zeros(B, dtype=torch.float32, device=dev())
    seeds = to_dev(np.arange(B, dtype=np.uint64))
    tk = to_dev(np.array([3, 20], dtype=np.int32))
    tp = to_dev(np.array([0.5, 0.95], dtype=np.float32))
    for c in range(12):
        kk = to_dev(np.array([c % (k + 1), k], dtype=np.int32))
        inps = [gen.cycle_inputs(cfg, W, 900 + 2 * c + b, seed=5) for b in range(B)]
        pos = to_dev(np.arange(B, dtype=np.int64) * 8 + c)
        for i in range(1, k + 1):
            cyc.draft(i, to_dev(np.stack([inp["Hd"][i - 1] for inp in inps])), temps, seeds, pos)
        cyc.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        cyc.accept(kk, temps, seeds, pos, cfg.eos_id, use_q=False)
        greedy = cyc.result().copy()
        _filtered(cyc, kk, temps, tk, tp, seeds, pos, cfg.eos_id)
        assert (cyc.result() == greedy).all(), c


def test_bad_filter_status_per_request(c0):
    cfg, W, Wd = c0
    B, k = 6, 0
    cyc = Cycle(cfg, Wd, B, 1, 0)
    temps = torch.ones(B, dtype=torch.float32, device=dev())
    seeds = to_dev(np.arange(B, dtype=np.uint64))
    pos = to_dev(np.zeros(B, dtype=np.int64))
    rng = np.random.default_rng(3)
    H = gen.encode(rng.standard_normal((B, cfg.d), dtype=np.float32), cfg.wdtype)
    cyc.verify(to_dev(H), temps)
    tk = to_dev(np.array([0, 33, 20, 20, 20, 20], dtype=np.int32))
    tp = to_dev(np.array([0.9, 0.9, 0.0, 1.5, np.nan, 0.9], dtype=np.float32))
    _filtered(cyc, to_dev(np.zeros(B, dtype=np.int32)), temps, tk, tp, seeds, pos, -1)
    o = cyc.result()
    assert list(o["status"]) == [spec.REQ_BAD_FILTER] * 5 + [spec.REQ_OK]
    assert list(o["n_emit"]) == [0] * 5 + [1]


@pytest.fixture(scope="module")
def c1():
    ensure_built()
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def test_full_size_filtered_k7(c1):
    """V = 151,936 x 2560 bf16, 8 requests x 8 rows at T = 1, top-k 20, top-p 0.95, planted
    targets; drafts follow the targets for a random prefix."""
    cfg, W, Wd = c1
    B, R, k = 8, 8, 7
    rng = np.random.default_rng(51)
    H, _, targets = gen.planted_rows(configs.get(2), W, B * R, rng)
    drafts = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        n_follow = int(rng.integers(0, k + 1))
        for i in range(k):
            drafts[b, i] = targets[b * R + i] if i < n_follow else int(rng.integers(0, cfg.V))
    ws = workspace(cfg.V, B)
    logits = torch.zeros((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    T = 1.0
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(H), B, R, temps, logits,
                            stats, ws)
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    seeds = np.arange(B, dtype=np.uint64) + 300
    pos = np.arange(B, dtype=np.int64) * 100 + 9000
    tp32 = float(np.float32(0.95))
    spec.spec_accept_filtered(B, k, to_dev(np.full(B, k, dtype=np.int32)), to_dev(drafts),
                              logits, stats, cfg.V, R, temps,
                              to_dev(np.full(B, 20, dtype=np.int32)),
                              to_dev(np.full(B, 0.95, dtype=np.float32)), cfg.eos_id,
                              to_dev(seeds), to_dev(pos), out, None, ws)
    torch.cuda.synchronize()
    o = to_np(out, spec.ACCEPT_OUT_DTYPE)
    z = o_lm.logits(W, H)
    compared = kept = mism = 0
    for b in range(B):
        r = o_accept.accept_request_filtered(z[b * R:(b + 1) * R], list(drafts[b]), k, T, 20,
                                             tp32, cfg.eos_id,
                                             o_ph.make_uniform_source(int(seeds[b])), int(pos[b]))
        if _near(r["margins"]):
            continue
        _compare(o[b], r, f"request {b}")
        compared += 1
        kept += r["n_accept"]
        mism += int(r["n_accept"] < k)
    assert compared >= 6 and kept > 0 and mism > 0


@pytest.mark.parametrize("top_k,lanes", [(20, (5, 9)), (5, (5,)), (32, (3,))])
def test_slice_topk_with_concentrated_keys(top_k, lanes):
    """Logits whose largest entries in every 1,024-entry slice sit at ids = l (mod 32) for the
    planted l: the slice selection's threshold cut then keeps more than 64 keys (two lanes at
    top-k 20; top-k 32) and falls back to rounds of a warp maximum, or few (one lane at top-k
    5). Decisions against the oracle on the same fp32 logits (statistics zero: at T > 0 the
    filtered mode reads them only for the NaN check)."""
    ensure_built()
    B, k, V = 2, 3, 4096
    R = k + 1
    rng = np.random.default_rng([61, top_k])
    z = (rng.standard_normal((B * R, V)) * 0.5).astype(np.float32)
    for s in range(V // 1024):
        for li, l in enumerate(lanes):
            for i in range(32):
                z[:, s * 1024 + 32 * i + l] = np.float32(3.0 + 0.05 * i + 0.3 * li + 0.001 * s)
    z += (np.arange(B * R, dtype=np.float32)[:, None] * np.float32(0.01))
    T = 1.0
    drafts = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        for i in range(k):
            row = z[b * R + i]
            drafts[b, i] = int(np.argmax(row)) if (b + i) % 2 == 0 else int(rng.integers(0, V))
    ws = workspace(V, B)
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    seeds = np.arange(B, dtype=np.uint64) + 71
    pos = np.arange(B, dtype=np.int64) * 10 + 5
    top_p = 0.95
    tp32 = float(np.float32(top_p))
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    compared = 0
    for rep in range(8):
        p_rep = pos + 1000 * rep
        spec.spec_accept_filtered(B, k, to_dev(np.full(B, k, dtype=np.int32)), to_dev(drafts),
                                  to_dev(z), stats, V, R, temps,
                                  to_dev(np.full(B, top_k, dtype=np.int32)),
                                  to_dev(np.full(B, top_p, dtype=np.float32)), -1,
                                  to_dev(seeds), to_dev(p_rep), out, None, ws)
        torch.cuda.synchronize()
        o = to_np(out, spec.ACCEPT_OUT_DTYPE)
        for b in range(B):
            r = o_accept.accept_request_filtered(z[b * R:(b + 1) * R].astype(np.float64),
                                                 list(drafts[b]), k, T, top_k, tp32, -1,
                                                 o_ph.make_uniform_source(int(seeds[b])),
                                                 int(p_rep[b]))
            if _near(r["margins"]):
                continue
            _compare(o[b], r, f"top-k {top_k} lanes {lanes} rep {rep} request {b}")
            compared += 1
    assert compared >= 12


@pytest.mark.parametrize("top_k", [16, 20])
def test_large_vocabulary_block_merge(top_k):
    """V = 300,000 (293 slices): past the one-warp-per-row merge (up to 256 slices) the last
    block merges a row's slice lists with the whole block, from shared memory when slices x
    top-k fits in 5,120 keys (top-k 16) and from L2 otherwise (top-k 20). Random fp32 logits,
    drafts partly the rows' argmax; against the oracle."""
    ensure_built()
    B, k, V = 2, 3, 300_000
    R = k + 1
    rng = np.random.default_rng([62, top_k])
    z = (rng.standard_normal((B * R, V)) * 2.0).astype(np.float32)
    T = 1.0
    drafts = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        for i in range(k):
            drafts[b, i] = (int(np.argmax(z[b * R + i])) if (b + i) % 2 == 0
                            else int(rng.integers(0, V)))
    ws = workspace(V, B)
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    seeds = np.arange(B, dtype=np.uint64) + 91
    top_p = 0.95
    tp32 = float(np.float32(top_p))
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    zd = to_dev(z)
    compared = 0
    for rep in range(6):
        pos = np.arange(B, dtype=np.int64) * 10 + 1000 * rep + 3
        spec.spec_accept_filtered(B, k, to_dev(np.full(B, k, dtype=np.int32)), to_dev(drafts),
                                  zd, stats, V, R, temps,
                                  to_dev(np.full(B, top_k, dtype=np.int32)),
                                  to_dev(np.full(B, top_p, dtype=np.float32)), -1,
                                  to_dev(seeds), to_dev(pos), out, None, ws)
        torch.cuda.synchronize()
        o = to_np(out, spec.ACCEPT_OUT_DTYPE)
        for b in range(B):
            r = o_accept.accept_request_filtered(z[b * R:(b + 1) * R].astype(np.float64),
                                                 list(drafts[b]), k, T, top_k, tp32, -1,
                                                 o_ph.make_uniform_source(int(seeds[b])),
                                                 int(pos[b]))
            if _near(r["margins"]):
                continue
            _compare(o[b], r, f"V={V} top-k {top_k} rep {rep} request {b}")
            compared += 1
    assert compared >= 9
