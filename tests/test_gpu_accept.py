"""GPU parity of drafting + verify + acceptance (through the C ABI) against the oracle.

* C0 (d=256, V=4,096, fp32, k=3): 1,000 cycles at temperature 0 and 1,000 at temperature 1,
  Philox seed 0, pos_base = 16 * cycle. Drafts, accepted counts, emitted tokens, EOS flags and
  the draw kinds must equal the oracle's exactly; cycles whose oracle margin is below the
  near-tie thresholds (top-2 gap < 1e-5, |u*q - p| < 1e-5, CDF boundary distance < 1e-5) are
  counted and reported separately.
* Forced cases: rejection at every draft position, EOS at every position, k = 0 (MTP off),
  p == q, one-hot q, out-of-range k and tokens, non-finite logits, missing logits.
* The law of the GPU's first emitted token at V=4,096 matches p_0 (chi-square).
"""

import numpy as np
import pytest
from scipy import stats as sstats

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import (CDF_EPS, GAP_EPS, RATIO_EPS, dev, ensure_built, to_dev,  # noqa: E402
                      to_np, wdt_of, workspace, ws_error, zeros_bytes)
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


@pytest.fixture(scope="module")
def c0():
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


class Cycle:
    """Device buffers for B requests x R verify rows with k_max drafts each."""

    def __init__(self, cfg, Wd, B, R, k_max):
        self.cfg, self.Wd, self.B, self.R, self.k_max = cfg, Wd, B, R, k_max
        V, Vd = cfg.V, cfg.Vd
        self.ws = workspace(V, B)
        self.logits = torch.zeros((B * R, V), dtype=torch.float32, device=dev())
        self.stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
        self.q = torch.zeros((max(k_max, 1) * B, Vd), dtype=torch.float32, device=dev())
        self.qs = zeros_bytes(max(k_max, 1) * B * spec.ROWSTATS_BYTES)
        self.drafts = torch.zeros((B, max(k_max, 1)), dtype=torch.int32, device=dev())
        self.out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
        self.counters = zeros_bytes(B * spec.COUNTERS_BYTES)

    def draft(self, i, h, temps, seeds, pos):
        """Draft i (1-based) for all requests from draft hidden rows h [B, d]."""
        B, Vd = self.B, self.cfg.Vd
        spec.spec_draft_argmax(self.Wd, wdt_of(self.cfg), Vd, self.cfg.d, h, B, temps, seeds, pos,
                               i - 1, self.drafts[:, i - 1:], self.k_max, self.q[(i - 1) * B:],
                               Vd, self.qs[(i - 1) * B * spec.ROWSTATS_BYTES:], None, self.ws)

    def verify(self, H, temps):
        spec.spec_lmhead_verify(self.Wd, wdt_of(self.cfg), self.cfg.V, self.cfg.d, H, self.B,
                                self.R, temps, self.logits, self.stats, self.ws)

    def accept(self, k, temps, seeds, pos, eos, use_q=True, logits=True):
        spec.spec_accept(self.B, self.k_max, k, self.drafts, self.logits if logits else None,
                         self.stats, self.cfg.V, self.R, self.q if use_q else None,
                         self.qs if use_q else None, self.cfg.Vd, self.cfg.Vd, temps, eos, seeds,
                         pos, self.out, self.counters, self.ws)

    def result(self):
        torch.cuda.synchronize()
        assert ws_error(self.ws) == 0
        return to_np(self.out, spec.ACCEPT_OUT_DTYPE)


def _oracle_cycle(cfg, W, inp, T, seed, pos_base, eos, forced=None):
    k = inp["k"]
    z = o_lm.logits(W, inp["H"])
    y = o_lm.logits(W, inp["Hd"], rows=cfg.Vd) if k else np.zeros((0, cfg.Vd))
    uni = o_ph.make_uniform_source(seed)
    if forced is None:
        d, dm = o_accept.draft_chain_tokens(y, T, uni, pos_base)
    else:
        d, dm = list(forced), []
    r = o_accept.accept_request(z, y if T > 0 else None, d, k, T, eos, uni, pos_base)
    return d, dm, r


def _near(margins):
    for kind, m in margins:
        if kind == "gap" and m < GAP_EPS:
            return True
        if kind == "ratio" and m < RATIO_EPS:
            return True
        if kind == "cdf" and m < CDF_EPS:
            return True
    return False


def _compare(o, r, tag):
    assert o["status"] == r["status"], tag
    assert o["n_accept"] == r["n_accept"], tag
    assert o["n_emit"] == r["n_emit"], tag
    assert list(o["tokens"][: o["n_emit"]]) == r["tokens"], tag
    assert all(t == -1 for t in o["tokens"][o["n_emit"]:]), tag
    assert bool(o["eos_hit"]) == r["eos_hit"], tag
    assert o["sample_kind"] == r["sample_kind"] and o["sample_row"] == r["sample_row"], tag


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_c0_thousand_cycles(c0, T):
    cfg, W, Wd = c0
    B, k = 2, cfg.k
    cyc = Cycle(cfg, Wd, B, k + 1, k)
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    seeds = to_dev(np.zeros(B, dtype=np.uint64))
    kk = to_dev(np.full(B, k, dtype=np.int32))
    near = compared = 0
    emitted = accepted = 0
    for c0_ in range(0, 1000, B):
        inps = [gen.cycle_inputs(cfg, W, c0_ + b, seed=int(T * 1000)) for b in range(B)]
        pos_np = np.array([16 * (c0_ + b) for b in range(B)], dtype=np.int64)
        pos = to_dev(pos_np)
        for i in range(1, k + 1):
            cyc.draft(i, to_dev(np.stack([inp["Hd"][i - 1] for inp in inps])), temps, seeds, pos)
        cyc.verify(to_dev(np.concatenate([inp["H"] for inp in inps])), temps)
        cyc.accept(kk, temps, seeds, pos, cfg.eos_id)
        out = cyc.result()
        drafts = to_np(cyc.drafts)
        for b in range(B):
            d, dm, r = _oracle_cycle(cfg, W, inps[b], T, 0, int(pos_np[b]), cfg.eos_id)
            tag = f"T={T} cycle {c0_ + b}"
            if _near(dm) and list(drafts[b, :k]) != d:
                near += 1
                continue
            assert list(drafts[b, :k]) == d, tag
            if _near(r["margins"]):
                near += 1
                continue
            _compare(out[b], r, tag)
            compared += 1
            emitted += r["n_emit"]
            accepted += r["n_accept"]
    print(f"\nC0 T={T}: {compared} cycles bit-exact, {near} near-tie cycles set aside, "
          f"{emitted} tokens, acceptance {accepted / (k * compared):.3f}")
    assert compared >= 900
    cnt = to_np(cyc.counters, spec.COUNTERS_DTYPE)
    assert cnt["cycles"].sum() == 1000 and cnt["drafted"].sum() == 1000 * k


def _planted_row(cfg, W, tok, rng, scale=60.0):
    g = rng.standard_normal(cfg.d).astype(np.float32)
    w = gen.as_f32(W[tok])
    return gen.encode((g + scale * w / np.linalg.norm(w)).astype(np.float32)[None], cfg.wdtype)[0]


def _run_forced(cfg, W, Wd, H, drafts, k, T, eos, use_q=False, Hd=None, seed=3, pos=100,
                logits=True):
    R = 8
    cyc = Cycle(cfg, Wd, 1, R, 7)
    Hfull = np.zeros((R, cfg.d), dtype=H.dtype)
    Hfull[: H.shape[0]] = H
    temps = torch.tensor([T], dtype=torch.float32, device=dev())
    cyc.verify(to_dev(Hfull), temps)
    dr = np.zeros((1, 7), dtype=np.int32)
    dr[0, :len(drafts)] = drafts
    cyc.drafts.copy_(to_dev(dr))
    if use_q:
        for i in range(1, k + 1):
            # q rows from the draft head; the sampled draft tokens are overwritten below
            cyc.draft(i, to_dev(Hd[i - 1:i]), temps, to_dev(np.array([seed], np.uint64)),
                      to_dev(np.array([pos], np.int64)))
        cyc.drafts.copy_(to_dev(dr))
    cyc.accept(to_dev(np.array([k], np.int32)), temps, to_dev(np.array([seed], np.uint64)),
               to_dev(np.array([pos], np.int64)), eos, use_q=use_q, logits=logits)
    return cyc.result()[0]


def test_greedy_rejection_at_every_position(c0):
    cfg, W, Wd = c0
    rng = np.random.default_rng(40)
    for k in range(0, 8):
        H = gen.encode(rng.standard_normal((k + 1, cfg.d), dtype=np.float32) * 3, cfg.wdtype)
        z = o_lm.logits(W, H)
        am = [int(np.argmax(z[r])) for r in range(k + 1)]
        for j in range(1, k + 2):  # j = first rejected draft; k+1 = all accepted
            d = [am[i] for i in range(k)]
            if j <= k:
                d[j - 1] = (am[j - 1] + 1) % cfg.V
            o = _run_forced(cfg, W, Wd, H, d, k, 0.0, -1)
            r = o_accept.accept_request(z, None, d, k, 0.0, -1, None, 100)
            _compare(o, r, f"k={k} j={j}")
            assert o["n_accept"] == j - 1 and o["n_emit"] == min(j, k + 1)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_eos_at_every_position(c0, T):
    cfg, W, Wd = c0
    rng = np.random.default_rng(41)
    eos, k = cfg.eos_id, 7
    for j in range(1, k + 1):
        toks = [int(t) for t in rng.integers(3, cfg.V, k + 1)]
        toks[j - 1] = eos
        H = np.stack([_planted_row(cfg, W, t, rng) for t in toks])
        z = o_lm.logits(W, H)
        d = [int(np.argmax(z[i])) for i in range(k)]
        assert d[j - 1] == eos
        o = _run_forced(cfg, W, Wd, H, d, k, T, eos)
        uni = o_ph.make_uniform_source(3)
        r = o_accept.accept_request(z, None, d, k, T, eos, uni, 100)
        if not _near(r["margins"]):
            _compare(o, r, f"T={T} eos at {j}")
        assert o["eos_hit"] == 1 and o["tokens"][o["n_emit"] - 1] == eos
        assert o["n_emit"] == j


def test_mtp_off_k0(c0):
    cfg, W, Wd = c0
    rng = np.random.default_rng(42)
    H = gen.encode(rng.standard_normal((1, cfg.d), dtype=np.float32) * 3, cfg.wdtype)
    z = o_lm.logits(W, H)
    for T in (0.0, 1.0):
        o = _run_forced(cfg, W, Wd, H, [], 0, T, -1, seed=9, pos=77)
        r = o_accept.accept_request(z, None, [], 0, T, -1, o_ph.make_uniform_source(9), 77)
        if not _near(r["margins"]):
            _compare(o, r, f"k=0 T={T}")
        assert o["n_emit"] == 1 and o["n_accept"] == 0


def test_sampled_with_q_rows_forced_drafts(c0):
    """Ratio rule with real q rows and arbitrary drafts (including tokens outside q's support)."""
    cfg, W, Wd = c0
    rng = np.random.default_rng(43)
    near = 0
    for trial in range(60):
        k = 1 + trial % 7
        H = gen.encode(rng.standard_normal((k + 1, cfg.d), dtype=np.float32) * 3, cfg.wdtype)
        Hd = gen.noisy_rows(gen.as_f32(H[:k]), 0.5, cfg.wdtype, rng)
        d = [int(t) for t in rng.integers(0, cfg.V if trial % 3 == 0 else cfg.Vd, k)]
        o = _run_forced(cfg, W, Wd, H, d, k, 1.0, cfg.eos_id, use_q=True, Hd=Hd, seed=trial,
                        pos=5000 + trial)
        z = o_lm.logits(W, H)
        y = o_lm.logits(W, Hd, rows=cfg.Vd)
        r = o_accept.accept_request(z, y, d, k, 1.0, cfg.eos_id,
                                    o_ph.make_uniform_source(trial), 5000 + trial)
        if _near(r["margins"]):
            near += 1
            continue
        _compare(o, r, f"trial {trial}")
    assert near <= 6


def test_p_equals_q_accepts_all(c0):
    cfg, W, Wd = c0
    rng = np.random.default_rng(44)
    k = 7
    H = gen.encode(rng.standard_normal((k + 1, cfg.d), dtype=np.float32) * 3, cfg.wdtype)
    cyc = Cycle(cfg, Wd, 1, 8, k)
    temps = torch.tensor([1.0], device=dev())
    cyc.verify(to_dev(H), temps)
    z = o_lm.logits(W, H)
    d = np.array([[int(np.argsort(z[i])[-2]) for i in range(k)]], dtype=np.int32)
    cyc.drafts.copy_(to_dev(d))
    # q := the verify rows themselves over the whole vocabulary (draft-major with B = 1)
    spec.spec_accept(1, k, to_dev(np.array([k], np.int32)), cyc.drafts, cyc.logits, cyc.stats,
                     cfg.V, 8, cyc.logits, cyc.stats, cfg.V, cfg.V, temps, -1,
                     to_dev(np.array([1], np.uint64)), to_dev(np.array([0], np.int64)), cyc.out,
                     None, cyc.ws)
    o = cyc.result()[0]
    assert o["n_accept"] == k and o["n_emit"] == k + 1 and o["sample_kind"] == 2


def test_status_codes(c0):
    cfg, W, Wd = c0
    rng = np.random.default_rng(45)
    H = gen.encode(rng.standard_normal((4, cfg.d), dtype=np.float32), cfg.wdtype)
    assert _run_forced(cfg, W, Wd, H, [1, 2, 3, 4, 5, 6, 7], 8, 0.0, -1)["status"] == 2
    assert _run_forced(cfg, W, Wd, H, [1, cfg.V, 3], 3, 0.0, -1)["status"] == 5
    assert _run_forced(cfg, W, Wd, H, [1, -1, 3], 3, 1.0, -1)["status"] == 5
    assert _run_forced(cfg, W, Wd, H, [1, 2, 3], 3, 1.0, -1, logits=False)["status"] == 4
    Hn = H.copy()
    Hn[2, 0] = np.inf
    o = _run_forced(cfg, W, Wd, Hn, [1, 2, 3], 3, 1.0, -1)
    assert o["status"] == 1 and o["n_emit"] == 0 and list(o["tokens"]) == [-1] * 8
    # the same non-finite row past the last row the cycle uses is harmless
    assert _run_forced(cfg, W, Wd, Hn, [1], 1, 0.0, -1)["status"] == 0


def test_first_token_law_chi_square(c0):
    """k = 1 at T = 1 with drafts drawn from q: the GPU's first token ~ p_0, bonus ~ p_1."""
    cfg, W, Wd = c0
    rng = np.random.default_rng(46)
    H = gen.encode(rng.standard_normal((2, cfg.d), dtype=np.float32), cfg.wdtype)
    Hd = gen.noisy_rows(gen.as_f32(H[:1]), cfg.draft_noise, cfg.wdtype, rng)
    z = o_lm.logits(W, H)
    y = o_lm.logits(W, Hd, rows=cfg.Vd)[0]
    p0, p1, q = o_lm.probs(z[0], 1.0), o_lm.probs(z[1], 1.0), o_lm.probs(y, 1.0)
    Bn, calls = 1024, 200
    one = Cycle(cfg, Wd, 1, 2, 1)
    temps1 = torch.tensor([1.0], device=dev())
    one.verify(to_dev(H), temps1)
    one.draft(1, to_dev(Hd), temps1, to_dev(np.array([0], np.uint64)),
              to_dev(np.array([0], np.int64)))
    torch.cuda.synchronize()
    logits = one.logits.repeat(Bn, 1)
    st = one.stats.view(1, -1).repeat(Bn, 1).reshape(-1)
    qrow = one.q[:1].repeat(Bn, 1)
    qst = one.qs[: spec.ROWSTATS_BYTES].view(1, -1).repeat(Bn, 1).reshape(-1)
    ws = workspace(cfg.V, Bn)
    out = zeros_bytes(Bn * spec.ACCEPT_OUT_BYTES)
    temps = torch.full((Bn,), 1.0, device=dev())
    kk = torch.ones(Bn, dtype=torch.int32, device=dev())
    seeds = to_dev(np.full(Bn, 11, dtype=np.uint64))
    first, second = [], []
    for c in range(calls):
        d = rng.choice(cfg.Vd, size=(Bn, 1), p=q / q.sum()).astype(np.int32)
        pos = to_dev((np.arange(Bn, dtype=np.int64) + c * Bn) * 16)
        spec.spec_accept(Bn, 1, kk, to_dev(d), logits, st, cfg.V, 2, qrow, qst, cfg.Vd, cfg.Vd,
                         temps, -1, seeds, pos, out, None, ws)
        o = to_np(out, spec.ACCEPT_OUT_DTYPE)
        first.append(o["tokens"][:, 0].copy())
        acc = o["n_accept"] == 1
        second.append(o["tokens"][acc, 1].copy())
    assert ws_error(ws) == 0
    first = np.concatenate(first)
    second = np.concatenate(second)

    def pval(counts, p):
        exp = p * counts.sum()
        order = np.argsort(exp)
        obs_m, exp_m, ao, ae = [], [], 0.0, 0.0
        for j in order:
            ao += counts[j]
            ae += exp[j]
            if ae >= 5:
                obs_m.append(ao)
                exp_m.append(ae)
                ao = ae = 0.0
        obs_m[-1] += ao
        exp_m[-1] += ae
        return sstats.chisquare(obs_m, exp_m).pvalue

    assert pval(np.bincount(first, minlength=cfg.V), p0) > 1e-3
    assert pval(np.bincount(second, minlength=cfg.V), p1) > 1e-3
