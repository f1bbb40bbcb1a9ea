"""GPU parity of the adaptive verify width (spec_adapt_width and the draft-step width gate of
spec_draft_argmax, through the C ABI) against the oracle's ``adapt`` module.

* The width kernel over 60 cycles of synthetic acceptance results for 16 requests at random
  widths: rates within 1e-5 of the float64 oracle, the same observed depths and cycle counts,
  and the same next width except where two widths' values are within 1e-5 (counted).
* The gate: a draft step no request needs writes nothing; one that some need gives those
  requests the tokens an ungated call gives.
* The cost fit: the kernel's moving averages and fitted ratio against the oracle's, with
  explicit per-request cycle costs (noise, missing costs, host pauses).
* The engine in adaptive mode at C0, as a width graph and as gated draft steps: identical
  results cycle for cycle, and widths equal to an oracle replay of those results; with no
  cost given, the graph's cycles are timed on the device.
* Host-scheduled widths (one cycle late, spec_adapt_width_mirror): every cycle's result equals
  a fixed-width cycle's at the width it ran, the width of cycle n + 2 is the oracle's choice
  after cycle n, and the host-visible copy equals the device's widths.
"""

import numpy as np
import pytest

from oracle import adapt as o_adapt
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, wdt_of, workspace, zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402
from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine  # noqa: E402


def _near_tie(vals, k):
    best = vals[k]
    return any(j != k and abs(vals[j] - best) <= 1e-5 * abs(best) for j in range(len(vals)))


def test_width_kernel_against_oracle():
    """Rates, cost fit and next width over 60 cycles of synthetic results and measured costs
    (each request its own a + b*k with noise, some failed cycles, some without a cost, one host
    pause per request) against the float64 oracle."""
    ensure_built()
    rng = np.random.default_rng(5)
    B, k_max, alpha = 16, 7, 0.15
    cost = np.array([1.0 + 0.35 * k for k in range(k_max + 1)], dtype=np.float32)
    cost_d = to_dev(cost)
    state = zeros_bytes(B * spec.WIDTH_STATE_BYTES)
    ref = [o_adapt.new_state(k_max) for _ in range(B)]
    k_next = torch.zeros(B, dtype=torch.int32, device=dev())
    ca = rng.uniform(80, 160, B)
    cb = rng.uniform(20, 80, B)
    near = fitted = 0
    for c in range(60):
        k_used = rng.integers(0, k_max + 1, B).astype(np.int32)
        out = np.zeros(B, dtype=spec.ACCEPT_OUT_DTYPE)
        cyc = np.zeros(B, dtype=np.float32)
        for b in range(B):
            k = int(k_used[b])
            out[b]["status"] = 0 if rng.random() < 0.9 else 1
            n_acc = int(rng.integers(0, k + 1))
            out[b]["n_accept"] = n_acc
            out[b]["eos_hit"] = int(n_acc > 0 and rng.random() < 0.1)
            out[b]["n_emit"] = n_acc + (0 if out[b]["eos_hit"] else 1)
            cyc[b] = ca[b] + cb[b] * k + rng.normal(0, 3.0)
            if rng.random() < 0.05:
                cyc[b] = 0.0  # no measurement
            if c == 40 + b % 10:
                cyc[b] *= 10.0  # a host pause between two cycles
        spec.spec_adapt_width(B, k_max, to_dev(out.view(np.uint8)), to_dev(k_used), cost_d,
                              to_dev(cyc), alpha, state, k_next)
        torch.cuda.synchronize()
        st = to_np(state, spec.WIDTH_STATE_DTYPE)
        kn = to_np(k_next)
        for b in range(B):
            o = out[b]
            o_adapt.observe(ref[b], int(o["status"]), int(o["n_accept"]), bool(o["eos_hit"]),
                            int(k_used[b]), alpha)
            o_adapt.observe_cost(ref[b], int(o["status"]), int(k_used[b]), float(cyc[b]), alpha)
            kb, vals = o_adapt.choose(ref[b], cost.astype(np.float64), k_max)
            for d in range(1, k_max + 1):
                seen = bool((int(st[b]["seen"]) >> d) & 1)
                assert seen == (ref[b]["rate"][d] is not None), (c, b, d)
                if seen:
                    assert abs(float(st[b]["rate"][d]) - ref[b]["rate"][d]) < 1e-5, (c, b, d)
            assert int(st[b]["cycles"]) == ref[b]["cycles"]
            assert bool(int(st[b]["seen"]) & 1) == (ref[b]["fit"] is not None), (c, b)
            if ref[b]["fit"] is not None:
                assert np.allclose(st[b]["fit"], ref[b]["fit"], rtol=1e-4), (c, b)
            assert (float(st[b]["rate"][0]) > 0) == (ref[b]["ratio"] > 0), (c, b)
            if ref[b]["ratio"] > 0:
                fitted += 1
                assert abs(float(st[b]["rate"][0]) - ref[b]["ratio"]) <= 1e-3 * ref[b]["ratio"]
            if _near_tie(vals, kb):
                near += 1
                continue
            assert int(kn[b]) == kb == int(st[b]["k"]), (c, b)
    assert near < 60 * B // 10
    assert fitted > 40 * B  # the fit is in use for most of the run


@pytest.fixture(scope="module")
def c0():
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def _draft(cfg, Wd, h, temps, seeds, pos, off, tok, q, qs, ws, k_active):
    spec.spec_draft_argmax(Wd, wdt_of(cfg), cfg.Vd, cfg.d, h, h.shape[0], temps, seeds, pos, off,
                           tok, 1, q, cfg.Vd, qs, k_active, ws)


def test_draft_width_gate(c0):
    cfg, W, Wd = c0
    B = 2
    rng = np.random.default_rng(9)
    h = to_dev(gen.encode(rng.standard_normal((B, cfg.d), dtype=np.float32), cfg.wdtype))
    temps = torch.tensor([0.0, 1.0], dtype=torch.float32, device=dev())
    seeds = to_dev(np.array([3, 4], dtype=np.uint64))
    pos = to_dev(np.array([10, 20], dtype=np.int64))
    ws = workspace(cfg.V, B)
    q = torch.full((B, cfg.Vd), -5.0, dtype=torch.float32, device=dev())
    qs = zeros_bytes(B * spec.ROWSTATS_BYTES)
    # draft 2 (pos_offset 1): nobody needs it -> nothing written
    tok = torch.full((B,), -7, dtype=torch.int32, device=dev())
    _draft(cfg, Wd, h, temps, seeds, pos, 1, tok, q, qs, ws, to_dev(np.array([1, 0], np.int32)))
    torch.cuda.synchronize()
    assert (to_np(tok) == -7).all() and (to_np(q) == -5.0).all()
    # request 0 needs it, request 1 does not: request 0 gets the ungated token
    ref = torch.full((B,), -7, dtype=torch.int32, device=dev())
    _draft(cfg, Wd, h, temps, seeds, pos, 1, ref, q, qs, ws, None)
    got = torch.full((B,), -7, dtype=torch.int32, device=dev())
    _draft(cfg, Wd, h, temps, seeds, pos, 1, got, q, qs, ws, to_dev(np.array([2, 0], np.int32)))
    torch.cuda.synchronize()
    assert int(to_np(got)[0]) == int(to_np(ref)[0]) >= 0


def _adaptive_engine(cfg, Wd, cost, alpha, graph, cycle_cost):
    eng = SpecVerifyEngine(Wd, wdt_of(cfg), cfg.V, cfg.d, cfg.Vd, 1, cfg.k + 1, cfg.k,
                           cfg.eos_id, device=dev(), adaptive_cost=cost, alpha=alpha,
                           cycle_cost=cycle_cost, width_graph=graph)
    eng.set_requests(temps=[0.0], seeds=[1], pos=[0], k=[cfg.k])
    return eng


def test_engine_adaptive_widths_replay(c0):
    """The engine's adaptive cycles, as a width graph (the device-chosen width's body: its draft
    steps, a verify of width + 1 rows, acceptance, next width) and as k_max gated draft steps
    with a verify of k_max + 1 rows: the same results cycle for cycle, and widths equal to an
    oracle replay of those results (no measured costs: the prior cost table decides)."""
    cfg, W, Wd = c0
    k_max, alpha = cfg.k, 0.2
    cost = [1.0 + 0.25 * k for k in range(k_max + 1)]
    zero = torch.zeros(1, dtype=torch.float32, device=dev())
    engs = {"graph": _adaptive_engine(cfg, Wd, cost, alpha, True, zero),
            "gated": _adaptive_engine(cfg, Wd, cost, alpha, False, zero)}
    ref = o_adapt.new_state(k_max)
    widths = []
    for c in range(40):
        inp = gen.cycle_inputs(cfg, W, c, seed=21, k=k_max)
        res = {}
        for name, eng in engs.items():
            k_used = int(to_np(eng.k)[0])
            eng.cycle(to_dev(inp["H"]), to_dev(inp["Hd"])[:, None, :], k_max)
            torch.cuda.synchronize()
            res[name] = (k_used, to_np(eng.out, spec.ACCEPT_OUT_DTYPE)[0].copy(),
                         int(to_np(eng.k)[0]))
        (kg, og, ng), (kt, ot, nt) = res["graph"], res["gated"]
        assert kg == kt and ng == nt and og.tobytes() == ot.tobytes(), c
        assert og["status"] == 0 and og["n_accept"] <= kg
        o_adapt.observe(ref, 0, int(og["n_accept"]), bool(og["eos_hit"]), kg, alpha)
        kb, vals = o_adapt.choose(ref, [float(x) for x in cost], k_max)
        if not _near_tie(vals, kb):
            assert ng == kb, c
        widths.append(ng)
    cg = to_np(engs["graph"].counters, spec.COUNTERS_DTYPE)[0]
    ct = to_np(engs["gated"].counters, spec.COUNTERS_DTYPE)[0]
    assert cg.tobytes() == ct.tobytes()
    print(f"\nC0 adaptive widths: {widths}")
    for eng in engs.values():
        eng.close()


def test_engine_width_graph_times_its_cycles(c0):
    """With no cost given, the width kernel times the cycles on the device: after cycles at
    several widths the request's fit holds finite moving averages and the last timestamp."""
    cfg, W, Wd = c0
    eng = _adaptive_engine(cfg, Wd, [1.0 + 0.25 * k for k in range(cfg.k + 1)], 0.3, True,
                           None)
    for c in range(30):
        inp = gen.cycle_inputs(cfg, W, c, seed=22, k=cfg.k)
        eng.cycle(to_dev(inp["H"]), to_dev(inp["Hd"])[:, None, :], cfg.k)
    torch.cuda.synchronize()
    st = to_np(eng.width_state, spec.WIDTH_STATE_DTYPE)[0]
    assert int(st["seen"]) & 1 and int(st["t_last"]) != 0
    assert np.isfinite(st["fit"]).all() and st["fit"][2] > 0  # mean cycle cost > 0
    assert np.isfinite(st["rate"]).all()
    eng.close()


@pytest.mark.parametrize("fused", [False, True])
def test_engine_host_scheduled_widths(c0, fused):
    """width_lag at C0, 40 cycles: each cycle's acceptance result is bitwise the one a
    fixed-width engine gives at the width the cycle ran; the width of cycle n + 2 is the
    oracle's choice from the results of cycles 0..n (no measured costs: the prior decides, a
    nearly flat one so that deeper widths pay at C0's acceptance and the width moves); the
    pinned copy the width update writes equals the device's widths. Run with the width
    update as its own launch and fused into the verify's last block (fuse_greedy)."""
    cfg, W, Wd = c0
    k_max, alpha = cfg.k, 0.2
    cost = [1.0 + 0.005 * k for k in range(k_max + 1)]
    zero = torch.zeros(1, dtype=torch.float32, device=dev())
    eng = SpecVerifyEngine(Wd, wdt_of(cfg), cfg.V, cfg.d, cfg.Vd, 1, k_max + 1, k_max,
                           cfg.eos_id, device=dev(), adaptive_cost=cost, alpha=alpha,
                           cycle_cost=zero, width_lag=True, fuse_greedy=fused)
    eng.set_requests(temps=[0.0], seeds=[1], pos=[0], k=[1])  # widths grow from 1
    fixed = {}

    def fixed_out(w, H, Hd):
        if w not in fixed:
            f = SpecVerifyEngine(Wd, wdt_of(cfg), cfg.V, cfg.d, cfg.Vd, 1, w + 1, w, cfg.eos_id,
                                 device=dev())
            f.set_requests(temps=[0.0], seeds=[1], pos=[0], k=[w])
            fixed[w] = f
        fixed[w].cycle(H[:w + 1], Hd[:w], w)
        torch.cuda.synchronize()
        return to_np(fixed[w].out, spec.ACCEPT_OUT_DTYPE)[0].copy()

    ref = o_adapt.new_state(k_max)
    chosen, widths, near = {}, [], 0
    for n in range(40):
        inp = gen.cycle_inputs(cfg, W, n, seed=23, k=k_max)
        H, Hd = to_dev(inp["H"]), to_dev(inp["Hd"])[:, None, :]
        eng.cycle(H, Hd, k_max)
        torch.cuda.synchronize()
        w = eng.last_width
        widths.append(w)
        o = to_np(eng.out, spec.ACCEPT_OUT_DTYPE)[0].copy()
        assert o["status"] == 0 and o["n_accept"] <= w
        assert o.tobytes() == fixed_out(w, H, Hd).tobytes(), n
        if n >= 2 and chosen.get(n - 2) is not None:
            assert w == chosen[n - 2], n
        s = n % 2
        assert eng.k_seen[s].tolist() == to_np(eng.k_ring[s]).tolist(), n
        o_adapt.observe(ref, 0, int(o["n_accept"]), bool(o["eos_hit"]), w, alpha)
        kb, vals = o_adapt.choose(ref, [float(x) for x in cost], k_max)
        if _near_tie(vals, kb):
            near += 1
            chosen[n] = None
        else:
            chosen[n] = kb
            assert int(eng.k_seen[s][0]) == kb, n
    assert near < 10
    assert len(set(widths)) > 1  # the width moved
    print(f"\nC0 host-scheduled widths: {widths}")
