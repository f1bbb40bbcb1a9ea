"""Full-size cycle-by-cycle GPU parity with the oracle on the sampled, adaptive-rollback and
batched workloads (d = 2560, V = 151,936 bf16 LM head, draft head over the first 64,000 rows),
every step through the C ABI.

* Sampled k = 7 at temperature 1 (DS4Server issue #98, *Implementation*: exact
  probability-ratio acceptance with residual correction; *Verification*: EOS at every
  position, deterministic seeded sampling): 200 cycles, Philox seeds 0..99 two cycles each,
  seven draft steps writing real q rows, an 8-row verify, one spec_accept call for all 200
  cycles, EOS injected in 5% of the cycles at a random proposal position.
* Adaptive width with rollback at a 64K context (*Completion requirements*: rejected rows leave
  every cache and recurrent component identical to ordinary decoding; lucebox-hub PR #15,
  *Exactness*): k ~ U{1..7} per cycle from P0 = 63,488, each cycle's acceptance driving
  spec_commit_rollback (snapshot and replay cycles alternating), the KV, recurrent and conv
  bytes equal to the oracle's sequential no-draft run after every cycle.
* Batched serving: 32 requests x 8 rows on the tensor-core LM head, half greedy and half at
  T = 1 with real q rows, then one snapshot commit of all 32 requests' state at a 16K context,
  per request against the oracle.

Drafts are compared with the oracle's draft draws; the acceptance then runs on the oracle's
draft tokens (uploaded over the GPU's own, which they equal outside near-tie draws), so that a
near-tie draft draw does not take the rest of its cycle out of the comparison. The oracle's
logits are computed once per test for all cycles' rows stacked. Near-ties are counted and set
aside as ``cycle_parity`` describes; each test prints its counts and asserts how many cycles
were compared.
"""

import numpy as np
import pytest

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from oracle import state as o_st
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from cycle_parity import Tally, check_drafts  # noqa: E402
from gpu_util import dev, ensure_built, to_dev, to_np, workspace, ws_error, zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402

RS = spec.ROWSTATS_BYTES


@pytest.fixture(scope="module")
def head():
    ensure_built()
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    return W, to_dev(W)


def _draft(Wd, cfg, h_dev, B, temps, seeds, pos, i, drafts, k_max, q, qs, q_row0, kact, ws):
    """Draft step i (1-based) for B requests whose q rows start at draft-major row q_row0."""
    spec.spec_draft_argmax(Wd, spec.SPEC_BF16, cfg.Vd, cfg.d, h_dev, B, temps, seeds, pos,
                           i - 1, drafts[:, i - 1:], k_max,
                           None if q is None else q[q_row0:], cfg.Vd, qs[q_row0 * RS:], kact, ws)


def test_sampled_k7_seeds_0_99_with_eos_injection(head):
    W, Wd = head
    cfg = configs.get(2)
    k, R, B, T = cfg.k, cfg.k + 1, 200, 1.0
    seeds_np = np.array([b // 2 for b in range(B)], dtype=np.uint64)      # seeds 0..99
    pos_np = np.array([5000 + 16 * (b % 2) for b in range(B)], dtype=np.int64)
    eos_at = [gen.eos_injection(cfg, b, k, seed=2) for b in range(B)]
    inps = [gen.cycle_inputs(cfg, W, b, seed=2, eos_at=eos_at[b]) for b in range(B)]
    assert 3 <= sum(e > 0 for e in eos_at) <= 25

    # ---- the oracle, all cycles' rows stacked
    z = o_lm.logits(W, np.concatenate([inp["H"] for inp in inps]))
    y = o_lm.logits(W, np.concatenate([inp["Hd"] for inp in inps]), rows=cfg.Vd)
    ref_drafts, ref_dm, ref = [], [], []
    for b in range(B):
        uni = o_ph.make_uniform_source(int(seeds_np[b]))
        yb = y[k * b:k * (b + 1)]
        d, dm = o_accept.draft_chain_tokens(yb, T, uni, int(pos_np[b]))
        ref_drafts.append(list(d))
        ref_dm.append(dm)
        if eos_at[b]:
            d = list(d)
            d[eos_at[b] - 1] = cfg.eos_id
        ref.append((d, o_accept.accept_request(z[R * b:R * (b + 1)], yb, d, k, T, cfg.eos_id,
                                               uni, int(pos_np[b]))))

    # ---- the GPU: 7 draft steps and an 8-row verify per cycle, one acceptance for all cycles
    ws = workspace(cfg.V, B)
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    seeds, pos = to_dev(seeds_np), to_dev(pos_np)
    drafts = torch.zeros((B, k), dtype=torch.int32, device=dev())
    q = torch.empty((k * B, cfg.Vd), dtype=torch.float32, device=dev())
    qs = zeros_bytes(k * B * RS)
    logits = torch.empty((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * RS)
    for b in range(B):
        Hd = to_dev(inps[b]["Hd"])
        for i in range(1, k + 1):
            _draft(Wd, cfg, Hd[i - 1:i], 1, temps[b:], seeds[b:], pos[b:], i, drafts[b:], k, q,
                   qs, (i - 1) * B + b, None, ws)
        spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(inps[b]["H"]), 1, R,
                                temps[b:], logits[R * b:], stats[R * b * RS:], ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    g_drafts = to_np(drafts)
    tally = Tally()
    for b in range(B):
        tally.draft_ties += check_drafts(g_drafts[b], ref_drafts[b], ref_dm[b])
    acc_drafts = to_dev(np.array([d for d, _ in ref], dtype=np.int32))
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    counters = zeros_bytes(B * spec.COUNTERS_BYTES)
    kk = torch.full((B,), k, dtype=torch.int32, device=dev())
    spec.spec_accept(B, k, kk, acc_drafts, logits, stats, cfg.V, R, q, qs, cfg.Vd, cfg.Vd, temps,
                     cfg.eos_id, seeds, pos, out, counters, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    o = to_np(out, spec.ACCEPT_OUT_DTYPE)
    eos_cycles = eos_hits = 0
    for b in range(B):
        tally.add(o[b], ref[b][1])
        if eos_at[b]:
            eos_cycles += 1
            eos_hits += int(ref[b][1]["eos_hit"])
    acc = sum(r["n_accept"] for _, r in ref) / (k * B)
    print("\n" + tally.line("sampled k=7, T=1, seeds 0-99") +
          f"; oracle acceptance {acc:.3f}; EOS injected in {eos_cycles} cycles, "
          f"{eos_hits} of them ended on EOS")
    assert tally.compared >= 0.95 * B
    assert tally.n["exact"] >= 0.5 * B
    assert eos_hits >= 1
    cnt = to_np(counters, spec.COUNTERS_DTYPE)
    assert int(cnt["cycles"].sum()) == B and int(cnt["drafted"].sum()) == k * B


class _ChainState:
    """Device state of one request at the 64K-context workload plus its spec_state_desc."""

    def __init__(self, cfg, init, n_slots):
        L, H, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
        self.kv = to_dev(init["kv_pre"])
        self.kv_len = to_dev(np.array([init["P"]], dtype=np.int64))
        self.live = to_dev(init["S0"])
        self.conv = to_dev(init["conv0"])
        self.slots = torch.zeros((n_slots, L, H, dk, dv), device=dev())
        self.cslots = torch.zeros((n_slots, L, cfg.conv_rows, cfg.conv_width), device=dev())
        self.a = torch.zeros((n_slots - 1, L, H), device=dev())
        self.b = torch.zeros((n_slots - 1, L, H, dk), device=dev())
        self.c = torch.zeros((n_slots - 1, L, H, dv), device=dev())
        self.x = torch.zeros((n_slots - 1, L, cfg.conv_width), device=dev())
        d = spec.spec_state_desc()
        d.kv, d.kv_request_stride, d.kv_layers = self.kv.data_ptr(), self.kv.numel(), cfg.kv_layers
        d.kv_capacity, d.kv_row_bytes = cfg.kv_capacity, cfg.kv_row_bytes
        d.kv_len = self.kv_len.data_ptr()
        d.rec_layers, d.rec_heads, d.rec_dk, d.rec_dv = L, H, dk, dv
        d.rec_live, d.rec_slots = self.live.data_ptr(), self.slots.data_ptr()
        d.conv_rows, d.conv_width = cfg.conv_rows, cfg.conv_width
        d.conv_live, d.conv_slots, d.n_slots = self.conv.data_ptr(), self.cslots.data_ptr(), n_slots
        d.step_a, d.step_b, d.step_c = self.a.data_ptr(), self.b.data_ptr(), self.c.data_ptr()
        d.conv_in = self.x.data_ptr()
        self.desc = d


def test_adaptive_rollback_chain_64k(head):
    """k ~ U{1..7} per cycle at T = 0; each cycle: draft steps, verify of k+1 rows, acceptance,
    the verify rows written into the KV cache, then the commit driven on the device by that
    acceptance. After every cycle the whole KV buffer, the length, the recurrent state and the
    conv rows equal the oracle's ordinary decoding of the kept inputs, byte for byte."""
    W, Wd = head
    cfg = configs.get(3)
    n_slots, cycles, seed = 9, 24, 3
    init = gen.state_inputs(cfg, 0, seed=seed, n_slots=n_slots)
    inps = [gen.cycle_inputs(cfg, W, c, seed=seed) for c in range(cycles)]
    ks = [inp["k"] for inp in inps]
    z = o_lm.logits(W, np.concatenate([inp["H"] for inp in inps]))
    y = o_lm.logits(W, np.concatenate([inp["Hd"] for inp in inps]), rows=cfg.Vd)
    zoff = np.cumsum([0] + [k + 1 for k in ks])
    yoff = np.cumsum([0] + ks)

    st = _ChainState(cfg, init, n_slots)
    ws = workspace(cfg.V, 1)
    temps = torch.zeros(1, dtype=torch.float32, device=dev())
    seeds = to_dev(np.array([seed], dtype=np.uint64))
    logits = torch.empty((8, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(8 * RS)
    drafts = torch.zeros((1, 7), dtype=torch.int32, device=dev())
    qs = zeros_bytes(7 * RS)
    out = zeros_bytes(spec.ACCEPT_OUT_BYTES)
    cstat = torch.zeros(1, dtype=torch.int32, device=dev())
    kv_ref, P = init["kv_pre"].copy(), init["P"]
    S_ref, conv_ref = init["S0"].copy(), init["conv0"].copy()
    tally = Tally()
    emitted = 0
    for c in range(cycles):
        k = ks[c]
        pos = to_dev(np.array([P], dtype=np.int64))
        Hd = to_dev(inps[c]["Hd"])
        for i in range(1, k + 1):
            _draft(Wd, cfg, Hd[i - 1:i], 1, temps, seeds, pos, i, drafts, 7, None, qs, i - 1,
                   None, ws)
        spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(inps[c]["H"]), 1, k + 1,
                                temps, logits, stats, ws)
        kd = to_dev(np.array([k], dtype=np.int32))
        d_ref, dm = o_accept.draft_chain_tokens(y[yoff[c]:yoff[c + 1]], 0.0, None, P)
        g = to_np(drafts)[0, :k]
        ties = check_drafts(g, d_ref, dm)
        tally.draft_ties += ties
        if ties:
            drafts[0, :k].copy_(to_dev(np.array(d_ref, dtype=np.int32)))
        spec.spec_accept(1, 7, kd, drafts, logits, stats, cfg.V, k + 1, None, None, cfg.Vd,
                         cfg.Vd, temps, cfg.eos_id, seeds, pos, out, None, ws)
        # what the verify forward of this cycle wrote: KV rows P..P+k and the row snapshots
        si = gen.step_inputs(cfg, c, k, seed=seed, n_slots=n_slots)
        st.kv.view(cfg.kv_layers, 2, cfg.kv_capacity, cfg.kv_row_bytes)[:, :, P:P + k + 1, :] \
            .copy_(to_dev(np.ascontiguousarray(si["kv_rows"][:k + 1].transpose(1, 2, 0, 3))))
        for name in ("a", "b", "c", "x"):
            getattr(st, name).copy_(to_dev(si[name]))
        mode = spec.SPEC_COMMIT_SNAPSHOT if c % 2 == 0 else spec.SPEC_COMMIT_REPLAY
        if mode == spec.SPEC_COMMIT_SNAPSHOT:
            sS, sC = o_st.verify_snapshots(S_ref, conv_ref, si["a"], si["b"], si["c"], si["x"],
                                           k + 1)
            st.slots[:k + 2].copy_(to_dev(sS))
            st.cslots[:k + 2].copy_(to_dev(sC))
        else:  # replay starts from the state before the cycle: the live state itself
            st.slots[0].copy_(st.live)
            st.cslots[0].copy_(st.conv)
        spec.spec_commit_rollback(1, st.desc, out, kd, mode, cstat)
        torch.cuda.synchronize()
        assert ws_error(ws) == 0 and int(to_np(cstat)[0]) == 0
        r = o_accept.accept_request(z[zoff[c]:zoff[c + 1]], None, d_ref, k, 0.0, cfg.eos_id,
                                    None, P)
        o = to_np(out, spec.ACCEPT_OUT_DTYPE)[0]
        tally.add(o, r)
        assert int(o["n_emit"]) == r["n_emit"], f"cycle {c}"  # the chain needs the same m
        m = o_st.kept_rows(r["status"], r["n_emit"])
        kv_ref, P, S_ref, conv_ref = o_st.sequential_no_draft(
            kv_ref, P, si["kv_rows"], S_ref, conv_ref, si["a"], si["b"], si["c"], si["x"], m)
        emitted += m
        assert int(to_np(st.kv_len)[0]) == P, f"cycle {c}"
        assert np.array_equal(to_np(st.kv).reshape(kv_ref.shape), kv_ref), f"KV, cycle {c}"
        assert to_np(st.live).tobytes() == S_ref.tobytes(), f"recurrent state, cycle {c}"
        assert to_np(st.conv).tobytes() == conv_ref.tobytes(), f"conv rows, cycle {c}"
    print("\n" + tally.line("adaptive k~U{1..7} at 64K, T=0") +
          f"; {emitted} tokens kept over {cycles} cycles (P {init['P']} -> {P})")
    assert tally.n["exact"] == cycles


def test_batched_32_requests_mixed_temperature_with_commit_16k(head):
    W, Wd = head
    cfg = configs.get(4)
    B, R, k_max, n_slots = cfg.batch, cfg.rows_per_request, 7, 9
    temps_np = np.array(cfg.temps, dtype=np.float32)
    seeds_np = np.arange(B, dtype=np.uint64) + 40
    pos_np = cfg.context + 17 * np.arange(B, dtype=np.int64)
    inps = [gen.cycle_inputs(cfg, W, b, seed=4) for b in range(B)]
    ks = [inp["k"] for inp in inps]
    H = np.zeros((B * R, cfg.d), dtype=np.uint16)
    for b, inp in enumerate(inps):
        H[R * b:R * b + ks[b] + 1] = inp["H"]
    z = o_lm.logits(W, H)
    y = o_lm.logits(W, np.concatenate([inp["Hd"] for inp in inps]), rows=cfg.Vd)
    yoff = np.cumsum([0] + ks)

    ws = workspace(cfg.V, B)
    temps, seeds, pos = to_dev(temps_np), to_dev(seeds_np), to_dev(pos_np)
    kd = to_dev(np.array(ks, dtype=np.int32))
    drafts = torch.zeros((B, k_max), dtype=torch.int32, device=dev())
    q = torch.empty((k_max * B, cfg.Vd), dtype=torch.float32, device=dev())
    qs = zeros_bytes(k_max * B * RS)
    for i in range(1, k_max + 1):
        for g0 in range(0, B, 8):  # the draft head takes up to 8 requests per call
            h = np.zeros((8, cfg.d), dtype=np.uint16)
            for j in range(8):
                if i <= ks[g0 + j]:
                    h[j] = inps[g0 + j]["Hd"][i - 1]
            _draft(Wd, cfg, to_dev(h), 8, temps[g0:], seeds[g0:], pos[g0:], i, drafts[g0:],
                   k_max, q, qs, (i - 1) * B + g0, kd[g0:], ws)
    logits = torch.empty((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * RS)
    spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(H), B, R, temps, logits,
                            stats, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    tally = Tally()
    g_drafts = to_np(drafts)
    ref = []
    for b in range(B):
        T = float(temps_np[b])
        uni = o_ph.make_uniform_source(int(seeds_np[b]))
        yb = y[yoff[b]:yoff[b + 1]]
        d, dm = o_accept.draft_chain_tokens(yb, T, uni, int(pos_np[b]))
        tally.draft_ties += check_drafts(g_drafts[b, :ks[b]], d, dm)
        ref.append((d, o_accept.accept_request(z[R * b:R * (b + 1)], yb if T > 0 else None, d,
                                               ks[b], T, cfg.eos_id, uni, int(pos_np[b]))))
    acc_d = np.zeros((B, k_max), dtype=np.int32)
    for b, (d, _) in enumerate(ref):
        acc_d[b, :len(d)] = d
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    spec.spec_accept(B, k_max, kd, to_dev(acc_d), logits, stats, cfg.V, R, q, qs, cfg.Vd, cfg.Vd,
                     temps, cfg.eos_id, seeds, pos, out, None, ws)

    # ---- the 32 requests' state at a 16K context: KV window around P, tagged snapshots
    L, Hh, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
    P, win = cfg.context, 64
    rng = np.random.default_rng(44)
    base = rng.standard_normal((L, Hh, dk, dv), dtype=np.float32)
    cbase = rng.standard_normal((L, cfg.conv_rows, cfg.conv_width), dtype=np.float32)
    kv = torch.zeros((B, cfg.kv_layers, 2, cfg.kv_capacity, cfg.kv_row_bytes), dtype=torch.uint8,
                     device=dev())
    kvw = rng.integers(0, 256, (B, cfg.kv_layers, 2, win + R, cfg.kv_row_bytes), dtype=np.uint8)
    for b in range(B):
        kvw[b, :, :, win + ks[b] + 1:, :] = 0  # nothing written past the cycle's k+1 rows
    kv[:, :, :, P - win:P + R, :].copy_(to_dev(kvw))
    kv_len = torch.full((B,), P, dtype=torch.int64, device=dev())
    live = torch.full((B, L, Hh, dk, dv), -1.0, device=dev())
    clive = torch.full((B, L, cfg.conv_rows, cfg.conv_width), -1.0, device=dev())
    slots = torch.empty((B, n_slots, L, Hh, dk, dv), device=dev())
    cslots = torch.empty((B, n_slots, L, cfg.conv_rows, cfg.conv_width), device=dev())
    for b in range(B):
        for r in range(n_slots):
            slots[b, r].copy_(torch.from_numpy(gen.tagged(base, b * n_slots + r)))
            cslots[b, r].copy_(torch.from_numpy(gen.tagged(cbase, b * n_slots + r)))
    d_ = spec.spec_state_desc()
    d_.kv, d_.kv_request_stride, d_.kv_layers = kv.data_ptr(), kv[0].numel(), cfg.kv_layers
    d_.kv_capacity, d_.kv_row_bytes, d_.kv_len = cfg.kv_capacity, cfg.kv_row_bytes, kv_len.data_ptr()
    d_.rec_layers, d_.rec_heads, d_.rec_dk, d_.rec_dv = L, Hh, dk, dv
    d_.rec_live, d_.rec_slots = live.data_ptr(), slots.data_ptr()
    d_.conv_rows, d_.conv_width = cfg.conv_rows, cfg.conv_width
    d_.conv_live, d_.conv_slots, d_.n_slots = clive.data_ptr(), cslots.data_ptr(), n_slots
    cst = torch.full((B,), -9, dtype=torch.int32, device=dev())
    spec.spec_commit_rollback(B, d_, out, kd, spec.SPEC_COMMIT_SNAPSHOT, cst)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0 and (to_np(cst) == 0).all()

    o = to_np(out, spec.ACCEPT_OUT_DTYPE)
    lens = to_np(kv_len)
    state_checked = 0
    for b in range(B):
        kind = tally.n.copy()
        tally.add(o[b], ref[b][1])
        if tally.n["tie"] != kind["tie"]:
            continue  # the GPU kept another number of rows at a near-tie: nothing to compare
        m = o_st.kept_rows(ref[b][1]["status"], ref[b][1]["n_emit"])
        assert lens[b] == P + m, b
        kv_b = to_np(kv[b])
        win_ref, _ = o_st.kv_commit(kvw[b], win, ks[b], m)
        assert np.array_equal(kv_b[:, :, P - win:P + R, :], win_ref), b
        assert not kv_b[:, :, :P - win, :].any() and not kv_b[:, :, P + R:, :].any(), b
        sS = np.stack([gen.tagged(base, b * n_slots + r) for r in range(n_slots)])
        sC = np.stack([gen.tagged(cbase, b * n_slots + r) for r in range(n_slots)])
        S_ref, c_ref = o_st.commit_snapshot(sS, sC, m)
        assert to_np(live[b]).tobytes() == S_ref.tobytes(), b
        assert to_np(clive[b]).tobytes() == c_ref.tobytes(), b
        state_checked += 1
    print("\n" + tally.line("batched 32 x 8, half T=0 / half T=1") +
          f"; state of {state_checked} requests committed byte-exact at 16K")
    assert tally.compared >= B - 2 and state_checked >= B - 2
