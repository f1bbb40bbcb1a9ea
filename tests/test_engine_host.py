"""Host logic of SpecVerifyEngine on the CPU: which library calls one cycle enqueues, in which
order and with which arguments, for each acceptance mode and for adaptive widths. The library
calls are replaced by a recorder (no kernel runs); buffers live on the CPU."""

import pytest

torch = pytest.importorskip("torch")

import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402
from mtp_speculative_decoding_spec_gb300 import engine as eng_mod  # noqa: E402

V, d, Vd, B, R, K_MAX = 4096, 256, 1024, 2, 4, 3


@pytest.fixture
def calls(monkeypatch):
    log = []

    def rec(name):
        def f(*args, **kw):
            log.append((name, args))
        return f

    for name in ("spec_draft_argmax", "spec_lmhead_verify", "spec_accept", "spec_accept_exact",
                 "spec_accept_filtered", "spec_commit_rollback", "spec_adapt_width",
                 "spec_adapt_width_mirror", "spec_verify_accept_greedy",
                 "spec_graph_capture_begin", "spec_graph_capture_end", "spec_graph_launch",
                 "spec_graph_destroy"):
        monkeypatch.setattr(eng_mod, name, rec(name))

    def create(n, k_next, B_):
        log.append(("spec_width_graph_create", (n, k_next, B_)))
        return 1000, [2000 + i for i in range(n)]

    def instantiate(g):
        log.append(("spec_graph_instantiate", (g,)))
        return 3000

    monkeypatch.setattr(eng_mod, "spec_width_graph_create", create)
    monkeypatch.setattr(eng_mod, "spec_graph_instantiate", instantiate)
    monkeypatch.setattr(eng_mod, "spec_workspace_bytes", lambda V_, B_: 4096)
    return log


def _engine(b=B, **kw):
    W = torch.zeros((V, d), dtype=torch.float32)
    return eng_mod.SpecVerifyEngine(W, spec.SPEC_F32, V, d, Vd, b, R, K_MAX, eos_id=2,
                                    device="cpu", **kw)


def _names(log):
    return [n for n, _ in log]


def test_ratio_cycle_order_and_draft_slots(calls):
    e = _engine()
    H = torch.zeros((B * R, d))
    Hd = torch.zeros((K_MAX, B, d))
    e.cycle(H, Hd, 2)
    assert _names(calls) == ["spec_draft_argmax", "spec_draft_argmax", "spec_lmhead_verify",
                             "spec_accept"]
    for i, (_, a) in enumerate(calls[:2], start=1):
        assert a[9] == i - 1                      # pos_offset: draft i predicts pos + i - 1
        assert a[6] is e.temps                    # drafts sampled at the requests' temperatures
        assert a[15] is None                      # fixed widths: no k_active gate
        assert a[10].data_ptr() == e.drafts[:, i - 1:].data_ptr()   # draft column i - 1
        assert a[12].data_ptr() == e.q[(i - 1) * B:].data_ptr()     # q rows draft-major
    acc = calls[3][1]
    assert acc[8] is e.q and acc[9] is e.qs       # the ratio rule reads the draft logits


def test_exact_and_filtered_modes(calls):
    e = _engine(acceptance="exact")
    e.verify_cycle(torch.zeros((B * R, d)))
    assert _names(calls) == ["spec_lmhead_verify", "spec_accept_exact"]
    calls.clear()
    f = _engine(acceptance="filtered")
    f.set_requests(top_k=[20, 5], top_p=[0.95, 0.5])
    f.draft_step(1, torch.zeros((B, d)))
    f.verify_cycle(torch.zeros((B * R, d)))
    assert _names(calls) == ["spec_draft_argmax", "spec_lmhead_verify", "spec_accept_filtered"]
    assert calls[0][1][6] is f.zero_temps         # argmax drafts: the draft head runs at T = 0
    a = calls[2][1]
    assert a[9] is f.top_k and a[10] is f.top_p
    assert f.top_k.tolist() == [20, 5] and abs(f.top_p[1].item() - 0.5) < 1e-7
    with pytest.raises(ValueError):
        _engine(acceptance="other")


def test_adaptive_enqueues_every_draft_step_and_the_width_update(calls):
    e = _engine(adaptive_cost=[1.0, 1.5, 2.0, 2.5])
    e.cycle(torch.zeros((B * R, d)), torch.zeros((K_MAX, B, d)), 1)
    names = _names(calls)
    assert names == ["spec_draft_argmax"] * K_MAX + ["spec_lmhead_verify", "spec_accept",
                                                      "spec_adapt_width"]
    for _, a in calls[:K_MAX]:
        assert a[15] is e.k                       # steps past a request's width return at once
    ad = calls[-1][1]
    assert ad[3] is e.k and ad[8] is e.k          # widths read and written in place
    assert ad[4] is e.cost and ad[5] is None      # the prior table; cycles timed on the device
    with pytest.raises(ValueError):
        _engine(adaptive_cost=[1.0, 2.0])         # needs k_max + 1 entries
    with pytest.raises(ValueError):
        _engine(adaptive_cost=[1.0, 1.5, 2.0, 2.5], width_graph=True)  # one request only


def test_adaptive_single_request_runs_a_width_graph(calls):
    """One request: the first cycle captures one body per width -- w draft steps (no gate), a
    verify and an acceptance of w + 1 rows, the width update -- and every cycle launches the
    graph; no call is enqueued outside it."""
    e = _engine(b=1, adaptive_cost=[1.0, 1.5, 2.0, 2.5])
    H, Hd = torch.ones((K_MAX + 1, d)), torch.ones((K_MAX, 1, d))
    e.cycle(H, Hd, K_MAX)
    names = _names(calls)
    assert names[0] == "spec_width_graph_create" and calls[0][1][0] == K_MAX + 1
    assert calls[0][1][1] is e.k                  # the select kernel reads the chosen widths
    assert names[-2:] == ["spec_graph_instantiate", "spec_graph_launch"]
    bodies = names[1:-2]
    i = 0
    for w in range(K_MAX + 1):
        ww = max(w, 1)
        assert bodies[i] == "spec_graph_capture_begin" and calls[1 + i][1][0] == 2000 + w
        body = bodies[i + 1:i + 1 + ww + 4]
        assert body == ["spec_draft_argmax"] * ww + ["spec_lmhead_verify", "spec_accept",
                                                    "spec_adapt_width",
                                                    "spec_graph_capture_end"]
        for j in range(ww):
            assert calls[2 + i + j][1][15] is None  # the body is the width: no gate
        assert calls[2 + i + ww][1][6] == ww + 1    # verify of w + 1 rows
        assert calls[2 + i + ww + 1][1][7] == ww + 1
        i += ww + 5
    assert torch.equal(e.H_in, H) and torch.equal(e.Hd_in, Hd)
    calls.clear()
    e.cycle(H, Hd, K_MAX)
    assert _names(calls) == ["spec_graph_launch"]
    e.close()
    assert _names(calls)[-1] == "spec_graph_destroy"


def test_adaptive_host_scheduled_widths_one_cycle_late(calls):
    """width_lag: cycle n runs at the width the device wrote to host-visible slot n % 2 after
    cycle n - 2 (the first two cycles at set_requests' k): exactly that many draft steps and no
    gate, a verify and an acceptance of width + 1 rows, and a width update that reads and
    writes device slot n % 2 and mirrors its choice into host slot n % 2."""
    e = _engine(b=1, adaptive_cost=[1.0, 1.5, 2.0, 2.5], width_lag=True)
    assert e.width_lag and not e.width_graph
    e.set_requests(k=[2])
    H, Hd = torch.ones((K_MAX + 1, d)), torch.ones((K_MAX, 1, d))
    widths = []
    for n in range(5):
        if n >= 2:  # what the device chose after cycle n - 2
            e.k_seen[n % 2, 0] = [3, 1, 2][n - 2]
        calls.clear()
        e.cycle(H, Hd, K_MAX)
        w = e.last_width
        widths.append(w)
        assert _names(calls) == ["spec_draft_argmax"] * w + [
            "spec_lmhead_verify", "spec_accept", "spec_adapt_width_mirror"]
        for j in range(w):
            assert calls[j][1][15] is None          # the cycle is its width: no gate
            assert calls[j][1][9] == j              # draft j + 1
        assert calls[w][1][6] == w + 1              # verify of w + 1 rows
        assert calls[w][1][4].shape[0] == w + 1
        acc = calls[w + 1][1]
        slot = e.k_ring[n % 2].data_ptr()
        assert acc[7] == w + 1 and acc[2].data_ptr() == slot
        ad = calls[w + 2][1]
        assert ad[3].data_ptr() == slot and ad[8].data_ptr() == slot
        assert ad[9] == e.k_seen[n % 2].data_ptr()  # the host-visible copy of the choice
        assert ad[4] is e.cost and ad[5] is None
    assert widths == [2, 2, 3, 1, 2]
    with pytest.raises(ValueError):
        _engine(b=2, adaptive_cost=[1.0, 1.5, 2.0, 2.5], width_lag=True)  # one request only
    with pytest.raises(ValueError):
        _engine(b=1, width_lag=True)                # adaptive widths only


def test_fused_greedy_verify_and_acceptance(calls):
    """fuse_greedy: while every request is greedy a cycle's verify and acceptance are one call
    (spec_verify_accept_greedy, with the engine's widths, drafts, results and counters); a
    request at T > 0, or another acceptance rule, brings back the two calls."""
    e = _engine(fuse_greedy=True)
    e.set_requests(temps=[0.0, 0.0])
    H, Hd = torch.zeros((B * R, d)), torch.zeros((K_MAX, B, d))
    e.cycle(H, Hd, 2)
    assert _names(calls) == ["spec_draft_argmax", "spec_draft_argmax",
                             "spec_verify_accept_greedy"]
    a = calls[-1][1]
    assert a[4] is H and a[5] == B and a[6] == R and a[10] == K_MAX
    assert a[11] is e.k and a[12] is e.drafts and a[13] == 2
    assert a[14] is e.out and a[15] is e.counters and a[16] is e.ws
    calls.clear()
    e.set_requests(temps=[0.0, 1.0])
    e.verify_cycle(H)
    assert _names(calls) == ["spec_lmhead_verify", "spec_accept"]
    calls.clear()
    f = _engine(fuse_greedy=True, acceptance="exact")
    f.set_requests(temps=[0.0, 0.0])
    f.verify_cycle(H)
    assert _names(calls) == ["spec_lmhead_verify", "spec_accept_exact"]


def test_host_scheduled_widths_with_the_update_fused(calls, monkeypatch):
    """width_lag with fuse_greedy, greedy requests, no state: a cycle is its draft steps and one
    fused launch that also takes the width update (k_used = k_next = the device slot, the
    host-visible slot as mirror); with a state attached the commit reads the widths before the
    update overwrites them, so the update stays a launch of its own after the commit."""
    kws = []

    def fused(*args, **kw):
        calls.append(("spec_verify_accept_greedy", args))
        kws.append(kw)
    monkeypatch.setattr(eng_mod, "spec_verify_accept_greedy", fused)
    e = _engine(b=1, adaptive_cost=[1.0, 1.5, 2.0, 2.5], width_lag=True, fuse_greedy=True)
    e.set_requests(temps=[0.0], k=[2])
    H, Hd = torch.ones((K_MAX + 1, d)), torch.ones((K_MAX, 1, d))
    e.cycle(H, Hd, K_MAX)
    assert _names(calls) == ["spec_draft_argmax"] * 2 + ["spec_verify_accept_greedy"]
    kw = kws[-1]
    slot = e.k_ring[0].data_ptr()
    assert calls[-1][1][11].data_ptr() == slot and kw["k_next"].data_ptr() == slot
    assert kw["state"] is e.width_state and kw["cost"] is e.cost
    assert kw["k_mirror"] == e.k_seen[0].data_ptr() and kw["alpha"] == e.alpha
    calls.clear()
    e.attach_state(object(), 0)
    e.cycle(H, Hd, K_MAX)
    assert _names(calls) == ["spec_draft_argmax"] * 2 + [
        "spec_verify_accept_greedy", "spec_commit_rollback", "spec_adapt_width_mirror"]
    assert kws[-1]["state"] is None  # no update inside the fused launch


def test_commit_only_with_attached_state(calls):
    e = _engine()
    e.verify_cycle(torch.zeros((B * R, d)))
    assert "spec_commit_rollback" not in _names(calls)
    calls.clear()
    desc = spec.spec_state_desc()
    e.attach_state(desc, spec.SPEC_COMMIT_REPLAY)
    e.verify_cycle(torch.zeros((B * R, d)))
    assert _names(calls)[-1] == "spec_commit_rollback"
    a = calls[-1][1]
    assert a[1] is desc and a[2] is e.out and a[4] == spec.SPEC_COMMIT_REPLAY
