"""Pins for the oracle's commit/rollback (CPU only).

Target fixed by the pages: "Rejected rows leave every cache and recurrent component identical
to ordinary decoding" and "capture-commit and fallback repair are both correct" (DS4Server
issue #98, *Completion requirements*); after a rollback the KV and recurrent state equal, bit
for bit, those of a run that never drafted
(lucebox-hub PR #15, *Exactness*). The reference run here is ordinary decoding: the m kept
inputs fed one at a time.
"""

import numpy as np
import pytest

from oracle import accept, state
from synth import configs, gen


def _cfg():
    return configs.get(0)


@pytest.mark.parametrize("k", [0, 1, 3, 7])
def test_commit_equals_sequential_no_draft_for_every_m(k):
    cfg = _cfg()
    n_slots = 9
    inp = gen.state_inputs(cfg, k, seed=1, n_slots=n_slots)
    P = inp["P"]
    slots_S, slots_conv = state.verify_snapshots(inp["S0"], inp["conv0"], inp["a"], inp["b"],
                                                 inp["c"], inp["x"], k + 1)
    # what the verify forward left in the KV cache: rows P..P+k written
    kv_verified = inp["kv_pre"].copy()
    for r in range(k + 1):
        kv_verified[:, :, P + r, :] = inp["kv_rows"][r]
    for m in range(0, k + 2):
        kv, L = state.kv_commit(kv_verified, P, k, m)
        S, cv = state.commit_snapshot(slots_S, slots_conv, m)
        S2, cv2 = state.commit_replay(inp["S0"], inp["conv0"], inp["a"], inp["b"], inp["c"],
                                      inp["x"], m)
        kv_ref, L_ref, S_ref, cv_ref = state.sequential_no_draft(
            inp["kv_pre"], P, inp["kv_rows"], inp["S0"], inp["conv0"], inp["a"], inp["b"],
            inp["c"], inp["x"], m)
        assert L == L_ref == P + m
        assert kv.tobytes() == kv_ref.tobytes()
        assert S.tobytes() == S_ref.tobytes() == S2.tobytes()
        assert cv.tobytes() == cv_ref.tobytes() == cv2.tobytes()


@pytest.mark.parametrize("k", [0, 3, 7])
def test_index_commit_selects_the_snapshot(k):
    """Index mode: with cycle snapshot r written to slot (L + r) mod n_slots (the live slot L
    holding the pre-cycle state) and every other slot holding unrelated values, the slot the
    index commit selects holds, for every L and m, the state ordinary decoding reaches."""
    cfg = _cfg()
    n_slots = 9
    inp = gen.state_inputs(cfg, k, seed=4, n_slots=n_slots)
    snaps_S, snaps_conv = state.verify_snapshots(inp["S0"], inp["conv0"], inp["a"], inp["b"],
                                                 inp["c"], inp["x"], k + 1)
    rng = np.random.default_rng(k)
    for L in range(n_slots):
        slots_S = rng.standard_normal((n_slots,) + snaps_S.shape[1:]).astype(np.float32)
        slots_conv = rng.standard_normal((n_slots,) + snaps_conv.shape[1:]).astype(np.float32)
        for r in range(k + 2):
            j = state.index_slot(L, r, n_slots)
            slots_S[j], slots_conv[j] = snaps_S[r], snaps_conv[r]
        for m in range(0, k + 2):
            L2 = state.commit_index(L, m, n_slots)
            _, _, S_ref, cv_ref = state.sequential_no_draft(
                inp["kv_pre"], inp["P"], inp["kv_rows"], inp["S0"], inp["conv0"], inp["a"],
                inp["b"], inp["c"], inp["x"], m)
            assert slots_S[L2].tobytes() == S_ref.tobytes(), (L, m)
            assert slots_conv[L2].tobytes() == cv_ref.tobytes(), (L, m)
            S_snap, cv_snap = state.commit_snapshot(snaps_S, snaps_conv, m)
            assert slots_S[L2].tobytes() == S_snap.tobytes()
    assert state.commit_index(5, 0, n_slots) == 5          # nothing kept: the live slot stays
    assert state.commit_index(7, 4, n_slots) == 2          # wraps around


def test_index_commit_over_chained_cycles():
    """Three cycles in index mode, each verify forward reading the live slot the previous commit
    chose and writing its snapshots after it: the live state after each commit equals ordinary
    decoding of all rows kept so far, and no cycle overwrites its own live slot."""
    cfg = _cfg()
    n_slots = 9
    inp0 = gen.state_inputs(cfg, 7, seed=6, n_slots=n_slots)
    slots_S = np.zeros((n_slots,) + np.asarray(inp0["S0"]).shape, dtype=np.float32)
    slots_conv = np.zeros((n_slots,) + np.asarray(inp0["conv0"]).shape, dtype=np.float32)
    L = 3
    slots_S[L], slots_conv[L] = inp0["S0"], inp0["conv0"]
    S_seq, cv_seq = np.array(inp0["S0"]), np.array(inp0["conv0"])
    for cyc, (k, m) in enumerate([(7, 5), (3, 0), (6, 7)]):
        inp = gen.state_inputs(cfg, k, seed=10 + cyc, n_slots=n_slots)
        S, cv = slots_S[L].copy(), slots_conv[L].copy()
        for r in range(k + 1):  # the verify forward, from the live slot
            S, cv = state.synthetic_step(S, cv, inp["a"][r], inp["b"][r], inp["c"][r],
                                         inp["x"][r])
            j = state.index_slot(L, r + 1, n_slots)
            assert j != L
            slots_S[j], slots_conv[j] = S, cv
        for r in range(m):  # ordinary decoding of the kept rows
            S_seq, cv_seq = state.synthetic_step(S_seq, cv_seq, inp["a"][r], inp["b"][r],
                                                 inp["c"][r], inp["x"][r])
        L = state.commit_index(L, m, n_slots)
        assert slots_S[L].tobytes() == S_seq.tobytes(), cyc
        assert slots_conv[L].tobytes() == cv_seq.tobytes(), cyc


def test_eos_keeps_no_state_past_eos():
    """An accepted EOS at draft position i emits i tokens; the state keeps x_0, d_1..d_{i-1}."""
    cfg = _cfg()
    k, eos = 5, 2
    rng = np.random.default_rng(4)
    inp = gen.state_inputs(cfg, k, seed=2)
    slots_S, slots_conv = state.verify_snapshots(inp["S0"], inp["conv0"], inp["a"], inp["b"],
                                                 inp["c"], inp["x"], k + 1)
    for pos in range(1, k + 1):
        z = rng.standard_normal((k + 1, 40))
        d = [int(np.argmax(z[i])) for i in range(k)]
        d[pos - 1] = eos
        z[pos - 1, eos] = z[pos - 1].max() + 1
        r = accept.accept_request(z, None, d, k, 0.0, eos, None, 0)
        m = state.kept_rows(r["status"], r["n_emit"])
        assert m == pos and r["tokens"][-1] == eos
        S, _ = state.commit_snapshot(slots_S, slots_conv, m)
        # rows fed: x_0, d_1..d_{pos-1}; the EOS itself (row pos) is not in the state
        S_ref, _ = state.commit_replay(inp["S0"], inp["conv0"], inp["a"], inp["b"], inp["c"],
                                       inp["x"], pos)
        assert S.tobytes() == S_ref.tobytes()


def test_failed_cycle_restores_pre_cycle_state():
    assert state.kept_rows(1, 3) == 0 and state.kept_rows(0, 3) == 3
    cfg = _cfg()
    inp = gen.state_inputs(cfg, 3, seed=3)
    slots_S, slots_conv = state.verify_snapshots(inp["S0"], inp["conv0"], inp["a"], inp["b"],
                                                 inp["c"], inp["x"], 4)
    S, cv = state.commit_snapshot(slots_S, slots_conv, 0)
    assert S.tobytes() == inp["S0"].tobytes() and cv.tobytes() == inp["conv0"].tobytes()
    kv, L = state.kv_commit(inp["kv_pre"], inp["P"], 3, 0)
    assert L == inp["P"] and not kv[:, :, inp["P"]:].any()


def test_kv_trim_clips_at_capacity():
    kv = np.full((1, 2, 10, 4), 7, dtype=np.uint8)
    out, L = state.kv_commit(kv, 8, 3, 1)   # rows 8..11 verified, capacity 10
    assert L == 9 and out[:, :, :9].min() == 7 and not out[:, :, 9:].any()


def test_synthetic_step_closed_forms():
    rng = np.random.default_rng(0)
    L, H, dk, dv, C, Wd = 2, 3, 4, 5, 3, 6
    S = rng.standard_normal((L, H, dk, dv)).astype(np.float32)
    conv = rng.standard_normal((L, C, Wd)).astype(np.float32)
    x = rng.standard_normal((L, Wd)).astype(np.float32)
    # a = 1, b = 0: state unchanged, conv shifts in x
    S1, c1 = state.synthetic_step(S, conv, np.ones((L, H)), np.zeros((L, H, dk)),
                                  np.zeros((L, H, dv)), x)
    assert S1.tobytes() == S.tobytes()
    assert np.array_equal(c1[:, :2], conv[:, 1:]) and np.array_equal(c1[:, 2], x)
    # S = 0: the outer product b (x) c
    b = rng.standard_normal((L, H, dk)).astype(np.float32)
    c = rng.standard_normal((L, H, dv)).astype(np.float32)
    S2, _ = state.synthetic_step(np.zeros_like(S), conv, np.full((L, H), 0.5), b, c, x)
    assert np.array_equal(S2, np.einsum("lhi,lhj->lhij", b, c).astype(np.float32))
    # small integers and a power-of-two decay: exact against integer arithmetic
    Si = rng.integers(-50, 50, (L, H, dk, dv))
    bi = rng.integers(-9, 9, (L, H, dk))
    ci = rng.integers(-9, 9, (L, H, dv))
    S3, _ = state.synthetic_step(Si.astype(np.float32), conv, np.full((L, H), 0.25), bi, ci, x)
    exact = Si * 0.25 + bi[..., :, None] * ci[..., None, :]
    assert np.array_equal(S3.astype(np.float64), exact)


def test_step_rounds_each_operation_separately():
    # fl(fl(a*s) + fl(b*c)) differs from a fused a*s + b*c for these values
    a = np.float32(1.0 + 2**-23)
    s = np.float32(1.0 + 2**-23)
    b = np.float32(-1.0)
    c = np.float32(1.0 + 2**-22)
    S, _ = state.synthetic_step(np.full((1, 1, 1, 1), s), np.zeros((1, 1, 1)),
                                np.full((1, 1), a), np.full((1, 1, 1), b), np.full((1, 1, 1), c),
                                np.zeros((1, 1)))
    unfused = np.float32(np.float32(a * s) + np.float32(b * c))
    fused = np.float32(float(a) * float(s) + float(b) * float(c))
    assert S[0, 0, 0, 0] == unfused and unfused != fused
