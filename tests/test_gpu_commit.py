"""GPU commit/rollback (through the C ABI) against the oracle, byte for byte.

Rejected rows leave every cache and recurrent component identical to ordinary decoding, and
capture-commit and replay agree (DS4Server issue #98, *Completion requirements*; lucebox-hub PR
#15, *Exactness*). Checked for every m = 0..k+1, both modes, several requests in one call, a
failed cycle, KV overflow, and the full-size state of a 64K-context workload. Index mode
(the live state kept in a slot, the commit moving only the index): the selected slot holds the
oracle's state, no state byte moves, and an invalid live slot is reported.
"""

import numpy as np
import pytest

from oracle import state as o_st
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402

N_SLOTS = 9


class DevState:
    """Device copies of B requests' state plus a spec_state_desc pointing at them."""

    def __init__(self, cfg, per_req):
        B = len(per_req)
        self.cfg, self.B = cfg, B
        self.kv = to_dev(np.stack([r["kv"] for r in per_req]))
        self.kv_len = to_dev(np.array([r["P"] for r in per_req], dtype=np.int64))
        self.rec_live = torch.full((B,) + per_req[0]["S0"].shape, -1.0, device=dev())
        self.rec_slots = to_dev(np.stack([r["slots_S"] for r in per_req]))
        self.conv_live = torch.full((B,) + per_req[0]["conv0"].shape, -1.0, device=dev())
        self.conv_slots = to_dev(np.stack([r["slots_conv"] for r in per_req]))
        self.a = to_dev(np.stack([r["a"] for r in per_req]))
        self.b = to_dev(np.stack([r["b"] for r in per_req]))
        self.c = to_dev(np.stack([r["c"] for r in per_req]))
        self.x = to_dev(np.stack([r["x"] for r in per_req]))
        d = spec.spec_state_desc()
        d.kv = self.kv.data_ptr()
        d.kv_request_stride = self.kv[0].numel()
        d.kv_layers = cfg.kv_layers
        d.kv_capacity = cfg.kv_capacity
        d.kv_row_bytes = cfg.kv_row_bytes
        d.kv_len = self.kv_len.data_ptr()
        d.rec_layers, d.rec_heads, d.rec_dk, d.rec_dv = (cfg.rec_layers, cfg.rec_heads,
                                                         cfg.rec_dk, cfg.rec_dv)
        d.rec_live = self.rec_live.data_ptr()
        d.rec_slots = self.rec_slots.data_ptr()
        d.conv_rows, d.conv_width = cfg.conv_rows, cfg.conv_width
        d.conv_live = self.conv_live.data_ptr()
        d.conv_slots = self.conv_slots.data_ptr()
        d.n_slots = N_SLOTS
        d.step_a, d.step_b, d.step_c = self.a.data_ptr(), self.b.data_ptr(), self.c.data_ptr()
        d.conv_in = self.x.data_ptr()
        self.desc = d


def _request(cfg, k, seed, P=None, capacity=None):
    inp = gen.state_inputs(cfg, k, seed=seed, n_slots=N_SLOTS, P=P, capacity=capacity)
    P = inp["P"]
    cap = inp["kv_pre"].shape[2]
    kv = inp["kv_pre"].copy()
    for r in range(k + 1):
        if P + r < cap:
            kv[:, :, P + r, :] = inp["kv_rows"][r]
    slots_S, slots_conv = o_st.verify_snapshots(inp["S0"], inp["conv0"], inp["a"], inp["b"],
                                                inp["c"], inp["x"], N_SLOTS - 1)
    return dict(inp, kv=kv, slots_S=slots_S, slots_conv=slots_conv, k=k)


def _acc(statuses, n_emits):
    o = np.zeros(len(statuses), dtype=spec.ACCEPT_OUT_DTYPE)
    o["status"] = statuses
    o["n_emit"] = n_emits
    return to_dev(o.view(np.uint8))


def _check(cfg, ds, reqs, ms, statuses, mode):
    kv = to_np(ds.kv)
    L = to_np(ds.kv_len)
    rec = to_np(ds.rec_live)
    conv = to_np(ds.conv_live)
    for b, r in enumerate(reqs):
        m = o_st.kept_rows(statuses[b], ms[b])
        kv_ref, len_ref = o_st.kv_commit(r["kv"], r["P"], r["k"], m)
        assert L[b] == len_ref and kv[b].tobytes() == kv_ref.tobytes(), (b, m, mode)
        if mode == spec.SPEC_COMMIT_SNAPSHOT:
            S_ref, c_ref = o_st.commit_snapshot(r["slots_S"], r["slots_conv"], m)
        else:
            S_ref, c_ref = o_st.commit_replay(r["S0"], r["conv0"], r["a"], r["b"], r["c"], r["x"], m)
        assert rec[b].tobytes() == S_ref.tobytes(), (b, m, mode)
        assert conv[b].tobytes() == c_ref.tobytes(), (b, m, mode)
        if r["P"] + r["k"] + 1 <= r["kv"].shape[2]:
            kv_seq, len_seq, S_seq, c_seq = o_st.sequential_no_draft(
                r["kv_pre"], r["P"], r["kv_rows"], r["S0"], r["conv0"], r["a"], r["b"], r["c"],
                r["x"], m)
            assert kv[b].tobytes() == kv_seq.tobytes() and rec[b].tobytes() == S_seq.tobytes()
            assert conv[b].tobytes() == c_seq.tobytes()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("k", [0, 1, 3, 7])
def test_commit_c0_every_m(mode, k):
    ensure_built()
    cfg = configs.get(0)
    for m in range(0, k + 2):
        reqs = [_request(cfg, k, seed=10 * k + m)]
        ds = DevState(cfg, reqs)
        cs = torch.full((1,), -9, dtype=torch.int32, device=dev())
        spec.spec_commit_rollback(1, ds.desc, _acc([0], [m]), to_dev(np.array([k], np.int32)),
                                  mode, cs)
        torch.cuda.synchronize()
        _check(cfg, ds, reqs, [m], [0], mode)
        assert to_np(cs)[0] == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_commit_batched_mixed_requests(mode):
    """Several requests in one call: different k, m, a failed cycle, and a KV overflow."""
    ensure_built()
    cfg = configs.get(0)
    ks = [2, 7, 5, 3, 4]
    ms = [1, 8, 0, 2, 3]
    statuses = [0, 0, 0, 1, 0]
    Ps = [100, 300, 7, 400, 509]     # the last one: P + k + 1 = 514 > 512 capacity
    reqs = [_request(cfg, k, seed=50 + i, P=P) for i, (k, P) in enumerate(zip(ks, Ps))]
    ds = DevState(cfg, reqs)
    cs = torch.full((len(ks),), -9, dtype=torch.int32, device=dev())
    spec.spec_commit_rollback(len(ks), ds.desc, _acc(statuses, ms),
                              to_dev(np.array(ks, np.int32)), mode, cs)
    torch.cuda.synchronize()
    _check(cfg, ds, reqs, ms, statuses, mode)
    assert list(to_np(cs)) == [0, 0, 0, 0, spec.REQ_KV_OVERFLOW]


def test_snapshot_equals_replay_full_size():
    """The 64K-context workload's state (36 layers of [16,128,128] + conv [3,8192], KV of
    4 heads x 256 bf16 at 65,536 positions): snapshot commit and replay give the bytes of the
    oracle's sequential run."""
    ensure_built()
    cfg = configs.get(3)
    for k, m in ((7, 3), (4, 5)):
        reqs = [_request(cfg, k, seed=k)]
        for mode in (0, 1):
            ds = DevState(cfg, reqs)
            spec.spec_commit_rollback(1, ds.desc, _acc([0], [m]),
                                      to_dev(np.array([k], np.int32)), mode, None)
            torch.cuda.synchronize()
            _check(cfg, ds, reqs, [m], [0], mode)
            del ds
            torch.cuda.empty_cache()


def test_invalid_descriptors_rejected():
    ensure_built()
    cfg = configs.get(0)
    ds = DevState(cfg, [_request(cfg, 1, seed=1)])
    acc = _acc([0], [1])
    k = to_dev(np.array([1], np.int32))
    bad = spec.spec_state_desc.from_buffer_copy(ds.desc)
    bad.kv_row_bytes = 24
    with pytest.raises(spec.SpecError):
        spec.spec_commit_rollback(1, bad, acc, k, 0)
    bad = spec.spec_state_desc.from_buffer_copy(ds.desc)
    bad.n_slots = 1
    with pytest.raises(spec.SpecError):
        spec.spec_commit_rollback(1, bad, acc, k, 0)
    with pytest.raises(spec.SpecError):
        spec.spec_commit_rollback(1, ds.desc, acc, k, 3)  # no such mode
    with pytest.raises(spec.SpecError):  # index mode without the live-slot array
        spec.spec_commit_rollback(1, ds.desc, acc, k, spec.SPEC_COMMIT_INDEX)


def _index_state(cfg, reqs, lives):
    """DevState whose slots follow the index convention: request b's snapshot r in slot
    (lives[b] + r) mod N_SLOTS, the live-slot array set to lives."""
    rot = []
    for r, L in zip(reqs, lives):
        S = np.empty_like(r["slots_S"])
        C = np.empty_like(r["slots_conv"])
        for j in range(N_SLOTS):
            S[o_st.index_slot(L, j, N_SLOTS)] = r["slots_S"][j]
            C[o_st.index_slot(L, j, N_SLOTS)] = r["slots_conv"][j]
        rot.append(dict(r, slots_S=S, slots_conv=C))
    ds = DevState(cfg, rot)
    ds.live = to_dev(np.array(lives, dtype=np.int32))
    ds.desc.live_slot = ds.live.data_ptr()
    return ds, rot


@pytest.mark.parametrize("k", [0, 3, 7])
def test_index_commit_c0(k):
    """Several requests, each at its own live slot (wrapping included), every m = 0..k+1 and a
    failed cycle: the new live slot is the oracle's, the KV trim is the oracle's, the selected
    slot holds the state ordinary decoding reaches, and no state byte moved."""
    ensure_built()
    cfg = configs.get(0)
    ms = list(range(0, k + 2)) + [k + 1]
    statuses = [0] * (k + 2) + [1]
    lives = [(3 * i + 5) % N_SLOTS for i in range(len(ms))]
    reqs = [_request(cfg, k, seed=200 + 10 * k + i, P=20 + 40 * i) for i in range(len(ms))]
    ds, rot = _index_state(cfg, reqs, lives)
    slots_before = to_np(ds.rec_slots).tobytes(), to_np(ds.conv_slots).tobytes()
    cs = torch.full((len(ms),), -9, dtype=torch.int32, device=dev())
    spec.spec_commit_rollback(len(ms), ds.desc, _acc(statuses, ms),
                              to_dev(np.array([k] * len(ms), np.int32)), spec.SPEC_COMMIT_INDEX,
                              cs)
    torch.cuda.synchronize()
    live, kv, L = to_np(ds.live), to_np(ds.kv), to_np(ds.kv_len)
    slots_S, slots_C = to_np(ds.rec_slots), to_np(ds.conv_slots)
    assert (slots_S.tobytes(), slots_C.tobytes()) == slots_before  # nothing moved
    assert (to_np(ds.rec_live) == -1.0).all() and (to_np(ds.conv_live) == -1.0).all()
    for b, r in enumerate(reqs):
        m = o_st.kept_rows(statuses[b], ms[b])
        assert live[b] == o_st.commit_index(lives[b], m, N_SLOTS), b
        kv_ref, len_ref = o_st.kv_commit(r["kv"], r["P"], r["k"], m)
        assert L[b] == len_ref and kv[b].tobytes() == kv_ref.tobytes(), b
        _, _, S_seq, c_seq = o_st.sequential_no_draft(
            r["kv_pre"], r["P"], r["kv_rows"], r["S0"], r["conv0"], r["a"], r["b"], r["c"],
            r["x"], m)
        assert slots_S[b, live[b]].tobytes() == S_seq.tobytes(), b
        assert slots_C[b, live[b]].tobytes() == c_seq.tobytes(), b
    assert (to_np(cs) == 0).all()


def test_index_commit_invalid_live_slot():
    """A live slot outside [0, n_slots): left as it is, SPEC_REQ_BAD_K; the KV trim still runs
    and the other requests commit."""
    ensure_built()
    cfg = configs.get(0)
    reqs = [_request(cfg, 2, seed=300 + i, P=50 + 60 * i) for i in range(3)]
    ds, _ = _index_state(cfg, reqs, [1, 4, 8])
    ds.live.copy_(torch.tensor([1, N_SLOTS, -2], dtype=torch.int32))
    cs = torch.full((3,), -9, dtype=torch.int32, device=dev())
    spec.spec_commit_rollback(3, ds.desc, _acc([0, 0, 0], [2, 2, 2]),
                              to_dev(np.array([2, 2, 2], np.int32)), spec.SPEC_COMMIT_INDEX, cs)
    torch.cuda.synchronize()
    assert list(to_np(ds.live)) == [3, N_SLOTS, -2]
    assert list(to_np(cs)) == [0, spec.REQ_BAD_K, spec.REQ_BAD_K]
    assert list(to_np(ds.kv_len)) == [r["P"] + 2 for r in reqs]
