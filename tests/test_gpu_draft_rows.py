"""GPU parity of the two-range draft set (spec_draft_argmax_rows and spec_accept_rows, through
the C ABI) against the oracle with its draft-row map (lucebox-hub PR #15, *What*: the draft head
covers the control and special tokens plus the lowest ids).

Draft set at V = 4,096, d = 256, bf16: ids [0, 3072) and the 256 ids from 3840.
* Draft tokens (vocabulary ids) and draft logits rows (draft-row order) against the oracle on
  the gathered rows, bf16 and 4-bit weights; touching ranges give bitwise what the plain call
  gives.
* 300 sampled cycles (T = 1, k = 3, q from the draft head) bit-exact against accept_request
  with the map, outside near-ties.
* Host limits.
"""

from dataclasses import replace

import numpy as np
import pytest

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from oracle import quant as o_q
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import (CDF_EPS, GAP_EPS, close, dev, ensure_built, to_dev, to_np,  # noqa: E402
                      workspace, ws_error, zeros_bytes)
from test_gpu_accept import _compare, _near  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402

N_LOW, HI, N_HIGH = 3072, 3840, 256
ROWS = o_accept.draft_rows(N_LOW, HI, N_HIGH)
VD = len(ROWS)


@pytest.fixture(scope="module")
def cb():
    ensure_built()
    cfg = replace(configs.get(0), wdtype="bf16")
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def _draft(Wd, wdt, cfg, h, temps, seeds, pos, off, n_low=N_LOW, hi=HI, n_high=N_HIGH):
    B = h.shape[0]
    Vd = n_low + n_high
    ws = workspace(cfg.V, B)
    q = torch.full((B, Vd), float("nan"), dtype=torch.float32, device=dev())
    qs = zeros_bytes(B * spec.ROWSTATS_BYTES)
    tok = torch.full((B,), -7, dtype=torch.int32, device=dev())
    spec.spec_draft_argmax_rows(Wd, wdt, n_low, hi, n_high, cfg.d, to_dev(h), B,
                                torch.tensor(temps, dtype=torch.float32, device=dev()),
                                to_dev(np.array(seeds, dtype=np.uint64)),
                                to_dev(np.array(pos, dtype=np.int64)), off, tok, 1, q, Vd, qs,
                                None, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    return to_np(tok), to_np(q), to_np(qs, spec.ROWSTATS_DTYPE)


def _check_draft(Wrows, h, temps, seeds, pos, off, tok, q, qs):
    """Wrows: bf16 bits of the draft rows in draft-row order."""
    y = o_lm.logits(Wrows, h)
    near = 0
    for b in range(h.shape[0]):
        T = temps[b]
        u = o_ph.uniform(seeds[b], pos[b] + off, o_ph.PURPOSE_DRAFT) if T > 0 else None
        t_ref, margin = o_accept.draft_token(y[b], T, u, ROWS)
        if T > 0:
            ok, _ = close(q[b], y[b], o_lm.fp32_abs_bound(Wrows, h[b:b + 1])[0])
            assert ok.all()
        st = o_lm.row_stats(y[b], T)
        if st["gap"] >= GAP_EPS:
            assert qs[b]["argmax"] == ROWS[st["argmax"]]
        if margin < (CDF_EPS if T > 0 else GAP_EPS):
            near += 1
        else:
            assert tok[b] == t_ref, (b, T, tok[b], t_ref)
    return near


def test_draft_tokens_two_ranges_bf16(cb):
    cfg, W, Wd = cb
    near = n = 0
    for trial in range(16):
        rng = np.random.default_rng([60, trial])
        B = [1, 3, 8][trial % 3]
        h = gen.encode(rng.standard_normal((B, cfg.d), dtype=np.float32) * 3, "bf16")
        # steer some rows to the special range so its argmax and draws are exercised
        for b in range(0, B, 2):
            t = int(rng.integers(HI, HI + N_HIGH))
            w = o_lm.bf16_to_f64(W[t]).astype(np.float32)
            h[b] = gen.f32_to_bf16(gen.bf16_to_f32(h[b]) + 40 * w / np.linalg.norm(w))
        temps = [[0.0, 1.0, 0.5][(b + trial) % 3] for b in range(B)]
        seeds = [trial * 5 + b for b in range(B)]
        pos = [100 * trial + b for b in range(B)]
        tok, q, qs = _draft(Wd, spec.SPEC_BF16, cfg, h, temps, seeds, pos, trial % 2)
        assert ((tok < N_LOW) | ((tok >= HI) & (tok < HI + N_HIGH))).all()
        near += _check_draft(W[ROWS], h, temps, seeds, pos, trial % 2, tok, q, qs)
        n += B
    assert near <= n // 10


def test_draft_tokens_two_ranges_q4(cb):
    cfg, W, _ = cb
    Wq = gen.q4_weights(cfg)
    Wqd = to_dev(Wq)
    rng = np.random.default_rng(61)
    h = gen.encode(rng.standard_normal((4, cfg.d), dtype=np.float32) * 3, "bf16")
    temps, seeds, pos = [0.0, 1.0, 0.0, 0.7], [1, 2, 3, 4], [5, 6, 7, 8]
    tok, q, qs = _draft(Wqd, spec.SPEC_Q4A32, cfg, h, temps, seeds, pos, 0)
    Wrows = o_q.dequantise(Wq[ROWS], cfg.d)
    assert _check_draft(Wrows, h, temps, seeds, pos, 0, tok, q, qs) <= 1


def test_touching_ranges_equal_the_plain_call(cb):
    cfg, W, Wd = cb
    rng = np.random.default_rng(62)
    h = gen.encode(rng.standard_normal((3, cfg.d), dtype=np.float32), "bf16")
    temps, seeds, pos = [1.0, 0.0, 0.8], [7, 8, 9], [1, 2, 3]
    a = _draft(Wd, spec.SPEC_BF16, cfg, h, temps, seeds, pos, 1, 2048, 2048, 1024)
    ws = workspace(cfg.V, 3)
    q = torch.full((3, 3072), float("nan"), dtype=torch.float32, device=dev())
    qs = zeros_bytes(3 * spec.ROWSTATS_BYTES)
    tok = torch.full((3,), -7, dtype=torch.int32, device=dev())
    spec.spec_draft_argmax(Wd, spec.SPEC_BF16, 3072, cfg.d, to_dev(h), 3,
                           torch.tensor(temps, dtype=torch.float32, device=dev()),
                           to_dev(np.array(seeds, dtype=np.uint64)),
                           to_dev(np.array(pos, dtype=np.int64)), 1, tok, 1, q, 3072, qs, None, ws)
    torch.cuda.synchronize()
    assert (a[0] == to_np(tok)).all()
    assert a[1].tobytes() == to_np(q).tobytes()
    assert a[2].tobytes() == to_np(qs, spec.ROWSTATS_DTYPE).tobytes()


def test_accept_rows_cycles(cb):
    cfg, W, Wd = cb
    B, k, T = 2, 3, 1.0
    R = k + 1
    ws = workspace(cfg.V, B)
    logits = torch.zeros((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    q = torch.zeros((k * B, VD), dtype=torch.float32, device=dev())
    qs = zeros_bytes(k * B * spec.ROWSTATS_BYTES)
    drafts = torch.zeros((B, k), dtype=torch.int32, device=dev())
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    temps = torch.full((B,), T, dtype=torch.float32, device=dev())
    seeds_np = np.full(B, 31, dtype=np.uint64)
    seeds = to_dev(seeds_np)
    kk = to_dev(np.full(B, k, dtype=np.int32))
    Wrows = W[ROWS]
    near = compared = kept = 0
    for c in range(0, 300, B):
        inps = [gen.cycle_inputs(cfg, W, c + b, seed=77) for b in range(B)]
        pos_np = np.array([16 * (c + b) + 3 for b in range(B)], dtype=np.int64)
        pos = to_dev(pos_np)
        for i in range(1, k + 1):
            hd = to_dev(np.stack([inp["Hd"][i - 1] for inp in inps]))
            spec.spec_draft_argmax_rows(Wd, spec.SPEC_BF16, N_LOW, HI, N_HIGH, cfg.d, hd, B, temps,
                                        seeds, pos, i - 1, drafts[:, i - 1:], k, q[(i - 1) * B:],
                                        VD, qs[(i - 1) * B * spec.ROWSTATS_BYTES:], None, ws)
        spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d,
                                to_dev(np.concatenate([inp["H"] for inp in inps])), B, R, temps,
                                logits, stats, ws)
        spec.spec_accept_rows(B, k, kk, drafts, logits, stats, cfg.V, R, q, qs, N_LOW, HI, N_HIGH,
                              VD, temps, cfg.eos_id, seeds, pos, out, None, ws)
        torch.cuda.synchronize()
        o = to_np(out, spec.ACCEPT_OUT_DTYPE)
        d_gpu = to_np(drafts)
        for b in range(B):
            uni = o_ph.make_uniform_source(31)
            z = o_lm.logits(W, inps[b]["H"])
            y = o_lm.logits(Wrows, inps[b]["Hd"])
            d, dm = o_accept.draft_chain_tokens(y, T, uni, int(pos_np[b]), ROWS)
            if list(d_gpu[b]) != d:
                assert _near(dm)
                near += 1
                continue
            r = o_accept.accept_request(z, y, d, k, T, cfg.eos_id, uni, int(pos_np[b]),
                                        rows=ROWS)
            if _near(r["margins"]):
                near += 1
                continue
            _compare(o[b], r, f"cycle {c + b}")
            compared += 1
            kept += r["n_accept"]
    print(f"\ntwo-range draft set: {compared} cycles bit-exact, {near} near-tie, {kept} kept")
    assert compared >= 200 and kept > 0  # ~8% of T = 1 draws at V = 4,096 sit within 1e-5


def test_host_limits(cb):
    cfg, W, Wd = cb
    lib = spec._abi.lib()
    ws = workspace(cfg.V, 1)
    h = torch.zeros((1, cfg.d), dtype=torch.int16, device=dev())
    t = torch.zeros(1, dtype=torch.float32, device=dev())
    sd = torch.zeros(1, dtype=torch.int64, device=dev())
    tok = torch.zeros(1, dtype=torch.int32, device=dev())

    def call(wdt, n_low, hi, n_high):
        return lib.spec_draft_argmax_rows(Wd.data_ptr(), wdt, n_low, hi, n_high, cfg.d,
                                          h.data_ptr(), 1, t.data_ptr(), sd.data_ptr(),
                                          sd.data_ptr(), 0, tok.data_ptr(), 1, None, 0, None,
                                          None, ws.data_ptr(), ws.numel(), None)

    assert call(spec.SPEC_BF16, 3000, 3840, 256) == 2   # n_low not a multiple of 32
    assert call(spec.SPEC_F32, 3072, 3840, 256) == 2    # fp32 weights: plain range only
    assert call(spec.SPEC_BF16, 3072, 3000, 256) == 1   # second range before the first ends
    assert call(spec.SPEC_BF16, 3072, 3840, 256) == 0
    torch.cuda.synchronize()
