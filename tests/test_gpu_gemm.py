"""GPU parity of the batched tensor-core LM head (spec_lmhead_verify with more than 8 rows)
against the float64 oracle: logits of every temperature > 0 row within tolerance, row statistics,
argmax exact outside near-ties; ragged vocabulary tiles, a partly filled second half of H, and the
full 32 requests x 8 rows x 151,936 x 2560 shape. Then one batched cycle (verify + acceptance
for 32 requests at mixed temperatures) against the oracle's acceptance."""

import numpy as np
import pytest

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import (GAP_EPS, close, dev, ensure_built, to_dev, to_np,  # noqa: E402
                      workspace, ws_error, zeros_bytes)
from test_gpu_accept import _compare, _near  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


def _cfg(V, d):
    return configs.Config(name="tc", d=d, V=V, Vd=min(V, 1024), wdtype="bf16", k=7,
                          k_mode="fixed", batch=1, rows_per_request=8, temps=(1.0,), cycles=1,
                          seeds=(0,), plant_scale=0.0, pi_draft=0.0, draft_noise=0.5)


def _run(cfg, Wd, H, B, R, temps):
    ws = workspace(cfg.V, B)
    logits = torch.full((B * R, cfg.V), float("nan"), device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(H), B, R,
                            torch.tensor(temps, dtype=torch.float32, device=dev()), logits, stats,
                            ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    return to_np(logits), to_np(stats, spec.ROWSTATS_DTYPE)


def _check(W, H, B, R, temps, logits, stats, max_near):
    z = o_lm.logits(W, H)
    bound = o_lm.fp32_abs_bound(W, H)
    near = 0
    for q in range(B * R):
        T = temps[q // R]
        ref = o_lm.row_stats(z[q], T)
        if ref["gap"] < GAP_EPS:
            near += 1
        else:
            assert stats[q]["argmax"] == ref["argmax"], q
        assert abs(stats[q]["max"] - ref["max"]) <= 2e-2 * abs(ref["max"]) + 1e-5, q
        assert abs(stats[q]["log_norm"] - ref["log_norm"]) <= 2e-2 * abs(ref["log_norm"]) + 1e-5
        if T > 0:
            ok, _ = close(logits[q], z[q], bound[q])
            assert ok.all(), (q, np.flatnonzero(~ok)[:5])
        else:
            assert np.isnan(logits[q]).all()
    assert near <= max_near


@pytest.mark.parametrize("V,d,B,R", [(4099, 256, 2, 8), (4099, 256, 25, 8), (1000, 128, 32, 8),
                                     (70001, 512, 16, 8), (517, 64, 9, 1)])
def test_batched_small_shapes(V, d, B, R):
    ensure_built()
    assert spec.spec_batched_supported()
    cfg = _cfg(V, d)
    W = gen.lm_weights(cfg, seed=V, cache=False)
    rng = np.random.default_rng([V, B])
    H = gen.encode(rng.standard_normal((B * R, d), dtype=np.float32) * 3, "bf16")
    temps = [[0.0, 1.0, 0.7][b % 3] for b in range(B)]
    logits, stats = _run(cfg, to_dev(W), H, B, R, temps)
    _check(W, H, B, R, temps, logits, stats, max_near=B * R // 20 + 1)


@pytest.fixture(scope="module")
def c4():
    ensure_built()
    cfg = configs.get(4)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def test_batched_full_shape_256_rows(c4):
    cfg, W, Wd = c4
    rng = np.random.default_rng(91)
    H, _, _ = gen.planted_rows(cfg, W, 256, rng)
    temps = list(cfg.temps)
    logits, stats = _run(cfg, Wd, H, 32, 8, temps)
    _check(W, H, 32, 8, temps, logits, stats, max_near=3)


def test_batched_cycle_acceptance_32_requests(c4):
    """32 requests x 8 rows (k per request from 1..7), half greedy and half at T = 1 with the
    ratio rule and one-hot q: verify on the tensor cores, acceptance for all 32 in one call."""
    cfg, W, Wd = c4
    B, R = 32, 8
    rng = np.random.default_rng(92)
    H, _, targets = gen.planted_rows(cfg, W, B * R, rng)
    temps = list(cfg.temps)
    ks = [int(x) for x in rng.integers(1, 8, B)]
    z = o_lm.logits(W, H)
    drafts = np.zeros((B, 7), dtype=np.int32)
    for b in range(B):  # drafts: the planted target of the previous verify row (mostly right)
        for i in range(ks[b]):
            drafts[b, i] = targets[b * R + i] if rng.random() < 0.8 else rng.integers(0, cfg.V)
    ws = workspace(cfg.V, B)
    logits = torch.zeros((B * R, cfg.V), device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    t = torch.tensor(temps, dtype=torch.float32, device=dev())
    spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, to_dev(H), B, R, t, logits, stats, ws)
    out = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    seeds = np.arange(B, dtype=np.uint64) + 500
    pos = np.arange(B, dtype=np.int64) * 1000 + 15360
    spec.spec_accept(B, 7, to_dev(np.array(ks, np.int32)), to_dev(drafts), logits, stats, cfg.V,
                     R, None, None, cfg.Vd, cfg.Vd, t, cfg.eos_id, to_dev(seeds), to_dev(pos),
                     out, None, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    o = to_np(out, spec.ACCEPT_OUT_DTYPE)
    compared = 0
    for b in range(B):
        r = o_accept.accept_request(z[b * R:(b + 1) * R], None, list(drafts[b]), ks[b], temps[b],
                                    cfg.eos_id, o_ph.make_uniform_source(int(seeds[b])),
                                    int(pos[b]))
        if _near(r["margins"]):
            continue
        _compare(o[b], r, f"request {b}")
        compared += 1
    assert compared >= 24
