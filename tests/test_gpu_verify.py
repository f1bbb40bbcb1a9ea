"""GPU parity of the LM-head verify GEMV and the draft head (through the C ABI) against the
float64 oracle: logits and statistics within tolerance, argmax and sampled draft tokens exact
outside near-ties, and bitwise batch invariance of every row for 1..8 rows (lucebox-hub PR
#15, "Exactness": up to eight rows, a row's verify logits may not depend on how many rows are
verified together)."""

import numpy as np
import pytest

from oracle import accept as o_accept
from oracle import lmhead as o_lm
from oracle import philox as o_ph
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import (CDF_EPS, GAP_EPS, Verifier, close, dev, ensure_built,  # noqa: E402
                      to_dev, to_np, wdt_of, workspace, ws_error, zeros_bytes)
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


@pytest.fixture(scope="module")
def c0():
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


@pytest.fixture(scope="module")
def c1():
    ensure_built()
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    return cfg, W, to_dev(W)


def _check_stats(st_gpu, z, T, tag):
    """Compare one row's statistics with the oracle; returns 1 if the argmax was a near-tie."""
    ref = o_lm.row_stats(z, T)
    if ref["gap"] < GAP_EPS:
        near = 1
    else:
        near = 0
        assert st_gpu["argmax"] == ref["argmax"], tag
    assert abs(st_gpu["max"] - ref["max"]) <= 2e-2 * abs(ref["max"]) + 1e-5, tag
    if np.isinf(ref["gap"]):
        assert np.isinf(st_gpu["gap"]), tag
    else:
        assert abs(st_gpu["gap"] - ref["gap"]) <= 2e-2 * abs(ref["gap"]) + 2e-5, tag
    assert abs(st_gpu["log_norm"] - ref["log_norm"]) <= 2e-2 * abs(ref["log_norm"]) + 1e-5, tag
    return near


def _verify_case(cfg, W, Wd, H, B, R, temps, seed_tag):
    ws = workspace(cfg.V, B)
    v = Verifier(Wd, wdt_of(cfg), cfg.V, cfg.d, B, R, ws)
    v.logits.fill_(float("nan"))
    v.run(to_dev(H), torch.tensor(temps, dtype=torch.float32, device=dev()))
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    logits = to_np(v.logits)
    stats = v.stats_np()
    z = o_lm.logits(W, H)
    bound = o_lm.fp32_abs_bound(W, H)
    near = 0
    for q in range(B * R):
        T = temps[q // R]
        tag = f"{seed_tag} row {q} T={T}"
        near += _check_stats(stats[q], z[q], T, tag)
        if T > 0:
            ok, _ = close(logits[q], z[q], bound[q])
            assert ok.all(), (tag, np.flatnonzero(~ok)[:5])
        else:
            assert np.isnan(logits[q]).all(), f"{tag}: greedy rows must be left untouched"
    return near


@pytest.mark.parametrize("B,R", [(1, 1), (1, 3), (1, 4), (1, 8), (2, 4), (4, 2), (8, 1)])
def test_verify_c0_logits_and_stats(c0, B, R):
    cfg, W, Wd = c0
    rng = np.random.default_rng([B, R])
    H = gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), cfg.wdtype)
    temps = [[0.0, 1.0, 0.7, 2.0][b % 4] for b in range(B)]
    _verify_case(cfg, W, Wd, H, B, R, temps, f"B={B} R={R}")


def test_verify_c0_ragged_vocab_and_odd_shapes():
    """V not a multiple of any tile, fewer rows than blocks, tiny d."""
    ensure_built()
    for V, d, wd in ((1, 64, "f32"), (37, 8, "bf16"), (4099, 256, "f32"), (70001, 128, "bf16")):
        cfg = configs.Config(name="odd", d=d, V=V, Vd=V, wdtype=wd, k=3, k_mode="fixed", batch=1,
                             rows_per_request=4, temps=(1.0,), cycles=1, seeds=(0,),
                             plant_scale=0.0, pi_draft=0.0, draft_noise=0.5)
        W = gen.lm_weights(cfg, seed=V, cache=False)
        rng = np.random.default_rng(V)
        H = gen.encode(rng.standard_normal((3, d), dtype=np.float32), wd)
        _verify_case(cfg, W, to_dev(W), H, 1, 3, [1.0], f"V={V} d={d}")


@pytest.mark.parametrize("bands,extra", [(5, 0), (6, 0), (7, 0), (8, 0), (13, 17)])
def test_verify_partial_last_tile_shapes(bands, extra):
    """d = 2560 (40 k-blocks of 64) and V = SMs x 32 x bands + extra: every block's last
    128-row tile holds 1, 2, 3 or 4 boxes of 32 rows (its stages packed with 12, 7, 5 or 4
    k-blocks), and with 17 extra rows a few blocks own one band more and the last band is
    ragged. Logits and statistics against the oracle, one sampled and one greedy request."""
    ensure_built()
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    V = sms * 32 * bands + extra
    cfg = configs.Config(name="tiles", d=2560, V=V, Vd=V, wdtype="bf16", k=3, k_mode="fixed",
                         batch=2, rows_per_request=2, temps=(1.0,), cycles=1, seeds=(0,),
                         plant_scale=0.0, pi_draft=0.0, draft_noise=0.5)
    W = gen.lm_weights(cfg, seed=bands, cache=False)
    rng = np.random.default_rng(bands)
    H = gen.encode(rng.standard_normal((4, cfg.d), dtype=np.float32), "bf16")
    near = _verify_case(cfg, W, to_dev(W), H, 2, 2, [1.0, 0.0], f"bands={bands} V={V}")
    assert near <= 1


@pytest.mark.parametrize("V,d", [(300_000, 1024), (400_000, 512)])
def test_verify_large_vocabulary_sixteen_tiles_per_block(V, d):
    """V = 300,000 at 152 SMs gives each block up to 62 bands of 32 rows, about 16 tiles of 128
    rows (the bf16 kernel's limit before its grid grows); V = 400,000 grows the grid past one
    block per SM. Logits and statistics against the oracle at T = 1 and T = 0."""
    ensure_built()
    cfg = configs.Config(name="wide", d=d, V=V, Vd=V, wdtype="bf16", k=3, k_mode="fixed",
                         batch=2, rows_per_request=3, temps=(1.0,), cycles=1, seeds=(0,),
                         plant_scale=0.0, pi_draft=0.0, draft_noise=0.5)
    W = gen.lm_weights(cfg, seed=V // 1000, cache=False)
    rng = np.random.default_rng(V // 1000)
    H = gen.encode(rng.standard_normal((6, d), dtype=np.float32), "bf16")
    near = _verify_case(cfg, W, to_dev(W), H, 2, 3, [1.0, 0.0], f"V={V} d={d}")
    assert near <= 1


def test_verify_nonfinite_rows_flagged(c0):
    cfg, W, Wd = c0
    H = np.zeros((2, cfg.d), dtype=np.float32)
    H[0, 0] = np.inf   # inf * w -> +-inf logits, inf - inf -> NaN
    H[1, :] = np.float32(1.0)
    ws = workspace(cfg.V, 1)
    v = Verifier(Wd, wdt_of(cfg), cfg.V, cfg.d, 1, 2, ws)
    v.run(to_dev(H), torch.tensor([1.0], device=dev()))
    torch.cuda.synchronize()
    st = v.stats_np()
    assert np.isnan(st[0]["max"]) and st[0]["argmax"] == -1
    assert not np.isnan(st[1]["max"])


def test_verify_batch_invariance_c0(c0):
    cfg, W, Wd = c0
    rng = np.random.default_rng(21)
    H = gen.encode(rng.standard_normal((8, cfg.d), dtype=np.float32), cfg.wdtype)
    ref_l = ref_s = None
    for R in range(8, 0, -1):
        ws = workspace(cfg.V, 1)
        v = Verifier(Wd, wdt_of(cfg), cfg.V, cfg.d, 1, R, ws)
        v.run(to_dev(H[:R]), torch.tensor([1.0], device=dev()))
        torch.cuda.synchronize()
        lg, st = to_np(v.logits), v.stats_np()
        if ref_l is None:
            ref_l, ref_s = lg, st
        assert lg.tobytes() == ref_l[:R].tobytes(), R
        assert st.tobytes() == ref_s[:R].tobytes(), R


def test_verify_batch_invariance_full_size(c1):
    cfg, W, Wd = c1
    rng = np.random.default_rng(22)
    H, _, _ = gen.planted_rows(cfg, W, 8, rng)
    ref_l = ref_s = None
    ws = workspace(cfg.V, 1)
    for R in (8, 7, 5, 4, 3, 2, 1):
        v = Verifier(Wd, wdt_of(cfg), cfg.V, cfg.d, 1, R, ws)
        v.run(to_dev(H[:R]), torch.tensor([1.0], device=dev()))
        torch.cuda.synchronize()
        lg, st = to_np(v.logits), v.stats_np()
        if ref_l is None:
            ref_l, ref_s = lg, st
        assert lg.tobytes() == ref_l[:R].tobytes(), R
        assert st.tobytes() == ref_s[:R].tobytes(), R
    assert ws_error(ws) == 0


def test_verify_full_size_against_oracle(c1):
    """C1/C2 shapes (d=2560, V=151,936, bf16): every logit of 8 rows within tolerance."""
    cfg, W, Wd = c1
    rng = np.random.default_rng(23)
    H, _, _ = gen.planted_rows(configs.get(2), W, 8, rng)
    near = _verify_case(cfg, W, Wd, H, 1, 8, [1.0], "full")
    assert near <= 1


def _draft_case(cfg, W, Wd, Vd, h, temps, seeds, pos, off):
    B = h.shape[0]
    ws = workspace(Vd, B)
    q = torch.full((B, Vd), float("nan"), dtype=torch.float32, device=dev())
    qs = zeros_bytes(B * spec.ROWSTATS_BYTES)
    tok = torch.full((B,), -7, dtype=torch.int32, device=dev())
    spec.spec_draft_argmax(Wd, wdt_of(cfg), Vd, cfg.d, to_dev(h), B,
                           torch.tensor(temps, dtype=torch.float32, device=dev()),
                           to_dev(np.array(seeds, dtype=np.uint64)),
                           to_dev(np.array(pos, dtype=np.int64)), off, tok, 1, q, Vd, qs, None, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    tok, q, qs = to_np(tok), to_np(q), to_np(qs, spec.ROWSTATS_DTYPE)
    y = o_lm.logits(W, h, rows=Vd)
    near = 0
    for b in range(B):
        T = temps[b]
        _check_stats(qs[b], y[b], T, f"draft {b}")
        if T > 0:
            u = o_ph.uniform(seeds[b], pos[b] + off, o_ph.PURPOSE_DRAFT)
            t_ref, margin = o_accept.draft_token(y[b], T, u)
            ok, _ = close(q[b], y[b], o_lm.fp32_abs_bound(W[:Vd], h[b:b + 1])[0])
            assert ok.all()
        else:
            t_ref, margin = o_accept.draft_token(y[b], 0.0)
            assert np.isnan(q[b]).all()
        eps = CDF_EPS if T > 0 else GAP_EPS
        if margin < eps:
            near += 1
        else:
            assert tok[b] == t_ref, (b, T, tok[b], t_ref, margin)
    return near


def test_draft_tokens_c0(c0):
    cfg, W, Wd = c0
    total_near = 0
    n = 0
    for trial in range(40):
        rng = np.random.default_rng([5, trial])
        B = [1, 2, 5, 8][trial % 4]
        h = gen.encode(rng.standard_normal((B, cfg.d), dtype=np.float32) * 3, cfg.wdtype)
        temps = [[0.0, 1.0, 0.5, 1.5][(b + trial) % 4] for b in range(B)]
        seeds = [trial * 17 + b for b in range(B)]
        pos = [1000 * trial + 7 * b for b in range(B)]
        total_near += _draft_case(cfg, W, Wd, cfg.Vd, h, temps, seeds, pos, trial % 3)
        n += B
    assert total_near <= n // 10


def test_draft_tokens_full_size(c1):
    cfg, W, Wd = c1
    rng = np.random.default_rng(31)
    h, h32, _ = gen.planted_rows(configs.get(2), W, 4, rng)
    h = gen.noisy_rows(h32, 1.0, "bf16", rng)
    near = _draft_case(cfg, W, Wd, cfg.Vd, h, [1.0, 1.0, 0.0, 0.7], [0, 1, 2, 3],
                       [63488, 63489, 5, 2**33 + 1], 0)
    assert near <= 2
