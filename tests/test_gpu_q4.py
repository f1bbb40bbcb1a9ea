"""GPU parity of the LM head over 4-bit affine weights in groups of 32 (SPEC_Q4A32, through
the C ABI) against the oracle's ``quant`` module: logits and statistics within the bf16 path's
tolerance (the dequantised weights are bf16, accumulated in fp32), argmax and sampled draft
tokens exact outside near-ties, bitwise batch invariance for 1..8 rows, ragged vocabularies and
hidden sizes, and the host-side limits of the format."""

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

from gpu_util import (CDF_EPS, GAP_EPS, Verifier, close, dev, ensure_built,  # noqa: E402
                      to_dev, to_np, workspace, ws_error, zeros_bytes)
from test_gpu_verify import _check_stats  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402

Q4 = spec.SPEC_Q4A32


def _cfg(base, **kw):
    return replace(base, wdtype="bf16", **kw)


@pytest.fixture(scope="module")
def c0():
    ensure_built()
    cfg = _cfg(configs.get(0))
    Wq = gen.q4_weights(cfg)
    return cfg, Wq, to_dev(Wq), o_q.dequantise(Wq, cfg.d)


@pytest.fixture(scope="module")
def c1():
    ensure_built()
    cfg = configs.get(1)
    Wq = gen.q4_weights(cfg)
    return cfg, Wq, to_dev(Wq), gen.lm_weights(cfg)


def _verify_case(cfg, Wq, Wd, H, B, R, temps, tag, Wdq=None):
    ws = workspace(cfg.V, B)
    v = Verifier(Wd, Q4, cfg.V, cfg.d, B, R, ws)
    v.logits.fill_(float("nan"))
    v.run(to_dev(H), torch.tensor(temps, dtype=torch.float32, device=dev()))
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    logits, stats = to_np(v.logits), v.stats_np()
    if Wdq is None:
        Wdq = o_q.dequantise(Wq, cfg.d)
    z = o_lm.logits(Wdq, H)
    bound = o_lm.fp32_abs_bound(Wdq, H)
    near = 0
    for q in range(B * R):
        T = temps[q // R]
        near += _check_stats(stats[q], z[q], T, f"{tag} row {q} T={T}")
        if T > 0:
            ok, _ = close(logits[q], z[q], bound[q])
            assert ok.all(), (tag, q, np.flatnonzero(~ok)[:5])
        else:
            assert np.isnan(logits[q]).all(), f"{tag}: greedy rows must be left untouched"
    return near


@pytest.mark.parametrize("B,R", [(1, 1), (1, 2), (1, 4), (1, 8), (2, 4), (4, 2), (8, 1)])
def test_q4_c0_logits_and_stats(c0, B, R):
    cfg, Wq, Wd, Wdq = c0
    rng = np.random.default_rng([40, B, R])
    H = gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), "bf16")
    temps = [[0.0, 1.0, 0.7, 2.0][b % 4] for b in range(B)]
    _verify_case(cfg, Wq, Wd, H, B, R, temps, f"B={B} R={R}", Wdq)


@pytest.mark.parametrize("V,d", [(1, 128), (37, 384), (4099, 256), (70001, 1024), (300, 4096),
                                 (2049, 640)])
def test_q4_ragged_vocab_and_hidden_sizes(V, d):
    """V not a multiple of a tile or a band; d a multiple of 128 that leaves half a stage (384,
    640), one code chunk (256) or the largest supported size (4096)."""
    ensure_built()
    cfg = configs.Config(name="odd", d=d, V=V, Vd=V, wdtype="bf16", k=3, k_mode="fixed",
                         batch=1, rows_per_request=4, temps=(1.0,), cycles=1, seeds=(0,),
                         plant_scale=0.0, pi_draft=0.0, draft_noise=0.5)
    Wq = gen.q4_quantise(gen.lm_weights(cfg, seed=V, cache=False))
    rng = np.random.default_rng(V + d)
    H = gen.encode(rng.standard_normal((3, d), dtype=np.float32), "bf16")
    _verify_case(cfg, Wq, to_dev(Wq), H, 1, 3, [1.0], f"V={V} d={d}")


def test_q4_nonfinite_rows_flagged(c0):
    cfg, Wq, Wd, _ = c0
    H = np.zeros((2, cfg.d), dtype=np.float32)
    H[0, 0] = np.inf
    H[1, :] = 1.0
    ws = workspace(cfg.V, 1)
    v = Verifier(Wd, Q4, cfg.V, cfg.d, 1, 2, ws)
    v.run(to_dev(gen.encode(H, "bf16")), torch.tensor([1.0], device=dev()))
    torch.cuda.synchronize()
    st = v.stats_np()
    assert np.isnan(st[0]["max"]) and st[0]["argmax"] == -1
    assert not np.isnan(st[1]["max"])


def _invariance(cfg, Wd, H, counts):
    ws = workspace(cfg.V, 1)
    ref_l = ref_s = None
    for R in counts:
        v = Verifier(Wd, Q4, cfg.V, cfg.d, 1, R, ws)
        v.run(to_dev(H[:R]), torch.tensor([1.0], device=dev()))
        torch.cuda.synchronize()
        lg, st = to_np(v.logits), v.stats_np()
        if ref_l is None:
            ref_l, ref_s = lg, st
        assert lg.tobytes() == ref_l[:R].tobytes(), R
        assert st.tobytes() == ref_s[:R].tobytes(), R
    assert ws_error(ws) == 0


def test_q4_batch_invariance_c0(c0):
    cfg, _, Wd, _ = c0
    rng = np.random.default_rng(41)
    H = gen.encode(rng.standard_normal((8, cfg.d), dtype=np.float32), "bf16")
    _invariance(cfg, Wd, H, range(8, 0, -1))


def test_q4_batch_invariance_full_size(c1):
    cfg, _, Wd, W = c1
    H, _, _ = gen.planted_rows(cfg, W, 8, np.random.default_rng(42))
    _invariance(cfg, Wd, H, (8, 7, 5, 4, 3, 2, 1))


def test_q4_full_size_against_oracle(c1):
    """d = 2560, V = 151,936 quantised: every logit of 8 rows within tolerance."""
    cfg, Wq, Wd, W = c1
    H, _, _ = gen.planted_rows(configs.get(2), W, 8, np.random.default_rng(43))
    near = _verify_case(cfg, Wq, Wd, H, 1, 8, [1.0], "full")
    assert near <= 1


def _draft_case(cfg, Wq, Wd, Vd, h, temps, seeds, pos, off):
    B = h.shape[0]
    ws = workspace(Vd, B)
    q = torch.full((B, Vd), float("nan"), dtype=torch.float32, device=dev())
    qs = zeros_bytes(B * spec.ROWSTATS_BYTES)
    tok = torch.full((B,), -7, dtype=torch.int32, device=dev())
    spec.spec_draft_argmax(Wd, Q4, Vd, cfg.d, to_dev(h), B,
                           torch.tensor(temps, dtype=torch.float32, device=dev()),
                           to_dev(np.array(seeds, dtype=np.uint64)),
                           to_dev(np.array(pos, dtype=np.int64)), off, tok, 1, q, Vd, qs, None, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    tok, q, qs = to_np(tok), to_np(q), to_np(qs, spec.ROWSTATS_DTYPE)
    Wdq = o_q.dequantise(Wq[:Vd], cfg.d)
    y = o_lm.logits(Wdq, h)
    near = 0
    for b in range(B):
        T = temps[b]
        _check_stats(qs[b], y[b], T, f"draft {b}")
        if T > 0:
            u = o_ph.uniform(seeds[b], pos[b] + off, o_ph.PURPOSE_DRAFT)
            t_ref, margin = o_accept.draft_token(y[b], T, u)
            ok, _ = close(q[b], y[b], o_lm.fp32_abs_bound(Wdq, h[b:b + 1])[0])
            assert ok.all()
        else:
            t_ref, margin = o_accept.draft_token(y[b], 0.0)
            assert np.isnan(q[b]).all()
        if margin < (CDF_EPS if T > 0 else GAP_EPS):
            near += 1
        else:
            assert tok[b] == t_ref, (b, T, tok[b], t_ref, margin)
    return near


def test_q4_draft_tokens_c0(c0):
    cfg, Wq, Wd, _ = c0
    near = n = 0
    for trial in range(24):
        rng = np.random.default_rng([44, trial])
        B = [1, 2, 5, 8][trial % 4]
        h = gen.encode(rng.standard_normal((B, cfg.d), dtype=np.float32) * 3, "bf16")
        temps = [[0.0, 1.0, 0.5, 1.5][(b + trial) % 4] for b in range(B)]
        near += _draft_case(cfg, Wq, Wd, cfg.Vd, h, temps, [trial * 17 + b for b in range(B)],
                            [1000 * trial + 7 * b for b in range(B)], trial % 3)
        n += B
    assert near <= n // 10


def test_q4_draft_tokens_full_size(c1):
    """The draft head over the first 64,000 rows of the quantised matrix (same buffer)."""
    cfg, Wq, Wd, W = c1
    rng = np.random.default_rng(45)
    h, h32, _ = gen.planted_rows(configs.get(2), W, 4, rng)
    h = gen.noisy_rows(h32, 1.0, "bf16", rng)
    near = _draft_case(cfg, Wq, Wd, cfg.Vd, h, [1.0, 1.0, 0.0, 0.7], [0, 1, 2, 3],
                       [63488, 63489, 5, 2**33 + 1], 0)
    assert near <= 2


def test_q4_host_limits(c0):
    cfg, _, Wd, _ = c0
    ws = workspace(cfg.V, 2)
    H = torch.zeros((16, 4224), dtype=torch.int16, device=dev())
    temps = torch.ones(2, dtype=torch.float32, device=dev())
    stats = zeros_bytes(16 * spec.ROWSTATS_BYTES)
    lib = spec._abi.lib()

    def call(d, B, R):
        return lib.spec_lmhead_verify(Wd.data_ptr(), Q4, cfg.V, d, H.data_ptr(), B, R,
                                      temps.data_ptr(), None, stats.data_ptr(), ws.data_ptr(),
                                      ws.numel(), None)

    assert call(192, 1, 2) == 1          # d not a multiple of 128: invalid
    assert call(4224, 1, 2) == 2         # d above 4096: unsupported
    assert call(cfg.d, 2, 8) == 2        # 16 rows: the batched path takes bf16 only
    torch.cuda.synchronize()
