"""The fused greedy verify + acceptance (spec_verify_accept_greedy) against the two calls it
replaces, spec_lmhead_verify then spec_accept at temperature <= 0, through the C ABI: the
acceptance records, the counters, the row statistics and the logits bit for bit.

Greedy acceptance (lucebox-hub PR #15, *Exactness*): a draft is kept while it is the argmax of
the verify row before it; the first mismatch emits that argmax, all k kept emit the bonus
argmax of row k; an emitted or accepted EOS ends the block (DS4Server issue #98,
*Implementation*). Cases: every acceptance depth, EOS accepted and EOS emitted, a bad k, a
draft outside the vocabulary, a non-finite row, several requests per call, each weight format
(fp32 at the tiny configuration, bf16 and 4-bit at full size), and the headline 2-row and the
8-row shapes. With the width update fused too, its state, next widths and mirror against
spec_adapt_width_mirror over 30 cycles.
"""

import numpy as np
import pytest

from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, workspace  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


def _pair(W, wdt, V, d, H, B, R, temps, k_max, k, drafts, eos):
    """Both paths on the same inputs: (out, counters, stats, logits) of each."""
    res = []
    for fused in (False, True):
        ws = workspace(V, B)
        logits = torch.full((B * R, V), -7.0, dtype=torch.float32, device=dev())
        stats = torch.zeros(B * R * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev())
        out = torch.zeros(B * spec.ACCEPT_OUT_BYTES, dtype=torch.uint8, device=dev())
        cnt = torch.zeros(B * spec.COUNTERS_BYTES, dtype=torch.uint8, device=dev())
        if fused:
            spec.spec_verify_accept_greedy(W, wdt, V, d, H, B, R, temps, logits, stats, k_max, k,
                                           drafts, eos, out, cnt, ws)
        else:
            spec.spec_lmhead_verify(W, wdt, V, d, H, B, R, temps, logits, stats, ws)
            zero = torch.zeros(B, dtype=torch.float32, device=dev())  # the greedy rule
            seeds = torch.zeros(B, dtype=torch.int64, device=dev())
            pos = torch.zeros(B, dtype=torch.int64, device=dev())
            spec.spec_accept(B, k_max, k, drafts, logits, stats, V, R, None, None, V, V, zero,
                             eos, seeds, pos, out, cnt, ws)
        torch.cuda.synchronize()
        assert int(to_np(ws[4:8]).view(np.uint32)[0]) == 0  # no wait gave up
        res.append((to_np(out).tobytes(), to_np(cnt).tobytes(), to_np(stats).tobytes(),
                    to_np(logits).tobytes()))
    return res


def _argmax(W, wdt, V, d, H, B, R, temps):
    ws = workspace(V, B)
    stats = torch.zeros(B * R * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev())
    spec.spec_lmhead_verify(W, wdt, V, d, H, B, R, temps, None, stats, ws)
    torch.cuda.synchronize()
    return to_np(stats).view(spec.ROWSTATS_DTYPE)["argmax"].reshape(B, R)


def _check_cases(W, wdt, V, d, Hs, B, R, k_max, rng, temps_list):
    """For each H batch: drafts equal to the argmax up to a per-request depth, then a wrong one;
    EOS planted at some accepted and some emitted positions; bad k and bad tokens; every result
    compared bitwise between the two paths."""
    n = 0
    for H in Hs:
        for temps in temps_list:
            am = _argmax(W, wdt, V, d, H, B, R, temps)
            k_np = np.full(B, R - 1, dtype=np.int32)
            drafts = np.zeros((B, max(k_max, 1)), dtype=np.int32)
            for b in range(B):
                depth = int(rng.integers(0, R))  # drafts 0..depth-1 match
                for i in range(R - 1):
                    drafts[b, i] = am[b, i] if i < depth else (am[b, i] + 1 + i) % V
            for eos in (-1, int(am[0, 0]), int(am[B - 1, R - 1])):
                out = _pair(W, wdt, V, d, H, B, R, temps, k_max, to_dev(k_np), to_dev(drafts),
                            eos)
                assert out[0] == out[1], (B, R, eos)
                n += 1
            # a bad k for request 0 and a draft outside the vocabulary for the last request
            k_bad = k_np.copy()
            k_bad[0] = k_max + 1
            d_bad = drafts.copy()
            if R > 1:
                d_bad[B - 1, 0] = V + 3
            out = _pair(W, wdt, V, d, H, B, R, temps, k_max, to_dev(k_bad), to_dev(d_bad), -1)
            assert out[0] == out[1]
            o = np.frombuffer(out[1][0], dtype=spec.ACCEPT_OUT_DTYPE)
            assert o[0]["status"] == spec.REQ_BAD_K
            if R > 1 and B > 1:
                assert o[B - 1]["status"] == spec.REQ_BAD_TOKEN
            n += 1
    return n


def test_fused_greedy_tiny_fp32():
    """fp32 weights at the tiny configuration (V = 4,096, d = 256): two requests of four rows,
    and one request of two rows; one temperature set greedy, one mixed (statistics and logits
    of the T > 0 rows written, acceptance still greedy)."""
    ensure_built()
    cfg = configs.get(0)
    W = to_dev(gen.lm_weights(cfg))
    rng = np.random.default_rng(1)
    for B, R in ((2, 4), (1, 2), (4, 2)):
        Hs = [to_dev(gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), "f32"))
              for _ in range(3)]
        temps = [torch.zeros(B, dtype=torch.float32, device=dev()),
                 torch.tensor([0.0, 1.0] * (B // 2) + [0.0] * (B % 2), dtype=torch.float32,
                              device=dev())]
        assert _check_cases(W, spec.SPEC_F32, cfg.V, cfg.d, Hs, B, R, R - 1, rng, temps) > 0


def test_fused_greedy_nonfinite_row():
    """A non-finite verify row: SPEC_REQ_NONFINITE from both paths, the same bytes."""
    ensure_built()
    cfg = configs.get(0)
    W = to_dev(gen.lm_weights(cfg))
    rng = np.random.default_rng(2)
    B, R = 2, 4
    H = rng.standard_normal((B * R, cfg.d), dtype=np.float32)
    H[1, 5] = np.nan  # request 0, row 1
    Hd = to_dev(gen.encode(H, "f32"))
    temps = torch.zeros(B, dtype=torch.float32, device=dev())
    k = to_dev(np.full(B, R - 1, dtype=np.int32))
    drafts = to_dev(np.ones((B, R - 1), dtype=np.int32))
    out = _pair(W, spec.SPEC_F32, cfg.V, cfg.d, Hd, B, R, temps, R - 1, k, drafts, -1)
    assert out[0] == out[1]
    o = np.frombuffer(out[1][0], dtype=spec.ACCEPT_OUT_DTYPE)
    assert o[0]["status"] == spec.REQ_NONFINITE and o[1]["status"] == 0


@pytest.fixture(scope="module")
def full():
    ensure_built()
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    return cfg, W


@pytest.mark.parametrize("R", [2, 8])
def test_fused_greedy_full_size_bf16(full, R):
    """bf16 LM head at full size (V = 151,936, d = 2560): the headline 2-row shape and 8 rows."""
    cfg, W = full
    Wd = torch.from_numpy(W.view(np.int16)).to(dev())
    rng = np.random.default_rng(10 + R)
    Hs = [torch.from_numpy(gen.encode(rng.standard_normal((R, cfg.d), dtype=np.float32),
                                      "bf16").view(np.int16)).to(dev()) for _ in range(2)]
    temps = [torch.zeros(1, dtype=torch.float32, device=dev())]
    assert _check_cases(Wd, spec.SPEC_BF16, cfg.V, cfg.d, Hs, 1, R, R - 1, rng, temps) > 0


def test_fused_greedy_full_size_q4(full):
    """4-bit LM head at full size, two requests of two rows."""
    cfg, W = full
    Wq = to_dev(gen.q4_weights(cfg))
    rng = np.random.default_rng(21)
    B, R = 2, 2
    Hs = [torch.from_numpy(gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32),
                                      "bf16").view(np.int16)).to(dev()) for _ in range(2)]
    temps = [torch.zeros(B, dtype=torch.float32, device=dev())]
    assert _check_cases(Wq, spec.SPEC_Q4A32, cfg.V, cfg.d, Hs, B, R, R - 1, rng, temps) > 0


def test_fused_width_update_matches_the_width_kernel():
    """30 cycles at the tiny configuration, one request of 4 rows: the fused launch with the
    width update (state set) against the fused launch without it followed by
    spec_adapt_width_mirror, each path with its own buffers. Records, counters, width state,
    next widths and the mirror bitwise equal after every cycle; the widths each path runs come
    from its own updates; cycle costs given (the cost fit in use), so both are deterministic."""
    ensure_built()
    cfg = configs.get(0)
    W = to_dev(gen.lm_weights(cfg))
    rng = np.random.default_rng(41)
    B, k_max = 1, 3
    R = k_max + 1
    cost = torch.tensor([1.0 + 0.3 * i for i in range(k_max + 1)], dtype=torch.float32,
                        device=dev())
    temps = torch.zeros(B, dtype=torch.float32, device=dev())
    paths = []
    for _ in range(2):
        paths.append(dict(
            ws=workspace(cfg.V, B),
            stats=torch.zeros(B * R * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev()),
            out=torch.zeros(B * spec.ACCEPT_OUT_BYTES, dtype=torch.uint8, device=dev()),
            cnt=torch.zeros(B * spec.COUNTERS_BYTES, dtype=torch.uint8, device=dev()),
            state=torch.zeros(B * spec.WIDTH_STATE_BYTES, dtype=torch.uint8, device=dev()),
            k=torch.full((B,), 1, dtype=torch.int32, device=dev()),
            mirror=torch.full((B,), -5, dtype=torch.int32, device=dev())))
    for c in range(30):
        H = to_dev(gen.encode(rng.standard_normal((R, cfg.d), dtype=np.float32), "f32"))
        am = _argmax(W, spec.SPEC_F32, cfg.V, cfg.d, H, B, R, temps)
        depth = int(rng.integers(0, R))
        drafts = to_dev(np.array([[am[0, i] if i < depth else (am[0, i] + 7) % cfg.V
                                   for i in range(k_max)]], dtype=np.int32))
        cyc = torch.tensor([100.0 + 40.0 * int(to_np(paths[0]["k"])[0]) + float(c % 5)],
                           dtype=torch.float32, device=dev())
        for fused_update, q in zip((False, True), paths):
            spec.spec_verify_accept_greedy(
                W, spec.SPEC_F32, cfg.V, cfg.d, H, B, R, temps, None, q["stats"], k_max, q["k"],
                drafts, -1, q["out"], q["cnt"], q["ws"], cost=cost if fused_update else None,
                cycle_cost=cyc if fused_update else None, alpha=0.2,
                state=q["state"] if fused_update else None,
                k_next=q["k"] if fused_update else None,
                k_mirror=q["mirror"] if fused_update else None)
            if not fused_update:
                spec.spec_adapt_width_mirror(B, k_max, q["out"], q["k"], cost, cyc, 0.2,
                                             q["state"], q["k"], q["mirror"])
        torch.cuda.synchronize()
        for key in ("out", "cnt", "state", "k", "mirror"):
            assert to_np(paths[0][key]).tobytes() == to_np(paths[1][key]).tobytes(), (c, key)
    st = to_np(paths[1]["state"]).view(spec.WIDTH_STATE_DTYPE)[0]
    assert int(st["cycles"]) == 30 and float(st["rate"][0]) > 0  # the fit in use
