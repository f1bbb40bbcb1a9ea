"""spec_lmhead_verify_noalloc: the verify LM head for callers that cannot allocate device
memory (a plugin handed only pre-allocated tensors by a framework that owns the memory budget,
or code that must not risk an allocation's implicit synchronisation). It takes no workspace and
uses a fixed scratch array inside the library instead.

Checked through the C ABI against spec_lmhead_verify (which uses a caller-allocated workspace)
on the same inputs, within the tolerances the other parity tests use, on two calls in a row (the
second call reuses the scratch the first one left behind). The file is named to be collected
last, and each test builds all of its own buffers, so it passes alone in a fresh process and
after the other tests.
"""

import numpy as np
import pytest

from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import close, dev, ensure_built, to_dev, to_np, wdt_of, workspace, ws_error, \
    zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


def _both(cfg, Wd, H, B, R, temps):
    """Run the allocating and the allocation-free entry points on the same inputs."""
    t = torch.tensor(temps, dtype=torch.float32, device=dev())
    Hd = to_dev(H)
    ref_l = torch.full((B * R, cfg.V), float("nan"), device=dev())
    ref_s = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    ws = workspace(cfg.V, B)
    spec.spec_lmhead_verify(Wd, wdt_of(cfg), cfg.V, cfg.d, Hd, B, R, t, ref_l, ref_s, ws)
    na_l = torch.full((B * R, cfg.V), float("nan"), device=dev())
    na_s = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    spec.spec_lmhead_verify_noalloc(Wd, wdt_of(cfg), cfg.V, cfg.d, Hd, B, R, t, na_l, na_s)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    return (to_np(ref_l), to_np(ref_s, spec.ROWSTATS_DTYPE), to_np(na_l),
            to_np(na_s, spec.ROWSTATS_DTYPE))


def _check(ref_l, ref_s, na_l, na_s, temps, R):
    for q in range(ref_s.shape[0]):
        if temps[q // R] > 0:
            ok, _ = close(na_l[q], ref_l[q])
            assert ok.all(), q
        else:
            assert np.isnan(na_l[q]).all()  # greedy rows stay untouched, as in the original
        assert na_s[q]["argmax"] == ref_s[q]["argmax"]
        for f in ("max", "log_norm", "gap"):
            a, b = float(na_s[q][f]), float(ref_s[q][f])
            assert (np.isinf(a) and np.isinf(b)) or abs(a - b) <= 2e-2 * abs(b) + 1e-6, (q, f)


@pytest.mark.parametrize("cfg_index", [0, 1])
def test_noalloc_matches_workspace_entry_point_two_calls(cfg_index):
    ensure_built()
    cfg = configs.get(cfg_index)
    W = gen.lm_weights(cfg)
    Wd = to_dev(W)
    assert spec.spec_noalloc_scratch_bytes() == 128 * 1024
    rng = np.random.default_rng(77 + cfg_index)
    for call, (B, R, temps) in enumerate([(1, 8, [1.0]), (2, 3, [0.0, 0.7])]):
        if cfg.plant_scale > 0:
            H, _, _ = gen.planted_rows(cfg, W, B * R, rng)
        else:
            H = gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), cfg.wdtype)
        ref_l, ref_s, na_l, na_s = _both(cfg, Wd, H, B, R, temps)
        _check(ref_l, ref_s, na_l, na_s, temps, R)


def test_noalloc_rejects_vocabularies_beyond_its_scratch():
    ensure_built()
    dummy = torch.zeros(64, dtype=torch.int16, device=dev())
    stats = zeros_bytes(spec.ROWSTATS_BYTES)
    t = torch.ones(1, device=dev())
    with pytest.raises(spec.SpecError) as e:
        spec.spec_lmhead_verify_noalloc(dummy, spec.SPEC_BF16, (1 << 24) - 1, 64, dummy, 1, 1, t,
                                        None, stats)
    assert e.value.status == 2  # SPEC_ERR_UNSUPPORTED: validated before any launch
