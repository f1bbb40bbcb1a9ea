"""spec_lmhead_verify_noalloc: the verify LM head for callers that cannot allocate device
memory (a plugin handed only pre-allocated tensors by a framework that owns the memory budget,
or code that must not risk an allocation's implicit synchronisation). It takes no workspace and
uses a fixed scratch array inside the library instead.

Checked through the C ABI against spec_lmhead_verify (which uses a caller-allocated workspace)
on the same inputs for the fp32, bf16 and 4-bit heads: the statistics and logits must be
bitwise equal, since the same kernel runs behind both, and the error word read back through
spec_noalloc_error_word must be zero, on two calls in a row (the second call reuses the scratch
the first one left behind). The file is named to be collected last, and each test builds all
of its own buffers, so it passes alone in a fresh process and after the other tests.
"""

import numpy as np
import pytest

from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, wdt_of, workspace, ws_error, \
    zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


def _noalloc_error():
    """The allocation-free entry point's error word, read through the C ABI."""
    err = torch.full((1,), -1, dtype=torch.int32, device=dev())
    spec.spec_noalloc_error_word(err)
    torch.cuda.synchronize()
    return int(to_np(err).view(np.uint32)[0])


def _both(cfg, Wd, wdt, H, B, R, temps):
    """Run the allocating and the allocation-free entry points on the same inputs."""
    t = torch.tensor(temps, dtype=torch.float32, device=dev())
    Hd = to_dev(H)
    ref_l = torch.full((B * R, cfg.V), float("nan"), device=dev())
    ref_s = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    ws = workspace(cfg.V, B)
    spec.spec_lmhead_verify(Wd, wdt, cfg.V, cfg.d, Hd, B, R, t, ref_l, ref_s, ws)
    na_l = torch.full((B * R, cfg.V), float("nan"), device=dev())
    na_s = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    spec.spec_lmhead_verify_noalloc(Wd, wdt, cfg.V, cfg.d, Hd, B, R, t, na_l, na_s)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    assert _noalloc_error() == 0
    return to_np(ref_l), to_np(ref_s), to_np(na_l), to_np(na_s)


@pytest.mark.parametrize("case", ["fp32", "bf16", "4-bit"])
def test_noalloc_matches_workspace_entry_point_two_calls(case):
    """The same kernel runs behind both entry points, so their outputs are bitwise equal; the
    second call reuses the scratch the first one left behind."""
    ensure_built()
    cfg = configs.get(0 if case == "fp32" else 1)
    W = gen.lm_weights(cfg)
    if case == "4-bit":
        Wd, wdt = to_dev(gen.q4_weights(cfg)), spec.SPEC_Q4A32
    else:
        Wd, wdt = to_dev(W), wdt_of(cfg)
    assert spec.spec_noalloc_scratch_bytes() == 128 * 1024
    rng = np.random.default_rng(77 + len(case))
    for call, (B, R, temps) in enumerate([(1, 8, [1.0]), (2, 3, [0.0, 0.7])]):
        if cfg.plant_scale > 0:
            H, _, _ = gen.planted_rows(cfg, W, B * R, rng)
        else:
            H = gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), cfg.wdtype)
        ref_l, ref_s, na_l, na_s = _both(cfg, Wd, wdt, H, B, R, temps)
        assert na_s.tobytes() == ref_s.tobytes(), (case, call)
        # NaN-filled rows of greedy requests stay untouched by both: compare the bit patterns
        assert na_l.view(np.uint32).tobytes() == ref_l.view(np.uint32).tobytes(), (case, call)
        if B == 2:  # request 0 is greedy (rows untouched), request 1 at T = 0.7 (written)
            assert np.isnan(na_l[:R]).all() and np.isfinite(na_l[R:]).all()


def test_noalloc_rejects_vocabularies_beyond_its_scratch():
    ensure_built()
    dummy = torch.zeros(64, dtype=torch.int16, device=dev())
    stats = zeros_bytes(spec.ROWSTATS_BYTES)
    t = torch.ones(1, device=dev())
    with pytest.raises(spec.SpecError) as e:
        spec.spec_lmhead_verify_noalloc(dummy, spec.SPEC_BF16, (1 << 24) - 1, 64, dummy, 1, 1, t,
                                        None, stats)
    assert e.value.status == 2  # SPEC_ERR_UNSUPPORTED: validated before any launch
