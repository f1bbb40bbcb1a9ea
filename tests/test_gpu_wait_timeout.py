"""Failure detection without a GPU fault: a bounded wait that runs out returns an error status
the host reads, and the GPU stays usable.

spec_test_verify_stalled runs the fp32 verify LM head (the CUDA-core kernel: no tensor memory
to release) with a producer warp that issues no copy, so no bulk copy is ever in flight and the
consumers' waits for the first stage can only run out, after a 2 ms limit. The kernel must then
set the ring-wait bit of the workspace error word, finish, and leave the workspace counters at
zero; the ordinary call that follows, on a fresh workspace, must match the oracle.
"""

import numpy as np
import pytest

from oracle import lmhead as o_lm
from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import close, dev, ensure_built, to_dev, to_np, workspace, ws_error, zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402

ERR_GEMV_WAIT_FULL = 1  # bit 0 of the error word: a consumer's wait for a stage gave up


def test_stalled_producer_wait_runs_out_and_reports():
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    Wd = to_dev(W)
    rng = np.random.default_rng(5)
    H = gen.encode(rng.standard_normal((4, cfg.d), dtype=np.float32), cfg.wdtype)
    Hd = to_dev(H)
    t = torch.ones(1, dtype=torch.float32, device=dev())
    logits = torch.zeros((4, cfg.V), device=dev())
    stats = zeros_bytes(4 * spec.ROWSTATS_BYTES)
    ws = workspace(cfg.V, 1)
    spec.spec_test_verify_stalled(Wd, cfg.V, cfg.d, Hd, 1, 4, t, logits, stats, 2000, ws)
    torch.cuda.synchronize()  # the kernel returned: every wait ended
    assert ws_error(ws) & ERR_GEMV_WAIT_FULL
    assert int(to_np(ws[0:4]).view(np.uint32)[0]) == 0  # the cross-block ticket is back at 0

    # the next ordinary call, on a fresh workspace, is unaffected
    ws2 = workspace(cfg.V, 1)
    spec.spec_lmhead_verify(Wd, spec.SPEC_F32, cfg.V, cfg.d, Hd, 1, 4, t, logits, stats, ws2)
    torch.cuda.synchronize()
    assert ws_error(ws2) == 0
    z = o_lm.logits(W, H)
    ok, _ = close(to_np(logits), z, o_lm.fp32_abs_bound(W, H))
    assert ok.all()
    st = to_np(stats, spec.ROWSTATS_DTYPE)
    assert list(st["argmax"]) == [int(np.argmax(z[r])) for r in range(4)]


def test_stalled_call_validates_its_limit():
    ensure_built()
    dummy = torch.zeros(64, dtype=torch.float32, device=dev())
    ws = workspace(64, 1)
    with pytest.raises(spec.SpecError):
        spec.spec_test_verify_stalled(dummy, 8, 8, dummy, 1, 1, dummy, None, dummy, 0, ws)
