"""Helpers for the GPU parity tests: device buffers, calls through the C ABI, host readback.

Only marshalling lives here: buffers are created from the seeded generators in ``synth``, the
CUDA library computes, and results come back as numpy arrays for comparison with ``oracle``.
"""

import numpy as np
import torch

import mtp_speculative_decoding_spec_gb300 as spec
from mtp_speculative_decoding_spec_gb300 import build as _build

# margins below which a decision is a near-tie, counted and reported separately
GAP_EPS = 1e-5     # top-2 logit gap (logit units)
RATIO_EPS = 1e-5   # |u*q(x) - p(x)| (probability units)
CDF_EPS = 1e-5     # distance from u*sum(w) to a cumulative boundary (probability units)

# logits and probabilities: 2e-2 relative, with an absolute floor (1e-6, or the rigorous fp32
# accumulation bound of the row when that is larger)
REL_TOL = 2e-2
ABS_TOL = 1e-6

_built = False


def ensure_built():
    global _built
    if not _built:
        _build.build()
        _built = True


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    """numpy array -> device tensor holding the same bytes."""
    a = np.ascontiguousarray(a)
    m = {np.uint16: torch.int16, np.uint64: torch.int64, np.uint32: torch.int32}
    t = torch.from_numpy(a.view(np.dtype(a.dtype.str.replace("u", "i"))) if a.dtype.type in m
                         else a)
    return t.to(dev())


def zeros_bytes(n):
    return torch.zeros(int(n), dtype=torch.uint8, device=dev())


def to_np(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(np.uint8).view(dtype)
    return a


def workspace(V, B):
    n = spec.spec_workspace_bytes(V, B)
    assert n > 0
    return torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device=dev())


def ws_error(ws):
    return int(to_np(ws[4:8]).view(np.uint32)[0])


def wdt_of(cfg):
    return spec.SPEC_BF16 if cfg.wdtype == "bf16" else spec.SPEC_F32


class Verifier:
    """Device-side buffers for one shape (V, d, rows) and calls of spec_lmhead_verify."""

    def __init__(self, W_dev, wdt, V, d, B, R, ws):
        self.W, self.wdt, self.V, self.d, self.B, self.R, self.ws = W_dev, wdt, V, d, B, R, ws
        self.logits = torch.empty((B * R, V), dtype=torch.float32, device=dev())
        self.stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)

    def run(self, H_dev, temps_dev, want_logits=True):
        spec.spec_lmhead_verify(self.W, self.wdt, self.V, self.d, H_dev, self.B, self.R, temps_dev,
                                self.logits if want_logits else None, self.stats, self.ws)

    def stats_np(self):
        return to_np(self.stats, spec.ROWSTATS_DTYPE)


def close(gpu, ref, bound=None, rel=REL_TOL, abs_=ABS_TOL):
    """Elementwise tolerance check; returns (ok mask, count passing only via the fp32 bound)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    base = rel * np.abs(ref) + abs_
    ok = err <= base
    via_bound = 0
    if bound is not None:
        ok2 = err <= rel * np.abs(ref) + np.maximum(abs_, bound)
        via_bound = int(np.sum(ok2 & ~ok))
        ok = ok2
    return ok, via_bound
