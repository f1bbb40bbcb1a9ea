"""Seeded synthetic inputs for the verify step: the only module both the CUDA path's tests and
the oracle's tests consume. It holds workload shapes and random-input recipes -- no logits,
softmax, acceptance, sampling or commit arithmetic.

All data come from numpy's PCG64 with fixed seeds (weights, hidden rows, drafts injected by
tests, state buffers); the method's own random draws are Philox uniforms that each side
computes from the published definition.
"""

from .configs import CONFIGS, Config, get  # noqa: F401
from . import gen  # noqa: F401
