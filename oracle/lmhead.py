"""LM-head logits and per-row statistics (oracle; test infrastructure only).

The verify step projects the k+1 verify rows through the shared LM head in one batched pass
(lucebox-hub PR #15 "MTP speculative decoding", section *What*: all drafts are checked by a
single batched trunk forward); the draft head is the same projection restricted to the first
64,000 vocabulary rows (same page and section). A logit
is a plain dot product, so the oracle is that definition in float64:

    z[r, v] = sum_j H[r, j] * W[v, j]

Inputs arrive as bf16 bit patterns (uint16) or float32 and are widened exactly to float64, so
every product is exact and the float64 sum carries a relative error of at most
d * 2^-53 * sum|W*H| -- far inside any fp32 tolerance. The loop over blocks of vocabulary rows
exists only to bound host memory; each logit is still one independent dot product.

Row statistics are the quantities the acceptance rule reads:

    max       = max_v z[v]
    argmax    = the lowest v with z[v] == max           (ties: lowest index)
    gap       = max - (largest z[v] over v != argmax)     (top-2 gap; +inf when V == 1)
    log_norm  = log sum_v exp((z[v] - max) / T)           (T == 0 uses T = 1)
    nonfinite = any z[v] is NaN or +Inf

and the temperature-T distribution is p[v] = exp((z[v] - max) / T - log_norm) (DS4Server issue
#98, *Implementation*: "probability-ratio acceptance ... for official non-greedy sampling";
temperature 0 means greedy).

Pinned by: exact integer dot products (small-integer bf16 inputs), scipy.special.logsumexp and
softmax, closed forms for constant and one-hot rows, and brute-force argmax/second-max.
"""

import numpy as np

_BLOCK_ROWS = 8192


def bf16_to_f64(bits):
    """Widen bf16 bit patterns (uint16 array) to float64 exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_f64(x):
    """Widen a bf16 (uint16 bit pattern) or float32/float64 array to float64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


def logits(W, H, rows=None):
    """z = H @ W[rows].T in float64.

    W: [V, d] bf16 bits (uint16) or float32. H: [R, d] same encoding. ``rows`` restricts the
    projection to vocabulary rows [0, rows) (the draft head). Returns float64 [R, rows or V].
    """
    Hf = to_f64(H)
    if Hf.ndim == 1:
        Hf = Hf[None, :]
    V = W.shape[0] if rows is None else int(rows)
    out = np.empty((Hf.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, _BLOCK_ROWS):
        v1 = min(V, v0 + _BLOCK_ROWS)
        Wb = to_f64(W[v0:v1])
        out[:, v0:v1] = Hf @ Wb.T
    return out


def logit(W, H_row, v):
    """One logit z[v] for one hidden row, computed alone (for sampled checks at full size)."""
    return float(np.dot(to_f64(W[v]), to_f64(H_row)))


def row_stats(z, T):
    """Statistics of one logit row (float64 [V]) at temperature T (see module docstring)."""
    z = np.asarray(z, dtype=np.float64)
    nonfinite = bool(np.any(np.isnan(z)) or np.any(np.isposinf(z)))
    if nonfinite or z.size == 0:
        return dict(max=float("nan"), argmax=-1, gap=float("nan"), log_norm=float("nan"),
                    nonfinite=True)
    mx = float(np.max(z))
    if mx == -np.inf:  # every token has probability zero: no distribution
        return dict(max=mx, argmax=0, gap=0.0, log_norm=float("nan"), nonfinite=True)
    am = int(np.flatnonzero(z == mx)[0])
    if z.size > 1:
        rest = np.concatenate([z[:am], z[am + 1:]])
        gap = mx - float(np.max(rest))
    else:
        gap = float("inf")
    Teff = T if T > 0 else 1.0
    log_norm = float(np.log(np.sum(np.exp((z - mx) / Teff))))
    return dict(max=mx, argmax=am, gap=gap, log_norm=log_norm, nonfinite=False)


def probs(z, T):
    """p[v] = exp((z[v] - max)/T - log_norm), the temperature-T distribution of one row (T > 0)."""
    st = row_stats(z, T)
    z = np.asarray(z, dtype=np.float64)
    return np.exp((z - st["max"]) / T - st["log_norm"])


def fp32_abs_bound(W, H):
    """Rigorous bound on |fp32 logit - exact logit| for any summation order (elementwise).

    For a sum of d exactly-representable products accumulated in float32, the error is at
    most (d - 1) * 2^-24 * sum_j |W[v,j] * H[r,j]| (standard recursive-summation bound; the
    products of bf16 values are exact in fp32). Returns float64 [R, V].
    """
    Hf = np.abs(to_f64(H))
    if Hf.ndim == 1:
        Hf = Hf[None, :]
    d = Hf.shape[1]
    V = W.shape[0]
    out = np.empty((Hf.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, _BLOCK_ROWS):
        v1 = min(V, v0 + _BLOCK_ROWS)
        out[:, v0:v1] = Hf @ np.abs(to_f64(W[v0:v1])).T
    return (d - 1) * 2.0 ** -24 * out
