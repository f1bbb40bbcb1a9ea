"""4-bit affine LM-head weights with 32-value groups (oracle; test infrastructure only).

DS4Server issue #98, closing comment: the MTP head's weights are 4-bit affine values in groups
of 32; lucebox-hub PR #15 "MTP speculative decoding", *Speed*, and llama.cpp PR #28104,
*Result*, run the MTP head quantised as well (Q4_K_M, Q8_0). The pages name the format's
parameters, not its byte layout or how a kernel widens it, so this build fixes both.

Layout of one vocabulary row of d elements (d a multiple of 128): 5d/8 bytes.

* Bytes [0, d/2): the 4-bit codes q in 0..15. The codes of elements 8w .. 8w+7 (e0 .. e7) form
  the little-endian 32-bit word w. Code e_{2i} sits in bits 4i .. 4i+3 and e_{2i+1} in bits
  16+4i .. 16+4i+3 (i = 0..3), so each 16-bit half holds alternate elements.
* Bytes [d/2, 5d/8): one (scale, bias) pair per group g = 0 .. d/32 - 1, group g being
  elements 32g .. 32g+31: the bf16 scale s_g, then the bf16 bias b_g, each little-endian.

Every row carries its own scales, so the first Vd rows of the matrix are a complete matrix of
Vd rows. The draft head reads them exactly as the verify head reads all V.

Dequantised weight, this build's reading: w_j = bf16(s_g * q_j + b_g), the exact value
rounded once to bf16 (round to nearest, ties to even). The LM head computes in bf16 with fp32
accumulation, so with that rounding the quantised head's logits are a plain bf16 projection of
the dequantised matrix, z = H w^T. That projection's oracle (lmhead.logits) then applies as it
stands.

Pinned by: the rounding against torch's float32 -> bfloat16 conversion and hand-derived ties
and overflow; the code layout against a hand-packed word; dequantisation against closed forms;
logits against exact integer dot products (s = 1, b = 0, integer H).
"""

import numpy as np

from . import lmhead

GROUP = 32


def row_bytes(d):
    """Bytes per vocabulary row: d/2 of codes and d/8 of (scale, bias) pairs."""
    return 5 * d // 8


def bf16_rne(x):
    """float64 -> bf16 bit patterns, the exact value rounded once (ties to even; overflow to
    +-inf; bf16 subnormals kept; NaN -> 0x7FC0)."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # |x| = m 2^e with 0.5 <= m < 1
    ulp_exp = np.maximum(e - 8, -133)       # 8 significant bits; subnormal spacing 2^-133
    with np.errstate(invalid="ignore", over="ignore"):
        y = np.ldexp(np.rint(np.ldexp(x, -ulp_exp)), ulp_exp)  # np.rint: ties to even
        y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, x), y)
    bits = (y.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def unpack_codes(code_bytes, d):
    """Codes [..., d/2 bytes] -> q [..., d] (uint8, 0..15), following the word layout above."""
    b = np.ascontiguousarray(code_bytes, dtype=np.uint8)
    words = b.reshape(b.shape[:-1] + (d // 8, 4)).view("<u4")[..., 0]
    q = np.empty(b.shape[:-1] + (d // 8, 8), dtype=np.uint8)
    for i in range(4):
        q[..., 2 * i] = (words >> np.uint32(4 * i)) & np.uint32(0xF)
        q[..., 2 * i + 1] = (words >> np.uint32(16 + 4 * i)) & np.uint32(0xF)
    return q.reshape(b.shape[:-1] + (d,))


def scales_biases(Wq, d):
    """(s, b) as float64 [..., d/32] each, widened exactly from their bf16 bits."""
    sb = np.ascontiguousarray(Wq[..., d // 2:row_bytes(d)], dtype=np.uint8)
    pairs = sb.reshape(sb.shape[:-1] + (d // GROUP, 2, 2)).view("<u2")[..., 0]
    return lmhead.bf16_to_f64(pairs[..., 0]), lmhead.bf16_to_f64(pairs[..., 1])


def dequantise(Wq, d):
    """Wq [V, 5d/8] uint8 -> the dequantised weights [V, d] as bf16 bit patterns."""
    Wq = np.asarray(Wq, dtype=np.uint8)
    q = unpack_codes(Wq[..., :d // 2], d).astype(np.float64)
    s, b = scales_biases(Wq, d)
    s = np.repeat(s, GROUP, axis=-1)
    b = np.repeat(b, GROUP, axis=-1)
    with np.errstate(invalid="ignore", over="ignore"):
        # exact in float64 (8-bit s and b, 4-bit q) unless the exponents of s*q and b lie more
        # than 40 apart; then the smaller term is far below half a bf16 ulp of the larger and
        # the float64 rounding cannot change the bf16 result
        exact = s * q + b
    return bf16_rne(exact)


def logits(Wq, d, H, rows=None):
    """z = H w^T over the dequantised rows [0, rows or V), float64 (see module docstring)."""
    V = Wq.shape[0] if rows is None else int(rows)
    Hf = lmhead.to_f64(H)
    if Hf.ndim == 1:
        Hf = Hf[None, :]
    out = np.empty((Hf.shape[0], V), dtype=np.float64)
    step = 8192
    for v0 in range(0, V, step):
        v1 = min(V, v0 + step)
        out[:, v0:v1] = lmhead.logits(dequantise(Wq[v0:v1], d), H)
    return out


def logit(Wq, d, H_row, v):
    """One logit of one hidden row, computed alone (sampled checks at full size)."""
    w = lmhead.bf16_to_f64(dequantise(Wq[v:v + 1], d)[0])
    return float(np.dot(w, lmhead.to_f64(H_row)))
