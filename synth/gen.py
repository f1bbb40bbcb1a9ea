"""Seeded generators for weights, hidden rows, drafts and state buffers (no method arithmetic).

Encodings: bf16 tensors are numpy uint16 bit patterns (round-to-nearest-even from float32);
fp32 tensors are float32; KV buffers are raw bytes (uint8). The CUDA tests copy these arrays
to the device unchanged, and the oracle widens them to float64 itself.
"""

import numpy as np

W_STD = 0.02
_W_CACHE = {}


def f32_to_bf16(x):
    """float32 -> bf16 bit patterns, round to nearest even (NaN -> canonical quiet NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    out = ((u + bias) >> np.uint64(16)).astype(np.uint16)
    out[np.isnan(x)] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits):
    """bf16 bit patterns -> float32 (exact); input construction only (e.g. noise on rows)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(x):
    x = np.asarray(x)
    return bf16_to_f32(x) if x.dtype == np.uint16 else x.astype(np.float32)


def encode(x32, wdtype):
    return f32_to_bf16(x32) if wdtype == "bf16" else np.ascontiguousarray(x32, dtype=np.float32)


def lm_weights(cfg, seed=0, cache=True):
    """LM-head weights [V, d] ~ N(0, 0.02^2), bf16 bits or float32 per ``cfg.wdtype``."""
    key = (cfg.V, cfg.d, cfg.wdtype, seed)
    if cache and key in _W_CACHE:
        return _W_CACHE[key]
    rng = np.random.default_rng(seed)
    dt = np.uint16 if cfg.wdtype == "bf16" else np.float32
    W = np.empty((cfg.V, cfg.d), dtype=dt)
    step = 16384
    for v0 in range(0, cfg.V, step):
        v1 = min(cfg.V, v0 + step)
        blk = rng.standard_normal((v1 - v0, cfg.d), dtype=np.float32) * np.float32(W_STD)
        W[v0:v1] = encode(blk, cfg.wdtype)
    if cache:
        _W_CACHE[key] = W
    return W


def planted_rows(cfg, W, n, rng, force=None):
    """n trunk hidden rows: g ~ N(0, I), plus s * W[t]/|W[t]| for a planted target t when
    ``cfg.plant_scale`` > 0 (t from the draft rows with probability pi_draft). ``force`` maps
    row -> token to plant instead of the drawn one (the draws are made all the same, so the
    other rows do not change). Returns (rows encoded like W, float32 copy, targets or -1)."""
    g = rng.standard_normal((n, cfg.d), dtype=np.float32)
    targets = np.full(n, -1, dtype=np.int64)
    if cfg.plant_scale > 0:
        in_draft = rng.random(n) < cfg.pi_draft
        t_draft = rng.integers(0, cfg.Vd, n)
        t_rest = rng.integers(cfg.Vd, cfg.V, n)
        targets = np.where(in_draft, t_draft, t_rest)
        for r, tok in (force or {}).items():
            targets[r] = tok
        Wt = as_f32(W[targets])
        norms = np.linalg.norm(Wt.astype(np.float64), axis=1).astype(np.float32)
        g = g + np.float32(cfg.plant_scale) * Wt / norms[:, None]
    enc = encode(g, cfg.wdtype)
    return enc, as_f32(enc), targets


def noisy_rows(rows32, sigma, wdtype, rng):
    """Draft-head hidden rows: trunk rows plus N(0, sigma^2) noise, encoded like the weights."""
    noise = rng.standard_normal(rows32.shape, dtype=np.float32) * np.float32(sigma)
    return encode(rows32 + noise, wdtype)


def cycle_inputs(cfg, W, cycle, seed=0, k=None, eos_at=0):
    """Inputs of one verify cycle for one request.

    Returns dict(H [k+1, d] verify rows, Hd [k, d] draft-head rows, k, targets). Draft i uses
    verify row i-1 plus noise (draft i predicts the position verify row i-1 predicts).
    eos_at = j > 0 injects the EOS id at proposal position j: verify row j-1 (and so the draft
    row derived from it) is planted on ``cfg.eos_id``; callers that need the proposal itself to
    be EOS also force draft j (``eos_injection`` says which cycles and where)."""
    rng = np.random.default_rng([seed, cycle, 0xC1C1E])
    if k is None:
        k = cfg.k if cfg.k_mode == "fixed" else int(rng.integers(1, cfg.k + 1))
    force = {eos_at - 1: cfg.eos_id} if 0 < eos_at <= k else None
    H, H32, targets = planted_rows(cfg, W, k + 1, rng, force=force)
    Hd = noisy_rows(H32[:k], cfg.draft_noise, cfg.wdtype, rng) if k > 0 else H[:0]
    return dict(H=H, Hd=Hd, k=k, targets=targets)


def eos_injection(cfg, cycle, k, seed=0):
    """Position (1..k) at which a test forces the EOS id into the drafts, or 0 for none."""
    rng = np.random.default_rng([seed, cycle, 0xE05])
    if k > 0 and rng.random() < cfg.eos_inject:
        return int(rng.integers(1, k + 1))
    return 0


def state_inputs(cfg, k, seed=0, capacity=None, P=None, n_slots=None):
    """State buffers for one request and one cycle with k drafts (k+1 verify rows).

    Returns dict with: kv_pre (uint8 [layers, 2, cap, row_bytes], random rows below P, zeros
    at and past P), kv_rows (uint8 [k+1, layers, 2, row_bytes], what each verify row writes),
    P, S0 [L,H,dk,dv] f32, conv0 [L,C,W] f32, and per-row step inputs a [R,L,H], b [R,L,H,dk],
    c [R,L,H,dv], x [R,L,W] (R = n_slots - 1 rows, zero past k+1)."""
    rng = np.random.default_rng([seed, k, 0x57A7E])
    cap = cfg.kv_capacity if capacity is None else capacity
    P = cfg.context if P is None else P
    L, nh, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
    R = (k + 1) if n_slots is None else n_slots - 1
    rb = cfg.kv_row_bytes
    kv_pre = np.zeros((cfg.kv_layers, 2, cap, rb), dtype=np.uint8)
    kv_pre[:, :, :P, :] = rng.integers(0, 256, (cfg.kv_layers, 2, P, rb), dtype=np.uint8)
    kv_rows = rng.integers(0, 256, (R, cfg.kv_layers, 2, rb), dtype=np.uint8)
    S0 = rng.standard_normal((L, nh, dk, dv), dtype=np.float32)
    conv0 = rng.standard_normal((L, cfg.conv_rows, cfg.conv_width), dtype=np.float32)
    a = rng.uniform(0.9, 1.0, (R, L, nh)).astype(np.float32)
    b = (rng.standard_normal((R, L, nh, dk), dtype=np.float32) * np.float32(0.1))
    c = (rng.standard_normal((R, L, nh, dv), dtype=np.float32) * np.float32(0.1))
    x = rng.standard_normal((R, L, cfg.conv_width), dtype=np.float32)
    for arr in (a, b, c, x):
        arr[k + 1:] = 0
    return dict(kv_pre=kv_pre, kv_rows=kv_rows, P=P, S0=S0, conv0=conv0, a=a, b=b, c=c, x=x)


def step_inputs(cfg, cycle, k, seed=0, n_slots=9):
    """Per-cycle inputs of a chained run of cycles (state evolving from one cycle to the next):
    what each of the cycle's verify rows writes into the KV cache and feeds the recurrent step.
    Returns dict kv_rows (uint8 [R, layers, 2, row_bytes]), a [R,L,H], b [R,L,H,dk],
    c [R,L,H,dv], x [R,L,W] with R = n_slots - 1 rows, zero past the k+1 rows of the cycle
    (same distributions as ``state_inputs``)."""
    rng = np.random.default_rng([seed, cycle, 0x5E9])
    L, nh, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
    R = n_slots - 1
    kv_rows = rng.integers(0, 256, (R, cfg.kv_layers, 2, cfg.kv_row_bytes), dtype=np.uint8)
    a = rng.uniform(0.9, 1.0, (R, L, nh)).astype(np.float32)
    b = rng.standard_normal((R, L, nh, dk), dtype=np.float32) * np.float32(0.1)
    c = rng.standard_normal((R, L, nh, dv), dtype=np.float32) * np.float32(0.1)
    x = rng.standard_normal((R, L, cfg.conv_width), dtype=np.float32)
    for arr in (kv_rows, a, b, c, x):
        arr[k + 1:] = 0
    return dict(kv_rows=kv_rows, a=a, b=b, c=c, x=x)


def tagged(base, tag):
    """A float32 array with the bits of ``base`` XOR (tag + 1) * 16 in every word: a cheap way to
    give many state snapshots contents that differ from each other in every element (tag <
    2^18 keeps the change inside the significand, so finite inputs stay finite)."""
    bits = np.ascontiguousarray(base, dtype=np.float32).view(np.uint32)
    return (bits ^ np.uint32((int(tag) + 1) << 4)).view(np.float32)


_Q4_CACHE = {}


def q4_pack(q, s_bits, b_bits):
    """4-bit codes q [V, d] (0..15) and bf16 scale / bias bits [V, d/32] -> rows of 5d/8 bytes:
    d/2 bytes of codes (in each little-endian 32-bit word of 8 consecutive codes e0..e7, e_{2i}
    in bits 4i..4i+3 and e_{2i+1} in bits 16+4i..16+4i+3), then the (scale, bias) pairs."""
    q = np.asarray(q, dtype=np.uint32)
    V, d = q.shape
    e = q.reshape(V, d // 8, 8)
    words = np.zeros((V, d // 8), dtype=np.uint32)
    for i in range(4):
        words |= e[:, :, 2 * i] << np.uint32(4 * i)
        words |= e[:, :, 2 * i + 1] << np.uint32(16 + 4 * i)
    sb = np.stack([np.asarray(s_bits, np.uint16), np.asarray(b_bits, np.uint16)], axis=-1)
    out = np.empty((V, 5 * d // 8), dtype=np.uint8)
    out[:, :d // 2] = words.astype("<u4").view(np.uint8).reshape(V, d // 2)
    out[:, d // 2:] = sb.astype("<u2").view(np.uint8).reshape(V, d // 8)
    return out


def q4_quantise(W):
    """Min/max affine quantisation of weights [V, d] (bf16 bits or float32) in groups of 32:
    s = bf16((max - min) / 15), b = bf16(min), q = clip(rint((w - b) / s), 0, 15). Input
    construction only: the quantised matrix is the workload, however it was made."""
    w = as_f32(W)
    V, d = w.shape
    g = w.reshape(V, d // 32, 32)
    lo, hi = g.min(axis=-1), g.max(axis=-1)
    s_bits = f32_to_bf16((hi - lo) / np.float32(15))
    b_bits = f32_to_bf16(lo)
    s, b = bf16_to_f32(s_bits)[..., None], bf16_to_f32(b_bits)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, np.rint((g - b) / np.where(s > 0, s, 1)), 0)
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(V, d)
    return q4_pack(q, s_bits, b_bits)


def q4_weights(cfg, seed=0, cache=True):
    """The bf16 LM head of ``cfg`` (lm_weights, same seed) quantised to 4-bit affine codes in
    groups of 32: [V, 5d/8] uint8. Planted hidden rows keep using the bf16 matrix."""
    key = (cfg.V, cfg.d, seed)
    if cache and key in _Q4_CACHE:
        return _Q4_CACHE[key]
    from dataclasses import replace
    W = lm_weights(replace(cfg, wdtype="bf16"), seed=seed, cache=cache)
    out = np.empty((cfg.V, 5 * cfg.d // 8), dtype=np.uint8)
    step = 16384
    for v0 in range(0, cfg.V, step):
        out[v0:v0 + step] = q4_quantise(W[v0:v0 + step])
    if cache:
        _Q4_CACHE[key] = out
    return out
