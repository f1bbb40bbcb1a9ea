"""Pins of the 4-bit affine LM-head oracle (oracle/quant.py) against what does not depend on
it: torch's float32 -> bfloat16 rounding, hand-derived ties and overflow, a hand-packed code
word, closed forms of the dequantised values, and exact integer dot products."""

import numpy as np
import pytest

from oracle import lmhead, quant

torch = pytest.importorskip("torch")


def _row(q, s_bits, b_bits):
    """One row in the documented layout, packed here by hand (words built code by code)."""
    d = len(q)
    words = []
    for w in range(d // 8):
        e = q[8 * w:8 * w + 8]
        x = 0
        for i in range(4):
            x |= int(e[2 * i]) << (4 * i)
            x |= int(e[2 * i + 1]) << (16 + 4 * i)
        words.append(x)
    codes = b"".join(x.to_bytes(4, "little") for x in words)
    sb = b"".join(int(s).to_bytes(2, "little") + int(b).to_bytes(2, "little")
                  for s, b in zip(s_bits, b_bits))
    return np.frombuffer(codes + sb, dtype=np.uint8)


def test_rounding_matches_torch_bfloat16():
    """Values exactly representable in float32 (so torch's float32 -> bfloat16 conversion is
    itself a single rounding), spanning normal, subnormal and near-overflow magnitudes."""
    rng = np.random.default_rng(0)
    mant = rng.integers(1 << 23, 1 << 24, 20000)
    expo = rng.integers(-150, 105, 20000)
    x = np.ldexp(mant.astype(np.float64), expo) * rng.choice([-1.0, 1.0], 20000)
    x = x[np.isfinite(x.astype(np.float32)) & (x.astype(np.float32).astype(np.float64) == x)]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert (quant.bf16_rne(x) == ref.view(np.uint16)).all()


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (1.0 + 2.0 ** -8, 0x3F80),                  # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                              # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),                     # just above the tie
    (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000),
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),                     # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),                     # halfway to 2^128 -> inf
    (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),               # smallest subnormal; tie -> 0
    (3 * 2.0 ** -134, 0x0002), (float("inf"), 0x7F80),
])
def test_rounding_hand_cases(x, bits):
    assert int(quant.bf16_rne(np.array([x]))[0]) == bits


def test_code_layout_hand_packed_word():
    """Codes 1..8 of elements 0..7: the low half holds 1, 3, 5, 7 and the high half 2, 4, 6, 8,
    so the word is 0x86427531, stored as bytes 31 75 42 86."""
    q = quant.unpack_codes(np.frombuffer(bytes.fromhex("31754286"), dtype=np.uint8), 8)
    assert list(q) == [1, 2, 3, 4, 5, 6, 7, 8]
    rng = np.random.default_rng(1)
    qq = rng.integers(0, 16, 256)
    row = _row(qq, [0x3F80] * 8, [0] * 8)
    assert (quant.unpack_codes(row[:128], 256) == qq).all()


def test_dequantise_closed_forms():
    d = 128
    q = np.arange(d) % 16
    # s = 0.5, b = -2: w = q/2 - 2, exact
    row = _row(q, [0x3F00] * 4, [0xC000] * 4)
    w = lmhead.bf16_to_f64(quant.dequantise(row[None, :], d)[0])
    assert (w == q / 2 - 2).all()
    # s = 2^-10, b = 1: w = 1 + q/1024 rounded to the bf16 grid of [1, 2) (spacing 1/128): the
    # multiple of 8/1024 nearest to q/1024, ties (q = 4, 12) to the even multiple
    row = _row(q, [0x3A80] * 4, [0x3F80] * 4)
    w = lmhead.bf16_to_f64(quant.dequantise(row[None, :], d)[0])
    want = 1 + np.array([{4: 0, 12: 16}.get(int(x), 8 * round(x / 8)) for x in q]) / 1024
    assert (w == want).all()
    # each group has its own pair: group g scaled by 2^g, biased by -g
    s_bits = [0x3F80 + (g << 7) for g in range(4)]
    b_bits = [int(quant.bf16_rne(np.array([-float(g)]))[0]) for g in range(4)]
    row = _row(q, s_bits, b_bits)
    w = lmhead.bf16_to_f64(quant.dequantise(row[None, :], d)[0])
    g = np.arange(d) // 32
    assert (w == q * 2.0 ** g - g).all()


def test_logits_integer_dot_products():
    """s = 1, b = 0: the weights are the codes, and with integer H every logit is an exact
    integer dot product."""
    rng = np.random.default_rng(2)
    V, d = 40, 256
    Q = rng.integers(0, 16, (V, d))
    Wq = np.stack([_row(Q[v], [0x3F80] * (d // 32), [0] * (d // 32)) for v in range(V)])
    Hi = rng.integers(-8, 9, (3, d))
    H = (Hi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # small ints: exact
    z = quant.logits(Wq, d, H)
    assert (z == (Hi @ Q.T).astype(np.float64)).all()
    assert quant.logit(Wq, d, H[1], 7) == float(Hi[1] @ Q[7])
    assert (quant.logits(Wq, d, H, rows=10) == z[:, :10]).all()


def test_planted_mistakes_fail_the_pins():
    """A layout read as plain nibble order, or a bias dropped, fails the pins above."""
    word = np.frombuffer(bytes.fromhex("31754286"), dtype=np.uint8)
    plain = [(int(b) >> (4 * h)) & 0xF for b in word for h in (0, 1)]
    assert plain != [1, 2, 3, 4, 5, 6, 7, 8]
    q = np.arange(128) % 16
    row = _row(q, [0x3F00] * 4, [0xC000] * 4)
    s, b = quant.scales_biases(row[None, :], 128)
    assert not (np.repeat(s, 32) * q == q / 2 - 2).all()


def test_generator_packs_the_documented_layout():
    """The synthetic quantiser's rows unpack to its own codes and pairs under the oracle's
    reading of the layout, and the dequantised matrix stays within half a step of the source."""
    from synth import gen
    rng = np.random.default_rng(3)
    W = gen.f32_to_bf16(rng.standard_normal((64, 256), dtype=np.float32) * np.float32(0.02))
    Wq = gen.q4_quantise(W)
    assert Wq.shape == (64, quant.row_bytes(256))
    s, b = quant.scales_biases(Wq, 256)
    w = lmhead.bf16_to_f64(quant.dequantise(Wq, 256))
    src = lmhead.to_f64(W)
    step = np.repeat(s, 32, axis=-1)
    assert (np.abs(w - src) <= 0.5 * step + 2.0 ** -8 * np.abs(src) + 1e-12).all()
    assert (quant.unpack_codes(Wq[:, :128], 256) <= 15).all()
