"""CPU checks of the byte-permute decodes the MXFP4 scores kernel uses, emulating PTX prmt.b32
(default mode) in Python: every E2M1 nibble times 2^X for X in [-13, 13] must come out as the
E5M2 byte of that value, and the E4M3 scale table must hold the values the format defines.
The expected values come from the oracle's E2M1 magnitudes and an independent E5M2 decoder."""
import numpy as np

import oracle


def prmt(a: int, b: int, c: int) -> int:
    """prmt.b32 d, a, b, c: byte i of d is byte (c >> 4i) & 7 of {b, a}; if bit 3 of that selector
    nibble is set, the selected byte's top bit is replicated over the whole byte."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    d = 0
    for i in range(4):
        sel = (c >> (4 * i)) & 0xF
        byte = src[sel & 7]
        if sel & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        d |= byte << (8 * i)
    return d


def e5m2_value(byte: int) -> float:
    s = -1.0 if byte & 0x80 else 1.0
    e, m = (byte >> 2) & 31, byte & 3
    if e == 0:
        return s * m / 4 * 2.0 ** -14
    return s * (1 + m / 4) * 2.0 ** (e - 15)


def e2m1x8_to_e5m2(cw: int, X: int) -> list[int]:
    """The kernel's conversion: magnitude table shifted by 4X, sign by a whole-nibble selector."""
    t0 = (0x3E3C3800 + X * 0x04040400) & 0xFFFFFFFF
    t1 = (0x46444240 + X * 0x04040404) & 0xFFFFFFFF
    hi = cw >> 16
    m0, m1 = prmt(t0, t1, cw & 0x7777), prmt(t0, t1, hi & 0x7777)
    n0 = (prmt(0x7F7F7F7F, 0x7F7F7F7F, cw) + 0x01010101) & 0xFFFFFFFF
    n1 = (prmt(0x7F7F7F7F, 0x7F7F7F7F, hi) + 0x01010101) & 0xFFFFFFFF
    w0, w1 = m0 | (~n0 & 0x80808080), m1 | (~n1 & 0x80808080)
    return [(w0 >> (8 * i)) & 0xFF for i in range(4)] + [(w1 >> (8 * i)) & 0xFF for i in range(4)]


def test_e2m1_to_e5m2_every_nibble_and_exponent():
    mags = oracle.E2M1_MAGNITUDES
    rng = np.random.default_rng(5)
    words = [sum(((n + k) % 16) << (4 * k) for k in range(8)) for n in range(16)]
    words += [int(v) for v in rng.integers(0, 2 ** 32, 300, dtype=np.uint64)]
    for X in range(-13, 14):
        for cw in words:
            out = e2m1x8_to_e5m2(cw, X)
            for i in range(8):
                nib = (cw >> (4 * i)) & 0xF
                want = (-1.0 if nib & 8 else 1.0) * mags[nib & 7] * 2.0 ** X
                assert e5m2_value(out[i]) == want, (X, hex(cw), i)


def test_query_bytes_from_magnitude_index():
    """Queries: the E5M2 byte of a magnitude index comes from the same shifted table."""
    mags = oracle.E2M1_MAGNITUDES
    for X in range(-13, 14):
        t0 = (0x3E3C3800 + X * 0x04040400) & 0xFFFFFFFF
        t1 = (0x46444240 + X * 0x04040404) & 0xFFFFFFFF
        for idx in range(8):
            assert e5m2_value(prmt(t0, t1, idx) & 0xFF) == mags[idx] * 2.0 ** X
