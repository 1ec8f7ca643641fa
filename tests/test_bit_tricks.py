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


def _bf16_value(h: int) -> float:
    return float(np.array([h << 16], dtype=np.uint32).view(np.float32)[0])


def e2m1x8_to_bf16(cw: int, e8: int) -> list[int]:
    """The kernel's bf16 decode: magnitude high/low bytes by byte permutes, the sign moved into
    place, and X = e8 - 127 added to the exponent field of every non-zero half (vadd2 under a
    vcmpne2 mask)."""
    lo, hi = cw & 0x07070707, (cw >> 4) & 0x07070707
    yl, yh = lo | (lo >> 4), hi | (hi >> 4)
    sel_l = (yl & 0xFF) | ((yl >> 8) & 0xFF00)
    sel_h = (yh & 0xFF) | ((yh >> 8) & 0xFF00)
    hl = prmt(0x3F3F3F00, 0x40404040, sel_l) | ((cw << 4) & 0x80808080)
    ll = prmt(0xC0800000, 0xC0804000, sel_l)
    hh = prmt(0x3F3F3F00, 0x40404040, sel_h) | (cw & 0x80808080)
    lh = prmt(0xC0800000, 0xC0804000, sel_h)
    t0, t1 = prmt(ll, hl, 0x5140), prmt(lh, hh, 0x5140)
    t2, t3 = prmt(ll, hl, 0x7362), prmt(lh, hh, 0x7362)
    o = [prmt(t0, t1, 0x5410), prmt(t0, t1, 0x7632), prmt(t2, t3, 0x5410), prmt(t2, t3, 0x7632)]
    k16 = ((e8 - 127) << 7) & 0xFFFF
    out = []
    for w in o:
        for half in (w & 0xFFFF, w >> 16):
            out.append(((half + k16) & 0xFFFF) if (half & 0x7FFF) != 0 else half)
    return out   # elements 0, 1, ..., 7 as bf16 bit patterns


def test_e2m1_to_bf16_every_nibble_and_scale():
    mags = oracle.E2M1_MAGNITUDES
    rng = np.random.default_rng(6)
    words = [sum(((n + k) % 16) << (4 * k) for k in range(8)) for n in range(16)]
    words += [int(v) for v in rng.integers(0, 2 ** 32, 100, dtype=np.uint64)]
    for e8 in list(range(2, 253, 7)) + [2, 127, 252]:
        for cw in words:
            out = e2m1x8_to_bf16(cw, e8)
            for i in range(8):
                nib = (cw >> (4 * i)) & 0xF
                want = (-1.0 if nib & 8 else 1.0) * mags[nib & 7] * 2.0 ** (e8 - 127)
                assert _bf16_value(out[i]) == want, (e8, hex(cw), i)


def test_fp4_kv_decode_values():
    """The attention's fp4 row decode: the E4M3 scale byte -> fp32 from its bit fields (exact in
    bf16), times the E2M1 value (looked up by the byte-permute decoder checked above) -- every
    product exact in bf16 and equal to the oracle's decode for every code and finite scale."""
    def e4m3_to_f32(v: int) -> float:
        e, m, sg = (v >> 3) & 15, v & 7, (v & 0x80) << 24
        if e == 0:
            bits = sg | int(np.array([m * 0.001953125], dtype=np.float32).view(np.uint32)[0])
        else:
            bits = sg | ((e + 120) << 23) | (m << 20)
        return float(np.array([bits], dtype=np.uint32).view(np.float32)[0])

    mags = oracle.E2M1_MAGNITUDES
    for sb in range(256):
        if sb & 0x7F == 0x7F:
            continue
        s = e4m3_to_f32(sb)
        assert s == oracle.e4m3_value(np.array([sb], np.uint8))[0], hex(sb)
        for nib in range(16):
            v = np.float32((-1.0 if nib & 8 else 1.0) * mags[nib & 7]) * np.float32(s)
            bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0]) >> 16
            assert _bf16_value(bits) == float(v), (hex(sb), nib)   # exact in bf16
