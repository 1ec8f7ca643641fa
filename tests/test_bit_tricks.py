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


def test_e2m1_block_sums_are_exact_in_fp32():
    """The E2M1-operand scores kernel keeps one fp32 accumulator per 32-code scale block: every
    product of two E2M1 values is a multiple of 1/4 below 36 in magnitude, so a block's sum
    (at most 1152) is exact in fp32 whatever order the tensor core adds in."""
    mags = np.asarray(oracle.E2M1_MAGNITUDES)
    rng = np.random.default_rng(11)
    vals = np.concatenate([-mags[::-1], mags])          # every E2M1 value, both zeros
    worst = np.full(32, 6.0)                            # the extreme block: 32 x 6 x 6
    for trial in range(2000):
        a = rng.choice(vals, 32) if trial else worst
        b = rng.choice(vals, 32) if trial else worst
        exact = float(np.dot(a.astype(np.float64), b.astype(np.float64)))
        p = (a * b).astype(np.float32)
        for order in (np.arange(32), np.arange(32)[::-1], rng.permutation(32)):
            acc = np.float32(0.0)
            for i in order:
                acc = np.float32(acc + p[i])
            assert float(acc) == exact
        pair = p.copy()                                  # pairwise tree
        while len(pair) > 1:
            pair = (pair[0::2] + pair[1::2]).astype(np.float32)
        assert float(pair[0]) == exact


def test_e2m1_block_scaling_matches_the_decoded_dot_product():
    """The epilogue forms y = sum_j acc_j * (2^Xq_j * 2^Xk_j) over the four blocks with fp32
    multiplies and FMAs; against the fp64 dot product of the decoded values it stays within a few
    fp32 ulps of the terms, far inside the scores' 2e-3 relative tolerance, for scale exponents
    whose scaled products fit fp32 (e = 0 is 2^-127, a subnormal in fp32; scale products below
    2^-149 flush to zero, which costs at most 1152 * 2^-149 absolute)."""
    mags = np.asarray(oracle.E2M1_MAGNITUDES)
    vals = np.concatenate([-mags[::-1], mags])
    rng = np.random.default_rng(12)
    for trial in range(3000):
        a = rng.choice(vals, 128)
        b = rng.choice(vals, 128)
        ek = rng.integers(0, 201, 4) if trial % 3 == 0 else rng.integers(110, 145, 4)
        xq = rng.integers(-40, 27, 4)                                 # Xq + Xk <= 99
        sk = np.array([2.0 ** -127 if e == 0 else 2.0 ** (int(e) - 127) for e in ek])
        sq = 2.0 ** xq.astype(np.float64)
        acc = np.array([np.dot(a[32 * j:32 * j + 32], b[32 * j:32 * j + 32]) for j in range(4)], np.float32)
        y = np.float32(0.0)
        for j in range(4):
            f = np.float32(np.float32(sq[j]) * np.float32(sk[j]))      # exact: a power of two
            y = np.float32(float(acc[j]) * float(f) + float(y))        # one rounding, as an FMA
        ref = float(sum(float(acc[j]) * sq[j] * sk[j] for j in range(4)))
        mag = float(sum(abs(float(acc[j])) * sq[j] * sk[j] for j in range(4)))
        assert abs(float(y) - ref) <= 4 * 2.0 ** -24 * mag + 2.0 ** -137, (trial, float(y), ref)
