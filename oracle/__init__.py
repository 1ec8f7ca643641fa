"""CPU oracle for the DeepSeek V4.1 Indexer -> top-k -> sparse sink attention path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package; the product package never does.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation); this module only
builds it with gcc, loads it with ctypes and marshals numpy arrays.  bf16 tensors are
numpy ``uint16`` arrays holding the bf16 bit patterns.

Every function is pinned by the CPU tests in ``tests/test_oracle_*.py``:
  window_topk_idxs   worked rows of get_window_topk_idxs (tests/golden/window_idx.txt)
  visible / compress_len   closed forms and the worked Indexer rows (golden)
  index_score        one-hot closed forms, rank-one identity, head additivity, relu cut-off
  topk               numpy lexsort reference, subset brute force, vis <= k layout
  sparse_attn        textbook softmax (sink -> -inf), single-row closed form, empty rows,
                     duplicate-row sink shift, permutation invariance, mass + sink = 1
  dense_attn         independent of index lists; equal to sparse_attn when k >= visible
  mxfp4_quantize / mxfp4_decode / index_score_mxfp4   the E2M1 code table from the format's
                     definition, exact round trips of grid values, ties to even, saturation,
                     the scale rule against frexp, zero blocks, the error bound
  e4m3_value / e4m3_round / kvfp4_quantize / kvfp4_decode / sparse_attn_fp4kv   the E4M3 table
                     from the format's definition (bias, subnormals, NaN, 448), ties to even and
                     saturation, the scale rule, exact round trips, zero and tiny blocks, the
                     error bound, attention over the decoded rows equal to the plain attention
  window_topk_idxs_chunked   the prefill band of the pages when the chunk starts at 0 (rows
                     shifted past the ring), brute-force positions of every referenced row
  output_inverse_rope   identity at angle 0, the quarter-turn closed form, complex
                     multiplication by e^{-i theta}, and undoing the generator's rotation
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (portable flags, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_window_topk_idxs.argtypes = [I, I, I, I, P]
        lib.oracle_window_topk_idxs.restype = I
        lib.oracle_compress_len.argtypes = [I, I, I]
        lib.oracle_compress_len.restype = I
        lib.oracle_visible.argtypes = [I, I, I]
        lib.oracle_visible.restype = I
        lib.oracle_index_score.argtypes = [P, P, I64, P, D, P, I, I, I, I, I, I, P, I]
        lib.oracle_index_score.restype = None
        lib.oracle_topk.argtypes = [P, P, I, I, I, I, I, ctypes.c_int32, P, I]
        lib.oracle_topk.restype = None
        lib.oracle_sparse_attn.argtypes = [P, P, I64, P, I64, I, I, P, P, D, I, I, I, I, I, P, P, I]
        lib.oracle_sparse_attn.restype = None
        lib.oracle_dense_attn.argtypes = [P, P, I64, P, I64, P, P, D, I, I, I, I, I, I, P, I]
        lib.oracle_dense_attn.restype = None
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def window_topk_idxs(window_size: int, bsz: int, seqlen: int, start_pos: int) -> np.ndarray:
    """get_window_topk_idxs: [bsz, seqlen, min(seqlen, W)] in prefill, [bsz, 1, W] in decode."""
    lib = _load()
    if start_pos == 0:
        rows, width = seqlen, min(seqlen, window_size)
    else:
        rows, width = 1, window_size
    out = np.empty((bsz, rows, width), dtype=np.int32)
    got = lib.oracle_window_topk_idxs(window_size, bsz, seqlen, start_pos, _ptr(out))
    assert got == width
    return out


def window_topk_idxs_chunked(window_size: int, seqlen: int, start_pos: int) -> np.ndarray:
    """Window rows of a prefill chunk that continues a sequence (start_pos > 0): [seqlen, W].

    The pages cover prefill from position 0 (get_window_topk_idxs' band) and decode (the
    W-slot ring); a chunk starting later is not on them.  Reading: the chunk's window source is
    the ring as it stood before the chunk (rows [0, W): slot i holds the newest position
    p < start_pos with p % W == i) followed by the chunk's own raw rows (row W + i holds
    position start_pos + i).  Query t at position P = start_pos + t sees, as the prefill band
    does with t, the positions max(0, P - W + 1) + i for i < W, -1 past P; position p maps to
    row W + (p - start_pos) when p >= start_pos, else to ring slot p % W."""
    W = int(window_size)
    out = np.full((seqlen, W), -1, dtype=np.int32)
    for t in range(seqlen):
        P = start_pos + t
        first = max(0, P - W + 1)
        for i in range(W):
            p = first + i
            if p > P:
                continue
            out[t, i] = W + (p - start_pos) if p >= start_pos else p % W
    return out


# ------------------------------------------------------------------ MXFP4 (fp4 index keys and queries)
#
# Indexer.forward ("attend/selected" page) passes its keys and queries through fp4_act_quant(x,
# fp4_block_size, True) before the score einsum; the quantiser itself is not on the pages.
# Reading: the OCP Microscaling (MX) MXFP4 format -- blocks of 32 consecutive elements along the
# head dim share one E8M0 scale 2^X with X = floor(log2(max |x|)) - 2 (2 = the largest exponent of
# E2M1), each element x / 2^X rounded to the nearest E2M1 value (ties to the even code) and
# saturated at +-6.  The flag `True` is read as "in place": the einsum then runs on the
# dequantised values.

E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def mxfp4_decode(codes, scales, dim: int) -> np.ndarray:
    """Packed E2M1 codes [..., dim/2] (element 2j in the low nibble of byte j, 2j+1 in the high
    one; bit 3 of a nibble = sign) and E8M0 scales [..., dim/32] (byte e -> 2^(e-127)) ->
    float64 [..., dim]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (dim,))
    mag = np.asarray(E2M1_MAGNITUDES)[nib & 0x7]
    val = np.where(nib & 0x8, -mag, mag)
    sc = np.exp2(scales.astype(np.float64) - 127.0)
    return val * np.repeat(sc, 32, axis=-1)


def mxfp4_quantize(x):
    """float [..., dim] (dim a multiple of 32) -> (codes uint8 [..., dim/2], scales uint8 [..., dim/32])."""
    x = np.asarray(x, dtype=np.float64)
    dim = x.shape[-1]
    blk = x.reshape(x.shape[:-1] + (dim // 32, 32))
    amax = np.abs(blk).max(axis=-1)
    with np.errstate(divide="ignore"):
        X = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2.0, -127.0)
    X = np.clip(X, -127.0, 127.0)
    nib = _e2m1_nibbles(blk / np.exp2(X)[..., None]).reshape(x.shape)
    codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    scales = (X + 127.0).astype(np.uint8)
    return codes, scales


def _nearest_on_grid(grid, a):
    """Index of the value of the ascending grid nearest to a (a within [grid[0], grid[-1]]); on a
    tie the even index (for E2M1 and E4M3 codes: the one whose mantissa's last bit is clear)."""
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, len(grid) - 1)   # first grid value >= a
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo, d_hi = a - grid[lo], grid[hi] - a
    idx = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    return np.where(a == grid[hi], hi, idx)


def _e2m1_nibbles(p) -> np.ndarray:
    """Values already divided by their block scale -> E2M1 nibbles (bit 3 sign, bits 0-2 the
    magnitude code), nearest with ties to the even code, saturating at +-6; zero has no sign."""
    p = np.asarray(p, dtype=np.float64)
    code = _nearest_on_grid(np.asarray(E2M1_MAGNITUDES), np.minimum(np.abs(p), 6.0))
    sign = ((p < 0) & (code > 0)).astype(np.uint8) << 3
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def mxfp4_fake_quant(x) -> np.ndarray:
    """The values the einsum sees: quantise, then decode (float64)."""
    codes, scales = mxfp4_quantize(x)
    return mxfp4_decode(codes, scales, np.asarray(x).shape[-1])


def index_score_mxfp4(iq, ik_codes, ik_scales, w, c: float, start_pos, n_cols: int, ratio: int,
                      threads: int | None = None) -> np.ndarray:
    """Indexer scores with MXFP4 keys (stored quantised) and queries (quantised in the forward):
    index_score over the decoded values.  iq: [b, s, H, D] bf16 bits; ik_codes: [b, >= n_cols,
    D/2] uint8; ik_scales: [b, >= n_cols, D/32] uint8; w: [b, s, H] bf16 bits.  The decoded
    values are exact in bf16, so they go to index_score as bf16 bit patterns."""
    iq = _c(iq, np.uint16)
    D = iq.shape[-1]
    qf = (np.ascontiguousarray(iq).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    qd = mxfp4_fake_quant(qf)
    kd = mxfp4_decode(ik_codes, ik_scales, D)
    return index_score(_bf16_exact(qd), _bf16_exact(kd), w, c, start_pos, n_cols, ratio, threads)


# ------------------------------------------------------------------ fp4 compressed KV (E4M3 scales, groups of 16)
#
# Attention._compress_kv ("read-weights" page) applies the rotary embedding to the latent's last
# rope dims, then fp4_act_quant(latent, 16, True, scale_dtype=float8_e4m3fn) -- in place -- and
# writes the result to the compressed-KV cache; the page's comment there: the compressed KV uses
# groups of 16 with E4M3 scales.  The quantiser's body is not on the pages.  Reading (the
# NVFP4-style block format without a second, per-tensor scale): blocks of 16 consecutive
# elements along the row share one E4M3 scale s, the E4M3 value nearest to max|x| / 6 (ties to
# the even code, saturating at 448), and each element x / s is rounded to the nearest E2M1
# value as for MXFP4 (a block whose s is 0 is all zeros).  The cache (the attention's second KV
# source) holds the decoded values; the window rows stay bf16.

def e4m3_value(byte) -> np.ndarray:
    """E4M3 (the float8_e4m3fn format: sign, 4-bit exponent with bias 7, 3-bit mantissa,
    subnormals at exponent 0, no infinities, S.1111.111 = NaN) byte(s) -> float64."""
    b = np.asarray(byte, dtype=np.uint8).astype(np.int64)
    sgn = np.where(b & 0x80, -1.0, 1.0)
    e, m = (b >> 3) & 0xF, b & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sgn * mag


_E4M3_POSITIVE = e4m3_value(np.arange(0x7F, dtype=np.uint8))   # codes 0x00 .. 0x7E, ascending


def e4m3_round(a) -> np.ndarray:
    """Non-negative float(s) -> the byte of the nearest E4M3 value (ties to the even code),
    saturating at 448."""
    a = np.minimum(np.asarray(a, dtype=np.float64), 448.0)
    return _nearest_on_grid(_E4M3_POSITIVE, a).astype(np.uint8)


def kvfp4_quantize(x):
    """float [..., d] (d a multiple of 16) -> (codes uint8 [..., d/2], E4M3 scale bytes [..., d/16]);
    codes packed as for MXFP4 (element 2j in the low nibble of byte j)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    blk = x.reshape(x.shape[:-1] + (d // 16, 16))
    sbyte = e4m3_round(np.abs(blk).max(axis=-1) / 6.0)
    s = e4m3_value(sbyte)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(s > 0, blk / np.where(s > 0, s, 1.0), 0.0)
    nib = _e2m1_nibbles(p).reshape(x.shape)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8), sbyte


def kvfp4_decode(codes, scales, d: int) -> np.ndarray:
    """Packed E2M1 codes [..., d/2] and E4M3 scale bytes [..., d/16] -> float64 [..., d]."""
    codes = np.asarray(codes, dtype=np.uint8)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (d,))
    mag = np.asarray(E2M1_MAGNITUDES)[nib & 0x7]
    val = np.where(nib & 0x8, -mag, mag)
    return val * np.repeat(e4m3_value(scales), 16, axis=-1)


def sparse_attn_fp4kv(q, kv1, kv2_codes, kv2_scales, sink, idx, scale: float, threads: int | None = None,
                      rope_cs=None):
    """sparse_attn with the second (compressed) KV source stored as fp4 rows: kv2_codes [b, n2,
    d/2], kv2_scales [b, n2, d/16]; the attention runs over the decoded rows (exact in bf16: an
    E2M1 value times an E4M3 scale has at most 5 significant bits)."""
    d = np.asarray(q).shape[-1]
    kv2 = _bf16_exact(kvfp4_decode(kv2_codes, kv2_scales, d))
    return sparse_attn(q, kv1, sink, idx, scale, kv2=kv2, threads=threads, rope_cs=rope_cs)


def _bf16_exact(x) -> np.ndarray:
    """float64 values exactly representable in bf16 -> their bit patterns (checked)."""
    f = np.asarray(x, dtype=np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64)), "not exact in fp32"
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << np.uint32(16)).view(np.float32), f), "not exact in bf16"
    return bits


def compress_len(start_pos: int, seqlen: int, ratio: int) -> int:
    return int(_load().oracle_compress_len(start_pos, seqlen, ratio))


def visible(start_pos: int, t: int, ratio: int) -> int:
    return int(_load().oracle_visible(start_pos, t, ratio))


def index_score(iq, ik, w, c: float, start_pos, n_cols: int, ratio: int, threads: int | None = None) -> np.ndarray:
    """Scores [b, s, n_cols] (float64, -inf where not visible).

    iq: [b, s, H, D] bf16 bits; ik: [b, >= n_cols, D] bf16 bits; w: [b, s, H] bf16 bits."""
    iq = _c(iq, np.uint16)
    ik = _c(ik, np.uint16)
    w = _c(w, np.uint16)
    sp = _c(start_pos, np.int32)
    b, s, H, D = iq.shape
    assert ik.shape[0] == b and ik.shape[2] == D and ik.shape[1] >= n_cols
    assert w.shape == (b, s, H) and sp.shape == (b,)
    out = np.empty((b, s, n_cols), dtype=np.float64)
    _load().oracle_index_score(
        _ptr(iq), _ptr(ik), ik.shape[1] * D, _ptr(w), float(c), _ptr(sp), b, s, H, D, n_cols, ratio, _ptr(out),
        threads or default_threads(),
    )
    return out


def topk(score, start_pos, ratio: int, k: int, offset: int, threads: int | None = None) -> np.ndarray:
    """Top-k positions per row: [b, s, k] int32, ascending, +offset, -1 padded."""
    score = _c(score, np.float64)
    sp = _c(start_pos, np.int32)
    b, s, n_cols = score.shape
    out = np.empty((b, s, k), dtype=np.int32)
    _load().oracle_topk(_ptr(score), _ptr(sp), b, s, n_cols, ratio, k, offset, _ptr(out), threads or default_threads())
    return out


def output_inverse_rope(out, rope_cs):
    """The output's inverse rotary rotation, as Attention.forward applies it after sparse_attn
    (DeepSeek V4.1, "attend/selected" page: apply_rotary_emb on o[..., -rd:] with the inverse
    flag).  The rotation itself is not printed on the pages; its reading: the last rd dims form
    rd/2 interleaved pairs (x, y) = (o[2i], o[2i+1]) of a complex number x + iy, multiplied by
    conj(e^{i theta_i}) of the query's position.

    out: [b, s, h, d] float64 (rotated in place and returned); rope_cs: [b, s, rd/2, 2] with
    (cos theta_i, sin theta_i) per query and pair (any precision, widened to float64)."""
    cs = np.asarray(rope_cs, dtype=np.float64)
    b, s, h, d = out.shape
    rd = 2 * cs.shape[2]
    c = cs[..., 0][:, :, None, :]          # [b, s, 1, rd/2]
    sn = cs[..., 1][:, :, None, :]
    x = out[..., d - rd::2].copy()
    y = out[..., d - rd + 1::2].copy()
    out[..., d - rd::2] = x * c + y * sn
    out[..., d - rd + 1::2] = y * c - x * sn
    return out


def sparse_attn(q, kv1, sink, idx, scale: float, kv2=None, threads: int | None = None, rope_cs=None):
    """Sparse attention with sink; returns (out [b,s,h,d] float64, lse [b,s,h] float64).

    q: [b, s, h, d] bf16 bits; kv1: [b, n1, d]; kv2: optional [b, n2, d] (row r >= n1 of the
    concatenated KV is kv2[r - n1]); sink: [h] float32; idx: [b, s, k] int32; rope_cs: optional
    [b, s, rd/2, 2] (cos, sin) of the output's inverse rotation (output_inverse_rope)."""
    q = _c(q, np.uint16)
    kv1 = _c(kv1, np.uint16)
    kv2 = None if kv2 is None else _c(kv2, np.uint16)
    sink = _c(sink, np.float32)
    idx = _c(idx, np.int32)
    b, s, h, d = q.shape
    k = idx.shape[2]
    n1 = kv1.shape[1]
    n2 = 0 if kv2 is None else kv2.shape[1]
    out = np.empty((b, s, h, d), dtype=np.float64)
    lse = np.empty((b, s, h), dtype=np.float64)
    _load().oracle_sparse_attn(
        _ptr(q), _ptr(kv1), n1 * d, _ptr(kv2), n2 * d, n1, n2, _ptr(sink), _ptr(idx), float(scale), b, s, h, d, k,
        _ptr(out), _ptr(lse), threads or default_threads(),
    )
    if rope_cs is not None:
        output_inverse_rope(out, rope_cs)
    return out, lse


def dense_attn(q, win, comp, start_pos, sink, scale: float, window_size: int, ratio: int, threads: int | None = None):
    """Dense causal window + visible compressed attention with sink (no index lists)."""
    q = _c(q, np.uint16)
    win = _c(win, np.uint16)
    comp = _c(comp, np.uint16)
    sp = _c(start_pos, np.int32)
    sink = _c(sink, np.float32)
    b, s, h, d = q.shape
    out = np.empty((b, s, h, d), dtype=np.float64)
    _load().oracle_dense_attn(
        _ptr(q), _ptr(win), win.shape[1] * d, _ptr(comp), comp.shape[1] * d, _ptr(sp), _ptr(sink), float(scale),
        b, s, h, d, window_size, ratio, _ptr(out), threads or default_threads(),
    )
    return out
