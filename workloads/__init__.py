"""Seeded synthetic inputs for the Indexer -> top-k -> sparse sink attention path.

This module is shared by the tests, the benchmark and the oracle legs.  It only draws
random numbers and shapes them; it holds none of the path's arithmetic (no scores, no
selection, no attention).  bf16 tensors are numpy ``uint16`` arrays of bf16 bit patterns
(round-to-nearest-even from fp32); the CUDA side uploads them as ``torch.bfloat16``.

Random streams are numpy's counter-based Philox generator, keyed by (seed, tensor id), so
every tensor is reproducible on its own and identical on every machine.

Workloads (seed = 1000 + number):
  1 tiny prefill     b=1, s=256, start_pos=0, h=4, d=64 (RoPE theta 1e4 on the last 16 dims),
                     window 16, ratio 4 -> 64 compressed positions, index_topk 16, index heads 4x32,
                     weights N(0,1)/2
  2 decode           b=32, s=1, start_pos=65535, h=64, d=512, window 128, ratio 4 -> 16384
                     compressed rows, index heads 32x128 with RMS-normalised keys, index_topk 512
  3 prefill          b=1, s=8192, start_pos=0, same shapes as 2 -> 2048 compressed rows
  4 long decode      b=8, s=1, start_pos=131071 -> 32768 compressed rows; 1% of key rows carry a
                     planted rank-one bias so their scores sit about 3 sigma above the rest
  5 mixed serving    b=64, s=1, lengths uniform on [1024, 65536] (ragged start_pos), one index pass
                     and four attention layers (a source and three reuse layers) with their own
                     q / window / sink over one shared compressed KV
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))

# ------------------------------------------------------------------ bf16 bits


def to_bf16_bits(x) -> np.ndarray:
    """fp32/fp64 values -> bf16 bit patterns (round to nearest even, finite inputs)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rng_for(seed: int, stream: int) -> np.random.Generator:
    """Counter-based Philox stream `stream` of `seed`."""
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream])))


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return to_bf16_bits(x)


# ------------------------------------------------------------------ config


@dataclasses.dataclass
class Shape:
    """One workload's shapes.  start_pos is per sequence (ragged batches)."""

    name: str
    b: int
    s: int
    start_pos: np.ndarray      # int32 [b]
    h: int = 64                # attention heads
    d: int = 512               # head_dim (last rd dims carry RoPE)
    rd: int = 64
    rope_theta: float | None = None   # applied by the generator when set
    window: int = 128
    ratio: int = 4
    n_cols: int = 16384        # compressed positions held (capacity of the caches)
    topk: int = 512            # index_topk
    Hi: int = 32               # index heads
    Di: int = 128              # index head dim
    w_scale: float = 1.0       # weights_proj outputs ~ N(0, w_scale^2)
    rms_keys: bool = False     # RMS-normalise index key rows
    planted: bool = False      # planted rank-one score bias on 1% of keys
    n_layers: int = 1          # attention layers sharing one index pass (reuse layers)
    fp4_keys: bool = False     # index keys stored as MXFP4 (E2M1 codes + E8M0 scales)
    fp4_kv: bool = False       # compressed KV rows stored as fp4 (E2M1 codes + an E4M3 scale per 16)
    seed: int = 0

    @property
    def prefill(self) -> bool:
        """Several queries per sequence: a prefill from position 0, or a later chunk."""
        return self.s > 1

    @property
    def chunked(self) -> bool:
        """A prefill chunk that continues its sequence (start_pos > 0)."""
        return self.s > 1 and bool(np.any(self.start_pos != 0))

    @property
    def win_rows(self) -> int:
        """Rows of the window KV source: the s raw rows in prefill from 0, the ring before the
        chunk followed by its s rows in a later chunk, the W-slot ring in decode."""
        if self.chunked:
            return self.window + self.s
        return self.s if self.prefill else self.window

    @property
    def win_width(self) -> int:
        """Window slots per query: min(s, W) in prefill from 0, W otherwise."""
        return min(self.s, self.window) if (self.prefill and not self.chunked) else self.window

    @property
    def k_total(self) -> int:
        return self.win_width + self.topk

    @property
    def softmax_scale(self) -> float:
        return self.d ** -0.5

    @property
    def index_scale(self) -> float:
        return self.Di ** -0.5 * self.Hi ** -0.5

    def visible(self) -> np.ndarray:
        """Compressed positions each sequence's last query can see (capped by n_cols), [b]."""
        v = (self.start_pos.astype(np.int64) + self.s) // self.ratio
        return np.minimum(v, self.n_cols).astype(np.int64)


def config(n: int) -> Shape:
    """The named workloads: 1-5 as listed in the design notes, 6 and 7 the decode workload at
    compression ratios 2 and 1 (32768 and 65536 index rows per sequence), 8 a prefill chunk
    that continues its sequence, 9 workload 2 with MXFP4 index keys, 10 workload 3 and 11
    workload 2 with the compressed KV rows stored as fp4."""
    seed = 1000 + n
    if n == 1:
        return Shape("tiny_prefill_s256_h4_d64", b=1, s=256, start_pos=np.zeros(1, np.int32), h=4, d=64, rd=16,
                     rope_theta=10000.0, window=16, ratio=4, n_cols=64, topk=16, Hi=4, Di=32, w_scale=0.5, seed=seed)
    if n == 2:
        return Shape("decode_b32_ctx65536", b=32, s=1, start_pos=np.full(32, 65535, np.int32), n_cols=16384,
                     rms_keys=True, seed=seed)
    if n == 3:
        return Shape("prefill_s8192", b=1, s=8192, start_pos=np.zeros(1, np.int32), n_cols=2048, seed=seed)
    if n == 4:
        return Shape("long_decode_b8_ctx131072", b=8, s=1, start_pos=np.full(8, 131071, np.int32), n_cols=32768,
                     planted=True, seed=seed)
    if n == 5:
        lengths = rng_for(seed, 99).integers(1024, 65536, size=64, endpoint=True)
        sp = (lengths - 1).astype(np.int32)
        n_cols = int(lengths.max() // 4)
        return Shape("mixed_serving_b64_ctx1k-64k", b=64, s=1, start_pos=sp, n_cols=n_cols, rms_keys=True,
                     n_layers=4, seed=seed)
    if n == 9:   # workload 2 with MXFP4 index keys
        return Shape("decode_b32_ctx65536_mxfp4", b=32, s=1, start_pos=np.full(32, 65535, np.int32), n_cols=16384,
                     fp4_keys=True, seed=seed)
    if n == 11:  # workload 2 with fp4 compressed-KV rows
        return Shape("decode_b32_ctx65536_kvfp4", b=32, s=1, start_pos=np.full(32, 65535, np.int32), n_cols=16384,
                     rms_keys=True, fp4_kv=True, seed=seed)
    if n == 10:  # workload 3 with fp4 compressed-KV rows
        return Shape("prefill_s8192_kvfp4", b=1, s=8192, start_pos=np.zeros(1, np.int32), n_cols=2048, fp4_kv=True,
                     seed=seed)
    if n == 8:   # a prefill chunk of 2048 queries continuing a sequence at position 6144
        return Shape("chunked_prefill_s2048_at6144", b=1, s=2048, start_pos=np.full(1, 6144, np.int32), n_cols=2048,
                     seed=seed)
    if n in (6, 7):   # the model's own compression ratios (2 and 1) at context 65536
        r = 2 if n == 6 else 1
        return Shape(f"decode_b32_ctx65536_r{r}", b=32, s=1, start_pos=np.full(32, 65535, np.int32), ratio=r,
                     n_cols=65536 // r, rms_keys=True, seed=seed)
    raise ValueError(f"no workload {n}")


def custom(name: str, b: int, s: int, start_pos, seed: int, **kw) -> Shape:
    """A smaller workload of the same structure (tests: several tiles plus a ragged tail)."""
    sp = np.broadcast_to(np.asarray(start_pos, dtype=np.int32), (b,)).copy()
    return Shape(name, b=b, s=s, start_pos=sp, seed=seed, **kw)


# ------------------------------------------------------------------ RoPE (input preparation only)


def _rope_interleaved(x: np.ndarray, positions: np.ndarray, rd: int, theta: float) -> np.ndarray:
    """Rotate the last rd dims of x (pairs (2i, 2i+1)) by angle pos * theta^(-2i/rd).

    x: float64 [..., n, dim] with positions [n] along axis -2.  Input preparation for
    workload 1, whose recipe puts RoPE on the last rd dims; the path applies only the output's
    inverse rotation, from a table its caller passes (output_rope_table)."""
    y = x.copy()
    i = np.arange(rd // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / rd)
    ang = positions.astype(np.float64)[:, None] * inv[None, :]          # [n, rd/2]
    cos, sin = np.cos(ang), np.sin(ang)
    a = x[..., -rd::2]
    bb = x[..., -rd + 1::2]
    y[..., -rd::2] = a * cos - bb * sin
    y[..., -rd + 1::2] = a * sin + bb * cos
    return y


def planted_bias() -> float:
    """beta for workload 4, written by workloads/calibrate_planted_bias.py (oracle-calibrated)."""
    with open(os.path.join(_HERE, "planted_bias.json")) as f:
        return float(json.load(f)["beta"])


# ------------------------------------------------------------------ generator


def output_rope_table(shape: Shape, theta: float = 10000.0) -> np.ndarray:
    """(cos, sin) of the angles the output's inverse rotary rotation undoes, per query and pair:
    float32 [b, s, rd/2, 2] at positions start_pos + t, angle pos * theta^(-2i/rd) (the model's
    own frequencies come from a table these pages do not print; any table is an input here)."""
    theta = shape.rope_theta or theta
    i = np.arange(shape.rd // 2, dtype=np.float64)
    pos = shape.start_pos.astype(np.float64)[:, None] + np.arange(shape.s, dtype=np.float64)[None, :]
    ang = pos[..., None] * theta ** (-2.0 * i / shape.rd)
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


def make(shape: Shape, beta: float | None = None) -> dict:
    """Draw every input tensor of `shape`.

    Returns a dict with bf16-bit arrays
      q    [L, b, s, h, d]    attention queries per layer (L = n_layers)
      win  [L, b, win_rows, d] window KV per layer: raw rows (prefill) or ring (decode)
      comp [b, n_cols, d]     shared compressed KV (rows past a sequence's length are zero)
      iq   [b, s, Hi, Di]     index queries;  ik [b, n_cols, Di] index keys
      w    [b, s, Hi]         weights_proj outputs
    and float32 sink [L, h], int32 start_pos [b]."""
    sd = shape.seed
    L, b, s = shape.n_layers, shape.b, shape.s
    vis = shape.visible()
    out: dict = {"shape": shape, "start_pos": shape.start_pos.astype(np.int32)}

    r = rng_for(sd, 1)
    q = r.standard_normal(size=(L, b, s, shape.h, shape.d), dtype=np.float32)
    r = rng_for(sd, 2)
    win = r.standard_normal(size=(L, b, shape.win_rows, shape.d), dtype=np.float32)
    r = rng_for(sd, 3)
    comp = np.zeros((b, shape.n_cols, shape.d), dtype=np.uint16)
    r4 = rng_for(sd, 4)
    iq = r4.standard_normal(size=(b, s, shape.Hi, shape.Di), dtype=np.float32)
    r5 = rng_for(sd, 5)
    ik = np.zeros((b, shape.n_cols, shape.Di), dtype=np.uint16)
    r6 = rng_for(sd, 6)
    w = r6.standard_normal(size=(b, s, shape.Hi), dtype=np.float32) * np.float32(shape.w_scale)
    r7 = rng_for(sd, 7)
    sink = r7.standard_normal(size=(L, shape.h), dtype=np.float32)

    if shape.rope_theta is not None:
        th, rd = shape.rope_theta, shape.rd
        for bi in range(b):
            qpos = shape.start_pos[bi] + np.arange(s)
            q64 = np.moveaxis(q[:, bi].astype(np.float64), 1, -2)           # [L, h, s, d]
            q[:, bi] = np.moveaxis(_rope_interleaved(q64, qpos, rd, th), -2, 1)
            iq64 = np.moveaxis(iq[bi].astype(np.float64), 0, -2)            # [Hi, s, Di]
            iq[bi] = np.moveaxis(_rope_interleaved(iq64, qpos, rd, th), -2, 0)
            assert not shape.chunked, "RoPE inputs are drawn for prefill from 0 and decode only"
            if shape.prefill:
                wpos = np.arange(shape.win_rows)
            else:   # ring slot i holds the newest position p <= start_pos with p % W == i
                sp = int(shape.start_pos[bi])
                wpos = np.array([sp - ((sp - i) % shape.window) for i in range(shape.window)])
            win[:, bi] = _rope_interleaved(win[:, bi].astype(np.float64), wpos, rd, th)

    out["q"] = to_bf16_bits(q)
    out["win"] = to_bf16_bits(win)
    out["iq"] = to_bf16_bits(iq)
    out["w"] = to_bf16_bits(w)
    out["sink"] = sink

    beta = planted_bias() if (shape.planted and beta is None) else beta
    for bi in range(b):
        n = int(vis[bi])
        c = r.standard_normal(size=(n, shape.d), dtype=np.float32)
        k = r5.standard_normal(size=(n, shape.Di), dtype=np.float32)
        if shape.rope_theta is not None:
            pos = np.arange(n) * shape.ratio        # group j stands at position j*ratio
            c = _rope_interleaved(c.astype(np.float64), pos, shape.rd, shape.rope_theta)
            k = _rope_interleaved(k.astype(np.float64), pos, shape.rd, shape.rope_theta)
        if shape.rms_keys:
            k = k / np.sqrt(np.mean(np.square(k, dtype=np.float64), axis=-1, keepdims=True))
        if shape.planted:
            # direction: the weights-combined index query of this sequence, scaled to unit RMS
            qf = bf16_bits_to_f32(out["iq"][bi, 0]).astype(np.float64)              # [Hi, Di]
            wf = bf16_bits_to_f32(out["w"][bi, 0]).astype(np.float64)               # [Hi]
            u = (wf[:, None] * qf).sum(0)
            u = u / math.sqrt(float(np.mean(u * u)))
            n_plant = max(1, round(0.01 * n))
            rows = rng_for(sd, 100 + bi).choice(n, size=n_plant, replace=False)
            k = k.astype(np.float64)
            k[rows] += beta * u
            out.setdefault("planted_rows", {})[bi] = np.sort(rows)
        comp[bi, :n] = to_bf16_bits(c)
        ik[bi, :n] = to_bf16_bits(k)
    out["comp"] = comp
    if shape.fp4_keys:
        # MXFP4 keys are drawn directly as codes and scales: magnitude codes 0..7 with fixed
        # frequencies shaped like a half-normal on the E2M1 grid, random signs, and scale
        # bytes 125..127 (block scales 1/4 .. 1)
        rc = rng_for(sd, 8)
        mag = rc.choice(8, size=(b, shape.n_cols, shape.Di), p=FP4_CODE_FREQ).astype(np.uint8)
        sgn = (rc.random(size=mag.shape) < 0.5).astype(np.uint8) << 3
        nib = np.where(mag > 0, mag | sgn, 0).astype(np.uint8)
        codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        scales = rc.choice(np.array([125, 126, 127], np.uint8), size=(b, shape.n_cols, shape.Di // 32),
                           p=[0.2, 0.7, 0.1])
        for bi in range(b):   # rows past a sequence's visible count stay zero, as the bf16 keys do
            codes[bi, int(vis[bi]):] = 0
            scales[bi, int(vis[bi]):] = 0
        out["ik_codes"], out["ik_scales"] = codes, scales
    else:
        out["ik"] = ik
    if shape.fp4_kv:
        # fp4 compressed KV drawn directly as codes and E4M3 scales: the magnitude frequencies of
        # the MXFP4 keys, random signs, and scale bytes 0x28 .. 0x2E (1/4 .. 7/16: max|x| / 6 of a
        # 16-element block of N(0,1) values); rows past the sequence's compressed count are zero
        rc = rng_for(sd, 10)
        d2 = shape.d
        mag = rc.choice(8, size=(b, shape.n_cols, d2), p=FP4_CODE_FREQ).astype(np.uint8)
        sgn = (rc.random(size=mag.shape) < 0.5).astype(np.uint8) << 3
        nib = np.where(mag > 0, mag | sgn, 0).astype(np.uint8)
        kc = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        ksc = rc.integers(0x28, 0x2F, size=(b, shape.n_cols, d2 // 16), dtype=np.uint8)
        n_comp = np.minimum((shape.start_pos.astype(np.int64) + shape.s) // shape.ratio, shape.n_cols)
        for bi in range(b):
            kc[bi, int(n_comp[bi]):] = 0
            ksc[bi, int(n_comp[bi]):] = 0
        out["comp_codes"], out["comp_scales"] = kc, ksc
        del out["comp"]
    return out


FP4_CODE_FREQ = [0.10, 0.18, 0.17, 0.15, 0.13, 0.14, 0.09, 0.04]   # E2M1 magnitude codes 0..7


def index_lists(rng: np.random.Generator, b: int, s: int, k: int, n_rows: int, masked_frac: float = 0.1,
                empty_rows: int = 0) -> np.ndarray:
    """Random attention index lists [b, s, k] over rows [0, n_rows): distinct per query,
    a fraction set to -1, and the first `empty_rows` queries all -1."""
    out = np.empty((b, s, k), dtype=np.int32)
    for bi in range(b):
        for t in range(s):
            m = min(k, n_rows)
            sel = rng.choice(n_rows, size=m, replace=False).astype(np.int32)
            row = np.full(k, -1, dtype=np.int32)
            row[:m] = sel
            drop = rng.random(k) < masked_frac
            row[drop] = -1
            rng.shuffle(row)
            out[bi, t] = row
    flat = out.reshape(b * s, k)
    flat[:empty_rows] = -1
    return out
