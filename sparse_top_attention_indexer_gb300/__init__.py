"""sparse_top_attention_indexer_gb300 -- the DeepSeek V4.1 attention hot path on GB300.

Indexer scores -> top-k -> sliding-window indices -> sparse attention with an attention
sink, as hand-written sm_103a CUDA kernels behind the C ABI in ``include/sti.h``
(``libsti.so``).  This module is a thin ctypes binding: it checks dtypes/devices, passes
``data_ptr()``s, sizes and torch's current CUDA stream, and raises on a non-OK status.
Every step of the path runs in the library's kernels; there is no other implementation
here, and a missing library is an error.

Functions mirror the C entry points (``sti_`` prefix dropped):
  window_idxs, idx_scores, idx_topk, sparse_attn_sink, decode_fused, read_device_status
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# STI_LIB selects another build of the same library (for example one compiled with other
# tuning macros); by default the in-tree libsti.so
DEFAULT_LIB_PATH = os.path.join(_HERE, "libsti.so")
LIB_PATH = os.environ.get("STI_LIB") or DEFAULT_LIB_PATH

STATUS_NAMES = {0: "STI_OK", 1: "STI_ERR_INVALID_ARG", 2: "STI_ERR_UNSUPPORTED", 3: "STI_ERR_CUDA",
                4: "STI_ERR_INDEX_RANGE", 5: "STI_ERR_DEVICE_TIMEOUT", 6: "STI_ERR_DEVICE_UNSUPPORTED",
                7: "STI_ERR_TOO_LARGE"}
FLAG_INDEX_RANGE, FLAG_TIMEOUT, FLAG_CHUNKED = 1, 2, 4

EXPORTS = ["sti_status_string", "sti_last_cuda_error", "sti_version", "sti_read_device_status", "sti_window_idxs",
           "sti_idx_scores_workspace_size", "sti_idx_scores", "sti_idx_topk_workspace_size", "sti_idx_topk",
           "sti_sparse_attn_workspace_size", "sti_sparse_attn_sink", "sti_sparse_attn_sink_rope",
           "sti_sparse_attn_sink_fp4kv",
           "sti_decode_workspace_size",
           "sti_decode_fused", "sti_decode_kernel_count", "sti_decode_fused_noalloc", "sti_decode_noalloc_status",
           "sti_selftest_wait_timeout", "sti_window_idxs_chunked", "sti_idx_scores_mxfp4"]


class StiError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}" + (f" ({detail})" if detail else ""))


class DecodeArgs(ctypes.Structure):
    """Mirror of sti_decode_args."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("window_kv", ctypes.c_void_p), ("window_bstride", ctypes.c_int64),
        ("comp_kv", ctypes.c_void_p), ("comp_bstride", ctypes.c_int64), ("attn_sink", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_float), ("h", ctypes.c_int), ("d", ctypes.c_int), ("window_size", ctypes.c_int),
        ("iq", ctypes.c_void_p), ("ik", ctypes.c_void_p), ("ik_bstride", ctypes.c_int64), ("w", ctypes.c_void_p),
        ("index_scale", ctypes.c_float), ("Hi", ctypes.c_int), ("Di", ctypes.c_int), ("index_topk", ctypes.c_int),
        ("ratio", ctypes.c_int), ("n_cols", ctypes.c_int), ("start_pos", ctypes.c_void_p), ("b", ctypes.c_int),
        ("out", ctypes.c_void_p), ("topk_idxs", ctypes.c_void_p), ("q_ready", ctypes.c_void_p),
        ("rope_cs", ctypes.c_void_p), ("rope_dims", ctypes.c_int),
        ("ik_codes", ctypes.c_void_p), ("ik_codes_bstride", ctypes.c_int64), ("ik_scales", ctypes.c_void_p),
        ("ik_scales_bstride", ctypes.c_int64),
        ("comp_codes", ctypes.c_void_p), ("comp_codes_bstride", ctypes.c_int64), ("comp_scales", ctypes.c_void_p),
        ("comp_scales_bstride", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsti.so (built in-tree by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.sti_status_string.argtypes, L.sti_status_string.restype = [I], ctypes.c_char_p
        L.sti_last_cuda_error.argtypes, L.sti_last_cuda_error.restype = [], ctypes.c_char_p
        L.sti_version.argtypes, L.sti_version.restype = [], I
        L.sti_read_device_status.argtypes, L.sti_read_device_status.restype = [P, P, P], I
        L.sti_window_idxs.argtypes, L.sti_window_idxs.restype = [P, I, I, I, P, I64, P, P, P], I
        L.sti_window_idxs_chunked.argtypes, L.sti_window_idxs_chunked.restype = [P, I, I, I, P, I64, P, P], I
        L.sti_idx_scores_workspace_size.argtypes, L.sti_idx_scores_workspace_size.restype = [], SZ
        L.sti_idx_scores.argtypes = [P, P, I64, P, F, P, I, I, I, I, I, I, P, P, SZ, P]
        L.sti_idx_scores_mxfp4.argtypes = [P, P, I64, P, I64, P, F, P, I, I, I, I, I, I, P, P, SZ, P]
        L.sti_idx_scores_mxfp4.restype = I
        L.sti_idx_scores.restype = I
        L.sti_idx_topk_workspace_size.argtypes, L.sti_idx_topk_workspace_size.restype = [], SZ
        L.sti_idx_topk.argtypes = [P, P, I, I, I, I, I, ctypes.c_int32, P, I64, P, SZ, P]
        L.sti_idx_topk.restype = I
        L.sti_sparse_attn_workspace_size.argtypes = [I, I, I, I, I]
        L.sti_sparse_attn_workspace_size.restype = SZ
        L.sti_sparse_attn_sink.argtypes = [P, P, I64, P, I64, I, I, P, P, I64, F, I, I, I, I, I, P, P, P, SZ, P]
        L.sti_sparse_attn_sink.restype = I
        L.sti_sparse_attn_sink_rope.argtypes = [P, P, I64, P, I64, I, I, P, P, I64, F, I, I, I, I, I, P, I, P, P, P,
                                                SZ, P]
        L.sti_sparse_attn_sink_rope.restype = I
        L.sti_sparse_attn_sink_fp4kv.argtypes = [P, P, I64, P, I64, P, I64, I, I, P, P, I64, F, I, I, I, I, I, P, P,
                                                 P, SZ, P]
        L.sti_sparse_attn_sink_fp4kv.restype = I
        L.sti_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.sti_decode_workspace_size.restype = SZ
        L.sti_decode_kernel_count.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.sti_decode_kernel_count.restype = I
        L.sti_decode_fused.argtypes = [ctypes.POINTER(DecodeArgs), P, SZ, P, P]
        L.sti_decode_fused.restype = I
        L.sti_selftest_wait_timeout.argtypes = [P, SZ, ctypes.c_uint32, P]
        L.sti_selftest_wait_timeout.restype = I
        L.sti_decode_fused_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), P]
        L.sti_decode_fused_noalloc.restype = I
        L.sti_decode_noalloc_status.argtypes = [P, P]
        L.sti_decode_noalloc_status.restype = I
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        detail = lib().sti_last_cuda_error().decode() if status == 3 else ""
        raise StiError(status, where, detail)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str, contiguous: bool = True):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def upload_bf16(bits, device="cuda") -> torch.Tensor:
    """A numpy array of bf16 bit patterns (uint16) as a torch.bfloat16 tensor on `device`."""
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def upload(a, device="cuda") -> torch.Tensor:
    """A numpy array (any dtype torch knows) as a tensor on `device`."""
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (torch allocates it; the library never does)."""
    return torch.zeros(max(256, int(nbytes)), dtype=torch.uint8, device=device or "cuda")


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, return and clear the STI_FLAG_* bits of a workspace's status word."""
    flags = ctypes.c_uint32(0)
    lib().sti_read_device_status(_ptr(ws), ctypes.byref(flags), _stream(stream))
    return int(flags.value)


# ---------------------------------------------------------------------------- entry points


def window_idxs(start_pos: torch.Tensor, seqlen: int, window_size: int, out: torch.Tensor | None = None,
                ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """get_window_topk_idxs for a batch: [b, seqlen, width] int32 (width = min(seqlen, W) in
    prefill, W in decode).  `out` may be a strided view whose rows are longer than width."""
    _need(start_pos, torch.int32, "start_pos")
    b = start_pos.numel()
    width = min(seqlen, window_size) if seqlen > 1 else window_size
    if out is None:
        out = torch.empty(b, seqlen, width, dtype=torch.int32, device=start_pos.device)
    if out.stride(-1) != 1:
        raise ValueError("out rows must be contiguous")
    row_stride = out.stride(-2) if out.dim() >= 2 else width
    _check(lib().sti_window_idxs(_ptr(start_pos), b, seqlen, window_size, _ptr(out), row_stride, None, _ptr(ws),
                                 _stream(stream)), "sti_window_idxs")
    return out


def window_idxs_chunked(start_pos: torch.Tensor, seqlen: int, window_size: int, out: torch.Tensor | None = None,
                        ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Window rows [b, seqlen, W] of a prefill chunk continuing its sequence, over the source
    [ring before the chunk (W rows) ; the chunk's seqlen rows] (sti_window_idxs_chunked)."""
    _need(start_pos, torch.int32, "start_pos")
    b = start_pos.numel()
    if out is None:
        out = torch.empty(b, seqlen, window_size, dtype=torch.int32, device=start_pos.device)
    if out.stride(-1) != 1:
        raise ValueError("out rows must be contiguous")
    row_stride = out.stride(-2) if out.dim() >= 2 else window_size
    _check(lib().sti_window_idxs_chunked(_ptr(start_pos), b, seqlen, window_size, _ptr(out), row_stride, _ptr(ws),
                                         _stream(stream)), "sti_window_idxs_chunked")
    return out


def idx_scores(iq: torch.Tensor, ik: torch.Tensor, w: torch.Tensor, c: float, start_pos: torch.Tensor,
               n_cols: int, ratio: int, out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Indexer scores [b, s, n_cols] fp32.  iq [b,s,Hi,Di], ik [b,cap,Di] (cap >= n_cols), w [b,s,Hi] bf16."""
    _need(iq, torch.bfloat16, "iq")
    _need(w, torch.bfloat16, "w")
    _need(start_pos, torch.int32, "start_pos")
    _need(ik, torch.bfloat16, "ik", contiguous=False)
    b, s, Hi, Di = iq.shape
    if ik.dim() != 3 or ik.stride(2) != 1 or ik.stride(1) != Di:
        raise ValueError("ik must be [b, rows, Di] with contiguous rows")
    if out is None:
        out = torch.empty(b, s, n_cols, dtype=torch.float32, device=iq.device)
    ws = ws if ws is not None else workspace(lib().sti_idx_scores_workspace_size(), iq.device)
    _check(lib().sti_idx_scores(_ptr(iq), _ptr(ik), ik.stride(0), _ptr(w), float(c), _ptr(start_pos), b, s, Hi, Di,
                                n_cols, ratio, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "sti_idx_scores")
    return out


def idx_scores_mxfp4(iq: torch.Tensor, ik_codes: torch.Tensor, ik_scales: torch.Tensor, w: torch.Tensor, c: float,
                     start_pos: torch.Tensor, n_cols: int, ratio: int, out: torch.Tensor | None = None,
                     ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Indexer scores with MXFP4 keys: ik_codes uint8 [b, cap, Di/2], ik_scales uint8
    [b, cap, Di/32] (cap >= n_cols); the queries are quantised to MXFP4 in the kernel."""
    _need(iq, torch.bfloat16, "iq")
    _need(w, torch.bfloat16, "w")
    _need(start_pos, torch.int32, "start_pos")
    b, s, Hi, Di = iq.shape
    for name, t, inner in (("ik_codes", ik_codes, Di // 2), ("ik_scales", ik_scales, Di // 32)):
        if t.dtype != torch.uint8 or t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != inner:
            raise ValueError(f"{name} must be uint8 [b, rows, {inner}] with contiguous rows")
    if out is None:
        out = torch.empty(b, s, n_cols, dtype=torch.float32, device=iq.device)
    ws = ws if ws is not None else workspace(lib().sti_idx_scores_workspace_size(), iq.device)
    _check(lib().sti_idx_scores_mxfp4(_ptr(iq), _ptr(ik_codes), ik_codes.stride(0), _ptr(ik_scales),
                                      ik_scales.stride(0), _ptr(w), float(c), _ptr(start_pos), b, s, Hi, Di, n_cols,
                                      ratio, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "sti_idx_scores_mxfp4")
    return out


def idx_topk(scores: torch.Tensor, start_pos: torch.Tensor, ratio: int, k: int, offset: int,
             out: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Top-k visible positions per row, ascending, + offset, -1 padded: [b, s, k] int32.
    `out` may be a column slice of a wider index buffer (row stride taken from it)."""
    _need(scores, torch.float32, "scores")
    _need(start_pos, torch.int32, "start_pos")
    b, s, n_cols = scores.shape
    if out is None:
        out = torch.empty(b, s, k, dtype=torch.int32, device=scores.device)
    if out.stride(-1) != 1:
        raise ValueError("out rows must be contiguous")
    ws = ws if ws is not None else workspace(lib().sti_idx_topk_workspace_size(), scores.device)
    _check(lib().sti_idx_topk(_ptr(scores), _ptr(start_pos), b, s, n_cols, ratio, k, offset, _ptr(out),
                              out.stride(-2), _ptr(ws), ws.numel(), _stream(stream)), "sti_idx_topk")
    return out


def sparse_attn_workspace_size(b: int, s: int, h: int, d: int, k: int) -> int:
    return int(lib().sti_sparse_attn_workspace_size(b, s, h, d, k))


def sparse_attn_sink(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor, topk_idxs: torch.Tensor,
                     softmax_scale: float, kv2: torch.Tensor | None = None, out: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None,
                     rope_cs: torch.Tensor | None = None) -> torch.Tensor:
    """sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale) with an optional second KV source:
    row r < kv.shape[1] is kv[b, r], row r >= kv.shape[1] is kv2[b, r - kv.shape[1]].
    rope_cs: optional fp32 [b, s, rd/2, 2] (cos, sin): the output's last rd dims are rotated
    back by those angles in the same kernel (sti_sparse_attn_sink_rope)."""
    _need(q, torch.bfloat16, "q")
    _need(attn_sink, torch.float32, "attn_sink")
    _need(kv, torch.bfloat16, "kv", contiguous=False)
    if topk_idxs.dtype != torch.int32 or topk_idxs.stride(-1) != 1:
        raise ValueError("topk_idxs must be int32 with contiguous rows")
    b, s, h, d = q.shape
    k = topk_idxs.shape[-1]
    n1 = kv.shape[1]
    n2 = 0 if kv2 is None else kv2.shape[1]
    for name, t in (("kv", kv), ("kv2", kv2)):
        if t is not None and (t.stride(2) != 1 or t.stride(1) != d):
            raise ValueError(f"{name} must be [b, rows, d] with contiguous rows")
    if out is None:
        out = torch.empty_like(q)
    ws = ws if ws is not None else workspace(sparse_attn_workspace_size(b, s, h, d, k), q.device)
    if rope_cs is not None:
        _need(rope_cs, torch.float32, "rope_cs")
        if rope_cs.dim() != 4 or tuple(rope_cs.shape[:2]) != (b, s) or rope_cs.shape[3] != 2:
            raise ValueError("rope_cs must be [b, s, rd/2, 2]")
        _check(lib().sti_sparse_attn_sink_rope(
            _ptr(q), _ptr(kv), kv.stride(0), _ptr(kv2), 0 if kv2 is None else kv2.stride(0), n1, n2, _ptr(attn_sink),
            _ptr(topk_idxs), topk_idxs.stride(-2), float(softmax_scale), b, s, h, d, k, _ptr(rope_cs),
            2 * rope_cs.shape[2], _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
            "sti_sparse_attn_sink_rope")
        return out
    _check(lib().sti_sparse_attn_sink(
        _ptr(q), _ptr(kv), kv.stride(0), _ptr(kv2), 0 if kv2 is None else kv2.stride(0), n1, n2, _ptr(attn_sink),
        _ptr(topk_idxs), topk_idxs.stride(-2), float(softmax_scale), b, s, h, d, k, _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel(), _stream(stream)), "sti_sparse_attn_sink")
    return out


def sparse_attn_sink_fp4kv(q: torch.Tensor, kv: torch.Tensor, kv2_codes: torch.Tensor, kv2_scales: torch.Tensor,
                           attn_sink: torch.Tensor, topk_idxs: torch.Tensor, softmax_scale: float,
                           out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                           ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """sparse_attn_sink with the second (compressed) source as fp4 rows: kv2_codes uint8
    [b, rows, d/2] and kv2_scales uint8 [b, rows, d/16] (E4M3 scale per 16 elements), rows
    contiguous; row r >= kv.shape[1] of the index space is compressed row r - kv.shape[1]."""
    _need(q, torch.bfloat16, "q")
    _need(attn_sink, torch.float32, "attn_sink")
    _need(kv, torch.bfloat16, "kv", contiguous=False)
    if topk_idxs.dtype != torch.int32 or topk_idxs.stride(-1) != 1:
        raise ValueError("topk_idxs must be int32 with contiguous rows")
    b, s, h, d = q.shape
    k = topk_idxs.shape[-1]
    n1, n2 = kv.shape[1], kv2_codes.shape[1]
    if kv.stride(2) != 1 or kv.stride(1) != d:
        raise ValueError("kv must be [b, rows, d] with contiguous rows")
    for name, t, inner in (("kv2_codes", kv2_codes, d // 2), ("kv2_scales", kv2_scales, d // 16)):
        if t.dtype != torch.uint8 or t.dim() != 3 or t.shape[2] != inner or t.stride(2) != 1 or t.stride(1) != inner:
            raise ValueError(f"{name} must be uint8 [b, rows, {inner}] with contiguous rows")
    if kv2_scales.shape[1] < n2:
        raise ValueError("kv2_scales must hold as many rows as kv2_codes")
    if out is None:
        out = torch.empty_like(q)
    ws = ws if ws is not None else workspace(sparse_attn_workspace_size(b, s, h, d, k), q.device)
    _check(lib().sti_sparse_attn_sink_fp4kv(
        _ptr(q), _ptr(kv), kv.stride(0), _ptr(kv2_codes), kv2_codes.stride(0), _ptr(kv2_scales), kv2_scales.stride(0),
        n1, n2, _ptr(attn_sink), _ptr(topk_idxs), topk_idxs.stride(-2), float(softmax_scale), b, s, h, d, k,
        _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), "sti_sparse_attn_sink_fp4kv")
    return out


def decode_args(q, window_kv, comp_kv, attn_sink, softmax_scale, iq, ik, w, index_scale, start_pos, ratio, n_cols,
                index_topk, out=None, topk_idxs=None, q_ready=None, rope_cs=None, ik_codes=None,
                ik_scales=None, comp_codes=None, comp_scales=None) -> tuple[DecodeArgs, torch.Tensor, torch.Tensor]:
    """Fill sti_decode_args from tensors.  q [b,h,d] (or [b,1,h,d]), window_kv [b,W,d],
    comp_kv [b,cap,d], iq [b,Hi,Di] (or [b,1,Hi,Di]), ik [b,cap,Di], w [b,Hi] (or [b,1,Hi]).
    q_ready: optional torch.cuda.Event (already recorded once) the attention step waits for.
    rope_cs: optional fp32 [b, rd/2, 2] (cos, sin) of the output's inverse rotation.
    ik_codes / ik_scales: optional MXFP4 index keys (uint8 [b, cap, Di/2] / [b, cap, Di/32]);
    then `ik` is not read (it may be None).
    comp_codes / comp_scales: optional fp4 compressed KV rows (uint8 [b, cap, d/2] / [b, cap, d/16]);
    then `comp_kv` is not read (it may be None).
    The returned struct keeps references to every tensor it points to."""
    b = q.shape[0]
    h, d = q.shape[-2], q.shape[-1]
    Hi, Di = iq.shape[-2], iq.shape[-1]
    W = window_kv.shape[1]
    for name, t, dt in (("q", q, torch.bfloat16), ("iq", iq, torch.bfloat16), ("w", w, torch.bfloat16),
                        ("attn_sink", attn_sink, torch.float32), ("start_pos", start_pos, torch.int32)):
        _need(t, dt, name)
    for name, t, inner in (("window_kv", window_kv, d), ("comp_kv", comp_kv, d), ("ik", ik, Di)):
        if t is None and ((name == "ik" and ik_codes is not None) or (name == "comp_kv" and comp_codes is not None)):
            continue
        _need(t, torch.bfloat16, name, contiguous=False)
        if t.stride(2) != 1 or t.stride(1) != inner:
            raise ValueError(f"{name} must have contiguous rows")
    if out is None:
        out = torch.empty(b, h, d, dtype=torch.bfloat16, device=q.device)
    if topk_idxs is None:
        topk_idxs = torch.empty(b, W + index_topk, dtype=torch.int32, device=q.device)
    a = DecodeArgs(_ptr(q), _ptr(window_kv), window_kv.stride(0), _ptr(comp_kv),
                   0 if comp_kv is None else comp_kv.stride(0), _ptr(attn_sink),
                   float(softmax_scale), h, d, W, _ptr(iq), _ptr(ik), 0 if ik is None else ik.stride(0), _ptr(w),
                   float(index_scale), Hi,
                   Di, index_topk, ratio, n_cols, _ptr(start_pos), b, _ptr(out), _ptr(topk_idxs),
                   q_ready.cuda_event if q_ready is not None else None)
    if rope_cs is not None:
        _need(rope_cs, torch.float32, "rope_cs")
        if rope_cs.dim() != 3 or rope_cs.shape[0] != b or rope_cs.shape[2] != 2:
            raise ValueError("rope_cs must be [b, rd/2, 2]")
        a.rope_cs, a.rope_dims = _ptr(rope_cs), 2 * rope_cs.shape[1]
    if ik_codes is not None:
        for name, t, inner in (("ik_codes", ik_codes, Di // 2), ("ik_scales", ik_scales, Di // 32)):
            if t is None or t.dtype != torch.uint8 or t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != inner:
                raise ValueError(f"{name} must be uint8 [b, rows, {inner}] with contiguous rows")
        a.ik_codes, a.ik_codes_bstride = _ptr(ik_codes), ik_codes.stride(0)
        a.ik_scales, a.ik_scales_bstride = _ptr(ik_scales), ik_scales.stride(0)
    if comp_codes is not None:
        for name, t, inner in (("comp_codes", comp_codes, d // 2), ("comp_scales", comp_scales, d // 16)):
            if t is None or t.dtype != torch.uint8 or t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != inner:
                raise ValueError(f"{name} must be uint8 [b, rows, {inner}] with contiguous rows")
        a.comp_codes, a.comp_codes_bstride = _ptr(comp_codes), comp_codes.stride(0)
        a.comp_scales, a.comp_scales_bstride = _ptr(comp_scales), comp_scales.stride(0)
    # the struct holds raw device pointers: keep their tensors alive as long as it lives
    a.tensors = (q, window_kv, comp_kv, attn_sink, iq, ik, w, start_pos, out, topk_idxs, q_ready, rope_cs, ik_codes,
                 ik_scales, comp_codes, comp_scales)
    return a, out, topk_idxs


def decode_workspace_size(a: DecodeArgs) -> int:
    return int(lib().sti_decode_workspace_size(ctypes.byref(a)))


def decode_kernel_count(a: DecodeArgs) -> int:
    """Kernels one decode_fused call enqueues for these arguments (see sti_decode_kernel_count)."""
    n = int(lib().sti_decode_kernel_count(ctypes.byref(a)))
    if n < 0:
        raise StiError(1, "sti_decode_kernel_count")
    return n


def decode_fused(a: DecodeArgs, ws: torch.Tensor, stream=None, events=None):
    """One decode step of an index-source layer: scores, top-k with window indices, sparse
    attention.  `events`: optional 4 torch.cuda.Event(enable_timing=True), recorded before
    the first kernel and after each of the three."""
    ev = None
    if events is not None:
        for e in events:
            if e.cuda_event == 0:   # torch creates the event on first record
                e.record()
        ev = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    _check(lib().sti_decode_fused(ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream), ev), "sti_decode_fused")


def decode_fused_noalloc(a: DecodeArgs, stream=None):
    """The decode step of decode_fused without a workspace: its scratch is a fixed array inside
    the library (for callers that cannot allocate device memory).  Calls that overlap on the GPU
    race on that array; the first call on a device should come before any stream capture."""
    _check(lib().sti_decode_fused_noalloc(ctypes.byref(a), _stream(stream)), "sti_decode_fused_noalloc")


def decode_noalloc_status(stream=None) -> int:
    """Synchronise and return the STI_FLAG_* bits the last no-allocation call left."""
    flags = ctypes.c_uint32(0)
    lib().sti_decode_noalloc_status(ctypes.byref(flags), _stream(stream))
    return int(flags.value)


def selftest_wait_timeout(ws: torch.Tensor, limit_us: int = 2000, stream=None) -> None:
    """Launch the kernel whose wait nothing satisfies (see sti_selftest_wait_timeout)."""
    _check(lib().sti_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)),
           "sti_selftest_wait_timeout")
