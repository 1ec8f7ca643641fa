"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libsti():
    from sparse_top_attention_indexer_gb300 import _build

    _build.build()
    import sparse_top_attention_indexer_gb300 as m

    return m.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "sti.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(sti_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(libsti):
    names = _declared()
    assert "sti_idx_scores" in names and "sti_sparse_attn_sink" in names and "sti_decode_fused" in names
    for n in names:
        assert hasattr(libsti, n), f"{n} declared in sti.h but not exported"


def test_binding_lists_every_export():
    import sparse_top_attention_indexer_gb300 as m

    assert sorted(m.EXPORTS) == _declared()


def test_status_strings_and_version(libsti):
    assert libsti.sti_status_string(0) == b"STI_OK"
    assert libsti.sti_status_string(4) == b"STI_ERR_INDEX_RANGE"
    assert libsti.sti_version() >= 100


def test_host_argument_checks(libsti):
    """Invalid arguments return before any CUDA call (no GPU needed)."""
    fake = 1 << 20     # aligned non-null pointer value; never dereferenced on the host
    P = ctypes.c_void_p
    # workspace missing / misaligned
    assert libsti.sti_idx_scores(P(fake), P(fake), 128 * 100, P(fake), 1.0, P(fake), 1, 1, 32, 128, 100, 4, P(fake),
                                 None, 256, None) == 1
    assert libsti.sti_idx_scores(P(fake), P(fake), 128 * 100, P(fake), 1.0, P(fake), 1, 1, 32, 128, 100, 4, P(fake),
                                 P(fake + 8), 256, None) == 1
    # unsupported index head dim / head count
    assert libsti.sti_idx_scores(P(fake), P(fake), 100 * 96, P(fake), 1.0, P(fake), 1, 1, 32, 96, 100, 4, P(fake),
                                 P(fake), 256, None) == 2
    assert libsti.sti_idx_scores(P(fake), P(fake), 100 * 128, P(fake), 1.0, P(fake), 1, 1, 12, 128, 100, 4, P(fake),
                                 P(fake), 256, None) == 2
    # key batch stride too small / not a multiple of 8
    assert libsti.sti_idx_scores(P(fake), P(fake), 128 * 99, P(fake), 1.0, P(fake), 1, 1, 32, 128, 100, 4, P(fake),
                                 P(fake), 256, None) == 1
    assert libsti.sti_idx_scores(P(fake), P(fake), 128 * 100 + 4, P(fake), 1.0, P(fake), 1, 1, 32, 128, 100, 4,
                                 P(fake), P(fake), 256, None) == 1
    # top-k: k too large, row stride smaller than k
    assert libsti.sti_idx_topk(P(fake), P(fake), 1, 1, 100, 4, 5000, 0, P(fake), 5000, P(fake), 256, None) == 2
    assert libsti.sti_idx_topk(P(fake), P(fake), 1, 1, 100, 4, 64, 0, P(fake), 32, P(fake), 256, None) == 1
    # attention: too many heads, head dim not a multiple of 64, index row stride < k, small workspace
    assert libsti.sti_sparse_attn_sink(P(fake), P(fake), 100 * 512, None, 0, 100, 0, P(fake), P(fake), 640, 0.1, 1,
                                       1, 65, 512, 640, P(fake), None, P(fake), 1 << 30, None) == 2
    assert libsti.sti_sparse_attn_sink(P(fake), P(fake), 100 * 96, None, 0, 100, 0, P(fake), P(fake), 640, 0.1, 1, 1,
                                       64, 96, 640, P(fake), None, P(fake), 1 << 30, None) == 2
    assert libsti.sti_sparse_attn_sink(P(fake), P(fake), 100 * 512, None, 0, 100, 0, P(fake), P(fake), 100, 0.1, 1,
                                       1, 64, 512, 640, P(fake), None, P(fake), 1 << 30, None) == 1
    assert libsti.sti_sparse_attn_sink(P(fake), P(fake), 100 * 512, None, 0, 100, 0, P(fake), P(fake), 640, 0.1, 2,
                                       1, 64, 512, 640, P(fake), None, P(fake), 128, None) == 1
    # second source missing while n2 > 0
    assert libsti.sti_sparse_attn_sink(P(fake), P(fake), 100 * 512, None, 0, 100, 10, P(fake), P(fake), 640, 0.1,
                                       4096, 1, 64, 512, 640, P(fake), None, P(fake), 1 << 30, None) == 1
    # window: row stride shorter than the width; empty batch is a no-op
    assert libsti.sti_window_idxs(P(fake), 1, 1, 128, P(fake), 64, None, None, None) == 1
    assert libsti.sti_window_idxs(None, 0, 1, 128, None, 128, None, None, None) == 0


def test_output_rotation_argument_checks(libsti):
    """rope_dims must be even, in [1, d] (attention entry point; 0 allowed in the decode
    arguments), and come with a table; all of it is checked on the host."""
    fake = 1 << 20
    P = ctypes.c_void_p
    head = (P(fake), P(fake), 100 * 512, None, 0, 100, 0, P(fake), P(fake), 640, 0.1, 1, 1, 64, 512, 640)
    tail = (P(fake), None, P(fake), 1 << 30, None)
    for cs, rd in ((P(fake), 0), (P(fake), 63), (P(fake), 514), (P(fake), -2), (None, 64)):
        assert libsti.sti_sparse_attn_sink_rope(*head, cs, rd, *tail) == 1, (cs, rd)
    import sparse_top_attention_indexer_gb300 as m

    a = m.DecodeArgs()
    a.b, a.window_size, a.index_topk, a.n_cols, a.d = 1, 128, 512, 1024, 512
    for cs, rd in ((P(fake), 63), (P(fake), 514), (None, 64)):
        a.rope_cs, a.rope_dims = cs, rd
        assert libsti.sti_decode_fused(ctypes.byref(a), P(fake), 1 << 30, None, None) == 1, (cs, rd)
        assert libsti.sti_decode_fused_noalloc(ctypes.byref(a), None) == 1, (cs, rd)


def test_fp4kv_argument_checks(libsti):
    """The fp4 compressed rows' pointers and batch strides are checked on the host."""
    fake = 1 << 20
    P = ctypes.c_void_p
    n2, d = 100, 512

    def call(codes=P(fake), cb=n2 * d // 2, scales=P(fake), sb=n2 * d // 16):
        return libsti.sti_sparse_attn_sink_fp4kv(P(fake), P(fake), 128 * d, codes, cb, scales, sb, 128, n2, P(fake),
                                                 P(fake), 640, 0.1, 1, 1, 64, d, 640, P(fake), None, P(fake),
                                                 1 << 30, None)

    assert call(codes=P(fake + 8)) == 1          # codes not 16-byte aligned
    assert call(codes=None) == 1
    assert call(scales=None) == 1
    assert call(cb=n2 * d // 2 - 16) == 1        # codes batch stride short of n2 rows
    assert call(sb=n2 * d // 16 + 8) == 1        # scales batch stride not a multiple of 16


def test_decode_fp4kv_rows_need_the_fused_shape(libsti):
    """fp4 compressed rows in the decode arguments: a shape the fused kernel does not take (32
    heads) is refused on the host, before anything is enqueued, and the kernel count says so."""
    fake = 1 << 20
    P = ctypes.c_void_p
    import sparse_top_attention_indexer_gb300 as m

    a = m.DecodeArgs()
    a.q, a.window_kv, a.window_bstride, a.attn_sink = P(fake), P(fake), 128 * 512, P(fake)
    a.h, a.d, a.window_size, a.softmax_scale = 32, 512, 128, 0.04
    a.iq, a.ik, a.ik_bstride, a.w, a.index_scale = P(fake), P(fake), 1024 * 128, P(fake), 0.01
    a.Hi, a.Di, a.index_topk, a.ratio, a.n_cols = 32, 128, 512, 4, 1024
    a.start_pos, a.b, a.out, a.topk_idxs = P(fake), 2, P(fake), P(fake)
    a.comp_codes, a.comp_codes_bstride = P(fake), 1024 * 256
    a.comp_scales, a.comp_scales_bstride = P(fake), 1024 * 32
    assert libsti.sti_decode_kernel_count(ctypes.byref(a)) == -1
    assert libsti.sti_decode_fused(ctypes.byref(a), P(fake), 1 << 30, None, None) == 2
    assert libsti.sti_decode_fused_noalloc(ctypes.byref(a), None) == 2
    a.comp_codes = None   # the same shape with bf16 rows (none given here): three kernels
    a.comp_kv, a.comp_bstride = P(fake), 1024 * 512
    assert libsti.sti_decode_kernel_count(ctypes.byref(a)) == 3


def test_selftest_argument_checks(libsti):
    fake = 1 << 20
    P = ctypes.c_void_p
    assert libsti.sti_selftest_wait_timeout(None, 256, 1000, None) == 1
    assert libsti.sti_selftest_wait_timeout(P(fake), 256, 0, None) == 1
    assert libsti.sti_selftest_wait_timeout(P(fake), 256, 200000, None) == 1


def test_window_width_reported(libsti):
    w = ctypes.c_int(0)
    assert libsti.sti_window_idxs(None, 0, 300, 128, None, 128, ctypes.byref(w), None, None) == 0
    assert w.value == 128
    assert libsti.sti_window_idxs(None, 0, 37, 128, None, 128, ctypes.byref(w), None, None) == 0
    assert w.value == 37
    assert libsti.sti_window_idxs(None, 0, 1, 128, None, 128, ctypes.byref(w), None, None) == 0
    assert w.value == 128


def test_workspace_sizes(libsti):
    assert libsti.sti_idx_scores_workspace_size() >= 4
    assert libsti.sti_idx_topk_workspace_size() >= 4
    # attention: the status word, then (for batches that may split a query over a cluster) the
    # fp32 [queries, h, d] accumulator the cluster adds its partial outputs into
    assert libsti.sti_sparse_attn_workspace_size(2, 1, 64, 512, 640) == 256 + 2 * 64 * 512 * 4
    assert libsti.sti_sparse_attn_workspace_size(256, 1, 64, 512, 640) == 256 + 256 * 64 * 512 * 4
    assert libsti.sti_sparse_attn_workspace_size(4096, 1, 64, 512, 640) == 256
    assert libsti.sti_sparse_attn_workspace_size(1, 3, 4, 64, 32) == 256 + 3 * 4 * 64 * 4
