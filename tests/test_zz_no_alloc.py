"""The no-allocation decode entry point (sti_decode_fused_noalloc).

It exists for callers that cannot give the library a device workspace -- a plugin inside a
runtime that owns all device memory, or a serving loop that must not touch the allocator once
it runs.  Its scratch is a fixed array inside the library.  These tests call it through the C
ABI and check that two calls in a row give what the workspace entry point (sti_decode_fused)
gives, and that sizes beyond the fixed scratch are refused before anything runs.  The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from tests._util import bf16_out_to_f64, check_attn, to_dev, to_dev_any


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    """Host-side limit check: nothing is enqueued, so no GPU is needed."""
    from sparse_top_attention_indexer_gb300 import _build

    _build.build()
    import sparse_top_attention_indexer_gb300 as sti

    L = sti.lib()
    fake = 1 << 20
    a = sti.DecodeArgs()
    a.q = a.window_kv = a.comp_kv = a.attn_sink = a.iq = a.ik = a.w = a.start_pos = a.out = a.topk_idxs = fake
    a.h, a.d, a.window_size, a.Hi, a.Di, a.index_topk, a.ratio = 64, 512, 128, 32, 128, 512, 4
    a.b, a.n_cols = 257, 16                      # batch above STI_NOALLOC_MAX_BATCH
    assert L.sti_decode_fused_noalloc(ctypes.byref(a), None) == 7
    a.b, a.n_cols = 256, (1 << 21) // 256 + 1    # scores above STI_NOALLOC_MAX_SCORES
    assert L.sti_decode_fused_noalloc(ctypes.byref(a), None) == 7
    assert L.sti_status_string(7) == b"STI_ERR_TOO_LARGE"


# Batches that take each of the scratch's uses: the head-split attention (64 heads, few queries);
# the row-split attention whose clusters add partial outputs into the scratch's accumulator (16
# heads: not head-split), which the call must clear; and more than 128 queries, where the
# accumulator is not used and no query splits.
NOALLOC_CASES = {
    "head_split": dict(b=6, start_pos=[8191, 4095, 1500, 300, 40, 2], n_cols=2048, h=64),
    "row_split_acc": dict(b=20, start_pos=[8191 - 397 * i for i in range(20)], n_cols=2048, h=16),
    "many_queries": dict(b=140, start_pos=[4095 - 29 * i for i in range(140)], n_cols=1024, h=64),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", list(NOALLOC_CASES))
def test_noalloc_matches_workspace_entry_twice(case):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_top_attention_indexer_gb300 as sti

    sti.lib()
    kw = NOALLOC_CASES[case]
    # ragged decode batch: sequences longer and shorter than index_topk, one with a filling ring
    shape = workloads.custom(f"noalloc_decode_{case}", b=kw["b"], s=1, start_pos=kw["start_pos"], seed=9090,
                             n_cols=kw["n_cols"], topk=512, h=kw["h"], d=512)
    data = workloads.make(shape)
    args = dict(q=to_dev(data["q"][0]), window_kv=to_dev(data["win"][0]), comp_kv=to_dev(data["comp"]),
                attn_sink=to_dev_any(data["sink"][0]), softmax_scale=shape.softmax_scale, iq=to_dev(data["iq"]),
                ik=to_dev(data["ik"]), w=to_dev(data["w"]), index_scale=shape.index_scale,
                start_pos=to_dev_any(data["start_pos"]), ratio=shape.ratio, n_cols=shape.n_cols,
                index_topk=shape.topk)

    # the workspace entry point
    a_ref, out_ref, idx_ref = sti.decode_args(**args)
    ws = sti.workspace(sti.decode_workspace_size(a_ref))
    sti.decode_fused(a_ref, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    ref_o = bf16_out_to_f64(out_ref)
    ref_i = idx_ref.cpu().numpy()

    # the no-allocation entry point, two calls in a row into the same outputs
    a, out, idx = sti.decode_args(**args)
    for call in range(2):
        out.fill_(0)
        idx.fill_(-7)
        sti.decode_fused_noalloc(a)
        torch.cuda.synchronize()
        assert sti.decode_noalloc_status() == 0, f"call {call}: device status set"
        np.testing.assert_array_equal(idx.cpu().numpy(), ref_i)
        check_attn(bf16_out_to_f64(out), ref_o)
