"""GPU parity on the named workloads at full size, in the launch configuration bench.py times
(its GpuPath), against the CPU oracle on the same seeded inputs.

Decode workloads (b=32 ctx 65536 at compression ratios 4, 2 and 1, and with MXFP4 index keys;
b=8 ctx 131072 with planted keys; b=64 ragged with three reuse layers), the tiny prefill, the
8192-query prefill (bf16 and fp4 compressed KV) and the 2048-query chunk continuing a sequence
at position 6144 are compared element by element on every output."""
import numpy as np
import pytest

import workloads
from tests._util import (ATTN_MAX_ABS, ATTN_MEAN_ABS, bf16_out_to_f64, check_attn, check_scores, check_topk_rows,
                         score_error_stats)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_top_attention_indexer_gb300 as m

    m.lib()
    return torch.device("cuda", 0)


def _run(shape, data, device):
    import torch

    import bench

    path = bench.GpuPath(shape, data, device)
    path.step()
    torch.cuda.synchronize()
    assert path.read_status() == 0
    return path


@pytest.mark.parametrize("n", [1, 2, 4, 5, 6, 7, 9, 11])
def test_workload_full(gpu, orc, n):
    shape = workloads.config(n)
    data = workloads.make(shape)
    path = _run(shape, data, gpu)
    sp = data["start_pos"]
    W, width = shape.window, shape.win_width
    # scores, every row and column
    if shape.fp4_keys:
        ref_s = orc.index_score_mxfp4(data["iq"], data["ik_codes"], data["ik_scales"], data["w"], shape.index_scale, sp,
                                      shape.n_cols, shape.ratio)
    else:
        ref_s = orc.index_score(data["iq"], data["ik"], data["w"], shape.index_scale, sp, shape.n_cols, shape.ratio)
    got_s = path.scores_view().cpu().numpy()
    worst = check_scores(got_s, ref_s)
    print(f"workload {n} scores: {score_error_stats(got_s, ref_s)}")
    # indices: window part exact, compressed part the same set outside the boundary band
    ref_c = orc.topk(ref_s, sp, shape.ratio, shape.topk, shape.win_rows)
    if shape.prefill:
        ref_w = orc.window_topk_idxs(W, 1, shape.s, 0)
    else:
        ref_w = np.concatenate([orc.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0)
    got_i = path.idx.cpu().numpy()
    np.testing.assert_array_equal(got_i[..., :width], ref_w)
    banded = check_topk_rows(got_i[..., width:], ref_c, ref_s, shape.win_rows, shape.topk)
    # attention of every layer (the oracle on its own indices)
    ref_idx = np.concatenate([ref_w, ref_c], axis=-1)
    for i in range(shape.n_layers):
        if shape.fp4_kv:
            ref_o, _ = orc.sparse_attn_fp4kv(data["q"][i], data["win"][i], data["comp_codes"], data["comp_scales"],
                                             data["sink"][i], ref_idx, shape.softmax_scale)
        else:
            ref_o, _ = orc.sparse_attn(data["q"][i], data["win"][i], data["sink"][i], ref_idx, shape.softmax_scale,
                                       kv2=data["comp"])
        mx, mn = check_attn(bf16_out_to_f64(path.out[i]), ref_o)
        print(f"workload {n} layer {i}: score rel err {worst:.2e}, banded rows {banded}, attn max {mx:.2e} "
              f"mean {mn:.2e}")


@pytest.mark.parametrize("n", [3, 8, 10])
def test_workload_prefill_full(gpu, orc, n):
    """The 8192-query prefill from position 0 (with bf16 and with fp4 compressed KV), and the
    2048-query chunk continuing at 6144: every query row's scores, top-k set, window row and
    attention output against the oracle (the attention in chunks of query rows, so the oracle's
    fp64 outputs stay a few hundred MB)."""
    shape = workloads.config(n)
    data = workloads.make(shape)
    path = _run(shape, data, gpu)
    s, W, K, r = shape.s, shape.window, shape.topk, shape.ratio
    sp0 = int(shape.start_pos[0])
    off = shape.win_rows                      # compressed rows follow the window source's rows
    got_s = path.scores_view().cpu().numpy()  # [1, s, n_cols]
    got_i = path.idx.cpu().numpy()            # [1, s, W + K]
    # every row of the scores (query t sees (start_pos + t + 1)//ratio groups)
    ref_s = orc.index_score(data["iq"], data["ik"], data["w"], shape.index_scale, data["start_pos"], shape.n_cols, r)
    worst = check_scores(got_s, ref_s)
    # every index row: window part exact, compressed part the same set outside the boundary band
    ref_c = orc.topk(ref_s, data["start_pos"], r, K, off)
    ref_w = (orc.window_topk_idxs_chunked(W, s, sp0)[None] if shape.chunked else orc.window_topk_idxs(W, 1, s, 0))
    np.testing.assert_array_equal(got_i[..., :W], ref_w)
    banded = check_topk_rows(got_i[..., W:], ref_c, ref_s, off, K)
    del ref_s, got_s
    # every attention row, on the oracle's own indices
    idx = np.concatenate([ref_w, ref_c], axis=-1)
    q = data["q"][0]
    got_o = path.out[0]
    mx = mn_sum = 0.0
    step = 1024
    for t0 in range(0, s, step):
        t1 = min(s, t0 + step)
        if shape.fp4_kv:
            ref_o, _ = orc.sparse_attn_fp4kv(q[:, t0:t1], data["win"][0], data["comp_codes"], data["comp_scales"],
                                             data["sink"][0], idx[:, t0:t1], shape.softmax_scale)
        else:
            ref_o, _ = orc.sparse_attn(q[:, t0:t1], data["win"][0], data["sink"][0], idx[:, t0:t1],
                                       shape.softmax_scale, kv2=data["comp"])
        err = np.abs(bf16_out_to_f64(got_o[:, t0:t1]) - ref_o)
        mx = max(mx, float(err.max()))
        mn_sum += float(err.sum())
    mn = mn_sum / (s * shape.h * shape.d)
    assert mx <= ATTN_MAX_ABS and mn <= ATTN_MEAN_ABS, f"attention error max {mx:.3e} mean {mn:.3e}"
    print(f"workload {n}: every row; score rel err {worst:.2e}, banded rows {banded}, attn max {mx:.2e} mean {mn:.2e}")
