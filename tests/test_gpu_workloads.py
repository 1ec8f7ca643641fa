"""GPU parity on the named workloads at full size, in the launch configuration bench.py times
(its GpuPath), against the CPU oracle on the same seeded inputs.

Decode workloads (b=32 ctx 65536 at compression ratios 4, 2 and 1, and with MXFP4 index keys;
b=8 ctx 131072 with planted keys; b=64 ragged with three reuse layers) and the tiny prefill are compared element by element
on every output.  The 8192-query prefill and the 2048-query chunk continuing a sequence at
position 6144 are compared on a spread of sampled query rows (the oracle computes each one on
its own), and on properties that hold for every row at full size."""
import numpy as np
import pytest

import workloads
from tests._util import bf16_out_to_f64, check_attn, check_scores, check_topk_rows

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


@pytest.mark.parametrize("n", [1, 2, 4, 5, 6, 7, 9])
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
        ref_o, _ = orc.sparse_attn(data["q"][i], data["win"][i], data["sink"][i], ref_idx, shape.softmax_scale,
                                   kv2=data["comp"])
        mx, mn = check_attn(bf16_out_to_f64(path.out[i]), ref_o)
        print(f"workload {n} layer {i}: score rel err {worst:.2e}, banded rows {banded}, attn max {mx:.2e} "
              f"mean {mn:.2e}")


@pytest.mark.parametrize("n", [3, 8, 10])
def test_workload_prefill_sampled(gpu, orc, n):
    """The 8192-query prefill from position 0 (with bf16 and with fp4 compressed KV), and the
    2048-query chunk continuing at 6144."""
    shape = workloads.config(n)
    data = workloads.make(shape)
    path = _run(shape, data, gpu)
    s, W, K, r = shape.s, shape.window, shape.topk, shape.ratio
    sp0 = int(shape.start_pos[0])
    off = shape.win_rows                      # compressed rows follow the window source's rows
    got_s = path.scores_view()[0].cpu().numpy()
    got_i = path.idx[0].cpu().numpy()
    # properties of every row at full size
    t = np.arange(s)
    vis = np.minimum((sp0 + t + 1) // r, shape.n_cols)
    assert np.array_equal(np.isfinite(got_s).sum(axis=1), vis)
    n_valid = (got_i[:, W:] >= 0).sum(axis=1)
    assert np.array_equal(n_valid, np.minimum(vis, K))
    comp = got_i[:, W:]
    assert np.all((comp < 0) | ((comp >= off) & (comp < off + vis[:, None])))
    # sampled rows against the oracle (row t sees (start_pos + t + 1)//ratio groups)
    rows = np.unique(np.concatenate([np.arange(0, 8), np.linspace(8, s - 1, 40).astype(np.int64),
                                     [t for t in (2047, 2048, 2051) if t < s]]))
    sp = (sp0 + rows).astype(np.int32)
    iq = data["iq"][0][rows][:, None]
    w = data["w"][0][rows][:, None]
    ik = np.broadcast_to(data["ik"][0], (len(rows),) + data["ik"].shape[1:])
    ref_s = orc.index_score(iq, ik, w, shape.index_scale, sp, shape.n_cols, r)
    check_scores(got_s[rows][:, None], ref_s)
    ref_c = orc.topk(ref_s, sp, r, K, off)
    ref_w = (orc.window_topk_idxs_chunked(W, s, sp0) if shape.chunked else orc.window_topk_idxs(W, 1, s, 0)[0])[rows]
    np.testing.assert_array_equal(got_i[rows, :W], ref_w)
    check_topk_rows(got_i[rows, W:][:, None], ref_c, ref_s, off, K)
    idx = np.concatenate([ref_w[:, None], ref_c], axis=-1).reshape(1, len(rows), -1)
    if shape.fp4_kv:
        ref_o, _ = orc.sparse_attn_fp4kv(data["q"][0][0][rows][None], data["win"][0], data["comp_codes"],
                                         data["comp_scales"], data["sink"][0], idx, shape.softmax_scale)
    else:
        ref_o, _ = orc.sparse_attn(data["q"][0][0][rows][None], data["win"][0], data["sink"][0], idx,
                                   shape.softmax_scale, kv2=data["comp"])
    got_o = bf16_out_to_f64(path.out[0][0][rows])
    check_attn(got_o, ref_o[0])
