"""GPU parity of each kernel against the CPU oracle on the same seeded inputs (small and
ragged shapes that span several tiles).  Called through the C ABI via the thin binding."""
import numpy as np
import pytest

import workloads
from tests._util import bf16_out_to_f64, check_attn, check_scores, check_topk_rows, to_dev, to_dev_any
from workloads import index_lists, rng_for, to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sti():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_top_attention_indexer_gb300 as m

    m.lib()
    return m


# ----------------------------------------------------------------- window indices


@pytest.mark.parametrize("W,s,sps", [(4, 6, [0]), (16, 256, [0, 0]), (128, 300, [0]),
                                     (128, 1, [0, 1, 2, 127, 128, 65535, 131071]), (4, 1, [2, 7, 9])])
def test_window_idxs(sti, orc, W, s, sps):
    sp = np.array(sps, np.int32)
    got = sti.window_idxs(to_dev_any(sp), s, W).cpu().numpy()
    for bi, v in enumerate(sps):
        want = orc.window_topk_idxs(W, 1, s, int(v))[0]
        if s == 1 and v == 0:
            # the page's prefill branch gives the single row [0]; the ring layout lists the same
            # single slot among W entries (slot order does not matter to sparse_attn)
            assert sorted(int(x) for x in got[bi, 0] if x >= 0) == [0]
            continue
        np.testing.assert_array_equal(got[bi], want)


@pytest.mark.parametrize("W,s,sps", [(128, 300, [6144, 1, 5000]), (16, 40, [0, 3, 17]), (4, 1, [9])])
def test_window_idxs_chunked(sti, orc, W, s, sps):
    import torch

    sp = torch.tensor(sps, dtype=torch.int32, device="cuda")
    got = sti.window_idxs_chunked(sp, s, W).cpu().numpy()
    for bi, v in enumerate(sps):
        np.testing.assert_array_equal(got[bi], orc.window_topk_idxs_chunked(W, s, int(v)))


def test_window_idxs_flags_chunked_prefill(sti):
    ws = sti.workspace(256)
    got = sti.window_idxs(to_dev_any(np.array([0, 5], np.int32)), 4, 8, ws=ws).cpu().numpy()
    assert sti.read_device_status(ws) & sti.FLAG_CHUNKED
    assert np.all(got[1] == -1)


def test_wait_timeout_reports_and_the_context_survives(sti):
    """A kernel wait that nothing satisfies gives up, flags STI_FLAG_TIMEOUT and returns; the
    next launches on the same context work."""
    ws = sti.workspace(256)
    sti.selftest_wait_timeout(ws, 2000)
    assert sti.read_device_status(ws) & sti.FLAG_TIMEOUT
    assert sti.read_device_status(ws) == 0   # cleared
    got = sti.window_idxs(to_dev_any(np.array([7], np.int32)), 1, 4, ws=ws).cpu().numpy()
    assert sorted(got[0, 0].tolist()) == [0, 1, 2, 3]   # position p sits in ring slot p % W
    assert sti.read_device_status(ws) == 0


# ----------------------------------------------------------------- index scores


@pytest.mark.parametrize("b,s,Hi,Di,n_cols,sps,ratio", [
    (1, 1, 32, 128, 300, [1199], 4),             # decode, ragged last tile
    (3, 1, 32, 128, 1000, [3999, 1000, 17], 4),  # ragged batch, one sequence sees only 4 groups
    (1, 37, 32, 128, 20, [0], 4),                # prefill with a partial query tile
    (1, 256, 4, 32, 64, [0], 4),                 # tiny-prefill shapes (Hi=4, Di=32)
    (2, 1, 32, 64, 513, [2051, 600], 4),
    (2, 9, 16, 128, 200, [0, 0], 2),
])
def test_idx_scores(sti, orc, b, s, Hi, Di, n_cols, sps, ratio):
    rng = rng_for(500 + b * s, Hi)
    cap = n_cols + 5
    iq = to_bf16_bits(rng.standard_normal((b, s, Hi, Di)))
    ik = to_bf16_bits(rng.standard_normal((b, cap, Di)))
    w = to_bf16_bits(rng.standard_normal((b, s, Hi)))
    sp = np.array(sps, np.int32)
    c = Di ** -0.5 * Hi ** -0.5
    ref = orc.index_score(iq, ik, w, c, sp, n_cols, ratio)
    got = sti.idx_scores(to_dev(iq), to_dev(ik), to_dev(w), c, to_dev_any(sp), n_cols, ratio).cpu().numpy()
    check_scores(got, ref)


# ----------------------------------------------------------------- top-k (same fp32 input on both sides)


@pytest.mark.parametrize("b,s,Hi,Di,n_cols,sps", [
    (3, 1, 32, 128, 1500, [6000, 399, 5999]),     # decode: one query per unit, ragged visibility
    (2, 1, 16, 128, 900, [3599, 1000]),           # decode, N = 16: E2M1 operands
    (1, 1, 4, 128, 130, [519]),                   # 4 heads padded to N = 16; a 2-key last tile
    (1, 40, 32, 128, 300, [0]),                   # prefill: 8 queries per unit
    (2, 3, 8, 64, 700, [2799, 100]),
    (1, 70, 4, 64, 200, [0]),                     # 64 queries per unit, several units
])
def test_idx_scores_mxfp4(sti, orc, b, s, Hi, Di, n_cols, sps):
    """MXFP4 keys and queries quantised in the kernel give the oracle's scores over the decoded
    values (OCP MXFP4 reading of fp4_act_quant): one query per unit with Di == 128 runs the codes as
    E2M1 MMA operands with the scales applied per block; otherwise the keys are decoded in shared
    memory (E5M2 with Di == 128, else bf16)."""
    import torch

    rng = rng_for(790 + Di, n_cols)
    sp = np.broadcast_to(np.asarray(sps, np.int32), (b,)).copy()
    iq = to_bf16_bits(rng.standard_normal((b, s, Hi, Di)) * np.exp2(rng.integers(-3, 4, size=(b, s, Hi, 1))))
    cap = (n_cols + 40 + 7) // 8 * 8      # scale rows per batch a multiple of 16 bytes
    codes = rng.integers(0, 256, size=(b, cap, Di // 2), dtype=np.uint8)
    scales = rng.integers(115, 135, size=(b, cap, Di // 32), dtype=np.uint8)
    w = to_bf16_bits(rng.standard_normal((b, s, Hi)))
    c = Di ** -0.5 * Hi ** -0.5
    ref = orc.index_score_mxfp4(iq, codes, scales, w, c, sp, n_cols, 4)
    ws = sti.workspace(256)
    got = sti.idx_scores_mxfp4(to_dev(iq), to_dev_any(codes), to_dev_any(scales), to_dev(w), c, to_dev_any(sp),
                               n_cols, 4, ws=ws).cpu().numpy()
    assert sti.read_device_status(ws) == 0
    check_scores(got, ref)


@pytest.mark.parametrize("s", [1, 3])
@pytest.mark.parametrize("case", ["key_outliers", "query_outliers", "zero_blocks"])
def test_idx_scores_mxfp4_scale_ranges(sti, orc, case, s):
    """Far-out block scales.  One query per unit (s = 1): the E2M1 operands take any scale, applied
    per block in fp32.  Several queries per unit (s = 3): a key tile runs as E5M2 only when every
    scale block of its visible keys, and of the unit's queries, has X in [-13, 13]; other tiles
    (here: tiles with far-out key scales, or a unit whose query block is 2^20 or 2^-30 times larger
    or smaller) are decoded to bf16, in the same launch.  All give the oracle's scores."""
    b, Hi, Di, n_cols = 4, 32, 128, 1500
    sps = [5999, 3000, 5999, 1200]
    rng = rng_for(795, len(case))
    sp = np.asarray(sps, np.int32) - (s - 1)
    q = rng.standard_normal((b, s, Hi, Di))
    cap = (n_cols + 7) // 8 * 8
    codes = rng.integers(0, 256, size=(b, cap, Di // 2), dtype=np.uint8)
    scales = rng.integers(118, 132, size=(b, cap, Di // 32), dtype=np.uint8)
    if case == "key_outliers":
        scales[0, 130, 1] = 100            # X = -27: tile 1 of sequence 0
        scales[2, 700, 3] = 150            # X = 23: tile 5 of sequence 2
        scales[3, 299, 0] = 0              # tile 2 of sequence 3, the last one it sees
        scales[1, 900, 2] = 200            # past what sequence 1 sees (750 keys): no effect
    elif case == "query_outliers":
        q[1, 0, 3, 32:64] *= 2.0 ** 20
        q[2, 0, 17, 96:] *= 2.0 ** -30
    else:
        codes[0, 256:384] = 0              # whole tiles of zero keys with out-of-range scales
        scales[0, 256:384] = 0
        q[3, 0, 5, :32] = 0.0              # an all-zero query block
    iq = to_bf16_bits(q)
    w = to_bf16_bits(rng.standard_normal((b, s, Hi)))
    c = Di ** -0.5 * Hi ** -0.5
    ref = orc.index_score_mxfp4(iq, codes, scales, w, c, sp, n_cols, 4)
    ws = sti.workspace(256)
    got = sti.idx_scores_mxfp4(to_dev(iq), to_dev_any(codes), to_dev_any(scales), to_dev(w), c, to_dev_any(sp),
                               n_cols, 4, ws=ws).cpu().numpy()
    assert sti.read_device_status(ws) == 0
    check_scores(got, ref)


@pytest.mark.parametrize("b,s,n_cols,k,sps,ratio", [
    (2, 1, 16384, 512, [65535, 40000], 4),
    (4, 1, 1000, 512, [3999, 2047, 2048, 7], 4),
    (1, 64, 2048, 512, [0], 1),
    (1, 4200, 2048, 512, [0], 1),                 # many short rows: one warp per row
    (1, 300, 75, 16, [0], 4),
    (1, 1, 32768, 512, [131071], 4),
    (2, 1, 40000, 100, [159999, 100000], 4),     # beyond the shared-memory staging size
])
def test_topk_exact(sti, orc, b, s, n_cols, k, sps, ratio):
    rng = rng_for(600 + n_cols, k)
    scores = rng.standard_normal((b, s, n_cols)).astype(np.float32)
    scores[..., 5] = scores[..., 9]   # exact ties exercise the lower-position rule
    sp = np.array(sps, np.int32)
    offset = 128
    ref = orc.topk(scores.astype(np.float64), sp, ratio, k, offset)
    got = sti.idx_topk(to_dev_any(scores), to_dev_any(sp), ratio, k, offset).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("levels", [3, 40])
def test_topk_many_ties(sti, orc, levels):
    """Prefill rows (one warp a row) whose scores take only a few values: the k-th largest key is
    shared by many positions, so the lower-position rule decides most of the set."""
    rng = rng_for(602, levels)
    b, s, n_cols, k = 2, 2100, 2048, 512   # 4200 rows: the warp-per-row kernel
    scores = rng.integers(0, levels, size=(b, s, n_cols)).astype(np.float32) * 0.25 - 1.0
    scores[0, 2050, :] = 0.5                           # one row all equal (its bin too large to list)
    sp = np.array([0, 0], np.int32)
    ref = orc.topk(scores.astype(np.float64), sp, 1, k, 7)
    got = sti.idx_topk(to_dev_any(scores), to_dev_any(sp), 1, k, 7).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_topk_writes_into_wider_rows(sti, orc):
    import torch

    rng = rng_for(601, 0)
    scores = rng.standard_normal((3, 1, 700)).astype(np.float32)
    sp = np.array([2799, 100, 2000], np.int32)
    buf = torch.full((3, 1, 40 + 64), 7, dtype=torch.int32, device="cuda")
    sti.idx_topk(to_dev_any(scores), to_dev_any(sp), 4, 64, 40, out=buf[..., 40:])
    got = buf.cpu().numpy()
    assert np.all(got[..., :40] == 7)
    np.testing.assert_array_equal(got[..., 40:], orc.topk(scores.astype(np.float64), sp, 4, 64, 40))


# ----------------------------------------------------------------- sparse attention


@pytest.mark.parametrize("b,s,h,d,k,n1,n2,empty", [
    (2, 1, 64, 512, 640, 128, 3000, 0),     # decode shape: split over several CTAs
    (1, 3, 64, 512, 300, 200, 90, 1),       # k not a multiple of the tile, one all -1 query
    (1, 40, 4, 64, 32, 40, 10, 2),          # tiny-prefill shapes (h=4, d=64)
    (3, 2, 16, 128, 129, 64, 64, 0),
    (1, 200, 64, 512, 200, 256, 256, 3),    # enough queries that no split happens
])
def test_sparse_attn(sti, orc, b, s, h, d, k, n1, n2, empty):
    import torch

    rng = rng_for(700 + k, h)
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1 + n2, masked_frac=0.1, empty_rows=empty)
    scale = d ** -0.5
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, scale, kv2=kv2)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), scale, kv2=to_dev(kv2),
                               lse=lse)
    check_attn(bf16_out_to_f64(out), ref)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("b,s,h,d,k,n1,n2,ws_full", [
    (2, 1, 64, 512, 640, 128, 300, True),     # decode shape: window + compressed rows, split over a cluster
    (3, 1, 64, 512, 640, 128, 2000, False),   # decode shape, one CTA per query
    (1, 70, 64, 512, 256, 200, 100, False),   # several queries
    (1, 400, 48, 512, 640, 128, 900, False),  # more queries than SMs: the streamed kernel, 48 heads
    (2, 5, 16, 64, 300, 10, 700, True),       # small rows (d = 64: 4 scale bytes per row)
])
def test_sparse_attn_fp4kv(sti, orc, b, s, h, d, k, n1, n2, ws_full):
    """The compressed source as fp4 rows (E2M1 codes, an E4M3 scale per 16 elements; the form
    Attention._compress_kv gives the latent) decoded in the gather: the oracle's attention over
    the decoded rows.  Random masked slots, all -1 rows, both sources within a tile."""
    import torch

    rng = rng_for(800 + d, k + n2)
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    codes = rng.integers(0, 256, size=(b, n2, d // 2), dtype=np.uint8)
    # E4M3 1/4 .. 7/16 (rows of magnitude like N(0,1), which the absolute output tolerance assumes),
    # a few rows at 1/64 .. 1/32, and three zero rows
    scales = rng.integers(0x28, 0x2F, size=(b, n2, d // 16), dtype=np.uint8)
    scales[0, 3:9] = rng.integers(0x18, 0x1F, size=(6, d // 16))
    scales[0, :3] = 0
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1 + n2, masked_frac=0.15, empty_rows=1)
    ref, ref_lse = orc.sparse_attn_fp4kv(q, kv1, codes, scales, sink, idx, d ** -0.5)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    ws = sti.workspace(sti.sparse_attn_workspace_size(b, s, h, d, k) if ws_full else 256)
    out = sti.sparse_attn_sink_fp4kv(to_dev(q), to_dev(kv1), to_dev_any(codes), to_dev_any(scales),
                                     to_dev_any(sink), to_dev_any(idx), d ** -0.5, lse=lse, ws=ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got = bf16_out_to_f64(out)
    check_attn(got, ref)
    empty = np.all(idx < 0, axis=-1)
    assert np.all(got[empty] == 0)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("b,s,d,k,n1,n2", [
    (1, 300, 512, 200, 256, 256),    # k not a multiple of the 64-row tile
    (2, 150, 256, 130, 100, 300),
    (1, 260, 128, 640, 300, 700),
])
def test_sparse_attn_many_queries(sti, orc, b, s, d, k, n1, n2):
    """More than 256 queries of 64 heads (one CTA per query, no split): random masked slots, rows
    mixing both sources inside a four-row group, all -1 rows, and rows whose filled slots end
    early (whole trailing tiles of -1)."""
    import torch

    rng = rng_for(760 + d, k)
    h = 64
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1 + n2, masked_frac=0.15, empty_rows=2)
    for t in range(0, s, 7):                    # filled slots end early
        idx[0, t, rng.integers(0, k):] = -1
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    ws = sti.workspace(256)
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                               kv2=to_dev(kv2), lse=lse, ws=ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got = bf16_out_to_f64(out)
    check_attn(got, ref)
    empty = np.all(idx < 0, axis=-1)
    assert np.all(got[empty] == 0)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


def test_sparse_attn_streamed_prefill(sti, orc):
    """Many queries of up to 64 heads x 512 run on persistent CTAs that stream each tile by column
    block (several queries per CTA at 500 queries).  Index rows like the pages' prefill rows
    ([window | compressed], -1 where nothing is visible) plus what the stream must survive: rows
    whose middle or leading tiles are all -1, rows with no valid slot between live ones, four-row
    groups mixing both sources, an out-of-range index (flagged and masked), 48 heads, the output
    rotation and the lse."""
    import torch

    rng = rng_for(790, 0)
    b, s, h, d, k, n1, n2, rd = 2, 250, 48, 512, 640, 300, 900, 64
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = np.full((b, s, k), -1, np.int32)
    for bi in range(b):
        for t in range(s):
            w = min(128, t + 1)                                   # window slots, -1 before the start
            idx[bi, t, 128 - w:128] = np.arange(t + 1 - w, t + 1) % n1
            nc = int(rng.integers(0, 513))                        # compressed slots, ascending, -1 padded
            idx[bi, t, 128:128 + nc] = n1 + np.sort(rng.choice(n2, nc, replace=False))
    idx[0, 3] = -1                                                # no valid slot
    idx[1, 100] = -1
    idx[0, 10, :256] = -1                                         # leading tiles dead
    idx[0, 11, 128:512] = -1                                      # middle tiles dead, last tile live
    idx[0, 11, 600:620] = n1 + np.arange(20)
    idx[1, 7, 128:132] = [5, n1 + 9, -1, 6]                       # groups mixing both sources
    idx[1, 7, 40:44] = [n1 + 1, 3, n1 + 2, -1]
    bad = idx.copy()
    bad[1, 20, 130] = n1 + n2 + 5                                 # out of range: flagged, masked
    idx[1, 20, 130] = -1
    cs = _rope_table(rng, (b, s), rd)
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2, rope_cs=cs)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    ws = sti.workspace(256)
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(bad), d ** -0.5,
                               kv2=to_dev(kv2), lse=lse, ws=ws, rope_cs=to_dev_any(cs))
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == sti.FLAG_INDEX_RANGE
    got = bf16_out_to_f64(out)
    check_attn(got, ref)
    assert np.all(got[np.all(idx < 0, axis=-1)] == 0)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)
    # a second call on the same buffers gives the same bits
    out2 = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                                kv2=to_dev(kv2), ws=ws, rope_cs=to_dev_any(cs))
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    assert torch.equal(out, out2)


@pytest.mark.parametrize("b,s,h,k,n1,n2", [
    (1, 300, 1, 4096, 100, 6000),   # one head, the longest index row (32 tiles)
    (2, 170, 64, 129, 60, 300),     # a last tile of one slot
])
def test_sparse_attn_streamed_limits(sti, orc, b, s, h, k, n1, n2):
    """The streamed kernel at the ends of its range: 1 head (Q boxes one row high, 63 padded
    heads) with 32 tiles per query, and a last tile holding a single slot."""
    import torch

    rng = rng_for(795 + h, k)
    d = 512
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1 + n2, masked_frac=0.2, empty_rows=1)
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    ws = sti.workspace(256)
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                               kv2=to_dev(kv2), lse=lse, ws=ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got = bf16_out_to_f64(out)
    check_attn(got, ref)
    assert np.all(got[np.all(idx < 0, axis=-1)] == 0)
    fin = np.isfinite(ref_lse)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


def test_sparse_attn_whole_tiles_masked(sti, orc):
    """Decode-style rows where whole 128-slot tiles are -1 (short sequences), split over CTAs."""
    rng = rng_for(720, 0)
    b, s, h, d, k, n1, n2 = 4, 1, 64, 512, 640, 128, 400
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = np.full((b, s, k), -1, np.int32)
    idx[0, 0, :128] = np.arange(128)
    idx[0, 0, 128:128 + 300] = 128 + np.arange(300)
    idx[1, 0, 125:128] = [0, 1, 2]                      # three window slots, nothing compressed
    idx[2, 0, 600:] = 128 + np.arange(40)               # only the last tile has rows
    ref, _ = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2)
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                               kv2=to_dev(kv2))
    got = bf16_out_to_f64(out)
    check_attn(got, ref)
    assert np.all(got[3] == 0)


@pytest.mark.parametrize("b,k,h", [(1, 640, 64), (2, 640, 64), (40, 640, 64), (3, 129, 64), (2, 640, 32),
                                   (2, 640, 48), (5, 300, 48)])
def test_sparse_attn_split_queries(sti, orc, b, k, h):
    """Few decode queries run split over a thread-block cluster: with 32 or 64 heads the heads
    split (4 or 2 CTAs, tiles gathered once by multicast), otherwise the slots split (up to 8 CTAs
    adding into the workspace's fp32 accumulator).  The result matches the oracle and the
    unsplit run (256-byte workspace), the accumulator is zero again afterwards, and a second call
    on the same workspace agrees."""
    import torch

    rng = rng_for(730 + b, k + h)
    d, n1, n2 = 512, 128, 2000
    q = to_bf16_bits(rng.standard_normal((b, 1, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, 1, k, n1 + n2, masked_frac=0.2)
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2)
    args = (to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5)
    ws = sti.workspace(sti.sparse_attn_workspace_size(b, 1, h, d, k))
    assert ws.numel() == 256 + b * h * d * 4
    outs = []
    for _ in range(2):
        lse = torch.empty(b, 1, h, dtype=torch.float32, device="cuda")
        outs.append(sti.sparse_attn_sink(*args, kv2=to_dev(kv2), lse=lse, ws=ws))
        torch.cuda.synchronize()
        assert sti.read_device_status(ws) == 0
        assert int(torch.count_nonzero(ws[256:])) == 0, "accumulator not left zeroed"
        check_attn(bf16_out_to_f64(outs[-1]), ref)
        np.testing.assert_allclose(lse.cpu().numpy().astype(np.float64), ref_lse, rtol=1e-4, atol=1e-4)
    unsplit = sti.sparse_attn_sink(*args, kv2=to_dev(kv2), ws=sti.workspace(256))
    check_attn(bf16_out_to_f64(unsplit), ref)
    # the split and unsplit runs round the same fp32 values to bf16 except for summation order
    diff = np.abs(bf16_out_to_f64(outs[0]) - bf16_out_to_f64(unsplit))
    assert diff.max() <= 2e-2


def _rope_table(rng, lead, rd):
    theta = rng.uniform(-np.pi, np.pi, size=(*lead, rd // 2))
    return np.stack([np.cos(theta), np.sin(theta)], axis=-1).astype(np.float32)


@pytest.mark.parametrize("b,s,h,d,k,rd,label", [
    (2, 1, 64, 512, 640, 64, "head split, two row groups (merge epilogue)"),
    (40, 1, 64, 512, 640, 64, "head split, one row group"),
    (1, 300, 64, 512, 200, 64, "one CTA per query"),
    (3, 1, 48, 512, 640, 64, "slots split over a cluster (fp32 accumulator)"),
    (1, 40, 4, 64, 32, 16, "d = 64 (padded d block)"),
    (2, 1, 64, 512, 640, 512, "every dim rotated"),
])
def test_sparse_attn_output_rotation(sti, orc, b, s, h, d, k, rd, label):
    """The output's inverse rotary rotation fused into every attention epilogue equals the
    oracle's attention followed by its rotation."""
    import torch

    rng = rng_for(780 + h + d, k + rd)
    n1, n2 = 128, 900
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1 + n2, masked_frac=0.1, empty_rows=1)
    cs = _rope_table(rng, (b, s), rd)
    ref, ref_lse = orc.sparse_attn(q, kv1, sink, idx, d ** -0.5, kv2=kv2, rope_cs=cs)
    lse = torch.empty(b, s, h, dtype=torch.float32, device="cuda")
    ws = sti.workspace(sti.sparse_attn_workspace_size(b, s, h, d, k))
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                               kv2=to_dev(kv2), lse=lse, ws=ws, rope_cs=to_dev_any(cs))
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    check_attn(bf16_out_to_f64(out), ref)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse.cpu().numpy().astype(np.float64)[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)
    # the dims before the rotated ones are those of the plain call (bit for bit, except where the
    # cluster's partial sums meet in L2 atomics, whose order varies between runs)
    plain = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(idx), d ** -0.5,
                                 kv2=to_dev(kv2), ws=ws)
    if label.startswith("slots split"):
        assert float((out[..., :d - rd].float() - plain[..., :d - rd].float()).abs().max()) <= 2e-2
    else:
        assert torch.equal(out[..., :d - rd], plain[..., :d - rd])


def test_decode_fused_output_rotation(sti, orc):
    import torch

    shp = workloads.custom("decode_rope", b=3, s=1, start_pos=[4095, 700, 9000], seed=78, n_cols=2400, topk=512,
                           h=64, d=512)
    data = workloads.make(shp)
    sp = data["start_pos"]
    W = shp.window
    ref_scores = orc.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, sp, shp.n_cols, shp.ratio)
    ref_idx = np.concatenate([np.concatenate([orc.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0),
                              orc.topk(ref_scores, sp, shp.ratio, shp.topk, W)], axis=-1)
    cs = _rope_table(rng_for(79, 0), (shp.b,), shp.rd)
    ref_out, _ = orc.sparse_attn(data["q"][0], data["win"][0], data["sink"][0], ref_idx, shp.softmax_scale,
                                 kv2=data["comp"], rope_cs=cs[:, None])
    a, out, tk = sti.decode_args(to_dev(data["q"][0]), to_dev(data["win"][0]), to_dev(data["comp"]),
                                 to_dev_any(data["sink"][0]), shp.softmax_scale, to_dev(data["iq"]),
                                 to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale, to_dev_any(sp), shp.ratio,
                                 shp.n_cols, shp.topk, rope_cs=to_dev_any(cs))
    ws = sti.workspace(sti.decode_workspace_size(a))
    sti.decode_fused(a, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    check_attn(bf16_out_to_f64(out).reshape(ref_out.shape), ref_out)


def test_sparse_attn_flags_out_of_range(sti, orc):
    rng = rng_for(710, 0)
    b, s, h, d, k, n1 = 1, 2, 8, 64, 20, 30
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    idx = index_lists(rng, b, s, k, n1, masked_frac=0.0)
    bad = idx.copy()
    bad[0, 0, 3] = n1 + 7
    bad[0, 1, 4] = -5
    ws = sti.workspace(sti.sparse_attn_workspace_size(b, s, h, d, k))
    out = sti.sparse_attn_sink(to_dev(q), to_dev(kv1), to_dev_any(sink), to_dev_any(bad), d ** -0.5, ws=ws)
    assert sti.read_device_status(ws) & sti.FLAG_INDEX_RANGE
    assert sti.read_device_status(ws) == 0   # cleared
    masked = bad.copy()
    masked[0, 0, 3] = -1
    masked[0, 1, 4] = -1
    ref, _ = orc.sparse_attn(q, kv1, sink, masked, d ** -0.5)
    check_attn(bf16_out_to_f64(out), ref)


# ----------------------------------------------------------------- fused decode layer


def test_decode_fused_small(sti, orc):
    import torch

    shp = workloads.custom("decode_small", b=5, s=1, start_pos=[4095, 1023, 300, 2, 5000], seed=77, n_cols=1300,
                           topk=512, h=64, d=512)
    data = workloads.make(shp)
    sp = data["start_pos"]
    W = shp.window
    ref_scores = orc.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, sp, shp.n_cols, shp.ratio)
    ref_cidx = orc.topk(ref_scores, sp, shp.ratio, shp.topk, W)
    ref_widx = np.concatenate([orc.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0)
    ref_idx = np.concatenate([ref_widx, ref_cidx], axis=-1)
    ref_out, _ = orc.sparse_attn(data["q"][0], data["win"][0], data["sink"][0], ref_idx, shp.softmax_scale,
                                 kv2=data["comp"])
    a, out, tk = sti.decode_args(to_dev(data["q"][0]), to_dev(data["win"][0]), to_dev(data["comp"]),
                                 to_dev_any(data["sink"][0]), shp.softmax_scale, to_dev(data["iq"]),
                                 to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale, to_dev_any(sp), shp.ratio,
                                 shp.n_cols, shp.topk)
    ws = sti.workspace(sti.decode_workspace_size(a))
    for _ in range(2):   # the second call checks that the workspace was left ready (histograms re-zeroed)
        sti.decode_fused(a, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got_idx = tk.cpu().numpy().reshape(shp.b, 1, -1)
    np.testing.assert_array_equal(got_idx[..., :W], ref_widx)
    check_topk_rows(got_idx[..., W:], ref_cidx, ref_scores, W, shp.topk)
    check_attn(bf16_out_to_f64(out).reshape(ref_out.shape), ref_out)


def test_decode_fused_fp4kv(sti, orc):
    """The decode step with the compressed KV as fp4 rows (codes + E4M3 scales, the form
    Attention._compress_kv writes): the fused kernel stages and decodes the packed rows; ragged
    batch with rows short of index_topk (masked slots), a filling ring, and one sequence with no
    compressed rows yet.  A shape the fused kernel does not take is refused on the host."""
    import torch

    shp = workloads.custom("decode_fp4kv", b=5, s=1, start_pos=[8191, 700, 5, 3000, 2], seed=91, n_cols=2048,
                           topk=512, h=64, d=512, fp4_kv=True)
    data = workloads.make(shp)
    sp = data["start_pos"]
    W = shp.window
    ref_scores = orc.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, sp, shp.n_cols, shp.ratio)
    ref_cidx = orc.topk(ref_scores, sp, shp.ratio, shp.topk, W)
    ref_widx = np.concatenate([orc.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0)
    ref_idx = np.concatenate([ref_widx, ref_cidx], axis=-1)
    ref_out, _ = orc.sparse_attn_fp4kv(data["q"][0], data["win"][0], data["comp_codes"], data["comp_scales"],
                                       data["sink"][0], ref_idx, shp.softmax_scale)
    codes, scales = to_dev_any(data["comp_codes"]), to_dev_any(data["comp_scales"])
    a, out, tk = sti.decode_args(to_dev(data["q"][0]), to_dev(data["win"][0]), None, to_dev_any(data["sink"][0]),
                                 shp.softmax_scale, to_dev(data["iq"]), to_dev(data["ik"]), to_dev(data["w"]),
                                 shp.index_scale, to_dev_any(sp), shp.ratio, shp.n_cols, shp.topk,
                                 comp_codes=codes, comp_scales=scales)
    assert sti.decode_kernel_count(a) == 2
    ws = sti.workspace(sti.decode_workspace_size(a))
    for _ in range(2):
        sti.decode_fused(a, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got_idx = tk.cpu().numpy().reshape(shp.b, 1, -1)
    np.testing.assert_array_equal(got_idx[..., :W], ref_widx)
    check_topk_rows(got_idx[..., W:], ref_cidx, ref_scores, W, shp.topk)
    check_attn(bf16_out_to_f64(out).reshape(ref_out.shape), ref_out)
    # 32 heads: not the fused shape, so fp4 rows are refused before anything is enqueued
    a32, _, _ = sti.decode_args(to_dev(data["q"][0][:, :, :32]), to_dev(data["win"][0]), None,
                                to_dev_any(data["sink"][0][:32]), shp.softmax_scale, to_dev(data["iq"]),
                                to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale, to_dev_any(sp), shp.ratio,
                                shp.n_cols, shp.topk, comp_codes=codes, comp_scales=scales)
    with pytest.raises(RuntimeError):   # sti_decode_kernel_count returns -1
        sti.decode_kernel_count(a32)
    with pytest.raises(RuntimeError):   # STI_ERR_UNSUPPORTED
        sti.decode_fused(a32, sti.workspace(sti.decode_workspace_size(a32)))


@pytest.mark.parametrize("n_cols,sps,label", [
    (2101, [127, 126, 95, 31, 1, 2047, 2051, 8399],
     "ring full / one slot short / whole ring slices empty; vis = K, K+1; score rows not 16-byte aligned"),
    (20000, [79999, 65535, 17000, 130], "score rows past 16384 positions (quarters read twice from L2)"),
])
def test_decode_fused_boundaries(sti, orc, n_cols, sps, label):
    """The decode step's fused top-k + attention kernel: each CTA of a query's cluster owns 32
    ring slots and a quarter of the score row; these start positions put the ring's filling edge
    and the visible count at every boundary of that split."""
    import torch

    shp = workloads.custom("decode_bounds", b=len(sps), s=1, start_pos=sps, seed=83, n_cols=n_cols, topk=512, h=64,
                           d=512)
    data = workloads.make(shp)
    sp = data["start_pos"]
    W = shp.window
    ref_scores = orc.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, sp, shp.n_cols, shp.ratio)
    ref_cidx = orc.topk(ref_scores, sp, shp.ratio, shp.topk, W)
    ref_widx = np.concatenate([orc.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0)
    ref_out, _ = orc.sparse_attn(data["q"][0], data["win"][0], data["sink"][0],
                                 np.concatenate([ref_widx, ref_cidx], axis=-1), shp.softmax_scale, kv2=data["comp"])
    a, out, tk = sti.decode_args(to_dev(data["q"][0]), to_dev(data["win"][0]), to_dev(data["comp"]),
                                 to_dev_any(data["sink"][0]), shp.softmax_scale, to_dev(data["iq"]),
                                 to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale, to_dev_any(sp), shp.ratio,
                                 shp.n_cols, shp.topk)
    assert sti.decode_kernel_count(a) == 2, "the fused kernel takes this shape"
    ws = sti.workspace(sti.decode_workspace_size(a))
    sti.decode_fused(a, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got_idx = tk.cpu().numpy().reshape(shp.b, 1, -1)
    np.testing.assert_array_equal(got_idx[..., :W], ref_widx)
    check_topk_rows(got_idx[..., W:], ref_cidx, ref_scores, W, shp.topk)
    check_attn(bf16_out_to_f64(out).reshape(ref_out.shape), ref_out)


@pytest.mark.parametrize("probs,label", [((0.02, 0.49, 0.49), "tau bin fits: ~800 tied keys across every chunk"),
                                         ((0.34, 0.33, 0.33), "tau bin too large: whole-row passes")])
def test_decode_fused_topk_ties(sti, orc, probs, label):
    """Index keys drawn from three distinct rows, so every score is one of three values and the
    k-th largest is tied across the whole row: the selection must take the tied keys in position
    order, across the chunks the row is split into."""
    import torch

    shp = workloads.custom("decode_ties", b=2, s=1, start_pos=[159999, 100000], seed=81, n_cols=40000, topk=512,
                           h=64, d=512)
    data = workloads.make(shp)
    rng = rng_for(820, int(probs[0] * 100))
    groups = to_bf16_bits(rng.standard_normal((3, shp.Di)))
    pick = rng.choice(3, size=(shp.b, shp.n_cols), p=probs)
    data["ik"] = np.ascontiguousarray(groups[pick])
    sp = data["start_pos"]
    ref_scores = orc.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, sp, shp.n_cols, shp.ratio)
    for bi in range(shp.b):   # the three values must be well apart for the order to be unambiguous
        vals = np.unique(ref_scores[bi, 0][np.isfinite(ref_scores[bi, 0])])
        assert len(vals) == 3 and np.min(np.diff(vals)) > 1e-3 * np.max(np.abs(vals)), label
    ref_cidx = orc.topk(ref_scores, sp, shp.ratio, shp.topk, shp.window)
    a, out, tk = sti.decode_args(to_dev(data["q"][0]), to_dev(data["win"][0]), to_dev(data["comp"]),
                                 to_dev_any(data["sink"][0]), shp.softmax_scale, to_dev(data["iq"]),
                                 to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale, to_dev_any(sp), shp.ratio,
                                 shp.n_cols, shp.topk)
    ws = sti.workspace(sti.decode_workspace_size(a))
    sti.decode_fused(a, ws)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws) == 0
    got = tk.cpu().numpy().reshape(shp.b, 1, -1)[..., shp.window:]
    np.testing.assert_array_equal(got, ref_cidx)


def test_decode_fused_waits_for_q_ready(sti):
    """q uploaded on another stream: the attention step waits for the q_ready event and the
    result equals the call with q already in place."""
    import torch

    shp = workloads.custom("decode_qready", b=4, s=1, start_pos=[4095, 2047, 300, 9000], seed=78, n_cols=2300,
                           topk=512, h=64, d=512)
    data = workloads.make(shp)
    common = (to_dev(data["win"][0]), to_dev(data["comp"]), to_dev_any(data["sink"][0]), shp.softmax_scale,
              to_dev(data["iq"]), to_dev(data["ik"]), to_dev(data["w"]), shp.index_scale,
              to_dev_any(data["start_pos"]), shp.ratio, shp.n_cols, shp.topk)
    a0, out0, _ = sti.decode_args(to_dev(data["q"][0]), *common)
    sti.decode_fused(a0, sti.workspace(sti.decode_workspace_size(a0)))
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    h_q = torch.from_numpy(data["q"][0].view(np.int16)).view(torch.bfloat16).pin_memory()
    d_q = torch.zeros(h_q.shape, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(2_000_000)   # the upload lands well after the call is enqueued
        d_q.copy_(h_q, non_blocking=True)
        ev.record(side)
    a1, out1, _ = sti.decode_args(d_q, *common, q_ready=ev)
    ws1 = sti.workspace(sti.decode_workspace_size(a1))
    sti.decode_fused(a1, ws1)
    torch.cuda.synchronize()
    assert sti.read_device_status(ws1) == 0
    assert torch.equal(out0, out1)
