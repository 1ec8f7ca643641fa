"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test checks an oracle function against something other than itself: hand-worked rows
of the page's definitions (tests/golden), closed forms, a textbook/library computation, or
brute force, chosen so a dropped term, a wrong sign or index, or a transposed operand fails.
"""
import itertools
import math
import os

import numpy as np
import pytest

import workloads
from workloads import bf16_bits_to_f32, index_lists, rng_for, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(spec):
    return [[int(v) for v in r.split()] for r in spec.split(";")]


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ----------------------------------------------------------------- window indices


def test_window_idx_golden(orc):
    for ln in _golden_lines("window_idx.txt"):
        head, rows = ln.split("|")
        W, s, sp = (int(v) for v in head.split())
        want = np.array(_rows(rows), dtype=np.int32)
        got = orc.window_topk_idxs(W, 2, s, sp)
        assert got.shape == (2,) + want.shape
        np.testing.assert_array_equal(got[0], want)
        np.testing.assert_array_equal(got[1], want)


@pytest.mark.parametrize("W,s", [(1, 1), (4, 9), (16, 256), (128, 300), (7, 7)])
def test_window_idx_prefill_positions(orc, W, s):
    got = orc.window_topk_idxs(W, 1, s, 0)[0]
    assert got.shape == (s, min(s, W))
    for t in range(s):
        valid = sorted(int(v) for v in got[t] if v >= 0)
        assert valid == list(range(max(0, t - W + 1), t + 1))


@pytest.mark.parametrize("W", [1, 4, 16, 128])
def test_window_idx_decode_ring(orc, W):
    for sp in list(range(1, 3 * W)) + [65535, 131071]:
        got = orc.window_topk_idxs(W, 1, 1, sp)[0, 0]
        assert got.shape == (W,)
        valid = [int(v) for v in got if v >= 0]
        positions = list(range(max(0, sp - W + 1), sp + 1))
        # slots listed oldest first: slot of each held position, in increasing position order
        assert valid == [p % W for p in positions]


# ----------------------------------------------------------------- lengths


def test_compress_len_and_visible_closed_forms(orc):
    for sp in [0, 1, 3, 4, 5, 127, 65535]:
        for s in [1, 2, 7, 64]:
            for r in [1, 2, 4]:
                assert orc.compress_len(sp, s, r) == (sp + s) // r
                for t in range(s):
                    # group j sits at position j*r and becomes visible once (j+1)*r <= p+1
                    brute = sum(1 for j in range(0, (sp + s) // r + 2) if (j + 1) * r <= sp + t + 1)
                    assert orc.visible(sp, t, r) == brute
    # the last query of a chunk sees exactly compress_len groups
    for sp, s, r in [(0, 8, 4), (9, 1, 4), (65535, 1, 4), (100, 13, 2)]:
        assert orc.visible(sp, s - 1, r) == orc.compress_len(sp, s, r)


# ----------------------------------------------------------------- top-k


def test_indexer_rows_golden(orc):
    for ln in _golden_lines("indexer_rows.txt"):
        head, scores, rows = ln.split("|")
        s, sp, r, k, off = (int(v) for v in head.split())
        vals = np.array([float(v) for v in scores.split()], dtype=np.float64)
        n_cols = (sp + s) // r
        assert vals.size == n_cols
        score = np.tile(vals, (1, s, 1))
        want = np.array(_rows(rows), dtype=np.int32).reshape(1, s, k)
        got = orc.topk(score, np.array([sp], np.int32), r, k, off)
        np.testing.assert_array_equal(got, want)


def _topk_numpy(row, vis, k, offset):
    """Independent restatement: lexsort by (-score, position), keep min(k, vis), ascending."""
    pos = np.arange(vis)
    order = np.lexsort((pos, -row[:vis]))
    m = min(k, vis)
    sel = np.sort(pos[order[:m]])
    return np.concatenate([sel + offset, np.full(k - m, -1)]).astype(np.int32)


@pytest.mark.parametrize("n_cols,k,sp,s", [(300, 16, 0, 1300), (2048, 512, 65535 - 2047 * 4, 1), (97, 100, 600, 1)])
def test_topk_matches_lexsort(orc, n_cols, k, sp, s):
    rng = rng_for(7, n_cols)
    s_eff = min(s, 40)
    score = rng.standard_normal((2, s_eff, n_cols))
    spv = np.array([sp, sp + 4], np.int32)
    got = orc.topk(score, spv, 4, k, 128)
    for bi in range(2):
        for t in range(s_eff):
            vis = min((int(spv[bi]) + t + 1) // 4, n_cols)
            np.testing.assert_array_equal(got[bi, t], _topk_numpy(score[bi, t], vis, k, 128))


def test_topk_brute_force_subsets(orc):
    rng = rng_for(11, 0)
    for trial in range(30):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 6))
        row = rng.standard_normal(n)
        got = orc.topk(row.reshape(1, 1, n), np.array([n * 2 - 1], np.int32), 2, k, 0)[0, 0]
        m = min(k, n)
        best = max(itertools.combinations(range(n), m), key=lambda c: sum(row[list(c)]))
        assert list(got[:m]) == sorted(best)
        assert all(v == -1 for v in got[m:])


def test_topk_ties_prefer_lower_position(orc):
    row = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 2.0])
    got = orc.topk(row.reshape(1, 1, 6), np.array([23], np.int32), 4, 3, 0)[0, 0]
    np.testing.assert_array_equal(got, [1, 2, 3])


def test_topk_all_visible_when_k_exceeds(orc):
    rng = rng_for(12, 0)
    score = rng.standard_normal((1, 1, 50))
    got = orc.topk(score, np.array([4 * 30 - 1], np.int32), 4, 40, 7)[0, 0]
    np.testing.assert_array_equal(got, np.concatenate([np.arange(30) + 7, np.full(10, -1)]))


# ----------------------------------------------------------------- index scores


def _f(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def test_index_score_hand_values(orc):
    q = to_bf16_bits(np.array([[[[1, 2], [-1, 1]]]], np.float32))          # [1,1,2,2]
    k = to_bf16_bits(np.array([[[1, 0], [0, 1], [1, 1], [-2, 1]]], np.float32))
    w = to_bf16_bits(np.array([[[0.5, 2.0]]], np.float32))
    for ln in _golden_lines("index_score_hand.txt"):
        head, vals = ln.split("|")
        sp, r = (int(v) for v in head.split())
        want = np.array([-np.inf if v == "-inf" else float(v) for v in vals.split()])
        got = orc.index_score(q, k, w, 1.0, np.array([sp], np.int32), 4, r)[0, 0]
        np.testing.assert_array_equal(got, want)


def _rand_index_inputs(seed, b=2, s=3, H=4, D=32, n=70):
    rng = rng_for(seed, 0)
    iq = to_bf16_bits(rng.standard_normal((b, s, H, D)))
    ik = to_bf16_bits(rng.standard_normal((b, n, D)))
    w = to_bf16_bits(rng.standard_normal((b, s, H)))
    return iq, ik, w


def test_index_score_relu_identity(orc):
    """relu(x) - relu(-x) = x, so S(q) - S(-q) = c * sum_h w_h q_h . k (a plain matmul)."""
    iq, ik, w = _rand_index_inputs(21)
    neg = iq ^ np.uint16(0x8000)
    sp = np.array([400, 400], np.int32)
    c = 0.37
    a = orc.index_score(iq, ik, w, c, sp, 70, 4)
    bneg = orc.index_score(neg, ik, w, c, sp, 70, 4)
    lin = c * np.einsum("bsh,bshd,bnd->bsn", _f(w), _f(iq), _f(ik))
    np.testing.assert_allclose(a - bneg, lin, rtol=1e-12, atol=1e-12)
    # and relu really cuts: the two are not equal to +-lin individually
    assert np.abs(a - lin).max() > 1e-3


def test_index_score_rank_one_when_all_positive(orc):
    """All dots positive -> S = c * (sum_h w_h q_h) . k_j."""
    rng = rng_for(22, 0)
    iq = to_bf16_bits(np.abs(rng.standard_normal((1, 2, 3, 16))))
    ik = to_bf16_bits(np.abs(rng.standard_normal((1, 40, 16))))
    w = to_bf16_bits(rng.standard_normal((1, 2, 3)))
    got = orc.index_score(iq, ik, w, 0.5, np.array([1000], np.int32), 40, 4)
    u = (_f(w)[..., None] * _f(iq)).sum(2)                    # [1,2,16]
    want = 0.5 * u @ _f(ik)[0].T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_index_score_head_additivity(orc):
    """Splitting heads into two groups (zeroed weights) sums back to the full score:
    the partial-head sums a head-sharded run would all-reduce."""
    iq, ik, w = _rand_index_inputs(23)
    sp = np.array([299, 311], np.int32)
    wf = _f(w)
    mask = np.zeros(4)
    mask[[0, 2]] = 1
    wa = to_bf16_bits(wf * mask)
    wb = to_bf16_bits(wf * (1 - mask))
    full = orc.index_score(iq, ik, w, 0.1, sp, 70, 4)
    part = orc.index_score(iq, ik, wa, 0.1, sp, 70, 4) + orc.index_score(iq, ik, wb, 0.1, sp, 70, 4)
    np.testing.assert_allclose(full, part, rtol=1e-12, atol=1e-12)


def test_index_score_batches_and_mask(orc):
    iq, ik, w = _rand_index_inputs(24)
    sp = np.array([7, 150], np.int32)         # batch 0 sees (7+t+1)//4 = 2..2 columns, batch 1 37..38
    a = orc.index_score(iq, ik, w, 1.0, sp, 70, 4)
    for bi in range(2):
        for t in range(3):
            vis = (int(sp[bi]) + t + 1) // 4
            assert np.all(np.isfinite(a[bi, t, :vis]))
            assert np.all(a[bi, t, vis:] == -np.inf)
    ik2 = ik.copy()
    ik2[1] = to_bf16_bits(rng_for(25, 0).standard_normal(ik[1].shape))
    b2 = orc.index_score(iq, ik2, w, 1.0, sp, 70, 4)
    np.testing.assert_array_equal(a[0], b2[0])
    assert not np.array_equal(a[1], b2[1])
    # scale c multiplies every visible entry
    c2 = orc.index_score(iq, ik, w, 2.0, sp, 70, 4)
    fin = np.isfinite(a)
    np.testing.assert_allclose(c2[fin], 2 * a[fin], rtol=1e-15)


# ----------------------------------------------------------------- sparse attention


def _attn_inputs(seed, b=2, s=2, h=3, d=16, n1=12, n2=20):
    rng = rng_for(seed, 0)
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    kv2 = to_bf16_bits(rng.standard_normal((b, n2, d)))
    sink = rng.standard_normal(h).astype(np.float32)
    return q, kv1, kv2, sink


def _softmax_attn_numpy(qf, rows, scale):
    """Textbook softmax attention of one query head over the given rows."""
    from scipy.special import softmax

    p = softmax(scale * rows @ qf)
    return p @ rows


def test_attn_textbook_when_sink_vanishes(orc):
    q, kv1, kv2, _ = _attn_inputs(31)
    sink = np.full(3, -1e30, np.float32)
    idx = index_lists(rng_for(31, 1), 2, 2, 9, 32, masked_frac=0.2)
    out, _ = orc.sparse_attn(q, kv1, sink, idx, 0.25, kv2=kv2)
    allkv = np.concatenate([_f(kv1), _f(kv2)], axis=1)
    for bi in range(2):
        for t in range(2):
            rows = allkv[bi, [i for i in idx[bi, t] if i >= 0]]
            for hh in range(3):
                want = _softmax_attn_numpy(_f(q)[bi, t, hh], rows, 0.25)
                np.testing.assert_allclose(out[bi, t, hh], want, rtol=1e-12, atol=1e-12)


def test_attn_single_row_closed_form(orc):
    q, kv1, _, sink = _attn_inputs(32, b=1, s=1)
    idx = np.full((1, 1, 5), -1, np.int32)
    idx[0, 0, 3] = 7
    out, lse = orc.sparse_attn(q, kv1, sink, idx, 0.3)
    v = _f(kv1)[0, 7]
    for hh in range(3):
        sc = 0.3 * float(_f(q)[0, 0, hh] @ v)
        want = v / (1.0 + math.exp(float(sink[hh]) - sc))
        np.testing.assert_allclose(out[0, 0, hh], want, rtol=1e-13, atol=1e-13)
        assert lse[0, 0, hh] == pytest.approx(math.log(math.exp(sc) + math.exp(float(sink[hh]))), rel=1e-13)


def test_attn_empty_rows_are_zero(orc):
    q, kv1, kv2, sink = _attn_inputs(33)
    idx = np.full((2, 2, 6), -1, np.int32)
    idx[1, 1, 0] = 3
    out, lse = orc.sparse_attn(q, kv1, sink, idx, 0.25, kv2=kv2)
    assert np.all(out[0] == 0) and np.all(out[1, 0] == 0)
    assert np.all(lse[0] == -np.inf)
    assert np.any(out[1, 1] != 0)


def test_attn_mass_plus_sink_is_one(orc):
    q, kv1, kv2, sink = _attn_inputs(34)
    idx = index_lists(rng_for(34, 1), 2, 2, 11, 32, masked_frac=0.3)
    _, lse = orc.sparse_attn(q, kv1, sink, idx, 0.25, kv2=kv2)
    allkv = np.concatenate([_f(kv1), _f(kv2)], axis=1)
    for bi in range(2):
        for t in range(2):
            rows = allkv[bi, [i for i in idx[bi, t] if i >= 0]]
            for hh in range(3):
                s_i = 0.25 * rows @ _f(q)[bi, t, hh]
                total = np.exp(s_i - lse[bi, t, hh]).sum() + math.exp(float(sink[hh]) - lse[bi, t, hh])
                assert total == pytest.approx(1.0, abs=1e-12)


def test_attn_slot_order_masked_and_duplicates(orc):
    q, kv1, kv2, sink = _attn_inputs(35)
    idx = index_lists(rng_for(35, 1), 2, 2, 8, 32, masked_frac=0.25)
    base, _ = orc.sparse_attn(q, kv1, sink, idx, 0.25, kv2=kv2)
    perm = idx[..., rng_for(35, 2).permutation(8)]
    out_p, _ = orc.sparse_attn(q, kv1, sink, perm, 0.25, kv2=kv2)
    np.testing.assert_allclose(out_p, base, rtol=1e-13, atol=1e-13)
    padded = np.concatenate([idx, np.full((2, 2, 5), -1, np.int32)], axis=-1)
    out_m, _ = orc.sparse_attn(q, kv1, sink, padded, 0.25, kv2=kv2)
    np.testing.assert_allclose(out_m, base, rtol=1e-13, atol=1e-13)
    # a slot listed twice counts twice: same as listing it once with the sink lowered by ln 2
    one = np.array([[[5, -1]]], np.int32)
    two = np.array([[[5, 5]]], np.int32)
    o1, _ = orc.sparse_attn(q[:1, :1], kv1[:1], (sink - np.float32(math.log(2))).astype(np.float32), one, 0.25)
    o2, _ = orc.sparse_attn(q[:1, :1], kv1[:1], sink, two, 0.25)
    np.testing.assert_allclose(o2, o1, rtol=1e-6, atol=1e-7)   # float32 sink shift


def test_attn_two_sources_equal_concatenation(orc):
    q, kv1, kv2, sink = _attn_inputs(36)
    idx = index_lists(rng_for(36, 1), 2, 2, 10, 32, masked_frac=0.1)
    a, la = orc.sparse_attn(q, kv1, sink, idx, 0.25, kv2=kv2)
    cat = np.concatenate([kv1, kv2], axis=1)
    b, lb = orc.sparse_attn(q, cat, sink, idx, 0.25)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    # indices past the end of both sources hold nothing (treated as masked)
    bad = idx.copy()
    bad[0, 0, 0] = 32 + 5
    c, _ = orc.sparse_attn(q, kv1, sink, bad, 0.25, kv2=kv2)
    ref = idx.copy()
    ref[0, 0, 0] = -1
    d, _ = orc.sparse_attn(q, kv1, sink, ref, 0.25, kv2=kv2)
    np.testing.assert_array_equal(c, d)


# ----------------------------------------------------------------- dense reference


def test_dense_is_textbook_causal_window(orc):
    """Prefill with ratio > s: no compressed group visible -> causal sliding-window softmax + sink."""
    rng = rng_for(41, 0)
    s, h, d, W = 9, 2, 8, 4
    q = to_bf16_bits(rng.standard_normal((1, s, h, d)))
    win = to_bf16_bits(rng.standard_normal((1, s, d)))
    comp = to_bf16_bits(rng.standard_normal((1, 1, d)))
    sink = np.full(h, -1e30, np.float32)
    out = orc.dense_attn(q, win, comp, np.zeros(1, np.int32), sink, 0.5, W, 100)
    for t in range(s):
        rows = _f(win)[0, max(0, t - W + 1): t + 1]
        for hh in range(h):
            np.testing.assert_allclose(out[0, t, hh], _softmax_attn_numpy(_f(q)[0, t, hh], rows, 0.5), rtol=1e-12)


@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_sparse_equals_dense_when_topk_covers(orc, mode):
    """index_topk >= visible count: window indices + Indexer rows select everything the
    position-defined dense attention sees, so the two must agree."""
    rng = rng_for(42, 0 if mode == "prefill" else 1)
    h, d, W, r, Hi, Di = 3, 16, 8, 4, 2, 8
    if mode == "prefill":
        b, s, sp = 1, 37, np.zeros(1, np.int32)
        n_win_rows = s
    else:
        b, s, sp = 3, 1, np.array([5, 8, 61], np.int32)
        n_win_rows = W
    n_cols = int((sp.max() + s) // r)
    K = n_cols + 3
    q = to_bf16_bits(rng.standard_normal((b, s, h, d)))
    win = to_bf16_bits(rng.standard_normal((b, n_win_rows, d)))
    comp = to_bf16_bits(rng.standard_normal((b, n_cols, d)))
    iq = to_bf16_bits(rng.standard_normal((b, s, Hi, Di)))
    ik = to_bf16_bits(rng.standard_normal((b, n_cols, Di)))
    w = to_bf16_bits(rng.standard_normal((b, s, Hi)))
    sink = rng.standard_normal(h).astype(np.float32)
    score = orc.index_score(iq, ik, w, 1.0, sp, n_cols, r)
    comp_idx = orc.topk(score, sp, r, K, n_win_rows)
    win_idx = np.concatenate([orc.window_topk_idxs(W, 1, s, int(sp[bi])) for bi in range(b)], axis=0)
    idx = np.concatenate([win_idx, comp_idx], axis=-1)
    sparse, _ = orc.sparse_attn(q, win, sink, idx, d ** -0.5, kv2=comp)
    dense = orc.dense_attn(q, win, comp, sp, sink, d ** -0.5, W, r)
    np.testing.assert_allclose(sparse, dense, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ output inverse rotation


def test_inverse_rope_identity_and_quarter_turn(orc):
    rng = np.random.default_rng(5)
    o = rng.standard_normal((2, 3, 4, 16))
    cs0 = np.zeros((2, 3, 4, 2))
    cs0[..., 0] = 1.0                                   # angle 0: nothing moves
    np.testing.assert_array_equal(orc.output_inverse_rope(o.copy(), cs0), o)
    cs90 = np.zeros((2, 3, 4, 2))
    cs90[..., 1] = 1.0                                  # a quarter turn back: (x, y) -> (y, -x)
    got = orc.output_inverse_rope(o.copy(), cs90)
    np.testing.assert_array_equal(got[..., :8], o[..., :8])          # dims before the last rd
    np.testing.assert_array_equal(got[..., 8::2], o[..., 9::2])
    np.testing.assert_array_equal(got[..., 9::2], -o[..., 8::2])


def test_inverse_rope_is_complex_multiplication_by_conjugate(orc):
    rng = np.random.default_rng(6)
    o = rng.standard_normal((1, 2, 3, 12))
    theta = rng.uniform(-np.pi, np.pi, size=(1, 2, 4))
    cs = np.stack([np.cos(theta), np.sin(theta)], axis=-1)
    got = orc.output_inverse_rope(o.copy(), cs)
    z = (o[..., 4::2] + 1j * o[..., 5::2]) * np.exp(-1j * theta)[:, :, None, :]
    np.testing.assert_allclose(got[..., 4::2], z.real, rtol=0, atol=1e-14)
    np.testing.assert_allclose(got[..., 5::2], z.imag, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(got[..., :4], o[..., :4])


def test_inverse_rope_undoes_the_generators_rotation(orc):
    """The input generator rotates with its own code (position * theta^(-2i/rd), interleaved
    pairs); the oracle's inverse with the same angles gives the vector back."""
    rng = np.random.default_rng(7)
    rd, th = 16, 10000.0
    pos = np.array([0, 5, 1000])
    x = rng.standard_normal((len(pos), 32))
    rot = workloads._rope_interleaved(x.copy(), pos, rd, th)
    ang = pos[:, None] * th ** (-np.arange(0, rd, 2) / rd)
    cs = np.stack([np.cos(ang), np.sin(ang)], axis=-1)[None, :, None]          # [1, s, 1, rd/2, 2]
    back = orc.output_inverse_rope(rot[None, :, None].copy(), cs[:, :, 0])
    np.testing.assert_allclose(back[0, :, 0], x, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ window rows of a later prefill chunk


def test_chunked_window_from_position_zero_is_the_prefill_band(orc):
    """A chunk starting at 0 (an empty ring) lists the pages' prefill band, every row shifted
    past the W ring rows (golden rows of get_window_topk_idxs, W=4, s=6)."""
    W, s = 4, 6
    band = orc.window_topk_idxs(W, 1, s, 0)[0]                         # [s, min(s, W)]
    got = orc.window_topk_idxs_chunked(W, s, 0)
    np.testing.assert_array_equal(got[:, :band.shape[1]], np.where(band >= 0, band + W, -1))
    assert np.all(got[:, band.shape[1]:] == -1)


@pytest.mark.parametrize("W,s,sp", [(4, 6, 9), (8, 3, 5), (16, 40, 1000), (4, 1, 2)])
def test_chunked_window_rows_hold_the_last_w_positions(orc, W, s, sp):
    """Every referenced row of the [ring ; chunk] source holds one of the query's last W
    positions, each exactly once (brute force over what each row holds)."""
    got = orc.window_topk_idxs_chunked(W, s, sp)
    # what each source row holds: ring slot r -> the newest p < sp with p % W == r; chunk row
    held = {r: max([p for p in range(sp) if p % W == r], default=None) for r in range(W)}
    held.update({W + i: sp + i for i in range(s)})
    for t in range(s):
        P = sp + t
        want = set(range(max(0, P - W + 1), P + 1))
        rows = [int(v) for v in got[t] if v >= 0]
        assert sorted(held[r] for r in rows) == sorted(want)


# ------------------------------------------------------------------ MXFP4 quantiser (reading of fp4_act_quant)


def test_mxfp4_code_table_from_the_format_definition(orc):
    """E2M1: sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0; exponent 0 is subnormal
    (m * 0.5).  Every one of the 16 codes, under scale byte 127 (2^0) and 130 (2^3)."""
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        want = (m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)) * (-1) ** s
        packed = np.zeros(16, np.uint8)
        packed[0] = code | (code << 4)
        for sb, mul in ((127, 1.0), (130, 8.0)):
            got = orc.mxfp4_decode(packed[None], np.array([[sb]], np.uint8), 32)[0]
            assert got[0] == want * mul and got[1] == want * mul and np.all(got[2:] == 0)
    # element 2j is the low nibble of byte j, 2j+1 the high one; scale j covers elements 32j..
    packed = np.zeros((1, 32), np.uint8)
    packed[0, 0], packed[0, 16] = 0x21, 0xE5                 # (0.5, 1.0) and (3.0, -4.0)
    got = orc.mxfp4_decode(packed, np.array([[127, 126]], np.uint8), 64)[0]
    assert (got[0], got[1], got[32], got[33]) == (0.5, 1.0, 1.5, -2.0) and np.count_nonzero(got) == 4


def test_mxfp4_rounds_ties_to_even_and_saturates(orc):
    x = np.zeros((1, 32))
    x[0, :9] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -2.5]        # block max 7: X = 0
    got = orc.mxfp4_fake_quant(x)[0, :9]
    np.testing.assert_array_equal(got, [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -2.0])


def test_mxfp4_scale_rule_and_exact_round_trip(orc):
    rng = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for X in (-20, -3, 0, 5, 40):
        vals = rng.choice(grid, size=(3, 64)) * rng.choice([-1, 1], size=(3, 64))
        vals[:, 0] = 6.0                              # each 32-block's max is 6 * 2^X ...
        vals[:, 32] = -4.0                            # ... or 4 * 2^X: X = floor(log2) - 2
        x = vals * 2.0 ** X
        codes, scales = orc.mxfp4_quantize(x)
        assert np.all(scales == X + 127)
        np.testing.assert_array_equal(orc.mxfp4_decode(codes, scales, 64), x)
        amax = np.abs(x.reshape(3, 2, 32)).max(-1)
        assert np.all(scales == np.array([[math.frexp(a)[1] - 1 - 2 + 127 for a in row] for row in amax]))


def test_mxfp4_zero_block_and_error_bound(orc):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((50, 128)) * np.exp2(rng.integers(-8, 8, size=(50, 1)))
    x[3, 32:64] = 0.0
    codes, scales = orc.mxfp4_quantize(x)
    q = orc.mxfp4_decode(codes, scales, 128)
    assert np.all(q[3, 32:64] == 0)
    unit = np.repeat(np.exp2(scales.astype(np.float64) - 127), 32, axis=-1)
    # inside the grid the gap is at most 2 units (between 4 and 6); past 6 units it saturates,
    # and the block max is below 8 units
    assert np.all(np.abs(q - x) <= unit * 2 + 1e-300)
    inside = np.abs(x) <= 6 * unit
    assert np.all(np.abs(q - x)[inside] <= unit[inside])


def test_mxfp4_index_score_is_the_score_of_the_decoded_values(orc):
    """index_score_mxfp4 = index_score of independently decoded keys and quantised queries,
    checked against a plain numpy formula of the score."""
    rng = np.random.default_rng(13)
    b, s, H, D, n = 2, 1, 4, 64, 40
    iq = to_bf16_bits(rng.standard_normal((b, s, H, D)))
    codes = rng.integers(0, 256, size=(b, n, D // 2), dtype=np.uint8)
    scales = rng.integers(120, 130, size=(b, n, D // 32), dtype=np.uint8)
    w = to_bf16_bits(rng.standard_normal((b, s, H)))
    sp = np.array([4 * n - 1, 4 * 20 - 1], np.int32)
    got = orc.index_score_mxfp4(iq, codes, scales, w, 0.125, sp, n, 4)
    qd = orc.mxfp4_fake_quant(bf16_bits_to_f32(iq).astype(np.float64))
    kd = orc.mxfp4_decode(codes, scales, D)
    want = 0.125 * np.einsum("bsh,bsht->bst", bf16_bits_to_f32(w).astype(np.float64),
                             np.maximum(np.einsum("bshd,btd->bsht", qd, kd), 0.0))
    vis = np.minimum((sp + 1) // 4, n)
    for bi in range(b):
        np.testing.assert_allclose(got[bi, 0, :vis[bi]], want[bi, 0, :vis[bi]], rtol=1e-12, atol=1e-12)
        assert np.all(np.isneginf(got[bi, 0, vis[bi]:]))


# ----------------------------------------------------------------- fp4 compressed KV (E4M3 scales, 16)


def test_e4m3_table_equals_the_library_float8_e4m3fn(orc):
    """Every E4M3 byte decodes as torch's float8_e4m3fn does (an independent implementation of the
    format); the format's landmarks: 1.0 = 0x38, 448 the largest finite, 2^-9 the smallest
    subnormal, 2^-6 the smallest normal, 0x7F and 0xFF NaN."""
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = orc.e4m3_value(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    assert np.array_equal(lib[~np.isnan(lib)], ours[~np.isnan(ours)])
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and np.nanmax(ours) == 448.0


def test_e4m3_round_equals_the_library_cast_in_range_and_saturates(orc):
    """Round to nearest E4M3, ties to even: equal to torch's cast on [0, 448], including every
    midpoint between neighbouring codes; above 448 the reading saturates (a plain cast gives NaN
    past 464)."""
    torch = pytest.importorskip("torch")
    grid = orc.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    a = np.concatenate([np.random.default_rng(21).uniform(0, 448, 20000), (grid[1:] + grid[:-1]) / 2, grid])
    lib = torch.tensor(a, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(orc.e4m3_round(a), lib)
    assert orc.e4m3_round(np.array([1.0625]))[0] == 0x38      # 1 and 1.125 tie -> 1 (even code)
    assert orc.e4m3_round(np.array([1.1875]))[0] == 0x3A      # 1.125 and 1.25 tie -> 1.25
    np.testing.assert_array_equal(orc.e4m3_round(np.array([448.0, 464.0, 1e6])), [0x7E, 0x7E, 0x7E])


def test_kvfp4_scale_rule_and_exact_round_trip(orc):
    """Rows built as E2M1 values times an E4M3 scale s, each block holding +-6 s, quantise to
    exactly that scale byte and those codes, and decode back exactly."""
    rng = np.random.default_rng(22)
    d = 64
    mags = np.asarray(orc.E2M1_MAGNITUDES)
    sbytes = rng.integers(0x10, 0x70, size=(5, d // 16)).astype(np.uint8)
    s = orc.e4m3_value(sbytes)
    m = mags[rng.integers(0, 8, size=(5, d // 16, 16))]
    m[..., 3] = 6.0
    x = (np.where(rng.random(m.shape) < 0.5, -m, m) * s[..., None]).reshape(5, d)
    codes, scales = orc.kvfp4_quantize(x)
    np.testing.assert_array_equal(scales, sbytes)
    np.testing.assert_array_equal(orc.kvfp4_decode(codes, scales, d), x)


def test_kvfp4_zero_tiny_blocks_and_error_bound(orc):
    rng = np.random.default_rng(23)
    x = rng.standard_normal((40, 512)) * np.exp2(rng.integers(-6, 6, size=(40, 1)))
    x[1, 16:32] = 0.0
    x[2, 32:48] = rng.standard_normal(16) * 2.0 ** -16     # max/6 below half of E4M3's 2^-9
    codes, scales = orc.kvfp4_quantize(x)
    q = orc.kvfp4_decode(codes, scales, 512)
    assert scales[1, 1] == 0 and scales[2, 2] == 0 and np.all(q[1, 16:32] == 0) and np.all(q[2, 32:48] == 0)
    s = np.repeat(orc.e4m3_value(scales), 16, axis=-1)
    # the E2M1 grid's gaps are at most 2 (between 4 and 6): rounding costs at most 1 s; past 6 s
    # (s rounded down from max/6) the value saturates at 6 s
    assert np.all(np.abs(q - x) <= np.maximum(s, np.abs(x) - 6 * s) * (1 + 1e-12))
    assert np.all(np.abs(q) <= 6 * s)


def test_sparse_attn_fp4kv_is_the_sink_softmax_over_decoded_rows(orc):
    """Brute force in numpy on a tiny case: o = sum_i e^{s_i} v_i / (sum_i e^{s_i} + e^{sink})
    over the decoded compressed rows (selected by index r - n1) and the bf16 window rows."""
    rng = np.random.default_rng(24)
    b, s_, h, d, n1, n2, k = 1, 2, 2, 32, 3, 5, 6
    q = to_bf16_bits(rng.standard_normal((b, s_, h, d)))
    kv1 = to_bf16_bits(rng.standard_normal((b, n1, d)))
    codes = rng.integers(0, 256, size=(b, n2, d // 2), dtype=np.uint8)
    scales = rng.integers(0x28, 0x40, size=(b, n2, d // 16), dtype=np.uint8)
    sink = rng.standard_normal(h).astype(np.float32)
    idx = np.array([[[0, 4, -1, 7, 2, 3], [5, -1, -1, 6, 1, 0]]], np.int32)
    scale = d ** -0.5
    out, _ = orc.sparse_attn_fp4kv(q, kv1, codes, scales, sink, idx, scale)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    rows = np.concatenate([bf16_bits_to_f32(kv1).astype(np.float64), orc.kvfp4_decode(codes, scales, d)], axis=1)
    for t in range(s_):
        sel = [r for r in idx[0, t] if r >= 0]
        v = rows[0, sel]
        for hh in range(h):
            sc = scale * (v @ qf[0, t, hh])
            e = np.exp(sc)
            want = (e @ v) / (e.sum() + math.exp(float(sink[hh])))
            np.testing.assert_allclose(out[0, t, hh], want, rtol=1e-10, atol=1e-12)
