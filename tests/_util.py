"""Shared helpers of the tests: bf16 upload, tolerance checks, top-k set comparison."""
from __future__ import annotations

import numpy as np

from workloads import bf16_bits_to_f32

# Tolerances stated for the path: index scores within 2e-3 relative (floored at 1e-2 of the
# row's RMS where heads cancel to ~0); attention output max-abs 2e-2, mean-abs 2e-3 against
# the fp64 oracle; top-k index sets bit-exact outside a 1e-6 relative band around the k-th
# oracle score.
SCORE_RTOL = 2e-3
SCORE_FLOOR = 1e-2
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3
TOPK_BAND = 1e-6


def to_dev(bits: np.ndarray, device="cuda"):
    from sparse_top_attention_indexer_gb300 import upload_bf16

    return upload_bf16(bits, device)


def to_dev_any(a: np.ndarray, device="cuda"):
    from sparse_top_attention_indexer_gb300 import upload

    return upload(a, device)


def bf16_out_to_f64(t) -> np.ndarray:
    import torch

    return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def check_scores(gpu: np.ndarray, ref: np.ndarray):
    """gpu fp32 vs oracle fp64 scores: -inf exactly where the oracle has -inf, elsewhere
    |g-r| <= 2e-3 * max(|r|, 1e-2 * rms(row))."""
    assert gpu.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(gpu), ~fin), "masked (-inf) pattern differs"
    rows = ref.reshape(-1, ref.shape[-1])
    g = gpu.reshape(-1, ref.shape[-1]).astype(np.float64)
    worst = 0.0
    for i in range(rows.shape[0]):
        f = np.isfinite(rows[i])
        if not f.any():
            continue
        r = rows[i][f]
        rms = float(np.sqrt(np.mean(r * r)))
        if rms == 0.0:
            assert np.all(g[i][f] == 0.0)
            continue
        scale = np.maximum(np.abs(r), SCORE_FLOOR * rms)
        err = np.abs(g[i][f] - r) / scale
        worst = max(worst, float(err.max()))
    assert worst <= SCORE_RTOL, f"score relative error {worst:.3e} > {SCORE_RTOL}"
    return worst


def score_error_stats(gpu: np.ndarray, ref: np.ndarray) -> dict:
    """The score error three ways, for reporting beside check_scores: the floored relative error
    it asserts; the plain relative error |g-r|/|r| over the entries with |r| >= 1e-2 * rms(row)
    (where the floor does not act); and, below that, the absolute error in units of the row's
    rms (the entries where heads cancel to about zero)."""
    rows = ref.reshape(-1, ref.shape[-1])
    g = gpu.reshape(-1, ref.shape[-1]).astype(np.float64)
    floored = above = below = 0.0
    n_below = 0
    for i in range(rows.shape[0]):
        f = np.isfinite(rows[i])
        if not f.any():
            continue
        r, gi = rows[i][f], g[i][f]
        rms = float(np.sqrt(np.mean(r * r)))
        if rms == 0.0:
            continue
        err = np.abs(gi - r)
        big = np.abs(r) >= SCORE_FLOOR * rms
        floored = max(floored, float((err / np.maximum(np.abs(r), SCORE_FLOOR * rms)).max()))
        if big.any():
            above = max(above, float((err[big] / np.abs(r[big])).max()))
        if (~big).any():
            below = max(below, float(err[~big].max()) / rms)
            n_below += int((~big).sum())
    return {"floored_rel": floored, "rel_where_abs_ge_1e-2_rms": above, "abs_over_rms_below": below,
            "entries_below_floor": n_below}


def check_topk_rows(gpu_rows: np.ndarray, ref_rows: np.ndarray, ref_scores: np.ndarray | None, offset: int,
                    k: int, band: float = TOPK_BAND):
    """Index rows: same layout (ascending valid entries then -1) and the same set, except for
    oracle positions whose score lies within `band` (relative) of the k-th oracle score.
    Returns the number of rows that needed the band."""
    g = gpu_rows.reshape(-1, gpu_rows.shape[-1])
    r = ref_rows.reshape(-1, ref_rows.shape[-1])
    sc = None if ref_scores is None else ref_scores.reshape(-1, ref_scores.shape[-1])
    n_banded = 0
    for i in range(r.shape[0]):
        gv = g[i][g[i] >= 0]
        rv = r[i][r[i] >= 0]
        assert np.all(g[i][len(gv):] == -1) and np.all(g[i][:len(gv)] >= 0), f"row {i}: -1 padding not at the end"
        assert np.all(np.diff(gv) > 0), f"row {i}: not strictly ascending"
        assert len(gv) == len(rv), f"row {i}: {len(gv)} selected vs {len(rv)}"
        if np.array_equal(gv, rv):
            continue
        assert sc is not None, f"row {i}: index sets differ"
        srow = sc[i]
        vis = np.isfinite(srow)
        order = np.sort(srow[vis])[::-1]
        assert len(order) > k, f"row {i}: every visible position should be selected, sets differ"
        tau = order[k - 1]
        amb = set((np.nonzero(np.abs(srow - tau) <= band * abs(tau))[0] + offset).tolist())
        gs, rs = set(gv.tolist()) - amb, set(rv.tolist()) - amb
        assert gs == rs, f"row {i}: sets differ outside the boundary band: {sorted(gs ^ rs)[:8]}"
        n_banded += 1
    return n_banded


def check_attn(gpu: np.ndarray, ref: np.ndarray, max_abs=ATTN_MAX_ABS, mean_abs=ATTN_MEAN_ABS):
    err = np.abs(gpu - ref)
    mx, mn = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, f"attention error max {mx:.3e} mean {mn:.3e}"
    return mx, mn
