"""Host-side logic of the fp4 workloads (no GPU): the synthetic inputs, the bench's algorithmic
bytes, and the CPU reference arm on them."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_DATA = {}


def _make(n: int):
    """workloads.make(config(n)), built once per test session."""
    if n not in _DATA:
        shape = workloads.config(n)
        _DATA[n] = (shape, workloads.make(shape))
    return _DATA[n]


def test_mxfp4_key_inputs():
    """Workload 9: packed keys and E8M0 scales in their documented ranges, zero past the visible
    keys, no bf16 keys."""
    shape, data = _make(9)
    assert "ik" not in data
    codes, scales = data["ik_codes"], data["ik_scales"]
    assert codes.shape == (shape.b, shape.n_cols, shape.Di // 2) and codes.dtype == np.uint8
    assert scales.shape == (shape.b, shape.n_cols, shape.Di // 32) and scales.dtype == np.uint8
    vis = np.minimum((shape.start_pos.astype(np.int64) + 1) // shape.ratio, shape.n_cols)
    for bi in range(shape.b):
        assert set(np.unique(scales[bi, :vis[bi]])) <= {125, 126, 127}
        assert not codes[bi, vis[bi]:].any() and not scales[bi, vis[bi]:].any()
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1)
    assert not np.any(nib == 8)                    # zero magnitudes carry no sign
    freq = np.bincount((nib & 7).ravel(), minlength=8) / nib.size
    np.testing.assert_allclose(freq, workloads.FP4_CODE_FREQ, atol=0.01)


def test_fp4_compressed_kv_inputs():
    """Workload 10: the compressed rows as fp4 codes and E4M3 scale bytes 0x28..0x2E."""
    shape, data = _make(10)
    assert "comp" not in data and shape.prefill and shape.fp4_kv
    codes, scales = data["comp_codes"], data["comp_scales"]
    assert codes.shape == (1, shape.n_cols, shape.d // 2) and scales.shape == (1, shape.n_cols, shape.d // 16)
    assert scales.min() >= 0x28 and scales.max() <= 0x2E   # every compressed row is visible at s = 8192


def test_bench_bytes_of_the_fp4_workloads():
    """Algorithmic bytes: 68 B per MXFP4 key (64 code + 4 scale bytes) in the scores kernel; 288 B
    per fp4 compressed row (256 + 32) in the prefill attention."""
    import bench

    s9, d9 = _make(9)
    w9 = bench.work(s9, d9)
    keys = s9.b * s9.n_cols
    extra = s9.b * s9.Hi * s9.Di * 2 + s9.b * s9.Hi * 2 + s9.b * s9.n_cols * 4
    assert w9["idx_scores"]["bytes"] == keys * 68 + extra
    (s3, d3), (s10, d10) = _make(3), _make(10)
    w3, w10 = bench.work(s3, d3), bench.work(s10, d10)
    diff = w3["sparse_attn[0]"]["bytes"] - w10["sparse_attn[0]"]["bytes"]
    assert diff == s3.n_cols * (s3.d * 2 - (s3.d // 2 + s3.d // 16))
    assert w3["sparse_attn[0]"]["flops"] == w10["sparse_attn[0]"]["flops"]


@pytest.mark.parametrize("n", [9, 10])
def test_reference_arm_on_the_fp4_workloads(n):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", str(n),
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == workloads.config(n).name
