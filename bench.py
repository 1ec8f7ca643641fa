"""Benchmark of the Indexer -> top-k -> sparse sink attention path on one GB300.

    python bench.py [--steps K] [--warmup W] [--workload 1..10] [--impl ours|reference]

One step = one pass of the whole path over one batch of synthetic inputs resident in HBM:
window indices, Indexer scores, top-k, sparse sink attention (every attention layer),
launched through the C ABI on one stream (decode: a CUDA graph of the fused decode step and
any reuse layers).  Default workload: single-layer decode, b=32, context 65536 (16384
compressed rows), 64 heads x 512, index heads 32 x 128, top-512.  With the default workload
the same JSON line also carries sub-records for the other configurations the metric names:
`prefill` (b=1, 8192 queries), `long_decode` (b=8, context 131072) and `mixed` (b=64 ragged
sequences, one index pass + four attention layers).

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA events on the
launching stream; a 256 MiB buffer is written and then read before every step (outside the
events), so no step finds the previous step's data in L2 and no step pays for write-backs of
the flush itself.  Then K more steps with an event between every kernel give the per-kernel
durations (`kernel_us`); those events keep a kernel from starting its prologue under its
predecessor's tail, so their sum (`ms_per_step_with_kernel_events`) exceeds the step.

`roofline` is the whole step: the sum over its kernels of each kernel's floor time
(max(algorithmic bytes / HBM peak, algorithmic FLOPs / bf16 peak)) over the measured step time,
against the measured peaks.  `dominant_kernel_roofline` is the same for the kernel with the
largest share of the step, over its own event-timed duration; `kernel_roofline_frac` lists
every kernel's.  `e2e` is the same metric through the fused public entry point with the step's
inputs copied from one pinned host buffer and the output copied back every step (wall clock):
`value` overlaps each step's copies with its neighbours' kernels (double-buffered, as a serving
loop would), `serial_value` runs copy, call, copy back and synchronise one step at a time.
`cpu_baseline` times the CPU oracle on a bounded sample of the same workload.

The library runs on one GPU.  Asked for more (--gpus > 1, or WORLD_SIZE > 1 under torchrun),
rank 0 prints a line saying so and every rank exits 0 without touching a GPU; the reference
arm (the CPU oracle) still runs on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode tokens/s and prefill queries/s (indexer+topk+sparse_attn); % HBM/TC roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
FLUSH_BYTES = 256 << 20
# sub-records of the default line: (key, workload number)
SUB_WORKLOADS = (("prefill", 3), ("long_decode", 4), ("mixed", 5))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


KERNEL_SOURCES = {"idx_scores": ["idx_scores.cu"], "idx_topk": ["idx_topk.cu"],
                  "sparse_attn": ["sparse_attn.cu", "sparse_attn_stream.cu", "sparse_attn_hs.cu", "sti_attn_util.cuh",
                                  "sti_kvfp4.h"],
                  "window_idx": ["idx_topk.cu"],
                  "topk_sparse_attn": ["decode_attn.cu", "sti_attn_util.cuh", "sti_kvfp4.h"]}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is compiled from (its file and the shared headers), for
    matching the ncu counters profiles/ records against the kernel that runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_top_attention_indexer_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES.get(kernel, [])) + ["sti_internal.h", "sti_ptx.cuh"]:
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on these sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    with open(path) as f:
        for ln in f:
            m = re.match(r"\s*(\S+)\s+(\S+)\s+bytes_per_launch=(\d+)\s+sources=(\w+)", ln)
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == want:
                return int(m.group(3))
    return None


# ---------------------------------------------------------------------------------- GPU steps


class GpuPath:
    """Device-resident inputs of one workload and the step that runs the path on them."""

    def __init__(self, shape: workloads.Shape, data: dict, device, output_rope: bool = False):
        import torch

        import sparse_top_attention_indexer_gb300 as sti

        up, upb = sti.upload, sti.upload_bf16
        self.sti, self.torch, self.shape = sti, torch, shape
        self.dev = device
        self.b, self.s = shape.b, shape.s
        self.prefill = shape.prefill
        self.W = shape.window
        self.width = shape.win_width
        self.k_total = self.width + shape.topk
        self.L = shape.n_layers
        self.q = [upb(data["q"][i], device) for i in range(self.L)]
        self.win = [upb(data["win"][i], device) for i in range(self.L)]
        self.sink = [up(data["sink"][i], device) for i in range(self.L)]
        self.comp = upb(data["comp"], device) if "comp" in data else None
        # fp4 compressed KV (workload 10): packed codes and E4M3 scales instead of bf16 rows
        self.comp_codes = up(data["comp_codes"], device) if "comp_codes" in data else None
        self.comp_scales = up(data["comp_scales"], device) if "comp_scales" in data else None
        self.iq = upb(data["iq"], device)
        self.ik = upb(data["ik"], device) if "ik" in data else None
        # MXFP4 keys (workload 9): codes and scales instead of bf16 keys
        self.ik_codes = up(data["ik_codes"], device) if "ik_codes" in data else None
        self.ik_scales = up(data["ik_scales"], device) if "ik_scales" in data else None
        self.w = upb(data["w"], device)
        self.sp = up(data["start_pos"], device)
        self.scores = torch.empty(self.b, self.s, shape.n_cols, dtype=torch.float32, device=device)
        self.idx = torch.empty(self.b, self.s, self.k_total, dtype=torch.int32, device=device)
        self.out = [torch.empty_like(self.q[i]) for i in range(self.L)]
        ws_attn = sti.sparse_attn_workspace_size(self.b, self.s, shape.h, shape.d, self.k_total)
        self.ws = sti.workspace(max(ws_attn, 256), device)
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        # optional: the output's inverse rotary rotation, fused into the attention epilogue
        self.rope_cs = up(workloads.output_rope_table(shape), device) if output_rope else None
        if self.prefill:
            self.names = ["window_idx", "idx_scores", "idx_topk"] + [f"sparse_attn[{i}]" for i in range(self.L)]
            return
        # decode: the fused entry point (scores, top-k + window indices, attention -- the last two
        # as one kernel when the library fuses them), then the reuse layers' attention on the
        # published indices
        self.args, _, _ = sti.decode_args(self.q[0], self.win[0], self.comp, self.sink[0], shape.softmax_scale,
                                          self.iq, self.ik, self.w, shape.index_scale, self.sp, shape.ratio,
                                          shape.n_cols, shape.topk,
                                          out=self.out[0].view(self.b, shape.h, shape.d),
                                          topk_idxs=self.idx.view(self.b, self.k_total),
                                          rope_cs=None if self.rope_cs is None else self.rope_cs[:, 0],
                                          ik_codes=self.ik_codes, ik_scales=self.ik_scales,
                                          comp_codes=self.comp_codes, comp_scales=self.comp_scales)
        self.dws = sti.workspace(sti.decode_workspace_size(self.args), device)
        self.fused_kernels = sti.decode_kernel_count(self.args)
        first = (["idx_scores", "topk_sparse_attn[0]"] if self.fused_kernels == 2 else
                 ["idx_scores", "idx_topk", "sparse_attn[0]"])
        self.names = first + [f"sparse_attn[{i}]" for i in range(1, self.L)]

    def capture(self):
        """Capture the decode step in CUDA graphs: `pgraph` the plain step (what the timed steps
        replay), `graph` the single-layer step with timing events between its kernels."""
        torch = self.torch
        assert not self.prefill
        self.gevents = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in self.gevents:
            e.record()
        self.step()   # warm the library's per-shape caches before capture
        torch.cuda.synchronize()
        self.pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.pgraph):
            self.step()
        torch.cuda.synchronize()
        if self.L == 1:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                self.sti.decode_fused(self.args, self.dws, events=self.gevents)
            torch.cuda.synchronize()

    def graph_times_ms(self):
        """Per-kernel and whole-step milliseconds of the last evented replay."""
        ev = self.gevents
        if self.fused_kernels == 2:   # events 2 and 3 both follow the fused kernel
            return [ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[3])], ev[0].elapsed_time(ev[3])
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(3)], ev[0].elapsed_time(ev[3])

    def scores_view(self):
        """The index scores of the last step ([b, s, n_cols] fp32)."""
        if self.prefill:
            return self.scores
        n = self.b * self.s * self.shape.n_cols
        return self.dws[256:256 + 4 * n].view(self.torch.float32).view(self.b, self.s, self.shape.n_cols)

    def read_status(self) -> int:
        flags = self.sti.read_device_status(self.ws)
        if not self.prefill:
            flags |= self.sti.read_device_status(self.dws)
        return flags

    def launches_per_step(self) -> int:
        return len(self.names)

    def step(self, events=None):
        """One pass of the path; events (len = len(names)+1) are recorded around every kernel
        (prefill and reuse layers only; the fused decode step records its own)."""
        sti, shp = self.sti, self.shape
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        if not self.prefill:
            n0 = len(self.names) - (self.L - 1)
            if events is not None:
                dev = events[:n0 + 1] if self.fused_kernels == 3 else [events[0], events[1], events[2], events[2]]
            sti.decode_fused(self.args, self.dws, events=None if events is None else dev)
            for i in range(1, self.L):
                sti.sparse_attn_sink(self.q[i], self.win[i], self.sink[i], self.idx, shp.softmax_scale,
                                     kv2=self.comp, out=self.out[i], ws=self.ws, rope_cs=self.rope_cs)
                rec(n0 + i)
            return
        rec(0)
        if shp.chunked:
            sti.window_idxs_chunked(self.sp, self.s, self.W, out=self.idx[..., :self.width], ws=self.ws)
        else:
            sti.window_idxs(self.sp, self.s, self.W, out=self.idx[..., :self.width], ws=self.ws)
        rec(1)
        if self.ik_codes is not None:
            sti.idx_scores_mxfp4(self.iq, self.ik_codes, self.ik_scales, self.w, shp.index_scale, self.sp, shp.n_cols,
                                 shp.ratio, out=self.scores, ws=self.ws)
        else:
            sti.idx_scores(self.iq, self.ik, self.w, shp.index_scale, self.sp, shp.n_cols, shp.ratio,
                           out=self.scores, ws=self.ws)
        rec(2)
        # compressed rows follow the window source's rows: offset = s raw rows (prefill) or W slots (decode)
        sti.idx_topk(self.scores, self.sp, shp.ratio, shp.topk, shp.win_rows, out=self.idx[..., self.width:],
                     ws=self.ws)
        rec(3)
        for i in range(self.L):
            if self.comp_codes is not None:
                sti.sparse_attn_sink_fp4kv(self.q[i], self.win[i], self.comp_codes, self.comp_scales, self.sink[i],
                                           self.idx, shp.softmax_scale, out=self.out[i], ws=self.ws)
            else:
                sti.sparse_attn_sink(self.q[i], self.win[i], self.sink[i], self.idx, shp.softmax_scale,
                                     kv2=self.comp, out=self.out[i], ws=self.ws, rope_cs=self.rope_cs)
            rec(4 + i)

    l2_mode = "flush"

    def flush_l2(self):
        if self.l2_mode != "flush":
            return
        # write, then read: no data of the step stays in L2 and none of L2 is left dirty, so the
        # step neither hits on its own inputs nor pays for the flush's write-backs
        self.flush.fill_(1)
        self._flush_sink = self.flush.view(self.torch.int64).sum()


# ---------------------------------------------------------------------------------- work accounting


def work(shape: workloads.Shape, data: dict) -> dict:
    """Algorithmic bytes and FLOPs per kernel launch (what the method must move / compute)."""
    sp = data["start_pos"].astype(np.int64)
    b, s, Hi, Di, h, d = shape.b, shape.s, shape.Hi, shape.Di, shape.h, shape.d
    t = np.arange(s, dtype=np.int64)
    vis = np.minimum((sp[:, None] + t[None, :] + 1) // shape.ratio, shape.n_cols)   # [b, s]
    n_keys = np.minimum((sp + s) // shape.ratio, shape.n_cols)                       # unique keys per sequence
    sel = np.minimum(vis, shape.topk)
    if shape.prefill:
        win_valid = np.minimum(sp[:, None] + t[None, :] + 1, shape.window)
    else:
        win_valid = np.minimum(sp + 1, shape.window)[:, None]
    rows = (sel + win_valid).sum()                                                  # valid gathered rows
    w = {}
    key_bytes = (Di // 2 + Di // 32) if shape.fp4_keys else Di * 2                  # per key (MXFP4: codes + scales)
    w["idx_scores"] = {
        "bytes": float(n_keys.sum() * key_bytes + b * s * Hi * Di * 2 + b * s * Hi * 2 + b * s * shape.n_cols * 4),
        "flops": float(2 * Hi * Di * vis.sum()),
    }
    w["idx_topk"] = {"bytes": float(vis.sum() * 4 + b * s * shape.topk * 4), "flops": 0.0}
    w["window_idx"] = {"bytes": float(b * s * shape.win_width * 4), "flops": 0.0}
    if not shape.prefill:   # the decode top-k kernel also writes the window indices
        w["idx_topk"]["bytes"] += w.pop("window_idx")["bytes"]
    comp_row = (d // 2 + d // 16) if shape.fp4_kv else d * 2                        # per compressed row (fp4: codes + scales)
    if shape.prefill:
        kv_bytes = shape.win_rows * d * 2 + n_keys.sum() * comp_row                # unique rows (L2 serves reuse)
    else:   # every gathered row from HBM
        kv_bytes = win_valid.sum() * d * 2 + sel.sum() * comp_row
    attn = {"bytes": float(kv_bytes + 2 * b * s * h * d * 2 + b * s * shape.k_total * 4),
            "flops": float(4 * h * d * rows)}
    for i in range(shape.n_layers):
        w[f"sparse_attn[{i}]"] = dict(attn)
    # the fused decode kernel does the top-k (reading the scores, writing the index row) and the
    # first layer's attention (which then reads its indices from shared memory, not HBM)
    fused = {"bytes": w["idx_topk"]["bytes"] + attn["bytes"] - b * s * shape.k_total * 4, "flops": attn["flops"]}
    w["topk_sparse_attn[0]"] = fused
    return w


def floor_s(wk: dict, pk: dict) -> tuple[float, str]:
    """A kernel's roofline floor time and its bound."""
    t_mem = wk["bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = wk["flops"] / (pk["bf16_tflops"] * 1e12)
    return (t_tc, "tensor") if t_tc > t_mem else (t_mem, "hbm")


def roofline_of(kernel: str, wk: dict, avg_s: float, pk: dict, workload: str) -> dict:
    t_floor, bound = floor_s(wk, pk)
    if bound == "tensor":
        achieved = wk["flops"] / avg_s / 1e12
        out = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        achieved = wk["bytes"] / avg_s / 1e9
        out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s"}
    out["frac"] = round(achieved / out["peak"], 4)
    out["kernel"] = kernel
    out["peak_source"] = pk["source"]
    out["traffic"] = recorded_traffic(kernel.split("[")[0], workload)
    out["algorithmic_bytes"] = int(wk["bytes"])
    out["algorithmic_flops"] = int(wk["flops"])
    return out


def step_roofline(names: list, wk: dict, step_s: float, pk: dict, workload: str) -> dict:
    """The whole step against the roofline: sum of every kernel's floor time over the measured
    step time.  `achieved` is that fraction times the peak of the bound that dominates the sum
    (every decode kernel is HBM-bound: then it is the step's algorithmic bytes over its time)."""
    floors = [floor_s(wk[n], pk) for n in names]
    t_floor = sum(t for t, _ in floors)
    t_hbm = sum(t for t, bd in floors if bd == "hbm")
    bound = "hbm" if t_hbm >= t_floor - t_hbm else "tensor"
    frac = t_floor / step_s
    peak, unit = (pk["hbm_gbs"], "GB/s") if bound == "hbm" else (pk["bf16_tflops"], "TFLOP/s")
    traffic = [recorded_traffic(n.split("[")[0], workload) for n in names]
    return {"bound": bound, "achieved": round(frac * peak, 1), "peak": peak, "unit": unit, "frac": round(frac, 4),
            "scope": "step: " + " + ".join(names), "peak_source": pk["source"],
            "traffic": int(sum(traffic)) if all(x is not None for x in traffic) else None,
            "algorithmic_bytes": int(sum(wk[n]["bytes"] for n in names)),
            "algorithmic_flops": int(sum(wk[n]["flops"] for n in names)),
            "floor_us": round(t_floor * 1e6, 2)}


# ---------------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------- CPU oracle


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    try:   # Arm hosts often name only the part in lscpu
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def oracle_step(shape: workloads.Shape, data: dict, rows: np.ndarray | None = None, output_rope: bool = False,
                threads: int | None = None):
    """The path on the CPU oracle (test infrastructure), for a subset of query rows of batch
    element 0 in prefill (rows given) or for the whole decode batch."""
    import oracle

    W = shape.window
    if shape.prefill:
        t = rows
        sp = (int(shape.start_pos[0]) + t).astype(np.int32)   # query t sees (start_pos+t+1)//ratio groups
        iq = data["iq"][0][t][:, None]
        w = data["w"][0][t][:, None]
        ik = np.broadcast_to(data["ik"][0], (len(t),) + data["ik"].shape[1:])
        score = oracle.index_score(iq, ik, w, shape.index_scale, sp, shape.n_cols, shape.ratio, threads)
        cidx = oracle.topk(score, sp, shape.ratio, shape.topk, shape.win_rows, threads)
        widx = (oracle.window_topk_idxs_chunked(W, shape.s, int(shape.start_pos[0])) if shape.chunked else
                oracle.window_topk_idxs(W, 1, shape.s, 0)[0])[t][:, None]
        idx = np.concatenate([widx, cidx], axis=-1).reshape(1, len(t), -1)
        q = data["q"][0][0][t][None]
        cs = workloads.output_rope_table(shape)[:, t] if output_rope else None
        if shape.fp4_kv:
            oracle.sparse_attn_fp4kv(q, data["win"][0], data["comp_codes"], data["comp_scales"], data["sink"][0], idx,
                                     shape.softmax_scale, threads)
        else:
            oracle.sparse_attn(q, data["win"][0], data["sink"][0], idx, shape.softmax_scale, kv2=data["comp"],
                               rope_cs=cs, threads=threads)
        return len(t)
    sp = data["start_pos"]
    if shape.fp4_keys:
        score = oracle.index_score_mxfp4(data["iq"], data["ik_codes"], data["ik_scales"], data["w"], shape.index_scale,
                                         sp, shape.n_cols, shape.ratio, threads)
    else:
        score = oracle.index_score(data["iq"], data["ik"], data["w"], shape.index_scale, sp, shape.n_cols,
                                   shape.ratio, threads)
    cidx = oracle.topk(score, sp, shape.ratio, shape.topk, W, threads)
    widx = np.concatenate([oracle.window_topk_idxs(W, 1, 1, int(v)) for v in sp], axis=0)
    idx = np.concatenate([widx, cidx], axis=-1)
    cs = workloads.output_rope_table(shape) if output_rope else None
    for i in range(shape.n_layers):
        if shape.fp4_kv:
            oracle.sparse_attn_fp4kv(data["q"][i], data["win"][i], data["comp_codes"], data["comp_scales"],
                                     data["sink"][i], idx, shape.softmax_scale, threads)
        else:
            oracle.sparse_attn(data["q"][i], data["win"][i], data["sink"][i], idx, shape.softmax_scale,
                               kv2=data["comp"], rope_cs=cs, threads=threads)
    return shape.b * shape.s


def cpu_baseline(shape: workloads.Shape, data: dict, budget_s: float = 12.0, output_rope: bool = False) -> dict:
    """Oracle throughput on a bounded sample: decode runs whole batches, prefill a spread of
    query rows; repeated until about budget_s of CPU time.  Also the tiny prefill (workload 1)
    on one thread."""
    import oracle

    oracle.build()
    if shape.prefill:
        rows = np.linspace(0, shape.s - 1, 16).astype(np.int64)
        sample = f"16 query rows spread over the {shape.s}-query prefill, repeated"
    else:
        rows = None
        sample = f"the whole b={shape.b} decode batch (all {shape.n_layers} attention layer(s)), repeated"
    done, t0 = 0, time.perf_counter()
    reps = 0
    while True:
        done += oracle_step(shape, data, rows, output_rope)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    # single thread, tiny prefill: all 256 queries of workload 1, repeated for about 2 s
    s1 = workloads.config(1)
    d1 = workloads.make(s1)
    all_rows = np.arange(s1.s, dtype=np.int64)
    n1, t1, r1 = 0, time.perf_counter(), 0
    while True:
        n1 += oracle_step(s1, d1, all_rows, threads=1)
        r1 += 1
        e1 = time.perf_counter() - t1
        if e1 >= 2.0 or r1 >= 200:
            break
    return {"value": round(done / el, 3), "unit": "queries/s" if shape.prefill else "tokens/s",
            "cores": oracle.default_threads(), "kind": "oracle", "sample": f"{sample} x{reps} ({el:.1f} s)",
            "cpu_model": cpu_model(), "arch": platform.machine(),
            "single_thread_tiny_prefill": {"value": round(n1 / e1, 1), "unit": "queries/s", "cores": 1,
                                           "workload": s1.name,
                                           "sample": f"all {s1.s} queries x{r1} ({e1:.1f} s)"}}


def reference_arm(args, shape: workloads.Shape, cfg: dict) -> dict:
    """The oracle as the reference arm: W untimed and K timed steps, each the path over a
    bounded sample of the workload (the whole decode batch, or 16 query rows of a prefill)."""
    import oracle

    oracle.build()
    data = workloads.make(shape)
    rows = np.linspace(0, shape.s - 1, 16).astype(np.int64) if shape.prefill else None
    sample = (f"16 query rows spread over the {shape.s}-query prefill per step" if shape.prefill else
              f"the whole b={shape.b} decode batch (all {shape.n_layers} attention layer(s)) per step")
    for _ in range(args.warmup):
        oracle_step(shape, data, rows, args.output_rope)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        done += oracle_step(shape, data, rows, args.output_rope)
    el = time.perf_counter() - t0
    value = round(done / el, 3)
    unit = "queries/s" if shape.prefill else "tokens/s"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.default_threads(), "kind": "oracle",
                             "sample": f"{sample}, {args.steps} steps ({el:.1f} s)", "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def job_throughput(total_ms: float, units_per_step: int, steps: int):
    """Throughput of `steps` steps of `units_per_step` units that took total_ms: (units/s, ms)."""
    return units_per_step * steps / (float(total_ms) / 1e3), float(total_ms)


# ---------------------------------------------------------------------------------- main


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="default workload only: skip the prefill, long-decode "
                                                          "and mixed sub-records")
    ap.add_argument("--no-clocks", action="store_true", help="skip nvidia-smi sampling (profiler runs)")
    ap.add_argument("--output-rope", action="store_true",
                    help="fuse the output's inverse rotary rotation (last rd dims) into the attention")
    ap.add_argument("--l2", default="flush", choices=["flush", "none"],
                    help="flush: write then read 256 MiB before every step; none: no flush (every step of "
                         "the decode workloads touches more bytes than L2 holds)")
    return ap.parse_args(argv)


def workload_config(shape: workloads.Shape, args) -> dict:
    cfg = {"workload": shape.name, "b": shape.b, "seqlen": shape.s, "context": int(shape.start_pos.max()) + shape.s,
           "heads": shape.h, "head_dim": shape.d, "window": shape.window, "ratio": shape.ratio,
           "compressed_rows": shape.n_cols, "index_heads": shape.Hi, "index_head_dim": shape.Di,
           "index_topk": shape.topk, "attention_layers": shape.n_layers,
           "l2": ("256 MiB written then read before every step (outside the timed region)" if args.l2 == "flush" else
                  "no flush: inputs larger than L2 (each decode step streams the index keys, "
                  f"{shape.b * shape.n_cols * shape.Di * 2 / 1e6:.0f} MB, through the 129 MB L2)")}
    if args.output_rope:
        cfg["output_inverse_rope_dims"] = shape.rd
    if shape.fp4_kv:
        cfg["compressed_kv"] = ("fp4 rows (E2M1 codes, an E4M3 scale per 16 elements), gathered and decoded to "
                                "bf16 in the attention kernel")
    if shape.fp4_keys:
        cfg["index_keys"] = ("MXFP4 (E2M1 codes, an E8M0 scale per 32); queries quantised to MXFP4 in the scores "
                             "kernel; decode units run the codes as E2M1 tensor-core operands (kind::f8f6f4, one "
                             "fp32 accumulator per scale block, scales applied in the epilogue)")
    if shape.n_layers > 1:
        cfg["sequence_lengths"] = f"{int(shape.start_pos.min()) + 1}..{int(shape.start_pos.max()) + 1} (ragged)"
    return cfg


def bench_workload(n: int, args, device, primary: bool) -> dict:
    """Time workload n on the GPU and return its record (the main line, or a sub-record)."""
    import torch

    shape = workloads.config(n)
    if args.output_rope and shape.fp4_kv:
        raise SystemExit("--output-rope is not available with fp4 compressed KV")
    unit = "queries/s" if shape.prefill else "tokens/s"
    data = workloads.make(shape)
    path = GpuPath(shape, data, device, output_rope=args.output_rope and not shape.fp4_kv)
    path.l2_mode = args.l2
    sampler = None if args.no_clocks else ClockSampler(device.index)
    use_graph = not shape.prefill
    if use_graph:
        path.capture()

    def plain_step():
        # one step as a user runs it: the graph without events between its kernels (or direct calls)
        path.pgraph.replay() if use_graph else path.step()

    for _ in range(args.warmup):
        path.flush_l2()
        plain_step()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # timed region: K steps, each bracketed by CUDA events on this stream (the L2 flush before each
    # step stays outside them)
    se = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        path.flush_l2()
        se[k][0].record()
        plain_step()
        se[k][1].record()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in se]

    # per-kernel durations: K more steps with events between the kernels (those events also stop
    # one kernel's prologue from overlapping the previous one's tail, so these durations are
    # upper bounds of what each kernel costs inside a step)
    n_ev = len(path.names) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    graph_times = []
    for k in range(args.steps):
        path.flush_l2()
        if use_graph and path.L == 1:
            path.graph.replay()
            torch.cuda.synchronize()   # the graph's own events, read before the next replay
            graph_times.append(path.graph_times_ms())
        else:
            path.step(evs[k])
    torch.cuda.synchronize()
    clocks = None
    if sampler:
        # keep the GPU loaded until the clock sampler has seen the load
        t_end = time.perf_counter() + 0.6
        while time.perf_counter() < t_end:
            path.flush_l2()
            plain_step()
        torch.cuda.synchronize()
        clocks = sampler.stop()

    per_kernel = {n_: [] for n_ in path.names}
    evented_ms = []
    if use_graph and path.L == 1:
        for ks, st in graph_times:
            evented_ms.append(st)
            for n_, t in zip(path.names, ks):
                per_kernel[n_].append(t)
    else:
        for ev in evs:
            evented_ms.append(ev[0].elapsed_time(ev[-1]))
            for i, n_ in enumerate(path.names):
                per_kernel[n_].append(ev[i].elapsed_time(ev[i + 1]))
    status = path.read_status()
    value, total_ms = job_throughput(float(sum(step_ms)), shape.b * shape.s, args.steps)
    ms_per_step = total_ms / args.steps
    avg_us = {n_: round(1e3 * statistics.mean(v), 2) for n_, v in per_kernel.items()}

    wk = work(shape, data)
    pk = peaks()
    dominant = max(avg_us, key=lambda n_: avg_us[n_])
    rec = {"value": round(value, 1), "unit": unit, "ms_per_step": round(ms_per_step, 5),
           "roofline": step_roofline(path.names, wk, ms_per_step / 1e3, pk, shape.name),
           "dominant_kernel_roofline": roofline_of(dominant, wk[dominant], avg_us[dominant] / 1e6, pk, shape.name),
           "kernel_us": avg_us,
           "kernel_roofline_frac": {n_: roofline_of(n_, wk[n_], avg_us[n_] / 1e6, pk, shape.name)["frac"]
                                    for n_ in path.names},
           "ms_per_step_with_kernel_events": round(statistics.mean(evented_ms), 5),
           "gpu_launches": path.launches_per_step() * args.steps, "clocks": clocks,
           "launch": "CUDA graph of the decode step, replayed per step" if use_graph else "direct C-ABI calls",
           "device_status_flags": status}
    if primary:
        rec["dtype"] = "e2m1+bf16" if shape.fp4_keys else "fp4kv+bf16" if shape.fp4_kv else "bf16"
        rec["config"] = workload_config(shape, args)
        if not args.no_e2e and shape.n_layers == 1 and not shape.prefill:
            rec["e2e"] = measure_e2e(path, data, args.steps, args.warmup)
        if not args.no_cpu_baseline:
            rec["cpu_baseline"] = cpu_baseline(shape, data, output_rope=args.output_rope)
    else:
        rec["config"] = workload_config(shape, args)
    del path
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def main(argv=None):
    args = parse(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    shape = workloads.config(args.workload)

    if args.impl == "reference":
        if rank != 0:   # the CPU oracle runs once, on rank 0
            return
        print(json.dumps(reference_arm(args, shape, workload_config(shape, args))), flush=True)
        return
    if world > 1 or args.gpus > 1:
        # one GPU per process and one process: the path's kernels (clusters with multicast loads
        # inside this GPU's memory) are only ever launched by a single-GPU run
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus), "unavailable":
                              "single-GPU library: bench.py runs on one GPU only (no multi-GPU path)"}), flush=True)
        return
    if os.environ.get("STI_LIB"):
        raise SystemExit("bench.py measures the in-tree libsti.so: unset STI_LIB")

    import torch

    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)

    import __graft_entry__

    __graft_entry__.build()
    rec = bench_workload(args.workload, args, device, primary=True)
    line = {"metric": METRIC, "value": rec.pop("value"), "unit": rec.pop("unit"), "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec.pop("ms_per_step"), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": rec.pop("dtype"), "data": "synthetic",
            "config": rec.pop("config")}
    line.update(rec)
    if args.workload == 2 and not args.no_sub:
        for key, n in SUB_WORKLOADS:
            line[key] = bench_workload(n, args, device, primary=False)
        line["gpu_launches"] += sum(line[key]["gpu_launches"] for key, _ in SUB_WORKLOADS)
    print(json.dumps(line), flush=True)


def measure_e2e(path: GpuPath, data: dict, steps: int, warmup: int) -> dict:
    """Decode steps through sti_decode_fused with the step's inputs (q, index q, weights,
    start_pos, and the rotation table if any) packed in one pinned host buffer, uploaded with one
    copy into a device buffer the decode arguments point into, and the attention output copied
    back to pinned host memory: once one step at a time, synchronised (serial_value), and once as
    a double-buffered serving loop whose copies overlap the neighbouring steps' kernels (value)."""
    import torch

    sti = path.sti
    shp = path.shape
    parts = [("iq", data["iq"].view(np.uint8)), ("w", data["w"].view(np.uint8)),
             ("start_pos", data["start_pos"].astype(np.int32).view(np.uint8)), ("q", data["q"][0].view(np.uint8))]
    if path.rope_cs is not None:
        parts.append(("rope_cs", path.rope_cs[:, 0].cpu().numpy().view(np.uint8)))
    offs, off = {}, 0
    for name, arr in parts:
        offs[name] = off
        off = (off + arr.size + 255) // 256 * 256
    h_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    hv = h_buf.numpy()
    for name, arr in parts:
        hv[offs[name]:offs[name] + arr.size] = arr.reshape(-1)
    d_buf = torch.empty(off, dtype=torch.uint8, device=path.dev)

    def view(name, like, dtype):
        n = like.numel() * like.element_size()
        return d_buf[offs[name]:offs[name] + n].view(dtype).view(like.shape)

    d_q = view("q", path.q[0], torch.bfloat16)
    d_iq = view("iq", path.iq, torch.bfloat16)
    d_w = view("w", path.w, torch.bfloat16)
    d_sp = view("start_pos", path.sp, torch.int32)
    d_cs = None if path.rope_cs is None else view("rope_cs", path.rope_cs[:, 0].contiguous(), torch.float32)
    a, out, tk = sti.decode_args(d_q, path.win[0], path.comp, path.sink[0], shp.softmax_scale, d_iq, path.ik, d_w,
                                 shp.index_scale, d_sp, shp.ratio, shp.n_cols, shp.topk, rope_cs=d_cs,
                                 ik_codes=path.ik_codes, ik_scales=path.ik_scales,
                                 comp_codes=path.comp_codes, comp_scales=path.comp_scales)
    ws = sti.workspace(sti.decode_workspace_size(a), path.dev)
    h_out = torch.empty(out.numel(), dtype=torch.bfloat16).pin_memory()
    bi = sum(arr.size for _, arr in parts)
    bo = h_out.numel() * 2
    main = torch.cuda.current_stream()

    def serial():
        d_buf.copy_(h_buf, non_blocking=True)
        sti.decode_fused(a, ws)
        h_out.copy_(out.view(-1), non_blocking=True)
        main.synchronize()

    for _ in range(warmup):
        path.flush_l2()
        serial()
    el = 0.0
    for _ in range(steps):
        path.flush_l2()
        main.synchronize()
        t0 = time.perf_counter()
        serial()
        el += time.perf_counter() - t0
    serial_value = round(path.b * steps / el, 1)

    # A serving loop: two device input buffers and two outputs.  Step i's upload (one copy stream)
    # overlaps step i-1's kernels, its download (a second copy stream) overlaps step i+1's, and
    # the host waits for step i-1's result on the host before issuing step i+1.  Every step still
    # moves its own inputs and output; no L2 flush fits between overlapped steps (the index keys a
    # step streams, 134 MB at the decode shape, exceed L2).
    d_bufs = [d_buf, torch.empty_like(d_buf)]
    views1 = {}
    for name, like, dt in (("q", path.q[0], torch.bfloat16), ("iq", path.iq, torch.bfloat16),
                           ("w", path.w, torch.bfloat16), ("start_pos", path.sp, torch.int32)):
        n = like.numel() * like.element_size()
        views1[name] = d_bufs[1][offs[name]:offs[name] + n].view(dt).view(like.shape)
    d_cs1 = None
    if path.rope_cs is not None:
        n = path.rope_cs[:, 0].numel() * 4
        d_cs1 = d_bufs[1][offs["rope_cs"]:offs["rope_cs"] + n].view(torch.float32).view(path.rope_cs[:, 0].shape)
    a1, out1, _ = sti.decode_args(views1["q"], path.win[0], path.comp, path.sink[0], shp.softmax_scale, views1["iq"],
                                  path.ik, views1["w"], shp.index_scale, views1["start_pos"], shp.ratio, shp.n_cols,
                                  shp.topk, rope_cs=d_cs1, ik_codes=path.ik_codes, ik_scales=path.ik_scales,
                                 comp_codes=path.comp_codes, comp_scales=path.comp_scales)
    argv, outs = [a, a1], [out, out1]
    h_outs = [h_out, torch.empty(out.numel(), dtype=torch.bfloat16).pin_memory()]
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        main.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(ev_comp[k])   # step i-2's kernels have read d_bufs[k]
                d_bufs[k].copy_(h_buf, non_blocking=True)
                ev_up[k].record(s_up)
            main.wait_event(ev_up[k])
            sti.decode_fused(argv[k], ws)
            ev_comp[k].record(main)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_comp[k])
                h_outs[k].copy_(outs[k].view(-1), non_blocking=True)
                ev_down[k].record(s_down)
            if i >= 1:
                ev_down[(i - 1) & 1].synchronize()   # step i-1's output is on the host
        ev_down[(n - 1) & 1].synchronize()
        return time.perf_counter() - t0

    pipelined(max(warmup, 2))
    value = round(path.b * steps / pipelined(steps), 1)
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "serial_value": serial_value,
            "how": "sti_decode_fused with the step's inputs in one pinned host buffer (one host-to-device copy "
                   "into the device buffer the arguments point into) and the attention output copied back to "
                   "pinned host memory, every step; value: a serving loop that overlaps step i's upload and "
                   "step i-1's download with the kernels (double-buffered inputs and outputs, the host waiting "
                   "for each step's output); serial_value: copy, call, copy back and synchronise, one step at "
                   "a time with the L2 flushed between steps; wall clock"}


if __name__ == "__main__":
    main()
