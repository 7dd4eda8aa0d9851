#!/usr/bin/env python3
"""Benchmark of the fused row-wise RMSNorm on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole op (load, optional residual add, sum of
squares, scale, weighted store) over one batch of the workload: one launch of
the library through its C ABI.  The headline workload is the largest one that
fits a GPU: bf16 65536 x 8192 with a fused residual add and a weight (x with
0.1 % outliers; about 1 GiB a tensor), the bandwidth-roofline case.  The
metric is achieved HBM bandwidth over the op's algorithmic bytes (read x
[+ residual], write y [+ residual_out], read w once per launch), with rows/s
beside it; every other workload is timed the same way in ``per_config``.

Timing: inputs are resident on the device before the timed region; launches
are recorded in CUDA graphs and rotate through enough distinct buffer sets
that their footprint is at least 4x the L2 size (the headline's one set of
4 GiB already is), so each launch reads from HBM; CUDA events on the
launching stream bracket exactly K steps, with a barrier and a device
synchronise on both sides; nvidia-smi samples clocks during the timed region
and the half second of identical launches just before it.  ``e2e`` repeats
the measurement through the C ABI's host-buffer call (``rmsnorm_fwd_host``:
inputs in pinned host memory, outputs read back, every step), beside the
host link's own rate for the same copies with no launch (``link_gbs``),
which bounds it.  The CPU baseline is
the fp64 oracle on the host cores over a bounded sample of the headline's
rows.

Under torchrun each rank runs its own replica on its own GPU (the op has no
exchange between rows, so there is no collective on the data path); the
value is the work of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "bf16_res_65536x8192_w"
METRIC = "RMSNorm achieved HBM GB/s and % of GB300 peak; rows/s per config"
PER_CONFIG = ["bf16_4096x576", "f32_64x256", "bf16_res_16384x2048", "bf16_qk_262144x128", "bf16_decode_1x4096",
              "bf16_decode_8x4096", "bf16_decode_64x4096", "bf16_res_65536x8192_nw", "bf16_4096x32768_w",
              "bf16_res_4096x40960_w", "bf16_2048x65536_w", "bf16_res_2048x65536_w", "f32_res_2048x65536_w"]
# Workloads whose per-config entry also carries the launch-overhead context
# (copy floor, independent batches, hot L2, repeated runs).
SMALL_CONTEXT = ("bf16_4096x576",)
# Rows of the headline the CPU baseline's sample takes (64 MiB of each input),
# and the rows the reference arm's steps are taken from.
CPU_SAMPLE_ROWS = 4096
REF_POOL_ROWS = 16384
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description="fused RMSNorm benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-config table")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work for the oracle baseline (0 disables it)")
    ap.add_argument("--e2e-steps", type=int, default=0, help="steps of the e2e region (0: auto)")
    ap.add_argument("--ncu-case", default=None,
                    help="profiling mode: launch this workload --launches times and exit")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--rows", type=int, default=0, help="profiling mode: override the row count")
    ap.add_argument("--hidden", type=int, default=0, help="profiling mode: override the hidden size")
    ap.add_argument("--grid", type=int, default=0,
                    help="profiling mode: force this grid (blocks stride over row groups)")
    ap.add_argument("--misalign", action="store_true",
                    help="profiling mode: offset every tensor by one element (scalar path)")
    ap.add_argument("--plan", default="",
                    help="profiling mode: JSON object of plan fields set over the library's plan")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Host-side planning and argument checks: not device code, so not part of
# the hash that says whether a profile still describes the kernels.
HOST_ONLY_SOURCES = ("rmsnorm_api.cu", "rmsnorm_host.cu", "rmsnorm_host_static.cu")   # no kernel in them


def code_tokens(text):
    """C/C++ source with comments removed and whitespace collapsed (a comment
    edit does not change the code a profile describes)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                       # string or character literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the device code (kernels and their instantiations), comments
    and layout aside."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_reduction_norm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in HOST_ONLY_SOURCES:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, plan=None, with_source=False, rows=None):
    """DRAM bytes per launch from the committed ncu summary of this workload
    (profiles/ncu_*.md with a matching ``profile_workload:`` line), if it was
    taken on the current device code and, when ``plan`` is given, with the
    same launch plan; else None.  A summary of a row slice of the workload
    (``profile_workload: <name>@--rows<n>``, taken where the full workload is
    too large for a profiler capture) counts when ``rows`` is given: its
    bytes are scaled by rows / n (every row of a launch moves the same bytes)
    and its plan must match in everything but the grid.  ``with_source`` also
    returns which summary gave the figure, or why none did."""
    value, source = _profiled_traffic(workload, plan, rows)
    return (value, source) if with_source else value


def _profiled_traffic(workload, plan, rows=None):
    pdir = os.path.join(ROOT, "profiles")
    try:
        names = sorted(os.listdir(pdir))
    except OSError:
        return None, "no profiles/ directory"
    why = f"no ncu summary of {workload} in profiles/"
    found = []
    for name in names:
        if not (name.startswith("ncu_") and name.endswith(".md")):
            continue
        text = open(os.path.join(pdir, name)).read()
        m_wl = re.search(r"profile_workload:\s*(\S+)\s*$", text, re.M)
        if not m_wl:
            continue
        base, _, slice_arg = m_wl.group(1).partition("@")
        m_slice = re.fullmatch(r"--rows(\d+)", slice_arg)
        if base != workload or (slice_arg and (not m_slice or not rows)):
            continue
        found.append((0 if not slice_arg else 1, name, text, int(m_slice.group(1)) if m_slice else None))
    for _, name, text, slice_rows in sorted(found):
        m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
        m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
        m_plan = re.search(r"^Plan: `(\{.*\})`", text, re.M)
        if plan is not None:
            got = json.loads(m_plan.group(1)) if m_plan else None
            if got is not None and slice_rows:
                got, want = dict(got, grid=None), dict(plan, grid=None)
            else:
                want = plan
            if got != want:
                why = f"profiles/{name} was taken with another launch plan"
                continue
        if m_hash and m_bytes and m_hash.group(1) == kernel_source_hash():
            if slice_rows:
                scaled = int(round(int(m_bytes.group(1)) * rows / slice_rows))
                return scaled, (f"profiles/{name} (device code hash {m_hash.group(1)}, same plan but the grid): "
                                f"a {slice_rows}-row slice, its DRAM bytes scaled by {rows}/{slice_rows}")
            return int(m_bytes.group(1)), f"profiles/{name} (device code hash {m_hash.group(1)}, same plan)"
        why = f"profiles/{name} predates the current device code"
    return None, why


def aggregate(world, bytes_per_step, rows_per_step, steps, ms_max):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    secs = ms_max / 1e3
    return world * bytes_per_step * steps / secs / 1e9, world * rows_per_step * steps / secs


def reduce_max(value, dist, device):
    """Max over ranks of a float (identity without a process group)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples (host receive time attached) while the GPU works."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        window = [p for t, p in self.samples if t0 <= t <= t1]
        source = "timed region"
        if not window:
            window = [p for _, p in self.samples]
            source = "whole run (timed region shorter than the sampling period)"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm = [num(p[0]) for p in window if num(p[0]) is not None]
        mx = [num(p[1]) for p in window if num(p[1]) is not None]
        pw = [num(p[2]) for p in window if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in window:
            for name, v in zip(names, p[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons),
                "samples": len(window), "source": source}


def gpu_id_for(local_rank):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local_rank]
        return local_rank


# ------------------------------------------------------------ device side

class Launcher:
    """Buffer sets of one workload and a C-ABI launch over set i % n_sets."""

    def __init__(self, wl, device, stream, min_footprint, seed=0, n_sets=None):
        import torch
        from row_reduction_norm_gb300 import _native as N
        from row_reduction_norm_gb300 import api, workloads as W
        self.N = N
        self.wl = wl
        self.stream = stream
        per_set = wl.rows * wl.hidden * wl.elem_bytes * (4 if wl.has_res else 2)
        self.n_sets = n_sets or max(1, math.ceil(min_footprint / max(per_set, 1)))
        self.sets = []
        w = None
        for s in range(self.n_sets):
            x, r, w_s = W.make_inputs(wl, seed=seed + 16 * s, device=device)
            if w is None:
                w = w_s
            y = torch.empty_like(x)
            h = torch.empty_like(x) if r is not None else None
            self.sets.append((x, r, y, h))
        self.w = w
        self.code = api.dtype_code(self.sets[0][0].dtype)
        self.ptrs = [(x.data_ptr(), None if r is None else r.data_ptr(), y.data_ptr(),
                      None if h is None else h.data_ptr()) for x, r, y, h in self.sets]
        self.w_ptr = None if w is None else w.data_ptr()
        self.footprint = per_set * self.n_sets
        x0, r0, y0, h0 = self.sets[0]
        self.plan = api.plan_for(x0, w=w, residual=r0, out=y0, residual_out=h0)

    def launch(self, i):
        x, r, y, h = self.ptrs[i % self.n_sets]
        self.N.rmsnorm_fwd(x, r, self.w_ptr, y, h, self.wl.rows, self.wl.hidden, self.wl.eps, self.code,
                           self.stream.cuda_stream)

    def launch_with(self, i, slot, w_ptr):
        """Launch on buffer set `slot` with the given weight pointer."""
        x, r, y, h = self.ptrs[slot]
        self.N.rmsnorm_fwd(x, r, w_ptr, y, h, self.wl.rows, self.wl.hidden, self.wl.eps, self.code,
                           self.stream.cuda_stream)

    def graph(self, start, count):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(start, start + count):
                self.launch(i)
        return g


class ChainLauncher:
    """A dependent chain of the workload's launches: two buffers, launch i
    reads buffer i % 2 and writes the other, so every launch reads what the
    one before it wrote (x only: workloads without a residual)."""

    def __init__(self, L):
        import torch
        self.N, self.wl, self.stream, self.code, self.w_ptr = L.N, L.wl, L.stream, L.code, L.w_ptr
        x0 = L.sets[0][0]
        self.bufs = [x0.clone(), torch.empty_like(x0)]
        self.n_sets = 2

    def launch(self, i):
        src, dst = self.bufs[i % 2], self.bufs[(i + 1) % 2]
        self.N.rmsnorm_fwd(src.data_ptr(), None, self.w_ptr, dst.data_ptr(), None, self.wl.rows, self.wl.hidden,
                           self.wl.eps, self.code, self.stream.cuda_stream)

    graph = Launcher.graph


class CastLauncher(Launcher):
    """RMSNorm in the op-by-op cast order (rmsnorm_fwd_cast), same buffers."""

    def launch(self, i):
        x, r, y, h = self.ptrs[i % self.n_sets]
        self.N.rmsnorm_fwd_cast(x, r, self.w_ptr, y, h, self.wl.rows, self.wl.hidden, self.wl.eps, self.code,
                                None, self.stream.cuda_stream)


class LNLauncher(Launcher):
    """LayerNorm workloads: the Launcher's buffer sets plus a bias."""

    def __init__(self, wl, device, stream, min_footprint, seed=0):
        import torch
        from row_reduction_norm_gb300 import api, workloads as W
        super().__init__(wl, device, stream, min_footprint, seed)
        _, _, _, b = W.make_ln_inputs(wl, seed=seed, device=device, rows=1)
        self.b = b
        self.b_ptr = None if b is None else b.data_ptr()
        x0, r0, y0, h0 = self.sets[0]
        self.plan = api.layer_norm_plan_for(x0, w=self.w, b=b, residual=r0, out=y0, residual_out=h0)
        del torch

    def launch(self, i):
        x, r, y, h = self.ptrs[i % self.n_sets]
        self.N.layernorm_fwd(x, r, self.w_ptr, self.b_ptr, y, h, self.wl.rows, self.wl.hidden, self.wl.eps,
                             self.code, None, self.stream.cuda_stream)


class MXLauncher(Launcher):
    """RMSNorm with MXFP8 output: x (+ residual) in, codes and scales (+ residual_out) out."""

    def __init__(self, wl, device, stream, min_footprint, seed=0):
        import torch
        from row_reduction_norm_gb300 import api, workloads as W
        self.N = api.N
        self.wl = wl
        self.stream = stream
        e = wl.rows * wl.hidden
        per_set = e * wl.elem_bytes * (1 + (2 if wl.has_res else 0)) + e + e // 32
        self.n_sets = max(1, math.ceil(min_footprint / max(per_set, 1)))
        self.sets, self.scales = [], []
        w = None
        for s in range(self.n_sets):
            x, r, w_s = W.make_inputs(wl, seed=seed + 16 * s, device=device)
            w = w_s if w is None else w
            codes = torch.empty(x.shape, dtype=torch.uint8, device=device)
            sc = torch.empty((wl.rows, wl.hidden // 32), dtype=torch.uint8, device=device)
            h = torch.empty_like(x) if r is not None else None
            self.sets.append((x, r, codes, h))
            self.scales.append(sc)
        self.w = w
        self.code = api.dtype_code(self.sets[0][0].dtype)
        self.ptrs = [(x.data_ptr(), None if r is None else r.data_ptr(), c.data_ptr(),
                      None if h is None else h.data_ptr()) for x, r, c, h in self.sets]
        self.w_ptr = None if w is None else w.data_ptr()
        self.footprint = per_set * self.n_sets
        self.plan = api.rms_norm_mxfp8_plan_for(self.sets[0][0], w=w, residual=self.sets[0][1])

    def launch(self, i):
        x, r, c, h = self.ptrs[i % self.n_sets]
        self.N.rmsnorm_fwd_mxfp8(x, r, self.w_ptr, c, self.scales[i % self.n_sets].data_ptr(), h, self.wl.rows,
                                 self.wl.hidden, self.wl.eps, 0.0, self.code, None, self.stream.cuda_stream)


class NVLauncher(MXLauncher):
    """RMSNorm with NVFP4 output: codes are half a byte an element, one scale per 16."""

    def __init__(self, wl, device, stream, min_footprint, seed=0):
        import torch
        from row_reduction_norm_gb300 import api, workloads as W
        self.N = api.N
        self.wl = wl
        self.stream = stream
        e = wl.rows * wl.hidden
        per_set = e * wl.elem_bytes * (1 + (2 if wl.has_res else 0)) + e // 2 + e // 16
        self.n_sets = max(1, math.ceil(min_footprint / max(per_set, 1)))
        self.sets, self.scales = [], []
        w = None
        for s in range(self.n_sets):
            x, r, w_s = W.make_inputs(wl, seed=seed + 16 * s, device=device)
            w = w_s if w is None else w
            codes = torch.empty((wl.rows, wl.hidden // 2), dtype=torch.uint8, device=device)
            sc = torch.empty((wl.rows, wl.hidden // 16), dtype=torch.uint8, device=device)
            h = torch.empty_like(x) if r is not None else None
            self.sets.append((x, r, codes, h))
            self.scales.append(sc)
        self.w = w
        self.code = api.dtype_code(self.sets[0][0].dtype)
        self.ptrs = [(x.data_ptr(), None if r is None else r.data_ptr(), c.data_ptr(),
                      None if h is None else h.data_ptr()) for x, r, c, h in self.sets]
        self.w_ptr = None if w is None else w.data_ptr()
        self.footprint = per_set * self.n_sets
        self.tensor_scale = W.NV_TENSOR_SCALE
        self.plan = api.rms_norm_nvfp4_plan_for(self.sets[0][0], w=w, residual=self.sets[0][1])

    def launch(self, i):
        x, r, c, h = self.ptrs[i % self.n_sets]
        self.N.rmsnorm_fwd_nvfp4(x, r, self.w_ptr, c, self.scales[i % self.n_sets].data_ptr(), h, self.wl.rows,
                                 self.wl.hidden, self.wl.eps, 0.0, self.tensor_scale, self.code, None,
                                 self.stream.cuda_stream)


class QKLauncher(Launcher):
    """Buffer sets of a fused Q+K workload, normalised in place (the usual use on
    a packed projection), with the same launch interface as Launcher."""

    def __init__(self, wl, device, stream, min_footprint, seed=0):  # noqa: super().__init__ not used
        import torch
        from row_reduction_norm_gb300 import _native as N
        from row_reduction_norm_gb300 import api, workloads as W
        self.N = N
        self.wl = wl
        self.stream = stream
        per_set = wl.tokens * wl.width * wl.elem_bytes
        self.n_sets = max(1, math.ceil(min_footprint / max(per_set, 1)))
        self.sets = []
        qw = kw = None
        for s in range(self.n_sets):
            qkv, q_w, k_w = W.make_qk_inputs(wl, seed=seed + 16 * s, device=device)
            if qw is None:
                qw, kw = q_w, k_w
            self.sets.append((qkv, None, qkv, None))
        self.w, self.k_w = qw, kw
        self.code = api.dtype_code(self.sets[0][0].dtype)
        self.ptrs = [(x.data_ptr(), None, x.data_ptr(), None) for x, _, _, _ in self.sets]
        self.w_ptr = None if qw is None else qw.data_ptr()
        self.kw_ptr = None if kw is None else kw.data_ptr()
        self.footprint = per_set * self.n_sets
        self.plan = api.qk_plan_for(self.sets[0][0], wl.q_heads, wl.k_heads, wl.head_dim, qw, kw)
        self.stride = self.sets[0][0].stride(0)

    def launch(self, i):
        x, _, y, _ = self.ptrs[i % self.n_sets]
        wl = self.wl
        self.N.rmsnorm_qk_fwd(x, y, wl.tokens, self.stride, self.stride, wl.q_heads, wl.k_heads, wl.head_dim,
                              self.w_ptr, self.kw_ptr, wl.weight_bias, wl.eps, self.code, None,
                              self.stream.cuda_stream)


def time_launches(L, steps, warmup, barrier=None, sampler_window=None, graph_len=1024, soak_s=0.0):
    """Exactly `steps` launches between two events on L.stream; returns ms.
    Before them: at least `warmup` launches, continued (untimed, same
    launches) until `soak_s` seconds have passed, so that clock samples taken
    from the start of that soak to the end of the timed region describe the
    GPU under this load even when the timed region is shorter than the
    sampling period."""
    import torch
    with torch.cuda.stream(L.stream):
        L.launch(0)   # fills the library's per-device caches outside any capture
    L.stream.synchronize()
    G = max(1, min(steps, graph_len))
    G = max(1, (G // L.n_sets) * L.n_sets) if G >= L.n_sets else G
    g_main = L.graph(0, G)
    rem = steps % G
    g_rem = L.graph(0, rem) if rem else None
    with torch.cuda.stream(L.stream):
        for _ in range(max(1, math.ceil(warmup / G))):
            g_main.replay()
    L.stream.synchronize()
    t_soak = time.time()
    while time.time() - t_soak < soak_s:
        with torch.cuda.stream(L.stream):
            g_main.replay()
        L.stream.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(L.stream):
        ev0.record(L.stream)
        for _ in range(steps // G):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(L.stream)
    L.stream.synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    if barrier:
        barrier()
    if sampler_window is not None:
        sampler_window.extend([t_soak if soak_s > 0 else t0, t1])
    return ev0.elapsed_time(ev1)


def host_buffers(L):
    """Pinned host copies of buffer set 0's inputs (x, residual, w) and pinned
    host outputs (y, residual_out), with the bytes each step moves each way."""
    import torch
    x, r, y, h = L.sets[0]
    hx = x.cpu().pin_memory()
    hr = None if r is None else r.cpu().pin_memory()
    hw = None if L.w is None else L.w.cpu().pin_memory()
    hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    hh = None if h is None else torch.empty(h.shape, dtype=h.dtype).pin_memory()
    nbytes = lambda t: 0 if t is None else t.numel() * t.element_size()
    return hx, hr, hw, hy, hh, nbytes(hx) + nbytes(hr) + nbytes(hw), nbytes(hy) + nbytes(hh)


def host_link_gbs(L, reps=5):
    """The host link's rate for one step's copies alone: the uploads of x,
    residual and w into buffer set 0 on one stream while the read-backs of y
    and residual_out from buffer set 1 run on another, no launch between;
    (h2d + d2h bytes) / median time, GB/s.  It bounds the end-to-end rate,
    which moves the same bytes each step."""
    import torch
    hx, hr, hw, hy, hh, h2d, d2h = host_buffers(L)
    xd, rd, _, _ = L.sets[0]
    _, _, yd, hd = L.sets[min(1, L.n_sets - 1)]
    wd = None if L.w is None else torch.empty_like(L.w)
    s_k = L.stream
    s_up, s_dn = torch.cuda.Stream(s_k.device), torch.cuda.Stream(s_k.device)
    times = []
    for _ in range(reps + 1):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_k)
        s_up.wait_stream(s_k)
        s_dn.wait_stream(s_k)
        with torch.cuda.stream(s_up):
            for dst, src in ((xd, hx), (rd, hr), (wd, hw)):
                if dst is not None:
                    dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(s_dn):
            for dst, src in ((hy, yd), (hh, hd)):
                if dst is not None:
                    dst.copy_(src, non_blocking=True)
        s_k.wait_stream(s_up)
        s_k.wait_stream(s_dn)
        e1.record(s_k)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return (h2d + d2h) / statistics.median(times[1:]) / 1e6


E2E_CHUNK_BYTES = 64 << 20   # rows a chunk of the host call: about 64 MiB of each tensor


def e2e_chunk_rows(wl):
    return max(1, min(wl.rows, E2E_CHUNK_BYTES // (wl.hidden * wl.elem_bytes)))


def time_e2e_host(L, steps, chunk_rows):
    """End to end through the C ABI's host-buffer call: every step is one
    ``rmsnorm_fwd_host`` call on pinned host x, residual and w, writing pinned
    host y and residual_out; the library streams the rows through the device
    in chunks of ``chunk_rows`` rows (uploads, launches and read-backs on
    three streams over two halves of a device workspace).  Returns (ms for
    `steps` calls, h2d bytes per step, d2h bytes per step)."""
    import torch
    from row_reduction_norm_gb300 import _native as N
    hx, hr, hw, hy, hh, h2d, d2h = host_buffers(L)
    wl = L.wl
    nbytes = N.rmsnorm_host_workspace_bytes(chunk_rows, wl.hidden, L.code, hr is not None)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=L.stream.device)
    ptr = lambda t: None if t is None else t.data_ptr()

    def step():
        N.rmsnorm_fwd_host(ptr(hx), ptr(hr), ptr(hw), ptr(hy), ptr(hh), wl.rows, wl.hidden, wl.eps, L.code,
                           ws.data_ptr(), nbytes, chunk_rows, L.stream.cuda_stream)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(L.stream)
    for _ in range(steps):
        step()
    ev1.record(L.stream)
    torch.cuda.synchronize()
    del ws
    return ev0.elapsed_time(ev1), h2d, d2h


def copy_floor_us(L, steps=8192):
    """Mean time of a plain device copy (torch ``copy_``, y <- x) moving the
    same read + write bytes as one launch of the workload (no residual or
    weight traffic), in the same setting: CUDA graphs of dependent launches
    over the same rotating buffer sets.  It bounds what any kernel of this
    size achieves launch after launch on this device."""
    import torch
    G = max(1, min(steps, 1024))
    G = max(1, (G // L.n_sets) * L.n_sets) if G >= L.n_sets else G
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=L.stream):
        for i in range(G):
            x, _, y, _ = L.sets[i % L.n_sets]
            y.copy_(x)
    with torch.cuda.stream(L.stream):
        g.replay()
    L.stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps = max(1, steps // G)
    with torch.cuda.stream(L.stream):
        e0.record(L.stream)
        for _ in range(reps):
            g.replay()
        e1.record(L.stream)
    L.stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * G)


def independent_chains_us(L, steps=8192):
    """Mean time per launch when consecutive batches do not depend on each
    other: the same C-ABI launches split into two chains on two streams (even
    and odd buffer sets, disjoint), whose launches may then overlap.  Context
    for the dependent-chain figure, not a replacement for it: in a model each
    norm's input comes from the kernel before it."""
    import torch
    streams = [L.stream, torch.cuda.Stream(L.stream.device)]
    G = max(2, min(steps // 2, 1024))
    graphs = []
    saved = L.stream
    try:
        for c, st in enumerate(streams):
            L.stream = st
            with torch.cuda.stream(st):
                L.launch(c)   # library caches filled outside the capture
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for i in range(G):
                    L.launch(2 * i + c)
            graphs.append(g)
    finally:
        L.stream = saved
    for g, st in zip(graphs, streams):
        with torch.cuda.stream(st):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    joined = torch.cuda.Event()
    reps = max(1, steps // (2 * G))
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for _ in range(reps):
        for g, st in zip(graphs, streams):
            with torch.cuda.stream(st):
                g.replay()
    joined.record(streams[1])
    streams[0].wait_event(joined)
    e1.record(streams[0])
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * 2 * G)


def graph_launch_latency_us(L, reps=1000):
    """Device-side latency of one launch: CUDA events around the replay of a
    CUDA graph holding that single launch, median of `reps` (no Python or
    ctypes cost inside the events, unlike ``single_launch_latency_us``)."""
    import torch
    g = L.graph(0, 1)
    with torch.cuda.stream(L.stream):
        for _ in range(8):
            g.replay()
    L.stream.synchronize()
    ts = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        with torch.cuda.stream(L.stream):
            e0.record(L.stream)
            g.replay()
            e1.record(L.stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def single_launch_latency_us(L, reps=1000):
    """One C-ABI launch issued from Python between two CUDA events, median of
    `reps`: the device time plus the cost of issuing the call."""
    import torch
    ts = []
    for i in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(L.stream):
            e0.record(L.stream)
            L.launch(i)
            e1.record(L.stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def plan_summary(p):
    d = p.as_dict()
    out = {"kernel": d["kernel_name"], "regime": d["regime_name"], "threads_per_row": d["threads_per_row"],
           "chunks_per_thread": d["chunks_per_thread"], "vec_elems": d["vec_elems"],
           "block": d["block_threads"], "grid": d["grid"]}
    if d["rows_per_block"] != max(1, d["block_threads"] // max(1, d["threads_per_row"])):
        out["rows_per_block"] = d["rows_per_block"]     # fewer rows a block than row slots
    if d["cluster_ctas"]:
        out["cluster_ctas"] = d["cluster_ctas"]         # blocks of a cluster that share a row
    return out


# ------------------------------------------------------------ CPU oracle

def oracle_rate(wl, seconds, threads, host_inputs=None):
    """The oracle, as it stands, over the given rows of the workload (all of
    them by default), pass after pass until `seconds` of work; returns a dict."""
    import oracle
    from row_reduction_norm_gb300 import workloads as W
    if host_inputs is None:
        x, r, w = W.make_inputs(wl, seed=0, device="cpu")
        host_inputs = (W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w))
    xn, rn, wn = host_inputs
    rows_done = 0
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype=wl.dtype, threads=threads)
        rows_done += xn.shape[0]
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    per_launch_bytes = wl.algorithmic_bytes(rows=xn.shape[0])
    what = (f"the {wl.rows}x{wl.hidden} {wl.dtype} batch" if xn.shape[0] == wl.rows else
            f"the first {xn.shape[0]} rows of the {wl.rows}x{wl.hidden} {wl.dtype} batch")
    return {"value": per_launch_bytes * passes / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "rows_per_s": rows_done / dt,
            "sample": f"{passes} passes over {what} ({dt:.1f} s, fp64 C oracle, {threads} threads over row "
                      f"blocks; GB/s counts the algorithmic bytes of the rows done, the weight once a pass)"}


def bench_config(wl, world):
    """The ``config`` object of the JSON line: the workload and how L2 is kept
    out of the figure.  Both arms print exactly this object."""
    per_launch = wl.algorithmic_bytes()
    moved = wl.rows * wl.hidden * wl.elem_bytes
    return {
        "workload": wl.name, "rows": wl.rows, "hidden": wl.hidden, "dtype": wl.dtype, "eps": wl.eps,
        "residual": wl.has_res, "weight": wl.has_w, "outliers": wl.outlier_frac,
        "bytes_per_step": per_launch,
        "l2": (f"inputs larger than L2: one step reads {moved * (2 if wl.has_res else 1) // 2 ** 20} MiB; "
               "workloads whose launches fit in L2 rotate over buffer sets of at least 4x the L2 size"),
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def small_context(L, wl, steps):
    """Launch-overhead context for a workload whose launches move a few MB:
    the copy floor, independent batches, repeated runs and a hot-L2 figure."""
    import torch
    b = wl.algorithmic_bytes()
    floor_us = copy_floor_us(L)
    indep_us = independent_chains_us(L)
    rep_steps = 20000
    reps_us = sorted(time_launches(L, rep_steps, 8) * 1e3 / rep_steps for _ in range(10))
    LH = Launcher(wl, L.stream.device, L.stream, 0)
    hot_us = time_launches(LH, rep_steps, max(3, rep_steps // 20)) * 1e3 / rep_steps
    del LH
    chain_us = None
    if not wl.has_res:
        LC = ChainLauncher(L)
        chain_us = time_launches(LC, rep_steps, max(3, rep_steps // 20)) * 1e3 / rep_steps
        del LC
    torch.cuda.empty_cache()
    kernel_us = statistics.median(reps_us)
    return {
        "launch_floor": {"copy_us": round(floor_us, 3), "kernel_us": round(kernel_us, 3),
                         "kernel_vs_copy": round(floor_us / kernel_us, 3),
                         "what": "torch copy_ of the same x -> y bytes, same graphs and buffer rotation: the "
                                 "per-launch floor of a dependent chain of this size"},
        "independent_batches": {"gbs": round(b / (indep_us / 1e6) / 1e9, 1), "us_per_launch": round(indep_us, 3),
                                "streams": 2,
                                "what": "context, not the metric: the same launches as two chains of "
                                        "independent batches on two streams, free to overlap"},
        "repeats": {"n": len(reps_us), "steps_each": rep_steps, "median_us": round(kernel_us, 3),
                    "min_us": round(reps_us[0], 3), "max_us": round(reps_us[-1], 3),
                    "what": "the launches timed again as 10 separate runs of steps_each launches"},
        "hot_l2": {"us_per_launch": round(hot_us, 3), "gbs": round(b / (hot_us / 1e6) / 1e9, 1),
                   "what": "hot L2, not HBM: one buffer set reused by every launch, so the inputs stay in L2"},
        "dependent_chain": None if chain_us is None else {
            "us_per_launch": round(chain_us, 3), "gbs": round(b / (chain_us / 1e6) / 1e9, 1),
            "what": "each launch reads the y the launch before it wrote (two buffers; at this size they stay in "
                    "L2): the norm as a model runs it, where its input is the previous kernel's output"},
    }


def e2e_steps_for(wl, requested):
    """Steps of the end-to-end region: as asked, else about two seconds of
    host-link traffic at 150 GB/s (8 to 4096 steps)."""
    if requested:
        return requested
    link = wl.rows * wl.hidden * wl.elem_bytes * (4 if wl.has_res else 2)
    return int(max(8, min(4096, 2.0 / max(link / 150e9, 1e-9))))


# ------------------------------------------------------------------ arms

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    from row_reduction_norm_gb300 import build as B
    B.build()
    from row_reduction_norm_gb300 import workloads as W

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if dist is not None:
            dist.barrier()

    peak, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 128 * 2 ** 20)
    min_footprint = 4 * l2
    stream = torch.cuda.Stream(device)
    wl = W.WORKLOADS[args.workload]

    if args.ncu_case:
        run_profile_case(args, device, stream)
        return

    L = Launcher(wl, device, stream, min_footprint)
    headline_sets = L.n_sets
    sampler = ClockSampler(gpu_id_for(local)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    window = []
    ms = time_launches(L, args.steps, args.warmup, barrier=barrier, sampler_window=window, soak_s=0.5)
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    ms_max = reduce_max(ms, dist, device)
    launch_bytes = wl.algorithmic_bytes()
    per_launch_s = ms / 1e3 / args.steps
    achieved = launch_bytes / per_launch_s / 1e9
    value, rows_per_s = aggregate(world, launch_bytes, wl.rows, args.steps, ms_max)
    plan = plan_summary(L.plan)
    pdl = bool(L.plan.pdl)
    rep_steps = max(1, min(args.steps, int(math.ceil(0.2 / max(per_launch_s, 1e-9)))))
    reps_us = sorted(time_launches(L, rep_steps, 3) * 1e3 / rep_steps for _ in range(5))

    # end to end through the public call: a second buffer set lets uploads,
    # launches and read-backs of consecutive steps overlap
    e2e_steps = e2e_steps_for(wl, args.e2e_steps)
    del L
    torch.cuda.empty_cache()
    LE = Launcher(wl, device, stream, 0, n_sets=2)
    chunk = e2e_chunk_rows(wl)
    e_ms, h2d, d2h = time_e2e_host(LE, e2e_steps, chunk)
    e2e_value, _ = aggregate(world, launch_bytes, wl.rows, e2e_steps, reduce_max(e_ms, dist, device))
    serial_steps = max(2, e2e_steps // 4)
    s_ms, _, _ = time_e2e_host(LE, serial_steps, wl.rows)
    e2e_serial, _ = aggregate(world, launch_bytes, wl.rows, serial_steps, reduce_max(s_ms, dist, device))
    link = host_link_gbs(LE)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        n = min(wl.rows, CPU_SAMPLE_ROWS)
        x0, r0, _, _ = LE.sets[0]
        host = (W.to_numpy_bits(x0[:n]), W.to_numpy_bits(None if r0 is None else r0[:n]), W.to_numpy_bits(LE.w))
        cpu = oracle_rate(wl, args.cpu_seconds, os.cpu_count() or 1, host)
        one = oracle_rate(wl, max(1.0, args.cpu_seconds / 4), 1, host)
        cpu["single_thread"] = {"value": one["value"], "rows_per_s": one["rows_per_s"], "cores": 1,
                                "sample": one["sample"]}
    del LE
    torch.cuda.empty_cache()

    per_config = []
    if not args.no_per_config:
        for name, (cw, launcher_cls, bytes_of, kind) in per_config_table(W).items():
            qk, ln, mx, nv = kind == "qk", kind == "ln", kind == "mx", kind == "nv"
            CL = launcher_cls(cw, device, stream, min_footprint)
            # calibrate: about 0.3 s of launches
            cal = time_launches(CL, 64, 8)
            k = int(max(64, min(200000, 0.3 / max(cal / 1e3 / 64, 1e-9))))
            cms = time_launches(CL, k, max(3, k // 20), barrier=barrier)
            t_launch = cms / 1e3 / k
            b = bytes_of(cw)
            rows = cw.tokens * (cw.q_heads + cw.k_heads) if qk else cw.rows
            entry = {"workload": name, "rows": rows, "hidden": cw.head_dim if qk else cw.hidden,
                     "dtype": cw.dtype, "bytes_per_launch": b, "us_per_launch": round(t_launch * 1e6, 3),
                     "gbs": round(b / t_launch / 1e9, 1), "frac_of_peak": round(b / t_launch / 1e9 / peak, 4),
                     "rows_per_s": round(rows / t_launch, 1), "steps": k,
                     "buffer_sets": CL.n_sets, "plan": plan_summary(CL.plan)}
            if qk:
                entry.update({"op": "fused q+k head norm, in place", "tokens": cw.tokens,
                              "q_heads": cw.q_heads, "k_heads": cw.k_heads, "v_heads": cw.v_heads,
                              "weight_bias": cw.weight_bias})
            else:
                entry.update({"residual": cw.has_res, "weight": cw.has_w})
            if ln:
                entry.update({"op": "layernorm", "bias": cw.has_b})
            if mx:
                entry.update({"op": "rmsnorm, MXFP8 output (E4M3 codes, E8M0 scale per 32)"})
            if kind == "cast":
                entry.update({"op": "rmsnorm, cast order (normalised value rounded to bf16 before the weight)"})
            if nv:
                entry.update({"op": "rmsnorm, NVFP4 output (E2M1 codes, E4M3 scale per 16, tensor scale "
                                    f"{W.NV_TENSOR_SCALE})"})
            if rows <= 64 or (qk and cw.tokens <= 64):
                entry["graph_launch_latency_us"] = round(graph_launch_latency_us(CL), 3)
                entry["single_launch_latency_us"] = round(single_launch_latency_us(CL), 2)
            if name in SMALL_CONTEXT:
                entry.update(small_context(CL, cw, k))
            per_config.append(entry)
            del CL
            torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    clocks = sampler.summary(window[0], window[1]) if sampler and window else None
    if clocks is not None and clocks.get("source") == "timed region":
        clocks["source"] = "timed region and the 0.5 s of identical launches just before it"
    traffic, traffic_source = profiled_traffic(args.workload, plan, with_source=True, rows=wl.rows)
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic",
        "rows_per_s": round(rows_per_s, 1),
        "frac_of_peak": round(achieved / peak, 4),
        "config": bench_config(wl, world),
        "timing": f"CUDA graphs of C-ABI launches over {headline_sets} buffer set(s) (L2 {l2 // 2 ** 20} MiB), "
                  "CUDA events on the launching stream, exactly `steps` launches between them",
        "plan": plan,
        "pdl": pdl,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "traffic_source": traffic_source,
                     "kernel": f"rms_{plan['kernel']}_kernel",
                     "algorithmic_bytes_per_launch": launch_bytes},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "serial_value": round(e2e_serial, 2), "chunk_rows": chunk,
                "link_gbs": round(link, 2), "frac_of_link": round(e2e_value / world / link, 4),
                "link_what": "one step's uploads and read-backs alone, the two directions concurrent on two "
                             "streams, no launch (median of 5, same process, just after the e2e region)",
                "what": "every step one rmsnorm_fwd_host call (the C ABI's host-buffer entry point) on pinned "
                        "host x, residual and w, writing pinned host y and residual_out: the library copies "
                        "chunks of chunk_rows rows into a device workspace, launches on them and copies the "
                        "outputs back, uploads, launches and read-backs overlapping on three streams "
                        "(serial_value: the same call with the whole batch as one chunk, nothing overlapping)"},
        "repeats": {"n": len(reps_us), "steps_each": rep_steps, "median_us": round(statistics.median(reps_us), 3),
                    "min_us": round(reps_us[0], 3), "max_us": round(reps_us[-1], 3),
                    "what": "the headline launches timed again as separate runs of steps_each launches"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


def per_config_table(W):
    """name -> (workload, launcher class, algorithmic bytes of one launch, kind)
    for every workload the per-config table times, in order."""
    table = {}
    for name in PER_CONFIG:
        table[name] = (W.WORKLOADS[name], Launcher, lambda w: w.algorithmic_bytes(), "rms")
    for name, wl in W.CAST_WORKLOADS.items():
        table[name] = (wl, CastLauncher, lambda w: w.algorithmic_bytes(), "cast")
    for name, wl in W.QK_WORKLOADS.items():
        table[name] = (wl, QKLauncher, lambda w: w.algorithmic_bytes(), "qk")
    for name, wl in W.LN_WORKLOADS.items():
        table[name] = (wl, LNLauncher, lambda w: w.algorithmic_bytes(), "ln")
    for name, wl in W.MX_WORKLOADS.items():
        table[name] = (wl, MXLauncher, W.mx_algorithmic_bytes, "mx")
    for name, wl in W.NV_WORKLOADS.items():
        table[name] = (wl, NVLauncher, W.nv_algorithmic_bytes, "nv")
    return table


def run_profile_case(args, device, stream):
    """A few launches of one workload, for ncu (no timing)."""
    import dataclasses
    import torch
    from row_reduction_norm_gb300 import _native as N
    from row_reduction_norm_gb300 import api, workloads as W
    table = per_config_table(W)
    if args.ncu_case in table and table[args.ncu_case][3] != "rms":
        wl, launcher_cls, bytes_of, kind = table[args.ncu_case]
        qk = kind == "qk"
        if not qk and (args.rows or args.hidden):
            wl = dataclasses.replace(wl, rows=args.rows or wl.rows, hidden=args.hidden or wl.hidden)
        L = launcher_cls(wl, device, stream, 0)
        with torch.cuda.stream(stream):
            for i in range(args.launches):
                L.launch(i)
        stream.synchronize()
        nbytes = bytes_of(wl)
        rows = wl.tokens * (wl.q_heads + wl.k_heads) if qk else wl.rows
        print(json.dumps({"ncu_case": wl.name, "rows": rows, "hidden": wl.head_dim if qk else wl.hidden,
                          "launches": args.launches, "bytes_per_launch": nbytes, "plan": plan_summary(L.plan)}))
        return
    wl = W.WORKLOADS[args.ncu_case]
    if args.rows or args.hidden:
        wl = dataclasses.replace(wl, rows=args.rows or wl.rows, hidden=args.hidden or wl.hidden)
    x, r, w = W.make_inputs(wl, seed=0, device=device)
    off = 1 if args.misalign else 0

    def shifted(t):
        if t is None or not off:
            return t
        buf = torch.empty(t.numel() + off, dtype=t.dtype, device=t.device)
        v = buf[off:].view(t.shape)
        v.copy_(t)
        return v

    x, r, w = shifted(x), shifted(r), shifted(w)
    y = shifted(torch.empty_like(x))
    h = None if r is None else shifted(torch.empty_like(x))
    plan = api.plan_for(x, w=w, residual=r, out=y, residual_out=h)
    if args.plan:
        # fields of another kernel family's plan over the library's (that
        # family on this workload; the library validates the result)
        for k, v in json.loads(args.plan).items():
            setattr(plan, k, v)
    if args.grid:
        plan.grid = args.grid
        plan.persistent = 1
    with torch.cuda.stream(stream):
        for _ in range(args.launches):
            api.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h, stream=stream, plan=plan)
    stream.synchronize()
    print(json.dumps({"ncu_case": wl.name, "rows": wl.rows, "hidden": wl.hidden,
                      "launches": args.launches, "bytes_per_launch": wl.algorithmic_bytes(),
                      "plan": plan_summary(plan)}))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from row_reduction_norm_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    # the rows a step may take: the first REF_POOL_ROWS rows of the workload
    # as drawn on the host (the whole batch when it is smaller)
    pool = min(wl.rows, REF_POOL_ROWS)
    x, r, w = W.make_inputs(wl, seed=0, device="cpu", rows=pool)
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    del x, r, w
    # size each step so that warmup + steps take about a minute of host time.
    # A step spread over a thread pool pays the pool's set-up: below 64 rows a
    # thread it runs on one thread, sized from the single-thread row rate.
    budget = 60.0 / max(1, args.steps + args.warmup)
    probe = min(pool, 256)
    t0 = time.perf_counter()
    oracle.rmsnorm(xn[:probe], w=wn, residual=None if rn is None else rn[:probe], eps=wl.eps, dtype=wl.dtype,
                   threads=1)
    t_row1 = max(time.perf_counter() - t0, 1e-9) / probe
    if budget / t_row1 >= 64 * threads:
        t0 = time.perf_counter()
        oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype=wl.dtype, threads=threads)
        t_full = max(time.perf_counter() - t0, 1e-6)
        rows_per_step = int(max(1, min(pool, pool * budget / t_full)))
    else:
        threads = 1
        rows_per_step = int(max(1, min(pool, budget / t_row1)))

    def step(i):
        lo = (i * rows_per_step) % pool
        hi = min(pool, lo + rows_per_step)
        oracle.rmsnorm(xn[lo:hi], w=wn, residual=None if rn is None else rn[lo:hi], eps=wl.eps,
                       dtype=wl.dtype, threads=threads)
        return hi - lo

    for i in range(args.warmup):
        step(i)
    rows_done = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        rows_done += step(i)
    dt = time.perf_counter() - t0
    row_bytes = wl.algorithmic_bytes(rows=1) - (wl.hidden * wl.elem_bytes if wl.has_w else 0)
    wbytes = wl.hidden * wl.elem_bytes if wl.has_w else 0
    value = (rows_done * row_bytes + args.steps * wbytes) / dt / 1e9
    sample = (f"{rows_per_step} of {wl.rows} rows per step ({rows_per_step * wl.hidden} elements, taken in "
              f"turn from the first {pool} rows), fp64 C oracle, " +
              (f"{threads} threads over row blocks" if threads > 1 else
               "one thread (steps too small for a thread pool to pay)"))
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "rows_per_s": round(rows_done / dt, 1),
        "config": bench_config(wl, world),
        "timing": "host wall clock around exactly `steps` steps of the fp64 C oracle on the host cores",
        "plan": None,
        "pdl": None,
        "rows_per_step": rows_per_step,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out))


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
