#!/usr/bin/env python3
"""Benchmark of the FP8-blk decode GEMV hot path on GB300.

Headline workload (the largest configuration): the vocab-head GEMV fused with
the greedy argmax, W 131072 x 4096 e4m3 codes with a 1024 x 32 grid of e8m0
block scales (decoded to f32 on the host), x f32 [1, 4096]; the call returns
one u32 token.  One step = one fp8blk_gemv_argmax call (one kernel launch).
Weights, scales and x are resident in HBM before the timed region; calls
rotate over enough weight copies that their total exceeds L2, so every call
streams its weights from HBM.

Timing: W untimed warm-up calls, then CUDA graphs of exactly K back-to-back
calls (K = --steps), replayed as repetitions -- at least five, and until a
minimum time has passed -- each bracketed by a barrier and a device
synchronize and timed with CUDA events on the launch stream.  The reported
time per step is the median over repetitions (max over ranks); clock samples
come from inside the repetitions' window.  The other workloads of the path
(the 4096 x 4096 and 512 x 1024 GEMVs, the m = 8 verify on the tensor-core and
CUDA-core kernels, the NVFP4 and MXFP4 experts) are timed the same way into
`workloads`.

Metric: algorithmic bytes (codes + f32 scales + activations + outputs) per
second, GB/s, and its fraction of the measured HBM peak; microseconds per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the plain CPU oracle on this host on bounded row
samples of the same workload (the only other place this script runs the oracle
is the cpu_baseline leg).  Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (weak scaling, no data-path collective);
rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8-blk decode GEMV weight GB/s (fraction of GB300 HBM peak); us per call"
HEADLINE = "head_argmax_131072x4096_m1"
HEADLINE_ARGMAX = True
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "fp8_block_scaled_fp8blk_gb300", "csrc")


# ---------------------------------------------------------------- byte counts
KERNEL_NAMES = {0: "stream_gemv_kernel<{m},e4m3,{a}> (team kernel)",
                1: "rowwarp_gemv_kernel<e4m3,{a}> (row-per-warp kernel)",
                2: "tc8_gemv_kernel<{a}> (tensor-core kernel)"}


def kernel_name(ops, m: int, rows: int, cols: int, argmax: bool = False) -> str:
    """The kernel the library's planner picks for this shape on this device."""
    import torch
    prop = torch.cuda.get_device_properties(torch.cuda.current_device())
    kind = ops.plan_query(m, rows, cols, 1, sms=prop.multi_processor_count)["kernel"]
    return KERNEL_NAMES[kind].format(m=m, a=str(argmax).lower())


def fp8blk_bytes(rows: int, cols: int, m: int, argmax: bool = False) -> int:
    """codes + f32 scale grid + activations + outputs (tokens for argmax)."""
    grid = math.ceil(rows / 128) * math.ceil(cols / 128) * 4
    out = m * 4 if argmax else m * rows * 4
    return rows * cols + grid + m * cols * 4 + out


def nvfp4_bytes(n_active: int, rows: int, cols: int) -> int:
    """Per active expert: e2m1 codes + e4m3 scales + f32 global scale; + x + y."""
    per = rows * cols // 2 + rows * cols // 16 + 4
    return n_active * per + cols * 4 + n_active * rows * 4


# Sources that define the streaming kernels and their launch geometry.
KERNEL_SOURCES = ("device_common.cuh", "stream_gemv.cuh", "rowwarp_gemv.cuh", "tc8_gemv.cuh", "nvfp4_gemv.cuh",
                  "fp4tc_gemv.cuh", "launch.h", "abi.cu", "gemv_e4m3.cu", "gemv_bf16.cu", "gemv_tc.cu",
                  "nvfp4_dequant.cu", "nvfp4_gemv.cu")


# The sources that decide each profiled workload's dominant kernel and its
# launch shape: a committed traffic figure stays valid while these hash the same.
_PLAN_SOURCES = ("device_common.cuh", "launch.h", "abi.cu")
TRAFFIC_SOURCES = {
    "head_argmax_131072x4096_m1": _PLAN_SOURCES + ("stream_gemv.cuh", "tc8_gemv.cuh", "gemv_tc.cu"),
    "verify_16384x4096_m8": _PLAN_SOURCES + ("stream_gemv.cuh", "tc8_gemv.cuh", "gemv_tc.cu"),
    "gemv_4096x4096_m1": _PLAN_SOURCES + ("stream_gemv.cuh", "gemv_e4m3.cu"),
    "nvfp4_experts_6of64_2048x4096": _PLAN_SOURCES + ("tc8_gemv.cuh", "nvfp4_gemv.cuh", "fp4tc_gemv.cuh",
                                                      "nvfp4_gemv.cu"),
    "nvfp4_experts_64of64_2048x4096": _PLAN_SOURCES + ("tc8_gemv.cuh", "nvfp4_gemv.cuh", "fp4tc_gemv.cuh",
                                                       "nvfp4_gemv.cu"),
    "mxfp4_experts_6of64_2048x4096": _PLAN_SOURCES + ("tc8_gemv.cuh", "nvfp4_gemv.cuh", "fp4tc_gemv.cuh",
                                                      "nvfp4_gemv.cu"),
    "mxfp4_experts_64of64_2048x4096": _PLAN_SOURCES + ("tc8_gemv.cuh", "nvfp4_gemv.cuh", "fp4tc_gemv.cuh",
                                                       "nvfp4_gemv.cu"),
}


def _code_only(text: str) -> str:
    """C++ source without // comments, trailing blanks and empty lines: what
    the compiler sees, so that editing a comment keeps a kernel's hash."""
    out = []
    for line in text.splitlines():
        in_str, cut = False, len(line)
        for i, ch in enumerate(line):
            if ch == '"' and (i == 0 or line[i - 1] != "\\"):
                in_str = not in_str
            elif not in_str and line.startswith("//", i):
                cut = i
                break
        code = line[:cut].rstrip()
        if code:
            out.append(code)
    return "\n".join(out)


def source_hash(names=KERNEL_SOURCES) -> str:
    """Hash of kernel sources (all of them by default), comments left out; a
    committed ncu traffic figure is reported only while its workload's sources
    match (i.e. while the kernel is the one profiled)."""
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:12]


def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s earlier GB300 copy measurement)"


def profiled_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    if workload not in TRAFFIC_SOURCES:
        return None
    cur = source_hash(TRAFFIC_SOURCES[workload])
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == cur:
                return int(parts[2])
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) around the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str | None):
        self.samples = []
        self.error = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True, bufsize=1)
        except Exception as e:  # nvidia-smi missing
            self.proc, self.error = None, str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.samples.append(dict(t=ts, sm=float(parts[1]), sm_max=float(parts[2]),
                                         power=float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                                         reasons={r: parts[5 + k] == "Active"
                                                  for k, r in enumerate(self.REASONS)}))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"error": self.error or "nvidia-smi unavailable"}
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            inside = sorted(self.samples, key=lambda s: abs(s["t"] - 0.5 * (t0 + t1)))[:2]
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return {"error": "no nvidia-smi samples"}
        reasons = sorted({r for s in inside for r, on in s["reasons"].items() if on})
        powers = [s["power"] for s in inside if s["power"] is not None]
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["sm_max"] for s in inside),
                "reasons": reasons, "samples": len(inside), "note": note,
                "power_w_max": max(powers) if powers else None}


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """Slowest rank's value (all ranks get it).  Timing only: not a data path."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    if dist.get_backend() == "gloo":
        device = "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(bytes_per_call: int, us_per_call_slowest: float, world: int) -> float:
    """Whole-job GB/s of `world` independent replicas, each doing the same calls,
    timed by the slowest rank."""
    return world * bytes_per_call / (us_per_call_slowest * 1e-6) / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- timing core
def time_reps(calls, steps: int, warmup: int, stream, world: int, device, min_reps: int = 5,
              min_seconds: float = 0.3, max_reps: int = 3000, per_graph: int = 1000) -> dict:
    """`warmup` eager calls, then CUDA graphs of exactly `steps` back-to-back
    calls on `stream`, replayed as repetitions: at least `min_reps`, and until
    `min_seconds` of wall time have passed.  Each repetition is bracketed by a
    barrier and a device synchronize and timed with CUDA events on `stream`.
    Returns the median / min / max milliseconds per repetition (each the max
    over ranks), the repetition count and the host window of the repetitions."""
    import torch
    n = len(calls)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            calls[i % n]()
    stream.synchronize()

    def capture(first, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(first, first + count):
                calls[i % n]()
        return g

    graphs, done = [], 0
    while done < steps:  # one repetition = these graphs in order = exactly `steps` calls
        k = min(per_graph, steps - done)
        graphs.append(capture(done, k))
        done += k
    with torch.cuda.stream(stream):  # warm the graphs themselves (untimed)
        for g in graphs:
            g.replay()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    ms = []
    t0 = time.time()
    while len(ms) < min_reps or (time.time() - t0 < min_seconds and len(ms) < max_reps):
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            for g in graphs:
                g.replay()
            end.record(stream)
        torch.cuda.synchronize()
        ms.append(start.elapsed_time(end))
    t1 = time.time()
    barrier(world)
    med = statistics.median(ms)
    return {"ms": max_over_ranks(med, world, device), "ms_min": max_over_ranks(min(ms), world, device),
            "ms_max": max_over_ranks(max(ms), world, device), "reps": len(ms), "window": (t0, t1)}


# ---------------------------------------------------------------- workloads
def up(a, device, dtype=None):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def copies_for(nbytes: int) -> int:
    return max(2, math.ceil(2.5 * L2_BYTES / nbytes))


def setup_fp8blk(name: str, device, argmax: bool = False):
    import torch
    from fp8_block_scaled_fp8blk_gb300 import ops, synth
    w = synth.WORKLOADS[name]
    rows, cols, m = w["rows"], w["cols"], w["m"]
    case = synth.workload_case(name)
    s = up(ops.fp8blk_scales_from_e8m0(case.scale_e8m0), device)
    w0 = up(case.codes, device)
    n = copies_for(rows * cols)
    ws_ = [w0] + [w0.clone() for _ in range(n - 1)]
    x = up(case.x, device)
    calls = []
    wsp = toks = None
    if argmax:
        wsp = [ops.argmax_workspace(m, rows, cols, device) for _ in range(n)]
        toks = [torch.empty(m, dtype=torch.int32, device=device) for _ in range(n)]
        for i in range(n):
            calls.append(lambda i=i: ops.fp8blk_gemv_argmax(ws_[i], s, x, wsp[i], tokens=toks[i]))
    else:
        ys = [torch.empty((m, rows), dtype=torch.float32, device=device) for _ in range(n)]
        for i in range(n):
            calls.append(lambda i=i: ops.fp8blk_gemv(ws_[i], s, x, y=ys[i]))
    return dict(case=case, calls=calls, copies=n, rows=rows, cols=cols, m=m, weights=ws_, scales=s,
                x=x, workspaces=wsp, argmax=argmax, launches=1, bytes=fp8blk_bytes(rows, cols, m, argmax))


def setup_nvfp4(device, fused: bool = True, n_active: int | None = None):
    """C5 with ten rotating active-expert sets (the 64-expert pool is 301 MB, so
    the active experts' bytes come from HBM).  fused: one launch per call
    (ids and global scales on the device); otherwise the dequant-to-scratch +
    bf16 GEMV arm, two launches per active expert.  n_active: another number
    of active experts drawn from the same pool (default: C5's six)."""
    import numpy as np
    import torch
    from fp8_block_scaled_fp8blk_gb300 import ops, synth
    w = synth.NVFP4_WORKLOAD
    c = synth.nvfp4_case(w["n_experts"], w["rows"], w["cols"], w["n_active"], w["seed"])
    codes, scales, x = up(c.codes, device), up(c.scales, device), up(c.x, device)
    rows, cols = w["rows"], w["cols"]
    act = w["n_active"] if n_active is None else n_active
    rng = np.random.default_rng(w["seed"] + 100)
    id_sets = ([c.ids] if act == w["n_active"] else []) + [
        rng.choice(w["n_experts"], act, replace=False).astype(np.int32) for _ in range(9 if act == w["n_active"] else 10)]
    ys = [torch.empty((act, rows), dtype=torch.float32, device=device) for _ in id_sets]
    if fused:
        g_dev = up(c.gscale, device)
        ids_dev = [up(np.asarray(i, dtype=np.int32), device) for i in id_sets]
        calls = [lambda i=i: ops.nvfp4_expert_gemv(codes, scales, g_dev, ids_dev[i], x, y=ys[i])
                 for i in range(len(id_sets))]
        launches = 1
    else:
        scratch = torch.empty((rows, cols), dtype=torch.int16, device=device)
        calls = [lambda i=i: ops.nvfp4_expert_dequant_gemv(codes, scales, c.gscale, id_sets[i], x,
                                                           scratch, y=ys[i]) for i in range(len(id_sets))]
        launches = 2 * act
    return dict(calls=calls, bytes=nvfp4_bytes(act, rows, cols), launches=launches)


def mxfp4_bytes(n_active: int, rows: int, cols: int) -> int:
    """Algorithmic bytes of one MXFP4 expert call: codes + e8m0 scales of the
    active experts, x, y."""
    return n_active * (rows * cols // 2 + rows * cols // 32) + 4 * cols + 4 * n_active * rows


def setup_mxfp4(device, n_active: int | None = None):
    """The MTP block's OCP MXFP4 experts, C5 geometry, ten rotating active sets
    (of C5's six experts, or of `n_active`)."""
    import numpy as np
    import torch
    from fp8_block_scaled_fp8blk_gb300 import ops, synth
    w = synth.MXFP4_WORKLOAD
    c = synth.mxfp4_case(w["n_experts"], w["rows"], w["cols"], w["n_active"], w["seed"])
    codes, scales, x = up(c.codes, device), up(c.scales, device), up(c.x, device)
    act = w["n_active"] if n_active is None else n_active
    rng = np.random.default_rng(w["seed"] + 100)
    id_sets = ([c.ids] if act == w["n_active"] else []) + [
        rng.choice(w["n_experts"], act, replace=False).astype(np.int32) for _ in range(9)]
    ids_dev = [up(np.asarray(i, dtype=np.int32), device) for i in id_sets]
    ys = [torch.empty((act, w["rows"]), dtype=torch.float32, device=device) for _ in id_sets]
    calls = [lambda i=i: ops.mxfp4_expert_gemv(codes, scales, ids_dev[i], x, y=ys[i]) for i in range(len(id_sets))]
    return dict(calls=calls, bytes=mxfp4_bytes(act, w["rows"], w["cols"]), launches=1)


def summarize(st: dict, r: dict, steps: int, peak: float, sampler, **extra) -> dict:
    """One workload's entry: median us per call and its GB/s over the repetitions."""
    us = r["ms"] * 1e3 / steps
    gbs = st["bytes"] / (us * 1e-6) / 1e9
    out = {"us_per_call": round(us, 3), "gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
           "bytes_per_call": st["bytes"], "steps": steps, "repetitions": r["reps"],
           "us_per_call_min_max": [round(r["ms_min"] * 1e3 / steps, 3), round(r["ms_max"] * 1e3 / steps, 3)],
           "launches_per_call": st.get("launches", 1)}
    if sampler is not None:
        out["clocks"] = sampler.summary(*r["window"])
    out.update(extra)
    return out


def with_traffic(out: dict) -> dict:
    """Add each entry's committed ncu DRAM bytes per launch (while current).
    A `_tensor_core` entry takes its workload's figure: the tensor-core kernel
    is the by-shape default, and so the captured launch, of those workloads."""
    for name, entry in out.items():
        t = profiled_traffic(name)
        if t is None and name.endswith("_tensor_core"):
            t = profiled_traffic(name[: -len("_tensor_core")])
        if t is not None:
            entry["ncu_dram_bytes_per_launch"] = t
    return out


def measure_extra(device, stream, world, peak, steps, warmup, sampler):
    """The other workloads of the path, timed the same way (one JSON line)."""
    from fp8_block_scaled_fp8blk_gb300 import ops
    out = {}
    for name in ("gemv_512x1024_m1", "gemv_4096x4096_m1"):
        st = setup_fp8blk(name, device)
        r = time_reps(st["calls"], steps, warmup, stream, world, device)
        out[name] = summarize(st, r, steps, peak, sampler, weight_copies=st["copies"],
                              kernel=kernel_name(ops, st["m"], st["rows"], st["cols"]))
        del st
    # The vocab head on the CUDA cores (row-per-warp kernel), beside the
    # headline's tensor-core figure.
    st = setup_fp8blk(HEADLINE, device, HEADLINE_ARGMAX)
    ops.set_m1_kernel(1, 0)
    r = time_reps(st["calls"], steps, warmup, stream, world, device)
    out[HEADLINE + "_cuda_core"] = summarize(st, r, steps, peak, sampler, weight_copies=st["copies"],
                                             kernel=kernel_name(ops, st["m"], st["rows"], st["cols"], True))
    ops.set_m1_kernel(0, 0)
    del st
    # The m = 8 verify on both kernels: the tensor-core kernel (the library's
    # default for m >= 5 from 24 MiB of weights) and the CUDA-core team kernel.
    name = "verify_16384x4096_m8"
    st = setup_fp8blk(name, device)
    for arm, min_m in (("tensor_core", 0), ("cuda_core", 9)):
        ops.set_tensor_core_min_m(min_m, 0)
        r = time_reps(st["calls"], steps, warmup, stream, world, device)
        key = name if arm == "tensor_core" else name + "_cuda_core"
        out[key] = summarize(st, r, steps, peak, sampler, weight_copies=st["copies"],
                             kernel=kernel_name(ops, st["m"], st["rows"], st["cols"]))
    ops.set_tensor_core_min_m(0, 0)
    del st
    for fused, name, note in (
            (True, "nvfp4_experts_6of64_2048x4096",
             "one launch, the by-shape default (tensor cores here): e2m1 codes fed to tcgen05 kind::f8f6f4 "
             "as stored, expert ids and global scales on the device"),
            (False, "nvfp4_experts_6of64_2048x4096_two_step",
             "dequant to the reused bf16 scratch + bf16 GEMV per expert; algorithmic bytes exclude "
             "the 2 x 16 MiB scratch write+read per expert")):
        st = setup_nvfp4(device, fused)
        r = time_reps(st["calls"], steps, warmup, stream, world, device)
        out[name] = summarize(st, r, steps, peak, sampler, note=note)
        del st
    # The one-launch NVFP4 GEMV on both kernels, with C5's six and with all 64
    # experts active (the tensor-core kernel is the by-shape default from
    # 12288 active rows on, so for both).
    for act, name in ((6, "nvfp4_experts_6of64_2048x4096"), (64, "nvfp4_experts_64of64_2048x4096")):
        st = setup_nvfp4(device, True, act)
        for k, arm in ((2, "_tensor_core"), (1, "_cuda_core")):
            if act == 6 and k == 2:
                continue  # the default line above
            ops.set_fp4_kernel(k)
            r = time_reps(st["calls"], steps, warmup, stream, world, device)
            out[name + arm] = summarize(
                st, r, steps, peak, sampler,
                note="one launch on the tensor cores: e2m1 codes fed to tcgen05 kind::f8f6f4 as stored"
                if k == 2 else "one launch on the CUDA cores: NVFP4 decoded in registers")
        ops.set_fp4_kernel(0)
        del st
    # The MTP block's OCP MXFP4 experts (e8m0 per 32 columns), the same two
    # kernels and by-shape routing.
    st = setup_mxfp4(device)
    r = time_reps(st["calls"], steps, warmup, stream, world, device)
    out["mxfp4_experts_6of64_2048x4096"] = summarize(
        st, r, steps, peak, sampler,
        note="the MTP block's OCP MXFP4 experts: one launch, the by-shape default (tensor cores here)")
    for act, name in ((6, "mxfp4_experts_6of64_2048x4096"), (64, "mxfp4_experts_64of64_2048x4096")):
        if act != 6:
            st = setup_mxfp4(device, act)
        for k, arm in ((2, "_tensor_core"), (1, "_cuda_core")):
            if act == 6 and k == 2:
                continue  # the default line above
            ops.set_fp4_kernel(k)
            r = time_reps(st["calls"], steps, warmup, stream, world, device)
            out[name + arm] = summarize(
                st, r, steps, peak, sampler,
                note="one launch on the tensor cores: e2m1 codes fed to tcgen05 kind::f8f6f4 as stored"
                if k == 2 else "one launch on the CUDA cores: MXFP4 decoded in registers")
        ops.set_fp4_kernel(0)
        del st
    return with_traffic(out)


def measure_e2e(st, steps: int, device, min_seconds: float = 0.5) -> dict:
    """Same metric through the public API with host buffers: per step, copy x
    from pinned host memory, run the call, read its result (the u32 token for
    the argmax, y otherwise) back into pinned memory, synchronize."""
    import torch
    from fp8_block_scaled_fp8blk_gb300 import ops
    case = st["case"]
    x_h = torch.from_numpy(case.x.copy()).pin_memory()
    x_d = torch.empty_like(x_h, device=device)
    s = st["scales"]
    n = len(st["weights"])
    stream = torch.cuda.current_stream(device)
    if st["argmax"]:
        out_d = torch.empty(st["m"], dtype=torch.int32, device=device)
        wsp = st["workspaces"]

        def run(i):
            ops.fp8blk_gemv_argmax(st["weights"][i % n], s, x_d, wsp[i % n], tokens=out_d)
    else:
        out_d = torch.empty((st["m"], st["rows"]), dtype=torch.float32, device=device)

        def run(i):
            ops.fp8blk_gemv(st["weights"][i % n], s, x_d, y=out_d)
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()

    def one(i):
        x_d.copy_(x_h, non_blocking=True)
        run(i)
        out_h.copy_(out_d, non_blocking=True)
        stream.synchronize()

    def timed(step) -> tuple[float, int]:
        for i in range(10):
            step(i)
        k, t0 = 0, time.perf_counter()
        while k < max(steps, 5) or time.perf_counter() - t0 < min_seconds:
            step(k)
            k += 1
        return (time.perf_counter() - t0) / k, k

    dt_call, k_call = timed(one)
    # The same step recorded once per weight copy as a CUDA graph (the copy in,
    # the library call, the copy out), replayed and synchronized every step:
    # what a serving loop that captures its decode step pays.
    graphs = []
    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        for i in range(n):  # warm the library's per-shape host caches before capture
            run(i)
    cap.synchronize()
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            x_d.copy_(x_h, non_blocking=True)
            run(i)
            out_h.copy_(out_d, non_blocking=True)
        graphs.append(g)

    def one_graph(i):
        graphs[i % n].replay()
        stream.synchronize()

    dt, k = timed(one_graph)
    return {"value": round(st["bytes"] / dt / 1e9, 2), "unit": "GB/s", "us_per_call": round(dt * 1e6, 3),
            "steps": k, "h2d_bytes_per_step": x_h.numel() * 4,
            "d2h_bytes_per_step": out_h.numel() * out_h.element_size(),
            "path": "public binding, host buffers: per step one CUDA graph replay of (pinned x -> device, "
                    "one library call, result -> pinned host), then a stream sync",
            "per_call": {"value": round(st["bytes"] / dt_call / 1e9, 2), "us_per_call": round(dt_call * 1e6, 3),
                         "steps": k_call,
                         "path": "the same step issued call by call from Python (copy in, call, copy out, "
                                 "stream sync)"}}


def oracle_rate(name: str, argmax: bool, nthreads: int, budget_s: float, rows_per_call: int) -> dict:
    """The oracle, as it stands, on `nthreads` host threads: calls on the
    first `rows_per_call` rows of the workload (its argmax too, for the head)
    for about budget_s seconds; GB/s of the sampled rows' algorithmic bytes."""
    import oracle
    from fp8_block_scaled_fp8blk_gb300 import synth
    w = synth.WORKLOADS[name]
    case = synth.workload_case(name)
    oracle.build()
    r = min(rows_per_call, w["rows"])
    codes, grid = case.codes[:r], case.scale_e8m0[:math.ceil(r / 128)]
    t0 = time.perf_counter()
    n = 0
    while True:
        y, _ = oracle.fp8blk_gemv(codes, grid, case.x, nthreads=nthreads)
        if argmax:
            for i in range(w["m"]):
                oracle.argmax(y[i])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    nbytes = fp8blk_bytes(r, w["cols"], w["m"], argmax)
    return {"value": round(nbytes * n / el / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "sample": f"{n} calls on rows 0..{r - 1} of {w['rows']}x{w['cols']} m={w['m']}"
                      f"{' (+argmax)' if argmax else ''} in {el:.1f} s"}


def cpu_baseline(name: str, argmax: bool) -> dict:
    """The oracle timed on one host thread and on every host core."""
    cores = os.cpu_count() or 1
    one = oracle_rate(name, argmax, 1, 6.0, 2048)
    allc = oracle_rate(name, argmax, cores, 6.0, 16384)
    return {"value": allc["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": allc["sample"] + f"; double-precision oracle on {cores} threads",
            "single_thread": {"value": one["value"], "unit": "GB/s", "cores": 1, "sample": one["sample"]}}


# ---------------------------------------------------------------- arms
def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from fp8_block_scaled_fp8blk_gb300 import ops
    ops.set_tensor_core_min_m(args.tensor_core_min_m, args.tensor_core_min_bytes)
    peak, peak_src = hbm_peak()
    stream = torch.cuda.Stream(device)
    st = setup_fp8blk(HEADLINE, device, HEADLINE_ARGMAX)
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3)
    r = time_reps(st["calls"], args.steps, args.warmup, stream, world, device, min_seconds=1.0)
    clocks = sampler.summary(*r["window"]) if sampler else None
    ms = r["ms"]
    us = ms * 1e3 / args.steps
    per_gpu_gbs = st["bytes"] / (us * 1e-6) / 1e9
    value = replica_throughput(st["bytes"], us, world)
    status = ops.fp8blk_device_status()
    e2e = measure_e2e(st, args.steps, device)
    e2e["value"] = round(e2e["value"] * world, 2) if world > 1 else e2e["value"]
    del st
    extra = None
    if world == 1 and not args.no_extra:
        extra = measure_extra(device, stream, world, peak, args.steps, args.warmup, sampler)
    if sampler:
        sampler.stop()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(HEADLINE, HEADLINE_ARGMAX)
    if rank == 0:
        w = __import__("fp8_block_scaled_fp8blk_gb300.synth", fromlist=["WORKLOADS"]).WORKLOADS[HEADLINE]
        nbytes = fp8blk_bytes(w["rows"], w["cols"], w["m"], HEADLINE_ARGMAX)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
            "us_per_call": round(us, 4), "frac_of_hbm_peak": round(per_gpu_gbs / peak, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy: e4m3 codes uniform over finite codes, e8m0 2^[-8,0], x N(0,1))",
            "config": {"workload": HEADLINE, "rows": w["rows"], "cols": w["cols"], "m": w["m"],
                       "output": "one u32 greedy token per activation row (fused argmax), no logits",
                       "weights": "e4m3 codes + 128x128 f32 block scales (from e8m0)",
                       "bytes_per_call": nbytes,
                       "l2": "inputs larger than L2: rotating weight copies "
                             f"({copies_for(w['rows'] * w['cols'])} x {w['rows'] * w['cols'] / 2**20:.0f} MiB)",
                       "timing": f"median over {r['reps']} repetitions of exactly {args.steps} back-to-back "
                                 "calls (CUDA graphs), CUDA events on the launch stream, barrier + device "
                                 "synchronize around each repetition",
                       "parallelism": f"replicas x{world}"},
            "repetitions": r["reps"],
            "us_per_call_min_max": [round(r["ms_min"] * 1e3 / args.steps, 4), round(r["ms_max"] * 1e3 / args.steps, 4)],
            "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(per_gpu_gbs / peak, 4), "traffic": profiled_traffic(HEADLINE),
                         "peak_source": peak_src,
                         "kernel": kernel_name(ops, w["m"], w["rows"], w["cols"], HEADLINE_ARGMAX),
                         "algorithmic_bytes_per_launch": nbytes},
            "e2e": e2e,
            "gpu_launches": args.steps,
            "gpu_launches_note": f"one kernel launch per step; {args.steps} per repetition, "
                                 f"{args.steps * r['reps']} over all repetitions",
            "clocks": clocks,
            "device_status": status,
            "kernel_source_hash": source_hash(),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if extra is not None:
            line["workloads"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle on this host's cores, K steps of a bounded row sample each."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    from fp8_block_scaled_fp8blk_gb300 import synth
    w = synth.WORKLOADS[HEADLINE]
    rows, cols, m = w["rows"], w["cols"], w["m"]
    case = synth.workload_case(HEADLINE)
    cores = os.cpu_count() or 1
    oracle.build()
    t0 = time.perf_counter()
    oracle.fp8blk_gemv(case.codes[:1024], case.scale_e8m0[:8], case.x, nthreads=cores)
    per_row = (time.perf_counter() - t0) / 1024
    budget = 90.0 / max(1, args.steps + args.warmup)
    sample_rows = int(min(rows, max(128, budget / max(per_row, 1e-9))))
    sample_rows -= sample_rows % 128

    def step(i):
        r0 = (i * sample_rows) % rows
        r0 -= r0 % 128
        r1 = min(rows, r0 + sample_rows)
        y, _ = oracle.fp8blk_gemv(case.codes[r0:r1], case.scale_e8m0[r0 // 128:math.ceil(r1 / 128)], case.x,
                                  nthreads=cores)
        oracle.argmax(y[0])
        return r1 - r0

    for i in range(args.warmup):
        step(i)
    done = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        done += step(i)
    el = time.perf_counter() - t0
    per_step_rows = done / args.steps
    nbytes = per_step_rows * cols + math.ceil(per_step_rows / 128) * math.ceil(cols / 128) * 4 \
        + m * cols * 4 + m * 4
    value = nbytes * args.steps / el / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy, same generator as the GPU arm)",
        "config": {"workload": HEADLINE, "rows": rows, "cols": cols, "m": m,
                   "sample_rows_per_step": sample_rows},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample_rows} of {rows} rows (+ their argmax) per step, {args.steps} steps"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_workload(args):
    """Just `--calls` calls of one named workload, for an ncu capture."""
    import torch
    from fp8_block_scaled_fp8blk_gb300 import ops
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    ops.set_tensor_core_min_m(args.tensor_core_min_m, args.tensor_core_min_bytes)
    ops.set_fp4_kernel(args.fp4_kernel)
    if args.profile_workload == "mxfp4_experts_6of64_2048x4096":
        st = setup_mxfp4(device)
    elif args.profile_workload.startswith("nvfp4_experts_6of64_2048x4096"):
        st = setup_nvfp4(device, fused=not args.profile_workload.endswith("_two_step"))
    elif args.profile_workload == "nvfp4_experts_64of64_2048x4096":
        st = setup_nvfp4(device, True, 64)
    elif args.profile_workload == "mxfp4_experts_64of64_2048x4096":
        st = setup_mxfp4(device, 64)
    else:
        st = setup_fp8blk(args.profile_workload, device, args.profile_workload.startswith("head_argmax"))
    for i in range(args.calls):
        st["calls"][i % len(st["calls"])]()
    torch.cuda.synchronize()
    print(json.dumps({"profile_workload": args.profile_workload, "calls": args.calls,
                      "device_status": ops.fp8blk_device_status()}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200, help="calls per timed repetition")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-workload", default=None,
                    help="run --calls calls of this workload and exit (for ncu captures)")
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--fp4-kernel", type=int, default=0, choices=(0, 1, 2),
                    help="with --profile-workload: FP4 expert kernel (0 by shape, 1 CUDA cores, 2 tensor cores)")
    ap.add_argument("--tensor-core-min-m", type=int, default=0,
                    help="e4m3 GEMVs with m >= this use the tensor-core kernel (9 = never, 0 = library default)")
    ap.add_argument("--tensor-core-min-bytes", type=int, default=0,
                    help="... when the weights are at least this many bytes (1 = any, 0 = library default)")
    args = ap.parse_args()
    if args.profile_workload:
        run_profile_workload(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
