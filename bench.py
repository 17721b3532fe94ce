"""Benchmark of the LatentIndex decode indexer step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one decode step of the whole hot path for a 4-layer group over a
batch of sequences: absorb the queries into the decoders (eq. 6), score the
shared latent cache for all 4 layers in one pass (eq. 8), and take each
layer's top-k.  The default workload is the batched 32K-context decode with
an fp8 latent cache (32 sequences x 32,768 tokens, H=64, d=128, r=192,
k=2048).  In the same run the bench also times, on the same batch, the
hierarchical-selection variant (HS) and four native per-layer DSA indexer
scans with their top-k (the baseline LatentIndex replaces), and reports them
under "hs" and "native_x4".

Timing: W warm-up steps, then K timed steps; before every step, outside the
timed events, a 256 MiB buffer is read so that nothing of the step's inputs
is left in the L2 (126 MB).  Reading (not writing) that buffer leaves no dirty
lines behind, so the step does not pay for writing back someone else's data;
the step's inputs (205 MB of latent cache) are larger than the L2 as well.  Each
step is bracketed by CUDA events on the launching stream and the per-step
device times are summed; the max over ranks is taken.  `value` is the
algorithmic HBM bytes of the step (latent + scales + queries + decoders +
head weights + selected indices) per second.  `e2e` measures the same step
through the C ABI with host buffers: the step's new queries and head weights
are copied from pinned host memory and the selected indices copied back
inside the timed region (the latent cache is device-resident state).

With --impl reference the CPU oracle (fp64) is timed instead on a bounded
sample of the same workload.  Under torchrun each rank runs its own batch
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode indexer latency & HBM GB/s per 4-layer group at 8K-128K ctx"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="fp8_32k_b32")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-side", action="store_true", help="skip the HS / native side timings")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config records")
    ap.add_argument("--cpu-sample-seconds", type=float, default=12.0)
    ap.add_argument("--shape", default="",
                    help="override fields of the workload, e.g. T=256,pos0=130816 (a reduced case for "
                         "profiling; recorded in config.shape_overrides)")
    return ap.parse_args()


def shape_overrides(text):
    """'T=256,pos0=130816' -> {'T': 256, 'pos0': 130816} (integer fields only)."""
    out = {}
    for item in filter(None, (t.strip() for t in text.split(","))):
        key, val = item.split("=", 1)
        out[key.strip()] = int(val)
    return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device="cpu") -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if ws <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_step: int, ws: int, ms_per_step: float) -> float:
    """GB/s of the whole job: every rank's replica steps a batch of its own
    (weak scaling), so the bytes of all ranks over the slowest rank's time."""
    return bytes_per_step * ws / (ms_per_step * 1e-3) / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def step_bytes(w) -> dict:
    """Algorithmic bytes of one decode step (each tensor touched once)."""
    esz = {"f32": 4, "bf16": 2, "fp8": 1}[w.lat_dtype]
    qsz = {"f32": 4, "bf16": 2}[w.q_dtype]
    toks = w.B * w.L
    b = {
        "latent": toks * w.r * esz,
        "lat_scale": toks * 4 if w.lat_dtype == "fp8" else 0,
        "q": w.B * w.T * w.G * w.H * w.d * qsz,
        "D": w.G * w.r * w.d * qsz,
        "w": w.B * w.T * w.G * w.H * 4,
        "idx": w.B * w.T * w.G * w.k * 4,
    }
    b["total"] = sum(b.values())
    return b


def scan_bytes(w) -> int:
    """Algorithmic bytes of one group-scan launch: the latent (and its fp8 row
    scales) read once, the absorbed queries (stored in the latent's type) and
    the head weights; scores are the launch's output and are not counted."""
    esz = {"f32": 4, "bf16": 2, "fp8": 1}[w.lat_dtype]
    return (w.B * w.L * (w.r * esz + (4 if w.lat_dtype == "fp8" else 0)) +
            w.B * w.T * w.G * w.H * w.r * esz + w.B * w.T * w.G * w.H * 4)


def scan_flops(w, q_pos=None) -> int:
    """2 * G * H * r flops per (query, visible token) pair."""
    if q_pos is not None:
        pairs = w.B * sum(min(int(t) + 1, w.L) for t in q_pos)
    else:
        pairs = w.B * w.T * w.L
    return 2 * pairs * w.G * w.H * w.r


def source_hash(paths) -> str:
    """Hash of the code of `paths` with comments and blank space removed, so
    that only a change that can change the compiled kernel changes it."""
    import re
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


SCAN_SOURCES = ["shared_latent_key_cache_b300/csrc/score_tc.cu", "shared_latent_key_cache_b300/csrc/ptx.cuh",
                "shared_latent_key_cache_b300/csrc/li_internal.cuh"]


def ncu_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the scan kernel for this
    workload, from profiles/scan_dram_traffic.json (written from an ncu
    capture), if that capture was taken on the current kernel sources; else
    None."""
    p = os.path.join(ROOT, "profiles", "scan_dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("kernel_sources_sha256_16") != source_hash(SCAN_SOURCES):
        return None
    return int(rec["dram_bytes_per_launch"])


def spin_up(flush, dev, seconds: float = 0.25):
    """Keeps the GPU busy (L2-evicting reads) for `seconds` of wall time before
    a timed block that follows host-side set-up (the breakdown, the per-config
    records, the side timings).  After an idle spell of 0.2 s or more the GPU
    ran the next few milliseconds of work at about half speed (the reported
    clocks unchanged); 0.2 s of work first restored the full rate.  The
    contract's timed steps and the end-to-end leg follow their own warm-up
    steps instead."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(16):
            flush()
        torch.cuda.synchronize(dev)


class L2Flush:
    """Evicts the L2 by reading a buffer twice its size (a sum over it)."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.sum()


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, read through NVML
    (the library nvidia-smi itself uses), only ever reading settings.

    Every NVML query briefly stalls the GPU's work (measured here: 0.3-3 ms per
    query, which would inflate a ~30 ms timed region by several percent), so
    the timed loop takes as few samples as the timing rules allow: one per
    ~1000 steps and at least one, each taken while the GPU is still executing
    the steps the host has already enqueued."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.samples = []
        self.max_mhz = None
        self.h = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            self.h = h
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
                self.max_mhz = float(mx.value)
        except OSError:
            self.h = None

    def sample(self):
        if self.h is None:
            return
        import ctypes
        clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        ok = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        if ok:
            self.samples.append((float(clk.value), int(rs.value), pw.value / 1000.0))

    def summary(self):
        if self.h is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"]}
        reasons = sorted({name for _, r, _ in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "power_w_max": max(w for _, _, w in self.samples), "source": "NVML, during the timed steps"}


# ------------------------------------------------------------------ reference

CPU_SAMPLE = {  # name -> (unit of work timed on the host, how many at most)
    "tiny_f32": ("sequence", 1),
    "dsa_bf16_8k": ("sequence", 1),
    "fp8_32k_b32": ("sequence", 32),
    "fp8_128k_hs": ("sequence", 3),
    "prefill_bf16_128k": ("query", 6),
}


def cpu_oracle_rate(w, seed: int, budget_s: float, max_units: int | None = None):
    """Time the fp64 CPU oracle (absorb + score + TopK) on whole sequences of a
    decode workload, or on single query positions of a prefill workload, until
    about `budget_s` seconds of work or `max_units` units; returns the
    record's fields, the full step's time extrapolated from the sample when
    the sample is smaller than the step."""
    import numpy as np
    import torch

    import li_inputs
    import oracle

    oracle.build()
    cores = oracle.default_threads()
    unit, cap = CPU_SAMPLE.get(w.name, ("sequence", w.B))
    cap = cap if max_units is None else max_units
    total_units = w.B if unit == "sequence" else w.B * w.T
    cap = min(cap, total_units)
    elapsed, n = 0.0, 0
    qpos_all = None
    if unit == "query":
        # evenly spread query positions, first and last included
        qpos_all = [w.pos0 + round(i * (w.T - 1) / max(1, cap - 1)) for i in range(cap)]
    while n < cap and (n == 0 or elapsed < budget_s):
        if unit == "sequence":
            one = dataclasses.replace(w, B=1, native=False)
            x = li_inputs.make_workload(one, seed=seed + 1000 + n)
        else:
            one = dataclasses.replace(w, B=1, T=1, native=False, pos0=qpos_all[n])
            x = li_inputs.make_workload(one, seed=seed + 1000)
        t0 = time.perf_counter()
        qabs = oracle.absorb(x["q"], x["D"])
        u = oracle.score(x["latent"], x["lat_scale"], qabs, x["w"], q_pos=x["q_pos"])
        vl = None
        if x["q_pos"] is not None:
            vl = np.full(one.G, int(x["q_pos"][0]) + 1, dtype=np.int32)
        oracle.topk(u.reshape(-1, one.L), one.k, valid_len=vl)
        elapsed += time.perf_counter() - t0
        n += 1
        del x, qabs, u
    step_s = elapsed / n * total_units
    gbs = step_bytes(w)["total"] / step_s / 1e9
    extrap = n < total_units
    what = (f"{n} of {w.B} sequences of {w.name}" if unit == "sequence" else
            f"{n} of {w.T} query positions of {w.name} (spread over {w.pos0}..{w.pos0 + w.T - 1})")
    sample = what + f", fp64, {elapsed:.1f} s" + (", full step extrapolated from the sample" if extrap else "")
    rec = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
           "step_ms": step_s * 1e3, "extrapolated": extrap, "seconds": elapsed}
    if w.T > 1:
        q_pos = list(range(w.pos0, w.pos0 + w.T))
        rec["tflops"] = scan_flops(w, q_pos) / step_s / 1e12
    return rec


def run_reference(a, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    t0 = time.perf_counter()
    steps = []
    for i in range(max(1, a.steps if a.steps <= 3 else 1)):
        steps.append(cpu_oracle_rate(w, a.seed + i, a.cpu_sample_seconds))
    cb = steps[-1]
    ms = cb["step_ms"]
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s",
        "n_gpus": a.gpus, "steps": len(steps), "warmup": 0, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "L": w.L, "G": w.G, "H": w.H,
                                        "d": w.d, "r": w.r, "k": w.k, "T": w.T},
        "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ ours

PER_CONFIG = ["tiny_f32", "dsa_bf16_8k", "fp8_32k_b32", "fp8_128k_hs", "prefill_bf16_128k"]
NATIVE_SIDE = {"dsa_bf16_8k", "fp8_32k_b32", "fp8_128k_hs"}     # configs timed against 4 native scans


def _chk(li, st, what):
    if st != 0:
        raise RuntimeError(f"{what}: {li.li_status_string(st)}")


class Step:
    """Device buffers and the three launches of one step of a workload:
    absorb (eq. 6), group score (eq. 8), per-layer top-k."""

    def __init__(self, li, w, x, dev):
        import torch
        self.li, self.w, self.x = li, w, x
        B, T, G, H, r, L, k = w.B, w.T, w.G, w.H, w.r, w.L, w.k
        self.absd = {"f32": "f32", "bf16": "bf16", "fp8": "fp8"}[w.lat_dtype]
        self.q_abs = torch.empty(B, T, G, H, r, dtype={"f32": torch.float32, "bf16": torch.bfloat16,
                                                       "fp8": torch.uint8}[self.absd], device=dev)
        self.q_scale = torch.empty(B, T, G, H, dtype=torch.float32, device=dev) if self.absd == "fp8" else None
        self.scores = torch.empty(B, T, G, L, dtype=torch.float32, device=dev)
        self.idx = torch.empty(B, T, G, k, dtype=torch.int32, device=dev)
        self.vl = None
        if x["q_pos"] is not None:
            self.vl = (x["q_pos"] + 1).repeat_interleave(G).repeat(B).contiguous()
        n = li.li_topk_workspace_size(B * T * G, L, k)
        self.tws = torch.empty(n, dtype=torch.uint8, device=dev) if n > 0 else None
        self.launches = 4 if self.tws is not None else 3

    def __call__(self, stream, ev=None):
        li, x = self.li, self.x
        if ev is not None:
            ev[0].record(stream)
        _chk(li, li.li_absorb_queries(x["q"], x["D"], self.q_abs, self.q_scale, stream), "absorb")
        if ev is not None:
            ev[1].record(stream)
        _chk(li, li.li_score_group(x["latent"], x["lat_scale"], self.q_abs, self.q_scale, x["w"],
                                   self.scores, q_pos=x["q_pos"], stream=stream), "score")
        if ev is not None:
            ev[2].record(stream)
        _chk(li, li.li_topk(self.scores, self.w.k, self.idx, None, self.vl, self.tws, stream), "topk")
        if ev is not None:
            ev[3].record(stream)


def time_steps(step, n, flush, stream, dev, clk=None):
    """n steps, L2 evicted before each (outside the events); per-step device ms
    between events at the step's boundaries only (no event between kernels,
    which would end their programmatic launch overlap)."""
    import torch
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    nsamp = max(1, min(8, n // 1000))
    sample_at = {int((j + 0.5) * n / nsamp) for j in range(nsamp)} if clk is not None else set()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for i in range(n):
        flush()
        ev0[i].record(stream)
        step(stream)
        ev1[i].record(stream)
        if i in sample_at:
            clk.sample()          # the GPU is still running the steps enqueued so far
    torch.cuda.synchronize(dev)
    return [ev0[i].elapsed_time(ev1[i]) for i in range(n)], time.perf_counter() - t_wall


def breakdown(step, n, flush, stream, dev):
    """Median device us of absorb / score / top-k over n steps with events
    between the kernels."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for i in range(n):
        flush()
        step(stream, evs[i])
    torch.cuda.synchronize(dev)
    per = [[e[j].elapsed_time(e[j + 1]) * 1e3 for j in range(3)] for e in evs]
    return {name: statistics.median(p[j] for p in per) for j, name in enumerate(("absorb", "score", "topk"))}


def scored_positions(w, q_pos=None) -> int:
    """Positions scored per step, summed over (sequence, query, layer)."""
    if q_pos is not None:
        return w.B * w.G * sum(min(int(t) + 1, w.L) for t in q_pos)
    return w.B * w.T * w.G * w.L


def roofline(w, score_us, q_pos, pk, kernel_note=""):
    """The group scan's roofline: HBM for decode (algorithmic bytes per launch),
    the tensor pipe for prefill-shaped scoring (flops of the causal pairs)."""
    sbytes = scan_bytes(w)
    sflops = scan_flops(w, q_pos)
    if w.T > 1:
        achieved = sflops / (score_us * 1e-6) / 1e12
        peak = pk["bf16_tflops_sustained"] or pk["bf16_tflops"]
        return {"kernel": "score_tc_kernel (causal prefill scoring)" + kernel_note, "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": ncu_traffic(w.name), "peak_source": pk["source"] + " cuBLAS bf16, sustained",
                "algorithmic_bytes_per_launch": sbytes, "flops_per_launch": sflops}
    achieved = sbytes / (score_us * 1e-6) / 1e9
    kern = "score_simt_kernel (group scan, fp32)" if w.lat_dtype == "f32" else "score_tc_kernel (group scan)"
    return {"kernel": kern + kernel_note, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": ncu_traffic(w.name),
            "peak_source": pk["source"] + " copy bandwidth",
            "algorithmic_bytes_per_launch": sbytes, "flops_per_launch": sflops}


def config_record(a, name, li, dev, stream, flush, cpu=True):
    """One config's numbers: step latency, tokens scored per second, GB/s (and
    TFLOP/s for prefill), the scan's roofline fraction, the oracle on the host
    cores; HS and four native scans beside the 128K and 8K/32K decodes."""
    import torch
    import li_inputs
    w = li_inputs.spec(name, native=(name in NATIVE_SIDE and not a.no_side))
    x = li_inputs.make_workload(w, seed=a.seed, device=dev)
    step = Step(li, w, x, dev)
    n = {"tiny_f32": 200, "dsa_bf16_8k": 200, "fp8_32k_b32": 100, "fp8_128k_hs": 60,
         "prefill_bf16_128k": 4}[name]
    n = max(n, min(a.steps, 1000)) if w.T == 1 else n
    for _ in range(max(3, min(a.warmup, 20)) if w.T == 1 else 2):
        flush()
        step(stream)
    _chk(li, li.li_device_status(stream), name)
    spin_up(flush, dev)
    ts, _ = time_steps(step, n, flush, stream, dev)
    _chk(li, li.li_device_status(stream), name)
    lat_us = statistics.median(ts) * 1e3
    spin_up(flush, dev)
    kb = breakdown(step, min(n, 100), flush, stream, dev)
    _chk(li, li.li_device_status(stream), name)
    q_pos = x["q_pos"].tolist() if x["q_pos"] is not None else None
    sb = step_bytes(w)
    rec = {"workload": name, "B": w.B, "T": w.T, "L": w.L, "G": w.G, "H": w.H, "r": w.r, "k": w.k,
           "latent": w.lat_dtype, "steps_timed": n, "latency_us": lat_us,
           "tokens_scored_per_s": scored_positions(w, q_pos) / (lat_us * 1e-6),
           "gbs": sb["total"] / (lat_us * 1e-6) / 1e9, "step_bytes": sb["total"],
           "kernels_us": kb, "roofline": roofline(w, kb["score"], q_pos, peaks())}
    if w.T > 1:
        rec["tflops"] = scan_flops(w, q_pos) / (lat_us * 1e-6) / 1e12
    if name == "tiny_f32" or name == "dsa_bf16_8k":
        rec["note"] = "a few MB per step: launch-latency bound, not bandwidth bound"
    if w.T == 1 and not a.no_side:
        rec.update(side_timings(a, w, x, step, li, stream, flush, dev))
    if cpu:
        rec["cpu_baseline"] = config_cpu_baseline(a, name)
    del step, x
    torch.cuda.empty_cache()
    return rec


def config_cpu_baseline(a, name):
    """The oracle on the host cores for one config (the cpu_baseline field of
    its record)."""
    import li_inputs
    w = li_inputs.spec(name, native=False)
    cb = cpu_oracle_rate(w, a.seed, a.cpu_sample_seconds)
    out = {k2: cb[k2] for k2 in ("value", "unit", "cores", "kind", "sample", "step_ms", "extrapolated")}
    if "tflops" in cb:
        out["tflops"] = cb["tflops"]
    return out


class HostPool:
    """Page-locked host memory for the end-to-end leg: one cudaHostAlloc block
    (64 MB or more) handing out 2 MB-aligned buffers."""

    ALIGN = 2 << 20

    def __init__(self, nbytes):
        from cuda.bindings import runtime as rt
        self.rt = rt
        self.size = max(64 << 20, -(-nbytes // self.ALIGN) * self.ALIGN)
        err, self.ptr = rt.cudaHostAlloc(self.size, 0)
        if err != rt.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaHostAlloc failed: {err}")
        self.used = 0

    def buffer(self, like):
        """A HostBuffer holding a copy of the CPU tensor `like`."""
        n = like.numel() * like.element_size()
        if self.used + n > self.size:
            raise RuntimeError("host pool exhausted")
        b = HostBuffer(self.rt, self.ptr + self.used, like)
        self.used += -(-n // self.ALIGN) * self.ALIGN
        return b

    def free(self):
        self.rt.cudaFreeHost(self.ptr)


class HostBuffer:
    """A CPU tensor view of page-locked pool memory, filled once from `like`
    by one thread; copies to and from the device are cudaMemcpyAsync calls on
    the caller's stream.  (Host buffers written by torch's multi-threaded CPU
    copy were read by every later host-to-device DMA at ~11 GB/s instead of
    ~50 GB/s, the same bytes written by a single memmove at the full rate:
    the lines left in many cores' caches slow the device's reads.)"""

    def __init__(self, rt, ptr, like):
        import ctypes
        import torch
        self.rt = rt
        self.ptr = ptr
        self.nbytes = like.numel() * like.element_size()
        raw = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        self.t = torch.frombuffer(raw, dtype=torch.uint8).view(like.dtype).view(like.shape)
        src = like.contiguous().view(torch.uint8).numpy()
        ctypes.memmove(self.ptr, src.ctypes.data, self.nbytes)

    def _copy(self, dst, src, kind, stream):
        (err,) = self.rt.cudaMemcpyAsync(dst, src, self.nbytes, kind, stream.cuda_stream)
        if err != self.rt.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaMemcpyAsync failed: {err}")

    def to_device(self, dst, stream):
        self._copy(dst.data_ptr(), self.ptr, self.rt.cudaMemcpyKind.cudaMemcpyHostToDevice, stream)

    def from_device(self, src, stream):
        self._copy(self.ptr, src.data_ptr(), self.rt.cudaMemcpyKind.cudaMemcpyDeviceToHost, stream)


def e2e_timing(a, w, x, step, li, dev, ws):
    """The same step through the C ABI with host buffers: every step copies its
    queries and head weights from pinned host memory and reads its selections
    back.  Steps rotate over three streams with their own device buffers, so
    one step's copies overlap other steps' kernels, as a serving loop with a
    few requests in flight would run them (with two, a step's upload waits in
    its stream for the read-back of the step before it); the time is the
    whole run's, from one event before the first copy to
    the end of the last read-back.  No L2 flush here: every step streams the
    whole latent cache (more than the L2).  Also times a bare pinned copy of
    the same bytes each way on an idle GPU, the link's own bound.  Host
    buffers are page-locked, from one cudaHostAlloc block, and written once
    at set-up by one thread."""
    import torch
    stream = torch.cuda.current_stream(dev)
    NS = 3
    idx_bytes = step.idx.numel() * step.idx.element_size()
    pool = HostPool(x["q"].numel() * x["q"].element_size() + x["w"].numel() * x["w"].element_size() +
                    NS * idx_bytes + 4 * HostPool.ALIGN)
    q_h = pool.buffer(x["q"].cpu())
    w_h = pool.buffer(x["w"].cpu())
    streams = [torch.cuda.Stream(dev) for _ in range(NS)]
    slots = []
    for _ in range(NS):
        sx = dict(x)
        sx["q"], sx["w"] = torch.empty_like(x["q"]), torch.empty_like(x["w"])
        st = Step(li, w, sx, dev)
        slots.append({"step": st, "x": sx,
                      "idx_h": pool.buffer(torch.empty(st.idx.shape, dtype=torch.int32))})

    def e2e_step(i):
        st, sl = streams[i % NS], slots[i % NS]
        with torch.cuda.stream(st):
            q_h.to_device(sl["x"]["q"], st)
            w_h.to_device(sl["x"]["w"], st)
            sl["step"](st)
            sl["idx_h"].from_device(sl["step"].idx, st)

    # warm the streams, then keep stepping for 0.3 s of wall time: the set-up
    # above leaves the GPU idle long enough for its first milliseconds of work
    # to run slowly (see spin_up)
    t_warm = time.perf_counter()
    i = 0
    while i < 2 * NS or time.perf_counter() - t_warm < 0.3:
        e2e_step(i)
        i += 1
        if i % (4 * NS) == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    E = min(max(a.steps, 200), 500)
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    ev_start.record(stream)
    for st in streams:
        st.wait_event(ev_start)
    for i in range(E):
        e2e_step(i)
    for st in streams:
        j = torch.cuda.Event()
        j.record(st)
        stream.wait_event(j)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    _chk(li, li.li_device_status(stream), "e2e")
    e2e_ms = max_over_ranks(ev_start.elapsed_time(ev_end) / E, ws, dev)
    h2d = q_h.nbytes + w_h.nbytes
    d2h = slots[0]["idx_h"].nbytes

    # bare pinned copies of the same sizes, one direction at a time
    def bare(fn, reps=50):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps
    dq, dw = torch.empty_like(x["q"]), torch.empty_like(x["w"])
    h2d_ms = bare(lambda: (q_h.to_device(dq, stream), w_h.to_device(dw, stream)))
    d2h_ms = bare(lambda: slots[0]["idx_h"].from_device(slots[0]["step"].idx, stream))
    torch.cuda.synchronize(dev)
    pool.free()
    return {"ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": E, "streams": NS,
            "link": {"h2d_us": h2d_ms * 1e3, "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9,
                     "d2h_us": d2h_ms * 1e3, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
                     "how": "the step's own copies alone on an idle GPU, page-locked host memory "
                            "(one cudaHostAlloc block), mean of 50"}}


def run_ours(a, w):
    import torch

    import li_inputs
    import shared_latent_key_cache_b300 as li

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    x = li_inputs.make_workload(dataclasses.replace(w, native=False), seed=a.seed + rank, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    step = Step(li, w, x, dev)

    for _ in range(a.warmup):
        flush()
        step(stream)
    _chk(li, li.li_device_status(stream), "warm-up")

    K = a.steps
    barrier = (lambda: torch.distributed.barrier()) if ws > 1 else (lambda: None)
    barrier()
    clk = ClockSampler(local)
    ts, t_wall = time_steps(step, K, flush, stream, dev, clk)
    barrier()
    _chk(li, li.li_device_status(stream), "timed steps")
    ms_per_step = max_over_ranks(sum(ts), ws, dev) / K
    sb = step_bytes(w)
    value = whole_job_rate(sb["total"], ws, ms_per_step)
    spin_up(flush, dev)
    kb = breakdown(step, min(K, 400), flush, stream, dev)
    clocks = clk.summary()
    e2e = e2e_timing(a, w, x, step, li, dev, ws)
    q_pos = x["q_pos"].tolist() if x["q_pos"] is not None else None
    roof = roofline(w, kb["score"], q_pos, peaks())
    launches = step.launches * K
    del step, x
    torch.cuda.empty_cache()

    # Every GPU timing comes before the first run of the oracle on the host
    # cores: timings that include launches from the host came out up to twice
    # as long right after it.
    per_config = {}
    if rank == 0:
        main = {"workload": w.name, "latency_us": ms_per_step * 1e3,
                "tokens_scored_per_s": scored_positions(w, q_pos) * ws / (ms_per_step * 1e-3),
                "gbs": value, "kernels_us": kb, "roofline": roof,
                "note": "this record is the contract line itself"}
        if not a.no_side and w.T == 1:
            sx = li_inputs.make_workload(dataclasses.replace(w, native=True), seed=a.seed, device=dev)
            sstep = Step(li, w, sx, dev)
            main.update(side_timings(a, w, sx, sstep, li, stream, flush, dev))
            del sstep, sx
            torch.cuda.empty_cache()
        if ws == 1 and not a.no_configs:
            for name in PER_CONFIG:
                if name != w.name:
                    per_config[name] = config_record(a, name, li, dev, stream, flush, cpu=False)
        cb = None
        if ws == 1:
            cb = cpu_oracle_rate(w, a.seed, a.cpu_sample_seconds)
            cb = {k2: cb[k2] for k2 in ("value", "unit", "cores", "kind", "sample")}
            for name, rec in per_config.items():
                rec["cpu_baseline"] = config_cpu_baseline(a, name)
        main["cpu_baseline"] = cb
        per_config = {w.name: main, **per_config}
        per_config = {n: per_config[n] for n in PER_CONFIG if n in per_config}
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K,
            "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.lat_dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "L": w.L, "G": w.G, "H": w.H, "d": w.d,
                       "r": w.r, "k": w.k, "latent": {"fp8": "fp8 e4m3 + fp32 per-token scale",
                                                      "bf16": "bf16", "f32": "fp32"}[w.lat_dtype],
                       "step": "absorb + 4-layer group score + per-layer top-k",
                       "l2": "evicted before every step by reading a 256 MiB buffer (no dirty lines left), outside the timed events; inputs also exceed L2",
                       "parallelism": f"replicas{ws}" if ws > 1 else "single GPU",
                       **({"shape_overrides": shape_overrides(a.shape)} if a.shape else {})},
            "latency_us": ms_per_step * 1e3,
            "tokens_scored_per_s": main["tokens_scored_per_s"],
            "kernels_us": kb,
            "kernels_timing": f"medians of {min(K, 400)} further steps with an event between the kernels "
                              "(those events stop the launch overlap, so the three sum to more than latency_us)",
            "step_bytes": sb,
            "wall_s_timed": t_wall,
            "e2e": {"value": whole_job_rate(sb["total"], ws, e2e["ms_per_step"]), "unit": "GB/s",
                    **e2e,
                    "timing": "whole run of E steps between two events; steps rotate over three "
                              "streams so copies overlap other steps' kernels; no L2 flush (each step "
                              "streams the whole latent cache)",
                    "resident": "latent cache and decoders (device state across decode steps)"},
            "gpu_launches": launches,
            "roofline": roof,
            "clocks": clocks,
            "cpu_baseline": cb,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def side_timings(a, w, x, step, li, stream, flush, dev):
    """Beside a decode config: the latent append of one new token per sequence,
    hierarchical selection (total and per launch), and four native per-layer
    DSA scans with (and without) their top-k, on the same batch."""
    import torch
    import li_inputs
    B, G, H, r, L, k, d = w.B, w.G, w.H, w.r, w.L, w.k, w.d
    out = {}
    reps = max(5, min(200, a.steps // 10, 60 if L > 65536 else 200))

    def timeit(fn):
        spin_up(flush, dev)
        for _ in range(3):
            flush()
            fn()
        ts = []
        for i in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ts) * 1e3

    # latent-cache append of one new token per sequence (eqs. 1-2): hidden size
    # 7168 (DeepSeek-V3.2), RoPE branch 64 of the r latent values
    dm, rR = 7168, 64 if r >= 64 else 0
    xa, Pa = li_inputs.make_append_inputs(B, dm, r, "bf16", seed=a.seed, device=dev)
    lat_dt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[w.lat_dtype]
    lat_a = torch.zeros(B, 8, r, dtype=lat_dt, device=dev)
    sc_a = torch.zeros(B, 8, dtype=torch.float32, device=dev)
    pos_a = torch.full((B,), 7, dtype=torch.int32, device=dev)

    def append():
        assert li.li_append_latent(xa, Pa, pos_a, rR, lat_a, sc_a, stream=stream) == 0
    ap_us = timeit(append)
    ap_bytes = r * dm * 2 + B * dm * 2 + B * (r * lat_a.element_size() + 4)
    out["append"] = {"B": B, "d_model": dm, "r": r, "r_rope": rR, "latency_us": ap_us,
                     "bytes": ap_bytes, "gbs": ap_bytes / (ap_us * 1e-6) / 1e9}

    m = w.m if w.m else 8192
    q_abs, q_scale = step.q_abs, step.q_scale
    if m <= L:
        cand = torch.empty(B, m, dtype=torch.int32, device=dev)
        hidx = torch.empty(B, G, k, dtype=torch.int32, device=dev)
        wsb = torch.empty(li.li_hs_workspace_size(B, G, L, m, k), dtype=torch.uint8, device=dev)

        def hs():
            st = li.li_absorb_queries(x["q"], x["D"], q_abs, q_scale, stream)
            st |= li.li_hs_select(x["latent"], x["lat_scale"], q_abs, q_scale, x["w"], m, k, cand,
                                  hidx, wsb, None, stream)
            assert st == 0
        hs_us = timeit(hs)
        # per launch: absorb first, then the four launches of the selection between events
        stages = []
        for i in range(reps):
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            ev[0].record(stream)
            assert li.li_absorb_queries(x["q"], x["D"], q_abs, q_scale, stream) == 0
            assert li.li_hs_select_profiled(x["latent"], x["lat_scale"], q_abs, q_scale, x["w"], m, k,
                                            cand, hidx, wsb, ev[1:], None, stream) == 0
            stages.append(ev)
        torch.cuda.synchronize(dev)
        names = ["absorb", "anchor_scan", "anchor_top_m", "follower_rescore", "top_k_all_layers"]
        per = {nm: statistics.median(e[j].elapsed_time(e[j + 1]) * 1e3 for e in stages)
               for j, nm in enumerate(names)}
        out["hs"] = {"m": m, "latency_us": hs_us, "stages_us": per,
                     "stages_timing": "medians with an event between the launches",
                     "scored_positions_per_seq": L + (G - 1) * min(m, L),
                     "tokens_scored_per_s": B * (L + (G - 1) * min(m, L)) / (hs_us * 1e-6)}

    if "keys" in x:
        q8 = torch.empty(B, 1, 1, H, d, dtype=torch.uint8, device=dev)
        qs8 = torch.empty(B, 1, 1, H, dtype=torch.float32, device=dev)
        qls = [x["q"][:, :, l:l + 1].contiguous() for l in range(G)]
        wls = [x["w"][:, 0, l].contiguous() for l in range(G)]
        ns = torch.empty(B, L, dtype=torch.float32, device=dev)
        nidx = torch.empty(B, k, dtype=torch.int32, device=dev)
        nws_n = li.li_topk_workspace_size(B, L, k)
        nws = torch.empty(nws_n, dtype=torch.uint8, device=dev) if nws_n > 0 else None

        def native(with_topk=True):
            for l in range(G):
                st = li.li_absorb_queries(qls[l], None, q8, qs8, stream)
                st |= li.li_native_score(x["keys"][l], x["key_scale"][l], q8.view(B, H, d),
                                         qs8.view(B, H), wls[l], ns, stream)
                if with_topk:
                    st |= li.li_topk(ns, k, nidx, None, None, nws, stream)
                assert st == 0
        n_us = timeit(lambda: native(True))
        n_scan_us = timeit(lambda: native(False))
        nbytes = G * B * L * (d + 4)
        out["native_x4"] = {"latency_us": n_us, "scan_only_us": n_scan_us,
                            "cache_bytes": nbytes, "scan_gbs": nbytes / (n_scan_us * 1e-6) / 1e9}
    return out


def main():
    a = parse()
    import li_inputs
    w = li_inputs.spec(a.workload, **shape_overrides(a.shape))
    if a.impl == "reference":
        run_reference(a, w)
    else:
        run_ours(a, w)


if __name__ == "__main__":
    main()
