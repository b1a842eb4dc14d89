"""Benchmark of the fused cascaded-reduction kernels on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the hot path on one batch of the workload's synthetic
input, inputs already resident in HBM.  The default workload is the
non-causal fp16 attention forward (B=4 H=12 N=4096 D=64, seed 1); the line's
``parts`` object reports the other workloads (causal GQA bf16 attention,
split-KV decode, residual+LayerNorm and RMSNorm, softmax cross-entropy, the
sliding-window and ALiBi attention variants, rotary embedding of Q and K, tiny
fp32 attention) measured the
same way in the same run, and ``ablations`` times the fusion-level and
non-incremental variants of the LayerNorm and cross-entropy cascades.  Each
timed step is bracketed by CUDA events on the launching stream, with an L2
flush before every step, outside the events: a 512 MiB memset (larger than
the 129 MB L2), then a 256 MiB read so that no dirty flush line is left for
the timed kernel to write back.  Under torchrun each rank runs an
independent replica (no data-path collective: the work of one call does not
shard across GPUs here), ``value`` is the units all ranks processed divided by
the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (a deliberately slow baseline,
not a GPU reference implementation) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from cascaded_reductions_pass_gb300 import inputs, workmodel  # noqa: E402

L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(kernel_file, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    is unchanged since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, "cascaded_reductions_pass_gb300", "csrc", kernel_file)
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent["bytes_per_launch"] if ent.get("source_sha256_16") == digest else None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
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
        sel = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25] or [p for (_, p) in self.samples]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(p[0]) for p in sel if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in sel if p[1].replace(".", "").isdigit()]
        reasons = sorted({self.NAMES[i] for p in sel for i in range(4) if p[3 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


# ----------------------------------------------------------------------------- workloads
# metric, unit and bound per workload kind; both arms report the same metric and unit
METRICS = {
    "attn": ("attention forward TFLOP/s", "TFLOP/s", "tensor"),
    "decode": ("split-KV decode GB/s", "GB/s", "hbm"),
    "rope": ("rotary embedding GB/s", "GB/s", "hbm"),
    "xent": ("softmax cross-entropy GB/s", "GB/s", "hbm"),
    "rmsnorm": ("residual+RMSNorm GB/s", "GB/s", "hbm"),
    "layernorm": ("residual+LayerNorm GB/s", "GB/s", "hbm"),
}


def workload_config(w):
    """The workload part of the bench line's config, the same for both arms."""
    return {"workload": w.name, **w.dims, "dtype": w.dtype, "seed": w.seed}


class Runner:
    """One workload: its inputs on the device, one step of the hot path, its work."""

    def __init__(self, name, dev, batch=None):
        import dataclasses

        import cascaded_reductions_pass_gb300 as rf

        self.rf = rf
        self.w = inputs.WORKLOADS[name]
        if batch:  # a smaller case of the same kernel (for profiler captures)
            key = "rows" if self.w.kind in ("layernorm", "rmsnorm", "xent") else "B"
            self.w = dataclasses.replace(self.w, dims={**self.w.dims, key: int(batch)})
        self.dev = dev
        d = self.w.dims
        self.host = inputs.make(self.w)
        self.dtype = self.w.dtype
        if self.w.kind == "attn":
            self.scale = float(np.float32(1.0 / math.sqrt(d["D"])))
            self.flops = workmodel.attn_flops(d["B"], d["Hq"], d["N"], d["N"], d["D"], d["causal"], d.get("window", 0))
            self.window = d.get("window", 0)
            self.alibi = None
            if d.get("alibi"):
                self.alibi = rf.alibi_slopes(d["Hq"], device=dev)
            self.bytes = workmodel.attn_bytes(d["B"], d["Hq"], d["Hkv"], d["N"], d["N"], d["D"], self.dtype)
            self.metric, self.unit, self.bound = METRICS["attn"]
            self.units = self.flops / 1e12
            self.kernel_file = "attn_fwd_f32.cu" if self.dtype == "f32" else "attn_fwd_tc.cuh"
            self.kernel = "attn_fwd_f32" if self.dtype == "f32" else "attn_fwd_tc"
            if self.dtype != "f32" and d["D"] == 64 and 0 < self.window <= 1024:  # the persistent windowed kernel
                self.kernel_file, self.kernel = "attn_fwd_tc_window.cu", "attn_fwd_tc_window"
            if self.dtype == "f32":
                self.bound = "alu"
        elif self.w.kind == "decode":
            self.scale = float(np.float32(1.0 / math.sqrt(d["D"])))
            self.bytes = workmodel.decode_bytes(d["B"], d["Hq"], d["Hkv"], d["L"], d["D"], self.dtype)
            self.flops = workmodel.decode_flops(d["B"], d["Hq"], d["L"], d["D"])
            self.metric, self.unit, self.bound = METRICS["decode"]
            self.units = self.bytes / 1e9
            self.kernel_file, self.kernel = "decode_split.cu", "decode_split (+ lse_merge)"
        elif self.w.kind == "rope":
            self.bytes = workmodel.rope_bytes(d["B"], d["Hq"], d["Hkv"], d["N"], d["D"], self.dtype)
            self.flops = 6.0 * d["B"] * (d["Hq"] + d["Hkv"]) * d["N"] * d["D"] / 2
            self.metric, self.unit, self.bound = METRICS["rope"]
            self.units = self.bytes / 1e9
            self.kernel_file, self.kernel = "rope.cu", "rope"
        elif self.w.kind == "xent":
            self.bytes = workmodel.xent_bytes(d["rows"], d["vocab"], self.dtype)
            self.flops = 4.0 * d["rows"] * d["vocab"]
            self.metric, self.unit, self.bound = METRICS["xent"]
            self.units = self.bytes / 1e9
            self.kernel_file, self.kernel = "xent_fused.cu", "xent"
        elif self.w.kind == "rmsnorm":
            self.bytes = workmodel.layernorm_bytes(d["rows"], d["cols"], self.dtype, affine=False) + d["cols"] * 2
            self.flops = 4.0 * d["rows"] * d["cols"]
            self.metric, self.unit, self.bound = METRICS["rmsnorm"]
            self.units = self.bytes / 1e9
            self.kernel_file, self.kernel = "ln_fused.cu", "rms_fused"
        else:
            self.bytes = workmodel.layernorm_bytes(d["rows"], d["cols"], self.dtype)
            self.flops = 10.0 * d["rows"] * d["cols"]
            self.metric, self.unit, self.bound = METRICS["layernorm"]
            self.units = self.bytes / 1e9
            self.kernel_file, self.kernel = "ln_fused.cu", "ln_fused"
        self.dev_in = [t.to(dev) for t in self.host]
        self._alloc_outputs()

    def _alloc_outputs(self):
        d, dev = self.w.dims, self.dev
        if self.w.kind == "attn":
            q = self.dev_in[0]
            self.o = torch.empty_like(q)
            self.lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
            self.outs = [self.o, self.lse]
            # the unmasked 16-bit kernel splits a short last wave along the keys (two launches)
            self.ws = None
            if not d["causal"] and self.dtype != "f32":
                self.ws = self.rf.attn_workspace(q, self.dev_in[1], False)
            self.launches = 2 if self.ws is not None else 1
        elif self.w.kind == "rope":
            self.o = torch.empty_like(self.dev_in[0])
            self.ko = torch.empty_like(self.dev_in[1])
            self.outs = [self.o, self.ko]
        elif self.w.kind == "xent":
            self.o = torch.empty(d["rows"], dtype=torch.float32, device=dev)
            self.lse = torch.empty(d["rows"], dtype=torch.float32, device=dev)
            self.outs = [self.o, self.lse]
        elif self.w.kind == "decode":
            q = self.dev_in[0]
            self.ws = self.rf.decode_workspace(d["B"], d["Hq"], d["D"], d["splits"], dev)
            self.o = torch.empty((d["B"], d["Hq"], d["D"]), dtype=q.dtype, device=dev)
            self.lse = torch.empty((d["B"], d["Hq"]), dtype=torch.float32, device=dev)
            self.outs = [self.o, self.lse]
        else:
            self.o = torch.empty_like(self.dev_in[0])
            self.outs = [self.o]

    def step(self, ins=None):
        rf, d = self.rf, self.w.dims
        ins = ins or self.dev_in
        if self.w.kind == "attn" and (self.window or self.alibi is not None):
            rf.rf_attn_fwd_ex(ins[0], ins[1], ins[2], self.o, self.lse, scale=self.scale, causal=bool(d["causal"]),
                              window=self.window, alibi_slopes=self.alibi)
        elif self.w.kind == "attn":
            rf.rf_attn_fwd_ex(ins[0], ins[1], ins[2], self.o, self.lse, scale=self.scale, causal=bool(d["causal"]),
                              workspace=self.ws)
        elif self.w.kind == "decode":
            rf.rf_attn_decode_splitkv(ins[0], ins[1], ins[2], self.o, self.ws, d["splits"], lse=self.lse,
                                      scale=self.scale)
        elif self.w.kind == "rmsnorm":
            rf.rf_rmsnorm_fused(ins[0], ins[1], ins[2], self.o, eps=d["eps"])
        elif self.w.kind == "rope":
            rf.rf_rope_qk(ins[0], ins[1], self.o, self.ko, base=d["base"])
        elif self.w.kind == "xent":
            rf.rf_softmax_xent(ins[0], ins[1], self.o, self.lse)
        else:
            rf.rf_layernorm_fused(ins[0], ins[1], ins[2], ins[3], self.o, eps=d["eps"])

    def describe(self):
        return workload_config(self.w)


class L2Flush:
    """Leaves L2 cold and clean before a timed step: a 512 MiB memset (larger
    than the 129 MB L2) evicts every line of the step's inputs, then a 256 MiB
    read replaces the memset's dirty lines with clean ones.  Without the read,
    the next kernel pays the write-back of up to 129 MB of the flush buffer
    (measured: 5-9 us on an HBM-bound launch of 100-400 MB)."""

    def __init__(self, dev):
        self.write = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.read = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=dev)

    def zero_(self):
        self.write.zero_()
        self.read.sum()  # one read-only reduction: no temporary, nothing written back


def time_steps(runner, steps, warmup, flush):
    """Per-step device time (ms) with events around the step only; L2 flushed before each step."""
    for _ in range(warmup):
        flush.zero_()
        runner.step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        runner.step()
        ends[i].record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_e2e(runner, steps, warmup):
    """The step end to end through the public API with pinned host buffers,
    pipelined over steps the way a serving loop runs them: the host-to-device
    copy of step i+1's inputs and the device-to-host copy of step i-1's outputs
    run on streams of their own while step i computes, with two sets of device
    inputs and outputs and events ordering each reuse.  Every step's inputs are
    copied in and its outputs copied out inside the timed region, which runs
    from before the first copy in to after the last copy out."""
    names = [n for n in ("o", "lse", "ko") if any(getattr(runner, n, None) is t for t in runner.outs)]
    pinned_in = [t.pin_memory() for t in runner.host]
    sets_in = [[torch.empty_like(t) for t in runner.dev_in] for _ in range(2)]
    sets_out = [{n: getattr(runner, n) for n in names}, {n: torch.empty_like(getattr(runner, n)) for n in names}]
    pinned_out = [[torch.empty(sets_out[b][n].shape, dtype=sets_out[b][n].dtype, pin_memory=True) for n in names]
                  for b in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()

    def run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev_in, ev_comp, ev_out = [], [], []
        start.record(h2d_s)
        for i in range(n):
            b = i % 2
            if i >= 2:
                h2d_s.wait_event(ev_comp[i - 2])  # step i-2 has finished reading input set b
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(sets_in[b], pinned_in):
                    dst.copy_(src, non_blocking=True)
            ev_in.append(torch.cuda.Event())
            ev_in[i].record(h2d_s)
            comp.wait_event(ev_in[i])
            if i >= 2:
                comp.wait_event(ev_out[i - 2])  # step i-2's outputs (set b) have been read back
            for name, t in sets_out[b].items():
                setattr(runner, name, t)
            runner.step(sets_in[b])
            ev_comp.append(torch.cuda.Event())
            ev_comp[i].record(comp)
            d2h_s.wait_event(ev_comp[i])
            with torch.cuda.stream(d2h_s):
                for dst, name in zip(pinned_out[b], names):
                    dst.copy_(sets_out[b][name], non_blocking=True)
            ev_out.append(torch.cuda.Event())
            ev_out[i].record(d2h_s)
        end.record(d2h_s)
        return start, end

    run(warmup)
    torch.cuda.synchronize()
    start, end = run(steps)
    torch.cuda.synchronize()
    for name, t in sets_out[0].items():
        setattr(runner, name, t)
    ms = start.elapsed_time(end) / steps
    h2d = sum(t.numel() * t.element_size() for t in pinned_in)
    d2h = sum(t.numel() * t.element_size() for t in pinned_out[0])
    return ms, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(w, host, budget_s=12.0):
    """Time the fp64 oracle on a bounded sample of the workload; returns
    (value in the workload's unit, sample description, seconds)."""
    import oracle

    d = w.dims
    t_start = time.perf_counter()
    done_units, what = 0.0, ""
    if w.kind == "attn":
        q, k, v = host
        scale = float(np.float32(1.0 / math.sqrt(d["D"])))
        G = d["Hq"] // d["Hkv"]
        window = d.get("window", 0)
        slopes = oracle.alibi_slopes(d["Hq"]) if d.get("alibi") else None
        rows = min(d["N"], 1024)
        # blocks of query rows of one (batch, head) against all its keys, cycling
        # over the whole workload until the time budget is spent
        blocks = [(b, h, r0) for r0 in range(0, d["N"], rows) for b in range(d["B"]) for h in range(d["Hq"])]
        n = 0
        while n == 0 or time.perf_counter() - t_start < budget_s:
            b, h, r0 = blocks[n % len(blocks)]
            sel = np.arange(r0, min(r0 + rows, d["N"]))
            oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h // G:h // G + 1], v[b:b + 1, h // G:h // G + 1],
                             scale, bool(d["causal"]), rows=sel, window=window,
                             alibi_slopes=None if slopes is None else slopes[h:h + 1])
            if not d["causal"]:
                vis = len(sel) * d["N"]
            else:
                vis = int(np.minimum(sel + 1, window if window else d["N"]).sum())
            done_units += 4.0 * vis * d["D"] / 1e12
            n += 1
        what = (f"{n} blocks of up to {rows} query rows x all keys, cycling over the workload's "
                f"{len(blocks)} (batch, head, row-block) blocks")
    elif w.kind == "decode":
        q, k, v = host
        scale = float(np.float32(1.0 / math.sqrt(d["D"])))
        G = d["Hq"] // d["Hkv"]
        groups = [(b, hk) for b in range(d["B"]) for hk in range(d["Hkv"])]
        n = 0
        while n == 0 or time.perf_counter() - t_start < budget_s:
            b, hk = groups[n % len(groups)]
            oracle.decode(q[b:b + 1, hk * G:(hk + 1) * G], k[b:b + 1, hk:hk + 1], v[b:b + 1, hk:hk + 1], scale)
            done_units += workmodel.decode_bytes(1, G, 1, d["L"], d["D"], w.dtype) / 1e9
            n += 1
        what = f"{n} (batch, kv-head) groups of {G} query heads over all {d['L']} keys, cycling over {len(groups)}"
    elif w.kind == "rope":
        q, k = host
        pos = np.arange(d["N"])
        planes = [(t, b, h) for t in (0, 1) for b in range(d["B"]) for h in range(d["Hq"] if t == 0 else d["Hkv"])]
        n = 0
        while n == 0 or time.perf_counter() - t_start < budget_s:
            t, b, h = planes[n % len(planes)]
            oracle.rope((q if t == 0 else k)[b, h], pos, d["base"])
            done_units += 2 * d["N"] * d["D"] * (2 if w.dtype != "f32" else 4) / 1e9
            n += 1
        what = f"{n} (tensor, batch, head) planes of {d['N']} rows, cycling over {len(planes)}"
    else:
        # row blocks of the row-wise cascades, cycling over the workload until the budget is spent
        step = 64 if w.kind == "xent" else 512
        n_rows = d["rows"]
        n = 0
        rows_done = 0
        while n == 0 or time.perf_counter() - t_start < budget_s:
            r0 = (n * step) % n_rows
            r1 = min(r0 + step, n_rows)
            if w.kind == "xent":
                z, t = host
                oracle.softmax_xent(z[r0:r1], t[r0:r1])
            elif w.kind == "rmsnorm":
                x, r, g = host
                oracle.rmsnorm(x[r0:r1], r[r0:r1], g, d["eps"])
            else:
                x, r, g, b = host
                oracle.layernorm(x[r0:r1], r[r0:r1], g, b, d["eps"])
            rows_done += r1 - r0
            n += 1
        if w.kind == "xent":
            done_units = workmodel.xent_bytes(rows_done, d["vocab"], w.dtype) / 1e9
        elif w.kind == "rmsnorm":
            done_units = (workmodel.layernorm_bytes(rows_done, d["cols"], w.dtype, affine=False) + d["cols"] * 2) / 1e9
        else:
            done_units = workmodel.layernorm_bytes(rows_done, d["cols"], w.dtype) / 1e9
        what = f"{rows_done} rows in blocks of {step}, cycling over the workload's {n_rows} rows"
    secs = time.perf_counter() - t_start
    return done_units / secs, what, secs


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info

        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main
def measure(name, dev, steps, warmup, flush, peaks, with_e2e=True, batch=None):
    r = Runner(name, dev, batch)
    times = time_steps(r, steps, warmup, flush)
    ms = float(np.mean(times))
    val = r.units / (ms / 1e3)
    achieved_unit = "TFLOP/s" if r.bound == "tensor" else ("GB/s" if r.bound == "hbm" else "TFLOP/s")
    if r.bound == "hbm":
        achieved, peak = r.bytes / (ms / 1e3) / 1e9, peaks["hbm_gbs"]
    elif r.bound == "tensor":
        achieved, peak = r.flops / (ms / 1e3) / 1e12, peaks["bf16_tflops"]
    else:  # fp32 FFMA: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz
        achieved, peak = r.flops / (ms / 1e3) / 1e12, 152 * 128 * 2 * 2.07e9 / 1e12
    res = {
        "workload": name, "value": val, "unit": r.unit, "ms_per_step": ms,
        "ms_median": float(np.median(times)),
        "ms_p10": float(np.percentile(times, 10)), "ms_p90": float(np.percentile(times, 90)),
        "roofline": {"bound": r.bound, "achieved": achieved, "peak": peak, "unit": achieved_unit,
                     "frac": achieved / peak, "traffic": kernel_traffic(r.kernel_file, name),
                     "kernel": r.kernel,
                     "peak_source": peaks["source"] if r.bound != "alu" else "derived: 152 SMs x 128 FFMA x 2 x 2.07 GHz"},
        "algorithmic_bytes": r.bytes, "algorithmic_flops": r.flops, "config": r.describe(),
    }
    if with_e2e:
        e_ms, h2d, d2h = time_e2e(r, max(10, min(steps, 30)), 3)
        res["e2e"] = {"value": r.units / (e_ms / 1e3), "unit": r.unit, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
    return r, res


def measure_ablations(dev, steps, warmup, flush, peaks):
    """Each fusion-level / incremental-form variant of the residual+LayerNorm and
    softmax cross-entropy workloads (RedFuser, Figures 6-7), timed like a step.
    ``gbs`` is the fused form's algorithmic bytes over the variant's time, so it
    compares like for like; ``model_bytes`` is the variant's own compulsory
    traffic."""
    import cascaded_reductions_pass_gb300 as rf

    out = {}
    for name, op, variants in (("layernorm_residual_bf16", "layernorm", rf.LN_VARIANTS),
                               ("softmax_xent_bf16", "xent", rf.XENT_VARIANTS)):
        w = inputs.WORKLOADS[name]
        d = w.dims
        rows, cols = d["rows"], d["cols" if op == "layernorm" else "vocab"]
        dev_in = [t.to(dev) for t in inputs.make(w)]
        if op == "layernorm":
            o = torch.empty_like(dev_in[0])
        else:
            o = torch.empty(rows, dtype=torch.float32, device=dev)
            lse = torch.empty(rows, dtype=torch.float32, device=dev)
        fused_bytes = workmodel.ablation_bytes(op, 0, rows, cols, w.dtype)
        res = {}
        for v, label in variants.items():
            ws = rf.ablation_workspace(0 if op == "layernorm" else 1, v, rows, cols, dev_in[0].dtype, dev)

            class _Step:
                def step(self, _v=v, _ws=ws):
                    if op == "layernorm":
                        rf.rf_layernorm_ablation(*dev_in, o, _v, workspace=_ws, eps=d["eps"])
                    else:
                        rf.rf_softmax_xent_ablation(dev_in[0], dev_in[1], o, lse, _v, workspace=_ws)

            times = time_steps(_Step(), steps, warmup, flush)
            ms = float(np.mean(times))
            res[str(v)] = {"variant": label, "ms": ms, "gbs": fused_bytes / (ms / 1e3) / 1e9,
                           "model_bytes": workmodel.ablation_bytes(op, v, rows, cols, w.dtype),
                           "launches": {0: 1, 1: 1, 2: 2, 3: 4}[v] if op == "layernorm" else {0: 1, 1: 1, 2: 3}[v]}
            del ws
        base = res["0"]["ms"]
        for r in res.values():
            r["slowdown_vs_fused"] = r["ms"] / base
        out[name] = {"fused_algorithmic_bytes": fused_bytes, "hbm_peak_gbs": peaks["hbm_gbs"], "variants": res}
        del dev_in
        torch.cuda.empty_cache()
    return out


def rope_crossover(dev, flush, steps=10, warmup=3):
    """AttnFuse's "Rotation Calculus" question (Table 4) on this GPU: causal
    attention over rotary-embedded Q and K, with the rotation done
    (a) by the separate pass over Q and K, then attention;
    (b) by the separate pass over K only, Q turned inside the attention kernel;
    (c) inside the attention kernel for both Q and K;
    against (0) the same attention without rotation, for a range of N.
    Returns one row per shape with each variant's mean step time (ms)."""
    import cascaded_reductions_pass_gb300 as rf

    rows = []
    for B, H, D, dtype in ((4, 12, 64, "f16"), (2, 16, 128, "bf16")):
        for N in (1024, 2048, 4096, 8192, 16384):
            q, k, v = (t.to(dev) for t in inputs.attn_inputs(B, H, H, N, N, D, dtype, seed=N + D))
            scale = float(np.float32(1.0 / math.sqrt(D)))
            qo, ko, o = torch.empty_like(q), torch.empty_like(k), torch.empty_like(q)
            lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)

            def attn(qq, kk, mode):
                rf.rf_attn_fwd_ex(qq, kk, v, o, lse, scale=scale, causal=True, rope=mode)

            variants = {
                "attention, no rotation": lambda: attn(q, k, 0),
                "separate pass (Q, K) + attention": lambda: (rf.rf_rope_qk(q, k, qo, ko), attn(qo, ko, 0)),
                "separate pass (K) + Q in kernel": lambda: (rf.rf_rope_qk(k, None, ko), attn(q, ko, 1)),
                "Q and K in kernel": lambda: attn(q, k, 2),
            }
            res = {}
            for name, fn in variants.items():
                class _S:
                    step = staticmethod(fn)

                if not rows:  # the first shape also pays one-time costs: time it twice, keep the second
                    time_steps(_S(), steps, warmup, flush)
                res[name] = float(np.mean(time_steps(_S(), steps, warmup, flush)))
            rows.append({"B": B, "H": H, "N": N, "D": D, "dtype": dtype, "ms": res})
            del q, k, v, qo, ko, o, lse
            torch.cuda.empty_cache()
    return rows


# The five workload configurations of the headline metric, in their order, then the other workloads.
CONFIG_ORDER = ["attn_tiny_f32", "attn_fwd_f16_d64", "attn_fwd_causal_gqa_bf16_d128", "decode_splitkv_bf16",
                "layernorm_residual_bf16"]


def _r(x, nd=4):
    return None if x is None else float(f"{x:.{nd}g}")


def compact_summary(head_name, head, head_e2e, parts, ablations):
    """Every workload's result in a few fields (value, unit, ms per step,
    roofline fraction and bound, DRAM traffic per launch, end-to-end value),
    configurations first; and each ablation variant's slowdown against the
    fused incremental kernel."""
    allres = {head_name: {**head, "e2e": head_e2e}, **parts}
    names = [n for n in CONFIG_ORDER if n in allres] + [n for n in allres if n not in CONFIG_ORDER]
    out = {}
    for i, n in enumerate(names):
        r = allres[n]
        key = f"cfg{CONFIG_ORDER.index(n) + 1} {n}" if n in CONFIG_ORDER else n
        if "error" in r:
            out[key] = {"error": r["error"][:80]}
            continue
        rl, e = r["roofline"], r.get("e2e") or {}
        out[key] = {"v": _r(r["value"]), "u": r["unit"], "ms": _r(r["ms_per_step"]),
                    "frac": _r(rl["frac"], 3), "bound": rl["bound"], "traffic": rl["traffic"],
                    "e2e": _r(e.get("value"))}
    if isinstance(ablations, dict) and "error" not in ablations:
        out["ablation slowdowns"] = {n: [_r(v["slowdown_vs_fused"], 3) for v in a["variants"].values()]
                                     for n, a in ablations.items()}
    return out


def aggregate_over_ranks(local_ms, units_per_rank, world, device=None):
    """Replicas: every rank processed `units_per_rank`; the job's time is the slowest
    rank's.  Returns (max_ms, whole-job value in units/s).  With world > 1 this is a
    MAX all-reduce of one scalar -- the only collective, and it is outside the data path."""
    ms = float(local_ms)
    if world > 1:
        import torch.distributed as dist

        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units_per_rank / (ms / 1e3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="attn_fwd_f16_d64", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-parts", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--rope-crossover", action="store_true",
                    help="only time rotary causal attention three ways over N (AttnFuse's Rotation Calculus)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (attention, decode) or rows (LayerNorm): a smaller case for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = inputs.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        host = inputs.make(w)
        per_step = []
        for i in range(args.warmup + args.steps):
            v, what, secs = oracle_sample(w, host, budget_s=max(0.5, 60.0 / (args.warmup + args.steps)))
            if i >= args.warmup:
                per_step.append((v, secs))
        val = float(np.mean([v for v, _ in per_step]))
        metric, unit, _ = METRICS[w.kind]
        ms = float(np.mean([s for _, s in per_step]) * 1e3)
        print(json.dumps({
            "impl": "reference", "metric": metric, "value": val,
            "unit": unit, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w), "parallelism": "single-process (CPU oracle)",
            "cpu_baseline": {"value": val, "unit": unit, "cores": cpu_threads(), "kind": "oracle", "sample": what},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    import cascaded_reductions_pass_gb300 as rf

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rf.load()
    peaks = load_peaks()
    flush = L2Flush(dev)
    if args.rope_crossover:
        if rank == 0:
            print(json.dumps({"rope_crossover": rope_crossover(dev, flush),
                              "l2_flush": "before every step, outside the events", "steps": 10, "warmup": 3}))
        return
    sampler = ClockSampler(local)
    sampler.start()

    # the headline workload: replicas on every rank, bracketed by barriers
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    runner, res = measure(args.workload, dev, args.steps, args.warmup, flush, peaks, with_e2e=False,
                          batch=args.batch)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    ms, value = aggregate_over_ranks(res["ms_per_step"], runner.units, world, dev)
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = time_e2e(runner, max(10, min(args.steps, 30)), 3)
        e_ms, e2e_val = aggregate_over_ranks(e_ms, runner.units, world, dev)
        e2e = {"value": e2e_val, "unit": runner.unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms,
               "pipelining": "copies in of step i+1 and out of step i-1 overlap step i (two buffer sets)"}
    clocks = sampler.summary(t0, t1)
    launches = args.steps * (2 if w.kind == "decode" else getattr(runner, "launches", 1))

    parts = {}
    if not args.no_parts and rank == 0:
        for name in inputs.WORKLOADS:
            if name == args.workload:
                continue
            try:
                _, pres = measure(name, dev, max(10, args.steps // 2), args.warmup, flush, peaks, with_e2e=True)
                parts[name] = pres
            except Exception as exc:  # a workload whose kernel is unavailable is reported, not hidden
                parts[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
    ablations = None
    if not args.no_parts and rank == 0:
        try:
            ablations = measure_ablations(dev, 10, args.warmup, flush, peaks)
        except Exception as exc:
            ablations = {"error": f"{type(exc).__name__}: {exc}"}
    sampler.stop()
    status = rf.rf_device_status()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, what, secs = oracle_sample(w, runner.host, budget_s=15.0)
        cpu = {"value": v, "unit": runner.unit, "cores": cpu_threads(), "kind": "oracle", "sample": what,
               "seconds": secs}

    if rank == 0:
        line = {
            "metric": runner.metric, "value": value, "unit": runner.unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": runner.dtype, "data": "synthetic",
            "config": runner.describe(),
            "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
            "l2_flush": "before every step, outside the events: 512 MiB memset, then a 256 MiB read "
                        "so that L2 holds only clean lines",
            "roofline": res["roofline"],
            "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "cpu_baseline": cpu,
            "device_status": int(status),
            "ms_median": res["ms_median"], "ms_p10": res["ms_p10"], "ms_p90": res["ms_p90"],
            "parts": parts, "ablations": ablations,
            # last, so that the end of the line alone carries every workload's result
            "summary": compact_summary(args.workload, res, e2e, parts, ablations),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
