"""Benchmark: sink-attention forward + backward (incl. dS_h) on GB300.

One step = one pass of the whole hot path over one batch: sink_attn_fwd_ex
(O, o_lo and LSE), then sink_attn_bwd_preprocess_ex (delta from o + o_lo, and
dS_h) and sink_attn_bwd_main (dQ, dK, dV), all through the C ABI: the path
whose outputs the parity tests hold to the stated tolerance. The backward's
preparation pass (f16 copies of Q and K, the zeroed dQ accumulator), which
depends on Q and K alone, is issued with sink_attn_bwd_prepare on a
lower-priority stream right after the forward is queued, and
sink_attn_bwd_main runs with SINK_BWD_PREPARED once it is done (an event),
on layers whose forward outlasts it; with a window of at most 256 keys the
forward is short, the preparation would spill into the preprocess, and it
stays inside sink_attn_bwd_main on the one stream (as ``--serial-prepare``
does everywhere). The default workload is the GPT-OSS-20B-shaped
full-causal layer (B=2, N=8192, H_q=64, H_kv=8, d=64, bf16). Its inputs (302 MB
of Q/K/V/dO) exceed the 129 MB L2, so no extra flush is done between steps.

FLOP convention (algorithmic, unmasked (row, key) pairs only): forward 4*d per
pair (QK^T and PV), backward 10*d per pair (QK^T recompute, dP, dV, dK, dQ).

The line also carries: ``stage_rates`` (per-stage TFLOP/s and algorithmic
GB/s, the backward also without the recompute), ``roofline`` for the dominant
stage (the backward main loop; against HBM when its arithmetic intensity is
below the ridge point, as in the window layers), ``e2e`` (the same step with
inputs copied in from pinned host memory and every output copied back each
step, the copies overlapping the neighbouring steps' compute; the backward
as one sink_attn_bwd_ex call, whose preparation runs inside it; with the
copy rate of the pinned buffers measured alone), ``clocks``
sampled during the timed region and ``cpu_baseline`` (the oracle on the host
cores, bounded sample).

Prints ONE JSON line on rank 0. ``--impl reference`` times the fp64 CPU oracle
instead (the only reference this method has), on a bounded sample.
``--decode`` prints a separate line for the decode path (KV-cache bandwidth).

``--gpus N`` without a launcher starts N processes itself, one per GPU (it
fails with a clear message if fewer GPUs are visible); under torchrun the
launcher's ranks are used.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import datetime
import hashlib
import json
import math
import os
import platform
import socket
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_sink_softmax_gb300 import inputs  # noqa: E402

METRIC = "sink-attention fwd+bwd TFLOP/s (bf16) and % of GB300 dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- workload math
def pairs_of(w: inputs.Workload, window: int) -> int:
    """Number of unmasked (row, key) pairs summed over heads and sequences."""
    lengths = w.lengths if w.packed else [w.seqlen] * w.batch
    total = 0
    for L in lengths:
        if not w.causal:
            n = L * L
        elif window and window > 0:
            W = window
            full = max(L - W + 1, 0)  # rows i >= W-1 see W keys
            head = min(L, W - 1)      # rows i < W-1 see i+1 keys
            n = head * (head + 1) // 2 + full * W
        else:
            n = L * (L + 1) // 2
        total += n
    return total * w.h_q


def flops_of(w, window):
    p = pairs_of(w, window)
    return 4 * w.head_dim * p, 10 * w.head_dim * p


def bytes_of(w) -> dict:
    """Algorithmic bytes per step (each tensor read or written once):
    forward reads Q, K, V and writes O, o_lo (bf16) and LSE; the preprocess
    reads O, o_lo, dO and LSE and writes D; the backward main reads Q, K, V,
    dO, LSE and D and writes dQ, dK and dV. The fp32 dQ accumulator is
    implementation traffic, not counted."""
    T = w.total_tokens
    e = 2 if w.dtype == torch.bfloat16 else 4
    q = T * w.h_q * w.head_dim * e   # Q, O, dO, dQ each
    kv = T * w.h_kv * w.head_dim * e  # K, V, dK, dV each
    row = 4 * w.h_q * T               # LSE or D (fp32)
    lo = q if w.dtype == torch.bfloat16 else 0  # o_lo: written by the forward, read by the preprocess
    return {"fwd": q + 2 * kv + q + lo + row,
            "bwd_preprocess": 2 * q + lo + row + row,
            "bwd_main": q + 2 * kv + q + 2 * row + q + 2 * kv}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, every 100 ms, each with its
    timestamp; ``summary`` keeps the samples taken inside [mark_start,
    mark_end] (the timed region). nvidia-smi is started before the region and
    given up to 3 s to produce its first sample."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            deadline = time.time() + 3.0
            while time.time() < deadline and os.path.getsize(self.file.name) == 0:
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        if self.t0 is not None and self.t1 is not None:
            kept = []
            for r in rows:
                try:
                    ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if self.t0 <= ts <= self.t1:
                    kept.append(r)
            rows = kept
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no sample inside the timed region"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


class NvmlClockSampler:
    """Read-only NVML samples (SM clock, max SM clock, power, clock-event
    reasons) every ``period_s`` from a thread, between mark_start and
    mark_end, so that a timed region of a few tens of milliseconds still gets
    samples. Calls libnvidia-ml through ctypes; ``ok`` is False if it cannot
    be loaded or the device not found (then ClockSampler's nvidia-smi samples
    are used)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        self._run = threading.Event()
        self._thread = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            except Exception:
                uuid = None
            rc = -1
            if uuid:
                name = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                rc = self.nv.nvmlDeviceGetHandleByUUID(name.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h))
            self.ok = rc == 0
        except OSError:
            self.ok = False

    def _sample(self):
        sm, smax, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) != 0:
            return None
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(smax))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(reasons))
        return (sm.value, smax.value, mw.value / 1000.0, reasons.value)

    def _loop(self):
        while not self._stop.is_set():
            if self._run.is_set():
                x = self._sample()
                if x is not None:
                    self.samples.append(x)
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        return self

    def mark_start(self):
        self._run.set()

    def mark_end(self):
        self._run.clear()

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return None
        names = sorted({n for s in self.samples for bit, n in self.REASONS.items() if s[3] & bit})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": names,
                "samples": len(self.samples), "power_w_max": max(s[2] for s in self.samples),
                "source": f"NVML every {self.period * 1000:.0f} ms inside the timed region"}


class Clocks:
    """NVML samples when available, else nvidia-smi's (ClockSampler)."""

    def __init__(self, device_index: int):
        self.nvml = NvmlClockSampler(device_index)
        self.smi = None if self.nvml.ok else ClockSampler(device_index)

    def __enter__(self):
        (self.nvml if self.smi is None else self.smi).__enter__()
        return self

    def mark_start(self):
        (self.nvml if self.smi is None else self.smi).mark_start()

    def mark_end(self):
        (self.nvml if self.smi is None else self.smi).mark_end()

    def __exit__(self, *exc):
        (self.nvml if self.smi is None else self.smi).__exit__(*exc)

    def summary(self):
        if self.smi is None:
            got = self.nvml.summary()
            if got is not None:
                return got
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no NVML sample"], "samples": 0}
        return self.smi.summary()


# ----------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str) -> None:
    """One process per GPU (torchrun); ``backend`` is nccl on GPUs, gloo in tests."""
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend)


def rank_seed(w: inputs.Workload, rank: int) -> int:
    """Each replica draws its own batch (weak scaling: per-GPU work is fixed)."""
    return w.seed + rank


def aggregate_value(flops_per_rank_step: float, ws: int, ms_max: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_rank_step * ws / (ms_max / 1000) / 1e12


def emit(line: dict, rank: int) -> str | None:
    """Rank 0 alone prints the JSON line; returns what was printed."""
    if rank != 0:
        return None
    text = json.dumps(line)
    print(text, flush=True)
    return text


def config_of(w: inputs.Workload, window: int, ws: int) -> dict:
    return {"workload": w.name, "batch": w.batch, "seq_len": w.seqlen, "h_q": w.h_q,
            "h_kv": w.h_kv, "head_dim": w.head_dim, "causal": w.causal,
            "window": window, "tokens": w.total_tokens,
            "flops_per_step": sum(flops_of(w, window)), "l2": "inputs exceed L2 (no flush)",
            "parallelism": f"replicas x{ws} (independent batches, no collective)"}


def spawn_ranks(n: int, argv, extra_env=None) -> int:
    """Runs ``argv`` as n ranks of one job on this node (RANK, LOCAL_RANK,
    WORLD_SIZE, MASTER_ADDR=127.0.0.1, a free MASTER_PORT), each a fresh
    process; rank 0's output passes through, the others' is discarded unless
    they fail. Returns the largest exit code."""
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ)
        env.update({"RANK": str(r), "LOCAL_RANK": str(r), "WORLD_SIZE": str(n),
                    "LOCAL_WORLD_SIZE": str(n), "MASTER_ADDR": "127.0.0.1",
                    "MASTER_PORT": str(port)})
        env.update(extra_env or {})
        out = None if r == 0 else subprocess.PIPE
        procs.append(subprocess.Popen(list(argv), env=env, stdout=out, stderr=out))
    rc = 0
    for r, p in enumerate(procs):
        o, e = p.communicate()
        if p.returncode != 0 and r != 0:
            sys.stderr.write(f"rank {r} exited {p.returncode}\n")
            if e:
                sys.stderr.write(e.decode(errors="replace")[-4000:])
        rc = max(rc, p.returncode)
    return rc


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# The sources each profiled kernel is built from (its traffic entry is valid
# while their digest is the one the counters were taken on).
KERNEL_SOURCES = {
    "bwd_main": ["common.cuh", "tc.h", "tc_bwd.cu", "tc_common.cuh", "tc_ptx.cuh"],
    "fwd": ["common.cuh", "tc.h", "tc_fwd.cu", "tc_common.cuh", "tc_ptx.cuh"],
    "decode": ["common.cuh", "decode.cu", "tc_common.cuh", "tc_ptx.cuh"],
    "bwd_main_d128": ["common.cuh", "tc.h", "tc_bwd128.cu", "tc_common.cuh", "tc_ptx.cuh"],
}


def kernel_sources(stage):
    csrc = os.path.join(ROOT, "attention_sink_softmax_gb300", "csrc")
    return [os.path.join(csrc, f) for f in KERNEL_SOURCES[stage]]


def profiled_traffic(kernel_source, stage, workload):
    """DRAM traffic per launch of a stage's kernel(s) on a workload, from the
    committed ncu summary, if the kernel's source is unchanged since it was
    captured; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel_source)
    with open(path, encoding="utf-8") as f:
        for line in f:
            if not line.startswith("| "):
                continue
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            # | stage | workload | source digest | bytes per launch | ...
            if len(cells) >= 4 and cells[0] == stage and cells[1] == workload and cells[2] == digest:
                try:
                    return float(cells[3])
                except ValueError:
                    return None
    return None


# ----------------------------------------------------------------------------- CPU oracle timing
def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the machine)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return platform.machine()


def oracle_single_core_config0() -> dict:
    """The oracle's fp64 forward + backward of workload 0 (the whole problem) on
    one host core: a fresh interpreter with OMP_NUM_THREADS=1."""
    code = ("import sys, time, json; sys.path.insert(0, %r)\n"
            "import oracle\nfrom attention_sink_softmax_gb300 import inputs\n"
            "w = inputs.workload(0); p = inputs.make_inputs(w)\n"
            "kw = dict(scale=1 / 8, causal=True, window=0)\n"
            "best = 1e9\n"
            "for _ in range(5):\n"
            "    t = time.perf_counter()\n"
            "    oracle.forward(p['q'], p['k'], p['v'], p['sinks'], **kw)\n"
            "    oracle.backward(p['q'], p['k'], p['v'], p['sinks'], p['dout'], **kw)\n"
            "    best = min(best, time.perf_counter() - t)\n"
            "print(json.dumps({'seconds': best, 'threads': oracle.num_threads()}))\n") % ROOT
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                             env=env, timeout=300)
        d = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"error": f"{type(e).__name__}"}
    w = inputs.workload(0)
    f = sum(flops_of(w, w.window))
    return {"seconds": d["seconds"], "cores": d["threads"], "tflops": f / d["seconds"] / 1e12,
            "workload": w.name, "note": "best of 5, whole problem, fp64 forward + backward"}


def time_oracle(w, prob, window, budget_s=20.0, heads=None):
    """fp64 oracle fwd+bwd on a bounded sample: batch/sequence 0, the query heads
    of key/value head 0 (or ``heads`` of them), all rows. Returns a dict."""
    import oracle
    g = w.h_q // w.h_kv
    nh = heads or g
    if w.packed:
        cu = prob["cu_seqlens"]
        a, e = int(cu[0]), int(cu[1])
        q, k, v, do = (prob[n][a:e] for n in ("q", "k", "v", "dout"))
        L = e - a
    else:
        q, k, v, do = (prob[n][0] for n in ("q", "k", "v", "dout"))
        L = w.seqlen
    q, do = q[:, :nh], do[:, :nh]
    k, v = k[:, :1], v[:, :1]
    s = prob["sinks"][:nh]
    kw = dict(scale=w.scale if w.scale else 1 / math.sqrt(w.head_dim), causal=w.causal, window=window)
    t0 = time.perf_counter()
    oracle.forward(q, k, v, s, **kw)
    oracle.backward(q, k, v, s, do, **kw)
    dt = time.perf_counter() - t0
    sw = inputs.Workload("sample", 1, L, nh, 1, w.head_dim, w.dtype, w.causal, window, 0)
    f_fwd, f_bwd = flops_of(sw, window)
    return {"seconds": dt, "flops": f_fwd + f_bwd, "cores": oracle.num_threads(),
            "sample": f"sequence 0 (length {L}), query heads 0..{nh - 1} of key/value head 0, "
                      f"all rows, fp64 forward + backward",
            "value": (f_fwd + f_bwd) / dt / 1e12}


def run_reference(args, w, window):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    prob = inputs.make_inputs(w)
    for _ in range(args.warmup):
        time_oracle(w, prob, window, heads=1)
    times, flops, info = [], 0, None
    for _ in range(args.steps):
        info = time_oracle(w, prob, window, heads=1)
        times.append(info["seconds"])
        flops = info["flops"]
    ms = 1000 * sum(times) / len(times)
    value = flops / (ms / 1000) / 1e12
    full = sum(flops_of(w, window))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, window, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info["cores"],
                         "kind": "oracle", "sample": info["sample"], "cpu_model": cpu_model(),
                         "sample_fraction_of_step": flops / full,
                         "ms_per_full_step_at_this_rate": ms * full / flops},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, rank)


# ----------------------------------------------------------------------------- GPU arm
def run_e2e(args, ws, dev, stream, side, prob_host, q, k, v, sinks, dout, cu, p, o, o_lo, lse, dq,
            dk, dv, dsinks, delta, work_f, work, flops_step):
    """Same step through the public API with pinned host buffers: every step's
    inputs are copied in and every output copied back inside the timed region,
    as a training loop runs it: the next step's inputs are copied in on one
    stream and the previous step's outputs copied out on another while the
    current step computes (device buffers double-buffered, events order the
    reuse). Timed from the first copy in to the last copy out.

    The backward is the one-call sink_attn_bwd_ex (--overlap-e2e puts its
    preparation on the side stream as the device-timed loop does). The step
    is bound by the host link here: 742 MB of copies a step at about
    190-200 GB/s each way take about as long as the 4 ms of compute, so the
    overlapped preparation gains nothing, and a run whose host memory is
    busy with other work comes out slower. copy_gbs_alone gives the link's
    rate for these buffers, measured outside the timed region."""
    import attention_sink_softmax_gb300 as sa
    host_in = {n: prob_host[n].pin_memory() for n in ("q", "k", "v", "sinks", "dout")}
    outs0 = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "dsinks": dsinks}
    if o_lo is not None:
        outs0["o_lo"] = o_lo
    host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs0.items()}
    ins0 = {"q": q, "k": k, "v": v, "sinks": sinks, "dout": dout}
    dev_in = [ins0, {n: torch.empty_like(t) for n, t in ins0.items()}]
    dev_out = [outs0, {n: torch.empty_like(t) for n, t in outs0.items()}]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def copy_rate(stream_, pairs, nbytes):
        # one set of copies alone (outside the timed region), best of three:
        # the link's rate for these pinned buffers, to read the end-to-end
        # time against
        best = 0.0
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream_):
                a.record(stream_)
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
                b.record(stream_)
            b.synchronize()
            best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
        return best

    torch.cuda.synchronize(dev)
    h2d_gbs = copy_rate(s_in, [(dev_in[1][n], t) for n, t in host_in.items()], h2d)
    d2h_gbs = copy_rate(s_out, [(host_out[n], t) for n, t in dev_out[0].items()], d2h)
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]
    bwd_done = ev()
    bwd_done.record(stream)

    def e2e_step(i):
        b = i % 2
        din, dout_ = dev_in[b], dev_out[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])  # step i-2 has finished reading these inputs
            for n, t in host_in.items():
                din[n].copy_(t, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if used[b]:
            stream.wait_event(out_done[b])  # step i-2's outputs have been copied out
        if "o_lo" in dout_:
            sa.sink_attn_fwd_ex(din["q"], din["k"], din["v"], din["sinks"], cu, out=dout_["o"],
                                o_lo=dout_["o_lo"], lse=dout_["lse"], workspace=work_f, params=p,
                                stream=stream)
            if args.serial_prepare or not args.overlap_e2e:
                sa.sink_attn_bwd_ex(din["q"], din["k"], din["v"], din["sinks"], dout_["o"],
                                    dout_["o_lo"], dout_["lse"], din["dout"], cu, dq=dout_["dq"],
                                    dk=dout_["dk"], dv=dout_["dv"], dsinks=dout_["dsinks"],
                                    workspace=work, params=p, stream=stream)
            else:
                # the preparation beside the forward (q, k copied in; the last
                # backward, the workspace's previous user, done)
                side.wait_event(in_ready[b])
                side.wait_event(bwd_done)
                sa.sink_attn_bwd_prepare(p, din["q"], din["k"], workspace=work, stream=side)
                prepared = ev()
                prepared.record(side)
                sa.sink_attn_bwd_preprocess_ex(p, din["sinks"], dout_["o"], dout_["o_lo"],
                                               dout_["lse"], din["dout"], delta=delta,
                                               dsinks=dout_["dsinks"], workspace=work,
                                               stream=stream)
                stream.wait_event(prepared)
                sa.sink_attn_bwd_main(p, din["q"], din["k"], din["v"], dout_["lse"], delta,
                                      din["dout"], cu, dq=dout_["dq"], dk=dout_["dk"],
                                      dv=dout_["dv"], workspace=work, stream=stream, prepared=True)
                bwd_done.record(stream)
        else:
            sa.sink_attn_fwd(din["q"], din["k"], din["v"], din["sinks"], cu, out=dout_["o"],
                             lse=dout_["lse"], workspace=work_f, params=p, stream=stream)
            sa.sink_attn_bwd(din["q"], din["k"], din["v"], din["sinks"], dout_["o"], dout_["lse"],
                             din["dout"], cu, dq=dout_["dq"], dk=dout_["dk"], dv=dout_["dv"],
                             dsinks=dout_["dsinks"], workspace=work, params=p, stream=stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for n, t in dout_.items():
                host_out[n].copy_(t, non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    e2e_value = aggregate_value(flops_step, ws, ms_e2e)
    # the outputs that came back are the device's (spot check of the last copy)
    torch.testing.assert_close(host_out["dsinks"], dev_out[(args.steps - 1) % 2]["dsinks"].cpu(),
                               rtol=0, atol=0)
    return {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
            "overlap": "copies in and out on their own streams, overlapping the neighbouring steps' compute",
            "bwd": ("sink_attn_bwd_prepare on the side stream, then sink_attn_bwd_main"
                    if args.overlap_e2e and not args.serial_prepare and "o_lo" in dev_out[0]
                    else "one sink_attn_bwd call"),
            "copy_gbs_alone": {"h2d": h2d_gbs, "d2h": d2h_gbs}}



def check_step_outputs(sa, p, q, k, v, sinks, dout, cu, o, lse, dq, dk, dv, dsinks, stream):
    """The last timed step's outputs against one step run on the one stream
    with fresh buffers: O, LSE, dK, dV and dS_h bit for bit, dQ (fp32 reduce-adds
    in a varying order) within 2e-2 plus two ulps of its dtype. Guards the
    timed step's concurrency (the preparation beside the forward)."""
    with torch.cuda.stream(stream):
        if q.dtype == torch.bfloat16:
            o2, o_lo2, lse2 = sa.sink_attn_fwd_ex(q, k, v, sinks, cu, params=p)
            dq2, dk2, dv2, ds2 = sa.sink_attn_bwd_ex(q, k, v, sinks, o2, o_lo2, lse2, dout, cu,
                                                     params=p)
        else:
            o2, lse2 = sa.sink_attn_fwd(q, k, v, sinks, cu, params=p)
            dq2, dk2, dv2, ds2 = sa.sink_attn_bwd(q, k, v, sinks, o2, lse2, dout, cu, params=p)
    torch.cuda.synchronize()
    for name, a, b in (("o", o, o2), ("lse", lse, lse2), ("dk", dk, dk2), ("dv", dv, dv2),
                       ("dsinks", dsinks, ds2)):
        if not torch.equal(a, b):
            raise RuntimeError(f"timed step's {name} differs from a one-stream step")
    # two runs of the fused backward differ by the order of their fp32 dQ
    # reduce-adds, which can move a bf16 result by an ulp or two
    a, b = dq.float(), dq2.float()
    ulp = torch.ldexp(torch.ones_like(b), torch.frexp(b)[1] - (8 if dq.dtype == torch.bfloat16 else 24))
    if ((a - b).abs() - (2e-2 + 2 * ulp)).max().item() > 0:
        raise RuntimeError("timed step's dq differs from a one-stream step")


def overlaps_preparation(serial_prepare: bool, window: int) -> bool:
    """Whether the step issues the backward's preparation beside the forward
    on the lower-priority stream. Only where the forward outlasts it: on the
    window-128 layers the one-stream order measured faster (1.293 -> 1.276 ms
    at B 4 x N 8192; 8.27 -> 7.96 ms on the 48 packed sequences), the short
    forward leaving the preparation to run into the preprocess."""
    return not serial_prepare and not (0 < window <= 256)


def run_gpu(args, w, window):
    import attention_sink_softmax_gb300 as sa

    ws, rank, local = dist_env()
    init_dist(ws, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # the step's stream outranks the one the backward preparation runs on, so
    # the preparation's blocks only take SMs the forward leaves idle
    stream = torch.cuda.Stream(dev, priority=-1)
    side = torch.cuda.Stream(dev, priority=0)

    prob_host = inputs.make_inputs(w, seed=rank_seed(w, rank))
    d = {k: (v.to(dev) if v is not None else None) for k, v in prob_host.items()}
    q, k, v, sinks, dout, cu = d["q"], d["k"], d["v"], d["sinks"], d["dout"], d["cu_seqlens"]
    p = sa.make_params(q, k, cu, max_seqlen=w.seqlen, causal=w.causal, window=window,
                       softmax_scale=w.scale)
    o = torch.empty_like(q)
    o_lo = torch.empty_like(q) if q.dtype == torch.bfloat16 else None
    lse = torch.empty(p.h_q, p.total_tokens, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsinks = torch.empty_like(sinks)
    delta = torch.empty(p.h_q, p.total_tokens, dtype=torch.float32, device=dev)
    # the forward's and the backward's workspaces are separate buffers: the
    # backward's preparation writes its workspace while the forward runs
    work_f = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=dev)
    work = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device=dev)

    bwd_done = torch.cuda.Event()
    bwd_done.record(stream)
    overlap = overlaps_preparation(args.serial_prepare, window)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if o_lo is not None:
            sa.sink_attn_fwd_ex(q, k, v, sinks, cu, out=o, o_lo=o_lo, lse=lse, workspace=work_f,
                                params=p, stream=stream)
        else:
            sa.sink_attn_fwd(q, k, v, sinks, cu, out=o, lse=lse, workspace=work_f, params=p,
                             stream=stream)
        if overlap:
            # q and k are the step's inputs; the workspace's last user is the
            # previous step's backward
            side.wait_event(bwd_done)
            sa.sink_attn_bwd_prepare(p, q, k, workspace=work, stream=side)
            prepared = torch.cuda.Event()
            prepared.record(side)
        if ev is not None:
            ev[1].record(stream)
        if o_lo is not None:
            sa.sink_attn_bwd_preprocess_ex(p, sinks, o, o_lo, lse, dout, delta=delta,
                                           dsinks=dsinks, workspace=work, stream=stream)
        else:
            sa.sink_attn_bwd_preprocess(p, sinks, o, lse, dout, delta=delta, dsinks=dsinks,
                                        workspace=work, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        if overlap:
            stream.wait_event(prepared)
        sa.sink_attn_bwd_main(p, q, k, v, lse, delta, dout, cu, dq=dq, dk=dk, dv=dv,
                              workspace=work, stream=stream, prepared=overlap)
        if ev is not None:
            ev[3].record(stream)
        bwd_done.record(stream)

    def check_flags(when):
        for buf in (work_f, work):
            st, flags = sa.sink_attn_fetch_device_error(buf)
            if st != 0:
                raise RuntimeError(f"device flagged an error {when}: status {st}, flags {flags}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check_flags("during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = sa.sink_attn_kernel_launches()
    torch.cuda.synchronize(dev)
    barrier(ws)
    with Clocks(local) as clk:
        torch.cuda.synchronize(dev)
        clk.mark_start()
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    barrier(ws)
    launches = sa.sink_attn_kernel_launches() - launches0
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, ws, dev)
    stage_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / args.steps for j in range(3)]
    check_flags("in the timed steps")
    check_step_outputs(sa, p, q, k, v, sinks, dout, cu, o, lse, dq, dk, dv, dsinks, stream)

    f_fwd, f_bwd = flops_of(w, window)
    flops_step = f_fwd + f_bwd
    value = aggregate_value(flops_step, ws, ms)

    # ---- end to end through the public API with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, ws, dev, stream, side, prob_host, q, k, v, sinks, dout, cu, p, o, o_lo,
                      lse, dq, dk, dv, dsinks, delta, work_f, work, flops_step)

    pk, pk_src = peaks()
    # per-stage rates: FLOP/s (backward also without the S recompute, 8 d per
    # pair) and algorithmic bytes/s
    nbytes = bytes_of(w)
    f_bwd_norecompute = f_bwd * 8 // 10
    names = ("fwd", "bwd_preprocess", "bwd_main")
    stage_rates = {n: {"gb_per_s": nbytes[n] / (stage_ms[j] / 1000) / 1e9} for j, n in enumerate(names)}
    stage_rates["fwd"]["tflops"] = f_fwd / (stage_ms[0] / 1000) / 1e12
    bwd_ms = stage_ms[1] + stage_ms[2]
    stage_rates["bwd"] = {"tflops": f_bwd / (bwd_ms / 1000) / 1e12,
                          "tflops_no_recompute": f_bwd_norecompute / (bwd_ms / 1000) / 1e12,
                          "gb_per_s": (nbytes["bwd_preprocess"] + nbytes["bwd_main"]) / (bwd_ms / 1000) / 1e9}
    # dominant stage: the backward main loop (sink_attn_bwd_main), timed inside the step loop.
    # It is tensor-bound unless its arithmetic intensity is below the ridge point
    # (the short-window layers), then HBM-bound.
    main_ms = stage_ms[2]
    main_tflops = f_bwd / (main_ms / 1000) / 1e12
    # the 64-wide backward is one kernel; at d = 128 it is the dQ and dK/dV kernels
    # (their traffic entry is the sum of one launch of each)
    stage = "bwd_main" if w.head_dim == 64 else "bwd_main_d128"
    traffic = (profiled_traffic(kernel_sources(stage), stage, w.name) if stage in KERNEL_SOURCES
               else None)
    # The step lasts milliseconds and draws far below the power cap, so the
    # denominator is the burst bf16 peak (a GEMM timed alone); the sustained
    # figure (seconds-long loop under the power cap) is given beside it.
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if f_bwd / nbytes["bwd_main"] >= ridge:
        roofline = {"bound": "tensor", "achieved": main_tflops,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": main_tflops / pk["bf16_tflops"], "traffic": traffic,
                    "kernel": "sink_attn_bwd_main", "peak_kind": f"bf16 burst ({pk_src})",
                    "frac_of_sustained": main_tflops / pk["bf16_tflops_sustained"]}
    else:
        main_gbs = stage_rates["bwd_main"]["gb_per_s"]
        roofline = {"bound": "hbm", "achieved": main_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": main_gbs / pk["hbm_gbs"], "traffic": traffic,
                    "kernel": "sink_attn_bwd_main", "peak_kind": f"HBM copy ({pk_src})",
                    "algorithmic_bytes": nbytes["bwd_main"]}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": config_of(w, window, ws),
        "pct_of_peak": {"burst": 100 * value / ws / pk["bf16_tflops"],
                        "sustained": 100 * value / ws / pk["bf16_tflops_sustained"],
                        "source": pk_src, "headline": "burst"},
        "stages_ms": {"fwd": stage_ms[0], "bwd_preprocess": stage_ms[1], "bwd_main": stage_ms[2]},
        "bwd_prepare": ("inside sink_attn_bwd_main" if not overlap or w.head_dim != 64
                        or w.dtype != torch.bfloat16 else
                        "sink_attn_bwd_prepare on a lower-priority stream beside the forward"),
        "stage_rates": stage_rates,
        "clocks": clk.summary(),
        "e2e": e2e,
        "gpu_launches": int(launches),
        "roofline": roofline,
    }
    if rank == 0 and not args.no_cpu_baseline:
        info = time_oracle(w, prob_host, window)
        line["cpu_baseline"] = {"value": info["value"], "unit": "TFLOP/s", "cores": info["cores"],
                                "kind": "oracle", "sample": info["sample"],
                                "seconds": info["seconds"], "cpu_model": cpu_model(),
                                "single_core_config0": oracle_single_core_config0()}
    emit(line, rank)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_decode(args):
    """Decode (one newest token per sequence against its KV cache): bandwidth of
    sink_attn_decode on the decode workload, device-timed, one JSON line. Not
    the headline metric; the roofline is HBM (the cache is read once)."""
    import attention_sink_softmax_gb300 as sa

    ws_, rank, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    w = inputs.decode_workload()
    d = inputs.make_decode_inputs(w, device=str(dev))
    p = sa.make_decode_params(d["q"], d["k"], max_seqlen=w.ctx, window=w.window, softmax_scale=w.scale)
    work = torch.empty(sa.sink_attn_decode_workspace_bytes(p), dtype=torch.uint8, device=dev)
    o = torch.empty_like(d["q"])
    lse = torch.empty(w.h_q, w.batch, dtype=torch.float32, device=dev)

    def step(st=stream):
        sa.sink_attn_decode(d["q"], d["k"], d["v"], d["sinks"], d["kv_start"], d["kv_len"], params=p,
                            out=o, lse=lse, workspace=work, stream=st)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    # A serving loop issues decode steps from a captured graph: capture a run
    # of calls once and replay it, so the timing is the device's, not the
    # host's per-call marshalling.
    per_graph = 20
    graph, launch = None, "eager"
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            cs = torch.cuda.current_stream(dev)
            for _ in range(per_graph):
                step(cs)
        torch.cuda.synchronize(dev)
        launch = f"CUDA graph of {per_graph} calls, replayed"
    except Exception as e:  # time the calls one by one instead
        graph, launch = None, f"eager (graph capture failed: {type(e).__name__})"
    reps = max(1, (200 * args.steps + per_graph - 1) // per_graph)  # about a second: clocks get sampled
    steps = reps * per_graph
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph is not None:
        graph.replay()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark_start()
        start.record(stream)
        for _ in range(reps):
            if graph is not None:
                graph.replay()
            else:
                for _ in range(per_graph):
                    step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    st, flags = sa.sink_attn_fetch_device_error(work)
    if st != 0:
        raise RuntimeError(f"device flagged an error: status {st}, flags {flags}")
    ms = start.elapsed_time(end) / steps
    esz = d["q"].element_size()
    cache = 2 * w.cache_tokens * w.h_kv * w.head_dim * esz  # K and V, each read once
    qo = 2 * w.batch * w.h_q * w.head_dim * esz + 4 * w.h_q * w.batch
    gbs = (cache + qo) / (ms / 1000) / 1e9
    pk, pk_src = peaks()
    line = {
        "metric": "sink-attention decode bandwidth (bf16 KV cache read once)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "context": w.ctx, "h_q": w.h_q, "h_kv": w.h_kv,
                   "head_dim": w.head_dim, "window": w.window, "bytes_per_step": cache + qo,
                   "l2": "KV cache exceeds L2 (no flush)", "launch": launch},
        "clocks": clk.summary(),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": profiled_traffic(kernel_sources("decode"), "decode", w.name),
                     "kernel": "decode_mma_kernel",
                     "peak_kind": f"HBM copy ({pk_src})"},
    }
    emit(line, rank)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=1, help="workload index 0..5")
    ap.add_argument("--window", type=int, default=None, help="override the workload's window")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (padded workloads only): a smaller "
                         "case of the same layer, e.g. for profiler captures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--overlap-e2e", action="store_true",
                    help="end-to-end timing with the backward's preparation on the side stream "
                         "(default: the one-call backward; the host link bounds that step)")
    ap.add_argument("--serial-prepare", action="store_true",
                    help="run the backward preparation inside sink_attn_bwd_main on the step's "
                         "stream on every layer (by default it runs beside the forward on a "
                         "lower-priority stream, except with a window of at most 256 keys)")
    ap.add_argument("--decode", action="store_true",
                    help="measure the decode path (KV-cache bandwidth) instead of the training step")
    args = ap.parse_args()
    w = inputs.workload(args.config)
    if args.batch is not None:
        if w.packed or args.batch < 1:
            sys.exit("--batch takes a positive batch for a padded workload")
        w = dataclasses.replace(w, batch=args.batch,
                                name=w.name.replace(f"_B{w.batch}_", f"_B{args.batch}_"))
    window = w.window if args.window is None else args.window
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # no launcher: one process per GPU, started here
        if args.impl == "gb300" or args.decode:
            have = torch.cuda.device_count()
            if have < args.gpus:
                sys.exit(f"bench.py --gpus {args.gpus}: only {have} GPU(s) visible")
        sys.exit(spawn_ranks(args.gpus, [sys.executable, os.path.abspath(__file__)] + sys.argv[1:]))
    if args.decode:
        run_decode(args)
    elif args.impl == "reference":
        run_reference(args, w, window)
    else:
        run_gpu(args, w, window)


if __name__ == "__main__":
    main()
