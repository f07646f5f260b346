"""Benchmark: paged decode attention KV GB/s at Qwen3-4B heads on GB300.

One step = one pass of the whole hot path on one layer's caches: slot
mapping of the step's new rows, their append into the paged caches, and
attention of every query row through the block tables.  The default
workload is the Qwen3-4B decode step (batch 64, contexts uniform in
[512, 4096], 32 query heads, 8 KV heads, head dim 128, block size 16,
bf16, a shuffled pool of 20,000 blocks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
plain fp64 definition) on the host cores, on a bounded sample of the same
workload.  With N > 1 (torchrun), every rank runs its own replica of the
workload on its own GPU (no data exchange; weak scaling) and the slowest
rank's time counts.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_mapping_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s & % of GB300 HBM peak (Qwen3-4B heads, bs 64)"
UNIT = "GB/s"
WORKLOADS = ("decode", "layout-bs1-scattered", "layout-bs1-contiguous", "layout-bs16-scattered",
             "layout-bs16-contiguous", "layout-bs64-scattered", "layout-bs64-contiguous", "mixed",
             "mixed-chunks", "mixed-fp8", "mixed-chunks-fp8", "long-fp8", "lognormal-fp8")
DECODE_SOURCES = ["pkv_decode.cu", "pkv_pipeline.cuh", "pkv_common.cuh"]
PREFILL_SOURCES = ["pkv_prefill_tc.cu", "pkv_common.cuh"]


# ------------------------------------------------------------------ accounting
def step_bytes(wl, out_bytes=2, window_left=-1):
    """Algorithmic bytes of one step: attention reads each sequence's N_s K
    and V rows once per KV head plus Q and writes O; the append reads the new
    K/V rows and writes them into the caches; the slot step and the tables
    are listed separately.  With a sliding window a decoding row needs only
    the last window_left + 1 keys."""
    eb = {"f32": 4, "bf16": 2, "e4m3": 1}[wl.kv]
    sb = 4 if wl.src == "f32" else 2
    kv = wl.kv_bytes_read()
    if window_left >= 0:
        if int(wl.q_lens.max()) > 1:
            raise ValueError("window byte accounting is for decode workloads")
        n = wl.seq_lens[wl.q_lens > 0].astype(np.int64)
        kv = int(np.minimum(n, window_left + 1).sum()) * wl.Hkv * wl.D * eb * 2
    q = wl.T * wl.Hq * wl.D * sb
    o = wl.T * wl.Hq * wl.D * out_bytes
    app = wl.T * wl.Hkv * wl.D * 2 * (sb + eb)
    tables = int(sum(-(-int(n) // wl.block_size) for n in wl.seq_lens)) * 4 + wl.B * 8
    return {"attention": kv + q + o, "kv": kv, "q": q, "o": o, "append": app, "tables": tables,
            "total": kv + q + o + app}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != source_hash(DECODE_SOURCES):
        return None
    return rec


def source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_mapping_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """SM clocks, power and clock-event (throttle) reasons sampled while the
    timed regions run: NVML read through ctypes every millisecond from a
    thread (nothing is set, only read), else nvidia-smi every 100 ms.  Only
    samples taken while the sampler is armed count; arm() takes one sample at
    once and disarm() one more, so that a timed region of a few milliseconds
    still carries samples."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index, interval=0.001):
        self.gpu = gpu_index
        self.interval = interval
        self.rows = []  # (sm_mhz, max_mhz, power_w, reasons_mask)
        self.source = None
        self.proc = None
        self.thread = None
        self.armed = False
        self.regions = 0

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        idx = self.gpu
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        if vis and all(x.strip().isdigit() for x in vis.split(",")):
            idx = int(vis.split(",")[self.gpu])
        if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex failed")
        return lib, h

    def _sample(self):
        import ctypes
        lib, h = self.lib, self.h
        sm, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0  # NVML_CLOCK_SM
        lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
        if lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) != 0:
            lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(rs))
        if ok:
            self.rows.append((float(sm.value), float(self.max_mhz), mw.value / 1000.0, int(rs.value)))

    def _poll(self):
        while not self.stop:
            if self.armed:
                self._sample()
            time.sleep(self.interval)

    def __enter__(self):
        import ctypes
        import threading
        self.stop = False
        try:
            self.lib, self.h = self._nvml()
            mx = ctypes.c_uint()
            self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            self.source = f"nvml {self.interval * 1e3:g} ms"
        except (OSError, AttributeError, IndexError, ValueError):
            self.thread = None
            try:
                self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", "100"],
                                             stdout=self.f, stderr=subprocess.DEVNULL)
                self.source = "nvidia-smi 100 ms (whole run)"
            except (OSError, FileNotFoundError):
                self.proc = None
        return self

    def arm(self):
        self.regions += 1
        if self.thread is not None:
            self._sample()
        self.armed = True

    def disarm(self):
        if self.thread is not None and self.armed:
            self._sample()
        self.armed = False

    def __exit__(self, *a):
        self.armed = False
        if self.thread is not None:
            self.stop = True
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            with open(self.path) as f:
                lines = f.read().splitlines()
            os.remove(self.path)

            def num(x):
                try:
                    return float(x)
                except ValueError:
                    return None
            for line in lines:
                r = [x.strip() for x in line.split(",")]
                if len(r) >= 9 and num(r[1]) is not None:
                    mask = sum(self.BITS[n] for i, n in enumerate(names) if r[5 + i].lower() == "active")
                    self.rows.append((num(r[1]), num(r[2]) or 0.0, num(r[3]) or 0.0, mask))

    def summary(self):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": self.source}
        reasons = sorted(n for n, b in self.BITS.items() if any(r[3] & b for r in self.rows))
        return {"sm_mhz": statistics.median(r[0] for r in self.rows),
                "sm_max_mhz": max(r[1] for r in self.rows), "reasons": reasons, "samples": len(self.rows),
                "timed_regions": self.regions, "power_w_max": round(max(r[2] for r in self.rows), 1),
                "source": self.source}


# ------------------------------------------------------------------ ranks
def job_rate(ms_step, step_bytes, world, device):
    """Whole-job throughput over ranks that each run their own replica: the
    bytes all ranks move in one step over the slowest rank's step time.
    Returns (slowest ms per step, GB/s)."""
    total = float(step_bytes)
    if world > 1:
        import torch
        import torch.distributed as dist
        tm = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
        tb = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(tm, op=dist.ReduceOp.MAX)
        dist.all_reduce(tb, op=dist.ReduceOp.SUM)
        ms_step, total = float(tm.item()), float(tb.item())
    return ms_step, total / (ms_step * 1e-3) / 1e9


# ------------------------------------------------------------------ our arm
# Layers of one Qwen3-4B decode step.  The pages plan a step once and reuse
# the plan for the attention of every layer ("How Easy Is It to Start
# Serving LLMs?", "3. Load balancing: keep every SM busy"); the slot mapping
# is likewise made once per step.  A benchmark step is one layer.
LAYERS_PER_MODEL_STEP = 36


def layer_loop(ds, steps, layers, on_run=None):
    """steps consecutive layer steps from the start of a model step: slot
    mapping and plan at every model-step boundary, then append + attention
    run of the layer (on_run(i, fn) wraps the attention run, e.g. with
    events)."""
    from paged_kv_cache_mapping_gb300 import pkv_append
    wl = ds.wl
    for i in range(steps):
        if i % LAYERS_PER_MODEL_STEP == 0:
            ds.model_step_start()
        layer = i % layers
        kc, vc = ds.caches[layer]
        pkv_append(ds.k_new, ds.v_new, ds.slots, kc, vc, wl.k_scale, wl.v_scale)
        if on_run is None:
            ds.run(layer)
        else:
            on_run(i, lambda: ds.run(layer))


def timed_runs(ds, steps, layers, stream):
    """The attention run alone, with CUDA events on the launching stream
    around each call, inside the layer loop; returns ms per call."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def on_run(i, fn):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    layer_loop(ds, steps, layers, on_run)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def run_ours(args, rank, world):
    import torch

    from paged_kv_cache_mapping_gb300 import harness, pkv_device_errors

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    LAYERS = args.layers
    wl = make_workload(args.workload, rank)
    max_q = int(wl.q_lens.max())
    ds = harness.DeviceStep(wl, device=dev, out_dtype=torch.bfloat16, layers=LAYERS, max_q_len=max_q,
                            soft_cap=args.soft_cap, window_left=args.window_left)
    torch.cuda.synchronize()
    if pkv_device_errors(dev) != 0:
        raise RuntimeError("device error flags set during set-up")
    nb = step_bytes(wl, window_left=args.window_left)
    stream = torch.cuda.current_stream(dev)

    layer_loop(ds, args.warmup, LAYERS)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    with ClockSampler(dev.index) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        clk.arm()
        t_start.record(stream)
        layer_loop(ds, args.steps, LAYERS)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.disarm()
        flags = pkv_device_errors(dev)
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} in the timed region")
        ms_step = t_start.elapsed_time(t_end) / args.steps
        # The attention run alone, for the roofline: the same steps again with
        # events around each run (an event recorded between two launches keeps
        # the second from starting before the first ends, so these events stay
        # out of the step loop above, whose kernels overlap their neighbours'
        # launch and set-up); and the runs back to back over the same plan and
        # layer caches with events at the two ends only, which is the decode
        # kernel's launch rate when a model step reuses the plan for its layers.
        clk.arm()
        attn_ms = timed_runs(ds, args.steps, LAYERS, stream)
        clk.disarm()
        ds.model_step_start()
        for i in range(LAYERS):
            ds.run(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.arm()
        a.record(stream)
        for i in range(args.steps):
            ds.run(i % LAYERS)
        b.record(stream)
        torch.cuda.synchronize()
        clk.disarm()
        run_ms = a.elapsed_time(b) / args.steps
        # The step as it was before plan reuse: slot mapping, append and the
        # whole call (plan + run) in every step.
        clk.arm()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.steps):
            ds.step(i % LAYERS)
        b.record(stream)
        torch.cuda.synchronize()
        clk.disarm()
        ms_planned = a.elapsed_time(b) / args.steps
        flags = pkv_device_errors(dev)
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} in the attention timing passes")

        if world > 1:
            torch.distributed.barrier()
        # slowest rank, every rank's bytes
        ms_step, value = job_rate(ms_step, nb["total"], world, dev)
        _, value_planned = job_rate(ms_planned, nb["total"], world, dev)

        e2e = run_e2e(ds, wl, nb, args, dev, world, max_q, clk)
        graph = run_graph(ds, nb, args, dev, world, clk)
        secondary = None
        if rank == 0 and world == 1 and args.workload == "decode" and not args.no_secondary:
            del ds
            torch.cuda.empty_cache()
            secondary = run_secondary(args, dev, clk)
    if rank != 0:
        return None
    hbm, peak_kind = peaks()
    attn_avg_ms = statistics.mean(attn_ms)
    achieved = nb["attention"] / (run_ms * 1e-3) / 1e9
    achieved_ev = nb["attention"] / (attn_avg_ms * 1e-3) / 1e9
    rec = traffic_record()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64, N(0,1) rounded to bf16)",
        "config": {"workload": wl.name, "batch": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                   "block_size": wl.block_size, "num_blocks": wl.num_blocks,
                   "mean_ctx": float(wl.seq_lens.mean()), "out_dtype": "bf16",
                   "step": (f"one layer of a {LAYERS_PER_MODEL_STEP}-layer decode step: append of the layer's new "
                            f"rows + attention run over the step's plan; the slot mapping and the plan are made "
                            f"at the first layer of every model step (every {LAYERS_PER_MODEL_STEP} steps, "
                            f"step 0 included)"),
                   "l2": f"inputs larger than L2: {LAYERS} layer cache(s) rotated, "
                         f"{nb['kv'] / 1e6:.0f} MB of live KV each",
                   "bytes_per_step": nb, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   **({"variant": {"soft_cap": args.soft_cap, "window_left": args.window_left}}
                      if args.soft_cap > 0 or args.window_left >= 0 else {})},
        "roofline": {"bound": "hbm", "kernel": "pkv_attention_run (decode kernel)",
                     "achieved": round(achieved, 1), "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": rec["dram_bytes_per_launch"] if rec else None,
                     "algorithmic_bytes": nb["attention"], "avg_launch_us": round(run_ms * 1e3, 2),
                     "timing": f"{args.steps} pkv_attention_run calls back to back over one plan and the "
                               f"{LAYERS} layer caches, CUDA events on the launching stream at the two ends",
                     "per_call_events": {"avg_launch_us": round(attn_avg_ms * 1e3, 2),
                                         "achieved": round(achieved_ev, 1), "frac": round(achieved_ev / hbm, 4),
                                         "timing": "CUDA events around each run inside the layer loop (no "
                                                   "overlap with the neighbouring launches)"}},
        "plan_every_step": {"value": round(value_planned, 1), "unit": UNIT, "ms_per_step": round(ms_planned, 5),
                            "how": "slot mapping + append + pkv_attention (plan + run) in every step"},
        "e2e": e2e,
        "graph": graph,
        # per layer: append, decode (+ prefill); per model step: slot mapping, plan
        "gpu_launches": ((3 if max_q > 1 else 2) * args.steps
                         + 2 * -(-args.steps // LAYERS_PER_MODEL_STEP)),
        "clocks": clk.summary(),
    }
    if secondary is not None:
        line["configs"] = secondary
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, nb, budget_s=args.cpu_budget)
    return line


def run_graph(ds, nb, args, dev, world, clk):
    """A whole model step (slot mapping, plan, then append + run for each of
    its layers) captured into one CUDA graph after an eager warm-up and
    replayed: the launch cost of the kernels goes away.  Reported per layer
    beside the eager value, not instead of it."""
    import torch
    try:
        layers = len(ds.caches)
        L = LAYERS_PER_MODEL_STEP
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            layer_loop(ds, L, layers)
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer_loop(ds, L, layers)
        for _ in range(max(1, args.warmup // L)):
            g.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        stream = torch.cuda.current_stream(dev)
        reps = max(1, round(args.steps / L))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.arm()
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        clk.disarm()
        if world > 1:
            torch.distributed.barrier()
        ms, rate = job_rate(a.elapsed_time(b) / (reps * L), nb["total"], world, dev)
        return {"value": round(rate, 1), "unit": UNIT, "ms_per_step": round(ms, 5),
                "how": f"{reps} replay(s) of one CUDA graph holding a whole {L}-layer model step"}
    except Exception as e:  # reported, never fatal to the benchmark line
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def run_e2e(ds, wl, nb, args, dev, world, max_q, clk):
    """Same metric through the public API with host buffers: every step
    copies the step's inputs from pinned host memory and reads the output
    back.  The inputs of a step sit in one pinned staging buffer (one
    host-to-device copy); copies run on their own stream, double-buffered,
    so that step i + 1's inputs move and step i - 1's output comes back while
    step i computes.  The steps are layers of model steps as in the main
    loop: slot mapping and plan at the first layer of each."""
    import torch

    from paged_kv_cache_mapping_gb300 import (pkv_append, pkv_attention_plan, pkv_attention_run,
                                              pkv_slot_mapping)
    src = {"q": ds.q, "k": ds.k_new, "v": ds.v_new, "cu": ds.cu_q, "sl": ds.seq_lens, "bt": ds.bt}
    off, size, total = {}, {}, 0
    for k, t in src.items():
        off[k], size[k] = total, t.numel() * t.element_size()
        total += (size[k] + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k, t in src.items():
        host[off[k]:off[k] + size[k]].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [{k: buf[off[k]:off[k] + size[k]].view(t.dtype).view(t.shape) for k, t in src.items()} for buf in bufs]
    outs = [torch.empty_like(ds.out) for _ in range(2)]
    out_h = [torch.empty(ds.out.shape, dtype=ds.out.dtype).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    h2d = total
    d2h = out_h[0].numel() * out_h[0].element_size()

    def stage_in(i):
        b = i % 2
        with torch.cuda.stream(copy):
            if used[b]:
                copy.wait_event(comp_done[b])  # step i - 2 has finished with this buffer
            bufs[b].copy_(host, non_blocking=True)
            h2d_done[b].record(copy)

    def compute_and_read_back(i):
        b = i % 2
        comp.wait_event(h2d_done[b])
        d = views[b]
        kc, vc = ds.caches[i % len(ds.caches)]
        if i % LAYERS_PER_MODEL_STEP == 0:
            pkv_slot_mapping(d["cu"], d["sl"], d["bt"], wl.block_size, out=ds.slots)
            pkv_attention_plan(d["q"], d["cu"], d["sl"], d["bt"], kc, ds.ws, max_q_len=max_q,
                               window_left=args.window_left)
        pkv_append(d["k"], d["v"], ds.slots, kc, vc, wl.k_scale, wl.v_scale)
        pkv_attention_run(d["q"], d["cu"], d["sl"], d["bt"], kc, vc, wl.scale, outs[b], ds.ws, wl.k_scale,
                          wl.v_scale, max_q, soft_cap=args.soft_cap, window_left=args.window_left)
        comp_done[b].record(comp)
        used[b] = True
        with torch.cuda.stream(copy):
            copy.wait_event(comp_done[b])
            out_h[b].copy_(outs[b], non_blocking=True)

    def run(n):
        stage_in(0)
        for i in range(n):
            if i + 1 < n:
                stage_in(i + 1)
            compute_and_read_back(i)
        comp.wait_stream(copy)

    run(args.warmup)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.arm()
    a.record(comp)
    run(args.steps)
    b.record(comp)
    torch.cuda.synchronize()
    clk.disarm()
    ms = a.elapsed_time(b) / args.steps
    if not torch.equal(out_h[(args.steps - 1) % 2].to(dev), outs[(args.steps - 1) % 2]):
        raise RuntimeError("end-to-end read-back differs from the device output")
    if world > 1:
        torch.distributed.barrier()
    ms, rate = job_rate(ms, nb["total"], world, dev)
    return {"value": round(rate, 1), "unit": UNIT, "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "how": "inputs in one pinned staging buffer: one host-to-device copy and one read-back per step, "
                   "on a copy stream, double-buffered against the compute"}


# ------------------------------------------------------------------ the other workloads
def prefill_flops(wl):
    """Algorithmic FLOPs of the prefill rows: 4 * Hq * D per visible (query
    token, key) pair of every sequence with more than one query row."""
    pairs = 0
    for n, q in zip(wl.seq_lens.astype(np.int64), wl.q_lens.astype(np.int64)):
        if q > 1:
            pairs += int(q * (n - q) + q * (q + 1) // 2)
    return 4 * wl.Hq * wl.D * pairs


def time_runs(wl, dev, calls, layers=4, clk=None):
    """ms per pkv_attention_run, back to back over rotated layer caches after
    one plan (CUDA events at the two ends)."""
    import torch

    from paged_kv_cache_mapping_gb300 import harness, pkv_device_errors
    ds = harness.DeviceStep(wl, device=dev, out_dtype=torch.bfloat16, layers=layers)
    ds.model_step_start()
    for layer in range(layers):
        ds.layer_step(layer)
    for i in range(3 * layers):
        ds.run(i % layers)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.arm()
    a.record()
    for i in range(calls):
        ds.run(i % layers)
    b.record()
    torch.cuda.synchronize()
    if clk is not None:
        clk.disarm()
    if pkv_device_errors(dev):
        raise RuntimeError(f"device error flags set on {wl.name}")
    del ds
    torch.cuda.empty_cache()
    return a.elapsed_time(b) / calls


def run_secondary(args, dev, clk):
    """The other workloads of the survey, each as a secondary key of the
    bench line: the page-layout ratio, the mixed chunked-prefill step with
    the prefill's own tensor roofline, and the two fp8 workloads."""
    hbm, peak_kind = peaks()
    tflops, tflops_sus = tensor_peaks()
    out = {}
    t0 = time.time()
    try:
        out["layout"] = layout_ratio(dev, repeats=args.layout_repeats, clk=clk)
    except Exception as e:  # reported, never fatal to the benchmark line
        out["layout"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    calls = max(50, args.steps)
    for name, key in (("mixed", "mixed_prefill"), ("mixed-fp8", "mixed_prefill_fp8")):
        try:
            wl = make_workload(name)
            nb = step_bytes(wl)
            ms = time_runs(wl, dev, calls, clk=clk)
            chunks = wl.select([s for s in range(wl.B) if wl.q_lens[s] > 1])
            fl = prefill_flops(wl)
            # the prefill alone moves with where its few MB of K/V land: the
            # median over three fresh allocations
            ms_pf = statistics.median(time_runs(chunks, dev, calls, clk=clk) for _ in range(3))
            rec = prefill_record() if wl.kv == "bf16" else None
            out[key] = {
                "workload": wl.name, "call_us": round(ms * 1e3, 2),
                "kv_gbs": round(nb["attention"] / (ms * 1e-3) / 1e9, 1),
                "frac_hbm": round(nb["attention"] / (ms * 1e-3) / 1e9 / hbm, 4),
                "prefill": {"bound": "tensor", "flops": fl, "call_us": round(ms_pf * 1e3, 2),
                            "achieved": round(fl / (ms_pf * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                            "peak": tflops, "frac": round(fl / (ms_pf * 1e-3) / 1e12 / tflops, 4),
                            "frac_of_sustained": round(fl / (ms_pf * 1e-3) / 1e12 / tflops_sus, 4),
                            "tensor_pipe_active": rec.get("sm__pipe_tensor_cycles_active_pct") if rec else None,
                            "how": "the two prefill chunks alone (the tcgen05 prefill kernel and an empty decode "
                                   "launch), back-to-back runs, median of three allocations; FLOPs = 4 Hq D per "
                                   "visible (query, key) pair" + ("; f16 MMAs (the bf16 peak applies)"
                                                                  if wl.kv == "e4m3" else "")}}
        except Exception as e:
            out[key] = {"error": f"{type(e).__name__}: {e}"[:200]}
    for name in ("long-fp8", "lognormal-fp8"):
        try:
            wl = make_workload(name)
            nb = step_bytes(wl)
            ms = time_runs(wl, dev, calls, clk=clk)
            gbs = nb["attention"] / (ms * 1e-3) / 1e9
            out[name.replace("-", "_")] = {"workload": wl.name, "call_us": round(ms * 1e3, 2),
                                           "kv_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                           "algorithmic_bytes": nb["attention"]}
        except Exception as e:
            out[name.replace("-", "_")] = {"error": f"{type(e).__name__}: {e}"[:200]}
    out["peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tflops, "bf16_tflops_sustained": tflops_sus,
                    "kind": peak_kind}
    out["how"] = (f"{calls} back-to-back pkv_attention_run calls over 4 rotated layer caches after one plan, "
                  f"CUDA events at both ends; {time.time() - t0:.0f} s with set-up")
    return out


def layout_ratio(dev, repeats=2, calls=200, layers=4, clk=None):
    """Scattered against contiguous block tables on the layout workloads (B
    32 x 2048 keys, block sizes 1, 16, 64): each repeat allocates fresh
    caches for each layout (alternating which goes first) and times calls
    back-to-back runs over rotated layer caches.  Per-layout medians and
    their ratio."""
    times = {}
    wls = {}
    for r in range(repeats):
        for bs in (1, 16, 64):
            for contiguous in ((False, True) if r % 2 == 0 else (True, False)):
                key = (bs, contiguous)
                if key not in wls:
                    wls[key] = W.layout_sweep(bs, contiguous, seed=1003)
                times.setdefault(key, []).append(time_runs(wls[key], dev, calls, layers, clk) * 1e3)
    rows = []
    for bs in (1, 16, 64):
        s, c = statistics.median(times[(bs, False)]), statistics.median(times[(bs, True)])
        rows.append({"block_size": bs, "scattered_us": round(s, 2), "contiguous_us": round(c, 2),
                     "ratio": round(s / c, 4)})
    return {"ratio_max": max(r["ratio"] for r in rows), "rows": rows, "repeats": repeats,
            "workload": "layout B32 ctx2048, Qwen3-4B heads, bf16, block sizes 1/16/64"}


def tensor_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))
    return 1900.0, 1700.0


def prefill_record():
    """The tensor-core prefill kernel's ncu figures, if they were taken on its
    current source."""
    path = os.path.join(ROOT, "profiles", "prefill_tc_record.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != source_hash(PREFILL_SOURCES):
        return None
    return rec


# ------------------------------------------------------------------ oracle
def cpu_baseline(wl, nb, budget_s=20.0, nthreads=None, single_budget_s=6.0):
    """The oracle as it stands, on the host cores: its cache is built once
    (untimed), then whole steps (slot mapping, append of the new rows,
    attention of every row) are timed with all the cores until the budget is
    spent.  The same oracle on one thread is timed on a sample of the step's
    (token, head) rows (its attention is over rows, so a sample scales to the
    whole step by rows), with the full slot mapping and append."""
    import oracle

    nthreads = nthreads or oracle.cpu_count()
    kc = np.zeros(wl.cache_shape(), wl.cache_np_dtype())
    vc = np.zeros_like(kc)
    for s0, s1, cu, sl, k, v in wl.history_batches():
        if k.shape[0]:
            oracle.append(k, v, oracle.slot_mapping(cu, sl, wl.block_tables[s0:s1], wl.block_size),
                          kc, vc, wl.k_scale, wl.v_scale)
    kn, vn = wl.new_rows()
    times = []
    t_begin = time.perf_counter()
    while not times or (time.perf_counter() - t_begin < budget_s and len(times) < 50):
        t0 = time.perf_counter()
        slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, wl.block_size)
        oracle.append(kn, vn, slots, kc, vc, wl.k_scale, wl.v_scale)
        oracle.attention(wl.q, wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, kc, vc, wl.scale, wl.k_scale,
                         wl.v_scale, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    per = statistics.median(times)
    # one thread: append + slot mapping in full, attention over a row sample
    n_all = wl.T * wl.Hq
    order = np.random.default_rng(4243).permutation(n_all)
    t0 = time.perf_counter()
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, wl.block_size)
    oracle.append(kn, vn, slots, kc, vc, wl.k_scale, wl.v_scale)
    t_fixed = time.perf_counter() - t0
    done, t_rows = 0, 0.0
    while done < n_all and t_rows < single_budget_s:
        sel = order[done:done + 64]
        t0 = time.perf_counter()
        oracle.attention(wl.q, wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, kc, vc, wl.scale, wl.k_scale,
                         wl.v_scale, nthreads=1, rows=(sel // wl.Hq, (sel % wl.Hq).astype(np.int32)))
        t_rows += time.perf_counter() - t0
        done += sel.shape[0]
    per_1 = t_fixed + t_rows * n_all / done
    return {"value": round(nb["total"] / per / 1e9, 3), "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{len(times)} whole steps of the same workload (all {wl.T} query rows), "
                      f"median {per * 1e3:.1f} ms per step, fp64, {nthreads} threads",
            "single_thread": {"value": round(nb["total"] / per_1 / 1e9, 4), "unit": UNIT, "cores": 1,
                              "ms_per_step": round(per_1 * 1e3, 1),
                              "sample": f"{done} of {n_all} (token, head) rows on one thread, scaled to the "
                                        f"step by rows, plus the full slot mapping and append"}}


def make_workload(name, rank=0):
    """The benchmark workloads (seeded per rank: each rank owns a replica)."""
    off = 100 * rank
    if name == "decode":
        return W.qwen3_4b_decode(seed=1002 + off)
    if name.startswith("layout-"):
        _, bs, lay = name.split("-")
        return W.layout_sweep(int(bs[2:]), lay == "contiguous", seed=1003 + off)
    if name == "mixed":
        return W.mixed_prefill(seed=1004 + off)
    if name == "mixed-chunks":  # the two prefill chunks of the mixed step alone
        wl = W.mixed_prefill(seed=1004 + off)
        return wl.select([s for s in range(wl.B) if wl.q_lens[s] > 1])
    if name == "mixed-fp8":  # the mixed step on e4m3 caches
        return W.mixed_prefill(seed=1004 + off, kv="e4m3")
    if name == "mixed-chunks-fp8":
        wl = W.mixed_prefill(seed=1004 + off, kv="e4m3")
        return wl.select([s for s in range(wl.B) if wl.q_lens[s] > 1])
    if name == "long-fp8":
        return W.long_fp8(seed=1005 + off)
    if name == "lognormal-fp8":
        return W.lognormal_fp8(seed=1006 + off)
    raise ValueError(name)


def reference_row_bytes(wl):
    """Algorithmic bytes attributed to each (token, head) query row: its
    share of its sequence's K/V rows (N_s rows per KV head, shared by the
    sequence's q_s * Hq query rows) plus its own Q and O rows."""
    eb = {"f32": 4, "bf16": 2, "e4m3": 1}[wl.kv]
    sb = 4 if wl.src == "f32" else 2
    cu = wl.cu_seqlens_q
    per_tok = np.zeros(wl.T, np.float64)
    for s in range(wl.B):
        q_s = int(wl.q_lens[s])
        if q_s:
            per_tok[cu[s]:cu[s + 1]] = float(wl.seq_lens[s]) * wl.Hkv * wl.D * eb * 2 / (q_s * wl.Hq)
    return per_tok + wl.D * (sb + 2)


def run_reference(args, rank, world, budget_s=90.0):
    """The oracle as the reference arm, on the host cores.  Its caches are
    built once (untimed, like our set-up); each step runs the oracle's slot
    mapping and append of the step's rows and its attention on a bounded,
    rotating sample of the (token, head) rows, sized so that warm-up and
    timed steps take about budget_s together.  The value is the bytes those
    rows account for (plus the append) over the time taken."""
    if rank != 0:
        return None
    import oracle

    nt = oracle.cpu_count()
    wl = make_workload(args.workload)
    nb = step_bytes(wl)
    kc = np.zeros(wl.cache_shape(), wl.cache_np_dtype())
    vc = np.zeros_like(kc)
    for s0, s1, cu, sl, k, v in wl.history_batches():
        if k.shape[0]:
            oracle.append(k, v, oracle.slot_mapping(cu, sl, wl.block_tables[s0:s1], wl.block_size),
                          kc, vc, wl.k_scale, wl.v_scale)
    kn, vn = wl.new_rows()
    n_all = wl.T * wl.Hq
    order = np.random.default_rng(4242).permutation(n_all)
    row_b = np.repeat(reference_row_bytes(wl), wl.Hq)
    # calibrate the per-row cost on a probe sample of the rows path itself
    probe = order[:min(n_all, 8 * nt)]
    t0 = time.perf_counter()
    oracle.attention(wl.q, wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, kc, vc, wl.scale, wl.k_scale,
                     wl.v_scale, nthreads=nt, rows=(probe // wl.Hq, (probe % wl.Hq).astype(np.int32)))
    per_row = (time.perf_counter() - t0) / probe.shape[0]
    n_rows = int(min(n_all, max(1, round(budget_s / (args.steps + args.warmup) / per_row))))

    def step(i):
        sel = order[(i * n_rows + np.arange(n_rows)) % n_all]
        t, h = sel // wl.Hq, (sel % wl.Hq).astype(np.int32)
        slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, wl.block_size)
        oracle.append(kn, vn, slots, kc, vc, wl.k_scale, wl.v_scale)
        oracle.attention(wl.q, wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, kc, vc, wl.scale, wl.k_scale,
                         wl.v_scale, nthreads=nt, rows=(t, h))
        return float(row_b[sel].sum()) + nb["append"] + nb["tables"]

    for i in range(args.warmup):
        step(i)
    moved, t0 = 0.0, time.perf_counter()
    for i in range(args.steps):
        moved += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = moved / dt / 1e9
    sample = (f"{n_rows} of {n_all} (token, head) rows per step, rotating over a seeded permutation, "
              f"plus the full slot mapping and append of the step; fp64, {nt} threads")
    return {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64, N(0,1) rounded to bf16)", "impl": "reference",
            "config": {"workload": wl.name, "batch": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                       "block_size": wl.block_size, "num_blocks": wl.num_blocks,
                       "mean_ctx": float(wl.seq_lens.mean()), "step": "oracle: slot mapping + append + "
                       "attention of a row sample", "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": nt, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main
def run_layout_compare(args):
    """Scattered against contiguous block tables on the layout workloads, as
    its own JSON line (see layout_ratio)."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    with ClockSampler(dev.index) as clk:
        r = layout_ratio(dev, repeats=args.repeats, clk=clk)
    return {"metric": "pkv_attention_run time, scattered / contiguous block tables", "unit": "ratio",
            "value": r["ratio_max"], "higher_is_better": False, "repeats": args.repeats,
            "config": {"workload": r["workload"],
                       "timing": "median over repeats of 200 back-to-back runs, 4 layer caches rotated"},
            "rows": r["rows"], "clocks": clk.summary()}


def skew_workloads(B, mean_ctx=2048, seed=1007):
    """Decode batches of B sequences with the same total keys (B * mean_ctx):
    uniform (every sequence mean_ctx), one long (one sequence holds half of
    the keys, the others share the rest) and heavy-tailed (log-normal, sigma
    1.5, scaled to the total), at Qwen3-4B heads, bf16, block size 16."""
    total = B * mean_ctx
    uni = np.full(B, mean_ctx, np.int64)
    one = np.full(B, max(1, (total - total // 2) // max(1, B - 1)), np.int64)
    one[B // 2] = total - one.sum() + one[B // 2]
    g = W.rng(seed, 4, B)
    x = np.exp(g.normal(0.0, 1.5, size=B))
    tail = np.maximum(1, np.floor(x / x.sum() * total)).astype(np.int64)
    tail[int(np.argmax(tail))] += total - tail.sum()
    out = {}
    for name, lens in (("uniform", uni), ("one_long", one), ("heavy_tail", tail)):
        assert int(lens.sum()) == total and (lens >= 1).all()
        mb = -(-int(lens.max()) // 16)
        out[name] = W.build(f"skew {name} B{B} total {total}", Hq=32, Hkv=8, D=128, block_size=16,
                            seq_lens=lens.astype(np.int32), q_lens=np.ones(B, np.int32), src="bf16", kv="bf16",
                            seed=seed + B, max_blocks=mb, pool_slack=0.02)
    return out


def run_skew_compare(args):
    """Uniform against skewed batches at equal total keys, B = 4, 16, 64,
    128: pkv_attention_run time and its ratio to the uniform batch."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = []
    with ClockSampler(dev.index) as clk:
        for B in (4, 16, 64, 128):
            wls = skew_workloads(B)
            t = {name: time_runs(wl, dev, 200, clk=clk) * 1e3 for name, wl in wls.items()}
            rows.append({"batch": B, "total_keys": int(wls["uniform"].seq_lens.sum()),
                         "max_ctx": {k: int(w.seq_lens.max()) for k, w in wls.items()},
                         "us": {k: round(v, 2) for k, v in t.items()},
                         "ratio_one_long": round(t["one_long"] / t["uniform"], 4),
                         "ratio_heavy_tail": round(t["heavy_tail"] / t["uniform"], 4)})
    return {"metric": "pkv_attention_run time, skewed / uniform batch at equal total keys", "unit": "ratio",
            "value": max(max(r["ratio_one_long"], r["ratio_heavy_tail"]) for r in rows), "higher_is_better": False,
            "config": {"workload": "decode, Qwen3-4B heads, bf16, block size 16, mean context 2048",
                       "timing": "200 back-to-back runs over 4 rotated layer caches after one plan"},
            "rows": rows, "clocks": clk.summary()}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="decode")
    ap.add_argument("--layers", type=int, default=4, help="layer caches rotated across steps")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads' keys (layout, mixed prefill, fp8)")
    ap.add_argument("--layout-repeats", type=int, default=2, help="fresh allocations per layout in the line")
    ap.add_argument("--soft-cap", type=float, default=0.0, help="logits soft cap (variant; 0: off)")
    ap.add_argument("--window-left", type=int, default=-1, help="sliding window (variant; < 0: off)")
    ap.add_argument("--layout-compare", action="store_true",
                    help="print scattered / contiguous attention time on the layout workloads instead")
    ap.add_argument("--skew-compare", action="store_true",
                    help="print skewed / uniform attention time at equal total keys instead")
    ap.add_argument("--repeats", type=int, default=8, help="fresh allocations per layout (--layout-compare)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N > 1 with torch.distributed.run")
    if args.layout_compare:
        line = run_layout_compare(args) if rank == 0 else None
    elif args.skew_compare:
        line = run_skew_compare(args) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
