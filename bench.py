#!/usr/bin/env python
"""Benchmark of the KDA chunked forward on one GB300 (or N, as independent replicas).

One step = one kda_chunk_fwd call over one workload, inputs resident in HBM: by
default the headline workload (B=1, T=4096, H=HV=32, K=V=128, bf16 q/k/v/o, fp32
g/beta/state); --workload selects another of the five (2: B=4 T=16384 with an
initial state, 3: 16 packed sequences, 4: grouped value heads B=2 T=32768).
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl reference]

--impl reference times the fp64 CPU oracle (the only other implementation of
the method here) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA chunked fwd tokens/s & TFLOP/s on 1 GB300 (T=4096,H=32,K=V=128); % roofline"
WORKLOAD_INDEX = 1
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ["kimi_delta_attention_gb300/csrc/kda_chunk_tc.cu",
                  "kimi_delta_attention_gb300/csrc/kda_recurrent.cu",
                  "kimi_delta_attention_gb300/csrc/kda_decode.cu",
                  "kimi_delta_attention_gb300/csrc/kda_backward.cu",
                  "kimi_delta_attention_gb300/csrc/sm103.cuh",
                  "kimi_delta_attention_gb300/csrc/kda_common.cuh"]


# sources that only some entries depend on (the chunk-form backward's five kernels)
KERNEL_EXTRA_SOURCES = {"kda_backward_chunk": ["kimi_delta_attention_gb300/csrc/kda_backward_chunk.cu"]}


def kernel_source_hash(kernel: str | None = None) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES + KERNEL_EXTRA_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """Reads SM clocks and clock-event (throttle) reasons during the timed region
    through NVML (read-only queries), falling back to nvidia-smi."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) == 0:
                    self._nvml, self._handle = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = mx.value
        except OSError:
            pass

    def _sample(self):
        nv, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) != 0:
            return
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        reasons = rs.value if fn(h, ctypes.byref(rs)) == 0 else 0
        self.samples.append((clk.value, reasons))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(0.002)

    def start(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self):
        self._stop.set()
        if self._nvml is not None:
            self._t.join()
            if not self.samples:
                self._sample()

    def summary(self):
        if self._nvml is None:
            return self._smi_summary()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = [s for s, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle")
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml"}

    def _smi_summary(self):
        import subprocess
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                                  "clocks_event_reasons.active", "--format=csv,noheader,nounits"],
                                 capture_output=True, text=True, timeout=20).stdout.strip()
            sm, mx, act = [s.strip() for s in out.split(",")]
            bits = int(act, 16)
            reasons = sorted(n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle")
            return {"sm_mhz": float(sm), "sm_max_mhz": float(mx), "reasons": reasons, "samples": 1,
                    "source": "nvidia-smi after the timed region"}
        except Exception as e:  # noqa: BLE001
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": str(e)}


# ------------------------------------------------------------------ helpers --
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def load_traffic(kernel_name: str, workload: str):
    """Per-launch DRAM bytes of `kernel_name` on `workload` from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(f"{kernel_name}@{workload}")
    if not e or e.get("source_hash") != kernel_source_hash(kernel_name):
        return None
    return e.get("bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def sample_units(x, n):
    """n (sequence, value head) units spread over the workload: value heads in turn,
    sequences in turn (every unit of a small workload when n covers it)."""
    NS, HV = x.num_seqs, x.v.shape[2]
    units = [(s, h) for s in range(NS) for h in range(HV)]
    if n >= len(units):
        return units
    step = len(units) / n
    return [units[int(i * step)] for i in range(n)]


def unit_tokens(x, units):
    if x.cu_seqlens is None:
        return len(units) * x.q.shape[1]
    cu = x.cu_seqlens.numpy()
    return int(sum(int(cu[s + 1] - cu[s]) for s, _ in units))


def cpu_baseline(x, units: int | None = None, gate=None, min_cpu_s: float = 0.0):
    """Time the fp64 oracle (chunked form, C = 64) on a bounded sample of the
    workload: batches of `units` (sequence, value head) units, one thread each, taken in
    turn over the workload until the batches have used `min_cpu_s` thread-seconds or
    every unit is done (with `gate`, the oracle's pre-stage over the whole input first).
    Returns (tokens/s scaled so that a token counts all value heads, cores, sample text,
    wall s)."""
    import oracle
    cores = os.cpu_count() or 1
    HV = x.v.shape[2]
    total = x.num_seqs * HV
    if units is None:
        units = min(cores, total)
    f = lambda t: None if t is None else t.float().numpy()
    order = sample_units(x, total)
    if min_cpu_s <= 0.0:
        order = sample_units(x, units)
    cu = None if x.cu_seqlens is None else x.cu_seqlens.numpy()
    t0 = time.perf_counter()
    if gate is None:
        q, k, g, beta = f(x.q), f(x.k), f(x.g), f(x.beta)
    else:
        q, k, g, beta = oracle.prestage(f(x.q), f(x.k), f(x.g_raw), f(x.beta_raw), f(x.A_log), f(x.dt_bias),
                                        gate=gate[0], lower_bound=gate[1])
    v, h0 = f(x.v), f(x.initial_state)
    done = 0
    while done < len(order):
        sel = order[done:done + units]
        oracle.forward_units(q, k, v, g, beta, x.scale, sel, initial_state=h0, cu_seqlens=cu, form="chunked",
                             chunk=64, nthreads=len(sel))
        done += len(sel)
        if (time.perf_counter() - t0) * units >= min_cpu_s:
            break
    dt = time.perf_counter() - t0
    sel = order[:done]
    token_heads = unit_tokens(x, sel)
    sample = (f"{len(sel)} of {total} (sequence, value head) units ({token_heads} token-heads) of "
              f"{x.meta.get('workload', 'the workload')}, fp64 {'pre-stage + ' if gate else ''}chunked oracle "
              f"(C=64), {units} threads; {dt:.2f} s wall (~{dt * units:.0f} thread-s); tokens/s counts a "
              f"token as all {HV} value heads")
    return token_heads / HV / dt, units, sample, dt


# --------------------------------------------------------------------- arms --
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from kimi_delta_attention_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    x = W.workload_inputs(args.workload)
    vals, times = [], []
    cores = None
    sample = None
    n_steps = max(1, args.steps)
    for i in range(max(0, args.warmup) + n_steps):
        v, cores, sample, dt = cpu_baseline(x)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": n_steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w, x, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, x, n):
    d = {"workload": w.name, "model": None, "B": w.B, "T": int(x.q.shape[1]), "H": w.H, "HV": w.HV, "K": w.K,
         "V": w.V, "global_batch": x.num_seqs * n, "seq_len": w.T if not w.num_seqs else None, "chunk": 64,
         "parallelism": f"replicas x{n} (independent problems per GPU)",
         "l2": "flushed between timed steps (256 MiB device write outside the step events)",
         "initial_state": "read (0.1 N(0,1))" if w.init_state else "zeros (not read)", "final_state": "written"}
    if w.num_seqs:
        lens = [int(v) for v in (x.cu_seqlens[1:] - x.cu_seqlens[:-1]).tolist()]
        d.update({"num_seqs": w.num_seqs, "seq_lens": lens, "packed_tokens": int(x.q.shape[1])})
    return d


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", torch.cuda.current_device())
    import kimi_delta_attention_gb300 as kda
    from kimi_delta_attention_gb300 import workloads as W
    kda.build()
    kda.load_library()
    w = W.WORKLOADS[args.workload]
    gate = ("bounded", -5.0) if args.gated else None
    host = W.workload_raw_inputs(args.workload) if args.gated else W.workload_inputs(args.workload)
    x = host.to(dev)
    B, T, H, K = x.q.shape
    HV, V = x.v.shape[2], x.v.shape[3]
    NS = x.num_seqs
    out = torch.empty_like(x.v)
    fin = torch.empty((NS, HV, K, V), dtype=torch.float32, device=dev)
    shape = kda.make_shape(x.q, x.v, x.cu_seqlens)
    wsp = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        forward(kda, x, gate, out=out, final_state=fin, workspace=wsp, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if kda.kda_read_device_status(wsp) != 0:
        raise RuntimeError("device status not OK after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        torch.distributed.barrier()
    sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    status = kda.kda_read_device_status(wsp)

    tokens = host.tokens()
    value = ws * tokens / (ms * 1e-3)
    flops = tokens * HV * (6 * K * V + 6 * 64 * K + 4 * 64 * V)  # the flop convention (workloads.flops_convention)
    tflops = ws * flops / (ms * 1e-3) / 1e12
    alg_bytes = input_bytes(host) + 2 * x.v.numel() + NS * HV * K * V * 4  # inputs once, o and the final state
    hbm_gbs, bf16_tf, peak_src = load_peaks()
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    kernel_name = kda.kda_chunk_fwd_kernel_name(shape)
    # launches of that kernel per step (several for the split kernel over many units): a
    # launch moves its share of the step's bytes in its share of the step's time, so the
    # per-launch roofline fraction is the step's
    launches = kda.kda_chunk_fwd_kernel_launches(shape)

    # end to end through the public API with pinned host buffers
    e2e = e2e_measure(kda, host, gate, dev, stream, max(3, min(args.steps, 20 if tokens <= 1 << 16 else 5)))

    line = {
        "impl": "kda_gb300", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_dict(w, host, ws), **({"prestage": "fused: raw bf16 q, k, g_raw; bounded gate "
                                                        "lower_bound -5; beta sigmoid"} if gate else {})),
        "tflops": tflops,
        # the token recurrence's own arithmetic, 7 K V flop per token and value head: a
        # lower bound on any evaluation, reported beside the chunked convention
        "tflops_recurrent_lower_bound": ws * tokens * HV * 7 * K * V / (ms * 1e-3) / 1e12,
        "roofline_time_ms": max(alg_bytes / (hbm_gbs * 1e9), flops / (bf16_tf * 1e12)) * 1e3,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": load_traffic(kernel_name, w.name),
                     "kernel": kernel_name, "launches_per_step": launches,
                     "algorithmic_bytes_per_launch": alg_bytes / launches,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
        "clocks": sampler.summary(), "e2e": e2e, "gpu_launches": args.steps * launches,
        "device_status": status, "wall_s_timed_region": t_wall,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = cpu_baseline(host, gate=gate, min_cpu_s=10.0)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def input_tensors(x):
    """(name, tensor) of every input a forward reads, in the order of the call."""
    if hasattr(x, "g_raw"):
        names = ("q", "k", "v", "g_raw", "beta_raw", "A_log", "dt_bias", "initial_state", "cu_seqlens")
    else:
        names = ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")
    return [(n, getattr(x, n)) for n in names]


def input_bytes(x):
    return sum(t.numel() * t.element_size() for _, t in input_tensors(x) if t is not None)


def forward(kda, d, gate, **kw):
    """One forward on device tensors `d` (an Inputs, a RawInputs or a dict with the same
    fields) through the public entry point."""
    g = d.get if isinstance(d, dict) else (lambda n: getattr(d, n))
    if gate is None:
        return kda.kda_chunk_fwd(g("q"), g("k"), g("v"), g("g"), g("beta"), g("scale"), initial_state=g("initial_state"),
                                 cu_seqlens=g("cu_seqlens"), **kw)
    return kda.kda_chunk_fwd_gated(g("q"), g("k"), g("v"), g("g_raw"), g("beta_raw"), g("A_log"), g("dt_bias"),
                                   gate=gate[0], lower_bound=gate[1], scale=g("scale"),
                                   initial_state=g("initial_state"), cu_seqlens=g("cu_seqlens"), **kw)


def e2e_measure(kda, host, gate, dev, stream, steps):
    """Same metric through the public entry point with host buffers: every step copies
    the inputs (with the initial state and cu_seqlens when the workload has them) from
    pinned host memory to the device, runs the forward and copies o and the final
    state back.  Steps alternate between two streams with their own device buffers
    and workspaces, so that one step's copies overlap the previous step's forward;
    each stream keeps its own steps in order.  (Splitting a step's input copies over
    several streams did not raise the host-to-device rate, ~195 GB/s.)"""
    import torch
    hsrc = {n: (None if t is None else t.pin_memory()) for n, t in input_tensors(host)}
    B, T, H, K = host.q.shape
    HV, V = host.v.shape[2], host.v.shape[3]
    NS = host.num_seqs
    shape = kda.make_shape(hsrc["q"], hsrc["v"], hsrc["cu_seqlens"])
    wsz = kda.kda_chunk_fwd_workspace_size(shape)
    streams = [stream, torch.cuda.Stream(dev)]
    bufs = []
    for _ in range(2):
        d = {n: (None if t is None else torch.empty_like(t, device=dev)) for n, t in hsrc.items()}
        d["scale"] = host.scale
        d["o"] = torch.empty_like(d["v"])
        d["s"] = torch.empty((NS, HV, K, V), dtype=torch.float32, device=dev)
        d["ws"] = torch.empty(wsz, dtype=torch.uint8, device=dev)
        d["ho"] = torch.empty(host.v.shape, dtype=host.v.dtype).pin_memory()
        d["hs"] = torch.empty((NS, HV, K, V), dtype=torch.float32).pin_memory()
        bufs.append(d)
    h2d = sum(t.numel() * t.element_size() for t in hsrc.values() if t is not None)
    d2h = bufs[0]["ho"].numel() * bufs[0]["ho"].element_size() + bufs[0]["hs"].numel() * 4

    def step(i):
        d, st = bufs[i & 1], streams[i & 1]
        with torch.cuda.stream(st):
            for n, h in hsrc.items():
                if h is not None:
                    d[n].copy_(h, non_blocking=True)
            forward(kda, d, gate, out=d["o"], final_state=d["s"], workspace=d["ws"], stream=st.cuda_stream)
            d["ho"].copy_(d["o"], non_blocking=True)
            d["hs"].copy_(d["s"], non_blocking=True)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for i in range(steps):
        step(i)
    streams[0].wait_stream(streams[1])
    e1.record(streams[0])
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    status = max(kda.kda_read_device_status(d["ws"]) for d in bufs)
    return {"value": host.tokens() / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "overlap": "two streams, double-buffered: a step's copies overlap the previous step's forward",
            "device_status": status}


DECODE_METRIC = "KDA decode step (recurrent, state in place) tokens/s on 1 GB300 (B=128, T=1, H=HV=32, K=V=128); % roofline"


def run_decode(args):
    """One step = one kda_decode call: one new token for each of 128 sequences x 32
    value heads against fp32 states (537 MB read and written per step, more than L2).
    HBM-bound on the state."""
    import torch
    import kimi_delta_attention_gb300 as kda
    from kimi_delta_attention_gb300 import workloads as W
    kda.build()
    kda.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    B, T, H, HV, K, V = 128, 1, 32, 32, 128, 128
    host = W.make_inputs(B, T, H, HV, K, V, "bf16", seed=11, init_state=True)
    x = host.to(dev)
    state = x.initial_state.clone()
    out = torch.empty_like(x.v)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.kda_decode(x.q, x.k, x.v, x.g, x.beta, state, x.scale, out=out, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    el = lambda t: t.numel() * t.element_size()
    alg = 2 * el(x.initial_state) + el(x.q) + el(x.k) + el(x.v) + el(x.g) + el(x.beta) + el(out)
    hbm_gbs, _, peak_src = load_peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    line = {
        "impl": "kda_gb300", "metric": DECODE_METRIC, "value": B * T / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "decode_B128_T1_H32_K128", "B": B, "T": T, "H": H, "HV": HV, "K": K, "V": V,
                   "io": "bf16 q/k/v/o, fp32 g/beta/state", "l2": "flushed between timed steps; the state "
                   "(537 MB) is larger than L2 anyway"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": load_traffic("decode_kernel", "decode_B128_T1_H32_K128"),
                     "kernel": "decode_kernel",
                     "algorithmic_bytes_per_launch": alg, "peak_source": peak_src},
        "clocks": sampler.summary(), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


TWOPASS_METRIC = ("KDA chunked fwd in two passes (state scan writing h[n], then the parallel output kernel) "
                  "tokens/s on 1 GB300 (T=4096,H=32,K=V=128); % roofline")


def run_twopass(args):
    """One step = kda_chunk_states (the serial scan, writing the state entering every
    chunk, bf16) + kda_chunk_output (every chunk's output from those states, in parallel)
    over the headline workload.  Each pass is also timed on its own."""
    import torch
    import kimi_delta_attention_gb300 as kda
    from kimi_delta_attention_gb300 import workloads as W
    kda.build()
    kda.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[args.workload]
    host = W.workload_inputs(args.workload)
    if host.cu_seqlens is not None:
        raise SystemExit("the two-pass forward takes fixed-length workloads")
    x = host.to(dev)
    B, T, H, K = x.q.shape
    HV, V = x.v.shape[2], x.v.shape[3]
    h = torch.empty((B, HV, (T + 63) // 64, K, V), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((B, HV, K, V), dtype=torch.float32, device=dev)
    out = torch.empty_like(x.v)
    wsp = torch.empty(kda.kda_chunk_fwd_workspace_size(kda.make_shape(x.q, x.v)), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(256, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def states():
        kda.kda_chunk_states(x.q, x.k, x.v, x.g, x.beta, initial_state=x.initial_state, h=h, final_state=fin,
                             workspace=wsp, stream=stream.cuda_stream)

    def output():
        kda.kda_chunk_output(x.q, x.k, x.v, x.g, x.beta, h, x.scale, out=out, workspace=ws2, stream=stream.cuda_stream)

    def timed(fns):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            for f in fns:
                f()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            for f in fns:
                f()
            e1.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / len(evs)

    sampler = ClockSampler(dev.index)
    sampler.start()
    ms = timed([states, output])
    sampler.stop()
    ms_states, ms_output = timed([states]), timed([output])
    alg = W.algorithmic_bytes(host, final_state=True)
    h_bytes = h.numel() * 2
    hbm_gbs, _, peak_src = load_peaks()
    line = {
        "impl": "kda_gb300", "metric": TWOPASS_METRIC, "value": host.tokens() / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "ms_states_pass": ms_states, "ms_output_pass": ms_output, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_dict(w, host, 1), h_bytes=h_bytes),
        "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": alg / (ms * 1e-3) / 1e9 / hbm_gbs, "traffic": None,
                     "kernel": "kda_chunk_*_kernel (state pass) + kda_chunk_output_kernel",
                     "algorithmic_bytes_per_launch": alg,
                     "note": "the forward's algorithmic bytes; the two passes also write and read h once and "
                             "read the inputs twice", "peak_source": peak_src},
        "clocks": sampler.summary(), "gpu_launches": 2 * args.steps,
        "device_status": max(kda.kda_read_device_status(wsp), kda.kda_read_device_status(ws2)),
    }
    print(json.dumps(line), flush=True)
    return 0


BACKWARD_METRIC = ("KDA backward (gradients of q, k, v, g, beta and the initial state, chunk form with "
                   "split-operand tensor-core products) tokens/s on 1 GB300 (a workload; default T=4096, "
                   "H=HV=32, K=V=128); % of the TF32 tensor peak")
# nominal dense TF32 / bf16 tensor rates of the part (1.1 and 2.25 PFLOP/s): the TF32 peak
# is the measured bf16 peak scaled by their ratio
TF32_PER_BF16 = 1.1 / 2.25
BACKWARD_LAUNCHES = 5  # prep, chain, value-side, C x C and key-side gradient kernels
BACKWARD_KERNELS = "prep_kernel, chain_tc_kernel, grad_v_tc_kernel, grad_cc_kernel, grad_k_kernel"


def backward_flops(tokens_heads: int, K: int, V: int, C: int = 64) -> float:
    """Arithmetic of the chunk-form backward per (token, value head), every product counted
    once (triangular ones in full), per chunk of C tokens:
      prep      L and Aqk, W (2 C^2 K each), U, Aqk^T do (2 C^2 V each), Q (2 K^2 C),
                R (2 K C V), B (4 K C V);
      chains    the state and the state gradient (2 K^2 V each);
      value     v_new, dv_new, do S^T, dW, dkr (2 C K V each), dAqk, dAv, dv (2 C^2 V each);
      C x C     dA (2 C^2 K), dA A^T and T^T Y (2 C^3 each);
      key       A^T dW, two row-side and two column-side decayed products (2 C^2 K each).
    The split-TF32 evaluation issues three tensor products for each of these."""
    per_chunk = 18 * C * C * K + 10 * C * C * V + 2 * K * K * C + 16 * K * C * V + 4 * K * K * V + 4 * C ** 3
    return tokens_heads / C * per_chunk


def run_backward(args):
    """One step = one kda_backward call on a workload's inputs (default the headline shape;
    io dtype q, k, v and a seeded output gradient; fp32 g, beta; a final-state gradient; the
    workload's initial state), L2 flushed between steps."""
    import numpy as np
    import torch
    import kimi_delta_attention_gb300 as kda
    from kimi_delta_attention_gb300 import workloads as W
    kda.build()
    kda.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[args.workload]
    host = W.workload_inputs(args.workload)
    B, T, H, K = host.q.shape
    HV, V = host.v.shape[2], host.v.shape[3]
    NS = host.num_seqs
    rng = np.random.default_rng(22)
    io = torch.bfloat16 if w.io_dtype == "bf16" else torch.float32
    do_h = torch.from_numpy(rng.standard_normal(tuple(host.v.shape), dtype=np.float32)).to(io)
    dfin_h = torch.from_numpy(rng.standard_normal((NS, HV, K, V), dtype=np.float32))
    x = host.to(dev)
    do, dfin = do_h.to(dev), dfin_h.to(dev)
    shape = kda.make_shape(x.q, x.v, x.cu_seqlens)
    ws = torch.empty(kda.kda_backward_workspace_size(shape), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return kda.kda_backward(x.q, x.k, x.v, x.g, x.beta, do, x.scale, initial_state=x.initial_state,
                                cu_seqlens=x.cu_seqlens, d_final_state=dfin, workspace=ws, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    tokens = B * T
    wname = "backward_" + w.name
    flops = backward_flops(tokens * HV, K, V)
    achieved = flops / (ms * 1e-3) / 1e12
    _, bf16_tf, peak_src = load_peaks()
    tf32_peak = bf16_tf * TF32_PER_BF16
    line = {
        "impl": "kda_gb300", "metric": BACKWARD_METRIC, "value": tokens / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wname, "B": B, "T": T, "H": H, "HV": HV, "K": K, "V": V, "num_seqs": NS,
                   "io": f"{w.io_dtype} q/k/v/d_out, fp32 g/beta/d_final_state; fp32 gradients",
                   "products": ("each operand split into high and low parts, 3 products per product: tcgen05 bf16 "
                                "for the state chains, the value-side gradients and prep's K x K / K x V products, "
                                "warp-level TF32 for the rest"),
                   "l2": "flushed between timed steps"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf32_peak, "unit": "TFLOP/s",
                     "frac": achieved / tf32_peak, "kernel": f"the whole step ({BACKWARD_KERNELS})",
                     "traffic": load_traffic("kda_backward_chunk", wname),
                     "flops_per_step": flops, "launches_per_step": BACKWARD_LAUNCHES,
                     "peak_source": (f"{peak_src} bf16 peak x {TF32_PER_BF16:.3f} (nominal dense TF32 / bf16)")},
        "clocks": sampler.summary(), "gpu_launches": args.steps * BACKWARD_LAUNCHES,
        "device_status": kda.kda_read_device_status(ws),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kda_gb300", choices=["kda_gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gated", action="store_true",
                    help="raw bf16 inputs through kda_chunk_fwd_gated (pre-stage fused, bounded gate)")
    ap.add_argument("--mode", default="forward", choices=["forward", "decode", "twopass", "backward"],
                    help="decode: time kda_decode (one token per sequence) instead of the chunked forward")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="workload index (0-4); 1, the headline, is the default bench line")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "decode":
        return run_decode(args)
    if args.mode == "backward":
        return run_backward(args)
    if args.mode == "twopass":
        return run_twopass(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
