#!/usr/bin/env python
"""Benchmark: In-Place TTT fast-weight layer tokens/s on GB300.

One step = one ittt_forward call over one batch of synthetic inputs (the whole
hot path: conv, target GEMM, gate/up GEMM, snapshot 0, update walk, apply).
Default workload: the Qwen3-4B-shaped layer, B=2 x T=32768, d=2560,
d_ff=9728, C=2048, eta=0.01 (bf16 inputs, fp32 state).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 run under torchrun: every rank processes its own batch of
sequences (independent fast-weight states, no data-path collective) and
value = all ranks' tokens / the slowest rank's time (weak scaling).

`--impl reference` times the fp64 CPU oracle on the host cores instead (rank 0
only; other ranks exit at once).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TTT-MLP tokens/s per layer (d2560/ff9728, 32k ctx); % of GB300 bf16 peak"
DEFAULT_CONFIG = 2
# DRAM bytes (read + write) per launch of a kernel at a named workload, from
# one ncu capture (profiles/traffic_qwen3-4b-layer-B2-T32k-C2048.md: the
# kernels of one forward over 1 x 32768 tokens, scaled by the token count to
# the 2 x 32768 launch), with the hash of the kernel's sources at capture
# time: once the sources change the figure no longer describes the kernel
# and `traffic` is reported as null.
TRAFFIC_BYTES = {
    (2, "gateup"): (2656388096, "0f821ce53dc8d5a6"),
}
KERNEL_SOURCES = {
    "gateup": ["k_gateup.cu"], "target": ["k_target.cu"], "update": ["k_update.cu"],
    "apply": ["k_apply.cu"], "conv": ["k_target.cu"], "snapshot0": ["k_update.cu"],
}


def _code_only(text: str) -> str:
    """C++ source with comments and runs of white space removed (string
    literals kept)."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (not the comments) a kernel is built from: recorded
    DRAM traffic is reported only while it matches."""
    import hashlib
    csrc = os.path.join(ROOT, "chunk_wise_weight_gb300", "csrc")
    m = hashlib.sha1()
    for f in KERNEL_SOURCES[kernel] + ["pipeline.cuh", "pipeline_pair.cuh", "sm103.cuh"]:
        with open(os.path.join(csrc, f)) as fh:
            m.update(_code_only(fh.read()).encode())
    return m.hexdigest()[:16]


def recorded_traffic(config: int, kernel: str, shape_override: bool):
    entry = TRAFFIC_BYTES.get((config, kernel))
    if entry is None or shape_override or entry[1] != kernel_source_hash(kernel):
        return None
    return entry[0]
PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--shape", default=None,
                    help="B,T,d,f,C,eta instead of the named workload (profiling cases)")
    ap.add_argument("--cpu-tokens", type=int, default=1024,
                    help="tokens of the CPU-baseline sample (two chunks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused-conv", action="store_true",
                    help="compute the convolution inside the target GEMM")
    ap.add_argument("--dual", action="store_true",
                    help="force the dual form (scores Z Z^T) instead of the fast-weight walk")
    ap.add_argument("--primal", action="store_true",
                    help="force the fast-weight walk (the library otherwise picks the dual "
                         "form for short sequences)")
    ap.add_argument("--packed", action="store_true",
                    help="pack the workload's B*T tokens into one row of documents with "
                         "log-uniform lengths in [512, 16384] (state reset per document)")
    ap.add_argument("--l2norm", action="store_true",
                    help="normalise every updated fast weight row by row (one launch per chunk)")
    ap.add_argument("--eta-tok", action="store_true",
                    help="per-token learning-rate weights (seeded uniform [0.5, 1.5))")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step (with a caller workspace) into a CUDA graph and time "
                         "its replays; per-kernel phases then come from an eager pass")
    ap.add_argument("--fp32-inputs", action="store_true",
                    help="draw H, X0, W_gate, W_up and W_target unrounded and pass them as "
                         "fp32: the library splits each value into bf16 hi/lo parts and "
                         "runs the gate/up and target contractions over K = 3 d")
    ap.add_argument("--bf16-inputs", action="store_true",
                    help="round the tiny workload's fp32 inputs to bf16 first, as the other "
                         "workloads' inputs are (it otherwise runs them as fp32)")
    ap.add_argument("--seq-shards", type=int, default=0,
                    help="run the sequence-sharded schedule with this many spans, the spans "
                         "run in turn on this GPU (fold, exclusive prefix, apply); one rank only")
    return ap.parse_args()


def tensor_peak(peaks, peak_src, clocks):
    """The bf16 peak a tensor-bound kernel is held to: the sustained one
    when the clock record of the timed region shows the power cap active
    (the kernel then runs in the regime the sustained figure was measured
    in: seconds of back-to-back work under the cap), else the burst one."""
    burst = float(peaks["bf16_tflops"])
    sust = float(peaks["bf16_tflops_sustained"])
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    if capped:
        return sust, (f"bf16_tflops_sustained ({peak_src}; sw_power_cap active in the "
                      f"timed region)")
    return burst, f"bf16_tflops burst ({peak_src})"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(PEAK_FALLBACK), "fallback"


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, via
    ctypes) every 10 ms on a host thread, so even a timed region of a few
    tens of milliseconds gets several samples.  Read-only: it sets nothing.
    Falls back to nvidia-smi (ClockSampler) where NVML cannot be loaded."""

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, device=None):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        found = False
        if device is not None:  # match the CUDA device by its PCI address
            try:
                import torch
                pr = torch.cuda.get_device_properties(device)
                bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
                found = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(
                    bus.encode(), ctypes.byref(self.handle)) == 0
            except (AttributeError, RuntimeError):
                found = False
        if not found and self.nvml.nvmlDeviceGetHandleByIndex_v2(
                ctypes.c_uint(index), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
            or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _run(self):
        ctypes = self.ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            if (self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0):
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.01)

    def start(self):
        self.thread = self.threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self) -> dict | None:
        self.stop_flag.set()
        self.thread.join()
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "NVML every 10 ms in the timed region"}


def clock_sampler(index: int, device=None):
    try:
        return NvmlClockSampler(index, device)
    except (OSError, AttributeError):
        return ClockSampler(index)


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[5 + k].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "source": "nvidia-smi every 200 ms"}


def phase_model(B, T, d, f, C, dual=False, cu=None, fp32_inputs=False):
    """Algorithmic work per phase: ('tensor', FLOPs) or ('hbm', bytes).  The
    dual form's extra work (scores Z Z^T, S Vhat) is charged at the primal
    form's FLOPs, the work the layer needs.  With packed documents (cu) B is
    1, every document is chunked on its own and only the tokens before each
    document's last chunk update.  fp32 inputs: the conv phase also splits
    H and the three weights (4 B read, 6 B written per element: three bf16
    segments) and writes Xc split the same way; the target and gate/up
    contractions run over K = 3 d (three bf16 products per input product)."""
    lens = [b - a for a, b in zip(cu, cu[1:])] if cu else [T] * B
    upd_tokens = sum(L - (L - (-(-L // C) - 1) * C) for L in lens)
    M = B * T
    if fp32_inputs:
        conv = (2.0 * M * d + 2.0 * f * d + 1.0 * d * d) * (4 + 6) + d * 3 * 4
    else:
        conv = 2.0 * M * d * 2 + d * 3 * 4
    kx = 3.0 if fp32_inputs else 1.0
    return {
        "conv": ("hbm", conv),
        "target": ("tensor", kx * 2.0 * B * T * d * d),
        "gateup": ("tensor", kx * 4.0 * B * T * d * f),
        "snapshot0": ("hbm", 1.0 * d * f * 2 + len(lens) * d * f * 2),
        "update": ("tensor", 2.0 * upd_tokens * d * f),
        "apply": ("tensor", 2.0 * B * T * d * f),
    }


def launches_per_step(B, T, C, cu, l2norm, dual=False, d=2560, f=9728, pairs=76,
                      fp32_inputs=False):
    """Kernel launches of one forward with the bench's bf16 W_down0 and no
    snapshot buffer: conv, target, gate/up, the update walk, apply (the
    apply reads W_0 itself, so no snapshot-0 copy); packed documents add the
    table-staging kernel; the dual form runs scores and dual apply instead of
    walk and apply.  The walk is one launch; with L2 normalisation too when
    the batch is regular, d a multiple of 256, every chunk a multiple of 64
    tokens and a group of ceil(f/256) CTA pairs fits in the GPU's 76 (the
    state stays in TMEM), else one launch per chunk that updates plus a
    finalising launch.  fp32 inputs add the four hi/lo splits (H, W_gate,
    W_up, W_target); their convolution kernel replaces the bf16 one."""
    lens = [b - a for a, b in zip(cu, cu[1:])] if cu else [T] * B
    steps = max(-(-L // C) - 1 for L in lens)
    splits = 4 if fp32_inputs else 0
    if dual:
        return 5 + splits + (1 if cu else 0)
    in_tmem = not cu and d % 256 == 0 and C % 64 == 0 and -(-f // 256) <= pairs
    walk = (steps + 1 if l2norm and not in_tmem else 1) if steps > 0 else 0
    return 4 + walk + (1 if cu else 0) + splits


def run_seq_shards(args, cfg, tensors, stream, dev, peaks, peak_src, rates, local, cpu):
    """--seq-shards R: every span's work of the sequence-sharded schedule on
    this one GPU, span after span: fold each span into its delta
    (ITTT_FLAG_UPDATE_ONLY, from zero), take each span's exclusive prefix
    (ittt_state_prefix), then walk and apply each span from its prefix
    reusing Z and eta * Vhat.  ms_per_step is the time one GPU needs for all
    spans; on R GPUs each would run one span and all-gather the deltas."""
    import torch
    from chunk_wise_weight_gb300 import counted_flops, ittt
    from chunk_wise_weight_gb300.shard import sequence_span

    H, X0, Wg, Wu, W0, Wt, cw = tensors
    B, T, d = H.shape
    f = Wg.shape[0]
    C, eta, R = cfg["C"], cfg["eta"], args.seq_shards
    spans = [sequence_span(T, C, R, r) for r in range(R)]
    spans = [(a, b) for a, b in spans if b > a]
    n_sp = len(spans)
    bf, f32 = torch.bfloat16, torch.float32
    Hs = [H[:, a:b].contiguous() for a, b in spans]
    X0s = [X0[:, a:b].contiguous() for a, b in spans]
    ets = [None if rates is None else rates[:, a:b].contiguous() for a, b in spans]
    zs = [torch.empty(B, b - a, f, dtype=bf, device=dev) for a, b in spans]
    vs = [torch.empty(B, b - a, d, dtype=bf, device=dev) for a, b in spans]
    outs = [torch.empty(B, b - a, d, dtype=bf, device=dev) for a, b in spans]
    deltas = torch.empty(n_sp, B, d, f, dtype=f32, device=dev)
    states = [torch.empty(B, d, f, dtype=f32, device=dev) for _ in spans]

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        for k in range(n_sp):
            ittt.forward(Hs[k], X0s[k], Wg, Wu, None, Wt, cw, eta, C, stream=stream,
                         update_only=True, state_out=deltas[k], z_buf=zs[k], vhat_buf=vs[k],
                         eta_tok=ets[k])
        if ev:
            ev[1].record(stream)
        for k in range(n_sp):
            ittt.state_prefix(W0, deltas, k, states[k], stream=stream)
        if ev:
            ev[2].record(stream)
        for k in range(n_sp):
            ittt.forward(Hs[k], X0s[k], Wg, Wu, None, Wt, cw, eta, C, outs[k], stream=stream,
                         state_in=states[k], reuse_zv=True, z_buf=zs[k], vhat_buf=vs[k])
        if ev:
            ev[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    ittt.stream_status(stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = clock_sampler(local, dev)
    torch.cuda.synchronize(dev)
    sampler.start()
    if isinstance(sampler, ClockSampler):
        time.sleep(0.3)  # let nvidia-smi take its first reading
    for k in range(args.steps):
        step(ev[k])
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ittt.stream_status(stream)
    ms_per_step = sum(e[0].elapsed_time(e[3]) for e in ev) / args.steps
    part = [sum(e[p].elapsed_time(e[p + 1]) for e in ev) / args.steps for p in range(3)]
    # Algorithmic work: the fold is gate/up, target and one 2*d*f-FLOP
    # contraction per token; the prefix of span k reads k deltas and W_0 and
    # writes one state; the apply phase is the walk and the apply.
    fold_flops = B * T * (4 * d * f + 2 * d * d + 2 * d * f)
    prefix_bytes = sum(k * B * d * f * 4 + d * f * 2 + B * d * f * 4 for k in range(n_sp))
    F = counted_flops(B, T, d, f, C)
    phases = {
        "fold": {"ms": round(part[0], 4), "share": round(part[0] / ms_per_step, 4),
                 "tflops": round(fold_flops / (part[0] * 1e-3) / 1e12, 1)},
        "prefix": {"ms": round(part[1], 4), "share": round(part[1] / ms_per_step, 4),
                   "gbs": round(prefix_bytes / (part[1] * 1e-3) / 1e9, 1)},
        "apply": {"ms": round(part[2], 4), "share": round(part[2] / ms_per_step, 4)},
    }
    peak, peak_kind = tensor_peak(peaks, peak_src, clocks)
    achieved = fold_flops / (part[0] * 1e-3) / 1e12
    launches = 0
    for a, b in spans:
        n_k = -(-(b - a) // C)
        launches += 4 + 1 + 2 + (1 if n_k > 1 else 0)
    conf = arm_config(cfg, args, 1)
    conf["parallelism"] = f"sequence x{R} (spans run in turn on one GPU)"
    conf["spans"] = [b - a for a, b in spans]
    line = {
        "metric": METRIC, "value": B * T / (ms_per_step * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": conf,
        "layer_tflops": round(F / (ms_per_step * 1e-3) / 1e12, 1),
        "counted_tflop_per_step": round(F / 1e12, 4),
        "roofline": {"bound": "tensor", "kernel": "fold (conv, target, gate/up, update)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_kind": peak_kind,
                     "frac_of_burst": round(achieved / float(peaks["bf16_tflops"]), 4)},
        "phases": phases, "cpu_baseline": cpu, "clocks": clocks, "e2e": None,
        "gpu_launches": launches * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def init_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dual_form(cfg, args, cu=None) -> bool:
    """Whether the call runs the dual form: forced by --dual, else the
    library's choice for these options (the rule of ittt_plan_form: the dual
    form where allowed and T < 2.5 d f / (d + f))."""
    if args.dual:
        return True
    if args.primal or cu is not None or args.l2norm or args.fused_conv:
        return False
    T, d, f, C = cfg["T"], cfg["d"], cfg["f"], cfg["C"]
    return C % 64 == 0 and T % C == 0 and T // C >= 2 and 2 * T * (d + f) < 5 * d * f


def arm_config(cfg, args, world, cu=None):
    """The `config` object of a bench line (both arms report the same one)."""
    T = cfg["T"] if cu is None else cu[-1]
    return {"workload": cfg["name"], "B": cfg["B"] if cu is None else 1, "T": T,
            "d": cfg["d"], "f": cfg["f"], "C": cfg["C"], "eta": cfg["eta"],
            "chunks": -(-T // cfg["C"]) if cu is None else None,
            "parallelism": f"batch x{world} (replicas)",
            "packed_docs": None if cu is None else {
                "count": len(cu) - 1, "lengths": [b - a for a, b in zip(cu, cu[1:])],
                "mix": "log-uniform in [512, 16384] tokens, seeded"},
            "conv": "fused into target GEMM" if args.fused_conv else "own kernel",
            "schedule": ("dual (scores Z Z^T), forced" if args.dual else
                         "dual (scores Z Z^T), chosen for short sequences"
                         if dual_form(cfg, args, cu) else "primal walk"),
            "eta_tok": "per-token rates" if args.eta_tok else None,
            "update_rule": "L2-normalised rows" if args.l2norm else "additive",
            "launch": "CUDA graph replay" if getattr(args, "graph", False) else "eager",
            "inputs": "fp32" if getattr(args, "fp32_inputs", False) else "bf16",
            "l2": l2_note(cfg, T)}


def l2_note(cfg, T):
    """Whether one step's tensors outrun the 126 MB L2 (no flush is then
    needed between timed steps): H and X0, Z, and the weight snapshots the
    walk writes and the apply reads."""
    B = cfg["B"] if T == cfg["T"] else 1
    n = -(-T // cfg["C"])
    z_bytes = B * T * cfg["f"] * 2
    act_bytes = 2 * B * T * cfg["d"] * 2
    snap_bytes = B * max(n - 1, 0) * cfg["d"] * cfg["f"] * 2
    total = z_bytes + act_bytes + snap_bytes
    if total > 2 * 126e6:
        return (f"inputs larger than L2: H+X0 {act_bytes / 1e9:.2f} GB, Z "
                f"{z_bytes / 1e9:.2f} GB and snapshots {snap_bytes / 1e9:.2f} GB per step")
    return (f"small workload: {total / 1e6:.0f} MB of activations and snapshots per step, "
            "not flushed from L2 between steps")


def fp32_inputs_for(args) -> bool:
    """Whether the run passes fp32 inputs: asked for, or the tiny workload
    (whose inputs are fp32) unless its rounding is asked for."""
    if args.fp32_inputs:
        return True
    return (args.config == 0 and args.shape is None and not args.bf16_inputs
            and not args.fused_conv)


def run_reference(args):
    world, rank, _ = init_dist(args)
    if rank != 0:
        return 0
    args.fp32_inputs = fp32_inputs_for(args)
    import oracle
    from chunk_wise_weight_gb300 import CONFIGS, make_inputs
    cfg = CONFIGS[args.config]
    S = max(128, min(256, cfg["T"]))
    Cs = S // 2
    inp = make_inputs(1, S, cfg["d"], cfg["f"], seed=1234 + args.config,
                      round_bf16=not args.fp32_inputs)
    warmup = max(3, args.warmup)
    for _ in range(warmup):
        oracle.forward(inp, cfg["eta"], Cs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(inp, cfg["eta"], Cs)
    dt = time.perf_counter() - t0
    tok_s = S * args.steps / dt
    cores = oracle.num_threads()
    sample = (f"fp64 oracle, one sequence of {S} tokens in two chunks of {Cs} at "
              f"d={cfg['d']}, d_ff={cfg['f']} per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(cfg, args, world),
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def gpu_local_cpus(device) -> set:
    """The host CPUs NVML reports as closest to `device` (those sharing its
    NUMA node), intersected with the CPUs this process may use; empty when
    NVML cannot tell."""
    import ctypes
    try:
        import torch
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            return set()
        handle = ctypes.c_void_p()
        pr = torch.cuda.get_device_properties(device)
        bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) != 0:
            return set()
        words = 64
        mask = (ctypes.c_ulong * words)()
        if nvml.nvmlDeviceGetCpuAffinity(handle, ctypes.c_uint(words), mask) != 0:
            return set()
        bits = ctypes.sizeof(ctypes.c_ulong) * 8
        cpus = {w * bits + i for w in range(words) for i in range(bits) if mask[w] >> i & 1}
        return cpus & set(os.sched_getaffinity(0))
    except (OSError, AttributeError, RuntimeError):
        return set()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    architecture)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(cfg, index, tokens):
    """The oracle on a bounded sample of the workload, on every host core;
    then, single-threaded, on the tiny d 64 / d_ff 256 workload whole."""
    import oracle
    from chunk_wise_weight_gb300 import CONFIGS, make_inputs
    S = max(128, tokens)
    Cs = S // 2
    inp = make_inputs(1, S, cfg["d"], cfg["f"], seed=1234 + index)
    t0 = time.perf_counter()
    oracle.forward(inp, cfg["eta"], Cs)
    dt = time.perf_counter() - t0
    cores = oracle.num_threads()
    tiny = CONFIGS[0]
    tin = make_inputs(tiny["B"], tiny["T"], tiny["d"], tiny["f"], seed=1234)
    oracle.set_num_threads(1)
    try:
        t1 = time.perf_counter()
        oracle.forward(tin, tiny["eta"], tiny["C"])
        dt1 = time.perf_counter() - t1
    finally:
        oracle.set_num_threads(cores)
    return {"value": S / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"fp64 oracle on one sequence of {S} tokens in two chunks of {Cs} at "
                       f"d={cfg['d']}, d_ff={cfg['f']} ({dt:.1f} s)"),
            "cpu_model": cpu_model(),
            "single_thread": {"workload": tiny["name"], "cores": 1,
                              "value": tiny["B"] * tiny["T"] / dt1, "unit": "tokens/s",
                              "seconds": round(dt1, 4)}}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from chunk_wise_weight_gb300 import CONFIGS, counted_flops, ittt, make_inputs
    from chunk_wise_weight_gb300.inputs import counted_flops_packed, packed_offsets
    from chunk_wise_weight_gb300 import build as lib_build
    from chunk_wise_weight_gb300.shard import barrier, max_over_ranks, shard_range

    world, rank, local = init_dist(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    cfg = dict(CONFIGS[args.config])
    if args.shape:
        vals = args.shape.split(",")
        cfg.update(B=int(vals[0]), T=int(vals[1]), d=int(vals[2]), f=int(vals[3]),
                   C=int(vals[4]), eta=float(vals[5]))
        cfg["name"] = "B{B}-T{T}-d{d}-f{f}-C{C}".format(**cfg)
    B, T, d, f, C, eta = cfg["B"], cfg["T"], cfg["d"], cfg["f"], cfg["C"], cfg["eta"]
    args.fp32_inputs = fp32_inputs_for(args)
    peaks, peak_src = load_peaks()

    # CPU baseline first (rank 0, one GPU only), before the device is busy.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args.config, args.cpu_tokens)

    lib_build.build()
    ittt.load()

    # Inputs: the layer's weights are shared; the global batch is B * world
    # sequences and each rank draws and runs its own contiguous share.
    first, last = shard_range(B * world, world, rank)
    assert last - first == B
    inp = make_inputs(B, T, d, f, seed=1234 + args.config, round_bf16=not args.fp32_inputs)
    if first > 0:
        g = torch.Generator().manual_seed(1234 + args.config + 1000 * first)
        inp["H"] = torch.randn(B, T, d, generator=g)
        inp["X0"] = torch.randn(B, T, d, generator=g)
        if not args.fp32_inputs:
            inp["H"] = inp["H"].to(torch.bfloat16).float()
            inp["X0"] = inp["X0"].to(torch.bfloat16).float()
    cu = None
    if args.packed:
        # The same tokens as one packed row of documents.
        cu = packed_offsets(B * T, seed=2468 + first)
        inp["H"] = inp["H"].reshape(1, B * T, d)
        inp["X0"] = inp["X0"].reshape(1, B * T, d)
        B, T = 1, B * T
    bf = torch.bfloat16
    adt = torch.float32 if args.fp32_inputs else bf  # H, X0, W_gate, W_up, W_target
    H = inp["H"].to(dev, adt)
    X0 = inp["X0"].to(dev, adt)
    Wg, Wu = inp["W_gate"].to(dev, adt), inp["W_up"].to(dev, adt)
    W0, Wt = inp["W_down0"].to(dev, bf), inp["W_target"].to(dev, adt)
    cw = inp["conv_w"].to(dev, torch.float32)
    out = torch.empty(B, T, d, dtype=bf, device=dev)
    stream = torch.cuda.current_stream(dev)
    rates = None
    if args.eta_tok:
        g_rates = torch.Generator().manual_seed(4321 + first)
        rates = (torch.rand(B, T, generator=g_rates) + 0.5).to(dev)

    if args.fp32_inputs and args.fused_conv:
        raise SystemExit("--fp32-inputs runs the split convolution (no --fused-conv)")
    if args.seq_shards:
        if world > 1:
            raise SystemExit("--seq-shards runs its spans in turn on one GPU: one rank only")
        if args.packed or args.l2norm or args.dual or dual_form(cfg, args) or args.fp32_inputs:
            raise SystemExit("--seq-shards needs regular bf16 sequences and the additive update")
        return run_seq_shards(args, cfg, (H, X0, Wg, Wu, W0, Wt, cw), stream, dev, peaks,
                              peak_src, rates, local, cpu)

    workspace = None
    if args.graph:
        if cu is not None:
            raise SystemExit("--graph: packed documents stage host tables and cannot be captured")
        ws_bytes = ittt.workspace_bytes_ex(B, T, d, f, C, fused_conv=args.fused_conv,
                                           dual=args.dual, primal=args.primal,
                                           l2norm=args.l2norm, fp32_inputs=args.fp32_inputs,
                                           eta_tok=rates)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step(events=None):
        ittt.forward(H, X0, Wg, Wu, W0, Wt, cw, eta, C, out, stream=stream, events=events,
                     fused_conv=args.fused_conv, dual=args.dual, primal=args.primal,
                     eta_tok=rates, cu_seqlens=cu,
                     l2norm=args.l2norm, workspace=workspace)

    for _ in range(max(3, args.warmup)):
        step()
    ittt.stream_status(stream)
    graph = None
    if args.graph:
        # One step captured once; the timed loop replays it.  Capture runs on
        # a side stream, as CUDA graph capture requires.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ittt.forward(H, X0, Wg, Wu, W0, Wt, cw, eta, C, out, fused_conv=args.fused_conv,
                         dual=args.dual, primal=args.primal, eta_tok=rates, l2norm=args.l2norm,
                         workspace=workspace)
        for _ in range(max(3, args.warmup)):
            graph.replay()
        torch.cuda.synchronize(dev)
        ittt.stream_status(stream)

    # An untimed pass of the same length with every phase's events finds the
    # dominant kernel and gives the other phases' times; the timed steps then
    # record only the dominant kernel's two events (an event between two
    # kernels costs a little and keeps the second from starting early).
    nph = len(ittt.PHASES)
    ev_all = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nph)]
              for _ in range(args.steps)]
    for k in range(args.steps):
        step(ev_all[k])
    torch.cuda.synchronize(dev)
    ittt.stream_status(stream)
    pass_ms = {name: sum(ev_all[k][2 * p].elapsed_time(ev_all[k][2 * p + 1])
                         for k in range(args.steps)) / args.steps
               for p, name in enumerate(ittt.PHASES)}
    dominant = max(ittt.PHASES, key=lambda nm: pass_ms[nm])
    di = ittt.PHASES.index(dominant)
    ev_dom = []
    for _ in range(args.steps):
        row = [None] * (2 * nph)
        row[2 * di] = torch.cuda.Event(enable_timing=True)
        row[2 * di + 1] = torch.cuda.Event(enable_timing=True)
        ev_dom.append(row)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = clock_sampler(local, dev)
    barrier(dev)
    torch.cuda.synchronize(dev)
    if isinstance(sampler, ClockSampler):
        sampler.start()
        time.sleep(0.3)  # let nvidia-smi take its first reading
    else:
        sampler.start()
    t_start.record(stream)
    for k in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(ev_dom[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(dev)
    ittt.stream_status(stream)
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    ms_per_step = elapsed_ms / args.steps
    tokens = B * T * world * args.steps
    value = tokens / (elapsed_ms / 1e3)

    # Per-phase device durations: the dominant kernel's from the timed steps
    # (a replayed graph records none: then from the untimed pass), the
    # others' from the untimed pass.
    live = graph is None
    if live:
        pass_ms[dominant] = sum(ev_dom[k][2 * di].elapsed_time(ev_dom[k][2 * di + 1])
                                for k in range(args.steps)) / args.steps
    form_dual = dual_form(cfg, args, cu)
    assert form_dual == (ittt.plan_form(B, T, d, f, C, dual=args.dual, primal=args.primal,
                                        fused_conv=args.fused_conv, l2norm=args.l2norm,
                                        cu_seqlens=cu) == ittt.FORM_DUAL)
    model = phase_model(B, T, d, f, C, form_dual, cu, args.fp32_inputs)
    phases = {}
    for name in ittt.PHASES:
        ms = pass_ms[name]
        kind, work = model[name]
        entry = {"ms": round(ms, 4), "share": round(ms / ms_per_step, 4),
                 "timed": "timed steps" if (live and name == dominant) else "untimed pass"}
        if kind == "tensor":
            entry["tflops"] = round(work / (ms * 1e-3) / 1e12, 1) if ms > 0 else None
        else:
            entry["gbs"] = round(work / (ms * 1e-3) / 1e9, 1) if ms > 0 else None
        phases[name] = entry
    kind, work = model[dominant]
    dom_ms = phases[dominant]["ms"]
    if kind == "tensor":
        # Held to the sustained peak when the timed region ran under the
        # power cap, else to the burst peak; both fractions are reported.
        achieved = work / (dom_ms * 1e-3) / 1e12
        peak, peak_kind = tensor_peak(peaks, peak_src, clocks)
        roof = {"bound": "tensor", "kernel": dominant, "achieved": round(achieved, 1),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(args.config, dominant, bool(args.shape)),
                "peak_kind": peak_kind,
                "frac_of_burst": round(achieved / float(peaks["bf16_tflops"]), 4),
                "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4),
                "flops_per_launch": work,
                "timed": "CUDA events in the timed steps" if live else "untimed eager pass"}
    else:
        achieved = work / (dom_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                "peak_kind": f"hbm_gbs ({peak_src})", "bytes_per_launch": work,
                "timed": "CUDA events in the timed steps" if live else "untimed eager pass"}
    F = counted_flops_packed(cu, d, f, C) if cu else counted_flops(B, T, d, f, C)
    layer_tflops = F / (ms_per_step * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step copies
    # its activations (H, X0) from pinned host memory to the device, runs the
    # layer and reads O back into pinned host memory.  Copies run on their own
    # streams with two device buffer sets, so step k's compute overlaps the
    # upload of step k+1 and the download of step k-1.
    e2e = None
    if not args.no_e2e:
        # Pinned buffers on the GPU's own NUMA node: the pages are placed
        # where the allocating thread runs, and a far node's memory reaches
        # the GPU over the CPU-to-CPU link at a fraction of the C2C rate.
        near = gpu_local_cpus(dev)
        allowed = set(os.sched_getaffinity(0))
        if near:
            os.sched_setaffinity(0, near)
        try:
            H_h = inp["H"].to(adt).pin_memory()
            X0_h = inp["X0"].to(adt).pin_memory()
            O_h = [torch.empty(B, T, d, dtype=bf).pin_memory() for _ in range(2)]
        finally:
            os.sched_setaffinity(0, allowed)
        Hs, X0s, Os = [H, torch.empty_like(H)], [X0, torch.empty_like(X0)], [out, torch.empty_like(out)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        mk = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        uploaded, computed, downloaded = mk(), mk(), mk()

        def e2e_steps(count, e_start=None, e_end=None):
            if e_start is not None:
                e_start.record(up)
            for k in range(count):
                j = k % 2
                if k >= 2:
                    up.wait_event(computed[j])      # buffers j free again
                with torch.cuda.stream(up):
                    Hs[j].copy_(H_h, non_blocking=True)
                    X0s[j].copy_(X0_h, non_blocking=True)
                    uploaded[j].record(up)
                stream.wait_event(uploaded[j])
                if k >= 2:
                    stream.wait_event(downloaded[j])  # O_j read back before reuse
                ittt.forward(Hs[j], X0s[j], Wg, Wu, W0, Wt, cw, eta, C, Os[j], stream=stream,
                             fused_conv=args.fused_conv, dual=args.dual, primal=args.primal,
                             eta_tok=rates,
                             cu_seqlens=cu, l2norm=args.l2norm)
                computed[j].record(stream)
                down.wait_event(computed[j])
                with torch.cuda.stream(down):
                    O_h[j].copy_(Os[j], non_blocking=True)
                    downloaded[j].record(down)
            if e_end is not None:
                for j in range(2):
                    up.wait_event(downloaded[j])
                e_end.record(up)

        def copies_only(count, h2d, d2h):
            """The same copies with no compute: host-copy rates in this run."""
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            t0.record(up)
            down.wait_event(t0)
            for k in range(count):
                j = k % 2
                if h2d:
                    with torch.cuda.stream(up):
                        Hs[j].copy_(H_h, non_blocking=True)
                        X0s[j].copy_(X0_h, non_blocking=True)
                if d2h:
                    with torch.cuda.stream(down):
                        O_h[j].copy_(Os[j], non_blocking=True)
            up.wait_stream(down)
            t1.record(up)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1) / count

        # At least 30 steps: the first upload and the last download of the
        # region are not overlapped with compute, and over a short region
        # they weigh on the average.
        e2e_n = max(args.steps, 30)
        e2e_steps(3)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dev)
        torch.cuda.synchronize(dev)
        e2e_steps(e2e_n, e0, e1)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        h2d_b = H_h.numel() * H_h.element_size() + X0_h.numel() * X0_h.element_size()
        d2h_b = O_h[0].numel() * O_h[0].element_size()
        ms_up = copies_only(e2e_n, True, False)
        ms_down = copies_only(e2e_n, False, True)
        ms_both = copies_only(e2e_n, True, True)
        e2e = {"value": B * T * world * e2e_n / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
               "steps": e2e_n,
               "note": "per step: H2D of H and X0 from pinned host memory, ittt_forward, D2H "
                       "of O to pinned host memory; copies overlap compute on two buffer "
                       "sets; weights stay resident",
               "pinned_on": (f"the GPU's NUMA node ({len(near)} CPUs)" if near
                             else "the allocating thread's node"),
               "copies_alone": {"h2d_gbs": round(h2d_b / ms_up / 1e6, 1),
                                "d2h_gbs": round(d2h_b / ms_down / 1e6, 1),
                                "both_ms_per_step": round(ms_both, 3),
                                "both_gbs": round((h2d_b + d2h_b) / ms_both / 1e6, 1),
                                "note": "the same copies with no compute, same run"}}
        ittt.stream_status(stream)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": arm_config(cfg, args, world, cu),
            "layer_tflops": round(layer_tflops, 1),
            "layer_frac_of_peak": {
                "bf16_tflops": round(layer_tflops / float(peaks["bf16_tflops"]), 4),
                "bf16_tflops_sustained":
                    round(layer_tflops / float(peaks["bf16_tflops_sustained"]), 4),
                "peaks": peak_src},
            "counted_tflop_per_step": round(F / 1e12, 4),
            "roofline": roof,
            "phases": phases,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": launches_per_step(B, T, C, cu, args.l2norm, form_dual, d, f,
                                              fp32_inputs=args.fp32_inputs) * args.steps,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
