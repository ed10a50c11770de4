#!/usr/bin/env python
"""FAVOR+ forward attention throughput on GB300: tokens*heads per second.

One step = one pass of the whole forward hot path over one batch of the
very-long-context workload (B=1, H=16, L=65536, d=dv=64, m=256, bf16,
Q/K/V ~ N(0, 0.5^2), orthogonal omega per head): bidirectional and causal
attention, each with positive softmax features and with ReLU features (four
library calls).  value = token*heads processed per second, whole job, timed
with CUDA events around the steps and nothing else on the stream.

Beside the headline: per-kernel times from a separate pass with the
library's event hooks on, each call of the step timed on its own with its
whole-call roofline, and the same per-call numbers for the other workloads
(tiny_f32, approx_f32 over m, bidir_bf16, causal_bf16).

Arms:
  --impl ours (default)  the CUDA library through its C ABI, inputs resident
                         in HBM; plus an end-to-end number with host buffers
                         (host->device copies and the device->host read of
                         the outputs inside the timed region).
  --impl reference       the float64 CPU oracle on this host's cores, each
                         step a bounded sample (a few heads) of the workload.

Multi-GPU (torchrun, one process per GPU): each rank runs an independent
replica of the workload with its own seed (no collective on the data path);
scaling is weak and value sums over ranks, time is the max over ranks.
"""
from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402

from synth import CONFIGS, make_workload  # noqa: E402

STEP_CALLS = (("bidir", "softmax_pos"), ("causal", "softmax_pos"), ("bidir", "relu"), ("causal", "relu"))
UNIT = "tokens*heads/s"
METRIC = "FAVOR+ forward tokens*heads/sec (bidir & causal)"
SFU_EX2_PER_CLK_PER_SM = 32   # ex2.approx throughput per SM per clock (measured on GB300: 31.4)
GB300_SMS = 152


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="long_bf16", choices=sorted(CONFIGS))
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's sequence length L (profiling a smaller case of the same shape)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--decode-steps", type=int, default=200,
                    help="one-token causal steps timed for the decode line (0 = skip)")
    ap.add_argument("--backward-steps", type=int, default=2,
                    help="timed repetitions of the backward line (bidir + causal gradients; 0 = skip)")
    ap.add_argument("--variant-steps", type=int, default=2,
                    help="timed repetitions of each feature-variant / relative-position call (0 = skip)")
    ap.add_argument("--e2e-groups", type=int, default=4,
                    help="head groups pipelined over upload / compute / download streams in the e2e leg")
    ap.add_argument("--cpu-heads", type=int, default=2, help="heads of the workload in the CPU oracle sample")
    ap.add_argument("--no-config-lines", dest="config_lines", action="store_false",
                    help="skip the per-configuration lines (tiny_f32, approx_f32, bidir_bf16, causal_bf16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks/throttle samples for one GPU while the work runs."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.samples = []          # (t, sm_mhz, max_mhz, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            reasons = [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, fallback_t0):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "timed region"
        if not win:
            win = [s for s in self.samples if fallback_t0 <= s[0] <= t1]
            note = "warm-up and timed region (timed region shorter than the sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        reasons = sorted({r for s in win for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win), "window": note}


# ------------------------------------------------------------- algorithmic work
def per_token_head(w, slot, kind):
    """Algorithmic (bytes, flops, exps) per token*head for one kernel slot."""
    b = 2 if w.dtype == "bf16" else 4
    d, dv, m = w.d, w.dv, w.m
    e = m if kind == "softmax_pos" else 0
    if slot == "segment_state":          # reads K, V; phi_K and Phi_K^T [V 1]
        return (d + dv) * b, 2 * m * d + 2 * m * (dv + 1), e
    if slot == "bidir_readout":          # reads Q, writes out; phi_Q and Phi_Q [S z]
        return (d + dv) * b, 2 * m * d + 2 * m * (dv + 1), e
    if slot == "causal_chunks":          # reads Q, K, V, writes out (the method's whole per-token work)
        return (2 * d + 2 * dv) * b, 4 * m * d + 4 * m * (dv + 1), 2 * e
    if slot == "feature_map":
        return d * b + m * b, 2 * m * d, e
    return 0, 0, 0


FP64_NOMINAL_TFLOPS = 1.25   # GB300 FP64 (datasheet); the fp32-storage path computes in float64


def compute_path(w, kind="softmax_pos"):
    """Which units a forward call of workload w runs on."""
    if w.dtype == "bf16" and (w.d, w.dv, w.m) == (64, 64, 256):
        return "tensor cores"
    if w.dtype == "f32" and kind in ("softmax_pos", "relu", "softmax_hyp"):
        return "CUDA cores, float64"
    return "CUDA cores, fp32"


def call_roofline(w, kind, ms, peaks, sm_mhz):
    """Roofline of one whole forward call (every kernel it launches) from its
    algorithmic work per token*head: bytes (2d + 2dv) * sizeof(dtype) (read Q,
    K, V, write out), flops 4md + 4m(dv+1), exps 2m (exp features only).  The
    roofline time is the largest of bytes / HBM, flops / compute peak and exps /
    exp2 peak; frac = roofline time / measured time."""
    T = w.B * w.H * w.L
    b = 2 if w.dtype == "bf16" else 4
    nbytes = (2 * w.d + 2 * w.dv) * b * T
    flops = (4 * w.m * w.d + 4 * w.m * (w.dv + 1)) * T
    exps = (2 * w.m if kind in ("softmax_pos", "softmax_hyp", "softmax_trig") else 0) * T
    path = compute_path(w, kind)
    sec = ms / 1e3
    sfu = GB300_SMS * SFU_EX2_PER_CLK_PER_SM * sm_mhz * 1e6
    if path == "tensor cores":
        cpeak, cname = peaks["bf16_tflops"] * 1e12, "bf16 tensor (measured burst)"
    elif path == "CUDA cores, float64":
        cpeak, cname, sfu = FP64_NOMINAL_TFLOPS * 1e12, "FP64 (nominal 1.25 TFLOP/s)", None
    else:
        cpeak, cname = GB300_SMS * 128 * 2 * sm_mhz * 1e6, "FP32 FFMA (152 SMs x 128 lanes x 2 x SM clock)"
    times = {"hbm": nbytes / (peaks["hbm_gbs"] * 1e9), "compute": flops / cpeak}
    if sfu and exps:
        times["exp2"] = exps / sfu
    bound = max(times, key=times.get)
    return {"bound": bound, "roofline_us": times[bound] * 1e6, "measured_us": ms * 1e3,
            "frac": times[bound] / sec, "path": path, "compute_peak": cname,
            "achieved": {"GB/s": nbytes / sec / 1e9, "TFLOP/s": flops / sec / 1e12,
                         "Gexp/s": exps / sec / 1e9},
            "per_token_head": {"bytes": nbytes // T, "flops": flops // T, "exps": exps // T}}


def time_calls(fn, reps, stream, warm=2):
    """Average device time (ms) of fn() over reps calls, CUDA events on `stream`."""
    import torch
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def backward_flops_per_token_head(w):
    """Algorithmic flops of one backward call per token*head: the recomputed
    features (2md each for q and k), the forward state (2m(dv+1)), and the
    gradient contractions u = S dO (2m dv), sum phi_q D^T (2m(dv+1)),
    dq = G Omega (2md), dphi_k = H [v 1] (2m(dv+1)), dv = H^T phi_k (2m dv),
    dk = G_k Omega (2md)."""
    d, dv, m = w.d, w.dv, w.m
    return 8 * m * d + 6 * m * (dv + 1) + 4 * m * dv


# Source files that define the tensor-core kernels whose DRAM traffic
# profiles/ncu_traffic.json records: a change to any of them voids the record.
TC_SOURCES = ("favor_tc.cu", "tc_common.cuh", "tc_ptx.cuh")


def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "random_feature_gb300", "csrc")
    for f in TC_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(slot):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernels."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(slot)
    if not ent or ent.get("source_digest") != source_digest():
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------- CPU oracle arm
def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it: the model name, else (Arm hosts)
    the implementer and part codes, else the machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            lines = f.read().splitlines()
    except OSError:
        lines = []
    fields = {}
    for line in lines:
        if ":" in line:
            key, val = (x.strip() for x in line.split(":", 1))
            fields.setdefault(key, val)
    for key in ("model name", "Model"):
        if fields.get(key):
            return fields[key]
    if "CPU implementer" in fields or "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer')} part {fields.get('CPU part')}"
    return platform.machine() or "unknown"


def cpu_sample(w, heads, seed=0):
    """Time the oracle on the first `heads` heads of the workload, all four calls."""
    import oracle as O
    wh = w.replace(H=heads)
    omega, q, k, v = make_workload(wh, seed)
    t0 = time.perf_counter()
    for mode, kind in STEP_CALLS:
        fn = O.favor_causal if mode == "causal" else O.favor_bidir
        fn(q, k, v, omega, w.data_scale, kind)
    dt = time.perf_counter() - t0
    units = len(STEP_CALLS) * wh.B * wh.H * wh.L
    return units / dt, dt, units


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload_of(args)
    heads = max(1, min(args.cpu_heads, w.H))
    for _ in range(max(0, min(args.warmup, 1))):
        cpu_sample(w.replace(L=min(w.L, 4096)), 1)
    total_units = 0
    total_t = 0.0
    for _ in range(args.steps):
        _, dt, units = cpu_sample(w, heads)
        total_units += units
        total_t += dt
    value = total_units / total_t
    sample = (f"{heads} of {w.H} heads of {w.name} (B={w.B}, L={w.L}, d={w.d}, m={w.m}), all four calls "
              f"(bidir/causal x softmax_pos/relu) per step, float64 NumPy")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample_heads": heads},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch
    import torch.distributed as dist
    import random_feature_gb300 as R
    from random_feature_gb300.replicas import job_aggregate, replica_seed

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    w = workload_of(args)
    peaks = load_peaks()
    omega, q, k, v = make_workload(w, seed=replica_seed(0, rank))
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    qd, kd, vd = (torch.from_numpy(a).to(device=dev, dtype=tdt).contiguous() for a in (q, k, v))
    handles = {kind: R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L)
               for kind in sorted({kd_ for _, kd_ in STEP_CALLS})}
    outs = [torch.empty((w.B, w.H, w.L, w.dv), dtype=tdt, device=dev) for _ in STEP_CALLS]
    stream = torch.cuda.current_stream(dev)

    def step(qq=qd, kk=kd, vv=vd, oo=outs):
        for (mode, kind), o in zip(STEP_CALLS, oo):
            handles[kind].attn(qq, kk, vv, causal=(mode == "causal"), out=o, stream=stream)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    t_warm = time.time()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # The timed region: library profiling hooks off (no events between kernels).
    launches0 = R.favor_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        dist.barrier()
    launches = R.favor_launch_count() - launches0
    ms_total = ev0.elapsed_time(ev1)

    # Per-kernel device times from a separate pass of the same steps with the
    # library's event hooks on (an event pair around every kernel).
    prof_steps = max(3, min(args.steps, 20))
    for hd in handles.values():
        R.favor_profile_reset(hd.handle)
        R.favor_profile_enable(hd.handle, True)
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize(dev)
    for hd in handles.values():
        R.favor_profile_enable(hd.handle, False)

    # Each call of the step on its own (hooks off): whole-call time and roofline.
    sm_mhz_now = sampler.samples[-1][1] if sampler.samples else peaks["sm_max_mhz"]
    calls = {}
    for (mode, kind), o in zip(STEP_CALLS, outs):
        def one(mode=mode, kind=kind, o=o):
            handles[kind].attn(qd, kd, vd, causal=(mode == "causal"), out=o, stream=stream)
        ms_c = time_calls(one, max(5, min(args.steps, 50)), stream)
        calls[f"{mode}_{kind}"] = {"ms": ms_c, "value": w.B * w.H * w.L / (ms_c / 1e3), "unit": UNIT,
                                   "roofline": call_roofline(w, kind, ms_c, peaks, sm_mhz_now)}
    sampler.stop()

    # per-kernel device time over the profiled pass
    slots = {}
    for hd in handles.values():
        for sl in range(R.favor_profile_slots()):
            ms, n = R.favor_profile_read(hd.handle, sl)
            name = R.favor_profile_name(sl)
            a = slots.setdefault(name, [0.0, 0, {}])
            a[0] += ms
            a[1] += n
            a[2][hd.kind] = a[2].get(hd.kind, 0) + n

    units_step = len(STEP_CALLS) * w.B * w.H * w.L
    job_units, ms_step = job_aggregate(units_step, ms_total / args.steps, device=dev)
    value = job_units / (ms_step / 1e3)

    # The other workloads, each call timed on its own (hooks off): throughput and
    # whole-call roofline.  tiny_f32 and approx_f32 are parity cases on the
    # float64 CUDA-core path (no roofline target); bidir_bf16 and causal_bf16
    # are the L >= 4096 bf16 configurations next to long_bf16.
    configs = None
    if args.config_lines and world == 1:
        configs = {}
        plan = [("tiny_f32", None), ("approx_f32", (16, 32, 64, 128, 256)), ("bidir_bf16", None),
                ("causal_bf16", None)]
        for cname, msweep in plan:
            base = CONFIGS[cname]
            entry = {}
            for m_ in (msweep or (base.m,)):
                wc = base.replace(m=m_)
                om_c, qc, kc, vc = make_workload(wc, 0)
                tdc = torch.bfloat16 if wc.dtype == "bf16" else torch.float32
                qcd, kcd, vcd = (torch.from_numpy(a).to(device=dev, dtype=tdc).contiguous() for a in (qc, kc, vc))
                oc = torch.empty((wc.B, wc.H, wc.L, wc.dv), dtype=tdc, device=dev)
                with R.Favor(wc.H, wc.m, wc.d, wc.dv, "softmax_pos", wc.dtype, om_c, wc.data_scale, wc.B,
                             wc.L) as fc:
                    for mode in wc.modes:
                        def one(mode=mode):
                            fc.attn(qcd, kcd, vcd, causal=(mode == "causal"), out=oc, stream=stream)
                        reps = 3 if wc.dtype == "f32" and wc.L > 1024 else 20
                        ms_c = time_calls(one, reps, stream)
                        key = mode if msweep is None else f"m{m_}_{mode}"
                        entry[key] = {"ms": ms_c, "value": wc.B * wc.H * wc.L / (ms_c / 1e3), "unit": UNIT,
                                      "roofline": call_roofline(wc, "softmax_pos", ms_c, peaks, sm_mhz_now)}
                del qcd, kcd, vcd, oc
            entry["config"] = (f"B={base.B} H={base.H} L={base.L} d={base.d} dv={base.dv} "
                               f"m={'/'.join(map(str, msweep)) if msweep else base.m} {base.dtype}, positive "
                               f"features, seed 0")
            configs[cname] = entry
        torch.cuda.synchronize(dev)

    # Decoding: one new token per step continuing from a resident state
    # (favor_attn_causal_step, T = 1), positive features, state prefilled from
    # the workload's keys; timed with CUDA events on the stream.
    decode = None
    if args.decode_steps > 0:
        hd_ = handles["softmax_pos"]
        state = hd_.kv_state(kd, vd)
        q1, k1, v1 = (t[:, :, :1].contiguous() for t in (qd, kd, vd))
        o1 = torch.empty_like(v1)
        for _ in range(10):
            hd_.causal_step(q1, k1, v1, state, out=o1, stream=stream)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.decode_steps):
            hd_.causal_step(q1, k1, v1, state, out=o1, stream=stream)
        d1.record(stream)
        torch.cuda.synchronize(dev)
        us_eager = d0.elapsed_time(d1) * 1e3 / args.decode_steps
        # The same steps replayed from a CUDA graph (one captured launch per
        # step, as a serving loop would run them): device time per step,
        # without the host's per-call cost.
        us_graph = None
        try:
            cs = torch.cuda.Stream(dev)
            cs.wait_stream(stream)
            nstep = 50
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cs):
                with torch.cuda.graph(graph, stream=cs):
                    for _ in range(nstep):
                        hd_.causal_step(q1, k1, v1, state, out=o1, stream=cs)
            stream.wait_stream(cs)
            reps = max(1, args.decode_steps // nstep)
            graph.replay()
            torch.cuda.synchronize(dev)
            d0.record(stream)
            for _ in range(reps):
                graph.replay()
            d1.record(stream)
            torch.cuda.synchronize(dev)
            us_graph = d0.elapsed_time(d1) * 1e3 / (reps * nstep)
        except Exception as exc:   # capture unsupported here: report the eager number only
            print(f"decode graph capture skipped: {exc}", file=sys.stderr)
        us = us_graph if us_graph is not None else us_eager
        nbytes = 2 * 4 * w.B * w.H * w.m * (w.dv + 1)
        decode = {"us_per_step": us, "us_per_step_eager": us_eager, "us_per_step_graph": us_graph,
                  "value": w.B * w.H / (us * 1e-6), "unit": "tokens*heads/s",
                  "state_bytes_read_written": nbytes, "state_gbs": nbytes / (us * 1e-6) / 1e9,
                  "config": f"B={w.B} H={w.H} m={w.m} d={w.d} dv={w.dv}, one token per step, positive features; "
                            f"value from CUDA-graph replay when available"}

    # Backward (gradients of the bidirectional and causal calls, positive
    # features) on the same workload, one entry per call with the roofline of
    # the unit it runs on: on the tensor cores (bf16 shape) against the
    # sustained bf16 peak, else on the CUDA cores against the FP32 FFMA peak of
    # the SMs at the sampled clock.
    backward = None
    if args.backward_steps > 0:
        hd_ = handles["softmax_pos"]
        gd = torch.randn((w.B, w.H, w.L, w.dv), device=dev, dtype=torch.float32).to(tdt)
        grads = tuple(torch.empty_like(t) for t in (qd, kd, vd))
        for causal in (False, True):
            hd_.attn_backward(qd, kd, vd, gd, causal=causal, grads=grads, stream=stream)
        torch.cuda.synchronize(dev)
        T = w.B * w.H * w.L
        fpt = backward_flops_per_token_head(w)
        bw_mhz = sampler.samples[-1][1] if sampler.samples else peaks["sm_max_mhz"]
        fp32_peak = GB300_SMS * 128 * 2 * bw_mhz * 1e6
        tc_shape = w.dtype == "bf16" and (w.d, w.dv, w.m) == (64, 64, 256)
        backward = {"unit": UNIT, "flops_per_token_head": fpt,
                    "config": f"{w.name}: B={w.B} H={w.H} L={w.L}, dq/dk/dv of one call, positive features, "
                              f"dO ~ N(0,1)"}
        for causal in (False, True):
            R.favor_profile_reset(hd_.handle)
            R.favor_profile_enable(hd_.handle, True)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(args.backward_steps):
                hd_.attn_backward(qd, kd, vd, gd, causal=causal, grads=grads, stream=stream)
            b1.record(stream)
            torch.cuda.synchronize(dev)
            R.favor_profile_enable(hd_.handle, False)
            ms = b0.elapsed_time(b1) / args.backward_steps
            bk = {}
            for sl in range(R.favor_profile_slots()):
                kms, n = R.favor_profile_read(hd_.handle, sl)
                if n:
                    bk[R.favor_profile_name(sl)] = {"ms_per_call": kms / args.backward_steps,
                                                    "launches_per_call": n / args.backward_steps}
            tc = tc_shape
            pk = peaks["bf16_tflops_sustained"] * 1e12 if tc else fp32_peak
            ach = fpt * T / (ms / 1e3)
            backward["causal" if causal else "bidir"] = {
                "ms": ms, "value": T / (ms / 1e3), "path": "tensor cores" if tc else "CUDA cores",
                "roofline": {"bound": "tensor" if tc else "alu", "achieved": ach / 1e12, "peak": pk / 1e12,
                             "unit": "TFLOP/s", "frac": ach / pk,
                             "peak_source": ("measured sustained bf16" if tc else
                                             "FP32 FFMA: 152 SMs x 128 lanes x 2 flops x SM clock")},
                "kernels": bk}

    # Feature variants and relative positions on the same workload, one line each:
    # hyperbolic and trigonometric features and RFA-Gate gated causal (tensor
    # cores), PermuteFormer (CUDA cores).  Roofline: the forward's flops per
    # token*head (4md + 4m(dv+1)) against the tensor peak (tensor-core calls) or
    # the FP32 FFMA peak (CUDA-core calls).
    variants = None
    if args.variant_steps > 0:
        variants = {}
        T = w.B * w.H * w.L
        fl = 4 * w.m * w.d + 4 * w.m * (w.dv + 1)
        vmhz = sampler.samples[-1][1] if sampler.samples else peaks["sm_max_mhz"]
        fp32_peak = GB300_SMS * 128 * 2 * vmhz * 1e6
        gate = torch.rand((w.B, w.H, w.L), device=dev, dtype=torch.float32) * 0.2 + 0.8
        rng_v = np.random.default_rng(1)
        perm = np.stack([rng_v.permutation(w.m) for _ in range(w.H)]).astype(np.int32)
        rdec = np.full(w.H, 0.999, np.float32)
        half = np.ascontiguousarray(omega[:, : w.m // 2])
        cases = [("hyperbolic", "softmax_hyp", half, None), ("trigonometric", "softmax_trig", half, None),
                 ("rfa_gate", "softmax_pos", omega, "gate"), ("permuteformer", "softmax_pos", omega, "relpos")]
        vout = torch.empty_like(vd)
        for name, kind, om_, extra in cases:
            hv = R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, om_, w.data_scale, w.B, w.L)
            if extra == "relpos":
                hv.set_relpos(perm, rdec)
            modes = ("causal",) if extra == "gate" else ("bidir", "causal")
            res = {}
            for mode in modes:
                def call():
                    if extra == "gate":
                        hv.attn_causal_gated(qd, kd, vd, gate, out=vout, stream=stream)
                    else:
                        hv.attn(qd, kd, vd, causal=(mode == "causal"), out=vout, stream=stream)
                call()
                torch.cuda.synchronize(dev)
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                for _ in range(args.variant_steps):
                    call()
                c1.record(stream)
                torch.cuda.synchronize(dev)
                ms = c0.elapsed_time(c1) / args.variant_steps
                tc = (extra != "relpos" and w.dtype == "bf16" and (w.d, w.dv, w.m) == (64, 64, 256))
                pk = peaks["bf16_tflops_sustained"] * 1e12 if tc else fp32_peak
                res[mode] = {"ms": ms, "value": T / (ms / 1e3), "unit": UNIT,
                             "path": "tensor cores" if tc else "CUDA cores",
                             "roofline": {"bound": "tensor" if tc else "alu",
                                          "achieved": fl * T / (ms / 1e3) / 1e12, "peak": pk / 1e12,
                                          "unit": "TFLOP/s", "frac": fl * T / (ms / 1e3) / pk}}
            variants[name] = res
            hv.close()

    # End to end through the public API: pinned host inputs in, outputs back, every
    # step.  The heads are split into groups, one library handle per group (its
    # slice of omega), and three streams overlap the upload of group g+1, the four
    # calls on group g and the download of group g-1 (events order each group's
    # copies and calls, across steps too).
    e2e = None
    if args.e2e_steps > 0:
        G = max(1, min(args.e2e_groups, w.H))
        bounds = [(w.H * g_) // G for g_ in range(G + 1)]
        groups = []
        for g_ in range(G):
            h0, h1 = bounds[g_], bounds[g_ + 1]
            hw = h1 - h0
            gh = {kind: R.Favor(hw, w.m, w.d, w.dv, kind, w.dtype, omega[h0:h1], w.data_scale, w.B, w.L)
                  for kind in handles}
            hin = [torch.from_numpy(np.ascontiguousarray(a[:, h0:h1])).to(tdt).pin_memory() for a in (q, k, v)]
            din = [torch.empty_like(t, device=dev) for t in hin]
            dout = [torch.empty((w.B, hw, w.L, w.dv), dtype=tdt, device=dev) for _ in STEP_CALLS]
            hout = [torch.empty((w.B, hw, w.L, w.dv), dtype=tdt).pin_memory() for _ in STEP_CALLS]
            ev = {k_: torch.cuda.Event() for k_ in ("in", "comp", "out")}
            groups.append({"h": gh, "hin": hin, "din": din, "dout": dout, "hout": hout, "ev": ev, "first": True})
        s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

        def e2e_step():
            for gr in groups:
                ev = gr["ev"]
                with torch.cuda.stream(s_in):
                    if not gr["first"]:
                        s_in.wait_event(ev["comp"])          # previous step's calls have read the inputs
                    for hd_, dd in zip(gr["hin"], gr["din"]):
                        dd.copy_(hd_, non_blocking=True)
                    ev["in"].record(s_in)
                with torch.cuda.stream(s_comp):
                    s_comp.wait_event(ev["in"])
                    if not gr["first"]:
                        s_comp.wait_event(ev["out"])         # previous step's outputs are downloaded
                    for (mode, kind), o in zip(STEP_CALLS, gr["dout"]):
                        gr["h"][kind].attn(*gr["din"], causal=(mode == "causal"), out=o, stream=s_comp)
                    ev["comp"].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev["comp"])
                    for o, ho in zip(gr["dout"], gr["hout"]):
                        ho.copy_(o, non_blocking=True)
                    ev["out"].record(s_out)
                gr["first"] = False

        e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        s_comp.wait_event(a0)
        s_out.wait_event(a0)
        for _ in range(args.e2e_steps):
            e2e_step()
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_comp)
        a1.record(s_out)
        torch.cuda.synchronize(dev)
        e_units, e_ms = job_aggregate(units_step, a0.elapsed_time(a1) / args.e2e_steps, device=dev)
        nb = 2 if tdt == torch.bfloat16 else 4
        e2e = {"value": e_units / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(nb * (q.size + k.size + v.size)),
               "d2h_bytes_per_step": int(nb * len(STEP_CALLS) * w.B * w.H * w.L * w.dv), "ms_per_step": e_ms,
               "head_groups": G}
        for gr in groups:
            for hd_ in gr["h"].values():
                hd_.close()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    clocks = sampler.summary(t0, t1, t_warm)
    # roofline of the dominant kernel (among those with algorithmic work of their own)
    dom = max(((k_, v_) for k_, v_ in slots.items() if per_token_head(w, k_, "softmax_pos")[0] > 0),
              key=lambda kv: kv[1][0])
    dname, (dms, dn, by_kind) = dom
    per_launch_ms = dms / max(dn, 1)
    T = w.B * w.H * w.L
    b_sum = f_sum = e_sum = 0.0
    for kind, n in by_kind.items():
        bb, ff, ee = per_token_head(w, dname, kind)
        b_sum += n * bb * T
        f_sum += n * ff * T
        e_sum += n * ee * T
    bytes_l, flops_l, exps_l = b_sum / max(dn, 1), f_sum / max(dn, 1), e_sum / max(dn, 1)
    sec = per_launch_ms / 1e3
    sm_mhz = clocks["sm_mhz"] or peaks["sm_max_mhz"]
    sfu_peak = GB300_SMS * SFU_EX2_PER_CLK_PER_SM * sm_mhz * 1e6
    cands = {
        "hbm": (bytes_l / sec / 1e9, peaks["hbm_gbs"], "GB/s", bytes_l / (peaks["hbm_gbs"] * 1e9)),
        "tensor": (flops_l / sec / 1e12, peaks["bf16_tflops"], "TFLOP/s",
                   flops_l / (peaks["bf16_tflops"] * 1e12)),
        "alu": (exps_l / sec / 1e9, sfu_peak / 1e9, "Gexp/s", exps_l / sfu_peak),
    }
    bound = max(cands, key=lambda kk: cands[kk][3])
    ach, pk, unit, _ = cands[bound]
    traffic = ncu_traffic(dname)
    roofline = {"bound": bound, "achieved": ach, "peak": pk, "unit": unit, "frac": ach / pk,
                "traffic": traffic, "kernel": dname, "launch_ms": per_launch_ms,
                "peak_source": peaks["source"] + (" (burst bf16: a launch of well under a millisecond)"
                                                  if bound == "tensor" else "")
                + (" (32 ex2/clk/SM x 152 SMs x median SM clock)" if bound == "alu" else "")}
    roofline_all = {kk: {"achieved": c[0], "peak": c[1], "unit": c[2], "frac": c[0] / c[1]} for kk, c in cands.items()}
    kernels = {name: {"ms_total": v_[0], "launches": v_[1], "ms_per_launch": v_[0] / v_[1],
                      "share": v_[0] / max(1e-12, sum(x[0] for x in slots.values()))}
               for name, v_ in slots.items() if v_[1]}
    kernels["_pass"] = (f"{prof_steps} steps with the library's per-kernel event hooks on, after the timed "
                        f"region (which ran with them off)")

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        heads = max(1, min(args.cpu_heads, w.H))
        cval, cdt, _ = cpu_sample(w, heads)
        cpu = {"value": cval, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{heads} of {w.H} heads of {w.name}, all four calls, float64 NumPy, {cdt:.1f} s",
               "cpu_model": cpu_model()}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} L={w.L} d={w.d} dv={w.dv} m={w.m}, "
                                   f"calls per step: bidir+causal x softmax_pos+relu",
                       "global_batch": w.B * world, "seq_len": w.L, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (Q,K,V 384 MB per replica)"},
            "clocks": clocks, "e2e": e2e, "calls": calls, "configs": configs, "decode": decode,
            "backward": backward, "variants": variants,
            "gpu_launches": launches,
            "roofline": roofline,
            "roofline_all": roofline_all, "kernels": kernels, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)
    for hd in handles.values():
        hd.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def workload_of(args):
    w = CONFIGS[args.workload]
    if args.seq_len is not None:
        w = w.replace(name=f"{w.name}_L{args.seq_len}", L=args.seq_len)
    return w


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
