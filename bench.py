#!/usr/bin/env python
"""Benchmark of the head-wise recurrent scan on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
the forward scan (writing states and the backward's tape) followed by the
backward through time (reverse scan, dWx, dstates0, and the dR / db
reduction). Default workload: the largest one-GPU configuration, LSTM, bf16
storage / fp32 arithmetic, B=32, T=4096, N=1 head, D=1024 (R = 8 MB, larger
than one thread-block cluster holds: the cooperative grid kernels). The same
line carries `target_config`: the per-step roofline fractions of the LSTM fp32
B=2 T=16 N=1 D=32 workload, the configuration the >= 50% forward / >= 35%
backward target is stated on, measured in the same run.

Prints ONE JSON line (rank 0). value = timesteps*batch per second of the
forward + backward step, summed over all ranks (weak scaling: every rank runs
the full workload). --impl reference times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "timesteps·batch/s fwd and fwd+bwd; % of per-step roofline (1 GB300)"
UNIT = "timesteps*batch/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--function", default=None, help="override the workload's cell (workload 3: gru|elman)")
    ap.add_argument("--path", default="auto", choices=["auto", "fused", "alternating", "simt", "grid"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--input-proj", action="store_true",
                    help="time the tensor-core input projection (Wx = x W_x^T, I = N*D, and its backward) "
                         "on the workload's B*T rows instead of the scan")
    ap.add_argument("--proj-shape", default=None, metavar="ROWS,I,C",
                    help="with --input-proj: time this projection shape instead of the workload's")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run the workload with this T instead of its own (profiling captures of a smaller "
                         "case); the line's workload name records it")
    ap.add_argument("--no-target-config", action="store_true",
                    help="skip the per-step roofline fractions of the LSTM fp32 B=2 T=16 D=32 workload")
    ap.add_argument("--trace", action="store_true",
                    help="print the per-phase cycle medians of the persistent scan kernels (rnn_trace) "
                         "instead of the bench line")
    return ap.parse_args()


def proj_bench(args, w, fn, dev, _lib):
    """The input projection of one layer of the workload: x [B*T, I = N*D] ->
    Wx [B*T, G*N*D], and its backward (dx, dW_x, dbias), timed with CUDA
    events, the L2 flushed before every step outside the event window."""
    B, T, N, D = w["B"], w["T"], w["N"], w["D"]
    G = {"lstm": 4, "gru": 3, "elman": 1, "slstm": 4}[fn]
    BT, I, C = B * T, N * D, G * N * D
    if args.proj_shape:
        BT, I, C = (int(v) for v in args.proj_shape.split(","))
    g = torch.Generator().manual_seed(7)
    x = torch.randn(BT, I, generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn(C, I, generator=g) / I ** 0.5).to(torch.bfloat16).to(dev)
    bias = torch.randn(C, generator=g).to(torch.bfloat16).to(dev)
    dWx = torch.randn(BT, C, generator=g).to(torch.bfloat16).to(dev)
    Wx, dx, dW, db = (torch.empty(s, dtype=torch.bfloat16, device=dev) for s in ((BT, C), (BT, I), (C, I), (C,)))
    ws = torch.empty(_lib.rnn_input_proj_workspace_size(BT, I, C), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    fwd = lambda: _lib.rnn_input_proj_fwd(BT, I, C, x, W, bias, Wx, ws)
    bwd = lambda: _lib.rnn_input_proj_bwd(BT, I, C, x, W, dWx, dx, dW, db, ws)
    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    tf, tb = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        fwd()
        e[1].record()
        bwd()
        e[2].record()
        torch.cuda.synchronize()
        tf.append(e[0].elapsed_time(e[1]))
        tb.append(e[1].elapsed_time(e[2]))
    _lib.rnn_check_status(ws)
    pk = peaks()
    f_fl, b_fl = 2.0 * BT * I * C, 4.0 * BT * I * C
    f_ms, b_ms = statistics.median(tf), statistics.median(tb)
    ach = (f_fl + b_fl) / ((f_ms + b_ms) / 1e3) / 1e12
    return {"metric": "input projection TFLOP/s (forward + backward)", "value": ach, "unit": "TFLOP/s",
            "higher_is_better": True, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w["name"] if not args.proj_shape else "projection %dx%dx%d" % (BT, I, C),
                       "rows": BT, "I": I, "C": C,
                       "l2": "flushed (256 MiB write) before every step, outside the event window"},
            "fwd": {"ms": f_ms, "tflops": f_fl / (f_ms / 1e3) / 1e12},
            "bwd": {"ms": b_ms, "tflops": b_fl / (b_ms / 1e3) / 1e12},
            "roofline": {"bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": ach / pk["bf16"], "traffic": None,
                         "peak_source": f"{pk['source']} (MEASURED_PEAKS.json, burst)"}}


def phase_trace(step_fn, backward, T):
    """Median clock64 cycles between the phase points of the persistent
    kernels (CTA 0, thread 0), over up to 200 steps after the first 10.
    Point 11 of the forward kernels (the step's tail: states and tape stores) is
    reported against point 7; points 8-10 (inside the cell) are reported when
    a kernel build records them."""
    from recurrent_networks_gb300 import _lib
    steps = max(1, min(200, T - 20))
    buf = torch.zeros(16 * steps, dtype=torch.int64, device="cuda")
    out = {}
    for which in (("fwd", "bwd") if backward else ("fwd",)):
        buf.zero_()
        _lib.rnn_trace(buf, 10, steps)
        step_fn(which)
        torch.cuda.synchronize()
        _lib.rnn_trace(None)
        tr = buf.view(steps, 16).cpu().tolist()
        phases = {}
        for p in range(1, 8):
            d = [r[p] - r[p - 1] for r in tr if r[p] and r[p - 1]]
            if d:
                phases[f"{p - 1}->{p}"] = statistics.median(d)
        # the finer points inside a phase, each against the nearest earlier point
        for p in range(8, 16):
            prev = {8: 4, 9: 8, 10: 9, 11: 7}.get(p)
            if prev is None:
                continue
            d = [r[p] - r[prev] for r in tr if r[p] and r[prev]]
            if d:
                phases[f"{prev}->{p}"] = statistics.median(d)
        per = [tr[i + 1][0] - tr[i][0] for i in range(steps - 1) if tr[i + 1][0] and tr[i][0]]
        out[which] = {"step_cycles": statistics.median(per) if per else None, "phase_cycles": phases}
    return out


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def algorithmic(w, fn, esize):
    """Algorithmic work of one step per (b, n, t): forward F = 2 G D^2 flops,
    (G + S) D e bytes (Wx read, states written); backward F = 4 G D^2,
    (2S + 2G) D e bytes (dstates, states, gates read; dWx written)."""
    from recurrent_networks_gb300.synth import GATES, STATES
    G, S, D = GATES[fn], STATES[fn], w["D"]
    units = w["B"] * w["T"] * w["N"]
    return dict(units=units,
                fwd_flops=2.0 * G * D * D * units, fwd_bytes=float((G + S) * D * esize * units),
                bwd_flops=4.0 * G * D * D * units, bwd_bytes=float((2 * S + 2 * G) * D * esize * units))


KERNEL_SOURCES = {
    "fused_fwd_kernel": ["fused_fwd.cuh", "cells.cuh", "ptx.cuh", "layout.h", "kernels.cuh", "grid_place.cuh"],
    "fused_bwd_kernel": ["fused_bwd.cuh", "cells.cuh", "ptx.cuh", "layout.h", "kernels.cuh"],
    "grid_bwd_kernel": ["grid_bwd.cuh", "cells.cuh", "ptx.cuh", "layout.h", "kernels.cuh", "grid_place.cuh",
                        "dr_beside.cuh", "umma.cuh"],
}


def kernel_sources_sha(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "recurrent_networks_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def placement():
    """How the grid kernels place their batch groups on the GPU's dies."""
    from recurrent_networks_gb300 import _lib
    if os.environ.get("RNN_DIE_PLACEMENT", "1").startswith("0"):
        return "groups by block index (RNN_DIE_PLACEMENT=0)"
    layout = _lib.rnn_die_layout()
    if layout is None:
        return "groups by block index (no two-die structure measured)"
    return "grid groups on one die each (%d + %d SMs), step counters homed on the group's die" % layout


def measured_traffic(kernel, workload, path=None):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None when absent or when the kernel's
    sources changed since the counters were taken."""
    p = path or os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{kernel}@{workload}")
    if not rec or rec.get("sources_sha256") != kernel_sources_sha(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def aggregate(total_ms, fwd_ms, world, units_per_rank, steps, device=None):
    """Max over ranks of the timed totals (the slowest rank bounds the job);
    value = the units all ranks processed / that time. Returns (ms per step,
    value, forward-only value)."""
    t = torch.tensor([total_ms, fwd_ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tot, fwd = float(t[0]), float(t[1])
    ms_per_step = tot / steps
    value = world * units_per_rank / (ms_per_step / 1e3)
    fwd_value = world * units_per_rank / (fwd / steps / 1e3) if fwd > 0 else 0.0
    return ms_per_step, value, fwd_value


def target_config_fracs(dev, steps=50, warmup=5, index=1):
    """The per-step roofline fractions of one workload's scan kernels (default:
    LSTM fp32 B=2 T=16 N=1 D=32), as the metric defines them: the forward's
    roofline max(F / P_tensor, bytes / BW_HBM) over its T steps, divided by the
    forward scan kernel's CUDA-event time, and the same for the backward scan
    kernel. Timed after the main measurement, with the L2 flushed before every
    step outside the event windows; the medians over `steps` steps."""
    from recurrent_networks_gb300 import _lib
    from recurrent_networks_gb300.synth import WORKLOADS, workload_inputs
    w = WORKLOADS[index]
    fn = w["fns"][0]
    B, T, N, D, dtype = w["B"], w["T"], w["N"], w["D"], w["dtype"]
    esize = 2 if dtype == torch.bfloat16 else 4
    inp = {k: (v.to(dev) if v is not None else None) for k, v in workload_inputs(index, function=fn).items()}
    S = _lib.rnn_num_states(fn)
    dims = _lib.make_dims(B, T, N, D, fn, dtype, "auto")
    _, plan_f = _lib.rnn_plan_describe(dims, False)
    _, plan_b = _lib.rnn_plan_describe(dims, True)
    states = torch.empty((S, B, T, N, D), dtype=dtype, device=dev)
    last = torch.empty((S, B, 1, N, D), dtype=dtype, device=dev)
    tape = torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device=dev)
    ws = torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_BWD), dtype=torch.uint8, device=dev)
    dWx, dR, db, ds0 = (torch.empty_like(inp[k]) for k in ("Wx", "R", "b", "states0"))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    ev = {k: torch.cuda.Event(enable_timing=True) for k in ("f0", "f1", "b0", "b1", "s0", "s1")}
    for e in ev.values():
        e.record()
    _lib.rnn_profile_events(0, ev["f0"], ev["f1"])
    _lib.rnn_profile_events(1, ev["b0"], ev["b1"])
    tf, tb, ts = [], [], []
    for k in range(warmup + steps):
        flush.zero_()
        ev["s0"].record()
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, tape, ws)
        _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, tape, inp["dstates"], None,
                     dWx, dR, db, ds0, ws)
        ev["s1"].record()
        ev["s1"].synchronize()
        if k >= warmup:
            tf.append(ev["f0"].elapsed_time(ev["f1"]))
            tb.append(ev["b0"].elapsed_time(ev["b1"]))
            ts.append(ev["s0"].elapsed_time(ev["s1"]))
    _lib.rnn_check_status(ws)
    _lib.rnn_profile_events(0, None, None)
    _lib.rnn_profile_events(1, None, None)
    pk = peaks()
    alg = algorithmic(w, fn, esize)
    roof_f = max(alg["fwd_flops"] / (pk["bf16"] * 1e12), alg["fwd_bytes"] / (pk["hbm"] * 1e9))
    roof_b = max(alg["bwd_flops"] / (pk["bf16"] * 1e12), alg["bwd_bytes"] / (pk["hbm"] * 1e9))
    f_ms, b_ms, s_ms = statistics.median(tf), statistics.median(tb), statistics.median(ts)
    return {"workload": w["name"], "plan_fwd": plan_f, "plan_bwd": plan_b,
            "target": "forward >= 0.50, backward >= 0.35 of the per-step roofline",
            "fwd_frac": roof_f / (f_ms / 1e3), "bwd_frac": roof_b / (b_ms / 1e3),
            "fwd_roof_ns_per_step": roof_f / T * 1e9, "bwd_roof_ns_per_step": roof_b / T * 1e9,
            "fwd_kernel_ms": f_ms, "bwd_kernel_ms": b_ms, "step_ms": s_ms,
            "fwd_ns_per_timestep": f_ms * 1e6 / T, "bwd_ns_per_timestep": b_ms * 1e6 / T,
            "value": B * T / (s_ms / 1e3), "unit": UNIT, "steps": steps,
            "peaks": f"{pk['source']} (MEASURED_PEAKS.json: bf16 burst for the tensor term, HBM copy)",
            "l2": "flushed before every step, outside the event windows"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        smax = max(int(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ oracle
def cpu_oracle_step(fn, inp, nthreads, rows, steps, backward=True):
    """One forward (+ backward) of the oracle over the first `rows` batch rows
    and the first `steps` time steps; returns seconds."""
    from oracle import oracle
    Wx = inp["Wx"][:rows, :steps]
    s0 = inp["states0"][:, :rows]
    t0 = time.perf_counter()
    oracle.fwd(fn, Wx, inp["R"], inp["b"], s0, nthreads=nthreads)
    if backward:
        dst = inp["dstates"][:, :rows, :steps]
        oracle.bwd(fn, Wx, inp["R"], inp["b"], s0, dst, nthreads=nthreads)
    return time.perf_counter() - t0


# fp64 flops of the oracle per sample: the CPU baseline of the bench line takes
# about 15 s on the GPU machine's 16 host cores; each step of the reference arm
# (--impl reference, 20 + 3 steps by default) about 1.5 s
ORACLE_BUDGET_BASELINE = 700e9
ORACLE_BUDGET_REFERENCE_STEP = 60e9


def oracle_sample(w, fn, cores, budget=ORACLE_BUDGET_BASELINE):
    """(batch rows, time steps) of the workload that make one oracle run about
    `budget` fp64 flops: all rows when they fit, else a time prefix over at
    least `cores` sequences. The metric is per (row, step), so the sample's
    rate stands for the workload's."""
    from recurrent_networks_gb300.synth import GATES
    G, D, T, N, B = GATES[fn], w["D"], w["T"], w["N"], w["B"]
    per_row_step = (3.0 if w["backward"] else 1.0) * 2.0 * G * D * D * N  # fwd (+ bwd), fp64 loops
    if per_row_step * B * T <= budget:
        return B, T
    rows = min(B, max(1, -(-cores // N)))
    steps = max(8, min(T, int(budget // (per_row_step * rows))))
    return rows, steps


def workload_config(w, fn, world):
    """The `config` both arms print: the workload and how a step is timed."""
    return {"workload": w["name"], "function": fn, "B": w["B"], "T": w["T"], "N": w["N"], "D": w["D"],
            "backward": w["backward"],
            "l2": "GPU arm: flushed (256 MiB write) before every step, outside the event window; "
                  "host arm: no flush",
            "parallelism": f"replicas x{world}"}


def run_reference(args, w, fn):
    from recurrent_networks_gb300.synth import workload_inputs
    cores = host_cores()
    inp = workload_inputs(args.workload, function=fn, with_grads=True)
    rows, steps = oracle_sample(w, fn, cores, ORACLE_BUDGET_REFERENCE_STEP)
    times = []
    for k in range(args.warmup + args.steps):
        dt = cpu_oracle_step(fn, inp, cores, rows, steps, w["backward"])
        if k >= args.warmup:
            times.append(dt)
    per_step = sum(times) / len(times)
    value = rows * steps / per_step
    sample = (f"{fn} {'fwd+bwd' if w['backward'] else 'fwd'} over {rows} of {w['B']} batch rows x "
              f"{steps} of {w['T']} steps, N={w['N']}, D={w['D']}, fp64")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, fn, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ ours
def main():
    args = parse()
    from recurrent_networks_gb300.synth import WORKLOADS
    w = dict(WORKLOADS[args.workload])
    if args.seq_len:
        w.update(T=args.seq_len, name=f"{w['name']}_seq{args.seq_len}")
    fn = args.function or w["fns"][0]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, fn)), flush=True)
        return

    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from recurrent_networks_gb300 import _lib
    from recurrent_networks_gb300.synth import workload_inputs
    _lib.load()
    if args.input_proj:
        if rank == 0:
            print(json.dumps(proj_bench(args, w, fn, dev, _lib)), flush=True)
        return
    dtype = w["dtype"]
    esize = 2 if dtype == torch.bfloat16 else 4
    B, T, N, D = w["B"], w["T"], w["N"], w["D"]
    backward = w["backward"]
    host = workload_inputs(args.workload, function=fn, with_grads=backward)
    if args.seq_len:  # a time prefix of the workload's inputs
        host = {k: (None if v is None else v[:, :T].contiguous() if k == "Wx" else
                    v[:, :, :T].contiguous() if k == "dstates" else v) for k, v in host.items()}
    inp = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
    S = _lib.rnn_num_states(fn)
    dims = _lib.make_dims(B, T, N, D, fn, dtype, args.path)
    _, plan_f = _lib.rnn_plan_describe(dims, False)
    _, plan_b = _lib.rnn_plan_describe(dims, True)
    states = torch.empty((S, B, T, N, D), dtype=dtype, device=dev)
    last = torch.empty((S, B, 1, N, D), dtype=dtype, device=dev)
    tape = torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device=dev) if backward else None
    ws = torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_BWD if backward else _lib.WS_FWD),
                     dtype=torch.uint8, device=dev)
    if backward:
        dWx, dR, db, ds0 = (torch.empty_like(inp[k]) for k in ("Wx", "R", "b", "states0"))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, tape, ws)
        if backward:
            _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, tape, inp["dstates"],
                         None, dWx, dR, db, ds0, ws)

    ev = {k: torch.cuda.Event(enable_timing=True) for k in ("f0", "f1", "b0", "b1")}
    for e in ev.values():
        e.record()  # creates the underlying cudaEvent_t
    _lib.rnn_profile_events(0, ev["f0"], ev["f1"])
    if backward:
        _lib.rnn_profile_events(1, ev["b0"], ev["b1"])

    for _ in range(args.warmup):
        step()
    _lib.rnn_check_status(ws)
    torch.cuda.synchronize()

    if args.trace:
        def one(which):
            if which == "fwd":
                _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, tape, ws)
            else:
                _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, tape, inp["dstates"],
                             None, dWx, dR, db, ds0, ws)
        res = {"trace": phase_trace(one, backward, T), "workload": w["name"], "plan_fwd": plan_f,
               "plan_bwd": plan_b}
        _lib.rnn_check_status(ws)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    # timed region: per-step events; L2 flushed before every step, outside the event window
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    fscan, bscan = [], []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = _lib.rnn_kernel_launches()
    with ClockSampler(dev.index) as clk:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record()
            _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, tape, ws)
            mids[k].record()
            if backward:
                _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, tape, inp["dstates"],
                             None, dWx, dR, db, ds0, ws)
            ends[k].record()
            # the scan-kernel events are re-recorded every step: read them now
            ends[k].synchronize()
            fscan.append(ev["f0"].elapsed_time(ev["f1"]))
            if backward:
                bscan.append(ev["b0"].elapsed_time(ev["b1"]))
        torch.cuda.synchronize()
    launches = _lib.rnn_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    # the same steps back to back without the L2 flush (Wx of a small workload
    # may stay in the 129 MB L2): reported beside the flushed number, not as it
    warm = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    nwarm = min(args.steps, 10)
    torch.cuda.synchronize()
    warm[0].record()
    for _ in range(nwarm):
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, tape, ws)
        if backward:
            _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, tape, inp["dstates"],
                         None, dWx, dR, db, ds0, ws)
    warm[1].record()
    torch.cuda.synchronize()
    warm_ms = warm[0].elapsed_time(warm[1]) / nwarm
    _lib.rnn_check_status(ws)
    _lib.rnn_profile_events(0, None, None)
    _lib.rnn_profile_events(1, None, None)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    fwd_ms = [s.elapsed_time(m) for s, m in zip(starts, mids)]
    ms_per_step, value, fwd_value = aggregate(sum(step_ms), sum(fwd_ms), world, B * T, args.steps, dev)
    fwd_tot = fwd_value and world * B * T / fwd_value * 1e3 * args.steps

    pk = peaks()
    alg = algorithmic(w, fn, esize)
    f_ms = statistics.mean(fscan)
    b_ms = statistics.mean(bscan) if bscan else 0.0
    # per-step roofline of the method (max of tensor time and HBM time), per the metric
    roof_f = max(alg["fwd_flops"] / (pk["bf16"] * 1e12), alg["fwd_bytes"] / (pk["hbm"] * 1e9))
    roof_b = max(alg["bwd_flops"] / (pk["bf16"] * 1e12), alg["bwd_bytes"] / (pk["hbm"] * 1e9)) if backward else 0
    dom_bwd = backward and b_ms > f_ms
    kms = b_ms if dom_bwd else f_ms
    kbytes = alg["bwd_bytes"] if dom_bwd else alg["fwd_bytes"]
    kflops = alg["bwd_flops"] if dom_bwd else alg["fwd_flops"]
    hbm_bound = kbytes / (pk["hbm"] * 1e9) >= kflops / (pk["bf16"] * 1e12)
    if hbm_bound:
        achieved = kbytes / (kms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": None}
    else:
        achieved = kflops / (kms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16"], "traffic": None}
    plan_path = (plan_b if dom_bwd else plan_f).split()[0].split("=")[1]
    kname = {("fused", False): "fused_fwd_kernel", ("grid", False): "fused_fwd_kernel",
             ("fused", True): "fused_bwd_kernel", ("grid", True): "grid_bwd_kernel",
             ("alternating", False): "alt_fwd_step", ("alternating", True): "alt_bwd_step"}.get(
        (plan_path, bool(dom_bwd)), f"simt_{'bwd' if dom_bwd else 'fwd'}_kernel")
    roof["traffic"] = measured_traffic(kname, w["name"])
    roof.update({"kernel": kname, "kernel_ms": kms,
                 "peak_source": f"{pk['source']} (MEASURED_PEAKS.json, burst)" if pk["source"] == "measured"
                 else "fallback"})

    result = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
              "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
              "vs_baseline": None, "dtype": "bf16" if dtype == torch.bfloat16 else "f32",
              "data": "synthetic",
              "config": workload_config(w, fn, world),
              "plan": {"fwd": plan_f, "bwd": plan_b, "placement": placement()},
              "fwd_value": fwd_value, "fwd_ms": fwd_tot / args.steps,
              "warm_l2": {"value": B * T / (warm_ms / 1e3), "ms_per_step": warm_ms, "steps": nwarm,
                          "note": "this rank, steps back to back without the flush"},
              "scan_ms": {"fwd": f_ms, "bwd": b_ms},
              "per_step_roofline": {"fwd_ns": roof_f / T * 1e9, "fwd_frac": roof_f / (f_ms / 1e3),
                                    "bwd_ns": roof_b / T * 1e9,
                                    "bwd_frac": (roof_b / (b_ms / 1e3)) if backward else None,
                                    "step_frac": (roof_f + roof_b) / (ms_per_step / 1e3)},
              "step_latency_ns": {"fwd": f_ms * 1e6 / T, "bwd": (b_ms * 1e6 / T) if backward else None},
              "roofline": roof, "gpu_launches": launches}
    result["clocks"] = clk.summary()

    # ---- latency floor of the cluster exchange (outside the timed region): the
    # forward's per-step h exchange alone, for the plan's cluster size and slice
    if plan_f.startswith("path=fused"):
        pf = dict(kv.split("=") for kv in plan_f.split()[1:] if "=" in kv)
        C, U, NT = int(pf["C"]), int(pf["U"]), int(pf["NT"])
        slice_bytes = min(B, 8 * NT) * (U + 8) * 2
        fl = torch.zeros(2, dtype=torch.int64, device=dev)
        _lib.rnn_exchange_floor(C, slice_bytes, 2000, fl)
        torch.cuda.synchronize()
        cyc, st_fl = (int(x) for x in fl.cpu().tolist())
        mhz = result["clocks"].get("sm_mhz") or 2070.0
        fl_ns = cyc / mhz * 1e3
        result["latency_floor"] = {
            "what": f"h exchange alone: cluster of {C}, {slice_bytes} B bulk copy to each peer per step",
            "cycles_per_step": cyc, "ns_per_step": fl_ns, "status": st_fl,
            "fwd_step_over_floor": (f_ms * 1e6 / T) / fl_ns if fl_ns > 0 else None}

    if plan_f.startswith("path=grid"):
        pf = dict(kv.split("=") for kv in plan_f.split()[1:] if "=" in kv)
        C, NT, groups = int(pf["C"]), int(pf["NT"]), int(pf["groups"])
        rows = min(B, 8 * NT)
        scratch = torch.empty(2 * groups * rows * D * 2 + 32768, dtype=torch.uint8, device=dev)
        fl = torch.zeros(2, dtype=torch.int64, device=dev)
        _lib.rnn_exchange_floor_grid(C, groups, rows, D, 2000, scratch, fl)
        torch.cuda.synchronize()
        cyc, st_fl = (int(x) for x in fl.cpu().tolist())
        mhz = result["clocks"].get("sm_mhz") or 2070.0
        fl_ns = cyc / mhz * 1e3
        result["latency_floor"] = {
            "what": f"h exchange alone through L2: {groups} groups of {C} CTAs, {rows} rows of {D} bf16 pulled per "
                    f"step after a release/acquire step counter; CTAs placed as the grid kernels place theirs "
                    f"({placement()})",
            "cycles_per_step": cyc, "ns_per_step": fl_ns, "status": st_fl,
            "fwd_step_over_floor": (f_ms * 1e6 / T) / fl_ns if fl_ns > 0 else None}

    # ---- the configuration the per-step roofline target is stated on (LSTM fp32
    # B=2 T=16 N=1 D=32), measured in this run after the main measurement
    if not args.no_target_config and args.workload != 1:
        result["target_config"] = target_config_fracs(dev)

    # ---- e2e through the C ABI with host buffers (pinned), copies inside the window.
    # Every step copies all its inputs host -> device (Wx, R, b, the initial
    # states and the upstream gradients) and reads its result device -> host:
    # the parameter gradients dR and db, the initial-state gradients and the
    # last states (the forward alone: the states and the last states). The
    # per-step states and dWx stay on the device, where the neighbouring layers
    # of a model consume them. The copies overlap the compute, as a training
    # loop prefetching its batches would run them: the inputs in three buffer
    # sets (a step's inputs are copied while the two steps before it compute,
    # so one slow host-to-device copy does not stall the next step), the
    # outputs in two, on a host-to-device and a device-to-host stream.
    if not args.no_e2e:
        NIN = 3
        hin = [{k: v.pin_memory() for k, v in host.items() if v is not None} for _ in range(NIN)]
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in hin[0].items()} for _ in range(NIN)]
        out0 = [states, last] + ([dWx, dR, db, ds0] if backward else [])
        outs = [out0, [torch.empty_like(o) for o in out0]]
        read = [1, 3, 4, 5] if backward else [0, 1]  # which outputs are the step's result read back
        hout = [[torch.empty(out0[r].shape, dtype=out0[r].dtype, pin_memory=True) for r in read] for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in hin[0].values())
        d2h = sum(out0[r].numel() * out0[r].element_size() for r in read)
        cs = torch.cuda.current_stream()
        hs, ds = torch.cuda.Stream(), torch.cuda.Stream()
        ev_h2d = [torch.cuda.Event() for _ in range(NIN)]
        ev_free = [torch.cuda.Event() for _ in range(NIN)]  # the compute is done with an input set
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_free + ev_done + ev_out:
            e.record(cs)

        def e2e_step(k):
            i, j = k % NIN, k % 2
            with torch.cuda.stream(hs):
                hs.wait_event(ev_free[i])  # the compute of step k-3 is done with dev_in[i]
                for key, v in hin[i].items():
                    dev_in[i][key].copy_(v, non_blocking=True)
                ev_h2d[i].record(hs)
            cs.wait_event(ev_h2d[i])
            cs.wait_event(ev_out[j])  # step k-2's outputs have reached the host
            o = outs[j]
            x = dev_in[i]
            _lib.rnn_fwd(dims, x["Wx"], x["R"], x["b"], x["states0"], o[0], o[1], tape, ws)
            if backward:
                _lib.rnn_bwd(dims, x["Wx"], x["R"], x["b"], x["states0"], o[0], tape, x["dstates"], None,
                             o[2], o[3], o[4], o[5], ws)
            ev_free[i].record(cs)
            ev_done[j].record(cs)
            with torch.cuda.stream(ds):
                ds.wait_event(ev_done[j])
                for r, t_host in zip(read, hout[j]):
                    t_host.copy_(o[r], non_blocking=True)
                ev_out[j].record(ds)

        for k in range(args.warmup):
            e2e_step(k)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        hs.wait_stream(cs)
        ds.wait_stream(cs)
        for k in range(args.steps):
            e2e_step(k)
        cs.wait_stream(hs)
        cs.wait_stream(ds)
        e1.record(cs)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        if world > 1:
            t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t[0])
        result["e2e"] = {"value": world * B * T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                         "copies": "every step: all inputs host->device; the result device->host: "
                                   + ("dR, db, dstates0 and the last states" if backward else
                                      "the states and the last states")
                                   + " (pinned), overlapped with the compute on two copy streams (inputs "
                                     "copied up to two steps ahead, three input buffer sets); the per-step "
                                     "states and dWx stay on the device"}

    # ---- the oracle on the host cores (rank 0, N=1 only), bounded sample
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        rows, steps = oracle_sample(w, fn, cores)
        dt = cpu_oracle_step(fn, host, cores, rows, steps, backward)
        result["cpu_baseline"] = {"value": rows * steps / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
                                  "sample": f"{fn} {'fwd+bwd' if backward else 'fwd'}, {rows} of {B} batch rows x "
                                            f"{steps} of {T} steps, N={N}, D={D}, fp64, {dt:.1f} s"}
        # the same oracle on one core, over a shorter time prefix
        steps1 = max(8, steps // max(1, cores))
        dt1 = cpu_oracle_step(fn, host, 1, rows, steps1, backward)
        result["cpu_baseline"]["single_thread"] = {
            "value": rows * steps1 / dt1, "unit": UNIT, "cores": 1,
            "sample": f"{rows} of {B} batch rows x {steps1} of {T} steps, {dt1:.1f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
