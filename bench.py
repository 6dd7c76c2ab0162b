#!/usr/bin/env python3
"""Benchmark of the fused chunk-scheduled AG-GEMM / GEMM-RS / GEMM-AR on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  AG-GEMM  Llama-3-8B FFN up-projection, TP=8   (M=8192, K=4096, N=1792)
  GEMM-AR  Qwen2-7B FFN down-projection, TP=8   (M=4096, K=2368, N=3584)
  GEMM-RS  Llama-3-8B FFN down-projection, TP=8 (M=8192, K=1792, N=4096, send on)
each as one fused chunk-scheduled call through the C ABI, the 7 other ranks
simulated in the same HBM (Syncopate summary page, Experiments, paper §6.1).
In this order the tensor-bound AG-GEMM follows GEMM-RS and absorbs the
write-back of its 125 MB of outputs, which would otherwise fall on the
HBM-bound GEMM-AR (measured: step 293.6 vs 295.4 us).

Metric: TFLOP/s over the step (2*M*N*K summed over the three operators), with
each operator's fraction of its roofline beside it.  Inputs are resident in
HBM before the timed region; the step streams ~2 GB, far more than the 135 MB
L2, so no explicit flush is needed between steps.  `e2e` repeats the
measurement with the inputs copied from pinned host memory and the bf16
outputs copied back inside the timed region.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch with torch.distributed.run: every rank runs an independent
replica (the tensor-parallel ranks are already simulated inside one GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunk_scheduled_communication_gb300 import tuned  # noqa: E402
from chunk_scheduled_communication_gb300 import workloads as wl  # noqa: E402

METRIC = "fused AG-GEMM/GEMM-RS/GEMM-AR TFLOPS and % of roofline on 1 GB300"
UNIT = "TFLOP/s"
WORKLOAD_NAME = ("llama3-8b-ffn-tp8 step: AG-GEMM up (8192x4096x1792) + qwen2-7b GEMM-AR down "
                 "(4096x2368x3584) + GEMM-RS down (8192x1792x4096, send)")
STEP = [wl.LLAMA3_8B_UP_AG, wl.QWEN2_7B_DOWN_AR, wl.LLAMA3_8B_DOWN_RS]

# Knobs per operator: the autotuner's cache entries where present, else the
# measured best points (shared with the parity tests).
DEFAULT_KNOBS, KNOBS_SOURCE = tuned.bench_knobs()
# A2A-GEMM (the MoE all-to-all + expert GEMM) is measured beside the step, on
# its own line of the JSON ("a2a"), not inside the headline value.
A2A = wl.MIXTRAL_8X7B_EXPERT_UP_A2A

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic_bytes(w: wl.Workload, with_send=True, with_publish=False, rows_from=None, r=0) -> float:
    """Bytes the method must move through this HBM (each operand read once,
    each output written once; AG: staged peer shards read + written; RS/AR:
    each peer byte read once; RS: the fp32 send rows; AR: the fp32 publish of
    the local partial only when it is written -- the measured step leaves it
    NULL, since every AR flop already feeds `out`)."""
    M, N, K, R = w.M, w.N, w.K, w.R
    if w.op == "a2a":  # AG-GEMM over unequal blocks: every non-local row staged
        M = sum(rows_from)
        staged = (M - rows_from[r]) * K * 2
        return M * K * 2 + K * N * 2 + M * N * 2 + 2 * staged
    if w.op == "ag":
        staged = (R - 1) * w.M_r * K * 2
        return M * K * 2 + K * N * 2 + M * N * 2 + 2 * staged
    if w.op == "rs":
        peers = (R - 1) * w.M_r * N * 4
        send = (R - 1) * w.M_r * N * 4 if with_send else 0
        return M * K * 2 + K * N * 2 + peers + send + w.M_r * N * 2
    publish = M * N * 4 if with_publish else 0
    return M * K * 2 + K * N * 2 + (R - 1) * M * N * 4 + publish + M * N * 2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunk_scheduled_communication_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cuh", ".cu", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(op: str):
    """DRAM traffic per launch recorded from an ncu capture of the current
    kernel sources (profiles/dram_traffic.txt lines: `op src_hash bytes`);
    None when absent or when the kernels changed since the capture."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash()
    for line in open(p):
        parts = line.split("#")[0].split()
        if len(parts) >= 3 and parts[0] == op and parts[1] == cur:
            return float(parts[2])
    return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                smax.append(float(f[2].split()[0]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = os.environ.get("SYN_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def barrier(dist, dev=None):
    if dist is not None:
        if dev is not None:
            dist.barrier(device_ids=[dev])
        else:
            dist.barrier()


def max_over_ranks(dist, x: float, dev=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=f"cuda:{dev}" if dev is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle arm
def oracle_sample(inputs, frac: float):
    """Run the CPU oracle on `frac` of each operator's output rows (at least
    one row each).  Returns (seconds, flops, description)."""
    import oracle
    flops = 0.0
    desc = []
    t0 = time.perf_counter()
    for w, inp in zip(STEP, inputs):
        if w.op == "ag":
            rows = max(1, int(w.M * frac))
            oracle.ag_gemm(inp.shards, inp.B, 0, rows, want_gathered=False)
        elif w.op == "rs":
            rows = max(1, int(w.M_r * frac))
            oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, 0, 0, rows)
            srows = max(1, int((w.M - w.M_r) * frac))
            oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, 0, 0, 1, send_rows=(w.M_r, w.M_r + srows))
            rows = rows + srows + 1
        else:
            rows = max(1, int(w.M * frac))
            oracle.gemm_ar(inp.A, inp.B, inp.peers, w.R, 0, 0, rows)
        flops += 2.0 * rows * w.N * w.K
        desc.append(f"{w.op}:{rows} rows")
    return time.perf_counter() - t0, flops, ", ".join(desc)


def run_reference(args, dist, rank):
    """`--impl reference`: the CPU oracle timed on the host cores."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    inputs = [wl.make_inputs(w, r=0, seed=0) for w in STEP]
    # size each step so the whole run ends within a few minutes
    t_cal, f_cal, _ = oracle_sample(inputs, 1.0 / 1024)
    rate = f_cal / max(t_cal, 1e-6)
    full = sum(w.flops for w in STEP)
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    frac = min(1.0, max(1.0 / 8192, budget * rate / full))
    for _ in range(args.warmup):
        oracle_sample(inputs, frac)
    tot_t, tot_f, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        t, f, desc = oracle_sample(inputs, frac)
        tot_t += t
        tot_f += f
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal, Llama-3/Qwen FFN shapes)",
            "config": {"workload": WORKLOAD_NAME, "parallelism": f"tp8 simulated in one device x{args.gpus}"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"per step {desc} ({frac:.5f} of each operator's rows)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="syn", choices=["syn", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-frac", type=float, default=1.0,
                    help="fraction of each operator's rows the CPU oracle baseline computes")
    ap.add_argument("--no-baselines", action="store_true")
    ap.add_argument("--knobs", default="", help="JSON overriding the per-operator knobs")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the step: the Llama-3-70B AG-GEMM sweep (splits 1-8, tile order, "
                         "backend, comm SMs), one JSON line per point")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    dist, rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, dist, rank)
    if args.sweep:
        return run_sweep(args)

    import torch

    from chunk_scheduled_communication_gb300 import runner, syn

    torch.cuda.set_device(local)
    syn.lib()  # raises if the CUDA library is missing: there is no fallback
    knobs = {k: dict(v) for k, v in DEFAULT_KNOBS.items()}
    if args.knobs:
        for k, v in json.loads(args.knobs).items():
            knobs[k].update(v)
    peaks, peak_src = load_peaks()

    host_inputs = [wl.make_inputs(w, r=0, seed=0) for w in STEP]
    devs, plans = [], []
    for w, inp in zip(STEP, host_inputs):
        d = runner.upload(inp, with_f32_out=(w.op == "rs"))  # RS: send rows; AR: publish NULL
        kn = dict(knobs[w.op])
        split, order = kn.pop("split"), kn.pop("order")
        plans.append(runner.make_plan(d, split=split, order=order, **kn))
        devs.append(d)
    stream = torch.cuda.current_stream()
    n_ops = len(STEP)

    def step():
        for p, d in zip(plans, devs):
            runner.call(p, d, stream)

    for _ in range(args.warmup):
        step()
    for p in plans:
        p.check(stream)

    # ---------------- timed region (device-resident inputs) ----------------
    # The step loop carries no event between its kernels: an event recorded
    # between two launches costs the second its programmatic early launch
    # (measured: 288.9 us per step with per-operator events, 274.5 without).
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist, local)
    torch.cuda.synchronize()
    e0.record(stream)
    for k in range(args.steps):
        for p, d in zip(plans, devs):
            runner.call(p, d, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    for p in plans:
        p.check(stream)
    total_ms = e0.elapsed_time(e1)
    total_ms = max_over_ranks(dist, total_ms, local)
    ms_per_step = total_ms / args.steps

    # Each operator's launch duration: the kernel alone, `steps` back-to-back
    # calls between two events on the launching stream (inputs larger than
    # L2).  Beside it, the same operator inside the step bracketed by events
    # (which also pays for the previous operator's L2 write-back and for the
    # events themselves).
    op_ms = []
    for p, d in zip(plans, devs):
        for _ in range(3):
            runner.call(p, d, stream)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(max(args.steps, 20)):
            runner.call(p, d, stream)
        a1.record(stream)
        torch.cuda.synchronize()
        op_ms.append(max_over_ranks(dist, a0.elapsed_time(a1), local) / max(args.steps, 20))
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ops)]
          for _ in range(args.steps)]
    for k in range(args.steps):
        for i, (p, d) in enumerate(zip(plans, devs)):
            ev[k][i][0].record(stream)
            runner.call(p, d, stream)
            ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    for p in plans:
        p.check(stream)
    in_step_ms = [statistics.fmean(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                  for i in range(n_ops)]
    step_flops = sum(w.flops for w in STEP)
    value = step_flops * world / (ms_per_step * 1e-3) / 1e12

    # Tensor denominator: the sustained bf16 figure only when the timed loop
    # ran long enough to settle under the power cap (>= 1 s) and the SM clock
    # actually dropped (median more than 5 % below max); otherwise the kernels
    # ran at burst conditions and the burst figure applies.
    timed_s = (total_ms + sum(op_ms) * max(args.steps, 20) + sum(in_step_ms) * args.steps) * 1e-3
    sm_med, sm_max = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    clock_low = bool(sm_med and sm_max and sm_med < 0.95 * sm_max)
    if timed_s >= 1.0 and clock_low:
        tensor_peak, peak_kind = peaks["bf16_tflops_sustained"], "sustained bf16"
        peak_why = f"timed region {timed_s:.2f} s, median SM clock {sm_med:.0f} of {sm_max:.0f} MHz"
    else:
        tensor_peak, peak_kind = peaks["bf16_tflops"], "burst bf16"
        peak_why = (f"timed region {timed_s:.3f} s, median SM clock "
                    f"{(f'{sm_med:.0f}' if sm_med else '?')} of {(f'{sm_max:.0f}' if sm_max else '?')} MHz")
    per_op = {}
    for w, ms, ms_step in zip(STEP, op_ms, in_step_ms):
        byts = algorithmic_bytes(w)
        t_roof = max(w.flops / (tensor_peak * 1e12), byts / (peaks["hbm_gbs"] * 1e9))
        per_op[w.op] = {"workload": w.name, "us": ms * 1e3, "in_step_us_with_events": ms_step * 1e3,
                        "tflops": w.flops / (ms * 1e-3) / 1e12,
                        "gbs": byts / (ms * 1e-3) / 1e9, "algorithmic_bytes": byts,
                        "roofline_frac": t_roof / (ms * 1e-3),
                        "roofline_frac_burst_peak": max(w.flops / (peaks["bf16_tflops"] * 1e12),
                                                        byts / (peaks["hbm_gbs"] * 1e9)) / (ms * 1e-3),
                        "roofline_frac_sustained_peak": max(
                            w.flops / (peaks["bf16_tflops_sustained"] * 1e12),
                            byts / (peaks["hbm_gbs"] * 1e9)) / (ms * 1e-3),
                        "bound": "tensor" if w.flops / (tensor_peak * 1e12) >= byts / (peaks["hbm_gbs"] * 1e9) else "hbm",
                        "knobs": knobs[w.op], "knobs_source": KNOBS_SOURCE.get(w.op)}
    dom = max(per_op, key=lambda k: per_op[k]["us"])
    dw = STEP[[w.op for w in STEP].index(dom)]
    if per_op[dom]["bound"] == "tensor":
        achieved, peak, unit = per_op[dom]["tflops"], tensor_peak, "TFLOP/s"
    else:
        achieved, peak, unit = per_op[dom]["gbs"], peaks["hbm_gbs"], "GB/s"
    roofline = {"bound": per_op[dom]["bound"], "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": recorded_traffic(dom), "kernel": f"syn_fused_kernel<{dom}>",
                "workload": dw.name,
                "peak_source": f"{peak_src} ({peak_kind if unit == 'TFLOP/s' else 'copy'})",
                "peak_choice": peak_why,
                "duration": "mean launch duration of the kernel alone: back-to-back calls on the launching "
                            "stream between two CUDA events, inputs larger than L2",
                "algorithmic_per_launch": dw.flops if unit == "TFLOP/s" else algorithmic_bytes(dw)}

    # ---------------- end to end: pinned host inputs in, bf16 outputs out ----------------
    import torch as _t
    pinned = []
    h2d = d2h = 0
    for w, inp, d in zip(STEP, host_inputs, devs):
        pairs = []
        if w.op == "ag":
            for q in range(w.R):
                h = _t.from_numpy(inp.shards[q].view(np.int16)).view(_t.bfloat16).pin_memory()
                pairs.append((h, d.shards[q]))
        else:
            pairs.append((_t.from_numpy(inp.A.view(np.int16)).view(_t.bfloat16).pin_memory(), d.A))
            # the peers' partials the operator reads: GEMM-AR all rows; GEMM-RS
            # only the rows of the local block (the rows a reduce-scatter delivers
            # to this rank; the kernel reads no other row of a peer's partial)
            rows = slice(0, w.M) if w.op == "ar" else slice(inp.r * w.M_r, (inp.r + 1) * w.M_r)
            for q in range(w.R):
                if d.peers[q] is not None:
                    h = _t.from_numpy(np.ascontiguousarray(inp.peers[q][rows])).pin_memory()
                    pairs.append((h, d.peers[q][rows]))
        pairs.append((_t.from_numpy(inp.B.view(np.int16)).view(_t.bfloat16).pin_memory(), d.B))
        out_h = _t.empty(d.out.shape, dtype=d.out.dtype).pin_memory()
        pinned.append((pairs, out_h, d.out))
        h2d += sum(h.numel() * h.element_size() for h, _ in pairs)
        d2h += out_h.numel() * out_h.element_size()

    # Three streams: inputs in, compute, outputs out (the host link is full duplex).
    # Operator k's kernel waits for its inputs; its output copy waits for the
    # kernel; the next step's input copy of operator k waits until the kernel
    # has read the previous inputs, and its kernel until the previous output
    # has been copied out.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n_ops = len(pinned)
    ev = {k: [torch.cuda.Event() for _ in range(n_ops)] for k in ("in", "done", "out")}
    first = [True]

    def e2e_step():
        for k, ((pairs, out_h, out_d), p, d) in enumerate(zip(pinned, plans, devs)):
            if not first[0]:
                s_in.wait_event(ev["done"][k])
            with torch.cuda.stream(s_in):
                for h, dd in pairs:
                    dd.copy_(h, non_blocking=True)
            ev["in"][k].record(s_in)
            stream.wait_event(ev["in"][k])
            if not first[0]:
                stream.wait_event(ev["out"][k])
            runner.call(p, d, stream)
            ev["done"][k].record(stream)
            s_out.wait_event(ev["done"][k])
            with torch.cuda.stream(s_out):
                out_h.copy_(out_d, non_blocking=True)
            ev["out"][k].record(s_out)
        first[0] = False

    e2e_step()
    torch.cuda.synchronize()
    barrier(dist, local)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    s_in.wait_event(a0)  # the timed region starts before the first input copy
    for _ in range(args.e2e_steps):
        e2e_step()
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, a0.elapsed_time(a1), local) / args.e2e_steps
    for p in plans:
        p.check(stream)
    e2e = {"value": step_flops * world / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---------------- per-call distribution (rank 0): warm and L2-cold ----------------
    # 5 warm-up calls, then 50 calls each between CUDA events: back to back
    # ("warm"), and with a 512 MB buffer rewritten before each call ("cold",
    # the flush outside the events).  Plus the share of CTA time spent waiting
    # on chunk flags, from a traced plan (trace = 1).
    per_call = {}
    if rank == 0 and not args.no_baselines:
        flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=stream.device)
        for w, p, d in zip(STEP, plans, devs):
            res = {}
            for mode in ("warm", "cold"):
                for _ in range(5):
                    runner.call(p, d, stream)
                ts = []
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(50)]
                for a, b in evs:
                    if mode == "cold":
                        flush.fill_(1.0)
                    a.record(stream)
                    runner.call(p, d, stream)
                    b.record(stream)
                torch.cuda.synchronize()
                ts = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
                res[mode] = {"p10_us": ts[4], "median_us": ts[24], "p90_us": ts[44]}
            p.check(stream)
            kn = dict(knobs[w.op])
            split, order = kn.pop("split"), kn.pop("order")
            with runner.make_plan(d, split=split, order=order, trace=1, **kn) as tp:
                for _ in range(20):
                    runner.call(tp, d, stream)
                tp.check(stream)
                wait_ns, busy_ns = tp.stats()
            res["flag_wait_share"] = wait_ns / busy_ns if busy_ns else None
            per_call[w.op] = res
        del flush

    # ---------------- comparisons (rank 0): unfused / decomposed baselines, cuBLAS+copy ----------------
    baselines = {}
    if rank == 0 and not args.no_baselines:
        for w, inp, d in zip(STEP, host_inputs, devs):
            res = {}
            for be in ("unfused", "decomposed", "decomposed_per_shard"):
                kn = dict(knobs[w.op])
                split, order = kn.pop("split"), kn.pop("order")
                kn["backend"] = "decomposed" if be.startswith("decomposed") else be
                kn["stages"] = 0  # the default depth of the baseline kernel instance
                kn.pop("direct_fetch", None)
                if be in ("unfused", "decomposed_per_shard"):
                    # unfused: the whole copy in one piece per source; decomposed
                    # per shard: one GEMM launch per source shard / rank block
                    split = 1
                with runner.make_plan(d, split=split, order=order, **kn) as bp:
                    for _ in range(5):
                        runner.call(bp, d, stream)
                    bp.check(stream)
                    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    reps = 200
                    b0.record(stream)
                    for _ in range(reps):
                        runner.call(bp, d, stream)
                    b1.record(stream)
                    torch.cuda.synchronize()
                    bp.check(stream)
                    res[f"{be}_us"] = b0.elapsed_time(b1) / reps * 1e3
            res["fused_us"] = per_op[w.op]["us"]
            res["fused_speedup_vs_unfused"] = res["unfused_us"] / res["fused_us"]
            res["cublas_plus_copy_us"] = cublas_plus_copy_us(w, d, stream)
            baselines[w.op] = res

    a2a = measure_a2a(knobs["a2a"], peaks, stream) if rank == 0 and not args.no_baselines else None
    extra = {}
    if rank == 0 and not args.no_baselines:
        extra["cfg5"] = measure_cfg5(peaks, stream)
        extra["ar_split"] = measure_ar_split(peaks, stream)
        extra["rs_staged"] = measure_rs_variants(peaks, stream)
        extra["wave_quantization"] = measure_wave_quantization(peaks, stream)
    ring_attn = measure_attention(peaks, stream) if rank == 0 and not args.no_baselines else None

    # ---------------- CPU oracle baseline (rank 0, N = 1) ----------------
    cpu = None
    if rank == 0 and world == 1 and args.cpu_frac > 0:
        import oracle
        oracle.build()
        t, f, desc = oracle_sample(host_inputs, args.cpu_frac)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
               "seconds": t, "sample": f"{desc} of the same workload (seed 0, rank 0)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded normal; no dataset or weights)",
                "config": {"workload": WORKLOAD_NAME, "global_batch": None, "seq_len": None,
                           "parallelism": f"tp8 simulated in one device, {world} replica(s)",
                           "l2": "inputs > L2 (each step streams ~2 GB through the 135 MB L2); no flush"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": sum(launches_per_call(p) for p in plans) * args.steps,
                "per_call": per_call,
                "clocks": clk, "per_op": per_op, "baselines": baselines, "a2a": a2a, "ring_attention": ring_attn,
                **extra,
                "peaks": {**peaks, "source": peak_src}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """The pages' tuning-space study on the Llama-3-70B FFN up-projection AG-GEMM
    (Syncopate summary, §6.3, Fig. 11): chunk splits 1-8 x tile order x staging
    backend x communication SMs, each point timed with CUDA events (median of
    --steps calls after --warmup), next to the unfused baseline."""
    import torch

    from chunk_scheduled_communication_gb300 import runner, syn

    torch.cuda.set_device(0)
    syn.lib()
    peaks, peak_src = load_peaks()
    w = wl.LLAMA3_70B_UP_AG
    d = runner.upload(wl.make_inputs(w, r=0, seed=0))
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 20))
    points = [dict(backend="unfused", split=1, order="row", tile_m=256)]
    for split in range(1, 9):
        for order in ("row", "grouped", "col"):
            points.append(dict(backend="ce", split=split, order=order, tile_m=256))
            points.append(dict(backend="tma_colocated", split=split, order=order, tile_m=256))
            points.append(dict(backend="ldst_colocated", split=split, order=order, tile_m=256))
        for cs in (4, 8, 16):
            points.append(dict(backend="tma_dedicated", split=split, order="row", comm_sms=cs, tile_m=256))
            points.append(dict(backend="ldst_dedicated", split=split, order="row", comm_sms=cs, tile_m=256))
    for pt in points:
        kn = dict(pt)
        split, order = kn.pop("split"), kn.pop("order")
        with runner.make_plan(d, split=split, order=order, **kn) as plan:
            for _ in range(args.warmup):
                runner.call(plan, d, stream)
            plan.check(stream)
            times = []
            for _ in range(steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                runner.call(plan, d, stream)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            plan.check(stream)
        us = statistics.median(times) * 1e3
        # each point runs alone (a burst of calls): burst tensor peak
        t_roof = max(w.flops / (peaks["bf16_tflops"] * 1e12), algorithmic_bytes(w) / (peaks["hbm_gbs"] * 1e9))
        print(json.dumps({"sweep": w.name, **pt, "us": us, "tflops": w.flops / us / 1e6,
                          "roofline_frac": t_roof / (us * 1e-6), "peak_source": f"{peak_src} (burst)"}),
              flush=True)
    return 0


def measure_a2a(knobs, peaks, stream, reps=50):
    """A2A-GEMM on the expert-parallel MoE workload (rank 0's expert), timed
    alone: CUDA events around `reps` back-to-back calls after warm-up, the
    unfused baseline (all copies, then the GEMM) the same way, cuBLAS + copy
    for context (the same number of back-to-back calls, so all three run
    equally long under the power cap), and the flag-wait share from a traced
    plan."""
    import torch

    from chunk_scheduled_communication_gb300 import runner
    w, r = A2A, 0
    inp = wl.make_inputs(w, r=r, seed=0)
    d = runner.upload(inp)
    M = sum(inp.rows_from)
    flops = 2.0 * M * w.N * w.K
    byts = algorithmic_bytes(w, rows_from=inp.rows_from, r=r)

    def timed(kn):
        kn = dict(kn)
        split, order = kn.pop("split"), kn.pop("order")
        with runner.make_plan(d, split=split, order=order, **kn) as p:
            for _ in range(10):
                runner.call(p, d, stream)
            p.check(stream)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(reps):
                runner.call(p, d, stream)
            b1.record(stream)
            torch.cuda.synchronize()
            p.check(stream)
            return b0.elapsed_time(b1) / reps * 1e3, launches_per_call(p)

    us, launches = timed(knobs)
    unfused_us, _ = timed({**knobs, "backend": "unfused", "stages": 0})
    kn = dict(knobs)
    split, order = kn.pop("split"), kn.pop("order")
    with runner.make_plan(d, split=split, order=order, trace=1, **kn) as tp:
        for _ in range(20):
            runner.call(tp, d, stream)
        tp.check(stream)
        wait_ns, busy_ns = tp.stats()
    t_burst = max(flops / (peaks["bf16_tflops"] * 1e12), byts / (peaks["hbm_gbs"] * 1e9))
    return {"workload": w.name, "rank": r, "rows_from": inp.rows_from, "M": M, "N": w.N, "K": w.K,
            "us": us, "tflops": flops / (us * 1e-6) / 1e12, "algorithmic_bytes": byts,
            "bound": "tensor" if flops / (peaks["bf16_tflops"] * 1e12) >= byts / (peaks["hbm_gbs"] * 1e9) else "hbm",
            "roofline_frac_burst_peak": t_burst / (us * 1e-6),
            "unfused_us": unfused_us, "fused_speedup_vs_unfused": unfused_us / us,
            "cublas_plus_copy_us": cublas_plus_copy_us(w, d, stream),
            "flag_wait_share": wait_ns / busy_ns if busy_ns else None,
            "gpu_launches_per_call": launches, "knobs": knobs}


def measure_attention(peaks, stream, reps=20):
    """Ring attention (sequence parallel, chunk-scheduled KV exchange) on the
    Llama-3-8B 32K-context shape, timed alone: CUDA events around `reps`
    back-to-back calls after warm-up; the same kernel after copying every KV
    shard first ("unfused"); torch's scaled_dot_product_attention on the
    gathered keys as context."""
    import torch

    from chunk_scheduled_communication_gb300 import attn

    def dev(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()

    out = {}
    for w, r in ((wl.LLAMA3_8B_RING_ATTN, 0), (wl.LLAMA3_8B_RING_ATTN_CAUSAL, wl.LLAMA3_8B_RING_ATTN_CAUSAL.R - 1)):
        Q, Ks, Vs = wl.make_attn_inputs(w, 0)
        kg = torch.zeros((w.R * w.S_r, w.H_kv, w.d), dtype=torch.bfloat16, device="cuda")
        vg = torch.zeros_like(kg)
        ks, vs = [dev(k) for k in Ks], [dev(v) for v in Vs]
        sl = slice(r * w.S_r, (r + 1) * w.S_r)
        kg[sl], vg[sl] = ks[r], vs[r]
        ks[r], vs[r] = kg[sl], vg[sl]
        q = dev(Q)
        O = torch.empty((w.S_r, w.H_q, w.d), dtype=torch.bfloat16, device="cuda")
        res = {"workload": w.name, "rank": r, "flops": w.flops}
        for be in ("tma_colocated", "unfused"):
            with attn.AttnPlan(R=w.R, rank=r, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, causal=w.causal,
                               backend=be) as p:
                for _ in range(3):
                    p.run(q, ks, vs, kg, vg, O, stream=stream)
                p.check(stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    p.run(q, ks, vs, kg, vg, O, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize()
                p.check(stream)
            res[be + "_us"] = e0.elapsed_time(e1) / reps * 1e3
        us = res["tma_colocated_us"]
        res["tflops"] = w.flops / (us * 1e-6) / 1e12
        res["roofline_frac_burst_peak"] = res["tflops"] / peaks["bf16_tflops"]
        if not w.causal:  # (torch's masked path is not a flash kernel: no fair comparison)
            qq, kk, vv = (x.permute(1, 0, 2).unsqueeze(0) for x in (q, kg, vg))
            f = lambda: torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, enable_gqa=True)
            for _ in range(3):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                f()
            e1.record(stream)
            torch.cuda.synchronize()
            res["torch_sdpa_us"] = e0.elapsed_time(e1) / reps * 1e3
        if not w.causal:  # the ncu capture in profiles/ is of this launch (rank 0, non-causal)
            res["dram_traffic_per_launch"] = recorded_traffic("attn")
        out["causal" if w.causal else "full"] = res
    # head-parallel layout (the all-to-all form): rank 0's 4 query heads over all 32K tokens
    w = wl.LLAMA3_8B_RING_ATTN
    Qs, Ks, Vs = wl.make_head_attn_inputs(w, 0)
    hq, hkv = w.H_q // w.R, w.H_kv // w.R
    qs, ks, vs = [dev(x) for x in Qs], [dev(x) for x in Ks], [dev(x) for x in Vs]
    qg = torch.zeros((w.R * w.S_r, hq, w.d), dtype=torch.bfloat16, device="cuda")
    kg = torch.zeros((w.R * w.S_r, hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vg = torch.zeros_like(kg)
    O = torch.empty((w.R * w.S_r, hq, w.d), dtype=torch.bfloat16, device="cuda")
    res = {"workload": w.name.replace("ring-attn-sp8", "head-parallel-attn-hp8"), "rank": 0, "flops": w.flops}
    for be in ("tma_colocated", "unfused"):
        with attn.AttnPlan(R=w.R, rank=0, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, backend=be, head_parallel=True) as p:
            for _ in range(3):
                p.run_head(qs, ks, vs, qg, kg, vg, O, stream=stream)
            p.check(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                p.run_head(qs, ks, vs, qg, kg, vg, O, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            p.check(stream)
        res[be + "_us"] = e0.elapsed_time(e1) / reps * 1e3
    res["tflops"] = w.flops / (res["tma_colocated_us"] * 1e-6) / 1e12
    res["roofline_frac_burst_peak"] = res["tflops"] / peaks["bf16_tflops"]
    out["head_parallel"] = res
    return out


def time_calls(plan, d, stream, reps=20, warm=3) -> float:
    """Mean microseconds per call over `reps` back-to-back calls after `warm`
    untimed ones (CUDA events on the launching stream); checks the plan's
    error word afterwards."""
    import torch

    from chunk_scheduled_communication_gb300 import runner
    for _ in range(warm):
        runner.call(plan, d, stream)
    plan.check(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        runner.call(plan, d, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    plan.check(stream)
    return e0.elapsed_time(e1) / reps * 1e3


def measure_cfg5(peaks, stream):
    """The Llama-3-70B FFN up-projection AG-GEMM (the pages' tuning-space
    workload, Syncopate summary §6.3 / Fig. 11) at the best point of its sweep,
    timed alone (burst tensor peak), beside the unfused baseline and the
    flag-wait share of a traced plan."""
    from chunk_scheduled_communication_gb300 import runner
    w = wl.LLAMA3_70B_UP_AG
    d = runner.upload(wl.make_inputs(w, r=0, seed=0))
    split, order, kn = tuned.knobs_for("ag70")
    with runner.make_plan(d, split=split, order=order, **kn) as p:
        us = time_calls(p, d, stream)
    with runner.make_plan(d, split=split, order=order, **{**kn, "backend": "unfused", "stages": 0}) as p:
        unfused_us = time_calls(p, d, stream, reps=10)
    with runner.make_plan(d, split=split, order=order, trace=1, **kn) as p:
        time_calls(p, d, stream, reps=5, warm=1)
        wait_ns, busy_ns = p.stats()
    byts = algorithmic_bytes(w)
    t_roof = max(w.flops / (peaks["bf16_tflops"] * 1e12), byts / (peaks["hbm_gbs"] * 1e9))
    return {"workload": w.name, "knobs": tuned.STEP_KNOBS["ag70"], "us": us, "tflops": w.flops / us / 1e6,
            "roofline_frac_burst_peak": t_roof / (us * 1e-6), "unfused_us": unfused_us,
            "fused_speedup_vs_unfused": unfused_us / us, "flag_wait_share": wait_ns / busy_ns if busy_ns else None}


def measure_ar_split(peaks, stream):
    """GEMM-AR against chunk split and message size (the pages' GEMM-AR
    sensitivity, Syncopate summary §6.3 / Fig. 11: best near ~128 MB messages
    and 2-3 splits): the staged backends -- the copy engine and co-located TMA
    staging copy every peer partial into a receive buffer, chunk by chunk,
    and the epilogue waits on each chunk's flag -- at splits 1-4, for the
    Qwen2-7B shape (58.7 MB fp32 partial per rank) and the same layer over
    8192 tokens (117.4 MB), beside the resident-peer kernel the step uses."""
    from chunk_scheduled_communication_gb300 import runner
    out = []
    for w in (wl.QWEN2_7B_DOWN_AR, wl.scaled(wl.QWEN2_7B_DOWN_AR, M=8192)):
        d = runner.upload(wl.make_inputs(w, r=0, seed=0), with_f32_out=False)
        msg_mb = w.M * w.N * 4 / 1e6
        byts = algorithmic_bytes(w)
        pts = []
        for be in ("ce", "tma_colocated"):
            for split in (1, 2, 3, 4):
                with runner.make_plan(d, split=split, order="row", backend=be, tile_m=256, tile_n=256) as p:
                    us = time_calls(p, d, stream, reps=10)
                pts.append({"backend": be, "split": split, "us": us, "gbs": byts / us / 1e3})
        split, order, kn = tuned.knobs_for("ar")
        with runner.make_plan(d, split=split, order=order, **kn) as p:
            res_us = time_calls(p, d, stream, reps=20)
        best = min(pts, key=lambda x: x["us"])
        out.append({"workload": w.name, "message_mb_per_rank": msg_mb, "algorithmic_bytes": byts,
                    "staged": pts, "best_staged": best, "worst_over_best_staged": max(x["us"] for x in pts) / best["us"],
                    "resident_us": res_us, "resident_frac_hbm": byts / (res_us * 1e-6) / (peaks["hbm_gbs"] * 1e9)})
        del d
    return out


def measure_rs_variants(peaks, stream):
    """GEMM-RS beside the step's resident-peer pull kernel: staged backends
    whose epilogue waits on every peer chunk's flag (co-located TMA staging
    into the receive buffer, splits 1, 2, 4, with the flag-wait share), and
    the push mode (send rows added at the destination by TMA reduce-add),
    issued by the epilogue or by 8 / 32 dedicated push SMs."""
    from chunk_scheduled_communication_gb300 import runner
    w = wl.LLAMA3_8B_DOWN_RS
    d = runner.upload(wl.make_inputs(w, r=0, seed=0))
    split, order, kn = tuned.knobs_for("rs")
    with runner.make_plan(d, split=split, order=order, **kn) as p:
        pull_us = time_calls(p, d, stream)
    with runner.make_plan(d, split=split, order=order, rs_push=1, **kn) as p:
        push_us = time_calls(p, d, stream)
    push_ded = {}
    for n in (8, 32):  # the pushes issued by n dedicated push SMs instead of the epilogue
        with runner.make_plan(d, split=split, order=order, rs_push=1, push_sms=n, **kn) as p:
            push_ded[n] = time_calls(p, d, stream, reps=5)
    staged = []
    for s in (1, 2, 4):
        with runner.make_plan(d, split=s, order="row", backend="tma_colocated", tile_m=256, tile_n=256,
                              trace=1) as p:
            us = time_calls(p, d, stream, reps=10)
            wait_ns, busy_ns = p.stats()
        staged.append({"backend": "tma_colocated", "split": s, "us": us,
                       "flag_wait_share": wait_ns / busy_ns if busy_ns else None})
    return {"workload": w.name, "pull_us": pull_us, "push_us": push_us, "push_dedicated_sms_us": push_ded,
            "staged": staged}


def measure_wave_quantization(peaks, stream):
    """The pages' first observation (Syncopate summary, Observation 1, paper
    Fig. 2(a)): a GEMM over one chunk of rows leaves SMs idle when its tiles
    do not fill whole waves, which is why splitting a GEMM into per-chunk
    kernels (the decomposed baseline) loses.  The Llama-3-8B FFN up GEMM
    (K 4096, N 1792) over M rows for M from one 256-row tile row to the full
    8192: this library's kernel with nothing to stage (one rank, CTA pairs,
    256 x 256 tiles over 76 pair walkers) and cuBLAS (torch.matmul), each
    timed alone, as TFLOP/s and fraction of the burst peak."""
    import torch

    from chunk_scheduled_communication_gb300 import runner
    K, N = 4096, 1792
    out = []
    for M in (256, 512, 1024, 2048, 2560, 2816, 3072, 4096, 5120, 5632, 6144, 8192):
        w = wl.Workload(f"wave-M{M}", wl.OP_AG, 1, M, K, N, 1.0, 0.02)
        d = runner.upload(wl.make_inputs(w, r=0, seed=0))
        with runner.make_plan(d, split=1, order="grouped", backend="tma_colocated", tile_m=256, tile_n=256) as p:
            us = time_calls(p, d, stream, reps=20)
        for _ in range(3):
            torch.matmul(d.gathered, d.B, out=d.out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            torch.matmul(d.gathered, d.B, out=d.out)
        e1.record(stream)
        torch.cuda.synchronize()
        cub = e0.elapsed_time(e1) / 20 * 1e3
        tiles = (M // 256) * (N // 256)
        flops = 2.0 * M * N * K
        out.append({"M": M, "pair_tiles": tiles, "waves": tiles / 76, "us": us,
                    "frac_of_burst": flops / (us * 1e-6) / (peaks["bf16_tflops"] * 1e12),
                    "cublas_us": cub, "cublas_frac_of_burst": flops / (cub * 1e-6) / (peaks["bf16_tflops"] * 1e12)})
        del d
    return out


def launches_per_call(plan) -> int:
    i = plan.info()
    return 1 if i["backend"] != 5 else len(set(plan.tables()[1].tolist()))


def cublas_plus_copy_us(w, d, stream) -> float:
    """Context only: the staging copy plus torch.matmul (cuBLAS) on the same
    operands, and for RS/AR the peer sum in PyTorch (not a fused path)."""
    import torch
    reps = 50

    def once():
        if w.op == "ag":
            for q in range(w.R):
                if q != 0:
                    d.gathered[q * w.M_r:(q + 1) * w.M_r].copy_(d.shards[q])
            torch.matmul(d.gathered, d.B, out=d.out)
        elif w.op == "a2a":
            o = 0
            for q in range(w.R):
                m = d.rows_from[q]
                if q != d.r and m:
                    d.gathered[o:o + m].copy_(d.shards[q])
                o += m
            torch.matmul(d.gathered, d.B, out=d.out)
        else:
            P = torch.matmul(d.A, d.B).float()
            rows = slice(0, w.M_r) if w.op == "rs" else slice(0, w.M)
            acc = P[rows]
            for q in range(w.R):
                if d.peers[q] is not None:
                    acc = acc + d.peers[q][rows]
            d.out.copy_(acc)
    for _ in range(3):
        once()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(reps):
        once()
    b1.record(stream)
    torch.cuda.synchronize()
    return b0.elapsed_time(b1) / reps * 1e3


if __name__ == "__main__":
    sys.exit(main())
