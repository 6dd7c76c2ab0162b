"""Run one operator on one named workload with the given knobs.

    python -m chunk_scheduled_communication_gb300.run_case --op rs \
        --backend tma_colocated_smem --tile-m 256 --stages 4 --calls 4

Issues ``--calls`` back-to-back calls of the fused operator on seeded
synthetic inputs (rank 0 of the tensor-parallel group), checks the plan's
error word, and prints the mean call time measured with CUDA events on the
launching stream.  It is the single-kernel case that a kernel profiler
attaches to; the time it prints is not a benchmark figure (no L2 flush, few
calls).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import runner, workloads as wl

ATTN_WORKLOADS = {
    "ring_attn": wl.LLAMA3_8B_RING_ATTN,
    "ring_attn_causal": wl.LLAMA3_8B_RING_ATTN_CAUSAL,
}


def run_attention(a) -> int:
    """The ring-attention forward of rank `--rank` (default: the last rank, the
    one with the most visible keys when causal)."""
    import numpy as np

    from . import attn
    w = ATTN_WORKLOADS[a.op]
    r = w.R - 1 if a.rank < 0 else a.rank
    torch.cuda.set_device(0)
    Q, Ks, Vs = wl.make_attn_inputs(w, 0)
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    kg = torch.zeros((w.R * w.S_r, w.H_kv, w.d), dtype=torch.bfloat16, device="cuda")
    vg = torch.zeros_like(kg)
    ks, vs = [dev(k) for k in Ks], [dev(v) for v in Vs]
    sl = slice(r * w.S_r, (r + 1) * w.S_r)
    kg[sl], vg[sl] = ks[r], vs[r]
    ks[r], vs[r] = kg[sl], vg[sl]
    q = dev(Q)
    O = torch.empty((w.S_r, w.H_q, w.d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    backend = a.backend if a.backend in ("tma_colocated", "unfused") else "tma_colocated"
    with attn.AttnPlan(R=w.R, rank=r, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, causal=w.causal, split=a.split,
                       backend=backend) as p:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(a.calls):
            p.run(q, ks, vs, kg, vg, O, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        p.check(stream)
    print(json.dumps({"workload": w.name, "rank": r, "backend": backend, "split": a.split, "calls": a.calls,
                      "us_per_call": e0.elapsed_time(e1) / a.calls * 1e3}), flush=True)
    return 0

WORKLOADS = {
    "ag": wl.LLAMA3_8B_UP_AG,
    "rs": wl.LLAMA3_8B_DOWN_RS,
    "ar": wl.QWEN2_7B_DOWN_AR,
    "ag70": wl.LLAMA3_70B_UP_AG,
    "a2a": wl.MIXTRAL_8X7B_EXPERT_UP_A2A,
}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--op", choices=sorted(WORKLOADS) + sorted(ATTN_WORKLOADS), default="ag")
    ap.add_argument("--rank", type=int, default=-1, help="ring attention: the local rank (default R-1)")
    ap.add_argument("--backend", default="tma_colocated")
    ap.add_argument("--split", type=int, default=1)
    ap.add_argument("--order", default="row", choices=["row", "col", "grouped", "banded"])
    ap.add_argument("--group-m", type=int, default=8)
    ap.add_argument("--tile-m", type=int, default=0)
    ap.add_argument("--tile-n", type=int, default=256)
    ap.add_argument("--tile-k", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--comm-sms", type=int, default=8)
    ap.add_argument("--direct-fetch", type=int, default=0)
    ap.add_argument("--tuned", action="store_true",
                    help="the benchmark's launch configuration of the operator (other knob flags ignored)")
    ap.add_argument("--calls", type=int, default=4)
    a = ap.parse_args(argv)
    if a.op in ATTN_WORKLOADS:
        return run_attention(a)

    w = WORKLOADS[a.op]
    torch.cuda.set_device(0)
    d = runner.upload(wl.make_inputs(w, r=0), with_f32_out=(w.op == "rs"))  # RS: send rows; AR: no publish
    stream = torch.cuda.current_stream()
    if a.tuned:
        from . import tuned
        split, order, kn = tuned.knobs_for(a.op if a.op != "ag70" else "ag70")
    else:
        split, order = a.split, a.order
        kn = dict(backend=a.backend, tile_m=a.tile_m, tile_n=a.tile_n, tile_k=a.tile_k, stages=a.stages,
                  comm_sms=a.comm_sms, group_m=a.group_m, direct_fetch=a.direct_fetch)
    with runner.make_plan(d, split=split, order=order, **kn) as p:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(a.calls):
            runner.call(p, d, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        p.check(stream)
        info = p.info()
    print(json.dumps({"workload": w.name, "knobs": kn, "split": split, "order": order,
                      "tile_m": info.get("tile_m", a.tile_m), "calls": a.calls,
                      "us_per_call": e0.elapsed_time(e1) / a.calls * 1e3}), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
