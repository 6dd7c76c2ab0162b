"""Run the autotuner on the benchmark step's three operators and record the
winners in the tuner cache the benchmark reads.

    python -m chunk_scheduled_communication_gb300.tune_step [--budget 120] [--out PATH]

Each operator's shape (Llama-3-8B FFN up AG-GEMM, Qwen2-7B FFN down GEMM-AR,
Llama-3-8B FFN down GEMM-RS, rank 0 of 8) is tuned with syn_autotune on its
own scratch operands; the winners are appended to PATH (default: the cache
beside tuned.py) as the tuner's own JSON lines.
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import syn, tuned


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--budget", type=float, default=120.0, help="seconds per operator")
    ap.add_argument("--out", default=tuned.CACHE_PATH)
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    os.environ["SYN_TUNE_CACHE"] = os.path.abspath(a.out)
    for op, w in tuned.STEP_WORKLOADS.items():
        best = syn.autotune(op, w.R, 0, w.M, w.N, w.K, budget_s=a.budget)
        print(json.dumps({"op": op, "workload": w.name, **best}), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
