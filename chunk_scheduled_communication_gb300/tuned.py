"""Launch configurations of the benchmarked workloads.

The knobs each operator of the benchmark step (and the A2A-GEMM beside it) is
timed with: the measured best points on GB300 (256 x 256 output tiles on CTA
pairs; AG-GEMM and A2A-GEMM staged by the co-located TMA warps, the AG-GEMM
tiles whose chunks have not arrived yet reading the source shard in place;
GEMM-RS and GEMM-AR reading the resident peer partials in place).  The parity tests run the
same configurations, so what the benchmark times is what the tests check.
"""
from __future__ import annotations

STEP_KNOBS = {
    "ag": dict(backend="tma_colocated", split=4, order="grouped", tile_m=256, tile_n=256, comm_sms=8, stages=0,
               direct_fetch=1),
    "rs": dict(backend="tma_colocated_smem", split=1, order="row", tile_m=256, tile_n=256, comm_sms=8, stages=6),
    "ar": dict(backend="tma_colocated_smem", split=1, order="row", tile_m=256, tile_n=256, comm_sms=8, stages=4),
    "a2a": dict(backend="tma_colocated", split=1, order="banded", group_m=8, tile_m=256, tile_n=256, comm_sms=8,
                stages=5),
    # the Llama-3-70B FFN up-projection AG-GEMM: the best point of its sweep
    "ag70": dict(backend="tma_colocated", split=1, order="row", tile_m=256, tile_n=256, comm_sms=8, stages=0),
}


def knobs_for(op: str) -> tuple[int, str, dict]:
    """(split, order, remaining knobs) of operator `op`'s benchmark configuration."""
    kn = dict(STEP_KNOBS[op])
    return kn.pop("split"), kn.pop("order"), kn
