"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2).

The path itself shards as independent replicas (the tensor-parallel ranks are
simulated inside one GPU), so the only cross-rank operations are the barrier
and the max-over-ranks of the timed region.  Both are exercised here with two
CPU processes, including a rank that is slower than the other.
"""
import os
import socket
import time

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), SYN_DIST_BACKEND="gloo")
    import bench
    dist, r, ws, local = bench.dist_setup(world)
    assert (r, ws) == (rank, world)
    t0 = time.perf_counter()
    if rank == 1:
        time.sleep(0.2)  # the slow rank
    bench.barrier(dist)
    waited = time.perf_counter() - t0
    mine = 10.0 + rank  # per-rank timed region in ms
    worst = bench.max_over_ranks(dist, mine)
    q.put((rank, waited, worst))
    dist.destroy_process_group()


def test_gloo_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] >= 0.15  # rank 0 waited for the slow rank at the barrier
    assert res[0][2] == res[1][2] == 11.0  # both see the maximum


def test_weak_scaling_value_counts_all_ranks():
    import bench
    from chunk_scheduled_communication_gb300 import workloads as wl
    step_flops = sum(w.flops for w in bench.STEP)
    assert step_flops == pytest.approx(2 * (8192 * 1792 * 4096 + 8192 * 4096 * 1792 + 4096 * 3584 * 2368))
    # GEMM-AR: A, B, seven fp32 peer partials read; bf16 out (and, when written, fp32 publish)
    assert bench.algorithmic_bytes(wl.QWEN2_7B_DOWN_AR) == pytest.approx(476.8e6, rel=2e-3)
    assert bench.algorithmic_bytes(wl.QWEN2_7B_DOWN_AR, with_publish=True) == pytest.approx(535.5e6, rel=2e-3)
    assert bench.algorithmic_bytes(wl.LLAMA3_8B_UP_AG) == pytest.approx(228.6e6, rel=2e-3)
    assert bench.algorithmic_bytes(wl.LLAMA3_8B_DOWN_RS) == pytest.approx(287.3e6, rel=2e-3)
