"""GPU parity at the plan's limits: the most ranks (8) and the finest chunking
(64 chunks per rank block, two-row chunks), so one tile waits on up to 64
chunk flags and a call publishes 512 (AG-GEMM, GEMM-RS, GEMM-AR, A2A-GEMM).
Integer-valued inputs, every output compared with the CPU oracle bit for bit,
two calls in a row (fresh epochs on every flag)."""
import numpy as np
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import runner, syn
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

AG_MAX = wl.scaled(wl.TINY_AG, M=8 * 128, K=64, N=256, R=8)
RS_MAX = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=8 * 128, K=64, N=256, R=8)
AR_MAX = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=8 * 130, K=72, N=264, R=8)   # with M, K and N tails


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    syn.lib()
    oracle.build()


def _run_check(w, r, split, rows_from=None, **kn):
    inp = wl.make_inputs(w, r=r, seed=3, kind="int", rows_from=rows_from)
    d = runner.upload(inp)
    with runner.make_plan(d, split=split, order="row", **kn) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        assert plan.info()["n_row_chunks"] == w.R * split
    out = runner.dev_to_u16(d.out)
    if w.op in ("ag", "a2a"):
        g, C = (oracle.ag_gemm if w.op == "ag" else oracle.a2a_gemm)(inp.shards, inp.B)
        assert (runner.dev_to_u16(d.gathered) == g).all()
        assert (out == C).all()
        return
    if w.op == "rs":
        ref, f32 = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
        keep = np.ones(w.M, bool)
        keep[r * w.M_r:(r + 1) * w.M_r] = False
    else:
        ref, f32 = oracle.gemm_ar(inp.A, inp.B, inp.peers, w.R, r, want_publish=True)
        keep = np.ones(w.M, bool)
    assert (out == ref).all()
    assert (d.f32_out.cpu().numpy()[keep] == f32[keep]).all()


@pytest.mark.parametrize("backend,tile_m", [("ce", 128), ("tma_colocated", 128), ("tma_colocated", 256),
                                            ("tma_dedicated", 128), ("ldst_colocated", 256)])
def test_ag_64_chunks_per_shard(backend, tile_m):
    _run_check(AG_MAX, 5, 64, backend=backend, tile_m=tile_m, tile_n=256, comm_sms=4)


def test_ag_64_chunks_direct_fetch():
    _run_check(AG_MAX, 2, 64, backend="tma_colocated", tile_m=128, tile_n=256, direct_fetch=1)


@pytest.mark.parametrize("op_w", ["rs", "ar"])
@pytest.mark.parametrize("backend,tile_m", [("ce", 128), ("tma_colocated", 256), ("ldst_dedicated", 128),
                                            ("tma_colocated_smem", 256), ("tma_colocated_smem", 128)])
def test_rs_ar_64_chunks_per_block(op_w, backend, tile_m):
    w = RS_MAX if op_w == "rs" else AR_MAX
    _run_check(w, 6, 64, backend=backend, tile_m=tile_m, tile_n=256, comm_sms=4)


@pytest.mark.parametrize("backend", ["ce", "tma_colocated"])
def test_a2a_64_chunks_per_block(backend):
    rows = (130, 64, 0, 200, 65, 1, 99, 128)  # empty and one-row blocks: empty chunks publish flags too
    w = wl.Workload("a2a-max-split", wl.OP_A2A, 8, sum(rows), 72, 256, 1.0, 1.0, tokens=1, top_k=1)
    _run_check(w, 3, 64, rows_from=rows, backend=backend, tile_m=128, tile_n=256, comm_sms=4)
