"""syn_ag_gemm_noalloc: AG-GEMM for callers that cannot allocate device memory.

Plug-in hosts that hand an operator only its tensors, and serving loops that
forbid cudaMalloc/cudaFree after start-up, cannot use syn_plan_create (it
allocates the plan's flags and tables).  This entry point keeps that scratch in
one static device array instead.  The test calls it through the C ABI twice in
a row, on two different shapes, and checks each result against the CPU oracle
(gathered buffer bit-exact, C within the parity tolerance) and against the
plan-based syn_ag_gemm on the same inputs (within the same tolerance).  The
array keeps the previous call's contents, so the second call also checks that
the entry point clears what must start at zero.  It lives in its own file so
that it is collected last.
"""
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import runner, syn
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _plan_result(w, inp):
    d = runner.upload(inp)
    with runner.make_plan(d, split=2 if w.M_r % 2 == 0 else 1, order="row") as plan:
        runner.call(plan, d)
        plan.check()
    return runner.dev_to_u16(d.gathered), runner.dev_to_u16(d.out)


def _noalloc_result(w, inp, split):
    d = runner.upload(inp)
    status = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    syn.ag_gemm_noalloc(w.R, inp.r, w.M, w.N, w.K, d.shards, d.gathered, d.B, d.out, split=split,
                        order="row", status=status)
    torch.cuda.synchronize()
    return runner.dev_to_u16(d.gathered), runner.dev_to_u16(d.out), status.cpu().numpy()


def test_noalloc_matches_oracle_and_plan_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    oracle.build()
    cases = [(wl.scaled(wl.LLAMA3_8B_UP_AG, M=8 * 256, K=1024, N=768), 3, 2),
             (wl.TINY_AG, 1, 1)]
    for w, r, split in cases:
        inp = wl.make_inputs(w, r=r, seed=0)
        g_ora, c_ora = oracle.ag_gemm(inp.shards, inp.B)
        g_ref, c_ref = _plan_result(w, inp)
        g, c, status = _noalloc_result(w, inp, split)
        assert status[0] == 0, status
        assert (g == g_ora).all(), "gathered buffer differs from the oracle's"
        ok, exc, frob = runner.bf16_close(c, c_ora)
        assert ok, (w.name, "oracle", exc, frob)
        assert (g == g_ref).all(), "gathered buffer differs from the plan entry point's"
        ok, exc, frob = runner.bf16_close(c, c_ref)
        assert ok, (w.name, "plan entry point", exc, frob)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L = syn.lib()
    lay = syn.Layout(8 * 8192, 8192, 128, 0, 0, 0)  # 512 x 32 = 16384 tiles > 4096
    arr = (syn._P * 8)(*([16] * 8))
    st = L.syn_ag_gemm_noalloc(8, 0, lay, 1, 0, arr, 16, 16, 16, None, None)
    assert st == syn.ERR_UNSUPPORTED
    assert b"SYN_NOALLOC_MAX_TILES" in L.syn_last_error()
