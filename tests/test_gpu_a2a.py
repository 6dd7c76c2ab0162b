"""GPU parity of A2A-GEMM (the MoE all-to-all + expert GEMM that the Syncopate
paper's sensitivity study, §6.3 / Fig. 11, tunes beside AG-GEMM, GEMM-RS and
GEMM-AR) against the CPU oracle, through the C ABI on cuda:0.

Rank r's expert receives rows_from[q] rows from every source q (blocks of
unequal size, some empty) and multiplies their stack by B.  The bar is the
AG-GEMM one: the stacked input bit-exact; bf16 outputs within
|gpu-ref| <= 1e-2 + 1e-2*|ref| and relative Frobenius error <= 2e-3; integer
inputs bit-exact; every backend, split and tile shape bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import runner, syn
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

BACKENDS = ["ce", "tma_dedicated", "tma_colocated", "unfused", "decomposed", "ldst_dedicated",
            "ldst_colocated"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    syn.lib()
    oracle.build()


def a2a_case(R, rows_from, K, N, kind="normal", scale=1.0 / 16):
    w = wl.Workload(f"a2a-R{R}-K{K}-N{N}", wl.OP_A2A, R, sum(rows_from), K, N, scale, scale,
                    tokens=1, top_k=1)
    return w, tuple(rows_from), kind


def run(w, r, rows_from=None, kind="normal", backend="ce", split=1, order="row", calls=1,
        inplace_local=True, **knobs):
    inp = wl.make_inputs(w, r=r, seed=0, kind=kind, rows_from=rows_from)
    d = runner.upload(inp, inplace_local=inplace_local)
    knobs.setdefault("comm_sms", 2)
    with runner.make_plan(d, split=split, order=order, backend=backend, **knobs) as plan:
        for _ in range(calls):
            runner.call(plan, d)
        st = plan.sync()
        assert st == syn.OK, syn.lib().syn_last_error()
        info = plan.info()
        fin, _ = plan.flags()
    return inp, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered),
                 "info": info, "in_flags": fin}


def check(inp, got, kind="normal"):
    g_ref, c_ref = oracle.a2a_gemm(inp.shards, inp.B)
    assert (got["gathered"] == g_ref).all(), "stacked input not bit-exact"
    if kind == "int":
        assert (got["out"] == c_ref).all(), "integer inputs must match bit for bit"
    else:
        ok, exc, frob = runner.bf16_close(got["out"], c_ref)
        assert ok, f"out: excess={exc:.3g} frob={frob:.3g}"


# ----------------------------------------------------------------------------- skewed tiny routing
@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("r", [0, 1, 2, 3])
def test_tiny_a2a_every_rank_and_backend(r, backend):
    inp, got = run(wl.TINY_A2A, r, backend=backend)
    assert got["info"]["a2a"] == 1 and got["info"]["M"] == sum(inp.rows_from)
    check(inp, got)


# ----------------------------------------------------------------------------- empty and ragged blocks
RAGGED = [100, 0, 37, 300]          # an empty block inside a tile's rows; 437 rows, ragged tail


@pytest.mark.parametrize("backend", ["ce", "tma_dedicated", "tma_colocated"])
@pytest.mark.parametrize("split", [1, 3])
@pytest.mark.parametrize("r", [0, 1, 3])
def test_ragged_blocks_with_an_empty_one(r, split, backend):
    w, rows, _ = a2a_case(4, RAGGED, 256, 256)
    inp, got = run(w, r, rows, backend=backend, split=split)
    check(inp, got)


INT8 = [200, 0, 57, 129, 0, 1, 64, 190]  # 641 rows, two empty blocks, a 1-row block


@pytest.mark.parametrize("backend", ["ce", "tma_dedicated", "tma_colocated"])
@pytest.mark.parametrize("r,split,tile_m", [(0, 1, 128), (1, 3, 128), (4, 2, 128), (7, 1, 256),
                                            (1, 4, 256), (4, 3, 256)])
def test_integer_inputs_bit_exact(r, split, tile_m, backend):
    """Integer inputs: every partial sum is exact, so the oracle's bits come
    back for every backend, split, tile shape and rank (r = 1 and 4 have no
    local rows)."""
    w, rows, kind = a2a_case(8, INT8, 192, 512, kind="int")
    inp, got = run(w, r, rows, kind=kind, backend=backend, split=split, tile_m=tile_m, comm_sms=3)
    check(inp, got, kind)


@pytest.mark.parametrize("rows,r", [([2, 3, 0, 500], 0),    # blocks smaller than split: empty chunks
                                    ([0, 0, 0, 700], 3),    # only the local rank sends
                                    ([0, 0, 0, 700], 0),    # local block empty, one source
                                    ([1, 1, 1, 1], 2)])     # M = 4: one tile, four one-row blocks
@pytest.mark.parametrize("backend", ["ce", "tma_colocated"])
def test_degenerate_routings(rows, r, backend):
    w, rows, _ = a2a_case(4, rows, 128, 256)
    inp, got = run(w, r, rows, backend=backend, split=8 if max(rows) >= 8 else 1)
    check(inp, got)


def test_local_part_not_in_place_is_copied():
    w, rows, _ = a2a_case(4, RAGGED, 256, 256)
    inp, got = run(w, 2, rows, backend="tma_colocated", split=2, inplace_local=False)
    check(inp, got)


def test_repeated_calls_publish_every_flag():
    w, rows, _ = a2a_case(4, RAGGED, 256, 256)
    inp, got = run(w, 3, rows, backend="tma_colocated", split=2, calls=4)
    check(inp, got)
    R, split = 4, 2
    for rc in range(R * split):
        q = rc // split
        if q != 3:  # the local block is in place and never staged
            assert got["in_flags"][rc * R + q] == 4, (rc, q)


# ----------------------------------------------------------------------------- equal parts == AG-GEMM
def test_equal_parts_match_ag_gemm_bit_for_bit():
    w = wl.scaled(wl.TINY_AG, M=4 * 256, K=256, N=512)
    inp = wl.make_inputs(w, r=1)
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, backend="tma_colocated") as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK
    ag = runner.dev_to_u16(d.out)
    wa, rows, _ = a2a_case(4, [256] * 4, 256, 512, scale=w.a_scale)
    ina = wl.make_inputs(wa, r=1, rows_from=rows)
    ina.shards, ina.B = inp.shards, inp.B
    da = runner.upload(ina)
    with runner.make_plan(da, split=2, backend="tma_colocated") as plan:
        runner.call(plan, da)
        assert plan.sync() == syn.OK
    assert (runner.dev_to_u16(da.out) == ag).all()


def test_plans_are_not_interchangeable():
    w, rows, _ = a2a_case(4, RAGGED, 256, 256)
    inp = wl.make_inputs(w, r=0, rows_from=rows)
    d = runner.upload(inp)
    with runner.make_plan(d) as plan:
        with pytest.raises(syn.SynError) as e:
            plan.ag_gemm(d.shards, d.gathered, d.B, d.out)
        assert e.value.status == syn.ERR_INVALID
    wg = wl.TINY_AG
    dg = runner.upload(wl.make_inputs(wg, r=0))
    with runner.make_plan(dg) as plan:
        with pytest.raises(syn.SynError) as e:
            plan.a2a_gemm(dg.shards, dg.gathered, dg.B, dg.out)
        assert e.value.status == syn.ERR_INVALID


# ----------------------------------------------------------------------------- full size
@pytest.mark.parametrize("r", [0, 6])
def test_mixtral_expert_up_full_size_sampled_rows(r):
    """Full-size expert up-projection (rank 0: 7099 rows; rank 6, the most
    popular expert: 12649 rows), in the launch configuration the benchmark
    times (CTA pairs, stagers colocated): the whole stacked input bit-exact,
    sampled rows (block boundaries and the ragged tail included) against the
    oracle, and the single-CTA CE path bit-identical."""
    w = wl.MIXTRAL_8X7B_EXPERT_UP_A2A
    inp, got = run(w, r, backend="tma_colocated", split=1, order="banded", group_m=8, tile_m=256, stages=5)
    g_ref = np.concatenate(inp.shards)
    assert (got["gathered"] == g_ref).all()
    M = g_ref.shape[0]
    off = np.cumsum(inp.rows_from)
    rng = np.random.default_rng(r)
    rows = set(rng.choice(M, size=96, replace=False).tolist())
    rows |= {int(x) for o in off[:-1] for x in (o - 1, o) if 0 <= x < M}
    rows |= {M - 1, 0}
    for i in sorted(rows):
        _, ref = oracle.a2a_gemm(inp.shards, inp.B, i, i + 1, want_gathered=False)
        ok, exc, frob = runner.bf16_close(got["out"][i:i + 1], ref)
        assert ok, (i, exc, frob)
    _, ce = run(w, r, backend="ce", split=1)
    ok, exc, frob = runner.bf16_close(ce["out"], got["out"])
    assert ok, (exc, frob)


# ----------------------------------------------------------------------------- banded tile order
@pytest.mark.parametrize("group_m,tile_m,backend", [(2, 128, "tma_colocated"), (4, 256, "tma_colocated"),
                                                    (3, 128, "ce"), (2, 256, "decomposed")])
def test_banded_order_bit_exact(group_m, tile_m, backend):
    """The banded order (bands of group_m tile rows keyed by their latest
    chunk) moves tiles, never values: integer inputs give the oracle's bits."""
    w, rows, kind = a2a_case(8, INT8, 192, 512, kind="int")
    inp, got = run(w, 3, rows, kind=kind, backend=backend, split=2, order="banded", tile_m=tile_m,
                   group_m=group_m)
    check(inp, got, kind)


def test_banded_order_ag_gemm_bit_exact():
    w = wl.scaled(wl.TINY_AG, M=3 * 200, K=192, N=512, R=3)
    inp = wl.make_inputs(w, r=1, kind="int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="banded", backend="tma_colocated", group_m=2) as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK
    g_ref, c_ref = oracle.ag_gemm(inp.shards, inp.B)
    assert (runner.dev_to_u16(d.gathered) == g_ref).all()
    assert (runner.dev_to_u16(d.out) == c_ref).all()
