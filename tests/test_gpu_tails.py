"""GPU parity with K and N tails: K and N multiples of 8 but not of the
64-element k-block or of the tile width.

The TMA operand loads read zeros past K and N, so the last k-block and the
last column of tiles are partial; every store path (TMA tile stores, plain
row stores, the reducer warps' loads and stores, the peer ring, push mode)
must stop at column N.  Integer-valued inputs make every partial sum exact, so
each case is compared with the CPU oracle bit for bit: the gathered buffer,
out, and the fp32 send / publish rows.  Shapes: K = 200 / 328 / 136 / 72
(one to five full k-blocks plus 8, 8, 8, 8 elements), N = 520 / 392 / 600 /
544 (last tile column of 8, 136, 88, 32 columns; N % 32 != 0 and == 0).
"""
import numpy as np
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import runner, syn
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TAIL_AG = wl.scaled(wl.TINY_AG, M=3 * 200, K=200, N=520, R=3)              # M tail as well
TAIL_AG_ALIGNED = wl.scaled(wl.TINY_AG, M=4 * 256, K=200, N=520, R=4)      # tiles inside one shard
TAIL_RS = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 256, K=328, N=392, R=4)
TAIL_AR = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=2 * 333, K=136, N=600, R=2)     # M tail, N % 32 != 0
TAIL_AR32 = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=3 * 200, K=72, N=544, R=3)    # N % 32 == 0

PLAIN = ["ce", "tma_dedicated", "tma_colocated", "ldst_dedicated", "ldst_colocated", "unfused", "decomposed"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    syn.lib()
    oracle.build()


def _run(w, r, calls=2, with_f32=True, **knobs):
    inp = wl.make_inputs(w, r=r, seed=0, kind="int")
    d = runner.upload(inp, with_f32_out=with_f32)
    knobs.setdefault("comm_sms", 3)
    split = knobs.pop("split", 2)
    with runner.make_plan(d, split=split, order=knobs.pop("order", "row"), **knobs) as plan:
        for _ in range(calls):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    got = {"out": runner.dev_to_u16(d.out)}
    if w.op == "ag":
        got["gathered"] = runner.dev_to_u16(d.gathered)
    elif with_f32:
        got["f32"] = d.f32_out.cpu().numpy()
    return inp, got


def _check(w, r, inp, got):
    if w.op == "ag":
        g, C = oracle.ag_gemm(inp.shards, inp.B)
        assert (got["gathered"] == g).all(), "gathered buffer not bit-exact"
        assert (got["out"] == C).all(), "out not bit-exact"
        return
    if w.op == "rs":
        out, f32 = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
        keep = np.ones(w.M, bool)
        keep[r * w.M_r:(r + 1) * w.M_r] = False
    else:
        out, f32 = oracle.gemm_ar(inp.A, inp.B, inp.peers, w.R, r, want_publish=True)
        keep = np.ones(w.M, bool)
    assert (got["out"] == out).all(), "out not bit-exact"
    if "f32" in got:
        assert (got["f32"][keep] == f32[keep]).all(), "fp32 send / publish rows not bit-exact"


def _both_ends(w, **knobs):
    for r in (0, w.R - 1):
        inp, got = _run(w, r, **dict(knobs))
        _check(w, r, inp, got)


# ----------------------------------------------------------------------------- AG-GEMM
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("backend", PLAIN)
def test_ag_tails_every_backend(backend, tile_n):
    _both_ends(TAIL_AG, backend=backend, tile_n=tile_n)


@pytest.mark.parametrize("knobs", [dict(backend="tma_colocated", tile_m=256, tile_n=256),
                                   dict(backend="ce", tile_m=256, tile_n=256),
                                   dict(backend="tma_colocated", tile_n=256, tile_k=32, stages=8)],
                         ids=["pair", "pair-ce", "tile_k32"])
def test_ag_tails_pair_and_tile_k32(knobs):
    _both_ends(TAIL_AG, **knobs)


@pytest.mark.parametrize("tile_m", [128, 256])
def test_ag_tails_direct_fetch(tile_m):
    _both_ends(TAIL_AG_ALIGNED, backend="tma_colocated", tile_m=tile_m, tile_n=256, direct_fetch=1, split=4)


def test_ag_noalloc_tails():
    w, r = TAIL_AG, 1
    inp = wl.make_inputs(w, r=r, seed=0, kind="int")
    d = runner.upload(inp)
    status = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    syn.ag_gemm_noalloc(w.R, r, w.M, w.N, w.K, d.shards, d.gathered, d.B, d.out, split=2, order="row",
                        status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0, status.cpu().numpy()
    _check(w, r, inp, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)})


# ----------------------------------------------------------------------------- GEMM-RS
@pytest.mark.parametrize("backend", PLAIN)
def test_rs_tails_every_backend(backend):
    _both_ends(TAIL_RS, backend=backend, tile_n=256)


@pytest.mark.parametrize("knobs", [
    dict(tile_m=128, tile_n=256),                        # reducer warps
    dict(tile_m=128, tile_n=128),                        # epilogue peer ring (tile_n 128)
    dict(tile_m=128, tile_n=256, reduce_warps=-1),       # epilogue peer ring
    dict(tile_m=256, tile_n=256, stages=6),              # pair + reducer warps
    dict(tile_m=256, tile_n=256, stages=5, reduce_warps=-1),
], ids=["reducers", "ring-n128", "ring", "pair-reducers", "pair-ring"])
def test_rs_tails_resident_peers(knobs):
    _both_ends(TAIL_RS, backend="tma_colocated_smem", **knobs)


@pytest.mark.parametrize("push_sms", [0, 4])
def test_rs_tails_push_mode(push_sms):
    """Push mode over an N tail: init + P after one call, (init + P) + P after
    two, on the send rows; local rows untouched; out_r the oracle's bits."""
    w, r = TAIL_RS, 2
    inp = wl.make_inputs(w, r=r, seed=0, kind="int")
    init = np.random.default_rng(5).integers(-4, 5, size=(w.M, w.N)).astype(np.float32)
    d = runner.upload(inp)
    d.f32_out.copy_(torch.from_numpy(init))
    snaps = []
    with runner.make_plan(d, split=2, order="row", backend="tma_colocated_smem", tile_m=256, tile_n=256,
                          rs_push=1, push_sms=push_sms) as plan:
        for _ in range(2):
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
            snaps.append(d.f32_out.cpu().numpy())
    out, P = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
    keep = np.ones(w.M, bool)
    keep[r * w.M_r:(r + 1) * w.M_r] = False
    assert (snaps[0][keep] == init[keep] + P[keep]).all()
    assert (snaps[1][keep] == init[keep] + P[keep] + P[keep]).all()
    assert (snaps[1][~keep] == init[~keep]).all()
    assert (runner.dev_to_u16(d.out) == out).all()


# ----------------------------------------------------------------------------- GEMM-AR
@pytest.mark.parametrize("w", [TAIL_AR, TAIL_AR32], ids=["n600", "n544"])
@pytest.mark.parametrize("backend", PLAIN)
def test_ar_tails_every_backend(w, backend):
    _both_ends(w, backend=backend, tile_n=256)


@pytest.mark.parametrize("w", [TAIL_AR, TAIL_AR32], ids=["n600", "n544"])
@pytest.mark.parametrize("knobs", [
    dict(tile_m=128, tile_n=256, stages=3),                    # pre-summed peers (reducer warps)
    dict(tile_m=256, tile_n=256, stages=4),                    # pre-summed, CTA pair
    dict(tile_m=256, tile_n=256, stages=4, with_f32=False),    # pre-summed, no publish
    dict(tile_m=128, tile_n=128),                              # epilogue peer ring (tile_n 128)
    dict(tile_m=256, tile_n=256, stages=4, reduce_warps=-1),   # epilogue peer ring, pair
], ids=["presum", "presum-pair", "presum-nopub", "ring-n128", "ring-pair"])
def test_ar_tails_resident_peers(w, knobs):
    _both_ends(w, backend="tma_colocated_smem", **knobs)


# ----------------------------------------------------------------------------- A2A-GEMM
@pytest.mark.parametrize("backend", ["ce", "tma_colocated"])
def test_a2a_tails(backend):
    rows = (100, 0, 37, 300)
    w = wl.Workload("a2a-tails", wl.OP_A2A, 4, sum(rows), 200, 392, 1.0 / 16, 1.0 / 16, tokens=1, top_k=1)
    for r in (0, 3):
        inp = wl.make_inputs(w, r=r, seed=0, kind="int", rows_from=rows)
        d = runner.upload(inp)
        with runner.make_plan(d, split=3, order="row", backend=backend, comm_sms=2, tile_n=256) as plan:
            runner.call(plan, d)
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        g, C = oracle.a2a_gemm(inp.shards, inp.B)
        assert (runner.dev_to_u16(d.gathered) == g).all()
        assert (runner.dev_to_u16(d.out) == C).all()


# ----------------------------------------------------------------------------- GEMM-RS row-block tails
# Rank blocks of M/R rows that are not whole tiles: a tile may hold rows of two
# or more blocks, some sent and some reduced (each 32-row warp group lies in
# one block).  96-row blocks under 128-row tiles, 160-row blocks under 256-row
# CTA-pair tiles (ragged last tile), with K and N tails as well.
RS_STRADDLE = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 96, K=200, N=392, R=4)
RS_STRADDLE_PAIR = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=5 * 160, K=136, N=520, R=5)


def _every_rank(w, ranks=None, **knobs):
    for r in (ranks if ranks is not None else range(w.R)):
        inp, got = _run(w, r, **dict(knobs))
        _check(w, r, inp, got)


@pytest.mark.parametrize("backend", PLAIN)
def test_rs_straddling_tiles_every_backend(backend):
    _every_rank(RS_STRADDLE, backend=backend, tile_n=256)


@pytest.mark.parametrize("knobs", [
    dict(tile_m=128, tile_n=256),                   # reducer warps
    dict(tile_m=128, tile_n=256, reduce_warps=-1),  # epilogue peer ring
    dict(tile_m=128, tile_n=128),
], ids=["reducers", "ring", "ring-n128"])
def test_rs_straddling_tiles_resident_peers(knobs):
    _every_rank(RS_STRADDLE, backend="tma_colocated_smem", **knobs)


@pytest.mark.parametrize("knobs", [
    dict(backend="tma_colocated_smem", stages=6),                    # pair + reducer warps
    dict(backend="tma_colocated_smem", stages=5, reduce_warps=-1),   # pair + epilogue peer ring
    dict(backend="tma_colocated", stages=4),
    dict(backend="ce", stages=4),
], ids=["reducers", "ring", "tma_colocated", "ce"])
def test_rs_straddling_pair_tiles(knobs):
    _every_rank(RS_STRADDLE_PAIR, ranks=(0, 2, 4), tile_m=256, tile_n=256, **knobs)


@pytest.mark.parametrize("push_sms", [0, 4])
def test_rs_straddling_push_mode(push_sms):
    """Push mode where tiles straddle block edges: only the sent rows are added
    into `send`; the local block's rows of `send` stay untouched."""
    w = RS_STRADDLE_PAIR
    for r in (1, 4):
        inp = wl.make_inputs(w, r=r, seed=0, kind="int")
        init = np.random.default_rng(6).integers(-4, 5, size=(w.M, w.N)).astype(np.float32)
        d = runner.upload(inp)
        d.f32_out.copy_(torch.from_numpy(init))
        with runner.make_plan(d, split=5, order="row", backend="tma_colocated_smem", tile_m=256, tile_n=256,
                              rs_push=1, push_sms=push_sms) as plan:
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
            once = d.f32_out.cpu().numpy()
        out, P = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
        keep = np.ones(w.M, bool)
        keep[r * w.M_r:(r + 1) * w.M_r] = False
        assert (once[keep] == init[keep] + P[keep]).all()
        assert (once[~keep] == init[~keep]).all()
        assert (runner.dev_to_u16(d.out) == out).all()


@pytest.mark.parametrize("tile_m,backend", [(128, "tma_colocated"), (256, "tma_colocated"), (128, "ce")])
def test_rs_straddling_dropped_chunk_times_out_then_recovers(tile_m, backend):
    """A straddling GEMM-RS tile waits for the local chunks its rows touch: a
    staging transfer of the local block whose flag is never published ends
    the call in SYN_ERR_TIMEOUT (bounded waits, no hang), and the next plan
    gives the oracle's bits."""
    w = RS_STRADDLE if tile_m == 128 else RS_STRADDLE_PAIR
    r = 1
    inp = wl.make_inputs(w, r=r, seed=0, kind="int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=tile_m, tile_n=256, comm_sms=2,
                          drop_chunk=0, timeout_ns=20_000_000) as bad:
        runner.call(bad, d)
        assert bad.sync() == syn.ERR_TIMEOUT
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=tile_m, tile_n=256,
                          comm_sms=2) as good:
        runner.call(good, d)
        assert good.sync() == syn.OK, syn.lib().syn_last_error()
    _check(w, r, inp, {"out": runner.dev_to_u16(d.out), "f32": d.f32_out.cpu().numpy()})
