"""GPU parity: the fused chunk-scheduled kernels against the CPU oracle.

Everything is called through the C ABI (libsyn.so) on cuda:0.  The bar:
gathered buffers bit-exact; bf16 outputs within |gpu-ref| <= 1e-2 + 1e-2*|ref|
per element and relative Frobenius error <= 2e-3; fp32 send/publish within the
same per-element bound; integer-valued inputs bit-exact everywhere; and every
backend, split and tile order gives bit-identical GPU outputs (chunking changes
when data moves, never what is computed: Syncopate summary page, method
§5.1-§5.2; pith review, "outputs match").
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import runner, syn, tuned
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV_BACKENDS = ["ce", "tma_dedicated", "tma_colocated", "unfused", "decomposed", "ldst_dedicated",
                "ldst_colocated"]
RSAR_BACKENDS = DEV_BACKENDS + ["tma_colocated_smem"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    syn.lib()
    oracle.build()


@functools.lru_cache(maxsize=8)
def inputs(w, r, seed=0, kind="normal"):
    return wl.make_inputs(w, r=r, seed=seed, kind=kind)


@functools.lru_cache(maxsize=8)
def reference(w, r, seed=0, kind="normal", rows=None):
    """Oracle outputs (all rows, or the sampled row list `rows`)."""
    inp = inputs(w, r, seed, kind)
    if w.op == "ag":
        g, C = oracle.ag_gemm(inp.shards, inp.B)
        return {"gathered": g, "out": C}
    if w.op == "rs":
        out, send = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
        return {"out": out, "f32": send}
    out, pub = oracle.gemm_ar(inp.A, inp.B, inp.peers, w.R, r, want_publish=True)
    return {"out": out, "f32": pub}


def run(w, r, backend="ce", split=1, order="grouped", tile_n=None, comm_sms=8, kind="normal",
        inplace_local=True, with_f32=True, calls=1):
    if tile_n is None:
        tile_n = 256 if w.N % 256 == 0 else 128
    inp = inputs(w, r, 0, kind)
    d = runner.upload(inp, inplace_local=inplace_local, with_f32_out=with_f32)
    with runner.make_plan(d, split=split, order=order, backend=backend, tile_n=tile_n,
                          comm_sms=comm_sms) as plan:
        for _ in range(calls):
            runner.call(plan, d)
        st = plan.sync()
        assert st == syn.OK, syn.lib().syn_last_error()
        fin, fout = plan.flags()
        epoch = plan.info()["epoch"]
    out = {"out": runner.dev_to_u16(d.out), "flags": (fin, fout, epoch)}
    if w.op == "ag":
        out["gathered"] = runner.dev_to_u16(d.gathered)
    elif d.f32_out is not None:
        out["f32"] = d.f32_out.cpu().numpy()
    return out


def check_against_oracle(w, r, got, kind="normal"):
    ref = reference(w, r, 0, kind)
    if w.op == "ag":
        assert (got["gathered"] == ref["gathered"]).all(), "gathered buffer not bit-exact"
    if kind == "int":
        assert (got["out"] == ref["out"]).all(), "integer inputs must match bit for bit"
    else:
        ok, exc, frob = runner.bf16_close(got["out"], ref["out"])
        assert ok, f"out: excess={exc:.3g} frob={frob:.3g}"
    if "f32" in got and w.op != "ag":
        g, rf = got["f32"], ref["f32"]
        if w.op == "rs":
            keep = np.ones(w.M, bool)
            keep[r * w.M_r:(r + 1) * w.M_r] = False
            g, rf = g[keep], rf[keep]
        if kind == "int":
            assert (g == rf).all()
        else:
            ok, exc, frob = runner.f_close(g, rf)
            assert ok, f"f32 out: excess={exc:.3g} frob={frob:.3g}"


# ----------------------------------------------------------------------------- tiny AG, every rank
@pytest.mark.parametrize("backend", DEV_BACKENDS)
@pytest.mark.parametrize("r", [0, 1, 2, 3])
def test_tiny_ag_every_rank_and_backend(r, backend):
    got = run(wl.TINY_AG, r, backend=backend, order="row", comm_sms=2)
    check_against_oracle(wl.TINY_AG, r, got)


def test_tiny_ag_not_inplace_copies_local_slot():
    got = run(wl.TINY_AG, 2, inplace_local=False)
    check_against_oracle(wl.TINY_AG, 2, got)


# ----------------------------------------------------------------------------- exact integer cases
INT_AG = wl.scaled(wl.TINY_AG, M=3 * 200, K=192, N=512, R=3)        # M tail, chunks straddle tiles
INT_RS = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 256, K=320, N=256, R=4)
INT_AR = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=2 * 333, K=128, N=384, R=2)  # M tail


@pytest.mark.parametrize("w", [INT_AG, INT_RS, INT_AR], ids=["ag", "rs", "ar"])
@pytest.mark.parametrize("backend", ["ce", "tma_dedicated", "tma_colocated", "ldst_dedicated", "ldst_colocated"])
def test_integer_inputs_bit_exact(w, backend):
    for r in (0, w.R - 1):
        got = run(w, r, backend=backend, kind="int", comm_sms=3)
        check_against_oracle(w, r, got, kind="int")


INT_AR_N512 = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=2 * 333, K=128, N=512, R=2)


@pytest.mark.parametrize("w,tile_n", [(INT_AR, 128), (INT_AR_N512, 128), (INT_AR_N512, 256)])
def test_integer_ar_colocated_smem_both_tiles(w, tile_n):
    got = run(w, 1, backend="tma_colocated_smem", kind="int", tile_n=tile_n)
    check_against_oracle(w, 1, got, kind="int")


# ----------------------------------------------------------------------------- edge shapes
@pytest.mark.parametrize("shape", [
    dict(R=1, M=128, K=64, N=256),     # one rank, one k-block, one tile
    dict(R=2, M=2 * 40, K=64, N=128),  # M smaller than a tile
    dict(R=5, M=5 * 96, K=640, N=384),  # odd R, ragged tail, N/128 tiles
    dict(R=8, M=8 * 16, K=128, N=256),  # 8 chunks inside one tile
])
def test_ag_edge_shapes(shape):
    w = wl.scaled(wl.TINY_AG, **shape)
    for backend in ("ce", "tma_colocated", "tma_dedicated"):
        got = run(w, shape["R"] - 1, backend=backend, comm_sms=2)
        check_against_oracle(w, shape["R"] - 1, got)


# ----------------------------------------------------------------------------- full-size workloads
def test_llama3_8b_ag_full_all_splits_bit_identical():
    w = wl.LLAMA3_8B_UP_AG
    base = None
    for split in w.splits:
        got = run(w, 0, backend="ce", split=split)
        if base is None:
            check_against_oracle(w, 0, got)
            base = got
        else:
            assert (got["out"] == base["out"]).all() and (got["gathered"] == base["gathered"]).all()
    for backend in ("tma_dedicated", "tma_colocated", "unfused", "decomposed"):
        got = run(w, 0, backend=backend, split=2, order="row")
        assert (got["out"] == base["out"]).all(), backend
        assert (got["gathered"] == base["gathered"]).all(), backend


def test_llama3_8b_rs_full():
    w = wl.LLAMA3_8B_DOWN_RS
    base = run(w, 0, backend="ce", split=1)
    check_against_oracle(w, 0, base)
    fin, fout, epoch = base["flags"]
    # with split 1, row chunk rc is rank rc's block: every send chunk (rc != 0)
    # published this call's epoch, and every staged peer chunk arrived
    assert all(fout[rc] == epoch for rc in range(1, w.R))
    assert all(fin[0 * w.R + q] == epoch for q in range(1, w.R))
    for backend, split in (("tma_dedicated", 2), ("tma_colocated", 4), ("tma_colocated_smem", 1),
                           ("unfused", 2), ("decomposed", 2)):
        got = run(w, 0, backend=backend, split=split)
        assert (got["out"] == base["out"]).all(), backend
        keep = np.ones(w.M, bool)
        keep[:w.M_r] = False
        assert (got["f32"][keep] == base["f32"][keep]).all(), backend


def test_qwen2_7b_ar_full():
    w = wl.QWEN2_7B_DOWN_AR
    base = run(w, 0, backend="tma_colocated_smem", split=1)
    check_against_oracle(w, 0, base)
    for backend, split in (("ce", 2), ("tma_dedicated", 4), ("tma_colocated", 1), ("unfused", 1)):
        got = run(w, 0, backend=backend, split=split)
        assert (got["out"] == base["out"]).all(), backend
        assert (got["f32"] == base["f32"]).all(), backend


def test_llama3_70b_ag_full_sampled_rows():
    """Full-size 70B up-projection: sampled rows against the oracle (row by row),
    and every split 1..8 bit-identical on the GPU."""
    w = wl.LLAMA3_70B_UP_AG
    inp = inputs(w, 0)
    base = run(w, 0, backend="ce", split=1)
    g_ref = np.concatenate(inp.shards)
    assert (base["gathered"] == g_ref).all()
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.M, size=192, replace=False))
    for lo in range(0, len(rows), 64):
        for i in rows[lo:lo + 64]:
            _, ref = oracle.ag_gemm(inp.shards, inp.B, int(i), int(i) + 1, want_gathered=False)
            ok, exc, frob = runner.bf16_close(base["out"][i:i + 1], ref)
            assert ok, (i, exc, frob)
    for split in (2, 3, 4, 5, 6, 7, 8):
        got = run(w, 0, backend="ce", split=split, order="row")
        assert (got["out"] == base["out"]).all(), split
    for backend in ("tma_dedicated", "tma_colocated"):
        got = run(w, 0, backend=backend, split=4, comm_sms=16)
        assert (got["out"] == base["out"]).all(), backend


# ----------------------------------------------------------------------------- protocol
def test_repeated_calls_and_epochs():
    w = wl.TINY_AG
    got = run(w, 1, backend="tma_colocated", calls=5)
    check_against_oracle(w, 1, got)
    fin, fout, epoch = got["flags"]
    assert epoch == 5
    # every non-local transfer published epoch 5
    info, tl, tk, tr = syn.schedule_build("ag", 4, 1, 256, 256, 256)
    for code in tr:
        if code % 4 != 1:
            assert fin[code] == 5


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("backend", ["ce", "tma_dedicated", "tma_colocated"])
def test_dropped_chunk_times_out_then_recovers(backend, tile_m):
    """A staging transfer whose ready flag is never published ends the call in
    SYN_ERR_TIMEOUT (no hang, no trap); the next plan on the same device works.
    With tile_m 256 this also exercises the CTA pair's abort and drain path."""
    w = wl.TINY_AG
    inp = inputs(w, 0)
    d = runner.upload(inp)
    with runner.make_plan(d, backend=backend, comm_sms=2, drop_chunk=2, timeout_ns=20_000_000,
                          tile_m=tile_m) as bad:
        runner.call(bad, d)
        assert bad.sync() == syn.ERR_TIMEOUT
    with runner.make_plan(d, backend=backend, comm_sms=2, tile_m=tile_m) as good:
        runner.call(good, d)
        assert good.sync() == syn.OK
    check_against_oracle(w, 0, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)})


@pytest.mark.parametrize("backend,tile_m,op", [
    ("tma_colocated", 256, "ag"), ("tma_dedicated", 128, "ag"), ("ce", 128, "ag"), ("decomposed", 256, "ag"),
    ("tma_colocated_smem", 256, "rs"), ("tma_colocated_smem", 256, "ar"), ("tma_colocated_smem", 128, "ar")])
def test_corrupt_table_entry_is_caught(backend, tile_m, op):
    """A tile-list entry (and a transfer-list entry) outside its range in the
    device tables is caught by the kernel's bounds checks: SYN_ERR_BOUNDS on
    every call, no out-of-range access, and a clean plan works afterwards."""
    w = {"ag": INT_AG_PAIR, "rs": INT_RS_PAIR, "ar": INT_AR_PAIR}[op]
    inp = inputs(w, 1, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=tile_m, comm_sms=2,
                          corrupt_entry=4, timeout_ns=200_000_000) as bad:
        for _ in range(2):
            runner.call(bad, d)
            assert bad.sync() == syn.ERR_BOUNDS
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=tile_m, comm_sms=2) as good:
        runner.call(good, d)
        assert good.sync() == syn.OK
    got = {"out": runner.dev_to_u16(d.out)}
    if op == "ag":
        got["gathered"] = runner.dev_to_u16(d.gathered)
    else:
        got["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, 1, got, kind="int")


@pytest.mark.parametrize("backend", ["tma_colocated", "tma_dedicated"])
def test_late_flag_from_a_device_stager_only_delays(backend):
    """A chunk flag published 3 ms late (fault injection in the device
    stager) only lengthens the flag waits; the call succeeds and matches."""
    w, r = INT_AG_PAIR, 0
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp)
    waits = []
    for delay in (0, 3000):
        with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=256, comm_sms=2, trace=1,
                              delay_chunk=2, delay_us=delay) as plan:
            runner.call(plan, d)
            assert plan.sync() == syn.OK
            waits.append(plan.stats()[0])
        check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)},
                             kind="int")
    assert waits[1] > waits[0] + 1_000_000  # at least one CTA waited over a millisecond longer


def test_trace_counters():
    w = wl.scaled(wl.LLAMA3_8B_UP_AG, M=8 * 256, K=1024, N=512)
    inp = inputs(w, 0)
    d = runner.upload(inp)
    with runner.make_plan(d, backend="ce", trace=1, split=2) as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK
        wait_ns, busy_ns = plan.stats()
    assert busy_ns > 0 and 0 <= wait_ns <= busy_ns * 2


@pytest.mark.parametrize("tile_m", [128, 256])
def test_per_tile_trace_is_consistent(tile_m):
    """trace=2 stamps every tile: MMA start <= MMA end <= epilogue start <=
    epilogue end, and walker u runs the entries u, u + n, ... in list order."""
    w = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=8 * 512, K=512, N=1024)
    inp = inputs(w, 0)
    d = runner.upload(inp)
    with runner.make_plan(d, backend="tma_colocated_smem", trace=2, split=2, tile_m=tile_m) as plan:
        runner.call(plan, d)
        runner.call(plan, d)
        assert plan.sync() == syn.OK
        tr = plan.trace()
        units = plan.info()["grid_compute"] // (tile_m // 128)
    assert (tr[:, :4] > 0).all()
    assert (tr[:, 0] <= tr[:, 1]).all() and (tr[:, 2] <= tr[:, 3]).all()
    assert (tr[:, 1] <= tr[:, 3]).all()
    walker = tr[:, 4]
    for c in range(units):
        mine = np.nonzero(walker == c)[0]
        assert mine.tolist() == list(range(c, len(tr), units))
        assert (np.diff(tr[mine, 0]) >= 0).all()


@pytest.mark.parametrize("op", ["ag", "rs", "ar"])
def test_autotune_winner_is_fastest_and_passes_parity(op, tmp_path, monkeypatch):
    """The tuner returns the smallest re-timed median it recorded, the winning
    knobs give the oracle's bits on integer inputs of the tuned shape, and a
    second call is a cache hit with the same knobs."""
    import json
    w = {"ag": INT_AG_ALIGNED, "rs": INT_RS_PAIR, "ar": INT_AR_PAIR}[op]
    monkeypatch.setenv("SYN_TUNE_CACHE", str(tmp_path / "tune.jsonl"))
    monkeypatch.setenv("SYN_TUNE_LOG", str(tmp_path / "log.jsonl"))
    best = syn.autotune(op, w.R, 0, w.M, w.N, w.K, budget_s=30.0)
    assert best["backend"] in syn.BACKENDS and best["us"] > 0
    finals = [json.loads(x)["us"] for x in open(tmp_path / "log.jsonl") if '"phase":"final"' in x]
    assert finals
    assert finals and abs(best["us"] - min(finals)) <= 1e-4 * best["us"]
    kn = {k: best[k] for k in ("backend", "comm_sms", "tile_m", "tile_n", "group_m", "stages", "reduce_warps",
                               "direct_fetch")}
    inp = inputs(w, 0, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=best["split"], order=best["order"], **kn) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    got = {"out": runner.dev_to_u16(d.out)}
    if op == "ag":
        got["gathered"] = runner.dev_to_u16(d.gathered)
    else:
        got["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, 0, got, kind="int")
    again = syn.autotune(op, w.R, 0, w.M, w.N, w.K, budget_s=30.0)  # cache hit
    assert {k: again[k] for k in kn} == kn and again["split"] == best["split"] and again["order"] == best["order"]


def test_autotune_push_mode_searches_push_sms(tmp_path, monkeypatch):
    """Push-mode GEMM-RS is tuned as its own problem: the search includes the
    number of dedicated push SMs, returns push mode, and the winner is the
    smallest re-timed mean recorded."""
    import json
    w = INT_RS_PAIR
    monkeypatch.setenv("SYN_TUNE_CACHE", str(tmp_path / "tune.jsonl"))
    monkeypatch.setenv("SYN_TUNE_LOG", str(tmp_path / "log.jsonl"))
    best = syn.autotune("rs", w.R, 0, w.M, w.N, w.K, budget_s=30.0, rs_push=1)
    assert best["rs_push"] == 1 and best["us"] > 0
    rows = [json.loads(x) for x in open(tmp_path / "log.jsonl")]
    assert {0, 4, 8, 16, 32}.issubset({r["push_sms"] for r in rows})  # tried (timed or dropped)
    finals = [r["us"] for r in rows if r["phase"] == "final"]
    assert abs(best["us"] - min(finals)) <= 1e-4 * best["us"]
    pull = syn.autotune("rs", w.R, 0, w.M, w.N, w.K, budget_s=30.0)  # a separate cache entry
    assert pull["rs_push"] == 0 and pull["push_sms"] == 0


# ----------------------------------------------------------------------------- pipeline depths
INT_RS_SMALL = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 128, K=192, N=512, R=4)


@pytest.mark.parametrize("w", [INT_RS_SMALL, INT_AR_N512], ids=["rs", "ar"])
@pytest.mark.parametrize("tile_n,stages", [(256, 2), (256, 3), (256, 4), (128, 3), (128, 4), (128, 6)])
def test_smem_peer_ring_depths_bit_exact(w, tile_n, stages):
    """Every compiled (tile_n, stages) instance of the per-tile shared-memory
    peer path gives the oracle's bits on integer inputs."""
    inp = inputs(w, 1, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend="tma_colocated_smem", tile_n=tile_n,
                          stages=stages, reduce_warps=-1) as plan:
        runner.call(plan, d)
        runner.call(plan, d)
        assert plan.sync() == syn.OK
    got = {"out": runner.dev_to_u16(d.out), "f32": d.f32_out.cpu().numpy()}
    check_against_oracle(w, 1, got, kind="int")


@pytest.mark.parametrize("w,backend,stages", [
    (INT_AG, "tma_colocated", 8), (INT_AG, "ce", 9), (INT_AG, "tma_dedicated", 9),
    (INT_RS_SMALL, "tma_colocated_smem", 4), (INT_RS_SMALL, "tma_colocated_smem", 5),
    (INT_RS_SMALL, "tma_colocated_smem", 6), (INT_RS_SMALL, "tma_colocated", 6), (INT_RS_SMALL, "ce", 6),
    (INT_AR_N512, "tma_colocated_smem", 6), (INT_AR_N512, "tma_colocated", 6), (INT_AR_N512, "ce", 4),
], ids=lambda v: str(getattr(v, "op", v)))
def test_tile_k32_instances_bit_exact(w, backend, stages):
    """k-blocks of 32 (64-byte swizzled A, half-size stages) give the oracle's
    bits on integer inputs, for every compiled tile_k 32 instance."""
    r = w.R - 1
    got = run(w, r, backend=backend, kind="int", comm_sms=3, split=2)
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_n=256, tile_k=32,
                          stages=stages, comm_sms=3) as plan:
        runner.call(plan, d)
        runner.call(plan, d)
        assert plan.sync() == syn.OK
    k32 = {"out": runner.dev_to_u16(d.out)}
    if w.op == "ag":
        k32["gathered"] = runner.dev_to_u16(d.gathered)
    else:
        k32["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, r, k32, kind="int")
    assert (k32["out"] == got["out"]).all()


# ----------------------------------------------------------------------------- CTA pairs (tile_m 256)
INT_AG_PAIR = wl.scaled(wl.TINY_AG, M=3 * 200, K=192, N=512, R=3)       # ragged: last pair half past M
INT_RS_PAIR = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 256, K=320, N=512, R=4)
INT_AR_PAIR = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=2 * 333, K=128, N=512, R=2)


@pytest.mark.parametrize("w,backend,stages", [
    (INT_AG_PAIR, "tma_colocated", 6), (INT_AG_PAIR, "tma_colocated", 5), (INT_AG_PAIR, "tma_colocated", 4),
    (INT_AG_PAIR, "ce", 7),
    (INT_AG_PAIR, "ce", 5), (INT_AG_PAIR, "tma_dedicated", 7), (INT_AG_PAIR, "unfused", 7),
    (INT_AG_PAIR, "decomposed", 7), (INT_AG_PAIR, "ldst_colocated", 7), (INT_AG_PAIR, "ldst_colocated", 5),
    (INT_AG_PAIR, "ldst_dedicated", 7),
    (INT_RS_PAIR, "smem_ring", 3), (INT_RS_PAIR, "smem_ring", 4),
    (INT_RS_PAIR, "smem_ring", 5), (INT_RS_PAIR, "smem_ring", 6),
    (INT_RS_PAIR, "tma_colocated_smem", 4), (INT_RS_PAIR, "tma_colocated_smem", 5),
    (INT_RS_PAIR, "tma_colocated_smem", 6), (INT_RS_PAIR, "tma_colocated_smem", 7),
    (INT_RS_PAIR, "tma_colocated", 4), (INT_RS_PAIR, "ce", 4), (INT_RS_PAIR, "ldst_colocated", 4),
    (INT_RS_PAIR, "ldst_dedicated", 4),
    (INT_AR_PAIR, "smem_ring", 4), (INT_AR_PAIR, "smem_ring", 6),
    (INT_AR_PAIR, "tma_colocated_smem", 4), (INT_AR_PAIR, "tma_colocated_smem", 5),
    (INT_AR_PAIR, "tma_colocated", 4), (INT_AR_PAIR, "ce", 3), (INT_AR_PAIR, "ldst_colocated", 3),
    (INT_AR_PAIR, "ldst_dedicated", 3),
], ids=lambda v: str(getattr(v, "op", v)))
def test_cta_pair_instances_bit_exact(w, backend, stages):
    """256-row tiles shared by a CTA pair (2-CTA UMMA) give the oracle's bits
    on integer inputs, for every compiled pair instance and both ranks' ends
    ("smem_ring": resident peers reduced by the epilogue through the
    shared-memory peer ring instead of the reducer warps)."""
    extra = {}
    if backend == "smem_ring":
        backend, extra = "tma_colocated_smem", {"reduce_warps": -1}
    for r in (0, w.R - 1):
        inp = inputs(w, r, 0, "int")
        d = runner.upload(inp)
        with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=256, tile_n=256,
                              stages=stages, comm_sms=4, **extra) as plan:
            runner.call(plan, d)
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
            assert plan.info()["grid_compute"] % 2 == 0
        got = {"out": runner.dev_to_u16(d.out)}
        if w.op == "ag":
            got["gathered"] = runner.dev_to_u16(d.gathered)
        else:
            got["f32"] = d.f32_out.cpu().numpy()
        check_against_oracle(w, r, got, kind="int")


@pytest.mark.parametrize("w,backend", [(wl.LLAMA3_8B_UP_AG, "tma_colocated"),
                                       (wl.LLAMA3_8B_DOWN_RS, "tma_colocated_smem"),
                                       (wl.QWEN2_7B_DOWN_AR, "tma_colocated_smem")],
                         ids=["ag", "rs", "ar"])
def test_cta_pair_full_size_against_oracle(w, backend):
    got = run(w, 0, backend=backend, split=2, order="row")  # single-CTA reference run
    inp = inputs(w, 0)
    d = runner.upload(inp, with_f32_out=(w.op != "ag"))
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=256) as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK
    pair = {"out": runner.dev_to_u16(d.out)}
    if w.op == "ag":
        pair["gathered"] = runner.dev_to_u16(d.gathered)
    else:
        pair["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, 0, pair)
    ok, exc, frob = runner.bf16_close(pair["out"], got["out"])
    assert ok, (exc, frob)


INT_RS_SPREAD = wl.scaled(wl.LLAMA3_8B_DOWN_RS, M=4 * 512, K=256, N=1024, R=4)   # 32 pair tiles


@pytest.mark.parametrize("spread,stages,reduce_warps", [
    (-1, 6, 0), (4, 5, 0), (3, 7, 0), (0, 6, 0), (0, 4, 0), (-1, 4, -1), (4, 4, -1), (2, 3, -1)])
def test_smem_reduce_spread_bit_exact(spread, stages, reduce_warps):
    """Where the GEMM-RS reduce tiles sit in the walk changes when bytes move,
    not what is computed: integer inputs give the oracle's bits for every
    placement, pipeline depth and reduction path."""
    w, r = INT_RS_SPREAD, 1
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=1, order="row", backend="tma_colocated_smem", tile_m=256,
                          tile_n=256, stages=stages, reduce_spread=spread,
                          reduce_warps=reduce_warps) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        tl, _, _ = plan.tables()
    assert sorted(tl.tolist()) == list(range(len(tl)))
    got = {"out": runner.dev_to_u16(d.out), "f32": d.f32_out.cpu().numpy()}
    check_against_oracle(w, r, got, kind="int")


@pytest.mark.parametrize("w", [wl.LLAMA3_8B_DOWN_RS, wl.QWEN2_7B_DOWN_AR], ids=["rs", "ar"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_reducer_warps_bit_identical_to_epilogue_ring(w, tile_m):
    """Full size, normal inputs: the reducer warps make the same additions in
    the same order as the epilogue's peer ring, so every output bit matches;
    and both stay within tolerance of the oracle."""
    outs = []
    for rw in (0, -1):
        inp = inputs(w, 0)
        d = runner.upload(inp)
        with runner.make_plan(d, split=1, order="row", backend="tma_colocated_smem", tile_m=tile_m,
                              reduce_warps=rw) as plan:
            runner.call(plan, d)
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        outs.append({"out": runner.dev_to_u16(d.out), "f32": d.f32_out.cpu().numpy()})
    assert (outs[0]["out"] == outs[1]["out"]).all()
    keep = np.ones(w.M, bool)
    if w.op == "rs":
        keep[:w.M_r] = False
    assert (outs[0]["f32"][keep] == outs[1]["f32"][keep]).all()
    check_against_oracle(w, 0, outs[0])


def test_reducer_warps_ar_without_publish():
    """GEMM-AR with no publish buffer (the reducer warps' peer sums live in the
    plan's own buffer either way): three calls, oracle bits on integer inputs."""
    w, r = INT_AR_PAIR, 1
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp, with_f32_out=False)
    with runner.make_plan(d, split=1, order="row", backend="tma_colocated_smem", tile_m=256,
                          tile_n=256) as plan:
        for _ in range(3):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out)}, kind="int")


@pytest.mark.parametrize("ce_streams", [1, 3, 16])
def test_copy_engine_streams_bit_exact(ce_streams):
    """Copy-engine staging spread over several side streams: every chunk's
    flag still follows its own copy, so outputs and the gathered buffer stay
    bit-exact (integer inputs) for any stream count."""
    w, r = INT_AG_PAIR, 1
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend="ce", tile_m=256, tile_n=256,
                          ce_streams=ce_streams) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)},
                         kind="int")


@pytest.mark.parametrize("w,stages,kind", [(INT_RS_SPREAD, 5, "int"), (INT_RS_PAIR, 6, "int"),
                                           (wl.LLAMA3_8B_DOWN_RS, 6, "normal")], ids=["spread", "pair", "full"])
def test_rs_push_mode_adds_send_rows(w, stages, kind):
    """GEMM-RS push mode: every send row is added (fp32, TMA reduce-add) into
    `send`, the destination ranks' receive accumulators; rows of the local
    block are untouched and out_r is unchanged.  Checked against the oracle's
    P (its send rows): init + P after one call and (init + P) + P after two,
    bit-exact for integer inputs and within the fp32 tolerance otherwise.  The
    added value is also the same P the pull mode stores (bit-exact)."""
    r = 1
    inp = inputs(w, r, 0, kind)
    rng = np.random.default_rng(7)
    init = rng.integers(-4, 5, size=(w.M, w.N)).astype(np.float32) if kind == "int" else \
        rng.standard_normal((w.M, w.N)).astype(np.float32)
    common = dict(split=1, order="row", backend="tma_colocated_smem", tile_m=256, tile_n=256, stages=stages)
    d = runner.upload(inp)
    with runner.make_plan(d, **common) as pull:  # P rows as the pull mode stores them
        runner.call(pull, d)
        assert pull.sync() == syn.OK
    P = d.f32_out.cpu().numpy()
    d.f32_out.copy_(torch.from_numpy(init))
    with runner.make_plan(d, rs_push=1, **common) as push:
        runner.call(push, d)
        assert push.sync() == syn.OK, syn.lib().syn_last_error()
        once = d.f32_out.cpu().numpy()
        runner.call(push, d)
        assert push.sync() == syn.OK
        twice = d.f32_out.cpu().numpy()
    keep = np.ones(w.M, bool)
    keep[r * w.M_r:(r + 1) * w.M_r] = False
    _, P_ora = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
    want_once = init[keep] + P_ora[keep]
    want_twice = want_once + P_ora[keep]
    if kind == "int":
        assert (once[keep] == want_once).all() and (twice[keep] == want_twice).all()
    else:
        for got_, want_ in ((once[keep], want_once), (twice[keep], want_twice)):
            ok, exc, frob = runner.f_close(got_, want_)
            assert ok, (exc, frob)
    assert (once[keep] == (init[keep] + P[keep])).all()
    assert (twice[keep] == ((init[keep] + P[keep]) + P[keep])).all()
    assert (once[~keep] == init[~keep]).all() and (twice[~keep] == init[~keep]).all()
    check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out)}, kind=kind)


def test_rs_push_mode_rejected_where_unsupported():
    inp = inputs(INT_AR_PAIR, 0, 0, "int")
    d = runner.upload(inp)
    with pytest.raises(syn.SynError) as e:
        runner.make_plan(d, backend="tma_colocated_smem", tile_m=256, rs_push=1)
    assert e.value.status == syn.ERR_UNSUPPORTED
    inp = inputs(INT_RS_PAIR, 0, 0, "int")
    d = runner.upload(inp)
    with pytest.raises(syn.SynError) as e:
        runner.make_plan(d, backend="ce", tile_m=256, rs_push=1)
    assert e.value.status == syn.ERR_UNSUPPORTED


def test_uncompiled_stage_count_is_rejected():
    inp = inputs(INT_AR_N512, 0, 0, "int")
    d = runner.upload(inp)
    with pytest.raises(syn.SynError) as e:
        runner.make_plan(d, backend="tma_colocated_smem", tile_n=256, stages=5)
    assert e.value.status == syn.ERR_UNSUPPORTED


# ----------------------------------------------------------------------------- the benchmark's configuration
@pytest.mark.parametrize("w", [wl.LLAMA3_8B_UP_AG, wl.LLAMA3_8B_DOWN_RS, wl.QWEN2_7B_DOWN_AR],
                         ids=["ag", "rs", "ar"])
def test_benchmark_configuration_full_size_against_oracle(w):
    """Full size, normal inputs, in exactly the launch configuration the
    benchmark times (its knobs, GEMM-RS with `send`, GEMM-AR with publish
    NULL so the plan keeps the partial sums in its own buffer), two calls in a
    row on one plan: every output element against the oracle."""
    split, order, kn = tuned.knobs_for(w.op)
    inp = inputs(w, 0)
    d = runner.upload(inp, with_f32_out=(w.op == "rs"))
    with runner.make_plan(d, split=split, order=order, **kn) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    got = {"out": runner.dev_to_u16(d.out)}
    if w.op == "ag":
        got["gathered"] = runner.dev_to_u16(d.gathered)
    elif w.op == "rs":
        got["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, 0, got)


@pytest.mark.parametrize("w,r", [(w, r) for w in (wl.LLAMA3_8B_UP_AG, wl.LLAMA3_8B_DOWN_RS, wl.QWEN2_7B_DOWN_AR)
                                 for r in range(1, 8)],
                         ids=[f"{o}-r{r}" for o in ("ag", "rs", "ar") for r in range(1, 8)])
def test_benchmark_configuration_other_ranks(w, r):
    """The benchmark's launch configuration at full size for every rank other
    than 0: every output element against the oracle."""
    split, order, kn = tuned.knobs_for(w.op)
    inp = wl.make_inputs(w, r=r, seed=0)
    d = runner.upload(inp, with_f32_out=(w.op == "rs"))
    with runner.make_plan(d, split=split, order=order, **kn) as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    got = {"out": runner.dev_to_u16(d.out)}
    if w.op == "ag":
        got["gathered"] = runner.dev_to_u16(d.gathered)
        g, C = oracle.ag_gemm(inp.shards, inp.B)
        assert (got["gathered"] == g).all()
        ok, exc, frob = runner.bf16_close(got["out"], C)
        assert ok, (exc, frob)
        return
    if w.op == "rs":
        ref, f32 = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
        keep = np.ones(w.M, bool)
        keep[r * w.M_r:(r + 1) * w.M_r] = False
        ok, exc, frob = runner.f_close(d.f32_out.cpu().numpy()[keep], f32[keep])
        assert ok, ("send", exc, frob)
    else:
        ref, _ = oracle.gemm_ar(inp.A, inp.B, inp.peers, w.R, r)
    ok, exc, frob = runner.bf16_close(got["out"], ref)
    assert ok, (exc, frob)


# ----------------------------------------------------------------------------- pre-summed GEMM-AR
# 704 pair tiles over 76 walkers (or 1408 single tiles over 152): walkers run
# 9 or 10 tiles, more than the reducer warps' 8 completion slots, so reducer
# items of a walker's ninth tile wait for the epilogue's acknowledgement of
# its first
INT_AR_LONG_WALK = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=2 * 2816, K=64, N=8192, R=2)


@pytest.mark.parametrize("tile_m,stages,publish", [(256, 5, False), (256, 4, True), (128, 3, False),
                                                   (128, 3, True)])
def test_presum_ar_long_walks_bit_exact(tile_m, stages, publish):
    """GEMM-AR with reducer warps that sum the peer partials ahead of the
    MMAs: walks longer than the completion ring, with and without publish,
    two calls in a row, give the oracle's bits on integer inputs."""
    w, r = INT_AR_LONG_WALK, 1
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp, with_f32_out=publish)
    with runner.make_plan(d, split=1, order="row", backend="tma_colocated_smem", tile_m=tile_m, tile_n=256,
                          stages=stages) as plan:
        for _ in range(2):
            runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    got = {"out": runner.dev_to_u16(d.out)}
    if publish:
        got["f32"] = d.f32_out.cpu().numpy()
    check_against_oracle(w, r, got, kind="int")


@pytest.mark.parametrize("R", [1, 3, 8])
def test_presum_ar_rank_counts_bit_exact(R):
    """Pre-summed GEMM-AR for one rank (no peer: out = rne(P)), an odd rank
    count and eight ranks, with an M tail: oracle bits on integer inputs for
    the first and the last rank."""
    w = wl.scaled(wl.QWEN2_7B_DOWN_AR, M=R * 200, K=192, N=512, R=R)
    for r in sorted({0, R - 1}):
        inp = inputs(w, r, 0, "int")
        d = runner.upload(inp)
        with runner.make_plan(d, split=1, order="row", backend="tma_colocated_smem", tile_m=256,
                              tile_n=256) as plan:
            runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out), "f32": d.f32_out.cpu().numpy()},
                             kind="int")



# ----------------------------------------------------------------------------- direct fetch (AG-GEMM)
INT_AG_ALIGNED = wl.scaled(wl.TINY_AG, M=4 * 256, K=192, N=512, R=4)   # every tile's rows in one shard


@pytest.mark.parametrize("backend,tile_m", [("tma_colocated", 256), ("tma_colocated", 128), ("tma_dedicated", 256),
                                            ("ce", 256), ("ldst_colocated", 256), ("tma_colocated_ragged", 256)])
def test_direct_fetch_bit_exact(backend, tile_m):
    """Tiles whose chunks have not arrived read the source shard in place:
    C and the gathered buffer are the oracle's bits (integer inputs), two
    calls in a row, for both ends of the rank range; on the ragged shape
    (shards of 200 rows) tiles that straddle two shards wait as usual."""
    w = INT_AG_ALIGNED
    if backend == "tma_colocated_ragged":
        backend, w = "tma_colocated", INT_AG_PAIR
    for r in (0, w.R - 1):
        inp = inputs(w, r, 0, "int")
        d = runner.upload(inp)
        with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=tile_m, tile_n=256, comm_sms=2,
                              direct_fetch=1) as plan:
            for _ in range(2):
                runner.call(plan, d)
            assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)},
                             kind="int")


@pytest.mark.parametrize("backend", ["tma_colocated", "ce"])
def test_direct_fetch_reads_an_unpublished_chunk_in_place(backend):
    """A transfer whose ready flag is never published (its bytes are still
    copied) stalls no tile when direct fetch is on: the tiles that need it
    read the source shard, the call succeeds and matches the oracle.  (With
    direct fetch off the same plan ends in SYN_ERR_TIMEOUT, as tested above.)"""
    w, r = INT_AG_ALIGNED, 1
    inp = inputs(w, r, 0, "int")
    d = runner.upload(inp)
    with runner.make_plan(d, split=2, order="row", backend=backend, tile_m=256, drop_chunk=2,
                          timeout_ns=50_000_000, direct_fetch=1) as plan:
        runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
    check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out), "gathered": runner.dev_to_u16(d.gathered)},
                         kind="int")


def test_direct_fetch_rejected_for_rs_ar():
    d = runner.upload(inputs(INT_AR_PAIR, 0, 0, "int"))
    with pytest.raises(syn.SynError) as e:
        runner.make_plan(d, backend="tma_colocated", tile_m=256, direct_fetch=1)
    assert e.value.status == syn.ERR_UNSUPPORTED



@pytest.mark.parametrize("w,push_sms,kind", [(INT_RS_PAIR, 2, "int"), (INT_RS_SPREAD, 6, "int"),
                                             (wl.LLAMA3_8B_DOWN_RS, 16, "normal")], ids=["pair", "spread", "full"])
def test_rs_push_dedicated_sms_adds_send_rows(w, push_sms, kind):
    """GEMM-RS push mode with dedicated push CTAs: the epilogue stores the send
    rows, and the push CTAs add each produced chunk into `send` (TMA
    tile reduce-add) and publish its delivered flag.  Against the oracle's P: init
    + P after one call and (init + P) + P after two (bit-exact for integer
    inputs), local rows untouched, out_r unchanged, every chunk delivered."""
    r = 1
    inp = inputs(w, r, 0, kind)
    rng = np.random.default_rng(11)
    init = rng.integers(-4, 5, size=(w.M, w.N)).astype(np.float32) if kind == "int" else \
        rng.standard_normal((w.M, w.N)).astype(np.float32)
    d = runner.upload(inp)
    d.f32_out.copy_(torch.from_numpy(init))
    with runner.make_plan(d, split=2, order="row", backend="tma_colocated_smem", tile_m=256, tile_n=256,
                          rs_push=1, push_sms=push_sms) as plan:
        assert plan.info()["grid_comm"] == push_sms
        runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        once = d.f32_out.cpu().numpy()
        runner.call(plan, d)
        assert plan.sync() == syn.OK, syn.lib().syn_last_error()
        twice = d.f32_out.cpu().numpy()
        fin, _ = plan.flags()
        info = plan.info()
    keep = np.ones(w.M, bool)
    keep[r * w.M_r:(r + 1) * w.M_r] = False
    _, P = oracle.gemm_rs(inp.A, inp.B, inp.peers, w.R, r, send_rows=(0, w.M))
    want_once = init[keep] + P[keep]
    want_twice = want_once + P[keep]
    if kind == "int":
        assert (once[keep] == want_once).all() and (twice[keep] == want_twice).all()
    else:
        for got_, want_ in ((once[keep], want_once), (twice[keep], want_twice)):
            ok, exc, frob = runner.f_close(got_, want_)
            assert ok, (exc, frob)
    assert (once[~keep] == init[~keep]).all() and (twice[~keep] == init[~keep]).all()
    for rc in range(info["n_row_chunks"]):
        if rc // info["split"] != r:
            assert fin[rc * w.R + r] == info["epoch"]
    check_against_oracle(w, r, {"out": runner.dev_to_u16(d.out)}, kind=kind)


def test_push_sms_needs_push_mode():
    d = runner.upload(inputs(INT_RS_PAIR, 0, 0, "int"))
    with pytest.raises(syn.SynError) as e:
        runner.make_plan(d, backend="tma_colocated_smem", tile_m=256, push_sms=4)
    assert e.value.status == syn.ERR_INVALID
