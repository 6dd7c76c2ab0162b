"""GPU parity of the fused ring attention (sequence-parallel attention over
the keys of all ranks with chunk-scheduled KV exchange; the pages'
RingAttention workload, Syncopate summary Experiments, paper §6.1) against
the fp64 CPU oracle, through the C ABI on cuda:0.

Tolerance, from the kernel's arithmetic: the probabilities are rounded to
bf16 (relative error <= 2^-9 each) before the P.V product and the output is
rounded once to bf16, so per element |gpu - ref| <= 2^-8 * max|V| + 2^-8 * |ref|
(the rest -- fp32 scores, exp2's ~2^-22 error, fp32 sums -- is far
smaller); relative Frobenius error <= 4e-3.  lse within 1e-3 absolute.
The gathered K and V buffers are bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from chunk_scheduled_communication_gb300 import attn, syn
from chunk_scheduled_communication_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    syn.lib()
    oracle.build()


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def upload(w, r, Q, Ks, Vs, inplace=True):
    kg = torch.zeros((w.R * w.S_r, w.H_kv, w.d), dtype=torch.bfloat16, device="cuda")
    vg = torch.zeros_like(kg)
    ks, vs = [], []
    for q in range(w.R):
        if q == r and inplace:
            kg[q * w.S_r:(q + 1) * w.S_r] = dev(Ks[q])
            vg[q * w.S_r:(q + 1) * w.S_r] = dev(Vs[q])
            ks.append(kg[q * w.S_r:(q + 1) * w.S_r])
            vs.append(vg[q * w.S_r:(q + 1) * w.S_r])
        else:
            ks.append(dev(Ks[q]))
            vs.append(dev(Vs[q]))
    O = torch.empty((w.S_r, w.H_q, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S_r, w.H_q), dtype=torch.float32, device="cuda")
    return dev(Q), ks, vs, kg, vg, O, lse


def run(w, r, backend="tma_colocated", split=1, calls=1, inplace=True, seed=0, **cfg):
    Q, Ks, Vs = wl.make_attn_inputs(w, seed)
    q, ks, vs, kg, vg, O, lse = upload(w, r, Q, Ks, Vs, inplace)
    with attn.AttnPlan(R=w.R, rank=r, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, d=w.d, causal=w.causal, split=split,
                       backend=backend, **cfg) as plan:
        for _ in range(calls):
            plan.run(q, ks, vs, kg, vg, O, lse)
        plan.check()
        flags, info = plan.flags(), plan.info()
    return (Q, Ks, Vs), {"O": to_f64(O), "lse": lse.cpu().numpy().astype(np.float64), "kg": kg, "vg": vg,
                         "flags": flags, "info": info}


def check(w, r, inp, got, rows=None):
    Q, Ks, Vs = inp
    assert (got["kg"].view(torch.int16).cpu().numpy().view(np.uint16) == np.concatenate(Ks)).all()
    assert (got["vg"].view(torch.int16).cpu().numpy().view(np.uint16) == np.concatenate(Vs)).all()
    spans = rows or [(0, w.S_r)]
    vmax = max(np.abs(wl.bf16_bits_to_f32(v)).max() for v in Vs)
    num = den = 0.0
    for a, b in spans:
        ref, ref_lse = oracle.ring_attention(Q, Ks, Vs, r, causal=w.causal, row0=a, row1=b)
        g = got["O"][a:b]
        bound = 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(ref)
        bad = np.abs(g - ref) > bound
        assert not bad.any(), (np.argwhere(bad)[:4], g[bad][:4], ref[bad][:4])
        num += ((g - ref) ** 2).sum()
        den += (ref ** 2).sum()
        assert np.abs(got["lse"][a:b] - ref_lse).max() < 1e-3
    assert np.sqrt(num / den) <= 4e-3, np.sqrt(num / den)


@pytest.mark.parametrize("backend", ["tma_colocated", "unfused"])
@pytest.mark.parametrize("r", [0, 1, 3])
def test_tiny_every_rank(r, backend):
    w = wl.TINY_RING_ATTN
    inp, got = run(w, r, backend=backend)
    check(w, r, inp, got)


@pytest.mark.parametrize("r,split", [(0, 2), (2, 1), (3, 2)])
def test_tiny_causal(r, split):
    w = wl.AttnWorkload("tiny-causal", 4, 256, 4, 2, causal=True)
    inp, got = run(w, r, split=split)
    check(w, r, inp, got)


@pytest.mark.parametrize("H_q,H_kv", [(2, 2), (8, 1), (6, 3)])
def test_head_groupings(H_q, H_kv):
    w = wl.AttnWorkload("heads", 2, 512, H_q, H_kv)
    inp, got = run(w, 1, split=3)
    check(w, 1, inp, got)


def test_single_rank_is_plain_attention():
    w = wl.AttnWorkload("one-rank", 1, 512, 2, 1, causal=True)
    inp, got = run(w, 0)
    check(w, 0, inp, got)


def test_local_shard_not_in_place_is_copied():
    w = wl.TINY_RING_ATTN
    inp, got = run(w, 2, inplace=False, split=2)
    check(w, 2, inp, got)


def test_repeated_calls_publish_every_chunk():
    w = wl.TINY_RING_ATTN
    inp, got = run(w, 1, split=2, calls=3)
    check(w, 1, inp, got)
    for q in range(w.R):
        for j in range(2):
            if q != 1:
                assert got["flags"][q * 2 + j] == 3


def test_dropped_chunk_times_out_then_recovers():
    w = wl.TINY_RING_ATTN
    Q, Ks, Vs = wl.make_attn_inputs(w, 0)
    q, ks, vs, kg, vg, O, lse = upload(w, 0, Q, Ks, Vs)
    with attn.AttnPlan(R=w.R, rank=0, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, split=2, drop_chunk=3,
                       timeout_ns=50_000_000) as plan:
        plan.run(q, ks, vs, kg, vg, O, lse)
        assert plan.sync() == syn.ERR_TIMEOUT
    with attn.AttnPlan(R=w.R, rank=0, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, split=2) as plan:
        plan.run(q, ks, vs, kg, vg, O, lse)
        plan.check()


@pytest.mark.parametrize("kw,status", [
    (dict(S_r=200), syn.ERR_UNSUPPORTED), (dict(S_r=384), syn.ERR_UNSUPPORTED), (dict(d=64), syn.ERR_UNSUPPORTED), (dict(H_q=3, H_kv=2), syn.ERR_INVALID),
    (dict(split=3, S_r=256), syn.ERR_INVALID), (dict(backend="ce"), syn.ERR_UNSUPPORTED),
    (dict(R=2, rank=2), syn.ERR_INVALID)])
def test_invalid_configurations_rejected(kw, status):
    with pytest.raises(syn.SynError) as e:
        attn.AttnPlan(**kw)
    assert e.value.status == status


@pytest.mark.parametrize("w,r", [(wl.LLAMA3_8B_RING_ATTN, 0), (wl.LLAMA3_8B_RING_ATTN_CAUSAL, 7)])
def test_llama3_8b_full_size_sampled_rows(w, r):
    """Full size (32K keys, 32 query heads): the gathered K/V bit-exact and
    sampled query rows (first, middle, tile boundaries, last) against the
    oracle, in the launch configuration the benchmark times."""
    inp, got = run(w, r, split=2)
    rows = [(0, 2), (127, 129), (w.S_r // 2, w.S_r // 2 + 2), (w.S_r - 2, w.S_r)]
    check(w, r, inp, got, rows=rows)


# ----------------------------------------------------------------------------- head-parallel layout
def run_head(w, r, split=1, calls=1, seed=0, **cfg):
    Qs, Ks, Vs = wl.make_head_attn_inputs(w, seed)
    hq, hkv = w.H_q // w.R, w.H_kv // w.R
    qs, ks, vs = [dev(x) for x in Qs], [dev(x) for x in Ks], [dev(x) for x in Vs]
    qg = torch.zeros((w.R * w.S_r, hq, w.d), dtype=torch.bfloat16, device="cuda")
    kg = torch.zeros((w.R * w.S_r, hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vg = torch.zeros_like(kg)
    O = torch.empty((w.R * w.S_r, hq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.R * w.S_r, hq), dtype=torch.float32, device="cuda")
    with attn.AttnPlan(R=w.R, rank=r, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, causal=w.causal, split=split,
                       head_parallel=True, **cfg) as plan:
        for _ in range(calls):
            plan.run_head(qs, ks, vs, qg, kg, vg, O, lse)
        plan.check()
    return (Qs, Ks, Vs), {"O": to_f64(O), "lse": lse.cpu().numpy().astype(np.float64), "qg": qg, "kg": kg, "vg": vg}


def check_head(w, r, inp, got, rows=None):
    """The head-parallel result is plain attention (one rank, global positions)
    over the gathered local heads: the oracle with R = 1 on the gathered rows."""
    Qs, Ks, Vs = inp
    hq, hkv = w.H_q // w.R, w.H_kv // w.R
    Qg = np.ascontiguousarray(np.concatenate([x[:, r * hq:(r + 1) * hq] for x in Qs]))
    Kg = np.ascontiguousarray(np.concatenate([x[:, r * hkv:(r + 1) * hkv] for x in Ks]))
    Vg = np.ascontiguousarray(np.concatenate([x[:, r * hkv:(r + 1) * hkv] for x in Vs]))
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (bits(got["qg"]) == Qg).all() and (bits(got["kg"]) == Kg).all() and (bits(got["vg"]) == Vg).all()
    vmax = np.abs(wl.bf16_bits_to_f32(Vg)).max()
    num = den = 0.0
    for a, b in rows or [(0, w.R * w.S_r)]:
        ref, ref_lse = oracle.ring_attention(Qg, [Kg], [Vg], 0, causal=w.causal, row0=a, row1=b)
        g = got["O"][a:b]
        bad = np.abs(g - ref) > 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(ref)
        assert not bad.any(), (np.argwhere(bad)[:4], g[bad][:4], ref[bad][:4])
        num += ((g - ref) ** 2).sum()
        den += (ref ** 2).sum()
        assert np.abs(got["lse"][a:b] - ref_lse).max() < 1e-3
    assert np.sqrt(num / den) <= 4e-3, np.sqrt(num / den)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("r,split", [(0, 1), (1, 2), (3, 1)])
def test_head_parallel_tiny(r, split, causal):
    w = wl.AttnWorkload("tiny-head", 4, 256, 8, 4, causal=causal)
    inp, got = run_head(w, r, split=split)
    check_head(w, r, inp, got)


def test_head_parallel_unfused_and_repeated_calls():
    w = wl.AttnWorkload("tiny-head-gqa", 2, 512, 8, 2, causal=True)
    inp, got = run_head(w, 1, split=3, backend="unfused")
    check_head(w, 1, inp, got)
    inp, got = run_head(w, 0, split=3, calls=3)
    check_head(w, 0, inp, got)


def test_layouts_are_not_interchangeable():
    w = wl.AttnWorkload("two-ranks", 2, 256, 4, 2)
    Q, Ks, Vs = wl.make_attn_inputs(w, 0)
    q, ks, vs, kg, vg, O, lse = upload(w, 0, Q, Ks, Vs)
    with attn.AttnPlan(R=w.R, rank=0, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv, head_parallel=True) as plan:
        with pytest.raises(syn.SynError) as e:
            plan.run(q, ks, vs, kg, vg, O, lse)
        assert e.value.status == syn.ERR_INVALID
    with attn.AttnPlan(R=w.R, rank=0, S_r=w.S_r, H_q=w.H_q, H_kv=w.H_kv) as plan:
        with pytest.raises(syn.SynError) as e:
            plan.run_head([q, q], ks, vs, q, kg, vg, O, lse)
        assert e.value.status == syn.ERR_INVALID
    with pytest.raises(syn.SynError) as e:  # H_kv = 2 is not divisible by R = 4
        attn.AttnPlan(R=4, rank=0, S_r=256, H_q=4, H_kv=2, head_parallel=True)
    assert e.value.status == syn.ERR_INVALID


def test_head_parallel_llama3_8b_full_size_sampled_rows():
    """Llama-3-8B heads split over 8 ranks (4 query heads, 1 KV head each),
    32K tokens, causal, rank 5: gathered Q/K/V bit-exact, sampled rows."""
    w = wl.AttnWorkload("llama3-8b-head-parallel", 8, 4096, 32, 8, causal=True)
    inp, got = run_head(w, 5, split=2)
    rows = [(0, 2), (4095, 4097), (16384, 16386), (32766, 32768)]
    check_head(w, 5, inp, got, rows=rows)


@pytest.mark.parametrize("causal,r", [(False, 2), (True, 7)])
def test_ring_attention_64_chunks_per_shard(causal, r):
    """The finest KV chunking the plan takes: eight ranks, 64 chunks of one
    128-key block each per shard (512 chunk flags, one wait per block),
    two calls in a row; sampled query rows against the oracle."""
    w = wl.AttnWorkload("ring-attn-max-split", 8, 64 * 128, 2, 1, causal=causal)
    inp, got = run(w, r, split=64, calls=2)
    assert got["info"]["n_transfers"] == (w.R - 1) * 64
    check(w, r, inp, got, rows=[(0, 16), (4096, 4112), (w.S_r - 16, w.S_r)])
