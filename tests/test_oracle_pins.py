"""Pins for the CPU oracle, against facts that do not come from the oracle.

Each test ties one oracle entry point to something fixed independently of it:
hand-worked values (tests/golden), the IEEE rounding rule, an exact fp64
brute force under a rigorous error bound, integer inputs where every order is
exact, identity and one-hot matrices, a library matmul, and the invariants of
the operators (row-block independence, concat-K, zero peers, R = 1).

Operators: the Syncopate summary page, Experiments (paper §6.1) — AG-GEMM,
GEMM-RS, GEMM-AR in their standard tensor-parallel meaning; chunking never
changes the result (method, paper §5.1-§5.2; pith review: outputs of the fused
and the original kernel must match).
"""
import json
import os

import numpy as np
import pytest
import torch

from chunk_scheduled_communication_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24      # fp32 unit roundoff
U_BF16 = 2.0 ** -8  # bf16 unit roundoff (8-bit significand)


def gamma(n):
    return n * U / (1 - n * U)


def bits_to_f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def torch_rne(x64):
    """Library rounding of fp64 values to bf16 bits (independent of the oracle)."""
    t = torch.from_numpy(np.asarray(x64, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- bf16 rounding
def test_bf16_rne_golden_cases(oracle_lib):
    rows = []
    with open(os.path.join(GOLD, "bf16_rne_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                a, b = line.split()[:2]
                rows.append((int(a, 16), int(b, 16)))
    f32 = np.array([r[0] for r in rows], dtype=np.uint32).view(np.float32)
    want = np.array([r[1] for r in rows], dtype=np.uint16)
    got = oracle_lib.bf16_rne(f32)
    assert (got == want).all(), list(zip([hex(x) for x in got], [hex(x) for x in want]))


def test_bf16_rne_matches_library_on_random_and_ties(oracle_lib):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # force a quarter of them onto exact ties and exclude NaN payloads
    bits[::4] = (bits[::4] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (oracle_lib.bf16_rne(x) == lib).all()


# --------------------------------------------------------------------------- hand-worked values
def _bits(a):
    return wl.to_bf16_bits(np.array(a, dtype=np.float32))


def test_hand_worked_ag(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["ag_gemm"]
    shards = [_bits(s) for s in g["shards"]]
    gathered, C = oracle_lib.ag_gemm(shards, _bits(g["B"]))
    assert (gathered == _bits(g["gathered"])).all()
    assert (C == np.array(g["C_bits"], dtype=np.uint16)).all()


def test_hand_worked_rs(oracle_lib):
    for g in json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["gemm_rs"]:
        peers = [None if p is None else np.array(p, dtype=np.float32) for p in g["peers"]]
        out, send = oracle_lib.gemm_rs(_bits(g["A"]), _bits(g["B"]), peers, g["R"], g["r"],
                                       send_rows=tuple(g["send_rows"]))
        assert (out == np.array(g["out_bits"], dtype=np.uint16)).all()
        assert (send == np.array(g["send"], dtype=np.float32)).all()


def test_hand_worked_ar_and_peer_order(oracle_lib):
    for g in json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["gemm_ar"]:
        peers = [None if p is None else np.array(p, dtype=np.float32) for p in g["peers"]]
        out, pub = oracle_lib.gemm_ar(_bits(g["A"]), _bits(g["B"]), peers, g["R"], g["r"],
                                      want_publish=True)
        assert (out == np.array(g["out_bits"], dtype=np.uint16)).all(), g["derivation"]
        assert (pub == np.array(g["publish"], dtype=np.float32)).all()


def test_hand_worked_sequential_k(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["sequential_k"]
    A = np.array(g["A_bits"], dtype=np.uint16)
    B = np.array(g["B_bits"], dtype=np.uint16)
    _, C = oracle_lib.ag_gemm([A], B)
    assert (C == np.array(g["C_bits"], dtype=np.uint16)).all()
    P = oracle_lib.gemm_f32(A, B)
    assert P[0, 0] == 0.0  # the fp64 sum would be 1


# --------------------------------------------------------------------------- brute force fp64
def _rand_bits(rng, shape, scale=1.0):
    return wl.to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def _check_bound(got_bits, exact, abs_terms, n_sum):
    """|rne(fl(sum)) - exact| <= gamma_n * S + 2^-8 (|exact| + gamma_n * S)."""
    got = bits_to_f64(got_bits)
    e = gamma(n_sum) * abs_terms
    bound = e + U_BF16 * (np.abs(exact) + e)
    bad = np.abs(got - exact) > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], exact[bad][:5])


@pytest.mark.parametrize("R,M_r,K,N", [(2, 16, 48, 24), (4, 8, 64, 40), (3, 5, 33, 7)])
def test_ag_brute_force_fp64(oracle_lib, R, M_r, K, N):
    rng = np.random.default_rng(R * 1000 + K)
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    B = _rand_bits(rng, (K, N), 0.5)
    gathered, C = oracle_lib.ag_gemm(shards, B)
    G = np.concatenate([bits_to_f64(s) for s in shards])
    Bf = bits_to_f64(B)
    exact = G @ Bf
    S = np.abs(G) @ np.abs(Bf)
    _check_bound(C, exact, S, K)
    # the unrounded fp32 P, checked without the bf16 term
    P = oracle_lib.gemm_f32(gathered, B).astype(np.float64)
    assert (np.abs(P - exact) <= gamma(K) * S).all()


@pytest.mark.parametrize("R,r", [(2, 0), (2, 1), (4, 2), (8, 7)])
def test_rs_brute_force_fp64(oracle_lib, R, r):
    rng = np.random.default_rng(7 + R + r)
    M_r, K, N = 4, 40, 12
    M = R * M_r
    A = _rand_bits(rng, (M, K))
    B = _rand_bits(rng, (K, N), 0.3)
    peers = [None if q == r else rng.standard_normal((M, N), dtype=np.float32) for q in range(R)]
    out, send = oracle_lib.gemm_rs(A, B, peers, R, r, send_rows=(0, M))
    Af, Bf = bits_to_f64(A), bits_to_f64(B)
    P = Af @ Bf
    S = np.abs(Af) @ np.abs(Bf)
    rows = slice(r * M_r, (r + 1) * M_r)
    exact = P[rows] + sum(peers[q][rows].astype(np.float64) for q in range(R) if q != r)
    abs_terms = S[rows] + sum(np.abs(peers[q][rows]).astype(np.float64) for q in range(R) if q != r)
    _check_bound(out, exact, abs_terms, K + R)
    for q in range(R):
        rq = slice(q * M_r, (q + 1) * M_r)
        if q == r:
            assert np.isnan(send[rq]).all()  # rows of rank r are not written
        else:
            assert (np.abs(send[rq].astype(np.float64) - P[rq]) <= gamma(K) * S[rq]).all()


@pytest.mark.parametrize("R,r", [(1, 0), (2, 1), (8, 3)])
def test_ar_brute_force_fp64(oracle_lib, R, r):
    rng = np.random.default_rng(70 + R + r)
    M, K, N = 10, 56, 9
    A = _rand_bits(rng, (M, K))
    B = _rand_bits(rng, (K, N), 0.3)
    peers = [None if q == r else rng.standard_normal((M, N), dtype=np.float32) for q in range(R)]
    out, pub = oracle_lib.gemm_ar(A, B, peers, R, r, want_publish=True)
    Af, Bf = bits_to_f64(A), bits_to_f64(B)
    P = Af @ Bf
    S = np.abs(Af) @ np.abs(Bf)
    exact = P + sum((peers[q].astype(np.float64) for q in range(R) if q != r), np.zeros_like(P))
    abs_terms = S + sum((np.abs(peers[q]).astype(np.float64) for q in range(R) if q != r), np.zeros_like(P))
    _check_bound(out, exact, abs_terms, K + R)
    assert (np.abs(pub.astype(np.float64) - P) <= gamma(K) * S).all()


# --------------------------------------------------------------------------- exact integer cases
@pytest.mark.parametrize("r", [0, 3])
def test_integer_inputs_exact_all_ops(oracle_lib, r):
    rng = np.random.default_rng(11)
    R, M_r, K, N = 4, 6, 96, 20
    M = R * M_r
    ints = lambda shape: rng.integers(-3, 4, size=shape).astype(np.float32)
    shards = [wl.to_bf16_bits(ints((M_r, K))) for _ in range(R)]
    B = wl.to_bf16_bits(ints((K, N)))
    A = wl.to_bf16_bits(ints((M, K)))
    peers = [None if q == r else ints((M, N)) for q in range(R)]
    Bf = bits_to_f64(B)
    # AG
    _, C = oracle_lib.ag_gemm(shards, B)
    exact = np.concatenate([bits_to_f64(s) for s in shards]) @ Bf
    assert (C == torch_rne(exact)).all()
    # RS and AR
    P = bits_to_f64(A) @ Bf
    red = P + sum(peers[q].astype(np.float64) for q in range(R) if q != r)
    out_r, send = oracle_lib.gemm_rs(A, B, peers, R, r, send_rows=(0, M))
    assert (out_r == torch_rne(red[r * M_r:(r + 1) * M_r])).all()
    keep = np.ones(M, bool)
    keep[r * M_r:(r + 1) * M_r] = False
    assert (send[keep] == P[keep]).all()
    out, pub = oracle_lib.gemm_ar(A, B, peers, R, r, want_publish=True)
    assert (out == torch_rne(red)).all()
    assert (pub == P).all()


# --------------------------------------------------------------------------- special matrices
def test_identity_B_returns_gathered(oracle_lib):
    rng = np.random.default_rng(3)
    R, M_r, K = 3, 7, 32
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    eye = wl.to_bf16_bits(np.eye(K, dtype=np.float32))
    gathered, C = oracle_lib.ag_gemm(shards, eye)
    assert (C == gathered).all()
    assert (gathered == np.concatenate(shards)).all()


def test_one_hot_selects_single_element(oracle_lib):
    rng = np.random.default_rng(4)
    R, M_r, K, N = 2, 5, 24, 10
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    for k0, j0 in [(0, 0), (23, 9), (11, 4)]:
        Bf = np.zeros((K, N), np.float32)
        Bf[k0, j0] = 1.0
        gathered, C = oracle_lib.ag_gemm(shards, wl.to_bf16_bits(Bf))
        assert (C[:, j0] == gathered[:, k0]).all()
        other = np.ones(N, bool)
        other[j0] = False
        assert (bits_to_f64(C[:, other]) == 0).all()
    # one-hot rows of A pick rows of B (transpose check)
    A = np.zeros((4, K), np.float32)
    for i, k in enumerate([0, 5, 17, 23]):
        A[i, k] = 1.0
    B = _rand_bits(rng, (K, N))
    _, C = oracle_lib.ag_gemm([wl.to_bf16_bits(A)], B)
    assert (C == B[[0, 5, 17, 23]]).all()


def test_row_block_independence(oracle_lib):
    rng = np.random.default_rng(5)
    R, M_r, K, N = 4, 6, 40, 16
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    B = _rand_bits(rng, (K, N))
    _, C0 = oracle_lib.ag_gemm(shards, B)
    shards2 = list(shards)
    shards2[2] = _rand_bits(rng, (M_r, K))
    _, C1 = oracle_lib.ag_gemm(shards2, B)
    changed = (C0 != C1).any(axis=1)
    assert not changed[:2 * M_r].any() and not changed[3 * M_r:].any()
    assert changed[2 * M_r:3 * M_r].any()


def test_row_ranges_compose(oracle_lib):
    rng = np.random.default_rng(6)
    R, M_r, K, N = 4, 8, 64, 24
    M = R * M_r
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    B = _rand_bits(rng, (K, N))
    _, C = oracle_lib.ag_gemm(shards, B)
    parts = [oracle_lib.ag_gemm(shards, B, a, b, want_gathered=False)[1]
             for a, b in [(0, 5), (5, 19), (19, M)]]
    assert (np.concatenate(parts) == C).all()
    A = np.concatenate(shards)
    peers = [None] + [rng.standard_normal((M, N), dtype=np.float32) for _ in range(R - 1)]
    out, _ = oracle_lib.gemm_ar(A, B, peers, R, 0)
    out2 = np.concatenate([oracle_lib.gemm_ar(A, B, peers, R, 0, a, b)[0] for a, b in [(0, 13), (13, M)]])
    assert (out == out2).all()
    rs, _ = oracle_lib.gemm_rs(A, B, peers, R, 0)
    rs2 = np.concatenate([oracle_lib.gemm_rs(A, B, peers, R, 0, a, b)[0] for a, b in [(0, 3), (3, M_r)]])
    assert (rs == rs2).all()


def test_library_matmul_cross_check(oracle_lib):
    rng = np.random.default_rng(8)
    A = _rand_bits(rng, (64, 512))
    B = _rand_bits(rng, (512, 96), 0.02)
    P = oracle_lib.gemm_f32(A, B).astype(np.float64)
    lib = (torch.from_numpy(wl.bf16_bits_to_f32(A)) @ torch.from_numpy(wl.bf16_bits_to_f32(B))).double().numpy()
    S = np.abs(bits_to_f64(A)) @ np.abs(bits_to_f64(B))
    # both are within gamma_K * S of the exact value
    assert (np.abs(P - lib) <= 2 * gamma(512) * S).all()


# --------------------------------------------------------------------------- operator invariants
def test_concat_k_invariant_rs_ar_exact(oracle_lib):
    """sum_q A_q . B_q == [A_0|...|A_{R-1}] . [B_0;...;B_{R-1}] (integer inputs: exact)."""
    rng = np.random.default_rng(9)
    R, M_r, Kq, N = 4, 3, 32, 8
    M = R * M_r
    ints = lambda shape: wl.to_bf16_bits(rng.integers(-3, 4, size=shape).astype(np.float32))
    As = [ints((M, Kq)) for _ in range(R)]
    Bs = [ints((Kq, N)) for _ in range(R)]
    Acat, Bcat = np.concatenate(As, axis=1), np.concatenate(Bs, axis=0)
    _, full = oracle_lib.ag_gemm([Acat], Bcat)
    for r in range(R):
        peers = [None if q == r else oracle_lib.gemm_f32(As[q], Bs[q]) for q in range(R)]
        out_r, _ = oracle_lib.gemm_rs(As[r], Bs[r], peers, R, r)
        assert (out_r == full[r * M_r:(r + 1) * M_r]).all()
        out, _ = oracle_lib.gemm_ar(As[r], Bs[r], peers, R, r)
        assert (out == full).all()


def test_concat_k_invariant_random_within_bound(oracle_lib):
    rng = np.random.default_rng(10)
    R, M_r, Kq, N = 4, 4, 48, 12
    M = R * M_r
    As = [_rand_bits(rng, (M, Kq)) for _ in range(R)]
    Bs = [_rand_bits(rng, (Kq, N), 0.2) for _ in range(R)]
    Acat = np.concatenate([bits_to_f64(a) for a in As], axis=1)
    Bcat = np.concatenate([bits_to_f64(b) for b in Bs], axis=0)
    exact, S = Acat @ Bcat, np.abs(Acat) @ np.abs(Bcat)
    r = 1
    peers = [None if q == r else oracle_lib.gemm_f32(As[q], Bs[q]) for q in range(R)]
    out, _ = oracle_lib.gemm_ar(As[r], Bs[r], peers, R, r)
    _check_bound(out, exact, S, Kq + R)


def test_zero_peers_reduce_rs_to_plain_gemm_rows(oracle_lib):
    rng = np.random.default_rng(12)
    R, M_r, K, N = 4, 5, 64, 16
    M = R * M_r
    A = _rand_bits(rng, (M, K))
    B = _rand_bits(rng, (K, N))
    _, C = oracle_lib.ag_gemm([A], B)
    for r in range(R):
        peers = [None if q == r else np.zeros((M, N), np.float32) for q in range(R)]
        out_r, _ = oracle_lib.gemm_rs(A, B, peers, R, r)
        assert (out_r == C[r * M_r:(r + 1) * M_r]).all()


def test_single_rank_ar_is_plain_gemm(oracle_lib):
    rng = np.random.default_rng(13)
    A = _rand_bits(rng, (9, 40))
    B = _rand_bits(rng, (40, 11))
    _, C = oracle_lib.ag_gemm([A], B)
    out, _ = oracle_lib.gemm_ar(A, B, [None], 1, 0)
    assert (out == C).all()


# --------------------------------------------------------------------------- A2A-GEMM
# The all-to-all + expert GEMM of the paper's sensitivity study (§6.3, Fig. 11):
# rank r's expert multiplies the rows every source q sends it (rows_from[q],
# possibly 0), stacked in ascending q.
def _parts(rng, rows_from, K, make=None):
    make = make or (lambda shape: _rand_bits(rng, shape))
    return [make((m, K)) for m in rows_from]


def test_hand_worked_a2a(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["a2a_gemm"]
    parts = [_bits(np.array(x, dtype=np.float32).reshape(-1, 2)) for x in g["parts"]]
    gathered, C = oracle_lib.a2a_gemm(parts, _bits(g["B"]))
    assert (gathered == _bits(g["gathered"])).all()
    assert (C == np.array(g["C_bits"], dtype=np.uint16)).all(), g["derivation"]


@pytest.mark.parametrize("rows_from", [[5, 0, 9, 1], [0, 0, 7], [3], [1, 1, 1, 1, 1, 1, 1, 1], [0, 12]])
def test_a2a_brute_force_fp64(oracle_lib, rows_from):
    rng = np.random.default_rng(sum(rows_from) + len(rows_from))
    K, N = 48, 20
    parts = _parts(rng, rows_from, K)
    B = _rand_bits(rng, (K, N), 0.5)
    gathered, C = oracle_lib.a2a_gemm(parts, B)
    G = np.concatenate([bits_to_f64(p) for p in parts])
    assert (bits_to_f64(gathered) == G).all()
    Bf = bits_to_f64(B)
    _check_bound(C, G @ Bf, np.abs(G) @ np.abs(Bf), K)


def test_a2a_integer_inputs_exact(oracle_lib):
    rng = np.random.default_rng(21)
    rows_from, K, N = [4, 0, 11, 2, 0, 6], 96, 18
    ints = lambda shape: wl.to_bf16_bits(rng.integers(-3, 4, size=shape).astype(np.float32))
    parts = _parts(rng, rows_from, K, ints)
    B = ints((K, N))
    _, C = oracle_lib.a2a_gemm(parts, B)
    exact = np.concatenate([bits_to_f64(p) for p in parts]) @ bits_to_f64(B)
    assert (C == torch_rne(exact)).all()


def test_a2a_rows_come_from_their_own_part(oracle_lib):
    """Each part filled with its own constant: row i of C must carry the
    constant of the part that holds row i (catches a wrong offset or an index
    into the wrong part)."""
    rows_from, K, N = [3, 0, 5, 1, 0, 2], 64, 8
    parts = [wl.to_bf16_bits(np.full((m, K), q + 1, np.float32)) for q, m in enumerate(rows_from)]
    B = wl.to_bf16_bits(np.full((K, N), 1.0, np.float32))
    _, C = oracle_lib.a2a_gemm(parts, B)
    want = np.concatenate([np.full(m, (q + 1) * K, np.float64) for q, m in enumerate(rows_from)])
    assert (bits_to_f64(C) == want[:, None]).all()


def test_a2a_equal_parts_is_ag_gemm(oracle_lib):
    rng = np.random.default_rng(22)
    R, M_r, K, N = 4, 6, 64, 24
    shards = [_rand_bits(rng, (M_r, K)) for _ in range(R)]
    B = _rand_bits(rng, (K, N))
    g0, C0 = oracle_lib.ag_gemm(shards, B)
    g1, C1 = oracle_lib.a2a_gemm(shards, B)
    assert (g0 == g1).all() and (C0 == C1).all()


def test_a2a_part_independence_and_row_ranges(oracle_lib):
    rng = np.random.default_rng(23)
    rows_from, K, N = [7, 2, 0, 13], 40, 16
    parts = _parts(rng, rows_from, K)
    B = _rand_bits(rng, (K, N))
    _, C = oracle_lib.a2a_gemm(parts, B)
    off = np.concatenate([[0], np.cumsum(rows_from)])
    for q, m in enumerate(rows_from):
        if m:
            _, Cq = oracle_lib.ag_gemm([parts[q]], B)   # the part alone
            assert (C[off[q]:off[q + 1]] == Cq).all()
    M = int(off[-1])
    pieces = [oracle_lib.a2a_gemm(parts, B, a, b, want_gathered=False)[1] for a, b in [(0, 8), (8, 9), (9, M)]]
    assert (np.concatenate(pieces) == C).all()


# --------------------------------------------------------------------------- ring attention
# Sequence-parallel attention over the keys of all ranks (the pages'
# RingAttention workload, summary Experiments, paper §6.1): the oracle is the
# plain softmax(scale Q K^T [+ causal mask]) V in fp64.
def _attn_inputs(rng, R, S_r, H_q, H_kv, d, scale=1.0):
    b = lambda shape: wl.to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))
    return b((S_r, H_q, d)), [b((S_r, H_kv, d)) for _ in range(R)], [b((S_r, H_kv, d)) for _ in range(R)]


def test_hand_worked_ring_attention(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "hand_worked_ops.json")))["ring_attention"]
    Q, K, V = (_bits(np.array(g[k], dtype=np.float32)) for k in ("Q", "K", "V"))
    for causal, ko, kl in ((False, "O", "lse"), (True, "O_causal", "lse_causal")):
        O, lse = oracle_lib.ring_attention(Q, [K], [V], 0, causal=causal, scale=1.0)
        assert np.abs(O - np.array(g[ko])).max() < 1e-15, (causal, O)
        assert np.abs(lse - np.array(g[kl])).max() < 1e-15, (causal, lse)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R,r,H_q,H_kv", [(3, 1, 4, 2), (2, 0, 2, 2), (4, 3, 4, 1)])
def test_ring_attention_matches_library_sdpa(oracle_lib, causal, R, r, H_q, H_kv):
    """torch's scaled_dot_product_attention in float64 over the concatenated
    keys (GQA heads expanded by hand), with the global-position causal mask."""
    rng = np.random.default_rng(40 + R + r)
    S_r, d = 7, 16
    Q, Ks, Vs = _attn_inputs(rng, R, S_r, H_q, H_kv, d)
    O, lse = oracle_lib.ring_attention(Q, Ks, Vs, r, causal=causal)
    q = torch.from_numpy(bits_to_f64(Q)).permute(1, 0, 2)                       # [H_q, S_r, d]
    k = torch.from_numpy(np.concatenate([bits_to_f64(x) for x in Ks])).permute(1, 0, 2)
    v = torch.from_numpy(np.concatenate([bits_to_f64(x) for x in Vs])).permute(1, 0, 2)
    k = k.repeat_interleave(H_q // H_kv, dim=0)
    v = v.repeat_interleave(H_q // H_kv, dim=0)
    pos_q = r * S_r + torch.arange(S_r)[:, None]
    pos_k = torch.arange(R * S_r)[None, :]
    mask = (pos_k <= pos_q) if causal else torch.ones(S_r, R * S_r, dtype=torch.bool)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask).permute(1, 0, 2).numpy()
    assert np.abs(O - ref).max() < 1e-12
    scores = (q @ k.transpose(1, 2)) / np.sqrt(d)
    ref_lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1).T.numpy()
    assert np.abs(lse - ref_lse).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_zero_queries_average_the_visible_values(oracle_lib, causal):
    rng = np.random.default_rng(50)
    R, r, S_r, H, d = 3, 2, 5, 2, 8
    _, Ks, Vs = _attn_inputs(rng, R, S_r, H, H, d)
    Q = np.zeros((S_r, H, d), np.uint16)
    O, lse = oracle_lib.ring_attention(Q, Ks, Vs, r, causal=causal)
    V = np.concatenate([bits_to_f64(v) for v in Vs])
    for i in range(S_r):
        n = r * S_r + i + 1 if causal else R * S_r
        assert np.allclose(O[i], V[:n].mean(axis=0), rtol=0, atol=1e-13)
        assert np.allclose(lse[i], np.log(n), rtol=0, atol=1e-13)


def test_ring_attention_one_dominant_key_selects_its_value(oracle_lib):
    """Scores 0 everywhere but one key at 64: its weight is 1 - O(e^-64)."""
    rng = np.random.default_rng(51)
    R, r, S_r, H, d = 2, 1, 4, 1, 4
    _, _, Vs = _attn_inputs(rng, R, S_r, H, H, d)
    for jstar in (0, 5, 7):
        Q = np.zeros((S_r, H, d), np.float32)
        Q[:, :, 1] = 8.0
        Ks = [np.zeros((S_r, H, d), np.float32) for _ in range(R)]
        Ks[jstar // S_r][jstar % S_r, 0, 1] = 16.0
        O, _ = oracle_lib.ring_attention(_bits(Q), [_bits(k) for k in Ks], Vs, r, scale=0.5)
        want = bits_to_f64(Vs[jstar // S_r][jstar % S_r, 0])
        bound = (R * S_r - 1) * np.exp(-64.0) * 2 * np.abs(np.stack([bits_to_f64(v) for v in Vs])).max()
        assert np.abs(O[:, 0, :] - want).max() <= bound


def test_ring_attention_lse_merges_per_rank_partials(oracle_lib):
    """RingAttention's combination rule: attention over all keys equals the
    per-rank partial attentions weighted by exp(lse_q - lse), lse = logsumexp_q lse_q."""
    rng = np.random.default_rng(52)
    R, r, S_r, H_q, H_kv, d = 4, 1, 6, 4, 2, 16
    Q, Ks, Vs = _attn_inputs(rng, R, S_r, H_q, H_kv, d)
    O, lse = oracle_lib.ring_attention(Q, Ks, Vs, r)
    parts = [oracle_lib.ring_attention(Q, [Ks[q]], [Vs[q]], 0, scale=1.0 / np.sqrt(d)) for q in range(R)]
    lse_all = np.logaddexp.reduce(np.stack([p[1] for p in parts]), axis=0)
    merged = sum(np.exp(p[1] - lse_all)[..., None] * p[0] for p in parts)
    assert np.abs(lse - lse_all).max() < 1e-12 and np.abs(O - merged).max() < 1e-12


def test_ring_attention_gqa_equals_repeated_heads(oracle_lib):
    rng = np.random.default_rng(53)
    R, r, S_r, H_q, H_kv, d = 2, 0, 5, 6, 2, 8
    Q, Ks, Vs = _attn_inputs(rng, R, S_r, H_q, H_kv, d)
    O, lse = oracle_lib.ring_attention(Q, Ks, Vs, r, causal=True)
    rep = lambda xs: [np.ascontiguousarray(np.repeat(x, H_q // H_kv, axis=1)) for x in xs]
    O2, lse2 = oracle_lib.ring_attention(Q, rep(Ks), rep(Vs), r, causal=True)
    assert (O == O2).all() and (lse == lse2).all()
