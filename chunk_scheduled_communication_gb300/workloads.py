"""Seeded synthetic workloads (shapes and input generators only).

This module holds no arithmetic of the operators: it draws random inputs and
quantises them to bf16 with PyTorch's own conversion.  The same bytes are
handed to the CUDA path and to the CPU oracle.

Shapes follow the workloads the Syncopate summary page evaluates ("Experiments",
paper §6.1: AG-GEMM, GEMM-RS and GEMM-AR on Llama-3 and Qwen FFN shapes), at
tensor-parallel degree 8 with the other ranks simulated in one GPU's memory.
No dataset or trained weights are involved: activations are N(0,1), weights
N(0, 0.02) (0.02 is a standard deviation), peer partials N(0,1) fp32.

Recipe (fixed order, numpy PCG64 ``default_rng(seed)``):
  AG : shards q = 0..R-1 (each [M_r, K]), then B [K, N]
  RS : A [M, K], then B [K, N], then the peers q != r in ascending q ([M, N] fp32)
  AR : same as RS
  A2A: parts q = 0..R-1 (each [rows_from[q], K]), then B [K, N]; the routing
       counts come from a generator of their own, ``default_rng(seed)`` in
       ``Workload.rows_from`` (the same matrix of counts for every rank)
A2A-GEMM (the MoE all-to-all + expert GEMM that the paper's sensitivity study,
§6.3 / Fig. 11, tunes) has no shapes on the pages; the workload here is an
expert-parallel mixture-of-experts FFN: R ranks, one expert each, every rank
holding ``tokens`` tokens routed to ``top_k`` experts.  Routing counts: expert
popularity p = softmax(skew * z), z ~ N(0, I_R); each source rank q sends
expert r the count r of Multinomial(tokens * top_k, p), drawn for q = 0..R-1
in order.  So blocks differ in size, the expert's row count M = sum_q rows_from[q]
varies with r and the seed, and small configurations can have empty blocks.
Every normal draw is ``standard_normal(float32) * scale``; bf16 operands are
then rounded to nearest-even by ``torch.Tensor.to(torch.bfloat16)``.
``kind="int"`` draws integers in [-3, 3] instead (exactly representable, and
small enough that every partial sum is exact in fp32 for K <= 512 * 8).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

OP_AG, OP_RS, OP_AR, OP_A2A = "ag", "rs", "ar", "a2a"


@dataclass(frozen=True)
class Workload:
    name: str
    op: str              # "ag" | "rs" | "ar"
    R: int               # simulated tensor-parallel ranks
    M: int               # gathered / output rows (all ranks)
    K: int
    N: int
    a_scale: float       # std of activations (A / shards)
    b_scale: float       # std of the weight B
    peer_scale: float = 1.0
    splits: tuple = (1,)  # chunks per shard (AG) or per rank row block (RS/AR)
    note: str = ""
    tokens: int = 0      # A2A: tokens per source rank
    top_k: int = 0       # A2A: experts per token
    skew: float = 0.0    # A2A: spread of the expert popularity logits

    @property
    def M_r(self) -> int:
        return self.M // self.R

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def rows_from(self, r: int, seed: int = 0) -> list:
        """A2A: the rows each source rank sends rank r's expert (recipe above)."""
        assert self.op == OP_A2A
        rng = np.random.default_rng(seed)
        z = rng.standard_normal(self.R)
        p = np.exp(self.skew * (z - z.max()))
        p /= p.sum()
        return [int(rng.multinomial(self.tokens * self.top_k, p)[r]) for _ in range(self.R)]

    def a2a_flops(self, r: int, seed: int = 0) -> float:
        return 2.0 * sum(self.rows_from(r, seed)) * self.N * self.K


# The five workloads.  Names say what they are; sizes are the full ones.
TINY_AG = Workload("tiny-ag-R4-M256-K256-N256", OP_AG, 4, 256, 256, 256, 1.0 / 16, 1.0 / 16,
                   splits=(1,), note="4 shards of 64 rows; each 128-row tile straddles 2 shards")
LLAMA3_8B_UP_AG = Workload("llama3-8b-ffn-up-ag-tp8-M8192-K4096-N1792", OP_AG, 8, 8192, 4096, 1792,
                           1.0, 0.02, splits=(1, 2, 4))
LLAMA3_8B_DOWN_RS = Workload("llama3-8b-ffn-down-rs-tp8-M8192-K1792-N4096", OP_RS, 8, 8192, 1792, 4096,
                             1.0, 0.02, 1.0, splits=(1, 2, 4))
QWEN2_7B_DOWN_AR = Workload("qwen2-7b-ffn-down-ar-tp8-M4096-K2368-N3584", OP_AR, 8, 4096, 2368, 3584,
                            1.0, 0.02, 1.0, splits=(1, 2, 4))
LLAMA3_70B_UP_AG = Workload("llama3-70b-ffn-up-ag-tp8-M16384-K8192-N3584", OP_AG, 8, 16384, 8192, 3584,
                            1.0, 0.02, splits=(1, 2, 3, 4, 5, 6, 7, 8))

# Expert-parallel MoE FFN up-projection in the shape of Mixtral-8x7B (hidden
# 4096, expert FFN 14336, 8 experts, top-2): 8 ranks, one expert each, 4096
# tokens per rank.  M is the nominal rows per expert (tokens * top_k); the
# drawn counts vary around it.
MIXTRAL_8X7B_EXPERT_UP_A2A = Workload("mixtral-8x7b-expert-up-a2a-ep8-T4096-top2-K4096-N14336", OP_A2A, 8,
                                      4096 * 2, 4096, 14336, 1.0, 0.02, splits=(1, 2, 4),
                                      tokens=4096, top_k=2, skew=0.5)
TINY_A2A = Workload("tiny-a2a-R4-T96-top2-K256-N256", OP_A2A, 4, 96 * 2, 256, 256, 1.0 / 16, 1.0 / 16,
                    tokens=96, top_k=2, skew=1.5, note="skewed routing: blocks of very different sizes")

ALL = (TINY_AG, LLAMA3_8B_UP_AG, LLAMA3_8B_DOWN_RS, QWEN2_7B_DOWN_AR, LLAMA3_70B_UP_AG)


def scaled(w: Workload, M: int | None = None, K: int | None = None, N: int | None = None,
           R: int | None = None, tokens: int | None = None) -> Workload:
    """Same workload family at another size (for small parity cases)."""
    return Workload(f"{w.name}-scaled", w.op, R or w.R, M or w.M, K or w.K, N or w.N,
                    w.a_scale, w.b_scale, w.peer_scale, w.splits, w.note, tokens or w.tokens, w.top_k, w.skew)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16) via PyTorch's round-to-nearest-even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _draw(rng: np.random.Generator, shape, scale: float, kind: str) -> np.ndarray:
    if kind == "int":
        return rng.integers(-3, 4, size=shape).astype(np.float32)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


@dataclass
class Inputs:
    w: Workload
    r: int
    shards: list = field(default_factory=list)   # AG: R x uint16 [M_r, K]; A2A: parts [rows_from[q], K]
    rows_from: list | None = None                # A2A: rows each source sends
    A: np.ndarray | None = None                  # RS/AR: uint16 [M, K]
    B: np.ndarray | None = None                  # uint16 [K, N]
    peers: list = field(default_factory=list)    # RS/AR: R entries, fp32 [M, N], None at r


def make_inputs(w: Workload, r: int = 0, seed: int = 0, kind: str = "normal",
                rows_from: tuple | None = None) -> Inputs:
    """Draw the inputs of workload ``w`` for local rank ``r`` (A2A: ``rows_from``
    overrides the drawn routing counts)."""
    rng = np.random.default_rng(seed)
    out = Inputs(w=w, r=r)
    if w.op == OP_AG:
        out.shards = [to_bf16_bits(_draw(rng, (w.M_r, w.K), w.a_scale, kind)) for _ in range(w.R)]
        out.B = to_bf16_bits(_draw(rng, (w.K, w.N), w.b_scale, kind))
    elif w.op == OP_A2A:
        out.rows_from = list(rows_from) if rows_from is not None else w.rows_from(r, seed)
        out.shards = [to_bf16_bits(_draw(rng, (m, w.K), w.a_scale, kind)) for m in out.rows_from]
        out.B = to_bf16_bits(_draw(rng, (w.K, w.N), w.b_scale, kind))
    else:
        out.A = to_bf16_bits(_draw(rng, (w.M, w.K), w.a_scale, kind))
        out.B = to_bf16_bits(_draw(rng, (w.K, w.N), w.b_scale, kind))
        out.peers = [None if q == r else _draw(rng, (w.M, w.N), w.peer_scale, kind)
                     for q in range(w.R)]
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (via PyTorch)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float32).numpy()


# --------------------------------------------------------------------------- ring attention
@dataclass(frozen=True)
class AttnWorkload:
    """Sequence-parallel attention: R ranks of S_r tokens each, H_q query
    heads over H_kv KV heads, head dimension d."""
    name: str
    R: int
    S_r: int
    H_q: int
    H_kv: int
    d: int = 128
    causal: bool = False

    @property
    def flops(self) -> float:
        """Tensor-core FLOPs of one rank's forward (Q.K^T and P.V)."""
        keys = self.R * self.S_r
        full = 4.0 * self.S_r * keys * self.d * self.H_q
        if not self.causal:
            return full
        # keys up to each query's position: sum over the rank-r rows (taken at the last rank)
        r = self.R - 1
        visible = sum(r * self.S_r + i + 1 for i in range(self.S_r))
        return 4.0 * visible * self.d * self.H_q


# Llama-3-8B attention (32 query heads, 8 KV heads, d 128) over a 32K-token
# context split across 8 ranks (4096 tokens each): the long-context ring
# attention shape of the pages' attention workloads.
LLAMA3_8B_RING_ATTN = AttnWorkload("llama3-8b-ring-attn-sp8-S32768-Hq32-Hkv8-d128", 8, 4096, 32, 8)
LLAMA3_8B_RING_ATTN_CAUSAL = AttnWorkload("llama3-8b-ring-attn-causal-sp8-S32768-Hq32-Hkv8-d128", 8, 4096, 32, 8,
                                          causal=True)
TINY_RING_ATTN = AttnWorkload("tiny-ring-attn-R4-S256-Hq4-Hkv2", 4, 256, 4, 2)


def make_attn_inputs(w: AttnWorkload, seed: int = 0):
    """Q (rank-independent draw: every rank's queries come from the same
    stream, the rank picks nothing), then K_q and V_q for q = 0..R-1, all
    N(0,1) bf16 token-major.  Returns (Q [S_r, H_q, d], Ks, Vs) as uint16."""
    rng = np.random.default_rng(seed)
    Q = to_bf16_bits(_draw(rng, (w.S_r, w.H_q, w.d), 1.0, "normal"))
    Ks, Vs = [], []
    for _ in range(w.R):
        Ks.append(to_bf16_bits(_draw(rng, (w.S_r, w.H_kv, w.d), 1.0, "normal")))
        Vs.append(to_bf16_bits(_draw(rng, (w.S_r, w.H_kv, w.d), 1.0, "normal")))
    return Q, Ks, Vs


def make_head_attn_inputs(w: AttnWorkload, seed: int = 0):
    """Head-parallel layout: every rank's tokens of all heads.  For q = 0..R-1
    in order: Q_q [S_r, H_q, d], K_q, V_q [S_r, H_kv, d], N(0,1) bf16."""
    rng = np.random.default_rng(seed)
    Qs, Ks, Vs = [], [], []
    for _ in range(w.R):
        Qs.append(to_bf16_bits(_draw(rng, (w.S_r, w.H_q, w.d), 1.0, "normal")))
        Ks.append(to_bf16_bits(_draw(rng, (w.S_r, w.H_kv, w.d), 1.0, "normal")))
        Vs.append(to_bf16_bits(_draw(rng, (w.S_r, w.H_kv, w.d), 1.0, "normal")))
    return Qs, Ks, Vs
