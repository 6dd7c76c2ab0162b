"""Convenience layer over the binding: device buffers for a workload, one call
of the plan's operator, outputs back on the host, and the tolerance check.

Everything computed here is computed by libsyn; this module only allocates
(PyTorch), copies, and compares numbers it is given.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import syn
from .workloads import Inputs

# Tolerances for floating-point outputs (bf16 and fp32), against the oracle:
# per element |gpu - ref| <= ATOL + RTOL * |ref|, and relative Frobenius error
# ||gpu - ref|| / ||ref|| <= FROB.
ATOL, RTOL, FROB = 1e-2, 1e-2, 2e-3


def _u16_to_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def dev_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclass
class DeviceInputs:
    op: str
    R: int
    r: int
    M: int
    N: int
    K: int
    shards: list = field(default_factory=list)   # AG / A2A: shard (part) tensors (shards[r] aliases gathered)
    rows_from: list | None = None                # A2A: rows each source sends
    gathered: torch.Tensor | None = None
    A: torch.Tensor | None = None
    B: torch.Tensor | None = None
    peers: list = field(default_factory=list)
    out: torch.Tensor | None = None              # C / out_r / out
    f32_out: torch.Tensor | None = None          # send / publish


def upload(inp: Inputs, device="cuda", inplace_local=True, with_f32_out=True) -> DeviceInputs:
    """Device buffers for one call.  AG: the local shard is written into its
    slot of the gathered buffer (in-place) unless ``inplace_local`` is False."""
    w = inp.w
    d = DeviceInputs(op=w.op, R=w.R, r=inp.r, M=w.M, N=w.N, K=w.K)
    d.B = _u16_to_dev(inp.B, device)
    if w.op == "a2a":
        d.rows_from = list(inp.rows_from)
        d.M = M = sum(d.rows_from)
        off = np.concatenate([[0], np.cumsum(d.rows_from)]).astype(int)
        d.gathered = torch.zeros((M, w.K), dtype=torch.bfloat16, device=device)
        for q in range(w.R):
            if d.rows_from[q] == 0:
                d.shards.append(None)  # nothing sent: a NULL part
            elif q == inp.r and inplace_local:
                slot = d.gathered[off[q]:off[q + 1]]
                slot.copy_(_u16_to_dev(inp.shards[q], device))
                d.shards.append(slot)
            else:
                d.shards.append(_u16_to_dev(inp.shards[q], device))
        d.out = torch.empty((M, w.N), dtype=torch.bfloat16, device=device)
    elif w.op == "ag":
        d.gathered = torch.zeros((w.M, w.K), dtype=torch.bfloat16, device=device)
        for q in range(w.R):
            if q == inp.r and inplace_local:
                slot = d.gathered[q * w.M_r:(q + 1) * w.M_r]
                slot.copy_(_u16_to_dev(inp.shards[q], device))
                d.shards.append(slot)
            else:
                d.shards.append(_u16_to_dev(inp.shards[q], device))
        d.out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
    else:
        d.A = _u16_to_dev(inp.A, device)
        d.peers = [None if p is None else torch.from_numpy(p).to(device) for p in inp.peers]
        rows = w.M_r if w.op == "rs" else w.M
        d.out = torch.empty((rows, w.N), dtype=torch.bfloat16, device=device)
        if with_f32_out:
            d.f32_out = torch.full((w.M, w.N), float("nan"), dtype=torch.float32, device=device)
    return d


def call(plan: syn.Plan, d: DeviceInputs, stream=None):
    """Issue one asynchronous call of the plan's operator."""
    if d.op == "ag":
        plan.ag_gemm(d.shards, d.gathered, d.B, d.out, stream)
    elif d.op == "a2a":
        plan.a2a_gemm(d.shards, d.gathered, d.B, d.out, stream)
    elif d.op == "rs":
        plan.gemm_rs(d.A, d.B, d.peers, d.f32_out, d.out, stream)
    else:
        plan.gemm_ar(d.A, d.B, d.peers, d.f32_out, d.out, stream)


def make_plan(d: DeviceInputs, split=1, order="row", **knobs) -> syn.Plan:
    if d.op == "a2a":
        return syn.Plan.a2a(d.R, d.r, d.rows_from, d.N, d.K, split=split, order=order, **knobs)
    return syn.Plan(d.op, d.R, d.r, d.M, d.N, d.K, split=split, order=order, **knobs)


def bf16_close(gpu_bits: np.ndarray, ref_bits: np.ndarray):
    """Tolerance check of bf16 outputs.  Returns (ok, max_abs_excess, rel_frob)."""
    g = torch.from_numpy(gpu_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    r = torch.from_numpy(ref_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    return f_close(g, r)


def f_close(g: np.ndarray, r: np.ndarray):
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if g.shape != r.shape:
        return False, float("inf"), float("inf")
    if not np.isfinite(g).all():
        return False, float("inf"), float("inf")
    diff = np.abs(g - r)
    excess = float((diff - (ATOL + RTOL * np.abs(r))).max()) if diff.size else 0.0
    nr = float(np.linalg.norm(r))
    frob = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g - r))
    return (excess <= 0.0 and frob <= FROB), excess, frob
