"""ctypes binding of the ring-attention entry points (include/syn_attn.h).

Argument marshalling only: every step of the operator runs in libsyn.so."""
from __future__ import annotations

import ctypes

import numpy as np

from . import syn

_P = ctypes.c_void_p


class AttnCfg(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("rank", ctypes.c_int), ("S_r", ctypes.c_int64), ("H_q", ctypes.c_int),
                ("H_kv", ctypes.c_int), ("d", ctypes.c_int), ("causal", ctypes.c_int), ("split", ctypes.c_int),
                ("backend", ctypes.c_int), ("scale", ctypes.c_float), ("timeout_ns", ctypes.c_uint64),
                ("debug_drop_chunk", ctypes.c_int), ("head_parallel", ctypes.c_int)]


class AttnInfo(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("rank", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int),
                ("d", ctypes.c_int), ("causal", ctypes.c_int), ("split", ctypes.c_int), ("backend", ctypes.c_int),
                ("S_r", ctypes.c_int64), ("n_qtiles", ctypes.c_int), ("grid", ctypes.c_int),
                ("n_transfers", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("epoch", ctypes.c_uint32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


SIGS = {
    "syn_attn_cfg_default": (ctypes.c_int, [ctypes.POINTER(AttnCfg)]),
    "syn_attn_plan_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.POINTER(AttnCfg)]),
    "syn_attn_plan_destroy": (ctypes.c_int, [_P]),
    "syn_ring_attention": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "syn_head_attention": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "syn_attn_sync_status": (ctypes.c_int, [_P, _P]),
    "syn_attn_plan_query": (ctypes.c_int, [_P, ctypes.POINTER(AttnInfo)]),
    "syn_attn_plan_flags": (ctypes.c_int, [_P, _P]),
}

_bound = None


def lib():
    """libsyn.so with the attention signatures bound (raises if the library is missing)."""
    global _bound
    L = syn.lib()
    if _bound is not L:
        for name, (res, args) in SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _bound = L
    return L


def make_cfg(R=1, rank=0, S_r=256, H_q=1, H_kv=1, d=128, causal=False, split=1, backend="tma_colocated", scale=0.0,
             timeout_ns=0, drop_chunk=-1, head_parallel=False) -> AttnCfg:
    c = AttnCfg()
    _check(lib().syn_attn_cfg_default(ctypes.byref(c)), "syn_attn_cfg_default")
    c.R, c.rank, c.S_r, c.H_q, c.H_kv, c.d = R, rank, S_r, H_q, H_kv, d
    c.causal, c.split = int(bool(causal)), split
    c.backend = syn.BACKENDS[backend] if isinstance(backend, str) else int(backend)
    c.scale, c.timeout_ns, c.debug_drop_chunk = scale, timeout_ns, drop_chunk
    c.head_parallel = int(bool(head_parallel))
    return c


def _check(status, where):
    if status != syn.OK:
        raise syn.SynError(status, where)


class AttnPlan:
    """A ring-attention plan on the current CUDA device (wraps syn_attn_plan_t)."""

    def __init__(self, **cfg):
        self._L = lib()
        self._h = _P()
        self.cfg = make_cfg(**cfg)
        _check(self._L.syn_attn_plan_create(ctypes.byref(self._h), ctypes.byref(self.cfg)), "syn_attn_plan_create")

    def close(self):
        if self._h:
            self._L.syn_attn_plan_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def info(self) -> dict:
        i = AttnInfo()
        _check(self._L.syn_attn_plan_query(self._h, ctypes.byref(i)), "syn_attn_plan_query")
        return i.as_dict()

    def flags(self):
        n = self.cfg.R * self.cfg.split
        out = np.empty(n, np.uint32)
        _check(self._L.syn_attn_plan_flags(self._h, out.ctypes.data), "syn_attn_plan_flags")
        return out

    def run(self, Q, K_shards, V_shards, K_gathered, V_gathered, O, lse=None, stream=None):
        R = self.cfg.R
        ks = (_P * R)(*[syn._ptr(t) for t in K_shards])
        vs = (_P * R)(*[syn._ptr(t) for t in V_shards])
        _check(self._L.syn_ring_attention(self._h, syn._ptr(Q), ks, vs, syn._ptr(K_gathered), syn._ptr(V_gathered),
                                          syn._ptr(O), syn._ptr(lse), syn._stream(stream)), "syn_ring_attention")

    def run_head(self, Q_shards, K_shards, V_shards, Q_gathered, K_gathered, V_gathered, O, lse=None, stream=None):
        R = self.cfg.R
        arr = lambda ts: (_P * R)(*[syn._ptr(t) for t in ts])
        _check(self._L.syn_head_attention(self._h, arr(Q_shards), arr(K_shards), arr(V_shards), syn._ptr(Q_gathered),
                                          syn._ptr(K_gathered), syn._ptr(V_gathered), syn._ptr(O), syn._ptr(lse),
                                          syn._stream(stream)), "syn_head_attention")

    def sync(self, stream=None) -> int:
        return int(self._L.syn_attn_sync_status(self._h, syn._stream(stream)))

    def check(self, stream=None):
        _check(self.sync(stream), "syn_attn_sync_status")
