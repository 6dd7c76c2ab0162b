"""Python binding of libsyn's C ABI (argument marshalling only).

Every computation happens in libsyn.so (CUDA kernels for sm_103a plus the
copy-engine stager).  This module loads the in-tree library, mirrors the
structs of ``include/syn.h`` with ctypes and turns torch tensors into device
pointers and torch streams into ``cudaStream_t`` handles.  PyTorch is only the
allocator and stream provider.  If the library is missing this module raises:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsyn.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, -1, -2, -3, -4, -5
OP_AG_GEMM, OP_GEMM_RS, OP_GEMM_AR = 0, 1, 2
ORDER_ROW_MAJOR, ORDER_COL_MAJOR, ORDER_GROUPED, ORDER_BANDED = 0, 1, 2, 3
(BACKEND_CE, BACKEND_TMA_DEDICATED, BACKEND_TMA_COLOCATED, BACKEND_TMA_COLOCATED_SMEM,
 BACKEND_UNFUSED, BACKEND_DECOMPOSED, BACKEND_LDST_DEDICATED, BACKEND_LDST_COLOCATED) = range(8)
BACKEND_NAMES = {BACKEND_CE: "ce", BACKEND_TMA_DEDICATED: "tma_dedicated",
                 BACKEND_TMA_COLOCATED: "tma_colocated", BACKEND_TMA_COLOCATED_SMEM: "tma_colocated_smem",
                 BACKEND_UNFUSED: "unfused", BACKEND_DECOMPOSED: "decomposed",
                 BACKEND_LDST_DEDICATED: "ldst_dedicated", BACKEND_LDST_COLOCATED: "ldst_colocated"}
BACKENDS = {v: k for k, v in BACKEND_NAMES.items()}
ORDERS = {"row": ORDER_ROW_MAJOR, "col": ORDER_COL_MAJOR, "grouped": ORDER_GROUPED, "banded": ORDER_BANDED}
OPS = {"ag": OP_AG_GEMM, "rs": OP_GEMM_RS, "ar": OP_GEMM_AR}


class Layout(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64)]


class Knobs(ctypes.Structure):
    _fields_ = [("backend", ctypes.c_int), ("comm_sms", ctypes.c_int), ("tile_m", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("group_m", ctypes.c_int), ("slice_kb", ctypes.c_int),
                ("timeout_ns", ctypes.c_uint64), ("debug_drop_chunk", ctypes.c_int),
                ("trace", ctypes.c_int), ("stages", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("reduce_spread", ctypes.c_int), ("reduce_warps", ctypes.c_int),
                ("ce_streams", ctypes.c_int), ("rs_push", ctypes.c_int), ("debug_delay_chunk", ctypes.c_int),
                ("debug_delay_us", ctypes.c_int), ("debug_corrupt_entry", ctypes.c_int),
                ("direct_fetch", ctypes.c_int), ("push_sms", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int), ("R", ctypes.c_int), ("rank", ctypes.c_int),
                ("backend", ctypes.c_int), ("order", ctypes.c_int),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("M_r", ctypes.c_int64), ("chunk_rows", ctypes.c_int64), ("split", ctypes.c_int),
                ("n_row_chunks", ctypes.c_int), ("n_transfers", ctypes.c_int),
                ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int), ("tiles_m", ctypes.c_int),
                ("tiles_n", ctypes.c_int), ("n_tiles", ctypes.c_int), ("grid_compute", ctypes.c_int),
                ("grid_comm", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("epoch", ctypes.c_uint32), ("recv_bytes", ctypes.c_uint64), ("a2a", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


# Every function the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_SIGS = {
    "syn_schedule_build": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Layout),
                                          ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Knobs),
                                          ctypes.POINTER(PlanInfo), _P, _P, _P]),
    "syn_knobs_default": (ctypes.c_int, [ctypes.POINTER(Knobs)]),
    "syn_plan_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(Layout), ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(Knobs)]),
    "syn_plan_create_a2a": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int, ctypes.c_int, _P, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Knobs)]),
    "syn_schedule_build_a2a": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int, ctypes.c_int, ctypes.POINTER(Knobs),
                                              ctypes.POINTER(PlanInfo), _P, _P, _P]),
    "syn_a2a_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "syn_plan_destroy": (ctypes.c_int, [_P]),
    "syn_ag_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "syn_gemm_rs": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "syn_gemm_ar": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "syn_sync_status": (ctypes.c_int, [_P, _P]),
    "syn_plan_query": (ctypes.c_int, [_P, ctypes.POINTER(PlanInfo)]),
    "syn_plan_tables": (ctypes.c_int, [_P, _P, _P, _P]),
    "syn_plan_flags": (ctypes.c_int, [_P, _P, _P]),
    "syn_plan_stats": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "syn_plan_trace": (ctypes.c_int, [_P, _P]),
    "syn_autotune": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Layout),
                                    ctypes.c_double, ctypes.POINTER(Knobs), ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]),
    "syn_device_sms": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
    "syn_ag_gemm_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.POINTER(Layout), ctypes.c_int,
                                           ctypes.c_int, _P, _P, _P, _P, _P, _P]),
    "syn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "syn_last_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def lib():
    """Load libsyn.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build(); "
                                   "there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
        return _lib


class SynError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = lib()
        msg = L.syn_last_error().decode(errors="replace")
        super().__init__(f"{where}: {L.syn_status_string(status).decode()} ({status}): {msg}")
        self.status = status


def _check(status: int, where: str):
    if status != OK:
        raise SynError(status, where)


def make_knobs(backend="tma_colocated", comm_sms=8, tile_n=256, group_m=8, slice_kb=128, timeout_ns=0,
               drop_chunk=-1, trace=0, stages=0, tile_k=0, tile_m=0, reduce_spread=0,
               reduce_warps=0, ce_streams=0, delay_chunk=-1, delay_us=0, corrupt_entry=0,
               rs_push=0, direct_fetch=0, push_sms=0) -> Knobs:
    k = Knobs()
    _check(lib().syn_knobs_default(ctypes.byref(k)), "syn_knobs_default")
    k.backend = BACKENDS[backend] if isinstance(backend, str) else int(backend)
    k.comm_sms, k.tile_n, k.group_m, k.slice_kb = comm_sms, tile_n, group_m, slice_kb
    k.timeout_ns, k.debug_drop_chunk, k.trace, k.stages, k.tile_k = timeout_ns, drop_chunk, trace, stages, tile_k
    k.tile_m = tile_m
    k.reduce_spread = reduce_spread
    k.reduce_warps = reduce_warps
    k.ce_streams = ce_streams
    k.rs_push = rs_push
    k.debug_delay_chunk, k.debug_delay_us, k.debug_corrupt_entry = delay_chunk, delay_us, corrupt_entry
    k.direct_fetch = direct_fetch
    k.push_sms = push_sms
    return k


def _op(op):
    return OPS[op] if isinstance(op, str) else int(op)


def _order(order):
    return ORDERS[order] if isinstance(order, str) else int(order)


def schedule_build(op, R, rank, M, N, K, chunk_rows=0, split=1, order="row", **knobs):
    """Host-only schedule (no GPU needed): info dict + tile_list, tile_key, transfers arrays."""
    L = lib()
    lay = Layout(M, N, K, 0, 0, 0)
    kn = make_knobs(**knobs)
    info = PlanInfo()
    _check(L.syn_schedule_build(_op(op), R, rank, ctypes.byref(lay), chunk_rows, split, _order(order),
                                ctypes.byref(kn), ctypes.byref(info), None, None, None), "syn_schedule_build")
    tl = np.empty(info.n_tiles, np.int32)
    tk = np.empty(info.n_tiles, np.int32)
    tr = np.empty(max(info.n_transfers, 1), np.int32)
    _check(L.syn_schedule_build(_op(op), R, rank, ctypes.byref(lay), chunk_rows, split, _order(order),
                                ctypes.byref(kn), ctypes.byref(info), tl.ctypes.data, tk.ctypes.data,
                                tr.ctypes.data), "syn_schedule_build")
    return info.as_dict(), tl, tk, tr[:info.n_transfers]


def schedule_build_a2a(R, rank, rows_from, N, K, split=1, order="row", **knobs):
    """Host-only A2A-GEMM schedule: info dict + tile_list, tile_key, transfers."""
    L = lib()
    rows = np.ascontiguousarray(rows_from, dtype=np.int64)
    if rows.shape != (R,):
        raise ValueError("rows_from needs R entries")
    kn = make_knobs(**knobs)
    info = PlanInfo()
    _check(L.syn_schedule_build_a2a(R, rank, rows.ctypes.data, N, K, split, _order(order), ctypes.byref(kn),
                                    ctypes.byref(info), None, None, None), "syn_schedule_build_a2a")
    tl = np.empty(info.n_tiles, np.int32)
    tk = np.empty(info.n_tiles, np.int32)
    tr = np.empty(max(info.n_transfers, 1), np.int32)
    _check(L.syn_schedule_build_a2a(R, rank, rows.ctypes.data, N, K, split, _order(order), ctypes.byref(kn),
                                    ctypes.byref(info), tl.ctypes.data, tk.ctypes.data, tr.ctypes.data),
           "syn_schedule_build_a2a")
    return info.as_dict(), tl, tk, tr[:info.n_transfers]


def _ptr(t) -> int:
    if t is None:
        return 0
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Plan:
    """A chunk plan on the current CUDA device (wraps syn_plan_t)."""

    def __init__(self, op, R, rank, M, N, K, chunk_rows=0, split=1, order="row", **knobs):
        self._L = lib()
        self._h = _P()
        lay = Layout(M, N, K, 0, 0, 0)
        self.knobs = make_knobs(**knobs)
        _check(self._L.syn_plan_create(ctypes.byref(self._h), _op(op), R, rank, ctypes.byref(lay),
                                       chunk_rows, split, _order(order), ctypes.byref(self.knobs)),
               "syn_plan_create")
        self.op, self.R, self.rank, self.M, self.N, self.K = _op(op), R, rank, M, N, K

    @classmethod
    def a2a(cls, R, rank, rows_from, N, K, split=1, order="row", **knobs):
        """An A2A-GEMM plan: rank `rank`'s expert receives rows_from[q] rows from rank q."""
        self = cls.__new__(cls)
        self._L = lib()
        self._h = _P()
        rows = np.ascontiguousarray(rows_from, dtype=np.int64)
        if rows.shape != (R,):
            raise ValueError("rows_from needs R entries")
        self.knobs = make_knobs(**knobs)
        _check(self._L.syn_plan_create_a2a(ctypes.byref(self._h), R, rank, rows.ctypes.data, N, K, split,
                                           _order(order), ctypes.byref(self.knobs)), "syn_plan_create_a2a")
        self.op, self.R, self.rank, self.M, self.N, self.K = OPS["ag"], R, rank, int(rows.sum()), N, K
        self.rows_from = rows
        return self

    # -- lifetime
    def close(self):
        if self._h:
            self._L.syn_plan_destroy(self._h)
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

    # -- introspection
    def info(self) -> dict:
        i = PlanInfo()
        _check(self._L.syn_plan_query(self._h, ctypes.byref(i)), "syn_plan_query")
        return i.as_dict()

    def tables(self):
        i = self.info()
        tl = np.empty(i["n_tiles"], np.int32)
        tk = np.empty(i["n_tiles"], np.int32)
        tr = np.empty(max(i["n_transfers"], 1), np.int32)
        _check(self._L.syn_plan_tables(self._h, tl.ctypes.data, tk.ctypes.data, tr.ctypes.data), "syn_plan_tables")
        return tl, tk, tr[:i["n_transfers"]]

    def flags(self):
        i = self.info()
        fin = np.empty(i["n_row_chunks"] * i["R"], np.uint32)
        fout = np.empty(i["n_row_chunks"], np.uint32)
        _check(self._L.syn_plan_flags(self._h, fin.ctypes.data, fout.ctypes.data), "syn_plan_flags")
        return fin, fout

    def stats(self):
        a, b = ctypes.c_uint64(), ctypes.c_uint64()
        _check(self._L.syn_plan_stats(self._h, ctypes.byref(a), ctypes.byref(b)), "syn_plan_stats")
        return a.value, b.value

    def trace(self):
        """Per-tile timeline of the last call (trace=2): int64 [n_tiles, 5] of
        (MMA start, MMA end, epilogue start, epilogue end) global-timer ns and
        the walker that ran the tile, rows in tile-list order."""
        n = self.info()["n_tiles"]
        out = np.zeros((n, 5), np.uint64)
        _check(self._L.syn_plan_trace(self._h, out.ctypes.data), "syn_plan_trace")
        return out.astype(np.int64)

    # -- operators (asynchronous on `stream`)
    def ag_gemm(self, shards, gathered, B, C, stream=None):
        arr = (_P * self.R)(*[_ptr(s) for s in shards])
        _check(self._L.syn_ag_gemm(self._h, arr, _ptr(gathered), _ptr(B), _ptr(C), _stream(stream)),
               "syn_ag_gemm")

    def a2a_gemm(self, parts, gathered, B, C, stream=None):
        arr = (_P * self.R)(*[_ptr(s) for s in parts])
        _check(self._L.syn_a2a_gemm(self._h, arr, _ptr(gathered), _ptr(B), _ptr(C), _stream(stream)),
               "syn_a2a_gemm")

    def gemm_rs(self, A, B, peers, send, out_r, stream=None):
        arr = (_P * self.R)(*[_ptr(p) for p in peers])
        _check(self._L.syn_gemm_rs(self._h, _ptr(A), _ptr(B), arr, _ptr(send), _ptr(out_r), _stream(stream)),
               "syn_gemm_rs")

    def gemm_ar(self, A, B, peers, publish, out, stream=None):
        arr = (_P * self.R)(*[_ptr(p) for p in peers])
        _check(self._L.syn_gemm_ar(self._h, _ptr(A), _ptr(B), arr, _ptr(publish), _ptr(out), _stream(stream)),
               "syn_gemm_ar")

    def sync(self, stream=None) -> int:
        """Synchronise and return the status (does not raise)."""
        return int(self._L.syn_sync_status(self._h, _stream(stream)))

    def check(self, stream=None):
        _check(self.sync(stream), "syn_sync_status")


def autotune(op, R, rank, M, N, K, budget_s=60.0, rs_push=0):
    L = lib()
    lay = Layout(M, N, K, 0, 0, 0)
    kn = Knobs()
    kn.rs_push = rs_push
    split = ctypes.c_int()
    order = ctypes.c_int()
    us = ctypes.c_double()
    _check(L.syn_autotune(_op(op), R, rank, ctypes.byref(lay), budget_s, ctypes.byref(kn), ctypes.byref(split),
                          ctypes.byref(order), ctypes.byref(us)), "syn_autotune")
    return {"backend": BACKEND_NAMES.get(kn.backend, kn.backend), "comm_sms": kn.comm_sms,
            "tile_m": kn.tile_m, "tile_n": kn.tile_n, "group_m": kn.group_m, "stages": kn.stages,
            "reduce_warps": kn.reduce_warps, "direct_fetch": kn.direct_fetch, "rs_push": kn.rs_push,
            "push_sms": kn.push_sms,
            "split": split.value, "order": order.value, "us": us.value}


def ag_gemm_noalloc(R, rank, M, N, K, shards, gathered, B, C, split=1, order="row", status=None,
                    stream=None):
    """AG-GEMM through syn_ag_gemm_noalloc (no device allocation; see include/syn.h)."""
    lay = Layout(M, N, K, 0, 0, 0)
    arr = (_P * R)(*[_ptr(s) for s in shards])
    _check(lib().syn_ag_gemm_noalloc(R, rank, ctypes.byref(lay), split, _order(order), arr, _ptr(gathered),
                                     _ptr(B), _ptr(C), _ptr(status), _stream(stream)), "syn_ag_gemm_noalloc")


def device_sms() -> int:
    n = ctypes.c_int()
    _check(lib().syn_device_sms(ctypes.byref(n)), "syn_device_sms")
    return n.value
