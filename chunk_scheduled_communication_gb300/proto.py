"""ctypes binding of libsynproto.so: the CPU emulation of the chunk ready-flag
protocol (include/syn_proto.h).  Host threads run the plan builder's schedule
with the protocol logic the fused kernel uses; no GPU is involved."""
from __future__ import annotations

import ctypes

from . import build as _build

STALE_DATA = -100

_lib = None


class Cfg(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int), ("R", ctypes.c_int), ("rank", ctypes.c_int),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("split", ctypes.c_int), ("order", ctypes.c_int), ("tile_m", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("walkers", ctypes.c_int), ("stagers", ctypes.c_int),
                ("slice_bytes", ctypes.c_int64), ("calls", ctypes.c_int), ("drop_transfer", ctypes.c_int),
                ("drop_call", ctypes.c_int), ("delay_transfer", ctypes.c_int), ("delay_us", ctypes.c_int),
                ("timeout_us", ctypes.c_int), ("jitter_us", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("mutation", ctypes.c_int), ("rows_from", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build_proto())
        _lib.syn_proto_emulate.restype = ctypes.c_int
        _lib.syn_proto_emulate.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int64)]
        _lib.syn_proto_last_error.restype = ctypes.c_char_p
    return _lib


OPS = {"ag": 0, "rs": 1, "ar": 2}
ORDERS = {"row": 0, "col": 1, "grouped": 2, "banded": 3}


def emulate(op="ag", R=4, rank=0, M=1024, N=256, K=64, split=1, order="row", tile_m=128, tile_n=256,
            walkers=8, stagers=4, slice_bytes=4096, calls=3, drop_transfer=-1, drop_call=1,
            delay_transfer=-1, delay_us=0, timeout_us=200_000, jitter_us=20, seed=1, mutation=0, rows_from=None):
    """Run `calls` emulated calls; returns (statuses, tiles_checked) lists.
    rows_from (op "ag" only): A2A-GEMM row counts per source; M is ignored."""
    rows = None if rows_from is None else (ctypes.c_int64 * R)(*[int(x) for x in rows_from])
    c = Cfg(OPS[op], R, rank, M, N, K, split, ORDERS[order], tile_m, tile_n, walkers, stagers, slice_bytes,
            calls, drop_transfer, drop_call, delay_transfer, delay_us, timeout_us, jitter_us, seed, mutation,
            ctypes.cast(rows, ctypes.c_void_p) if rows is not None else None)
    st = (ctypes.c_int * calls)()
    tc = (ctypes.c_int64 * calls)()
    rc = lib().syn_proto_emulate(ctypes.byref(c), st, tc)
    if rc != 0:
        raise ValueError(f"emulation rejected ({rc}): {lib().syn_proto_last_error().decode()}")
    return list(st), list(tc)
