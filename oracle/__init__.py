"""Plain CPU oracle for AG-GEMM, GEMM-RS, GEMM-AR, A2A-GEMM and ring attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package; the product path
(``chunk_scheduled_communication_gb300``) never does, and shares no code with it.

The arithmetic lives in ``syn_oracle.c`` (plain C, fp32 sequential-k
accumulation over bf16 inputs, one round-to-nearest-even at the end, peers
added in ascending rank order).  This module only compiles it with gcc and
marshals numpy arrays through ctypes.

Every function follows the plain definition of the operator as the Syncopate
summary page names them ("Experiments", paper §6.1: AG-GEMM, GEMM-RS,
GEMM-AR; A2A-GEMM, the all-to-all + expert GEMM of the sensitivity study,
paper §6.3 / Fig. 11); chunking and tile order never change these values
(method section, paper §5.1-§5.2).

Parity pins for every entry point are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "syn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``syn_oracle.c`` into ``liboracle.so`` with gcc (no GPU needed)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_bf16_rne_array.restype = None
        lib.oracle_bf16_rne_array.argtypes = [p, i64, p]
        lib.oracle_threads.restype = i32
        lib.oracle_threads.argtypes = []
        lib.oracle_gather.argtypes = [i32, i64, i64, p, p]
        lib.oracle_gemm_f32.argtypes = [p, p, i64, i64, i64, i64, p]
        lib.oracle_ag_gemm.argtypes = [i32, i64, i64, i64, p, p, i64, i64, p, p]
        lib.oracle_gemm_rs_out.argtypes = [i32, i32, i64, i64, i64, p, p, p, i64, i64, p]
        lib.oracle_gemm_rs_send.argtypes = [i32, i32, i64, i64, i64, p, p, i64, i64, p]
        lib.oracle_gemm_ar.argtypes = [i32, i32, i64, i64, i64, p, p, p, i64, i64, p, p]
        lib.oracle_a2a_gemm.argtypes = [i32, p, i64, i64, p, p, i64, i64, p, p]
        lib.oracle_ring_attention.argtypes = [i32, i32, i64, i32, i32, i32, i32, ctypes.c_double, p, p, p,
                                              i64, i64, p, p]
        for f in ("oracle_gather", "oracle_gemm_f32", "oracle_ag_gemm", "oracle_gemm_rs_out",
                  "oracle_gemm_rs_send", "oracle_gemm_ar", "oracle_a2a_gemm", "oracle_ring_attention"):
            getattr(lib, f).restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrs):
    arr = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    return arr


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as raw uint16 bit patterns")
    return a


def _f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError("partials are float32")
    return a


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_threads())


def bf16_rne(x) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (uint16), ties to even."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


def gather(shards) -> np.ndarray:
    """AllGather: concat of the R shards along rows (bit copy)."""
    lib = _load()
    shards = [_u16(s) for s in shards]
    R, (M_r, K) = len(shards), shards[0].shape
    g = np.empty((R * M_r, K), dtype=np.uint16)
    lib.oracle_gather(R, M_r, K, _ptr_array(shards), _ptr(g))
    return g


def gemm_f32(A, B, row0: int = 0, row1: int | None = None) -> np.ndarray:
    """P = A·B over rows [row0, row1), fp32 sequential-k, not rounded."""
    lib = _load()
    A, B = _u16(A), _u16(B)
    K, N = B.shape
    assert A.shape[1] == K
    row1 = A.shape[0] if row1 is None else row1
    P = np.empty((row1 - row0, N), dtype=np.float32)
    lib.oracle_gemm_f32(_ptr(A), _ptr(B), K, N, row0, row1, _ptr(P))
    return P


def ag_gemm(shards, B, row0: int = 0, row1: int | None = None, want_gathered: bool = True):
    """AG-GEMM.  Returns (gathered or None, C rows [row0,row1) as bf16 bits)."""
    lib = _load()
    shards = [_u16(s) for s in shards]
    B = _u16(B)
    R, (M_r, K) = len(shards), shards[0].shape
    N = B.shape[1]
    assert B.shape[0] == K
    M = R * M_r
    row1 = M if row1 is None else row1
    C = np.empty((row1 - row0, N), dtype=np.uint16)
    g = np.empty((M, K), dtype=np.uint16) if want_gathered else None
    lib.oracle_ag_gemm(R, M_r, K, N, _ptr_array(shards), _ptr(B), row0, row1,
                       _ptr(g) if g is not None else None, _ptr(C))
    return g, C


def a2a_gemm(parts, B, row0: int = 0, row1: int | None = None, want_gathered: bool = True):
    """A2A-GEMM: parts[q] is the [rows_from[q], K] block source q sends (may
    have 0 rows).  Returns (stacked input or None, C rows [row0,row1) as bf16
    bits)."""
    lib = _load()
    B = _u16(B)
    K, N = B.shape
    parts = [_u16(np.asarray(x).reshape(-1, K)) for x in parts]
    R = len(parts)
    rows = np.array([x.shape[0] for x in parts], dtype=np.int64)
    M = int(rows.sum())
    row1 = M if row1 is None else row1
    assert 0 <= row0 <= row1 <= M
    C = np.empty((row1 - row0, N), dtype=np.uint16)
    g = np.empty((M, K), dtype=np.uint16) if want_gathered else None
    lib.oracle_a2a_gemm(R, _ptr(rows), K, N, _ptr_array(parts), _ptr(B), row0, row1,
                        _ptr(g) if g is not None else None, _ptr(C))
    return g, C


def ring_attention(Q, Ks, Vs, r: int, causal: bool = False, scale: float | None = None,
                   row0: int = 0, row1: int | None = None):
    """Ring attention forward of rank r over the keys of all ranks (fp64).

    Q: uint16 [S_r, H_q, d]; Ks, Vs: R arrays uint16 [S_r, H_kv, d].
    Returns (O float64 [row1-row0, H_q, d], lse float64 [row1-row0, H_q])."""
    lib = _load()
    Q = _u16(Q)
    Ks = [_u16(k) for k in Ks]
    Vs = [_u16(v) for v in Vs]
    S_r, H_q, d = Q.shape
    R = len(Ks)
    H_kv = Ks[0].shape[1]
    assert all(k.shape == (S_r, H_kv, d) for k in Ks + Vs) and H_q % H_kv == 0
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    row1 = S_r if row1 is None else row1
    O = np.empty((row1 - row0, H_q, d), dtype=np.float64)
    lse = np.empty((row1 - row0, H_q), dtype=np.float64)
    lib.oracle_ring_attention(R, r, S_r, H_q, H_kv, d, 1 if causal else 0, scale, _ptr(Q), _ptr_array(Ks),
                              _ptr_array(Vs), row0, row1, _ptr(O), _ptr(lse))
    return O, lse


def _peer_ptrs(peers, R, r, M, N):
    """Pointer array for the peers; the local slot may be None (never read)."""
    ptrs = []
    keep = []
    for q in range(R):
        if q == r or peers[q] is None:
            ptrs.append(None)
            continue
        p = _f32(peers[q])
        assert p.shape == (M, N)
        keep.append(p)
        ptrs.append(p.ctypes.data)
    arr = (ctypes.c_void_p * R)(*ptrs)
    return arr, keep


def gemm_rs(A, B, peers, R: int, r: int, i0: int = 0, i1: int | None = None,
            send_rows: tuple[int, int] | None = None):
    """GEMM-RS for rank r.

    Returns (out_r rows [i0,i1) as bf16 bits, send) where ``send`` is the fp32
    P rows for global rows ``send_rows`` (rows of rank r left as NaN), or None.
    """
    lib = _load()
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N = B.shape[1]
    M_r = M // R
    i1 = M_r if i1 is None else i1
    arr, keep = _peer_ptrs(peers, R, r, M, N)
    out = np.empty((i1 - i0, N), dtype=np.uint16)
    lib.oracle_gemm_rs_out(R, r, M, K, N, _ptr(A), _ptr(B), arr, i0, i1, _ptr(out))
    send = None
    if send_rows is not None:
        s0, s1 = send_rows
        send = np.full((s1 - s0, N), np.nan, dtype=np.float32)
        lib.oracle_gemm_rs_send(R, r, M, K, N, _ptr(A), _ptr(B), s0, s1, _ptr(send))
    del keep
    return out, send


def gemm_ar(A, B, peers, R: int, r: int, row0: int = 0, row1: int | None = None,
            want_publish: bool = False):
    """GEMM-AR for rank r.  Returns (out rows [row0,row1) bf16 bits, publish or None)."""
    lib = _load()
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N = B.shape[1]
    row1 = M if row1 is None else row1
    arr, keep = _peer_ptrs(peers, R, r, M, N)
    out = np.empty((row1 - row0, N), dtype=np.uint16)
    pub = np.empty((row1 - row0, N), dtype=np.float32) if want_publish else None
    lib.oracle_gemm_ar(R, r, M, K, N, _ptr(A), _ptr(B), arr, row0, row1, _ptr(out),
                       _ptr(pub) if pub is not None else None)
    del keep
    return out, pub
