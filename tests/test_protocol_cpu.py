"""The chunk ready-flag protocol, emulated with host threads (no GPU).

libsynproto.so runs the plan builder's real schedule and the protocol logic
the fused kernel shares (epoch flags, double-buffered slice counters,
last-arriver publication, the persistent walk, chunk ranges, transfer rows)
with std::thread stagers and walkers over std::atomic flags.  Every walker
checks the bytes of every chunk it waited for; faults are injected on the
host: a flag never published must end the call in SYN_ERR_TIMEOUT without a
hang, and the next call must succeed; a late flag only delays.
"""
import time

import pytest

from chunk_scheduled_communication_gb300 import proto, syn

TIMEOUT = syn.ERR_TIMEOUT


def n_tiles(M, N, tile_m, tile_n):
    return -(-M // tile_m) * (N // tile_n)


@pytest.mark.parametrize("op,R,rank,M,N,K,split,order,tile_m", [
    ("ag", 4, 1, 256, 256, 64, 1, "row", 128),        # 64-row shards: every tile straddles 2 chunks
    ("ag", 8, 0, 2048, 512, 64, 4, "grouped", 128),
    ("ag", 3, 2, 600, 512, 64, 2, "col", 128),        # M tail, odd R
    ("ag", 8, 5, 4096, 512, 64, 3, "row", 256),       # uneven 3-way split, 256-row tiles
    ("rs", 4, 2, 1024, 512, 64, 2, "row", 128),
    ("rs", 8, 7, 2048, 256, 64, 4, "grouped", 256),
    ("rs", 4, 1, 4 * 96, 256, 64, 2, "row", 128),      # blocks of 96 rows: tiles straddle block edges
    ("rs", 5, 3, 5 * 160, 256, 64, 3, "row", 256),     # odd R, pair tiles straddling, ragged last tile
    ("ar", 4, 0, 1000, 256, 64, 3, "row", 128),       # M tail, uneven chunks
    ("ar", 2, 1, 512, 512, 64, 1, "col", 256),
])
def test_every_tile_sees_its_chunks(op, R, rank, M, N, K, split, order, tile_m):
    st, tc = proto.emulate(op=op, R=R, rank=rank, M=M, N=N, K=K, split=split, order=order, tile_m=tile_m,
                           walkers=6, stagers=5, slice_bytes=2048, calls=3)
    assert st == [0, 0, 0]
    assert tc == [n_tiles(M, N, tile_m, 256)] * 3


@pytest.mark.parametrize("walkers,stagers,slice_bytes", [(1, 1, 16), (16, 3, 1000 // 16 * 16), (3, 16, 65536)])
def test_worker_counts_and_slice_sizes(walkers, stagers, slice_bytes):
    st, tc = proto.emulate(op="ag", R=4, rank=3, M=1024, N=512, K=64, split=2, walkers=walkers,
                           stagers=stagers, slice_bytes=slice_bytes, calls=2)
    assert st == [0, 0]


def test_dropped_flag_times_out_then_the_next_call_recovers():
    t0 = time.monotonic()
    st, tc = proto.emulate(op="ag", R=4, rank=0, M=1024, N=256, K=64, split=2, calls=3, drop_transfer=3,
                           drop_call=2, timeout_us=50_000)
    assert time.monotonic() - t0 < 10.0  # bounded: no hang
    assert st == [0, TIMEOUT, 0]
    assert tc[0] == tc[2] == n_tiles(1024, 256, 128, 256) and tc[1] < tc[0]


@pytest.mark.parametrize("op", ["rs", "ar"])
def test_dropped_peer_chunk_times_out(op):
    st, _ = proto.emulate(op=op, R=4, rank=1, M=1024, N=256, K=64, split=2, calls=2, drop_transfer=0,
                          drop_call=1, timeout_us=50_000)
    assert st == [TIMEOUT, 0]


def test_late_flag_only_delays():
    # arrival indices 0 and 1 are the local shard's two chunks (in place, not
    # staged); 3 is a peer chunk
    st, _ = proto.emulate(op="ag", R=4, rank=0, M=1024, N=256, K=64, split=2, calls=2, delay_transfer=3,
                          delay_us=20_000, timeout_us=500_000)
    assert st == [0, 0]
    st, _ = proto.emulate(op="ag", R=4, rank=0, M=1024, N=256, K=64, split=2, calls=2, delay_transfer=3,
                          delay_us=300_000, timeout_us=50_000)
    assert st[0] == TIMEOUT and st[1] == TIMEOUT  # every call publishes that flag too late


def test_a_broken_protocol_is_caught():
    """The harness has teeth: publishing a flag before the bytes land is seen
    by the consumers as stale data."""
    st, _ = proto.emulate(op="ag", R=4, rank=0, M=1024, N=256, K=64, split=1, calls=1, mutation=1,
                          timeout_us=500_000, jitter_us=0)
    assert st == [proto.STALE_DATA]


def test_rejected_plan_reports_invalid():
    with pytest.raises(ValueError):
        proto.emulate(op="rs", R=4, rank=0, M=4 * 100, N=256, K=64)  # M/R not a multiple of 32


# --------------------------------------------------------------------------- A2A-GEMM row blocks
@pytest.mark.parametrize("rows_from,rank,split,tile_m", [
    ([300, 0, 41, 1000], 2, 1, 128),      # an empty block inside a tile's rows
    ([300, 0, 41, 1000], 0, 3, 256),
    ([5, 7, 0, 1, 900, 64, 0, 33], 6, 4, 128),
    ([2, 3], 1, 8, 128),                  # blocks smaller than split: empty chunks
    ([0, 0, 0, 700], 3, 2, 128),          # only the local rank sends
])
def test_a2a_every_tile_sees_its_chunks(rows_from, rank, split, tile_m):
    M = sum(rows_from)
    st, tc = proto.emulate(op="ag", R=len(rows_from), rank=rank, M=0, N=256, K=64, split=split, tile_m=tile_m,
                           walkers=6, stagers=5, slice_bytes=2048, calls=3, rows_from=rows_from)
    assert st == [0, 0, 0]
    assert tc == [n_tiles(M, 256, tile_m, 256)] * 3


def test_a2a_dropped_flag_times_out_then_recovers():
    # rank 0 of [400, 100, 0, 250]: arrival 0 is the local chunk (in place);
    # arrival 1 is source 1's chunk, which tiles 3 and 4 read
    st, tc = proto.emulate(op="ag", R=4, rank=0, M=0, N=256, K=64, split=1, calls=3, drop_transfer=1,
                           drop_call=2, timeout_us=50_000, rows_from=[400, 100, 0, 250])
    assert st == [0, TIMEOUT, 0]


def test_a2a_rows_from_rejected_outside_ag():
    with pytest.raises(ValueError):
        proto.emulate(op="rs", R=2, rank=0, M=0, N=256, K=64, rows_from=[128, 128])
