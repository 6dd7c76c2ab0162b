"""Host-side chunk plan (no GPU): partition, arrival order, dependency keys
and the rewritten tile order (Syncopate summary page, method ¶2 and ¶4, paper
§5.2, Fig. 6; Entwine abstract for the producer-side send order).

Every property is recomputed here from its definition, independently of the
library's code, and compared with what syn_schedule_build returns.
"""
import itertools

import numpy as np
import pytest

from chunk_scheduled_communication_gb300 import syn


@pytest.fixture(scope="module", autouse=True)
def _lib():
    syn.lib()


def expected_transfers(op, R, r, split):
    """Arrival order by definition: local data first, then the ring q = r+1..r-1."""
    out = []
    if op == "ag":
        for d in range(R):
            q = (r + d) % R
            out += [(q * split + j) * R + q for j in range(split)]
    else:
        blocks = [r] if op == "rs" else [(r + d) % R for d in range(R)]
        for b in blocks:
            for j in range(split):
                out += [(b * split + j) * R + (r + d) % R for d in range(1, R)]
    return out


def chunk_bounds(M_r, split):
    """Local row boundaries of the split chunks of one rank block: chunk j is
    [ceil(j*M_r/split), ceil((j+1)*M_r/split)) -- written with integer ceil."""
    return [-(-j * M_r // split) for j in range(split + 1)]


def chunk_of(row, M_r, split):
    q, rr = divmod(row, M_r)
    b = chunk_bounds(M_r, split)
    j = max(k for k in range(split) if b[k] <= rr)
    return q * split + j


def deps(op, R, r, M, M_r, split, tm, tile_m=128):
    rows = range(tm * tile_m, min((tm + 1) * tile_m, M))
    rcs = sorted({chunk_of(i, M_r, split) for i in rows})
    if op == "ag":
        return [rc * R + rc // split for rc in rcs]
    if op == "rs" and (tm * tile_m) // M_r != r:
        return []
    return [rc * R + q for rc in rcs for q in range(R) if q != r]


CASES = [
    ("ag", 4, 1, 256, 256, 256, 1),     # tiny: each tile straddles 2 shards
    ("ag", 8, 0, 8192, 1792, 4096, 2),
    ("ag", 8, 5, 8192, 1792, 4096, 4),
    ("ag", 3, 2, 600, 512, 192, 1),     # ragged M tail, chunk rows 200
    ("ag", 8, 3, 16384, 3584, 8192, 8),
    ("ag", 8, 0, 16384, 3584, 8192, 3),   # split does not divide M/R: uneven chunks
    ("ag", 8, 6, 16384, 3584, 8192, 7),
    ("ag", 4, 2, 4 * 100, 256, 128, 3),   # 34/33/33-row chunks straddling tiles
    ("ar", 8, 5, 4096, 3584, 2368, 3),
    ("ag", 8, 7, 128, 256, 128, 1),     # 8 chunks inside one tile
    ("rs", 8, 0, 8192, 4096, 1792, 1),
    ("rs", 8, 6, 8192, 4096, 1792, 4),
    ("rs", 4, 1, 1024, 256, 320, 2),
    ("rs", 8, 2, 8192, 4096, 1792, 3),
    ("ar", 8, 0, 4096, 3584, 2368, 1),
    ("ar", 8, 4, 4096, 3584, 2368, 4),
    ("ar", 2, 1, 666, 384, 128, 1),
]


@pytest.mark.parametrize("op,R,r,M,N,K,split", CASES)
@pytest.mark.parametrize("order", ["row", "col", "grouped"])
def test_schedule_properties(op, R, r, M, N, K, split, order):
    tile_n = 256 if N % 256 == 0 else 128
    info, tl, tk, tr = syn.schedule_build(op, R, r, M, N, K, split=split, order=order, tile_n=tile_n)
    M_r = M // R
    tiles_m, tiles_n = -(-M // 128), N // tile_n
    assert info["chunk_rows"] == -(-M_r // split) and info["n_row_chunks"] == R * split
    assert info["n_tiles"] == tiles_m * tiles_n
    # the tile list is a permutation of all tiles
    assert sorted(tl.tolist()) == list(range(tiles_m * tiles_n))
    # arrival order
    assert tr.tolist() == expected_transfers(op, R, r, split)
    arrival = {code: a for a, code in enumerate(tr.tolist())}
    # each tile's key is the latest arrival among the chunks it consumes;
    # RS send tiles (consume nothing) are negative and come in ring order
    for t, key in zip(tl.tolist(), tk.tolist()):
        tm = t // tiles_n
        d = deps(op, R, r, M, M_r, split, tm)
        if d:
            assert key == max(arrival[c] for c in d), (t, key, d)
        else:
            assert op == "rs" and key < 0
            block = (tm * 128) // M_r
            j = chunk_of(tm * 128, M_r, split) - block * split
            assert key == (((block - r) % R) - 1) * split + j - (R - 1) * split
    # the list is sorted by key (chunks walked in arrival order)
    assert (np.diff(tk) >= 0).all()
    # within a key group, the chosen traversal
    for key, grp in itertools.groupby(zip(tk.tolist(), tl.tolist()), key=lambda x: x[0]):
        ids = [t for _, t in grp]
        coords = [(t // tiles_n, t % tiles_n) for t in ids]
        if order == "row":
            want = sorted(coords)
        elif order == "col":
            want = sorted(coords, key=lambda c: (c[1], c[0]))
        else:
            want = sorted(coords, key=lambda c: (c[0] // 8, c[1], c[0] % 8))
        assert coords == want


def test_tiny_each_tile_depends_on_two_chunks():
    info, tl, tk, tr = syn.schedule_build("ag", 4, 0, 256, 256, 256, split=1)
    assert info["n_tiles"] == 2 and info["chunk_rows"] == 64
    for tm in range(2):
        assert len(deps("ag", 4, 0, 256, 64, 1, tm)) == 2


def test_rs_send_tiles_first_reduce_tiles_last():
    info, tl, tk, tr = syn.schedule_build("rs", 8, 2, 8192, 4096, 1792, split=2)
    tiles_n = 4096 // 256
    blocks = [(t // tiles_n) * 128 // 1024 for t in tl]
    n_local = (1024 // 128) * tiles_n
    assert all(b == 2 for b in blocks[-n_local:])
    assert all(b != 2 for b in blocks[:-n_local])
    first = [b for b in blocks[:-n_local]]
    # destinations in ring order 3, 4, ..., 1
    seen = [b for i, b in enumerate(first) if i == 0 or first[i - 1] != b]
    assert seen == [3, 4, 5, 6, 7, 0, 1]


@pytest.mark.parametrize("kw,status", [
    (dict(op="ag", R=4, rank=4, M=256, N=256, K=256), syn.ERR_INVALID),
    (dict(op="ag", R=3, rank=0, M=256, N=256, K=256), syn.ERR_INVALID),      # M % R
    (dict(op="ag", R=4, rank=0, M=256, N=256, K=100), syn.ERR_UNSUPPORTED),  # K % 8
    (dict(op="ag", R=4, rank=0, M=256, N=204, K=256), syn.ERR_UNSUPPORTED),  # N % 8
    (dict(op="rs", R=4, rank=0, M=1024, N=256, K=60), syn.ERR_UNSUPPORTED),  # K % 8
    (dict(op="ag", R=16, rank=0, M=256, N=256, K=256), syn.ERR_UNSUPPORTED),  # R > 8
    (dict(op="rs", R=4, rank=0, M=4 * 100, N=256, K=256), syn.ERR_UNSUPPORTED),  # M_r % 32
    (dict(op="ag", R=4, rank=0, M=256, N=256, K=256, split=65), syn.ERR_INVALID),  # split > M_r
    (dict(op="ag", R=4, rank=0, M=256, N=256, K=256, chunk_rows=32, split=4), syn.ERR_INVALID),
])
def test_invalid_shapes_rejected(kw, status):
    kw = dict(kw)
    args = [kw.pop(k) for k in ("op", "R", "rank", "M", "N", "K")]
    with pytest.raises(syn.SynError) as e:
        syn.schedule_build(*args, **kw)
    assert e.value.status == status


def test_k_and_n_tails_give_a_partial_last_tile_column():
    """K and N need only be multiples of 8: the last column of tiles covers the
    N tail (ceil(N / tile_n) tile columns), and the tile list still holds every
    tile once."""
    for N, tile_n in [(520, 256), (520, 128), (392, 256), (8, 128)]:
        info, tl, _, _ = syn.schedule_build("ag", 4, 1, 4 * 150, N, 200, split=2, order="row", tile_n=tile_n)
        tiles_n = -(-N // tile_n)
        assert info["tiles_n"] == tiles_n
        assert sorted(tl.tolist()) == list(range(info["tiles_m"] * tiles_n))


def test_chunk_rows_and_split_agree():
    a = syn.schedule_build("ag", 8, 0, 8192, 1792, 4096, chunk_rows=256, split=0)
    b = syn.schedule_build("ag", 8, 0, 8192, 1792, 4096, chunk_rows=0, split=4)
    assert a[0]["split"] == b[0]["split"] == 4
    assert (a[1] == b[1]).all() and (a[3] == b[3]).all()


def test_smem_peer_backend_has_no_transfers_and_reduce_tiles_first():
    """TMA_COLOCATED_SMEM fetches the resident peer partials tile by tile: there
    is nothing to stage, every peer chunk is available at t = 0, so GEMM-RS
    reduce tiles (which read peers) come first and GEMM-AR keeps pure traversal
    order."""
    info, tl, tk, tr = syn.schedule_build("rs", 8, 3, 8192, 4096, 1792, split=2, order="row",
                                          backend="tma_colocated_smem")
    assert info["n_transfers"] == 0 and len(tr) == 0
    tiles_n = 4096 // 256
    blocks = [(t // tiles_n) * 128 // 1024 for t in tl]
    n_local = (1024 // 128) * tiles_n
    assert all(b == 3 for b in blocks[:n_local]) and all(b != 3 for b in blocks[n_local:])
    info, tl, tk, tr = syn.schedule_build("ar", 8, 3, 4096, 3584, 2368, split=1, order="row",
                                          backend="tma_colocated_smem")
    assert info["n_transfers"] == 0 and tl.tolist() == list(range(info["n_tiles"]))


@pytest.mark.parametrize("op,R,r,M,N,K,split", [
    ("ag", 8, 0, 8192, 1792, 4096, 2), ("ag", 3, 1, 600, 512, 192, 1), ("rs", 8, 2, 8192, 4096, 1792, 4),
    ("ar", 8, 5, 4096, 3584, 2368, 3), ("ar", 2, 1, 666, 512, 128, 1)])
def test_pair_tiles_of_256_rows(op, R, r, M, N, K, split):
    """tile_m = 256 (a CTA pair per tile): same rules over 256-row tiles."""
    info, tl, tk, tr = syn.schedule_build(op, R, r, M, N, K, split=split, order="row", tile_m=256)
    M_r = M // R
    tiles_m, tiles_n = -(-M // 256), N // 256
    assert info["tile_m"] == 256 and info["n_tiles"] == tiles_m * tiles_n
    assert sorted(tl.tolist()) == list(range(tiles_m * tiles_n))
    arrival = {code: a for a, code in enumerate(tr.tolist())}
    for t, key in zip(tl.tolist(), tk.tolist()):
        tm = t // tiles_n
        d = deps(op, R, r, M, M_r, split, tm, tile_m=256)
        if d:
            assert key == max(arrival[c] for c in d)
        else:
            assert op == "rs" and key < 0
    assert (np.diff(tk) >= 0).all()


def test_rs_row_blocks_need_32_row_multiples():
    """GEMM-RS row blocks need not be whole tiles (a tile may straddle a block
    edge) but must be whole 32-row warp groups."""
    syn.schedule_build("rs", 4, 0, 4 * 384, 256, 256, tile_m=256)
    syn.schedule_build("rs", 4, 0, 4 * 96, 256, 256, tile_m=128)
    for tile_m in (128, 256):
        with pytest.raises(syn.SynError) as e:
            syn.schedule_build("rs", 4, 0, 4 * 368, 256, 256, tile_m=tile_m)
        assert e.value.status == syn.ERR_UNSUPPORTED


@pytest.mark.parametrize("R,r,M_r,tile_m,split,backend", [
    (4, 1, 96, 128, 1, "tma_colocated"),     # block 1 = rows 96..191: straddles tiles 0 and 1
    (4, 2, 96, 128, 3, "ce"),
    (4, 3, 160, 256, 2, "tma_colocated"),    # pair tiles, block 3 = rows 480..639, ragged last tile
    (3, 0, 32, 128, 1, "tma_colocated"),     # the whole row space is one tile
    (8, 5, 96, 256, 1, "tma_colocated_smem"),
])
def test_rs_straddling_tiles_reduce_and_wait_on_local_chunks(R, r, M_r, tile_m, split, backend):
    """A GEMM-RS tile reduces when any of its rows lie in the local block; it
    then waits only for (is keyed after) the local chunks its rows touch.
    Tiles with no local rows are send tiles, ordered before the reduce tiles
    when peers are staged.  Every tile appears once."""
    M, N, K = R * M_r, 256, 128
    info, tl, tk, tr = syn.schedule_build("rs", R, r, M, N, K, split=split, order="row", tile_m=tile_m,
                                          backend=backend)
    T = info["n_tiles"]
    assert sorted(tl.tolist()) == list(range(T))
    tiles_n = N // 256
    lo, hi = r * M_r, (r + 1) * M_r
    red = np.array([max(lo, (t // tiles_n) * tile_m) < min(hi, (t // tiles_n + 1) * tile_m) for t in tl])
    assert red.any()
    if backend == "tma_colocated_smem":
        assert len(tr) == 0
        assert red[:int(red.sum())].all()  # resident peers: reduce tiles first
        return
    # staged peers: send tiles first, then reduce tiles by their latest local chunk's arrival
    assert not red[:int((~red).sum())].any()
    arrival = {code: a for a, code in enumerate(tr.tolist())}
    bounds = [lo + (j * M_r + split - 1) // split for j in range(split + 1)]
    for t, k, is_red in zip(tl.tolist(), tk.tolist(), red.tolist()):
        if not is_red:
            continue
        a, b = max(lo, (t // tiles_n) * tile_m), min(hi, (t // tiles_n + 1) * tile_m)
        chunks = [r * split + j for j in range(split) if bounds[j] < b and bounds[j + 1] > a]
        want = max(arrival[rc * R + q] for rc in chunks for q in range(R) if q != r)
        assert k == want


@pytest.mark.parametrize("R,r,M,N,K,tile_m,tile_n,units", [
    (8, 3, 8192, 4096, 1792, 256, 256, 76),   # Llama-3-8B FFN down, CTA pairs
    (8, 0, 8192, 4096, 1792, 128, 256, 152),  # same, one CTA per tile
    (8, 5, 8192, 4096, 1792, 128, 128, 76),   # more reduce tiles than walkers
    (4, 1, 4096, 1024, 512, 128, 256, 16),
])
@pytest.mark.parametrize("reduce_warps", [0, -1])
def test_smem_rs_reduce_tiles_spread_over_walkers(R, r, M, N, K, tile_m, tile_n, units, reduce_warps):
    """With resident peer partials the GEMM-RS reduce tiles can go anywhere;
    reduce_spread = units lays them out one per walker where possible, in
    evenly filled rounds before each walker's last round (with reducer warps:
    the first half of those rounds), and keeps the send tiles' order in the
    other entries."""
    kw = dict(split=1, order="row", backend="tma_colocated_smem", tile_m=tile_m, tile_n=tile_n,
              reduce_warps=reduce_warps)
    _, tl0, tk0, _ = syn.schedule_build("rs", R, r, M, N, K, **kw)
    info, tl, tk, _ = syn.schedule_build("rs", R, r, M, N, K, reduce_spread=units, **kw)
    T = info["n_tiles"]
    assert sorted(tl.tolist()) == list(range(T))
    tiles_n = N // tile_n
    M_r = M // R
    is_red = np.array([(t // tiles_n) * tile_m // M_r == r for t in tl])
    is_red0 = np.array([(t // tiles_n) * tile_m // M_r == r for t in tl0])
    n_red = int(is_red.sum())
    assert is_red0[:n_red].all()                      # default: all first
    # send tiles: same relative order as before; keys travel with their tiles
    assert tl[~is_red].tolist() == tl0[n_red:].tolist()
    key_of = dict(zip(tl0.tolist(), tk0.tolist()))
    assert all(key_of[t] == k for t, k in zip(tl.tolist(), tk.tolist()))
    pos = np.nonzero(is_red)[0]
    rounds = T // units
    walker, rnd = pos % units, pos // units
    # never in a walker's last round
    last_round = np.array([(T - 1 - w) // units for w in range(units)])
    assert (rnd < last_round[walker]).all()
    if n_red <= units:
        assert len(set(walker.tolist())) == n_red      # one per walker
    early = reduce_warps == 0 and tile_n == 256
    use_rounds = max(1, (rounds - 1) // 2) if early else rounds - 1
    if n_red <= units * use_rounds:
        assert (rnd < use_rounds).all()
    counts = np.bincount(rnd, minlength=use_rounds)[:use_rounds]
    assert counts.max() - counts.min() <= 1 + n_red // units
    # the walkers with one tile fewer take the first reduce tiles
    short = list(range(T % units, units))
    if n_red >= len(short) and short:
        assert set(short) <= set(walker.tolist())


def test_smem_rs_spread_noop_for_short_walks():
    kw = dict(split=1, order="row", backend="tma_colocated_smem", tile_m=128, tile_n=256)
    _, tl0, _, _ = syn.schedule_build("rs", 4, 1, 1024, 512, 256, **kw)
    _, tl1, _, _ = syn.schedule_build("rs", 4, 1, 1024, 512, 256, reduce_spread=8, **kw)
    assert tl0.tolist() == tl1.tolist()  # 16 tiles over 8 walkers: 2 rounds only


# --------------------------------------------------------------------------- A2A-GEMM
# Row blocks of unequal size (rows_from[q] rows from source q, stacked in
# ascending q); each block cut into `split` chunks, chunk j of block q holding
# block rows [ceil(j*m/split), ceil((j+1)*m/split)).
def a2a_chunk_rows(rows_from, split):
    """Global [row0, row1) of every row chunk rc = q*split + j, by definition."""
    off = np.concatenate([[0], np.cumsum(rows_from)]).tolist()
    out = []
    for q, m in enumerate(rows_from):
        for j in range(split):
            out.append((off[q] + -(-j * m // split), off[q] + -(-(j + 1) * m // split)))
    return out


def a2a_deps(rows_from, split, tm, tile_m=128):
    R, M = len(rows_from), int(sum(rows_from))
    rows = set(range(tm * tile_m, min((tm + 1) * tile_m, M)))
    spans = a2a_chunk_rows(rows_from, split)
    rcs = [rc for rc, (a, b) in enumerate(spans) if rows & set(range(a, b))]
    return [rc * R + rc // split for rc in rcs]


A2A_CASES = [
    ([300, 0, 41, 1000], 1, 2, 256),
    ([300, 0, 41, 1000], 3, 0, 512),
    ([0, 0, 0, 128], 2, 1, 256),           # one source sends everything
    ([5, 7, 0, 1, 900, 64, 0, 33], 4, 6, 256),
    ([128, 128, 128, 128], 2, 3, 512),     # equal parts
    ([2, 3], 8, 1, 256),                   # blocks smaller than split: empty chunks
    ([4096, 1500, 2600, 0, 3000, 700, 2048, 512], 2, 4, 1024),
]


@pytest.mark.parametrize("rows_from,split,r,N", A2A_CASES)
@pytest.mark.parametrize("order", ["row", "grouped"])
def test_a2a_schedule_properties(rows_from, split, r, N, order):
    R, M, K = len(rows_from), int(sum(rows_from)), 128
    tile_n = 256
    info, tl, tk, tr = syn.schedule_build_a2a(R, r, rows_from, N, K, split=split, order=order, tile_n=tile_n)
    tiles_m, tiles_n = -(-M // 128), N // tile_n
    assert info["a2a"] == 1 and info["M"] == M and info["M_r"] == 0
    assert info["n_row_chunks"] == R * split and info["n_tiles"] == tiles_m * tiles_n
    assert info["chunk_rows"] == max(-(-m // split) for m in rows_from)
    assert sorted(tl.tolist()) == list(range(tiles_m * tiles_n))
    # the same arrival order as AG-GEMM: local block first, then r+1, r+2, ...
    assert tr.tolist() == expected_transfers("ag", R, r, split)
    arrival = {code: a for a, code in enumerate(tr.tolist())}
    for t, key in zip(tl.tolist(), tk.tolist()):
        d = a2a_deps(rows_from, split, t // tiles_n)
        assert d and key == max(arrival[c] for c in d), (t, key, d)
    assert (np.diff(tk) >= 0).all()


def test_a2a_equal_parts_is_the_ag_schedule():
    for r, split in [(0, 1), (3, 2), (5, 3)]:
        a = syn.schedule_build("ag", 8, r, 8192, 1792, 4096, split=split)
        b = syn.schedule_build_a2a(8, r, [1024] * 8, 1792, 4096, split=split)
        for x, y in zip(a[1:], b[1:]):
            assert (x == y).all()
        assert a[0]["chunk_rows"] == b[0]["chunk_rows"] and b[0]["a2a"] == 1


@pytest.mark.parametrize("rows_from,split,status", [
    ([4, -1, 3], 1, syn.ERR_INVALID),
    ([0, 0, 0], 1, syn.ERR_INVALID),         # nothing to multiply
    ([64, 64], 65, syn.ERR_INVALID),         # split > 64
    ([1] * 9, 1, syn.ERR_UNSUPPORTED),       # R > 8
])
def test_a2a_invalid_rejected(rows_from, split, status):
    with pytest.raises(syn.SynError) as e:
        syn.schedule_build_a2a(len(rows_from), 0, rows_from, 256, 128, split=split)
    assert e.value.status == status


# --------------------------------------------------------------------------- banded order
@pytest.mark.parametrize("kind,args,group_m", [
    ("a2a", ([300, 0, 41, 1000], 14336, 4096), 8),
    ("a2a", ([869, 895, 930, 901, 841, 876, 904, 883], 14336, 4096), 4),
    ("ag", (16384, 3584, 8192), 8),
    ("ag", (4 * 100, 256, 128), 3),
])
@pytest.mark.parametrize("r,split", [(0, 1), (2, 3)])
def test_banded_order(kind, args, group_m, r, split):
    """Bands of group_m tile rows: a band's key is the latest arrival any of
    its rows waits for; bands run in key order, each column by column."""
    if kind == "a2a":
        rows_from, N, K = args
        R = len(rows_from)
        if r >= R:
            pytest.skip("no such rank")
        info, tl, tk, tr = syn.schedule_build_a2a(R, r, rows_from, N, K, split=split, order="banded",
                                                  group_m=group_m)
        _, tl0, tk0, _ = syn.schedule_build_a2a(R, r, rows_from, N, K, split=split, order="row")
    else:
        M, N, K = args
        R = 8 if M > 1000 else 4
        info, tl, tk, tr = syn.schedule_build("ag", R, r, M, N, K, split=split, order="banded", group_m=group_m)
        _, tl0, tk0, _ = syn.schedule_build("ag", R, r, M, N, K, split=split, order="row")
    tiles_n = info["tiles_n"]
    row_key = {}
    for t, k in zip(tl0.tolist(), tk0.tolist()):
        row_key[t // tiles_n] = k        # the chunk key of each tile row (row order)
    band_key = {}
    for tm, k in row_key.items():
        b = tm // group_m
        band_key[b] = max(band_key.get(b, -1), k)
    assert sorted(tl.tolist()) == sorted(tl0.tolist())
    for t, k in zip(tl.tolist(), tk.tolist()):
        assert k == band_key[(t // tiles_n) // group_m]
    want = sorted(tl.tolist(), key=lambda t: (band_key[(t // tiles_n) // group_m], (t // tiles_n) // group_m,
                                               t % tiles_n, (t // tiles_n) % group_m))
    assert tl.tolist() == want


@pytest.mark.parametrize("op", ["rs", "ar"])
def test_banded_order_rejected_for_rs_ar(op):
    with pytest.raises(syn.SynError) as e:
        syn.schedule_build(op, 8, 0, 8192, 4096, 1792, order="banded")
    assert e.value.status == syn.ERR_UNSUPPORTED
