// schedule.cpp -- host-side chunk plan builder (no CUDA calls).
//
// Chunks (Syncopate summary page, method ¶1, paper §5.1): a chunk is a block
// of rows of a logical tensor holding one or more compute tiles.  Here every
// operator's row space [0, M) is cut into row chunks: each rank's block of
// rows (M/R rows, or for A2A-GEMM the rows that rank sends) into `split`
// chunks of near-equal size (RowBlocks in schedule.h); rank q owns row chunks
// [q*split, (q+1)*split).  A staging transfer is (row chunk rc,
// source rank q): the rows of rc held by rank q that the local rank needs.
//
//   AG-GEMM : transfer (rc, q = rc / split) copies shard q's rows into the
//             gathered buffer; tiles wait on every row chunk their rows touch.
//   GEMM-RS : transfers (rc, q) for rc in the local block and q != r copy peer
//             q's partial rows_r; only reduce tiles (local block) wait; send
//             tiles of other blocks produce chunks.
//   GEMM-AR : transfers (rc, q) for every rc and q != r; every tile waits on
//             its row chunks from all peers.
//
// Arrival order (method ¶1: ring plans): the local rank's data first, then a
// ring pull q = r+1, r+2, ..., r-1; chunk index ascending within a rank.  For
// GEMM-RS/AR, row chunks are the outer loop (local block first, then the ring
// of blocks) and peers the inner ring, so each row chunk completes early.
//
// Tile order (method ¶4, paper §5.2, Fig. 6): tiles are sorted by the latest
// arrival index among the chunks they consume, so the persistent grid walks
// chunks in arrival order; ties keep the chosen intra-chunk traversal.  GEMM-RS
// send tiles come first, ordered by destination ring position (Entwine
// abstract: produce data for communication at a regular pace).  With resident
// peer partials (TMA_COLOCATED_SMEM) nothing is awaited, and the GEMM-RS
// reduce tiles are spread over the walk instead (spread_reduce_tiles), so
// their peer reads overlap MMA work rather than arriving as one burst.
#include "schedule.h"

#include <algorithm>
#include <numeric>
#include <tuple>

namespace syn {

static int ring_pos(int q, int r, int R) { return ((q - r) % R + R) % R; }

// GEMM-RS: does tile row tm hold rows of the local block (so it reduces)?
static bool reduces_rows(const Schedule &s, int tm) {
    int64_t a, b;
    local_rows_of(s.M_r, s.rank, (int64_t)tm * s.tile_m, s.tile_m, a, b);
    return a < b;
}

int build_schedule(syn_op_t op, int R, int rank, const syn_layout_t &L,
                   int64_t chunk_rows, int split, syn_order_t order,
                   const syn_knobs_t &kn, Schedule &s, std::string &err, const int64_t *block_rows) {
    if (op != SYN_OP_AG_GEMM && op != SYN_OP_GEMM_RS && op != SYN_OP_GEMM_AR) {
        err = "unknown op";
        return SYN_ERR_INVALID;
    }
    if (R < 1 || rank < 0 || rank >= R) {
        err = "need 1 <= R and 0 <= rank < R";
        return SYN_ERR_INVALID;
    }
    if (R > kMaxRanks) {
        err = "R > 8 is not supported";
        return SYN_ERR_UNSUPPORTED;
    }
    if (L.M <= 0 || L.N <= 0 || L.K <= 0) {
        err = "M, N, K must be positive";
        return SYN_ERR_INVALID;
    }
    const bool var_blocks = block_rows != nullptr;
    if (var_blocks) {
        if (op != SYN_OP_AG_GEMM) {
            err = "per-rank block sizes are for the A2A-GEMM (AG-GEMM) plan only";
            return SYN_ERR_INVALID;
        }
        int64_t sum = 0;
        for (int q = 0; q < R; ++q) {
            if (block_rows[q] < 0) {
                err = "block sizes must be >= 0";
                return SYN_ERR_INVALID;
            }
            sum += block_rows[q];
        }
        if (sum != L.M) {
            err = "M must equal the sum of the block sizes";
            return SYN_ERR_INVALID;
        }
    } else if (L.M % R != 0) {
        err = "M must be divisible by R";
        return SYN_ERR_INVALID;
    }
    if ((L.lda != 0 && L.lda != L.K) || (L.ldb != 0 && L.ldb != L.N) ||
        (L.ldc != 0 && L.ldc != L.N)) {
        err = "only dense row-major layouts are supported";
        return SYN_ERR_UNSUPPORTED;
    }
    if (order < SYN_ORDER_ROW_MAJOR || order > SYN_ORDER_BANDED) {
        err = "unknown tile order";
        return SYN_ERR_INVALID;
    }
    if (order == SYN_ORDER_BANDED && op != SYN_OP_AG_GEMM) {
        err = "the banded tile order is for AG-GEMM and A2A-GEMM";
        return SYN_ERR_UNSUPPORTED;
    }
    const int64_t M_r = var_blocks ? 0 : L.M / R;
    if (chunk_rows < 0 || split < 0) {
        err = "chunk_rows and split must be >= 0";
        return SYN_ERR_INVALID;
    }
    if (var_blocks && chunk_rows != 0) {
        err = "per-rank block sizes take a split, not chunk_rows";
        return SYN_ERR_INVALID;
    }
    if (chunk_rows == 0 && split == 0) split = 1;
    if (chunk_rows > 0 && split > 0 && chunk_rows * split != M_r) {
        err = "chunk_rows * split must equal M/R";
        return SYN_ERR_INVALID;
    }
    if (chunk_rows > 0 && split == 0) {
        if (M_r % chunk_rows != 0) {
            err = "chunk_rows must divide M/R";
            return SYN_ERR_INVALID;
        }
        split = (int)(M_r / chunk_rows);
    }
    if (!var_blocks && split > M_r) {
        err = "split must not exceed M/R";
        return SYN_ERR_INVALID;
    }
    if (var_blocks && split > 64) {
        err = "split must not exceed 64";
        return SYN_ERR_INVALID;
    }
    const int tile_m = kn.tile_m == 0 ? kTileM : kn.tile_m;
    const int tile_n = kn.tile_n == 0 ? 256 : kn.tile_n;
    if (tile_m != kTileM && tile_m != 2 * kTileM) {
        err = "tile_m must be 128 (one CTA per tile) or 256 (a CTA pair per tile)";
        return SYN_ERR_UNSUPPORTED;
    }
    if (tile_n != 128 && tile_n != 256) {
        err = "tile_n must be 128 or 256";
        return SYN_ERR_UNSUPPORTED;
    }
    // Tails: the last k-block and the last column of tiles may be partial (the
    // TMA loads fill past K and N with zeros, the stores stop at N); rows of
    // bf16 operands and fp32 partials must start on 16-byte boundaries.
    if (L.K % 8 != 0) {
        err = "K must be a multiple of 8 (16-byte bf16 rows)";
        return SYN_ERR_UNSUPPORTED;
    }
    if (L.N % 8 != 0) {
        err = "N must be a multiple of 8 (16-byte bf16 rows)";
        return SYN_ERR_UNSUPPORTED;
    }
    if (op == SYN_OP_GEMM_RS && M_r % 32 != 0) {
        // (a warp's 32 epilogue rows are either all sent or all reduced)
        err = "GEMM-RS needs (M/R) % 32 == 0";
        return SYN_ERR_UNSUPPORTED;
    }
    if (L.M > (int64_t)1 << 30 || L.N > (int64_t)1 << 30 || L.K > (int64_t)1 << 30) {
        err = "dimension too large";
        return SYN_ERR_UNSUPPORTED;
    }

    s = Schedule();
    s.op = op;
    s.R = R;
    s.rank = rank;
    s.M = L.M;
    s.N = L.N;
    s.K = L.K;
    s.M_r = M_r;
    s.split = split;
    if (var_blocks) {
        s.rb.R = R;
        s.rb.split = split;
        s.rb.off[0] = 0;
        for (int q = 0; q < kMaxRanks; ++q) s.rb.off[q + 1] = s.rb.off[q] + (q < R ? block_rows[q] : 0);
        s.cr = 0;
        for (int q = 0; q < R; ++q) {
            const int64_t c = (block_rows[q] + split - 1) / split;
            if (c > s.cr) s.cr = c;
        }
    } else {
        s.rb = uniform_blocks(R, M_r, split);
        s.cr = (M_r + split - 1) / split;
    }
    s.order = order;
    s.group_m = kn.group_m > 0 ? kn.group_m : 8;
    s.tile_m = tile_m;
    s.tile_n = tile_n;
    s.tiles_m = (int)((L.M + tile_m - 1) / tile_m);
    s.tiles_n = (int)((L.N + tile_n - 1) / tile_n);
    s.n_tiles = s.tiles_m * s.tiles_n;
    s.n_rc = R * split;

    // ---- staging transfers in arrival order -----------------------------
    s.arrival.assign((size_t)s.n_rc * R, -1);
    auto add = [&](int rc, int q) {
        s.arrival[(size_t)rc * R + q] = (int)s.transfers.size();
        s.transfers.push_back(rc * R + q);
    };
    if (op == SYN_OP_AG_GEMM) {
        for (int d = 0; d < R; ++d) {
            const int q = (rank + d) % R;
            for (int j = 0; j < split; ++j) add(q * split + j, q);
        }
    } else if (kn.backend != SYN_BACKEND_TMA_COLOCATED_SMEM) {
        // (TMA_COLOCATED_SMEM fetches resident peer partials per tile: no transfers)
        const int nblocks = (op == SYN_OP_GEMM_RS) ? 1 : R;  // RS: only the local block
        for (int db = 0; db < nblocks; ++db) {
            const int b = (rank + db) % R;
            for (int j = 0; j < split; ++j)
                for (int dq = 1; dq < R; ++dq) add(b * split + j, (rank + dq) % R);
        }
    }

    // ---- tile keys from the chunk -> tile dependency ranges ---------------
    struct Item {
        int32_t key;
        int64_t t0, t1, t2;
        int32_t tile;
    };
    std::vector<int32_t> row_key((size_t)s.tiles_m, -1);
    for (int tm = 0; tm < s.tiles_m; ++tm) {
        int lo, hi;
        tile_row_chunks(s, tm, lo, hi);
        int32_t key = -1;
        const int block = block_of_row(s.rb, (int64_t)tm * tile_m);
        if (op == SYN_OP_GEMM_RS && !reduces_rows(s, tm)) {
            // send tile: produces chunk(s) for rank `block`; ring order
            const int j = chunk_of_row(s.rb, (int64_t)tm * tile_m) - block * split;
            key = (ring_pos(block, rank, R) - 1) * split + j - (R - 1) * split;
        } else if (op == SYN_OP_GEMM_RS && kn.backend == SYN_BACKEND_TMA_COLOCATED_SMEM) {
            // the peers' rows_r are resident from the start: reduce tiles first
            key = -(R - 1) * split - 1;
        } else {
            for (int rc = lo; rc <= hi; ++rc)
                for (int q = 0; q < R && !chunk_empty(s.rb, rc); ++q) {
                    const int a = s.arrival[(size_t)rc * R + q];
                    if (a > key) key = a;
                }
        }
        row_key[(size_t)tm] = key;
    }
    if (order == SYN_ORDER_BANDED)  // a band waits for the latest chunk of any of its rows
        for (int b0 = 0; b0 < s.tiles_m; b0 += s.group_m) {
            const int b1 = std::min(s.tiles_m, b0 + s.group_m);
            const int32_t k = *std::max_element(row_key.begin() + b0, row_key.begin() + b1);
            std::fill(row_key.begin() + b0, row_key.begin() + b1, k);
        }
    std::vector<Item> items;
    items.reserve(s.n_tiles);
    for (int tm = 0; tm < s.tiles_m; ++tm) {
        for (int tn = 0; tn < s.tiles_n; ++tn) {
            Item it;
            it.key = row_key[(size_t)tm];
            it.tile = tm * s.tiles_n + tn;
            switch (order) {
                case SYN_ORDER_ROW_MAJOR:
                    it.t0 = tm, it.t1 = tn, it.t2 = 0;
                    break;
                case SYN_ORDER_COL_MAJOR:
                    it.t0 = tn, it.t1 = tm, it.t2 = 0;
                    break;
                default:
                    it.t0 = tm / s.group_m, it.t1 = tn, it.t2 = tm % s.group_m;
                    break;
            }
            items.push_back(it);
        }
    }
    std::stable_sort(items.begin(), items.end(), [](const Item &a, const Item &b) {
        return std::tie(a.key, a.t0, a.t1, a.t2) < std::tie(b.key, b.t0, b.t1, b.t2);
    });
    s.tile_list.resize(items.size());
    s.tile_key.resize(items.size());
    for (size_t i = 0; i < items.size(); ++i) {
        s.tile_list[i] = items[i].tile;
        s.tile_key[i] = items[i].key;
    }
    if (op == SYN_OP_GEMM_RS && kn.backend == SYN_BACKEND_TMA_COLOCATED_SMEM && kn.reduce_spread > 0)
        spread_reduce_tiles(s, kn.reduce_spread, uses_reducer_warps(op, kn, tile_n));
    return SYN_OK;
}

void spread_reduce_tiles(Schedule &s, int units, bool early) {
    const int T = (int)s.tile_list.size();
    if (units <= 0 || T == 0) return;
    const int rounds = T / units;  // full rounds of the walk
    if (rounds < 3) return;
    std::vector<int32_t> red, red_key, snd, snd_key;
    for (int i = 0; i < T; ++i) {
        const bool is_red = reduces_rows(s, s.tile_list[i] / s.tiles_n);
        (is_red ? red : snd).push_back(s.tile_list[i]);
        (is_red ? red_key : snd_key).push_back(s.tile_key[i]);
    }
    const int n_red = (int)red.size();
    if (n_red == 0) return;
    // Walkers [T mod units, units) run one tile fewer (no entry in the partial
    // last round): they take the first reduce tiles.  A walker's last tile is
    // in round rounds - 1 or rounds, so reduce tiles use rounds [0, rounds - 2]
    // (early: the first half of those).
    const int first_unit = T % units;
    const int use_rounds = early ? std::max(1, (rounds - 1) / 2) : rounds - 1;
    std::vector<int32_t> pos_tile(T, -1), pos_key(T, 0);
    std::vector<char> taken(T, 0);
    for (int j = 0; j < n_red; ++j) {
        const int u = (first_unit + j) % units;
        const int rho = (int)(((int64_t)j * use_rounds) / n_red);
        int pos = rho * units + u;
        // with more reduce tiles than walkers a walker's later reduce tile may
        // land on a taken entry: take the walker's next free round, else any
        // free entry before the last round
        while (pos < use_rounds * units && taken[pos]) pos += units;
        if (pos >= use_rounds * units) {
            pos = 0;
            while (taken[pos]) ++pos;
        }
        taken[pos] = 1;
        pos_tile[pos] = red[j];
        pos_key[pos] = red_key[j];
    }
    size_t k = 0;
    for (int i = 0; i < T; ++i) {
        if (taken[i]) {
            s.tile_list[i] = pos_tile[i];
            s.tile_key[i] = pos_key[i];
        } else {
            s.tile_list[i] = snd[k];
            s.tile_key[i] = snd_key[k];
            ++k;
        }
    }
}

}  // namespace syn
