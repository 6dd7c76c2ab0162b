// schedule.h -- host-side chunk plan: chunk partition, chunk->tile dependency
// ranges, arrival order of staging transfers and the rewritten tile order.
//
// Syncopate summary page, method ¶2 (the chunk-tile dependency graph: which
// chunks each tile consumes or produces, and where waits go) and ¶4 (paper
// §5.2, Fig. 6: order chunks by communication order, then keep or adjust the
// tile traversal inside a chunk).  The producer-side order of GEMM-RS (send
// tiles first) follows Entwine's abstract: produce data for communication at a
// regular pace.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "syn.h"

#if defined(__CUDACC__)
#define SYN_SCHED_HD __host__ __device__ __forceinline__
#else
#define SYN_SCHED_HD inline
#endif

namespace syn {

constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int kMaxRanks = 8;

// Row blocks of the R ranks: rank q owns rows [off[q], off[q+1]) of the row
// space.  AG-GEMM, GEMM-RS and GEMM-AR use uniform blocks, off[q] = q * M / R;
// A2A-GEMM has one block per source rank with its own size (the rows that
// rank sends).  Block q (of m_q = off[q+1] - off[q] rows) is cut into `split`
// chunks: chunk j covers rows off[q] + [ceil(j*m_q/split), ceil((j+1)*m_q/split)),
// so chunk sizes within a block differ by at most one row.  Row chunk
// rc = q*split + j.
struct RowBlocks {
    int R = 1, split = 1;
    int64_t off[kMaxRanks + 1] = {0};
};

SYN_SCHED_HD RowBlocks uniform_blocks(int R, int64_t M_r, int split) {
    RowBlocks b;
    b.R = R;
    b.split = split;
    for (int q = 0; q <= kMaxRanks; ++q) b.off[q] = (int64_t)(q <= R ? q : R) * M_r;
    return b;
}
SYN_SCHED_HD int64_t block_rows(const RowBlocks &b, int q) { return b.off[q + 1] - b.off[q]; }

// GEMM-RS: the rows [a, b) of rows [r0, r0 + nrows) that lie in block `rank`
// (rows [rank * M_r, (rank + 1) * M_r)), the ones a tile reduces with the
// peers' partials; empty (a >= b) for a tile that only sends.  A tile may
// straddle the block's edges when M_r is not a multiple of the tile height.
SYN_SCHED_HD void local_rows_of(int64_t M_r, int rank, int64_t r0, int64_t nrows, int64_t &a, int64_t &b) {
    const int64_t lo = (int64_t)rank * M_r, hi = lo + M_r;
    a = r0 > lo ? r0 : lo;
    b = r0 + nrows < hi ? r0 + nrows : hi;
}

// First row of row chunk rc (rc == R*split gives the end of the row space).
SYN_SCHED_HD int64_t chunk_row0(const RowBlocks &b, int rc) {
    const int q = rc / b.split, j = rc - q * b.split;
    if (q >= b.R) return b.off[b.R];
    const int64_t m = block_rows(b, q);
    return b.off[q] + ((int64_t)j * m + b.split - 1) / b.split;
}
// Row chunk rc holds no rows (A2A-GEMM: an empty block, or a block of fewer
// rows than split).  Its transfer still publishes a flag, but no tile waits
// for it.
SYN_SCHED_HD bool chunk_empty(const RowBlocks &b, int rc) { return chunk_row0(b, rc + 1) == chunk_row0(b, rc); }
// The rank whose block holds `row` (0 <= row < off[R]); empty blocks hold none.
SYN_SCHED_HD int block_of_row(const RowBlocks &b, int64_t row) {
    int q = 0;
    while (q + 1 < b.R && b.off[q + 1] <= row) ++q;
    return q;
}
SYN_SCHED_HD int chunk_of_row(const RowBlocks &b, int64_t row) {
    const int q = block_of_row(b, row);
    const int64_t m = block_rows(b, q);
    return q * b.split + (int)(((row - b.off[q]) * b.split) / m);
}

struct Schedule {
    int op = 0, R = 1, rank = 0;
    int64_t M = 0, N = 0, K = 0, M_r = 0;  // M_r: rows per rank (uniform blocks; 0 for A2A)
    int64_t cr = 0;      // rows of the largest chunk
    int split = 1;       // chunks per rank row block
    RowBlocks rb;        // row blocks and chunk geometry
    int order = 0, group_m = 8;
    int tile_m = kTileM, tile_n = 256;
    int tiles_m = 0, tiles_n = 0, n_tiles = 0;
    int n_rc = 0;        // row chunks over [0, M)
    std::vector<int32_t> tile_list;   // execution order (tile ids)
    std::vector<int32_t> tile_key;    // sort key of each entry of tile_list
    std::vector<int32_t> transfers;   // rc * R + q, arrival order
    std::vector<int32_t> arrival;     // arrival index of (rc * R + q), -1 if none
};

// Fills `s` or returns a SYN_ERR_* code with a message in `err`.  With
// `block_rows` (AG-GEMM only: A2A-GEMM) rank q's block has block_rows[q] rows
// and layout.M must be their sum; otherwise blocks are uniform, M / R rows.
int build_schedule(syn_op_t op, int R, int rank, const syn_layout_t &layout,
                   int64_t chunk_rows, int split, syn_order_t order,
                   const syn_knobs_t &knobs, Schedule &s, std::string &err,
                   const int64_t *block_rows = nullptr);

// GEMM-RS whose peer partials are resident (TMA_COLOCATED_SMEM): every chunk
// is available at t = 0, so the order is free to place the reduce tiles (each
// streams R-1 peer tiles through its epilogue) where their reads overlap the
// most MMA work.  This moves them from the head of the order into evenly
// spaced rounds of the walk by `units` persistent tile walkers (walker u runs
// entries u, u + units, ...), one walker each where there are enough walkers,
// never in the last round a walker runs; the send tiles keep their order in
// the remaining entries.  No-op when the walk has fewer than three rounds.
// `early`: with reducer warps the walker's epilogue is short and the reducer
// streams the peers afterwards, so the reduce tiles go into the first half of
// the rounds, leaving the reducers the rest of the walk to finish.
void spread_reduce_tiles(Schedule &s, int units, bool early);

// Whether a GEMM-RS/AR plan reduces resident peers with reducer warps (the
// default for TMA_COLOCATED_SMEM at tile_n 256, tile_k 64).
inline bool uses_reducer_warps(int op, const syn_knobs_t &kn, int tile_n) {
    return op != SYN_OP_AG_GEMM && kn.backend == SYN_BACKEND_TMA_COLOCATED_SMEM &&
           kn.reduce_warps >= 0 && tile_n == 256 && (kn.tile_k == 0 || kn.tile_k == 64);
}

// Row-chunk range [lo, hi] covered by tile row tm (rows clipped to M).
inline void tile_row_chunks(const Schedule &s, int tm, int &lo, int &hi) {
    int64_t r0 = (int64_t)tm * s.tile_m;
    int64_t r1 = r0 + s.tile_m;
    if (r1 > s.M) r1 = s.M;
    lo = chunk_of_row(s.rb, r0);
    hi = chunk_of_row(s.rb, r1 - 1);
}

}  // namespace syn
