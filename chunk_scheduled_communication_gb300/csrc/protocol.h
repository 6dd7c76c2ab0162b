// protocol.h -- the pure logic of the chunk ready-flag protocol, shared by the
// fused kernel (device) and the CPU emulation of the protocol (host threads).
//
// Syncopate summary page, method ¶2 (tiles wait only on the chunks they
// consume) and ¶3 (stagers publish a chunk once its bytes have landed):
//   - every staging transfer (row chunk, source rank) has a ready flag that
//     carries the epoch (call number) of the call that published it, so a
//     flag left over from an earlier or aborted call never satisfies a wait;
//   - a transfer is copied in slices by several stagers; each adds one to the
//     transfer's slice counter and the stager that completes the last slice
//     publishes the flag (release after its own copy has landed);
//   - slice counters are double-buffered by epoch parity: a call counts in
//     half (epoch & 1) and clears the other half for the next call, so no
//     reset is needed between calls;
//   - persistent walker u of n runs tile-list entries u, u + n, u + 2n, ...
#pragma once

#include <cstdint>

#include "schedule.h"

namespace syn {

// Ready test of an epoch flag (wrap-around safe).
SYN_SCHED_HD bool flag_ready(uint32_t flag, uint32_t epoch) { return (int32_t)(flag - epoch) >= 0; }

// Half of the double-buffered slice / producer counters a call counts in, and
// the half it clears for the next call.
SYN_SCHED_HD uint32_t counter_half(uint32_t epoch) { return epoch & 1u; }
SYN_SCHED_HD uint32_t spare_half(uint32_t epoch) { return (epoch + 1u) & 1u; }

// Given the counter value before this stager's increment, does its slice
// complete the transfer (so it publishes the flag)?
SYN_SCHED_HD bool completes_transfer(uint32_t old_count, uint32_t slices_per_transfer) {
    return old_count + 1u == slices_per_transfer;
}

// Tile-list entry i of walker `unit` of `n_units`, or -1 past the walk.
SYN_SCHED_HD int walk_entry_of(int t_begin, int t_end, int unit, int n_units, int i) {
    const int t = t_begin + unit + i * n_units;
    return t < t_end ? t : -1;
}

// Row chunks [lo, hi] that rows [r0, r0 + nrows) clipped to M touch; lo > hi
// when every row lies past M.
SYN_SCHED_HD void chunk_range_of(int64_t M, const RowBlocks &b, int64_t r0, int64_t nrows, int &lo, int &hi) {
    const int64_t r1 = r0 + nrows < M ? r0 + nrows : M;
    if (r0 >= r1) {
        lo = 0;
        hi = -1;
        return;
    }
    lo = chunk_of_row(b, r0);
    hi = chunk_of_row(b, r1 - 1);
}

// Receive-buffer slot of source rank q (the local rank has none).
SYN_SCHED_HD int recv_slot_of(int q, int rank) { return q - (q > rank ? 1 : 0); }

// Rows of staging transfer `code` = rc * R + q (row chunk rc, from source
// rank q): `rows` rows from row `src_row` of source q's buffer to row
// `dst_row` of the destination (op 0 AG / A2A: the gathered buffer; op 1 RS /
// 2 AR: the receive buffer, source q's slot at rows [slot * slot_rows, ...)).
//   AG : shard q rows [row0 - off[q], ...)  ->  gathered rows [row0, row1)
//   RS : peer q rows [row0, row1)            ->  slot q rows [row0 - off[rank], ...)
//   AR : peer q rows [row0, row1)            ->  slot q rows [row0, row1)
struct TransferRows {
    int q;
    int64_t src_row, dst_row, rows;
};
SYN_SCHED_HD TransferRows transfer_rows(int op, int rank, const RowBlocks &b, int64_t slot_rows, int code) {
    const int rc = code / b.R, q = code % b.R;
    const int64_t row0 = chunk_row0(b, rc);
    const int64_t row1 = chunk_row0(b, rc + 1);
    TransferRows t;
    t.q = q;
    t.rows = row1 - row0;
    if (op == 0) {
        t.src_row = row0 - b.off[q];
        t.dst_row = row0;
    } else {
        t.src_row = row0;
        t.dst_row = (int64_t)recv_slot_of(q, rank) * slot_rows + row0 - (op == 1 ? b.off[rank] : 0);
    }
    return t;
}

}  // namespace syn
