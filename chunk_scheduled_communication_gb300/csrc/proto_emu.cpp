// proto_emu.cpp -- CPU emulation of the chunk ready-flag protocol (see
// include/syn_proto.h).  Host threads stand in for the GPU's staging workers
// and persistent tile walkers; everything they decide comes from the plan
// builder (schedule.cpp) and the protocol's shared logic (protocol.h), the
// same code the fused kernel runs.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstring>
#include <random>
#include <string>
#include <thread>
#include <vector>

#include "protocol.h"
#include "schedule.h"
#include "syn.h"
#include "syn_proto.h"

using namespace syn;

namespace {

thread_local std::string g_err;

using Clock = std::chrono::steady_clock;

// Byte b of row `row` of source q in call `epoch`: differs between calls, so
// a consumer that proceeds on a stale flag reads the wrong bytes.
inline uint8_t src_byte(uint32_t epoch, int q, int64_t row, int64_t b, uint64_t seed) {
    uint64_t x = seed ^ (0x9E3779B97F4A7C15ull * (epoch + 1)) ^ ((uint64_t)q << 56) ^ ((uint64_t)row << 20) ^
                 (uint64_t)b;
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdull;
    x ^= x >> 33;
    return (uint8_t)x;
}

struct State {
    const syn_proto_cfg_t *cfg;
    Schedule s;
    int64_t row_bytes = 0, slot_rows = 0;
    bool local_inplace = true;
    std::vector<std::vector<uint8_t>> src;   // R sources (AG shards [M_r] rows, A2A parts; RS/AR peers [M] rows)
    std::vector<uint8_t> dst;                // AG gathered [M] rows; RS/AR receive buffer
    std::vector<std::atomic<uint32_t>> flags;
    std::vector<std::atomic<uint32_t>> cnt;  // [2][n_flags]
    std::atomic<int> err{0};
    std::atomic<int64_t> checked{0};
};

// Bounded acquire-wait for a flag of this epoch; on expiry the call fails.
bool wait_ready(State &st, int code, uint32_t epoch) {
    const auto t0 = Clock::now();
    for (;;) {
        if (flag_ready(st.flags[code].load(std::memory_order_acquire), epoch)) return true;
        if (st.err.load(std::memory_order_relaxed) != 0) return false;
        if (Clock::now() - t0 > std::chrono::microseconds(st.cfg->timeout_us)) {
            int expect = 0;
            st.err.compare_exchange_strong(expect, SYN_ERR_TIMEOUT);
            return false;
        }
        std::this_thread::yield();
    }
}

void stager(State &st, int worker, uint32_t epoch, int call) {
    const syn_proto_cfg_t &c = *st.cfg;
    const int n_tr = (int)st.s.transfers.size();
    const int64_t max_rows = st.s.cr;  // largest transfer, in rows
    const int spt = (int)((max_rows * st.row_bytes + c.slice_bytes - 1) / c.slice_bytes);
    const int n_flags = st.s.n_rc * st.s.R;
    std::mt19937_64 rng(c.seed * 7919u + (uint64_t)worker * 104729u + epoch);
    for (int g = worker; g < n_tr * spt; g += c.stagers) {
        if (st.err.load(std::memory_order_relaxed) != 0) return;
        const int a = g / spt, sl = g % spt;
        const int code = st.s.transfers[a];
        if (c.op == 0 && st.local_inplace && code % st.s.R == st.s.rank) continue;
        if (c.jitter_us > 0) std::this_thread::sleep_for(std::chrono::microseconds(rng() % (c.jitter_us + 1)));
        const TransferRows t = transfer_rows(c.op, st.s.rank, st.s.rb, st.slot_rows, code);
        const int64_t bytes = t.rows * st.row_bytes;
        const int64_t off = (int64_t)sl * c.slice_bytes;
        const int64_t len = std::min<int64_t>(c.slice_bytes, bytes - off);
        auto copy = [&]() {
            if (len > 0)
                std::memcpy(st.dst.data() + t.dst_row * st.row_bytes + off,
                            st.src[t.q].data() + t.src_row * st.row_bytes + off, (size_t)len);
        };
        if (c.mutation != 1) copy();
        const uint32_t old = st.cnt[(size_t)counter_half(epoch) * n_flags + code].fetch_add(
            1u, std::memory_order_acq_rel);
        const bool last = completes_transfer(old, (uint32_t)spt);
        if (last && !(a == c.drop_transfer && call == c.drop_call)) {
            if (a == c.delay_transfer) std::this_thread::sleep_for(std::chrono::microseconds(c.delay_us));
            st.flags[code].store(epoch, std::memory_order_release);
        }
        if (c.mutation == 1) {  // broken on purpose: the bytes land after the flag
            if (last) std::this_thread::sleep_for(std::chrono::milliseconds(2));
            copy();
        }
    }
}

// The chunks a tile waits on (as the kernel's producer / peer loader does).
void tile_waits(const State &st, int tile, std::vector<int> &codes) {
    const Schedule &s = st.s;
    const int op = st.cfg->op;
    codes.clear();
    int64_t r0 = (int64_t)(tile / s.tiles_n) * s.tile_m, nrows = s.tile_m;
    if (op == 1) {  // GEMM-RS: only the rows of the local block consume chunks
        int64_t a, b;
        local_rows_of(s.M_r, s.rank, r0, nrows, a, b);
        if (a >= b) return;  // a send tile: consumes nothing
        r0 = a;
        nrows = b - a;
    }
    int lo, hi;
    chunk_range_of(s.M, s.rb, r0, nrows, lo, hi);
    for (int rc = lo; rc <= hi; ++rc) {
        if (op == 0) {
            const int q = rc / s.split;
            if (!(st.local_inplace && q == s.rank) && !chunk_empty(s.rb, rc)) codes.push_back(rc * s.R + q);
        } else {
            for (int q = 0; q < s.R; ++q)
                if (q != s.rank) codes.push_back(rc * s.R + q);
        }
    }
}

// Every destination row of the tile's transfers must hold this call's bytes.
bool rows_match(const State &st, int code, uint32_t epoch) {
    const TransferRows t = transfer_rows(st.cfg->op, st.s.rank, st.s.rb, st.slot_rows, code);
    for (int64_t r = 0; r < t.rows; ++r) {
        const uint8_t *d = st.dst.data() + (t.dst_row + r) * st.row_bytes;
        for (int64_t b = 0; b < st.row_bytes; ++b)
            if (d[b] != src_byte(epoch, t.q, t.src_row + r, b, st.cfg->seed)) return false;
    }
    return true;
}

void walker(State &st, int unit, uint32_t epoch) {
    const syn_proto_cfg_t &c = *st.cfg;
    const int n_flags = st.s.n_rc * st.s.R;
    if (unit == 0)  // "CTA 0" clears the spare half of the counters
        for (int i = 0; i < n_flags; ++i)
            st.cnt[(size_t)spare_half(epoch) * n_flags + i].store(0u, std::memory_order_relaxed);
    std::vector<int> codes;
    for (int i = 0;; ++i) {
        const int t = walk_entry_of(0, st.s.n_tiles, unit, c.walkers, i);
        if (t < 0) return;
        tile_waits(st, st.s.tile_list[t], codes);
        for (int code : codes)
            if (!wait_ready(st, code, epoch)) return;
        for (int code : codes)
            if (!rows_match(st, code, epoch)) {
                int expect = 0;
                st.err.compare_exchange_strong(expect, SYN_PROTO_STALE_DATA);
                return;
            }
        st.checked.fetch_add(1, std::memory_order_relaxed);
    }
}

}  // namespace

extern "C" const char *syn_proto_last_error(void) { return g_err.c_str(); }

extern "C" int syn_proto_emulate(const syn_proto_cfg_t *cfg, int *status, int64_t *tiles_checked) {
    if (cfg == nullptr || status == nullptr) {
        g_err = "null argument";
        return SYN_ERR_INVALID;
    }
    const syn_proto_cfg_t &c = *cfg;
    if (c.op < 0 || c.op > 2 || c.walkers < 1 || c.stagers < 1 || c.slice_bytes < 16 || c.calls < 1 ||
        c.timeout_us < 1) {
        g_err = "invalid emulation parameters";
        return SYN_ERR_INVALID;
    }
    State st;
    st.cfg = cfg;
    if (c.rows_from != nullptr && (c.op != 0 || c.R < 1 || c.R > kMaxRanks)) {
        g_err = "rows_from is for op 0 with 1 <= R <= 8";
        return SYN_ERR_INVALID;
    }
    int64_t M = c.M;
    if (c.rows_from != nullptr) {
        M = 0;
        for (int q = 0; q < c.R; ++q) M += c.rows_from[q];
    }
    syn_layout_t L = {M, c.N, c.K, 0, 0, 0};
    syn_knobs_t kn;
    std::memset(&kn, 0, sizeof(kn));
    kn.backend = SYN_BACKEND_TMA_COLOCATED;
    kn.tile_m = c.tile_m;
    kn.tile_n = c.tile_n;
    kn.group_m = 8;
    kn.slice_kb = 128;
    std::string err;
    const int rc = build_schedule((syn_op_t)c.op, c.R, c.rank, L, 0, c.split, (syn_order_t)c.order, kn, st.s, err,
                                  c.rows_from);
    if (rc != SYN_OK) {
        g_err = err;
        return rc;
    }
    const Schedule &s = st.s;
    st.row_bytes = c.op == 0 ? c.K * 2 : c.N * 4;
    st.slot_rows = c.op == 1 ? s.M_r : s.M;
    auto src_rows = [&](int q) { return c.op == 0 ? block_rows(s.rb, q) : s.M; };
    st.src.resize((size_t)s.R);
    for (int q = 0; q < s.R; ++q) st.src[q].assign((size_t)(src_rows(q) * st.row_bytes), 0);
    st.dst.assign((size_t)((c.op == 0 ? s.M : (int64_t)(s.R - 1) * st.slot_rows) * st.row_bytes), 0);
    const int n_flags = s.n_rc * s.R;
    st.flags = std::vector<std::atomic<uint32_t>>((size_t)n_flags);
    st.cnt = std::vector<std::atomic<uint32_t>>((size_t)2 * n_flags);
    for (auto &f : st.flags) f.store(0u);
    for (auto &x : st.cnt) x.store(0u);
    for (int call = 1; call <= c.calls; ++call) {
        const uint32_t epoch = (uint32_t)call;
        // this call's sources; the destination poisoned so stale reads show
        for (int q = 0; q < s.R; ++q)
            for (int64_t r = 0; r < src_rows(q); ++r)
                for (int64_t b = 0; b < st.row_bytes; ++b)
                    st.src[q][(size_t)(r * st.row_bytes + b)] = src_byte(epoch, q, r, b, c.seed);
        std::fill(st.dst.begin(), st.dst.end(), (uint8_t)0xEE);
        if (c.op == 0)  // the local shard is in place in its slot of the gathered buffer
            std::memcpy(st.dst.data() + s.rb.off[s.rank] * st.row_bytes, st.src[s.rank].data(),
                        (size_t)(block_rows(s.rb, s.rank) * st.row_bytes));
        st.err.store(0);
        st.checked.store(0);
        std::vector<std::thread> th;
        for (int w = 0; w < c.stagers; ++w) th.emplace_back(stager, std::ref(st), w, epoch, call);
        for (int u = 0; u < c.walkers; ++u) th.emplace_back(walker, std::ref(st), u, epoch);
        for (auto &x : th) x.join();
        status[call - 1] = st.err.load();
        if (tiles_checked) tiles_checked[call - 1] = st.checked.load();
        if (status[call - 1] != 0)  // as syn_sync_status: clear the counters
            for (auto &x : st.cnt) x.store(0u);
    }
    return SYN_OK;
}
