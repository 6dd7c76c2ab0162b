// fused.cuh -- the fused, persistent, chunk-scheduled GEMM kernel for sm_103a.
//
// One launch computes a whole AG-GEMM, GEMM-RS or GEMM-AR (Syncopate summary
// page, Experiments, paper §6.1) while the chunks it consumes are still being
// staged: each output tile waits only on the chunks its rows touch (method ¶2:
// chunk-tile dependencies and inserted waits), and the persistent CTAs walk the
// host-built tile list, which is sorted by chunk arrival (method ¶4, paper
// §5.2, Fig. 6).  The chunks are staged by the copy engine, by dedicated
// staging CTAs of this same grid, or by a staging warp inside every GEMM CTA
// (method ¶3, paper §5.2, Fig. 7); all three publish per-chunk ready flags in
// global memory.
//
// CTA layout (256 threads, one CTA per SM, cooperative launch so that every
// CTA is resident and flag waits between CTAs cannot deadlock):
//   warp 0      TMA producer: waits on chunk flags (AG), then streams A/B
//               tiles into an S-stage shared-memory ring (mbarrier tx counts)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer into a
//               double-buffered fp32 TMEM accumulator
//   warps 2-5   epilogue: tcgen05.ld rows out of TMEM; AG: bf16 store;
//               RS/AR: add the peer partial tiles (ascending rank), bf16 store,
//               fp32 send/publish stores and producer counters
//   warp 6      RS/AR peer loader: waits on the peer chunks' flags, then TMA-
//               loads 128 x 32 fp32 peer sub-tiles into a P-slot ring
//   warp 7      co-located stager: copies this CTA's share of chunk slices with
//               TMA bulk copies (double-buffered) and publishes the chunk flags
// CTAs with blockIdx.x >= G are dedicated staging CTAs (7 single-buffer copier threads).
// RED instances (GEMM-RS/AR with resident peers) run 384 threads (GEMM-RS)
// or 640 (GEMM-AR): the epilogue stores a reducing tile's fp32 partial and
// frees the accumulator at once, and warps 8-11 (GEMM-AR: 6-19), joined by
// every other warp once its own role is done, add the peer partials to it
// with plain coalesced loads (same additions, same order, as the epilogue's
// own peer path).
//
// Two MMA shapes.  Single CTA: 128 x BN x 16 UMMAs (tcgen05 cta_group::1), each
// CTA stages its A rows and all BN columns of B.  CTA pair (PAIR, 2-CTA
// clusters): the even CTA issues 256 x BN x 16 UMMAs (cta_group::2) that read A
// rows 0-127 and B columns 0..BN/2 from its own shared memory and A rows 128-255
// and the other B columns from its peer's, and write each CTA's accumulator
// rows into that CTA's TMEM.  Per SM this halves the B bytes staged and read
// for the same MMA work, which is what lets the tensor pipe run near its peak
// on this architecture.  The peer's TMA loads complete on the even CTA's ring
// barrier; the MMA issuer commits each stage release and each accumulator-ready
// signal to the barrier of both CTAs (two single-target commits, the second to
// the peer's barrier through its shared::cluster address), and the peer's
// epilogue releases the accumulator with a remote mbarrier arrive.  (Forwarding
// those signals through a thread of the even CTA instead measured 2.5x slower.)
// No multicast form is used.
//
// Single-launch CTA-pair calls are launched with programmatic stream
// serialization: a CTA sets up its shared memory and TMEM, then waits
// (griddepcontrol.wait) for the previous kernel on the stream before it reads
// or writes global memory, so launch and set-up overlap that kernel's tail.
//
// Every wait is bounded (global timer) and ends in SYN_ERR_TIMEOUT written to
// the plan's error word; the CTA then drains its own outstanding asynchronous
// copies and MMAs, frees TMEM and returns.  Nothing traps.
#pragma once

#include <cuda_bf16.h>

#include "fused.h"
#include "protocol.h"
#include "ptx.cuh"

namespace syn {

// Shared memory given to the operand ring, the peer ring and the staging
// buffers (barriers and bookkeeping come on top).
constexpr int kSmemRings = 224 * 1024;

// Pre-summed GEMM-AR: most S chunk loads an epilogue warp keeps in flight.
// Two: every further slot takes shared memory from L1, and the reducer warps'
// peer stream slows as L1 shrinks (measured on the Qwen2-7B FFN down shape,
// 4 stages: 84.3 us with two slots, 91.8 us with four).
#ifndef SYN_PS_NSL_MAX
#define SYN_PS_NSL_MAX 2
#endif

// Compile-time shape of one kernel instance: operator, tile width BN, GEMM
// pipeline stages S, k-block depth BK (64: 128-byte A rows, 128-byte swizzle;
// 32: 64-byte A rows, 64-byte swizzle, half-size stages so twice as many fit),
// whether the CTA carries the co-located staging buffers (STG), and whether
// CTA pairs share 256-row tiles (PAIR).  For RS/AR the peer-tile ring takes
// whatever shared memory is left.
// Threads of a CTA: 256; RED instances add reducer warps, four for GEMM-RS
// (384: its few reducing tiles run beside MMAs that need the memory system)
// and twelve for GEMM-AR (640, 96 registers a thread: its reduction outlasts
// the MMAs, and the rate at which it streams the peers grows with the warps
// doing it -- 16 / 20 / 24 warps measured 98.0 / 97.2 / 104 us on the
// Qwen2-7B FFN down shape against 100.4 with 12; at 24 the registers spill).
constexpr int red_threads(int op, bool red) { return red ? (op == OP_AR ? 640 : 384) : 256; }

template <int OP, int BN, int S_, int BK_, bool STG, bool PAIR, bool RED>
struct KCfg {
    static constexpr int CTAS = PAIR ? 2 : 1;
    static constexpr int BM = 128, BK = BK_, UK = 16;
    static constexpr int TILE_M = BM * CTAS;          // output rows of one tile
    static constexpr int BN_CTA = BN / CTAS;          // B columns staged per CTA
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BK * BN_CTA * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TX_BYTES = CTAS * STAGE_BYTES;  // one ring phase, all CTAs
    static constexpr int S = S_;
    static constexpr int BN_ = BN;
    static constexpr bool STG_ = STG;
    static constexpr bool PAIR_ = PAIR;
    // RED (GEMM-RS/AR with resident peers): the epilogue only stores the fp32
    // partial of a reducing tile and frees the accumulator; more warps (8-11,
    // GEMM-AR 8-19) then stream the peer sum with plain loads, so no peer ring
    // is needed and every byte of the rings goes to pipeline stages
    static constexpr bool RED_ = RED;
    static constexpr int NTHREADS = red_threads(OP, RED);
    // PRESUM (GEMM-AR with reducer warps): the reducer warps sum the peer
    // partials of the walker's tiles, S = ((peer_q1 + peer_q2) + ...) over
    // q != rank ascending, from the start of the kernel into a plan buffer --
    // they depend on no tile's MMAs -- and the epilogue adds that one fp32
    // tile to the accumulator: out = rne(P + S).  Per epilogue warp: PS_NSL
    // shared-memory slots of 32 x 32 fp32 that TMA fills with S, and two
    // 32 x 32 bf16 slots for the TMA stores of out.  Reducer items of tile j
    // count into completion slot j % PS_NS; the epilogue's acknowledgement of
    // tile j lets items of tile j + PS_NS start.
    static constexpr bool PRESUM = RED && OP == OP_AR;
    static constexpr int PS_SLOT = 32 * 32 * 4;
    static constexpr int PS_OUT = 32 * 32 * 2;
    static constexpr int PS_ROOM = (kSmemRings - S * STAGE_BYTES) / 4 - 2 * PS_OUT;
    static constexpr int PS_NSL = PS_ROOM / PS_SLOT >= SYN_PS_NSL_MAX ? SYN_PS_NSL_MAX
                                                                      : PS_ROOM / PS_SLOT;  // S loads in flight
    static constexpr int PS_WARP = PS_NSL * PS_SLOT + 2 * PS_OUT;
    static constexpr int PS_NS = 8;
    // A (K-major): 8-row swizzle atoms of 8 * BK * 2 bytes
    static constexpr uint32_t A_SBO = 8 * BK * 2;
    static constexpr uint32_t A_SWZ = BK == 64 ? ptx::kSwizzle128B : ptx::kSwizzle64B;
    // B (N-major): one TMA box of 64 columns x BK rows per 64 staged columns
    static constexpr uint32_t B_BOX_BYTES = BK * 128;
    static constexpr int PEER_COLS = 32;
    static constexpr int PEER_BYTES = BM * PEER_COLS * 4;
    // Epilogue store staging: when the rings leave room, each epilogue warp
    // writes its 32 rows x 32 columns (GEMM-RS/AR fp32 with 128-byte swizzle,
    // AG bf16 with 64-byte swizzle) into one of two shared-memory buffers and
    // issues a TMA tile store (whole lines) instead of one 16-byte store per
    // thread and row.  AG takes its buffers before the stager's.
    static constexpr int EPI_SLOT = 32 * 32 * (OP == OP_AG ? 2 : 4);
    static constexpr int EPI_WANT = 8 * EPI_SLOT;
    static constexpr int STG_BYTES = 16384;
    static constexpr bool EPI_AG =
        OP == OP_AG && PAIR && kSmemRings - S * STAGE_BYTES >= EPI_WANT + (STG ? STG_BYTES : 0);
    // co-located staging buffers: two for RS/AR (the peer ring takes the rest);
    // for AG every 16 KiB the stages and the epilogue buffers leave (up to 8),
    // so shallower pipelines trade MMA lookahead for more staging copies
    static constexpr int NSTG_AG = (kSmemRings - S * STAGE_BYTES - (EPI_AG ? EPI_WANT : 0)) / STG_BYTES;
    static constexpr int NSTG = !STG ? 0 : OP != OP_AG ? 2 : (NSTG_AG > 8 ? 8 : NSTG_AG);
    static constexpr int P =
        OP == OP_AG || RED ? 0 : (kSmemRings - NSTG * STG_BYTES - S * STAGE_BYTES) / PEER_BYTES;
    static_assert(OP == OP_AG || RED || P >= 2, "peer ring needs at least two slots");
    static_assert(!RED || (OP != OP_AG && !STG), "deferred reduction: GEMM-RS/AR, resident peers");
    static_assert(S * STAGE_BYTES + P * PEER_BYTES + NSTG * STG_BYTES <= kSmemRings, "rings");
    static constexpr int EPI_LEFT = kSmemRings - S * STAGE_BYTES - P * PEER_BYTES - NSTG * STG_BYTES;
    static constexpr bool EPI_TMA = OP == OP_AG ? EPI_AG : EPI_LEFT >= EPI_WANT;
    static constexpr int EPI_BYTES = PRESUM ? 4 * PS_WARP : EPI_TMA ? EPI_WANT : 0;
    static_assert(!PRESUM || (PS_NSL >= 2 && EPI_LEFT >= 4 * PS_WARP), "pre-summed reduction: epilogue slots");
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + S * A_BYTES;
    static constexpr int OFF_PEER = OFF_B + S * B_BYTES;
    static constexpr int OFF_STG = OFF_PEER + P * PEER_BYTES;
    static constexpr int OFF_EPI = OFF_STG + NSTG * STG_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    // barrier slots
    static constexpr int BAR_FULL = 0;
    static constexpr int BAR_EMPTY = BAR_FULL + S;
    static constexpr int BAR_TFULL = BAR_EMPTY + S;
    static constexpr int BAR_TEMPTY = BAR_TFULL + 2;
    static constexpr int BAR_PFULL = BAR_TEMPTY + 2;
    static constexpr int BAR_PEMPTY = BAR_PFULL + P;
    static constexpr int BAR_STG = BAR_PEMPTY + P;
    static constexpr int BAR_DRAIN = BAR_STG + NSTG;
    static constexpr int BAR_PEERDONE = BAR_DRAIN + 1;  // PAIR: odd producer finished issuing
    static constexpr int BAR_SLD = BAR_PEERDONE + 1;     // PRESUM: S slot loads, PS_NSL per epilogue warp
    static constexpr int NBAR = BAR_SLD + (PRESUM ? 4 * PS_NSL : 0);
    static constexpr int COMM_BUF_BYTES = 32768;  // (one 256 x 32 fp32 push box)
    static constexpr int COMM_NBUF = OFF_BAR / COMM_BUF_BYTES;
    static constexpr int NBAR_ALL = NBAR > COMM_NBUF ? NBAR : COMM_NBUF;
    static constexpr int OFF_MISC = OFF_BAR + NBAR_ALL * 8;
    // misc words: +0 TMEM base, +4 abort flag, +8 odd CTA's k-block count,
    // +16 (RED) per TMEM lane quadrant: reducing tiles whose partial is stored,
    // +32 (RED) next reduction work item, +36 (RED) 1 + the walker's reducing
    // tiles once the epilogue has seen them all (0 before)
    static constexpr int OFF_RED_READY = OFF_MISC + 16;
    static constexpr int OFF_RED_NEXT = OFF_MISC + 32;
    static constexpr int OFF_RED_TOTAL = OFF_MISC + 36;
    // PRESUM: completed reducer items per (slot j % PS_NS, TMEM lane quadrant),
    // then per quadrant the tiles whose completion the epilogue has seen
    static constexpr int OFF_PS_DONE = OFF_MISC + 48;
    static constexpr int OFF_PS_ACK = OFF_PS_DONE + PS_NS * 4 * 4;
    static constexpr int SMEM_USED = OFF_MISC + 48 + (PRESUM ? PS_NS * 16 + 16 : 0);
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_B % 1024 == 0 && OFF_PEER % 1024 == 0 && OFF_STG % 1024 == 0 && OFF_EPI % 1024 == 0,
                  "1 KiB atoms");
    static_assert(S * STAGE_BYTES + P * PEER_BYTES + NSTG * STG_BYTES + EPI_BYTES <= kSmemRings, "epilogue");
    static_assert(BN == 128 || BN == 256, "tile_n");
    static_assert(BK == 64 || BK == 32, "tile_k");
    static_assert(BN_CTA % 64 == 0, "B is staged in 64-column boxes");
    static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(TILE_M, BN, true);
};

// ------------------------------------------------------------------ errors and bounded waits
__device__ __forceinline__ void raise_error(const KernelParams &p, int code, int where, int info) {
    if (atomicCAS(p.err, 0, code) == 0) {
        p.err[1] = where;
        p.err[2] = (int)blockIdx.x;
        p.err[3] = info;
    }
}

__device__ __forceinline__ bool grid_failed(const KernelParams &p) {
    return *reinterpret_cast<volatile int32_t *>(p.err) != 0;
}

template <bool CL>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
    if constexpr (CL)
        return ptx::mbar_try_wait_cluster(bar, parity);
    else
        return ptx::mbar_try_wait(bar, parity);
}

// Wait for the phase of parity `parity` of mbarrier `bar` (acquire at cluster
// scope when CL).  False once the CTA aborts, the grid reports an error, or the
// bound runs out (then raises).
template <bool CL = false>
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int *abort,
                                      const KernelParams &p) {
    if (try_wait<CL>(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    for (uint32_t n = 1;; ++n) {
        if (try_wait<CL>(bar, parity)) return true;
        if (*abort) return false;
        if ((n & 31u) == 0u) {
            if (grid_failed(p)) {
                *abort = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > limit) {
                raise_error(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)bar);
                *abort = 1;
                return false;
            }
        }
    }
}

// Wait used only while draining on the way out: ignores the abort flag.
template <bool CL = false>
__device__ __forceinline__ void bwait_drain(uint32_t bar, uint32_t parity, const KernelParams &p) {
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    for (uint32_t n = 0;; ++n) {
        if (try_wait<CL>(bar, parity)) return;
        if ((n & 31u) == 31u && ptx::globaltimer() - t0 > limit) {
            raise_error(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)bar);
            return;
        }
    }
}

// Acquire-wait until the ready flag of a chunk carries this call's epoch.
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, const KernelParams &p,
                                          volatile int *abort, int where, int info,
                                          unsigned long long &waited_ns) {
    if (flag_ready(ptx::ld_acquire_gpu(flag), p.epoch)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        __nanosleep(40);
        if (flag_ready(ptx::ld_acquire_gpu(flag), p.epoch)) {
            waited_ns += ptx::globaltimer() - t0;
            return true;
        }
        if (*abort) return false;
        if ((n & 15u) == 0u) {
            if (grid_failed(p)) {
                *abort = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > p.timeout_ns) {
                raise_error(p, SYN_ERR_TIMEOUT, where, info);
                *abort = 1;
                return false;
            }
        }
    }
}

// Acquire-wait until the shared-memory counter at `addr` reaches `want`
// (written by another warp of this CTA with a release store): 1.  2 once the
// word at `total` (1 + the final count, 0 while unknown) shows the counter
// will never get there; 0 on abort or timeout.
__device__ __forceinline__ int wait_smem_count(uint32_t addr, uint32_t total, uint32_t want,
                                               const KernelParams &p, volatile int *abort) {
    auto state = [&]() -> int {
        if ((int32_t)(ptx::ld_acquire_cta_shared(addr) - want) >= 0) return 1;
        const uint32_t tot = ptx::ld_acquire_cta_shared(total);
        return (tot != 0u && want > tot - 1u) ? 2 : -1;
    };
    int st = state();
    if (st >= 0) return st;
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    // back off up to ~1 us: a waiting warp must not take issue slots from the
    // MMA issuer and the epilogue of its SM for the whole walk
    uint32_t sleep_ns = 32;
    for (uint32_t n = 1;; ++n) {
        __nanosleep(sleep_ns);
        if (sleep_ns < 1024u) sleep_ns *= 2u;
        if ((st = state()) >= 0) return st;
        if (*abort) return 0;
        if ((n & 31u) == 0u) {
            if (grid_failed(p)) {
                *abort = 1;
                return 0;
            }
            if (ptx::globaltimer() - t0 > limit) {
                raise_error(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)want);
                *abort = 1;
                return 0;
            }
        }
    }
}

// Row chunks [lo, hi] that rows [r0, r0 + nrows) clipped to M touch; lo > hi
// when every row lies past M (the odd CTA of a ragged last pair tile).
__device__ __forceinline__ void chunk_range(const KernelParams &p, int r0, int nrows, int &lo,
                                            int &hi) {
    chunk_range_of(p.M, p.rb, r0, nrows, lo, hi);
}

// Do rows [r0, r0 + nrows) (a tile's, or one CTA's share of it) reduce peers?
// AR: always; RS: when some of them lie in the local row block (a tile may
// straddle the block's edges; each 32-row warp group lies wholly inside or
// outside it, since M_r % 32 == 0).
template <int OP>
__device__ __forceinline__ bool reduces(const KernelParams &p, int r0, int nrows) {
    if (OP == OP_AR) return true;
    if (OP == OP_RS) {
        const int lo = p.rank * p.M_r;  // (< M <= 2^30)
        return r0 < lo + p.M_r && r0 + nrows > lo;
    }
    return false;
}
// GEMM-RS: do rows [r0, r0 + nrows) clipped to M include rows outside the
// local block (rows to send)?
template <int OP>
__device__ __forceinline__ bool sends(const KernelParams &p, int r0, int nrows) {
    if (OP != OP_RS) return false;
    const int lo = p.rank * p.M_r, r1 = r0 + nrows < p.M ? r0 + nrows : p.M;
    return r0 < lo || r1 > lo + p.M_r;
}
// GEMM-RS: is row `row` one of the local block's (reduced, not sent)?  AR: all rows.
template <int OP>
__device__ __forceinline__ bool local_row(const KernelParams &p, int row) {
    const int lo = p.rank * p.M_r;  // (< M <= 2^30)
    return OP != OP_RS || (row >= lo && row < lo + p.M_r);
}

// ------------------------------------------------------------------ tile walk
// A walker (a CTA, or a CTA pair) runs tile-list entries one after another:
// walker u of n runs entries u, u + n, u + 2n, ...; -1 ends the walk.
__device__ __forceinline__ int walk_entry(const KernelParams &p, int unit, int n_units, int i) {
    return walk_entry_of(p.t_begin, p.t_end, unit, n_units, i);
}

// Tile id at tile-list entry t, or -1 (with SYN_ERR_BOUNDS raised and the CTA
// aborting) when the table holds an id outside the tile grid: no role ever
// addresses memory from an unchecked entry.
__device__ __forceinline__ int tile_at(const KernelParams &p, int t, volatile int *abort) {
    const int tile = p.tile_list[t];
    if (tile < 0 || tile >= p.tiles_m * p.tiles_n) {
        raise_error(p, SYN_ERR_BOUNDS, WHERE_BOUNDS, t);
        *abort = 1;
        return -1;
    }
    return tile;
}

// ------------------------------------------------------------------ staging (device backends)
// Copy `len` bytes src -> dst through an nbuf-slot shared-memory ring with TMA
// bulk copies (global -> smem with mbarrier completion, smem -> global bulk
// group).  `phase_bits` carries each slot's barrier parity across calls.
template <typename Landed>
__device__ __forceinline__ bool bulk_copy(const uint8_t *src, uint8_t *dst, int64_t len,
                                          uint32_t buf0, int nbuf, uint32_t buf_bytes,
                                          uint32_t bar0, uint32_t &phase_bits,
                                          volatile int *abort, const KernelParams &p, Landed &&prev_landed) {
    const int n = (int)((len + buf_bytes - 1) / buf_bytes);
    auto piece = [&](int i) -> uint32_t {
        const int64_t rem = len - (int64_t)i * buf_bytes;
        return (uint32_t)(rem < (int64_t)buf_bytes ? rem : (int64_t)buf_bytes);
    };
    auto issue = [&](int i) {
        const int b = i % nbuf;
        const uint32_t bytes = piece(i);
        ptx::mbar_arrive_expect_tx(bar0 + 8 * b, bytes);
        ptx::bulk_g2s(buf0 + b * buf_bytes, src + (int64_t)i * buf_bytes, bytes, bar0 + 8 * b);
    };
    // the previous range's stores must have read the buffers before they are
    // refilled; their completion in global memory is awaited only after this
    // range's first loads are in flight (prev_landed), so that wait and the
    // previous range's flag publication overlap the new loads
    ptx::bulk_wait_read_all();
    const int pre = n < nbuf ? n : nbuf;
    for (int i = 0; i < pre; ++i) issue(i);
    prev_landed();
    for (int i = 0; i < n; ++i) {
        const int b = i % nbuf;
        const uint32_t par = (phase_bits >> b) & 1u;
        if (!bwait(bar0 + 8 * b, par, abort, p)) {
            // drain every load still in flight, then the stores
            for (int j = i; j < n && j < i + nbuf; ++j) {
                const int bj = j % nbuf;
                bwait_drain(bar0 + 8 * bj, (phase_bits >> bj) & 1u, p);
                phase_bits ^= 1u << bj;
            }
            ptx::bulk_wait_all();
            return false;
        }
        phase_bits ^= 1u << b;
        ptx::fence_proxy_async_smem();
        ptx::bulk_s2g(dst + (int64_t)i * buf_bytes, buf0 + b * buf_bytes, piece(i));
        ptx::bulk_commit();
        if (i + nbuf < n) {
            ptx::bulk_wait_read_all();  // slot b has been read by its store
            issue(i + nbuf);
        }
    }
    return true;  // this range's stores may still be in flight
}

// Stage this worker's share of chunk slices (worker w of W takes global slices
// w, w+W, ... in arrival order) and publish a chunk's flag once its last slice
// has landed (last arriver on the epoch-parity slice counter).
__device__ __forceinline__ void stage_slices(const KernelParams &p, int worker, int W,
                                             uint32_t buf0, int nbuf, uint32_t buf_bytes,
                                             uint32_t bar0, volatile int *abort) {
    const int spt = p.slices_per_transfer;
    const int total = p.n_transfers * spt;
    const int n_flags = p.n_rc * p.R;
    uint32_t *cnt = p.in_cnt + (size_t)counter_half(p.epoch) * n_flags;
    uint32_t phase_bits = 0;
    // the slice whose stores were issued last and are not yet counted (-1: none)
    int pend_a = -1, pend_code = 0;
    auto count_slice = [&](int a, int code) {  // its bytes have landed
        ptx::fence_proxy_async();
        const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt + code, 1u);
        if (completes_transfer(old, (uint32_t)spt) && a != p.drop_transfer) {
            if (a == p.delay_transfer) {  // fault injection: publish late (bounded by the delay)
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < p.delay_ns && !*abort) __nanosleep(1000);
            }
            ptx::st_release_gpu(p.in_flags + code, p.epoch);
        }
    };
    auto land_pending = [&]() {
        if (pend_a >= 0) {
            ptx::bulk_wait_all();
            count_slice(pend_a, pend_code);
            pend_a = -1;
        }
    };
    for (int g = worker; g < total; g += W) {
        const int a = g / spt, sl = g % spt;
        const int code = p.transfers[a];
        if (code < 0 || code >= n_flags) {  // the transfer table holds a code outside the flags
            land_pending();
            raise_error(p, SYN_ERR_BOUNDS, WHERE_BOUNDS, a);
            *abort = 1;
            return;
        }
        if (p.op == OP_AG && p.local_inplace && code % p.R == p.rank) continue;
        const uint8_t *src;
        uint8_t *dst;
        int64_t bytes;
        transfer_span(p, code, src, dst, bytes);
        // slices past the end of a shorter chunk copy nothing but still count
        const int64_t off = (int64_t)sl * p.slice_bytes;
        const int64_t rem = bytes - off;
        const int64_t len = rem < p.slice_bytes ? rem : p.slice_bytes;
        if (len > 0) {
            if (!bulk_copy(src + off, dst + off, len, buf0, nbuf, buf_bytes, bar0, phase_bits, abort, p,
                           land_pending))
                return;
            pend_a = a;
            pend_code = code;
        } else {
            land_pending();
            count_slice(a, code);
        }
    }
    land_pending();
}

// Dedicated push (GEMM-RS push mode with push CTAs): worker `worker` of `W`
// takes boxes worker, worker + W, ... (32 rows x 256 columns, 32 KB) of the
// send chunks in production order.  Per chunk it waits until the chunk's rows
// are produced (out flag, acquire), then per box TMA-loads it from push_buf
// into its shared-memory buffer and adds it into the destination's receive
// accumulator (`send`) with a TMA tile reduce-add, reloading the buffer as
// soon as the add has read it.  Once its boxes of a chunk have landed it
// counts them; the worker that completes the chunk's count publishes the
// delivered flag (in_flags[rc * R + rank]: this rank's contribution to chunk
// rc has arrived).  Chunk rows are a multiple of 32 (the host checks).
__device__ __forceinline__ void push_slices(const KernelParams &p, const TensorMaps &tm, int worker, int W,
                                            uint32_t buf, uint32_t bar, volatile int *abort) {
    constexpr int BOX_COLS = kPushBoxCols, BOX_ROWS = 32;
    constexpr uint32_t BOX_BYTES = BOX_COLS * BOX_ROWS * 4;
    const int n_flags = p.n_rc * p.R;
    const int col_boxes = (p.N + BOX_COLS - 1) / BOX_COLS;
    uint32_t *cnt = p.in_cnt + (size_t)counter_half(p.epoch) * n_flags;
    uint32_t phase = 0;
    unsigned long long wait_ns = 0;
    for (int a = 0, g = 0; a < p.n_push; ++a) {
        const int rc = p.push_list[a];
        if (rc < 0 || rc >= p.n_rc) {  // the push table holds a chunk outside the plan
            ptx::bulk_wait_all();
            raise_error(p, SYN_ERR_BOUNDS, WHERE_BOUNDS, a);
            *abort = 1;
            return;
        }
        const int row0 = (int)chunk_row0(p.rb, rc);
        const int n_boxes = (int)(chunk_row0(p.rb, rc + 1) - row0) / BOX_ROWS * col_boxes;
        uint32_t mine = 0;
        for (int bx = 0; bx < n_boxes; ++bx, ++g) {
            if (g % W != worker) continue;
            if (mine == 0) {
                if (!wait_flag(p.out_flags + rc, p, abort, WHERE_STAGER, rc, wait_ns)) {
                    ptx::bulk_wait_all();
                    return;
                }
                ptx::fence_proxy_async();  // generic acquire -> async-proxy (TMA) reads
            }
            const int x = (bx % col_boxes) * BOX_COLS, y = row0 + (bx / col_boxes) * BOX_ROWS;
            ptx::bulk_wait_read_all();  // the previous box's add has read the buffer
            ptx::mbar_arrive_expect_tx(bar, BOX_BYTES);
            ptx::tma_load_2d(buf, &tm.push_src, bar, x, y);
            if (!bwait(bar, phase, abort, p)) {
                bwait_drain(bar, phase, p);  // the load in flight lands before the CTA leaves
                ptx::bulk_wait_all();
                return;
            }
            phase ^= 1u;
            ptx::tma_reduce_add_2d(&tm.push_dst, buf, x, y);
            ptx::bulk_commit();
            ++mine;
        }
        if (mine > 0) {
            ptx::bulk_wait_all();  // this worker's adds to the chunk have landed
            ptx::fence_proxy_async();
            const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt + rc * p.R + p.rank, mine);
            if (old + mine == (uint32_t)n_boxes) ptx::st_release_gpu(p.in_flags + rc * p.R + p.rank, p.epoch);
        }
    }
}

// Load/store staging (the pages' load/store lowerings): warp `worker` of `W`
// copies slices worker, worker + W, ... with every lane moving 16-byte
// vectors (eight in flight per lane); after a slice lane 0 fences, counts it,
// and the warp that completes a transfer publishes its flag (release).
__device__ __forceinline__ void stage_slices_ldst(const KernelParams &p, int worker, int W, int lane,
                                                  volatile int *abort) {
    const int spt = p.slices_per_transfer;
    const int total = p.n_transfers * spt;
    const int n_flags = p.n_rc * p.R;
    uint32_t *cnt = p.in_cnt + (size_t)counter_half(p.epoch) * n_flags;
    for (int g = worker; g < total; g += W) {
        if (*abort) return;
        const int a = g / spt, sl = g % spt;
        const int code = p.transfers[a];
        if (code < 0 || code >= n_flags) {  // the transfer table holds a code outside the flags
            if (lane == 0) {
                raise_error(p, SYN_ERR_BOUNDS, WHERE_BOUNDS, a);
                *abort = 1;
            }
            return;
        }
        if (p.op == OP_AG && p.local_inplace && code % p.R == p.rank) continue;
        const uint8_t *src;
        uint8_t *dst;
        int64_t bytes;
        transfer_span(p, code, src, dst, bytes);
        const int64_t off = (int64_t)sl * p.slice_bytes;
        const int64_t len = bytes - off < p.slice_bytes ? bytes - off : p.slice_bytes;
        // (slices past the end of a shorter chunk copy nothing but still count)
        for (int64_t b = (int64_t)lane * 16; b < len; b += 32 * 16 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (b + u * 512 < len) v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + off + b + u * 512));
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (b + u * 512 < len) *reinterpret_cast<uint4 *>(dst + off + b + u * 512) = v[u];
        }
        __syncwarp();
        if (lane == 0) {
            ptx::fence_acq_rel_gpu();  // the warp's stores, observed through the barrier, before the count
            const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt + code, 1u);
            if (completes_transfer(old, (uint32_t)spt) && a != p.drop_transfer) {
                if (a == p.delay_transfer) {  // fault injection: publish late (bounded by the delay)
                    const uint64_t t0 = ptx::globaltimer();
                    while (ptx::globaltimer() - t0 < p.delay_ns && !*abort) __nanosleep(1000);
                }
                ptx::st_release_gpu(p.in_flags + code, p.epoch);
            }
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ epilogue helpers
// 32-column chunks of tile column tni that hold columns < N (all BN / 32 but
// in the last tile column when N is not a multiple of the tile width); the
// chunks past N are neither read from TMEM nor stored nor fed with peers.
template <int BN>
__device__ __forceinline__ int live_chunks(const KernelParams &p, int tni) {
    const int left = p.N - tni * BN;
    return left >= BN ? BN / 32 : (left + 31) / 32;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// (lim: the columns left in the row from dst on; N is a multiple of 8, so a
// 16-byte vector is either wholly inside the row or wholly past its end)
__device__ __forceinline__ void store_bf16_row32(uint16_t *dst, const float (&f)[32], int lim) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (8 * j >= lim) break;
        uint4 v;
        v.x = pack_bf16x2(f[8 * j + 0], f[8 * j + 1]);
        v.y = pack_bf16x2(f[8 * j + 2], f[8 * j + 3]);
        v.z = pack_bf16x2(f[8 * j + 4], f[8 * j + 5]);
        v.w = pack_bf16x2(f[8 * j + 6], f[8 * j + 7]);
        d[j] = v;
    }
}

__device__ __forceinline__ void store_f32_row32(float *dst, const float (&f)[32], int lim) {
    float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (4 * j < lim) d[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
}

// Producer side of a tile that writes send/publish rows: once this warp's rows
// are stored, count the warp on every row chunk the tile (rows [r0, r0 +
// tile_m)) covers; the last of the 4 * ctas * tiles_n * (tile rows over the
// chunk) arrivals publishes the chunk's out flag.
__device__ __forceinline__ void count_produced(const KernelParams &p, int r0, int tile_m, int ctas,
                                               int lane) {
    __syncwarp();
    if (lane == 0) {
        ptx::fence_acq_rel_gpu();
        int lo, hi;
        chunk_range(p, r0, tile_m, lo, hi);
        uint32_t *cnt = p.out_cnt + (size_t)counter_half(p.epoch) * p.n_rc;
        for (int rc = lo; rc <= hi; ++rc) {
            const int64_t row0 = chunk_row0(p.rb, rc);
            const int64_t row1 = chunk_row0(p.rb, rc + 1);
            const int t_lo = (int)(row0 / tile_m);
            const int t_hi = (int)((row1 - 1) / tile_m);
            const uint32_t need = 4u * (uint32_t)ctas * (uint32_t)((t_hi - t_lo + 1) * p.tiles_n);
            const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt + rc, 1u);
            if (old + 1u == need) ptx::st_release_gpu(p.out_flags + rc, p.epoch);
        }
    }
}

// The order every GEMM-RS / GEMM-AR path adds in: the peer partials first,
// S = ((peer_q1 + peer_q2) + ...) over q != rank ascending, then the local
// partial, out = bf16(P + S) -- one order for every backend, so their outputs
// are bit-identical; and it lets the peer sum start before P exists.

// Deferred reduction of ROWS rows x BN columns starting at (row0, col0): out =
// bf16(P + S), P the fp32 partial the epilogue stored in red_buf -- the same
// additions in the same order as the epilogue's own peer path.  One warp;
// lane l takes columns 4l..4l+3 of every 128-column half, so every load and
// store of the warp is one contiguous row segment, and U rows x all sources
// are in flight at once.
// S of one float4 column group: the left fold over q != rank ascending of
// pv[q][u][h]; -0 (the identity of an fp32 sum) when there is no peer.
template <int U, int H>
__device__ __forceinline__ float4 peer_sum(const KernelParams &p, const float4 (&pv)[kMaxRanks][U][H], int u,
                                           int h) {
    float4 s = make_float4(-0.f, -0.f, -0.f, -0.f);
    bool first = true;
#pragma unroll
    for (int q = 0; q < kMaxRanks; ++q)
        if (q < p.R && q != p.rank) {
            if (first) {
                s = pv[q][u][h];
                first = false;
            } else {
                s.x = s.x + pv[q][u][h].x;
                s.y = s.y + pv[q][u][h].y;
                s.z = s.z + pv[q][u][h].z;
                s.w = s.w + pv[q][u][h].w;
            }
        }
    return s;
}

template <int OP, int BN, int ROWS>
__device__ __forceinline__ void reduce_rows(const KernelParams &p, int row0, int col0, int lane) {
    constexpr int H = BN / 128;
    constexpr int U = OP == OP_AR ? 1 : 2;  // (GEMM-AR's wider CTA has 128 registers a thread)
    static_assert(ROWS % U == 0, "rows per pass");
    const int64_t N = p.N;
#pragma unroll 1
    for (int rr = 0; rr < ROWS; rr += U) {
        float4 acc[U][H];
        float4 pv[kMaxRanks][U][H];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int row = row0 + rr + u;
            const float *src = p.red_buf + (int64_t)(row - p.red_row_off) * N + col0 + 4 * lane;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const bool live = row < p.M && col0 + 4 * lane + 128 * h < N;
                acc[u][h] = live ? ptx::ld_f4(src + 128 * h) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < kMaxRanks; ++q)
                    if (live && q < p.R && q != p.rank)
                        pv[q][u][h] = ptx::ld_nc_f4(reinterpret_cast<const float *>(p.stage_src[q]) +
                                                    (int64_t)row * N + col0 + 4 * lane + 128 * h);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int row = row0 + rr + u;
            if (row >= p.M) continue;
            const int orow = OP == OP_RS ? row - p.rank * p.M_r : row;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                if (col0 + 4 * lane + 128 * h >= N) continue;
                float4 a = acc[u][h];
                const float4 sum = peer_sum(p, pv, u, h);
                a.x = a.x + sum.x;
                a.y = a.y + sum.y;
                a.z = a.z + sum.z;
                a.w = a.w + sum.w;
                ptx::st_u32x2(p.out + (int64_t)orow * N + col0 + 4 * lane + 128 * h,
                              pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
            }
        }
    }
}

// The CTA's reduction work (RED), shared by every warp that has nothing else
// to do: item k is row group k % 4 (8 rows) of TMEM lane quadrant (k / 4) % 4
// of the walker's (k / 16)-th reducing tile, in this CTA's rows.  Warps claim
// items in order from a shared-memory counter; an item starts once the
// epilogue warp of its quadrant has stored that tile's partial.  Warps 8 on
// (GEMM-AR: 6 on) work from the start, the epilogue, producer and MMA warps
// join when their own work is done, so GEMM-AR's reduction, which outlasts
// its MMAs, ends up on all twenty warps.
template <class C, int OP, int BN>
__device__ __forceinline__ void reduce_worker(const KernelParams &p, uint8_t *sm, uint32_t sbase, int unit,
                                              int n_units, uint32_t crank, int lane, volatile int *abort) {
    // two rows per item (one pass of reduce_rows): the finest split measured
    // fastest (items of 32 / 8 / 4 / 2 rows: GEMM-RS 135 / 106 / 105 / 104 us,
    // GEMM-AR 117 / 117 / 116.5 / 113.5 us on the FFN shapes)
    constexpr int RG = 2;
    constexpr int PER_Q = 32 / RG;
    constexpr int PER_TILE = 4 * PER_Q;
    uint32_t *next = reinterpret_cast<uint32_t *>(sm + C::OFF_RED_NEXT);
    int scan_i = 0, scan_j = -1, cur_t = -1;  // cursor over this walker's reducing tiles
    for (;;) {
        uint32_t k = 0;
        if (lane == 0) k = atomicAdd(next, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        const int j = (int)(k / PER_TILE), q = (int)(k / PER_Q) % 4, g = (int)(k % PER_Q);
        int st = 1;
        if (lane == 0)
            st = wait_smem_count(sbase + C::OFF_RED_READY + 4 * q, sbase + C::OFF_RED_TOTAL, (uint32_t)(j + 1),
                                 p, abort);
        __syncwarp();  // orders lane 0's acquire before every lane's loads
        st = __shfl_sync(0xffffffffu, st, 0);
        if (st != 1) return;  // aborted, or the walk has no j-th reducing tile
        while (scan_j < j) {
            const int t = walk_entry(p, unit, n_units, scan_i++);
            if (t < 0) return;  // (cannot happen: the epilogue stored tile j)
            const int tl = tile_at(p, t, abort);
            if (tl < 0) return;
            if (reduces<OP>(p, (tl / p.tiles_n) * C::TILE_M + (int)crank * C::BM, C::BM)) {
                ++scan_j;
                cur_t = t;
            }
        }
        const int tile = p.tile_list[cur_t];
        const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
        const int row0 = tmi * C::TILE_M + (int)crank * C::BM + q * 32 + g * RG;
        // (GEMM-RS: a quadrant of a tile straddling the local block's edge may
        // hold sent rows; its 32 rows lie wholly in or out of the block)
        if (local_row<OP>(p, row0)) reduce_rows<OP, BN, RG>(p, row0, tni * BN, lane);
    }
}

// ------------------------------------------------------------------ pre-summed GEMM-AR reduction
// Acquire-wait until the shared-memory counter at `addr` reaches `want`
// (written by other warps of this CTA with release operations).  False on
// abort or timeout.
__device__ __forceinline__ bool wait_smem_at_least(uint32_t addr, uint32_t want, const KernelParams &p,
                                                   volatile int *abort) {
    if ((int32_t)(ptx::ld_acquire_cta_shared(addr) - want) >= 0) return true;
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    uint32_t sleep_ns = 32;
    for (uint32_t n = 1;; ++n) {
        __nanosleep(sleep_ns);
        if (sleep_ns < 512u) sleep_ns *= 2u;
        if ((int32_t)(ptx::ld_acquire_cta_shared(addr) - want) >= 0) return true;
        if (*abort) return false;
        if ((n & 31u) == 0u) {
            if (grid_failed(p)) {
                *abort = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > limit) {
                raise_error(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)want);
                *abort = 1;
                return false;
            }
        }
    }
}

// S for ROWS rows x BN columns at (row0, col0): the peer partials summed in
// ascending q (q != rank), stored fp32 into red_buf.  One warp, one row per
// pass; lane l takes columns 4l..4l+3 of every 128-column half, so every load
// and store of the warp is one contiguous row segment.
template <int BN, int ROWS>
__device__ __forceinline__ void presum_rows(const KernelParams &p, int row0, int col0, int lane) {
    constexpr int H = BN / 128;
    const int64_t N = p.N;
#pragma unroll 1
    for (int rr = 0; rr < ROWS; ++rr) {
        const int row = row0 + rr;
        if (row >= p.M) break;
        float4 pv[kMaxRanks][1][H];
#pragma unroll
        for (int h = 0; h < H; ++h)
#pragma unroll
            for (int q = 0; q < kMaxRanks; ++q)
                if (q < p.R && q != p.rank && col0 + 4 * lane + 128 * h < N) {
                    const float *src = reinterpret_cast<const float *>(p.stage_src[q]) + (int64_t)row * N +
                                       col0 + 4 * lane + 128 * h;
                    pv[q][0][h] = ptx::ld_nc_f4(src);
                }
#pragma unroll
        for (int h = 0; h < H; ++h)
            if (col0 + 4 * lane + 128 * h < N)
                ptx::st_f4(p.red_buf + (int64_t)(row - p.red_row_off) * N + col0 + 4 * lane + 128 * h,
                           peer_sum(p, pv, 0, h));
    }
}

// Reducer side of the pre-summed GEMM-AR: item k is row pair k % 16 of TMEM
// lane quadrant (k / 16) % 4 of the walker's (k / 64)-th tile, in this CTA's
// rows.  An item of tile j >= PS_NS first waits until the epilogue warp of
// its quadrant has seen tile j - PS_NS complete (so completion slot j % PS_NS
// is free), then sums the peers and counts itself complete (release).
// Returns 1 when done, 0 when the walk has no tile for item k, -1 on abort.
template <class C, int BN>
__device__ __forceinline__ int presum_item(const KernelParams &p, uint32_t sbase, int unit, int n_units,
                                           uint32_t crank, int lane, volatile int *abort, uint32_t k) {
    constexpr int RG = 2;
    constexpr int PER_Q = 32 / RG;
    constexpr int PER_TILE = 4 * PER_Q;
    const int j = (int)(k / PER_TILE), q = (int)(k / PER_Q) % 4, g = (int)(k % PER_Q);
    const int t = walk_entry(p, unit, n_units, j);
    if (t < 0) return 0;
    const int tile = tile_at(p, t, abort);
    if (tile < 0) return -1;
    if (j >= C::PS_NS) {
        int ok = 1;
        if (lane == 0)
            ok = wait_smem_at_least(sbase + C::OFF_PS_ACK + 4 * q, (uint32_t)(j - C::PS_NS + 1), p, abort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return -1;
    }
    const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
    presum_rows<BN, RG>(p, tmi * C::TILE_M + (int)crank * C::BM + q * 32 + g * RG, tni * BN, lane);
    // the stores before the count, for the epilogue's TMA loads
    ptx::fence_proxy_async_global();
    __threadfence_block();
    __syncwarp();
    if (lane == 0)
        ptx::red_add_release_cta_shared(sbase + C::OFF_PS_DONE + 4 * ((j % C::PS_NS) * 4 + q), 1u);
    return 1;
}

// Reducer warps claim items in order from a shared-memory counter until the
// walk has none left.
template <class C, int BN>
__device__ __forceinline__ void presum_worker(const KernelParams &p, uint8_t *sm, uint32_t sbase, int unit,
                                              int n_units, uint32_t crank, int lane, volatile int *abort) {
    uint32_t *next = reinterpret_cast<uint32_t *>(sm + C::OFF_RED_NEXT);
    for (;;) {
        uint32_t k = 0;
        if (lane == 0) k = atomicAdd(next, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (presum_item<C, BN>(p, sbase, unit, n_units, crank, lane, abort, k) != 1) return;
    }
}

// Epilogue side of the pre-summed GEMM-AR, one warp (TMEM lane quadrant qd),
// the whole walk: per tile, wait until the tile's S rows of this quadrant are
// complete, then per 32-column chunk TMA-load S into a slot, read the
// accumulator, out = bf16(P + S) through a TMA tile store (and publish = P,
// when given, from the S slot the warp has just read), and drop the S lines
// from L2 (dead once read).  Returns false when the CTA aborts.
template <class C, int BN>
__device__ __forceinline__ void presum_epilogue(const KernelParams &p, const TensorMaps &tm, uint32_t sbase,
                                                uint32_t bar0, uint32_t tmem_base, int unit, int n_units,
                                                uint32_t crank, bool leader, int warp, int lane,
                                                volatile int *abort) {
    constexpr int PER_Q = 16;
    const int qd = warp & 3;
    const uint32_t wbase = sbase + C::OFF_EPI + (uint32_t)((warp - 2) * C::PS_WARP);
    const uint32_t sbar = bar0 + 8 * (C::BAR_SLD + (warp - 2) * C::PS_NSL);
    const bool pub = p.f32_out != nullptr;
    uint32_t ph = 0;       // parity of each S slot's next phase
    uint32_t pending = 0;  // S slots with a load in flight (lane 0's view)
    uint32_t tc = 0;
    auto drain = [&]() {
        if (lane == 0) {
            for (int b = 0; b < C::PS_NSL; ++b)
                if ((pending >> b) & 1u) bwait_drain(sbar + 8 * b, (ph >> b) & 1u, p);
            ptx::bulk_wait_all();
        }
        __syncwarp();
    };
    for (int i = 0;; ++i) {
        const int t = walk_entry(p, unit, n_units, i);
        if (t < 0) break;
        const int tile = tile_at(p, t, abort);
        if (tile < 0) break;
        const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
        const int acc = (int)(tc & 1u);
        const uint32_t aph = (tc >> 1) & 1u;
        bool ok = bwait<C::PAIR_>(bar0 + 8 * (C::BAR_TFULL + acc), aph, abort, p);
        if (!__all_sync(0xffffffffu, ok)) break;
        ptx::tc_fence_after();
        if (p.trace != nullptr && leader && warp == 2 && lane == 0) p.trace[5 * t + 2] = ptx::globaltimer();
        const int wrow0 = tmi * C::TILE_M + (int)crank * C::BM + qd * 32;  // this warp's first row
        const bool valid = wrow0 < p.M;
        const int row = wrow0 + lane;
        const int sy = wrow0 - p.red_row_off;
        const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * BN);
        const int ncc = live_chunks<BN>(p, tni);
        auto load_s = [&](int cc) {  // lane 0
            const int b = cc % C::PS_NSL;
            ptx::mbar_arrive_expect_tx(sbar + 8 * b, C::PS_SLOT);
            ptx::tma_load_2d(wbase + (uint32_t)(b * C::PS_SLOT), &tm.red, sbar + 8 * b, tni * BN + cc * 32, sy);
            pending |= 1u << b;
        };
        const uint32_t done_addr = sbase + C::OFF_PS_DONE + 4 * ((i % C::PS_NS) * 4 + qd);
        const uint32_t want = (uint32_t)(PER_Q * (i / C::PS_NS + 1));
        // this quadrant's S rows of the tile are complete; acknowledge, so
        // items of tile i + PS_NS may reuse the completion slot
        int st = 1;
        if (lane == 0) {
            st = wait_smem_at_least(done_addr, want, p, abort) ? 1 : 0;
            if (st) {
                ptx::st_release_cta_shared(sbase + C::OFF_PS_ACK + 4 * qd, (uint32_t)(i + 1));
                ptx::fence_proxy_async_global();  // the reducers' generic stores before the TMA loads
                if (valid)
                    for (int cc = 0; cc < C::PS_NSL && cc < ncc; ++cc) load_s(cc);
            }
        }
        st = __shfl_sync(0xffffffffu, st, 0);
        if (!st) break;
        bool dead = false;
#pragma unroll 1
        for (int cc = 0; cc < ncc; ++cc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
            ptx::tmem_ld_wait();
            if (!valid) continue;
            const int b = cc % C::PS_NSL;
            ok = bwait(sbar + 8 * b, (ph >> b) & 1u, abort, p);
            if (!__all_sync(0xffffffffu, ok)) {
                dead = true;
                break;
            }
            ph ^= 1u << b;
            if (lane == 0) pending &= ~(1u << b);
            const int col = tni * BN + cc * 32;
            const uint32_t srow = wbase + (uint32_t)(b * C::PS_SLOT) + (uint32_t)(lane * 128);
            float f[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t a = srow + ((uint32_t)(c ^ (lane & 7)) << 4);
                const float4 x = ptx::ld_shared_f4(a);
                f[4 * c + 0] = __uint_as_float(v[4 * c + 0]) + x.x;
                f[4 * c + 1] = __uint_as_float(v[4 * c + 1]) + x.y;
                f[4 * c + 2] = __uint_as_float(v[4 * c + 2]) + x.z;
                f[4 * c + 3] = __uint_as_float(v[4 * c + 3]) + x.w;
                if (pub)  // publish = P, into this lane's own row of the slot it has just read
                    ptx::st_shared_f4(a, __uint_as_float(v[4 * c + 0]), __uint_as_float(v[4 * c + 1]),
                                      __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
            }
            const uint32_t ob = wbase + (uint32_t)(C::PS_NSL * C::PS_SLOT + (cc & 1) * C::PS_OUT);
            if (lane == 0) ptx::bulk_wait_read<1>();  // the stores of chunk cc - 2 have read their slots
            __syncwarp();
            // row `lane` (64 bytes), 16-byte chunk c at position c ^ ((lane >> 1) & 3) (64-byte swizzle)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                ptx::st_shared_u4(ob + (uint32_t)(lane * 64) + ((uint32_t)(c ^ ((lane >> 1) & 3)) << 4),
                                  pack_bf16x2(f[8 * c], f[8 * c + 1]), pack_bf16x2(f[8 * c + 2], f[8 * c + 3]),
                                  pack_bf16x2(f[8 * c + 4], f[8 * c + 5]),
                                  pack_bf16x2(f[8 * c + 6], f[8 * c + 7]));
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (pub) ptx::tma_store_2d(&tm.f32out, wbase + (uint32_t)(b * C::PS_SLOT), col, wrow0);
                ptx::tma_store_2d(&tm.c, ob, col, wrow0);
                ptx::bulk_commit();
                if (cc + C::PS_NSL < ncc) {
                    if (pub) ptx::bulk_wait_read<0>();  // the publish store has read slot b
                    load_s(cc + C::PS_NSL);
                }
            }
            // this lane's S line of the chunk is dead: drop it from L2 unwritten
            // (only whole 128-byte lines: with N % 32 != 0 rows do not start on one)
            if (row < p.M && (p.N & 31) == 0 && col + 32 <= p.N)
                ptx::discard_l2_128(p.red_buf + (int64_t)(row - p.red_row_off) * p.N + col);
        }
        if (dead) {
            drain();
            break;
        }
        // release the accumulator (the even CTA's MMA waits for both CTAs)
        ptx::tc_fence_before();
        __syncwarp();
        const uint32_t tempty = bar0 + 8 * (C::BAR_TEMPTY + acc);
        if (lane == 0) {
            if (leader)
                ptx::mbar_arrive(tempty);
            else
                ptx::mbar_arrive_remote(ptx::mapa(tempty, 0));
        }
        if (p.trace != nullptr && leader && warp == 2 && lane == 0) p.trace[5 * t + 3] = ptx::globaltimer();
        if (pub) {
            // publish rows land before their chunk's produced flag
            if (lane == 0) {
                ptx::bulk_wait_all();
                ptx::fence_proxy_async();
            }
            __syncwarp();
            count_produced(p, tmi * C::TILE_M, C::TILE_M, C::CTAS, lane);
        }
        ++tc;
    }
    if (lane == 0) ptx::bulk_wait_all();  // every out store has landed before the CTA exits
    __syncwarp();
}

// ------------------------------------------------------------------ the kernel
template <int OP, int BN, int S, int BK, bool STG, bool PAIR, bool RED>
__global__ void __launch_bounds__(red_threads(OP, RED), 1)
    syn_fused_kernel(const __grid_constant__ KernelParams p, const __grid_constant__ TensorMaps tm) {
    using C = KCfg<OP, BN, S, BK, STG, PAIR, RED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(sm);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t t_start = ptx::globaltimer();

    // ---- dedicated staging CTA -------------------------------------------
    if ((int)blockIdx.x >= p.G) {
        ptx::grid_dep_wait();  // (programmatic launch) the previous grid's writes are visible
        ptx::grid_dep_launch_dependents();
        // COMM_NBUF independent copiers (threads 0..COMM_NBUF-1), each with its
        // own 32 KiB buffer and barrier, so several bulk copies are in flight.
        if (threadIdx.x == 0) {
            *abort = 0;
            for (int b = 0; b < C::COMM_NBUF; ++b) ptx::mbar_init(bar0 + 8 * b, 1);
            ptx::fence_mbar_init();
            ptx::fence_proxy_async_smem();
        }
        __syncthreads();
        if (p.push_dedicated) {  // GEMM-RS push mode: add produced send chunks at their destinations
            if ((int)threadIdx.x < C::COMM_NBUF) {
                const int c = (int)threadIdx.x;
                push_slices(p, tm, ((int)blockIdx.x - p.G) * C::COMM_NBUF + c, p.n_comm * C::COMM_NBUF,
                            sbase + c * C::COMM_BUF_BYTES, bar0 + 8 * c, abort);
            }
        } else if (p.ldst) {  // every warp copies with vector loads and stores
            constexpr int NW = C::NTHREADS / 32;
            stage_slices_ldst(p, ((int)blockIdx.x - p.G) * NW + warp, p.n_comm * NW, lane, abort);
        } else if ((int)threadIdx.x < C::COMM_NBUF) {
            const int c = (int)threadIdx.x;
            stage_slices(p, ((int)blockIdx.x - p.G) * C::COMM_NBUF + c, p.n_comm * C::COMM_NBUF,
                         sbase + c * C::COMM_BUF_BYTES, 1, C::COMM_BUF_BYTES, bar0 + 8 * c, abort);
        }
        __syncthreads();
        if constexpr (PAIR) ptx::cluster_sync();  // the pair's CTAs leave together
        return;
    }

    // rank in the CTA pair (0 = the CTA that issues the MMAs) and tile walk
    const uint32_t crank = PAIR ? ptx::cluster_ctarank() : 0u;
    const int unit = (int)blockIdx.x / C::CTAS;  // pair (or CTA) index
    const int n_units = p.G / C::CTAS;
    const bool leader = crank == 0;

    // ---- GEMM CTA set-up ---------------------------------------------------
    if (threadIdx.x == 0) {
        *abort = 0;
        if constexpr (RED) {
            for (int q = 0; q < 4; ++q)
                reinterpret_cast<volatile uint32_t *>(sm + C::OFF_RED_READY)[q] = 0u;
            *reinterpret_cast<volatile uint32_t *>(sm + C::OFF_RED_NEXT) = 0u;
            *reinterpret_cast<volatile uint32_t *>(sm + C::OFF_RED_TOTAL) = 0u;
        }
        if constexpr (C::PRESUM) {
            for (int q = 0; q < C::PS_NS * 4 + 4; ++q)
                reinterpret_cast<volatile uint32_t *>(sm + C::OFF_PS_DONE)[q] = 0u;
            for (int b = 0; b < 4 * C::PS_NSL; ++b) ptx::mbar_init(bar0 + 8 * (C::BAR_SLD + b), 1);
        }
        for (int s = 0; s < C::S; ++s) {
            ptx::mbar_init(bar0 + 8 * (C::BAR_FULL + s), 1);
            ptx::mbar_init(bar0 + 8 * (C::BAR_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar0 + 8 * (C::BAR_TFULL + a), 1);
            ptx::mbar_init(bar0 + 8 * (C::BAR_TEMPTY + a), 4 * C::CTAS);  // one per epilogue warp
        }
        ptx::mbar_init(bar0 + 8 * C::BAR_PEERDONE, 1);
        for (int s = 0; s < C::P; ++s) {
            ptx::mbar_init(bar0 + 8 * (C::BAR_PFULL + s), 1);
            ptx::mbar_init(bar0 + 8 * (C::BAR_PEMPTY + s), 4);
        }
        for (int s = 0; s < C::NSTG; ++s) ptx::mbar_init(bar0 + 8 * (C::BAR_STG + s), 1);
        ptx::mbar_init(bar0 + 8 * C::BAR_DRAIN, 1);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // both CTAs' barriers exist before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched with programmatic stream serialization, this grid may start while
    // the previous kernel on the stream still runs (on SMs it has left): the
    // set-up above touches only this CTA's shared memory and TMEM; everything
    // from here on may read what the previous grid wrote, so wait for it.  Then
    // let the next grid launch early too.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();
    // CTA 0 clears the counters of the other epoch parity for the next call.
    if (blockIdx.x == 0) {
        const int nf = p.n_rc * p.R;
        uint32_t *nin = p.in_cnt + (size_t)spare_half(p.epoch) * nf;
        uint32_t *nout = p.out_cnt + (size_t)spare_half(p.epoch) * p.n_rc;
        for (int i = threadIdx.x; i < nf; i += blockDim.x) nin[i] = 0u;
        for (int i = threadIdx.x; i < p.n_rc; i += blockDim.x) nout[i] = 0u;
    }

    unsigned long long wait_ns = 0;
    const int KB = (p.K + C::BK - 1) / C::BK;  // a partial last k-block reads zeros past K

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            const uint32_t sA = sbase + C::OFF_A, sB = sbase + C::OFF_B;
            uint32_t it = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int t = walk_entry(p, unit, n_units, i);
                if (t < 0) break;
                const int tile = tile_at(p, t, abort);
                if (tile < 0) break;
                const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
                const int r0 = tmi * C::TILE_M + (int)crank * C::BM;  // this CTA's rows
                // direct fetch: the source rank whose shard this tile's A rows
                // are read from in place (-1: the staged copy in `gathered`)
                int dq = -1;
                if (OP == OP_AG && p.waits) {
                    int lo, hi;
                    chunk_range(p, r0, C::BM, lo, hi);
                    if (p.direct_fetch && lo <= hi && lo / p.split == hi / p.split) {
                        const int q = lo / p.split;
                        bool ready = true;
                        for (int rc = lo; ready && rc <= hi; ++rc)
                            if (!(p.local_inplace && q == p.rank) && !chunk_empty(p.rb, rc))
                                ready = flag_ready(ptx::ld_acquire_gpu(p.in_flags + rc * p.R + q), p.epoch);
                        if (!ready) dq = q;  // every row lies in source q's block
                    }
                    if (dq < 0)
                        for (int rc = lo; ok && rc <= hi; ++rc) {
                            const int q = rc / p.split;
                            if ((p.local_inplace && q == p.rank) || chunk_empty(p.rb, rc)) continue;
                            ok = wait_flag(p.in_flags + rc * p.R + q, p, abort, WHERE_AG_FLAG,
                                           rc * p.R + q, wait_ns);
                        }
                    if (!ok) break;
                    ptx::fence_proxy_async();  // generic acquire -> async-proxy (TMA) reads
                }
                const CUtensorMap *amap = dq < 0 ? &tm.a : &tm.peer[dq];
                const int ay = dq < 0 ? r0 : r0 - (int)p.rb.off[dq];
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = (int)(it % C::S);
                    const uint32_t ph = (it / C::S) & 1u;
                    const uint32_t empty = bar0 + 8 * (C::BAR_EMPTY + s);
                    // wait until the pair's MMAs released the stage (its first use is
                    // free); the MMA commit arrives on this barrier in both CTAs
                    if (!bwait<PAIR>(empty, ph ^ 1u, abort, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar0 + 8 * (C::BAR_FULL + s);
                    const uint32_t a_dst = sA + s * C::A_BYTES, b_dst = sB + s * C::B_BYTES;
                    const int bcol = tni * BN + (int)crank * C::BN_CTA;
                    if (leader) {
                        // arm the phase that both CTAs' bytes complete
                        ptx::mbar_arrive_expect_tx(full, C::TX_BYTES);
                        ptx::tma_load_2d(a_dst, amap, full, kb * C::BK, ay);
#pragma unroll
                        for (int i = 0; i < C::BN_CTA / 64; ++i)
                            ptx::tma_load_2d(b_dst + i * C::B_BOX_BYTES, &tm.b, full, bcol + i * 64,
                                             kb * C::BK);
                    } else {
                        // the odd CTA's bytes complete on the even CTA's ring barrier
                        const uint32_t rfull = ptx::mapa(full, 0);
                        ptx::tma_load_2d_pair(a_dst, amap, rfull, kb * C::BK, ay);
#pragma unroll
                        for (int i = 0; i < C::BN_CTA / 64; ++i)
                            ptx::tma_load_2d_pair(b_dst + i * C::B_BOX_BYTES, &tm.b, rfull,
                                                  bcol + i * 64, kb * C::BK);
                    }
                }
            }
            // drain: every phase this CTA (or, PAIR, the odd CTA) loaded into must
            // have landed before the CTA may exit.  In a pair both producers wake
            // on the same MMA commit, so the odd CTA can be one use of a stage
            // ahead of the even CTA's arming; it reports how many k-blocks it
            // issued, and the even CTA arms any phase only the odd CTA loaded
            // into (with the odd CTA's bytes alone) before waiting for the last
            // phase of every stage.  The pair's closing cluster barrier keeps the
            // odd CTA alive until then.
            uint32_t it_all = it;
            if constexpr (PAIR) {
                uint32_t *peer_it = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC + 8);
                const uint32_t done = bar0 + 8 * C::BAR_PEERDONE;
                if (!leader) {
                    ptx::st_shared_cluster_u32(ptx::mapa(ptx::smem_u32(peer_it), 0), it);
                    ptx::mbar_arrive_remote(ptx::mapa(done, 0));
                } else {
                    bwait_drain<true>(done, 0, p);
                    const uint32_t it_p = *reinterpret_cast<volatile uint32_t *>(peer_it);
                    for (uint32_t s = 0; s < (uint32_t)C::S; ++s) {
                        const uint32_t uses_l = it > s ? (it - 1u - s) / C::S + 1u : 0u;
                        const uint32_t uses_p = it_p > s ? (it_p - 1u - s) / C::S + 1u : 0u;
                        if (uses_p > uses_l)
                            ptx::mbar_arrive_expect_tx(bar0 + 8 * (C::BAR_FULL + s), C::STAGE_BYTES);
                    }
                    it_all = it_p > it ? it_p : it;
                }
            }
            if (leader)
                for (uint32_t s = 0; s < (uint32_t)C::S; ++s) {
                    if (it_all > s) {
                        const uint32_t last = s + ((it_all - 1u - s) / C::S) * C::S;
                        bwait_drain<PAIR>(bar0 + 8 * (C::BAR_FULL + s), (last / C::S) & 1u, p);
                    }
                }
        }
    } else if (warp == 1) {
        // ================= MMA issuer (the pair's even CTA) =================
        if (lane == 0 && leader) {
            const uint32_t sA = sbase + C::OFF_A, sB = sbase + C::OFF_B;
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int t = walk_entry(p, unit, n_units, i);
                if (t < 0) break;
                const int acc = (int)(tc & 1u);
                const uint32_t aph = (tc >> 1) & 1u;
                if (!bwait<PAIR>(bar0 + 8 * (C::BAR_TEMPTY + acc), aph ^ 1u, abort, p)) break;
                ptx::tc_fence_after();
                if (p.trace != nullptr) {
                    p.trace[5 * t + 0] = ptx::globaltimer();
                    p.trace[5 * t + 4] = (unsigned long long)unit;
                }
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = (int)(it % C::S);
                    const uint32_t ph = (it / C::S) & 1u;
                    if (!bwait<PAIR>(bar0 + 8 * (C::BAR_FULL + s), ph, abort, p)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = sA + s * C::A_BYTES, b0 = sB + s * C::B_BYTES;
#pragma unroll
                    for (int k = 0; k < C::BK / C::UK; ++k) {
                        // A: K-major, 128- or 64-byte swizzle (BK 64 / 32); SBO = next
                        // 8-row atom; a 16-wide K slice is +32 bytes inside the row
                        const uint64_t ad = ptx::sdesc(a0 + k * 32, 16, C::A_SBO, C::A_SWZ);
                        // B: N-major, 128-byte swizzle; LBO = next 64-column box,
                        // SBO = next 8 K-rows; a 16-deep K slice is +16 rows of 128 B
                        const uint64_t bd =
                            ptx::sdesc(b0 + k * 2048, C::B_BOX_BYTES, 1024, ptx::kSwizzle128B);
                        if constexpr (PAIR)
                            ptx::umma_bf16_pair(d, ad, bd, C::IDESC, (kb | k) != 0 ? 1u : 0u);
                        else
                            ptx::umma_bf16(d, ad, bd, C::IDESC, (kb | k) != 0 ? 1u : 0u);
                    }
                    if constexpr (PAIR) {
                        // the stage is free in both CTAs once these MMAs completed:
                        // commit to each CTA's ring barrier directly
                        ptx::umma_commit_pair(bar0 + 8 * (C::BAR_EMPTY + s));
                        ptx::umma_commit_pair(ptx::mapa(bar0 + 8 * (C::BAR_EMPTY + s), 1));
                    } else {
                        ptx::umma_commit(bar0 + 8 * (C::BAR_EMPTY + s));
                    }
                }
                if (!ok) break;
                if constexpr (PAIR) {
                    ptx::umma_commit_pair(bar0 + 8 * (C::BAR_TFULL + acc));
                    ptx::umma_commit_pair(ptx::mapa(bar0 + 8 * (C::BAR_TFULL + acc), 1));
                } else {
                    ptx::umma_commit(bar0 + 8 * (C::BAR_TFULL + acc));
                }
                if (p.trace != nullptr) p.trace[5 * t + 1] = ptx::globaltimer();
                ++tc;
            }
            // every MMA this thread issued must finish before TMEM is released
            if constexpr (PAIR)
                ptx::umma_commit_pair(bar0 + 8 * C::BAR_DRAIN);
            else
                ptx::umma_commit(bar0 + 8 * C::BAR_DRAIN);
            bwait_drain(bar0 + 8 * C::BAR_DRAIN, 0, p);
        }
    } else if (warp >= 2 && warp < 6 && C::PRESUM) {
        // ================= epilogue: pre-summed GEMM-AR =================
        if constexpr (C::PRESUM)
            presum_epilogue<C, BN>(p, tm, sbase, bar0, tmem_base, unit, n_units, crank, leader, warp, lane,
                                   abort);
    } else if (warp >= 2 && warp < 6) {
        // ================= epilogue =================
        const int qd = warp & 3;  // TMEM lane quadrant this warp may access
        const int lrow = qd * 32 + lane;
        uint32_t tc = 0, pit = 0, red_done = 0;
        const uint32_t sPeer = sbase + C::OFF_PEER;
        for (int i = 0;; ++i) {
            const int t = walk_entry(p, unit, n_units, i);
            if (t < 0) break;
            const int tile = tile_at(p, t, abort);
            if (tile < 0) break;
            const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
            const int acc = (int)(tc & 1u);
            const uint32_t aph = (tc >> 1) & 1u;
            const uint32_t tfull = bar0 + 8 * (C::BAR_TFULL + acc);
            bool ok = bwait<PAIR>(tfull, aph, abort, p);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            if (p.trace != nullptr && leader && warp == 2 && lane == 0)
                p.trace[5 * t + 2] = ptx::globaltimer();
            const int tr0 = tmi * C::TILE_M;                       // tile's first row
            const int row = tr0 + (int)crank * C::BM + lrow;       // this thread's row
            const bool in_range = row < p.M;
            // red: this CTA's rows of the tile reduce (it takes the peer ring, or
            // hands its quadrants to the reducer warps); wl: this warp's 32 rows
            // are reduced rather than sent (GEMM-RS: local-block rows; a tile may
            // straddle the block's edge)
            const bool red = reduces<OP>(p, tr0 + (int)crank * C::BM, C::BM);
            const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * BN);
            bool dead = false;
            // fp32 store of this tile (at most one): send / publish, or (RED) the
            // reducing tile's partial; with EPI_TMA through this warp's staging
            // buffers and TMA tile stores of its 32 rows
            const int wrow0 = tr0 + (int)crank * C::BM + qd * 32;  // this warp's first row
            const bool wl = local_row<OP>(p, wrow0);
            const CUtensorMap *fmap = nullptr;
            int fy = 0;
            if constexpr (C::EPI_TMA && OP == OP_AG) {
                if (p.epi_tma && wrow0 < p.M) fmap = &tm.c;
            } else if constexpr (C::EPI_TMA) {
                if (p.epi_tma && wrow0 < p.M) {
                    if (p.f32_out != nullptr && (OP == OP_AR || !wl)) {
                        fmap = &tm.f32out;
                        fy = wrow0;
                    } else if (RED && wl && p.red_buf != p.f32_out) {
                        fmap = &tm.red;
                        fy = wrow0 - p.red_row_off;
                    }
                }
            }
            const uint32_t ebuf = sbase + C::OFF_EPI + (uint32_t)((warp - 2) * 2 * C::EPI_SLOT);
            const int ncc = live_chunks<BN>(p, tni);
#pragma unroll 1
            for (int cc = 0; cc < ncc; ++cc) {
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
                ptx::tmem_ld_wait();
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                const int col = tni * BN + cc * 32;
                if constexpr (OP == OP_AG) {
                    if (C::EPI_TMA && fmap != nullptr) {
                        {
                            const uint32_t buf = ebuf + (uint32_t)((cc & 1) * C::EPI_SLOT);
                            if (lane == 0) ptx::bulk_wait_read<1>();  // the store of chunk cc - 2 read it
                            __syncwarp();
                            // row `lane` (64 bytes), 16-byte chunk c at position c ^ ((lane >> 1) & 3)
                            // (64-byte swizzle)
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                ptx::st_shared_u4(buf + (uint32_t)(lane * 64) +
                                                      ((uint32_t)(c ^ ((lane >> 1) & 3)) << 4),
                                                  pack_bf16x2(f[8 * c], f[8 * c + 1]),
                                                  pack_bf16x2(f[8 * c + 2], f[8 * c + 3]),
                                                  pack_bf16x2(f[8 * c + 4], f[8 * c + 5]),
                                                  pack_bf16x2(f[8 * c + 6], f[8 * c + 7]));
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d(&tm.c, buf, col, wrow0);
                                ptx::bulk_commit();
                            }
                        }
                    } else if (in_range) {
                        store_bf16_row32(p.out + (int64_t)row * p.N + col, f, p.N - col);
                    }
                    continue;
                } else {
                if (C::EPI_TMA && fmap != nullptr) {
                    {
                        const uint32_t buf = ebuf + (uint32_t)((cc & 1) * C::EPI_SLOT);
                        if (lane == 0) ptx::bulk_wait_read<1>();  // the store of chunk cc - 2 read it
                        __syncwarp();
                        // row `lane`, 16-byte chunk c at position c ^ (lane & 7) (128-byte swizzle)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            ptx::st_shared_f4(buf + (uint32_t)(lane * 128) + ((uint32_t)(c ^ (lane & 7)) << 4),
                                              f[4 * c], f[4 * c + 1], f[4 * c + 2], f[4 * c + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // GEMM-RS push mode: send rows are added into the
                            // destination's receive accumulator
                            if (OP == OP_RS && !wl && p.send_push)
                                ptx::tma_reduce_add_2d(fmap, buf, col, fy);
                            else
                                ptx::tma_store_2d(fmap, buf, col, fy);
                            ptx::bulk_commit();
                        }
                    }
                } else {
                    if (p.f32_out != nullptr && in_range && (OP == OP_AR || !wl))
                        store_f32_row32(p.f32_out + (int64_t)row * p.N + col, f, p.N - col);
                    if (RED && wl && in_range && p.red_buf != p.f32_out)
                        store_f32_row32(p.red_buf + (int64_t)(row - p.red_row_off) * p.N + col, f, p.N - col);
                }
                if constexpr (RED) {
                    continue;  // the reducer warps add the peers to the stored partial
                } else {
                if (!red) continue;
                // S = peer sum in ascending q, then out = P + S
                float sacc[32];
                bool first = true;
                for (int q = 0; q < p.R; ++q) {
                    if (q == p.rank) continue;
                    const int slot = (int)(pit % C::P);
                    const uint32_t ph = (pit / C::P) & 1u;
                    bool okp = bwait(bar0 + 8 * (C::BAR_PFULL + slot), ph, abort, p);
                    if (!__all_sync(0xffffffffu, okp)) {
                        dead = true;
                        break;
                    }
                    // 128 rows x 128 B, 128-byte swizzle: 16-byte chunk c of row r sits
                    // at chunk position c ^ (r & 7)
                    const uint32_t rowaddr = sPeer + slot * C::PEER_BYTES + lrow * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 x = ptx::ld_shared_f4(rowaddr + ((uint32_t)(c ^ (lrow & 7)) << 4));
                        if (first) {
                            sacc[4 * c + 0] = x.x;
                            sacc[4 * c + 1] = x.y;
                            sacc[4 * c + 2] = x.z;
                            sacc[4 * c + 3] = x.w;
                        } else {
                            sacc[4 * c + 0] = sacc[4 * c + 0] + x.x;
                            sacc[4 * c + 1] = sacc[4 * c + 1] + x.y;
                            sacc[4 * c + 2] = sacc[4 * c + 2] + x.z;
                            sacc[4 * c + 3] = sacc[4 * c + 3] + x.w;
                        }
                    }
                    first = false;
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar0 + 8 * (C::BAR_PEMPTY + slot));
                    ++pit;
                }
                if (dead) break;
                if (!first) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) f[j] = f[j] + sacc[j];
                }
                if (in_range && wl) {
                    const int orow = OP == OP_RS ? row - p.rank * p.M_r : row;
                    store_bf16_row32(p.out + (int64_t)orow * p.N + col, f, p.N - col);
                }
                }  // !RED
                }  // OP != OP_AG
            }
            // release the accumulator: one arrive per warp once all its lanes'
            // TMEM loads completed (the even CTA's MMA waits for both CTAs)
            ptx::tc_fence_before();
            __syncwarp();
            const uint32_t tempty = bar0 + 8 * (C::BAR_TEMPTY + acc);
            if (lane == 0) {
                if (leader)
                    ptx::mbar_arrive(tempty);
                else
                    ptx::mbar_arrive_remote(ptx::mapa(tempty, 0));
            }
            if (p.trace != nullptr && leader && warp == 2 && lane == 0)
                p.trace[5 * t + 3] = ptx::globaltimer();
            if constexpr (C::EPI_TMA) {
                // the tile's TMA stores must have landed before its chunk flags or
                // the reducer hand-off publish them (the accumulator is already free)
                if (fmap != nullptr && lane == 0) {
                    ptx::bulk_wait_all();
                    ptx::fence_proxy_async();
                }
                __syncwarp();
            }
            if (dead) break;
            if constexpr (RED) {
                if (red) {
                    // this quadrant's rows of the partial are stored: hand them to
                    // the reducer warp of the same quadrant
                    __threadfence_block();
                    __syncwarp();
                    if (lane == 0) {
                        ++red_done;
                        ptx::st_release_cta_shared(sbase + C::OFF_RED_READY + 4 * qd, red_done);
                    }
                }
            }
            if (OP != OP_AG && p.f32_out != nullptr && (OP == OP_AR || sends<OP>(p, tr0, C::TILE_M)))
                count_produced(p, tr0, C::TILE_M, C::CTAS, lane);
            ++tc;
        }
        if constexpr (RED) {
            // every reducing tile of the walk has been seen (or the CTA aborted)
            __syncwarp();
            if (lane == 0) ptx::st_release_cta_shared(sbase + C::OFF_RED_TOTAL, red_done + 1u);
        }
    } else if (warp == 6) {
        // ================= peer loader (GEMM-RS / GEMM-AR) =================
        if constexpr (OP != OP_AG && !RED) if (lane == 0) {
            const uint32_t sPeer = sbase + C::OFF_PEER;
            uint32_t pit = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int t = walk_entry(p, unit, n_units, i);
                if (t < 0) break;
                const int tile = tile_at(p, t, abort);
                if (tile < 0) break;
                const int tmi = tile / p.tiles_n, tni = tile - tmi * p.tiles_n;
                const int tr0 = tmi * C::TILE_M;
                const int r0 = tr0 + (int)crank * C::BM;  // this CTA's rows
                if (!reduces<OP>(p, r0, C::BM)) continue;
                if (p.waits) {
                    // the chunks of the rows this CTA reduces (GEMM-RS: its local-block rows)
                    int a = r0, b = r0 + C::BM;
                    if (OP == OP_RS) {
                        a = max(a, p.rank * p.M_r);
                        b = min(b, (p.rank + 1) * p.M_r);
                    }
                    int lo, hi;
                    chunk_range(p, a, b - a, lo, hi);
                    for (int rc = lo; ok && rc <= hi; ++rc)
                        for (int q = 0; ok && q < p.R; ++q) {
                            if (q == p.rank) continue;
                            ok = wait_flag(p.in_flags + rc * p.R + q, p, abort, WHERE_PEER_FLAG,
                                           rc * p.R + q, wait_ns);
                        }
                    if (!ok) break;
                    ptx::fence_proxy_async();
                }
                const int prow = r0 - p.peer_row_off;
                const int ncc = live_chunks<BN>(p, tni);
                for (int cc = 0; ok && cc < ncc; ++cc) {
                    for (int q = 0; q < p.R; ++q) {
                        if (q == p.rank) continue;
                        const int slot = (int)(pit % C::P);
                        const uint32_t ph = (pit / C::P) & 1u;
                        if (!bwait(bar0 + 8 * (C::BAR_PEMPTY + slot), ph ^ 1u, abort, p)) {
                            ok = false;
                            break;
                        }
                        const uint32_t full = bar0 + 8 * (C::BAR_PFULL + slot);
                        ptx::mbar_arrive_expect_tx(full, C::PEER_BYTES);
                        ptx::tma_load_2d(sPeer + slot * C::PEER_BYTES, &tm.peer[q], full,
                                         tni * BN + cc * 32, prow);
                        ++pit;
                    }
                }
            }
            for (uint32_t s = 0; s < (uint32_t)C::P; ++s) {
                if (pit > s) {
                    const uint32_t last = s + ((pit - 1u - s) / C::P) * C::P;
                    bwait_drain(bar0 + 8 * (C::BAR_PFULL + s), (last / C::P) & 1u, p);
                }
            }
        }
    } else if (warp == 7) {
        // ================= co-located stager =================
        if (p.colocated && p.ldst) stage_slices_ldst(p, (int)blockIdx.x, p.G, lane, abort);
        if constexpr (C::NSTG > 0)
            // one copier per CTA, double-buffered: with one worker per GEMM CTA the
            // first round of slices covers only the earliest chunks in arrival order
            if (p.colocated && lane == 0)
                stage_slices(p, (int)blockIdx.x, p.G, sbase + C::OFF_STG, C::NSTG, C::STG_BYTES,
                             bar0 + 8 * C::BAR_STG, abort);
    }
    // ================= reducers (RED) =================
    // warps 8 on from the start, the others once their own role is done.
    // Warps 6-7 have no role here: GEMM-AR, whose reduction outlasts the MMAs,
    // puts them to work at once; GEMM-RS, whose few reducing tiles run early
    // beside MMAs that need the memory system, keeps them out.
    if constexpr (C::PRESUM) {
        __syncwarp();
        presum_worker<C, BN>(p, sm, sbase, unit, n_units, crank, lane, abort);
    } else if constexpr (RED) {
        if (OP == OP_AR || (warp != 6 && warp != 7)) {
            __syncwarp();
            reduce_worker<C, OP, BN>(p, sm, sbase, unit, n_units, crank, lane, abort);
        }
    }

    // ---- teardown -----------------------------------------------------------
    if (p.stats != nullptr && wait_ns != 0ull) atomicAdd(p.stats + 0, wait_ns);
    ptx::tc_fence_before();
    __syncthreads();
    // the pair leaves together: no remote arrive may target a CTA that has exited,
    // and the even CTA's drain above covered the odd CTA's in-flight loads
    if constexpr (PAIR) ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && p.stats != nullptr)
        atomicAdd(p.stats + 1, (unsigned long long)(ptx::globaltimer() - t_start));
}

template <int OP, int BN, int S, int BK, bool STG, bool PAIR, bool RED>
cudaError_t launch_fused_t(const KernelParams &p, const TensorMaps &tm, int grid, cudaStream_t st,
                           bool overlap_prev) {
    using C = KCfg<OP, BN, S, BK, STG, PAIR, RED>;
    auto kern = syn_fused_kernel<OP, BN, S, BK, STG, PAIR, RED>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = st;
    // Single CTAs: a cooperative launch, which fails rather than run a grid
    // whose CTAs cannot all be resident.  CTA pairs: a 2-CTA cluster launch
    // whose grid the host sized to the co-resident cluster count
    // (cudaOccupancyMaxActiveClusters), so every CTA is resident as well; were
    // one not, the bounded waits would end the call in SYN_ERR_TIMEOUT.
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 1;
    if (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        if (overlap_prev) {
            // the kernel waits for the previous grid (griddepcontrol.wait) before
            // touching global memory, so its launch and set-up may overlap it
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            n_attr = 2;
        }
    } else {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, kern, p, tm);
}

// Co-resident 2-CTA clusters of one instance (0 when the query fails).
template <int OP, int BN, int S, int BK, bool STG, bool PAIR, bool RED>
int max_clusters_t() {
    using C = KCfg<OP, BN, S, BK, STG, PAIR, RED>;
    auto kern = syn_fused_kernel<OP, BN, S, BK, STG, PAIR, RED>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Every compiled kernel instance, per operator: (tile_m, tile_n, stages,
// tile_k, stg, red).  tile_m 256 is the CTA-pair kernel.  `Fn` receives the
// KCfg type; returns false when the combination is not compiled.
template <int OP, typename Fn>
bool dispatch_cfg(const LaunchCfg &lc, Fn &&fn) {
    const int tn = lc.tile_n, st = lc.stages, tk = lc.tile_k;
    const bool g = lc.stg, pr = lc.pair, rd = lc.red;
#define SYN_CFG_R(PR, TN, ST, TK, G, RD)                                           \
    if (pr == PR && tn == TN && st == ST && tk == TK && g == G && rd == RD)        \
        return fn(KCfg<OP, TN, ST, TK, G, PR, RD>{}), true;
#define SYN_CFG(PR, TN, ST, TK, G) SYN_CFG_R(PR, TN, ST, TK, G, false)
    if constexpr (OP == OP_AG) {
        SYN_CFG(false, 256, 4, 64, true) SYN_CFG(false, 256, 4, 64, false)
        SYN_CFG(false, 128, 6, 64, true) SYN_CFG(false, 128, 6, 64, false)
        SYN_CFG(false, 256, 8, 32, true) SYN_CFG(false, 256, 9, 32, false)
        SYN_CFG(true, 256, 6, 64, true) SYN_CFG(true, 256, 7, 64, false)
        SYN_CFG(true, 256, 5, 64, true) SYN_CFG(true, 256, 5, 64, false)
        SYN_CFG(true, 256, 4, 64, true)
        return false;
    } else {
        SYN_CFG(false, 256, 3, 64, true) SYN_CFG(false, 128, 4, 64, true) SYN_CFG(false, 256, 6, 32, true)
        SYN_CFG(false, 256, 2, 64, false) SYN_CFG(false, 256, 3, 64, false) SYN_CFG(false, 256, 4, 64, false)
        SYN_CFG(false, 128, 3, 64, false) SYN_CFG(false, 128, 4, 64, false) SYN_CFG(false, 128, 6, 64, false)
        SYN_CFG(false, 256, 4, 32, false) SYN_CFG(false, 256, 5, 32, false) SYN_CFG(false, 256, 6, 32, false)
        SYN_CFG(true, 256, 4, 64, true)
        SYN_CFG(true, 256, 3, 64, false) SYN_CFG(true, 256, 4, 64, false) SYN_CFG(true, 256, 5, 64, false)
        SYN_CFG(true, 256, 6, 64, false)
        if constexpr (OP == OP_RS) {
            SYN_CFG_R(false, 256, 4, 64, false, true)
            SYN_CFG_R(true, 256, 4, 64, false, true)
            SYN_CFG_R(true, 256, 5, 64, false, true) SYN_CFG_R(true, 256, 6, 64, false, true)
            SYN_CFG_R(true, 256, 7, 64, false, true)
        } else {
            // pre-summed GEMM-AR: the epilogue's S and out slots need 48 KB
            SYN_CFG_R(false, 256, 3, 64, false, true)
            SYN_CFG_R(true, 256, 3, 64, false, true) SYN_CFG_R(true, 256, 4, 64, false, true)
            SYN_CFG_R(true, 256, 5, 64, false, true)
        }
        return false;
    }
#undef SYN_CFG
#undef SYN_CFG_R
}

template <int OP>
cudaError_t launch_op(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                      cudaStream_t st) {
    cudaError_t err = cudaErrorInvalidValue;
    dispatch_cfg<OP>(lc, [&](auto c) {
        using C = decltype(c);
        err = launch_fused_t<OP, C::BN_, C::S, C::BK, C::STG_, C::PAIR_, C::RED_>(p, tm, lc.grid, st,
                                                                                lc.overlap_prev);
    });
    return err;
}

template <int OP>
int smem_bytes_op(const LaunchCfg &lc) {
    int bytes = -1;
    dispatch_cfg<OP>(lc, [&](auto c) { bytes = decltype(c)::SMEM_ALLOC; });
    return bytes;
}

// 1 when the instance stages its epilogue stores through TMA, 0 when not,
// -1 when it is not compiled.
template <int OP>
int epi_tma_op(const LaunchCfg &lc) {
    int e = -1;
    dispatch_cfg<OP>(lc, [&](auto c) { e = decltype(c)::EPI_TMA ? 1 : 0; });
    return e;
}

template <int OP>
int max_clusters_op(const LaunchCfg &lc) {
    int n = 0;
    dispatch_cfg<OP>(lc, [&](auto c) {
        using C = decltype(c);
        if constexpr (C::PAIR_) n = max_clusters_t<OP, C::BN_, C::S, C::BK, C::STG_, C::PAIR_, C::RED_>();
    });
    return n;
}

}  // namespace syn
