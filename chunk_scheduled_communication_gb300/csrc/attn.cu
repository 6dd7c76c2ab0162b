// attn.cu -- fused ring attention forward (sequence parallelism) whose KV
// loop walks the staged chunks in arrival order, and the C ABI of
// include/syn_attn.h.
//
// Syncopate summary page, Experiments (paper §6.1: head-/sequence-parallel
// attention and RingAttention) and method ¶2-¶4 (a tile waits only for the
// chunks it reads; tiles follow the communication order).  A persistent CTA
// (one per SM, a cooperative launch) takes work items of one head and two
// 128-row query tiles (t = 0, 1) in turn and computes them on the tensor
// cores, KV block by KV block (128 keys) in chunk-arrival order:
//
//   warp 0      TMA producer: an item's Q tiles, then for each KV block:
//               wait for the chunk flags of its rows, load K and V into a
//               two-slot ring
//   warps 1, 3  MMA issuers, one per tile: S_t = Q_t.K^T into the tile's
//               TMEM score buffer (two 64-key halves), then O_t += P_t.V
//   warp 2      staging: copy the other ranks' KV chunks, publish flags
//   warps 4-7   softmax of tile 0 (one query row per thread, its TMEM lane)
//   warps 8-11  softmax of tile 1
//
// TMEM (512 columns): S_t at 128t, O_t at 256 + 128t.  The softmax writes
// the bf16 probabilities over the upper 64 columns of the tile's score
// buffer, where P.V reads them as a TMEM operand.  A tile's Q.K^T of block
// g+1 runs in two 64-key halves: the lower half as soon as the softmax has
// loaded the scores of block g into registers, the upper half once P.V of
// block g has read the probabilities.  The two tiles take turns at the
// exponentials (tile 1's of block g after tile 0's, tile 0's of block g+1
// after tile 1's of block g), so one tile's MMAs run while the other's
// softmax does and neither shares the exp2 unit.  The
// exponentials use a reference max that may lag the row's true max by up to
// 8 (log2 units, so every p <= 2^8): only when a block raises it by more is
// the tile's TMEM accumulator (and sum) rescaled, between two P.V products.
// The softmax warps hold 200 registers each, the other warps 96 (setmaxnreg).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "host_util.h"
#include "protocol.h"
#include "ptx.cuh"
#include "syn.h"
#include "syn_attn.h"

namespace syn {
namespace attn {

constexpr int kD = 128;                      // head dimension
constexpr int kBQ = 128;                     // query rows per tile
constexpr int kTiles = 2;                    // query tiles per work item
constexpr int kBK = 128;                     // keys per KV block
constexpr int kTileBytes = 128 * 128 * 2;    // one 128 x 128 bf16 tile: two 64-wide boxes
constexpr int kBoxBytes = kTileBytes / 2;    // 128 rows x 128 bytes, 128-byte swizzle
constexpr int OFF_Q = 0;                     // kTiles tiles
constexpr int OFF_K = OFF_Q + kTiles * kTileBytes;  // 2 slots
constexpr int OFF_V = OFF_K + 2 * kTileBytes;
constexpr int OFF_BAR = OFF_V + 2 * kTileBytes;
enum {
    B_QF = 0,      // the item's Q tiles landed
    B_QE = 1,      // Q tiles read by the item's last Q.K^T
    B_KF = 2,      // K slot s landed (2)
    B_KE = 4,      // K slot s consumed by both tiles' Q.K^T (2; one commit per tile's issuer)
    B_VF = 6,      // V slot s landed (2)
    B_VE = 8,      // V slot s consumed by both tiles' P.V (2; one commit per tile's issuer)
    B_SF = 10,     // tile t's scores written (2)
    B_PF = 12,     // tile t's probabilities written over its scores (2)
    B_PV = 14,     // tile t's P.V done: O_t updated, its score buffer free (2)
    B_OE = 16,     // tile t's accumulator read out after an item's last P.V (2)
    B_DRAIN = 18,  // every MMA of tile t's issuer completed (2)
    B_XD = 20,     // tile t's exponentials of a block done (2): the tiles take turns
    B_SL = 22,     // tile t's scores loaded into the softmax registers (2)
    N_BAR = 24
};
constexpr int OFF_MISC = OFF_BAR + 8 * N_BAR;  // TMEM base, abort flag
constexpr int OFF_SEEN = OFF_MISC + 16;        // chunks the producer has acquired this call: 512 bits
constexpr int SMEM_USED = OFF_SEEN + 64;
constexpr int NTHREADS = 384;
constexpr int SMEM_BYTES = SMEM_USED + 1024;   // + the 1024-byte alignment of the tiles
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(128, 64, false);   // B = 64 keys of the K tile, K-major
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, 128, true);   // A = P in TMEM, B = V tile, MN-major
constexpr int WHERE_FLAG = 1, WHERE_PIPE = 3;

struct Params {
    // ring mode: Q [S_r, H_q, d] local, queries at global positions rank*S_r + i;
    // head mode: Q gathered [R*S_r, H_q, d] (H_q = the local query heads),
    // queries at positions i, their rows waited for like the keys'
    int32_t R, rank, S_r, H_q, G, causal, split, n_qtiles, n_items;
    int32_t head_mode, q_pos0;  // q_pos0: global position of Q row 0
    int32_t local_inplace, waits;
    float scale_log2;  // scale * log2(e)
    uint32_t epoch;
    uint64_t timeout_ns;
    const uint32_t *flags;  // [R * split]
    uint16_t *out;          // [S_r, H_q, d]
    float *lse;             // [S_r, H_q] or null
    int32_t *err;           // {code, site, CTA, info}
    // in-kernel staging (stage = 1): warp 2 of every CTA copies the other
    // ranks' chunks into the gathered buffers in arrival order.  Tensor x
    // (K, V, and in head mode Q): row i of source q's chunk rows copies
    // width[x] bytes from src[x][q] + i * src_pitch[x] + src_off[x] to
    // dst[x] + (q * S_r + i) * width[x]; slices of slice_rows[x] rows
    int32_t stage, n_transfers, n_tensors, drop_transfer;
    int32_t slice_rows[3], slices_of[3];  // slices per chunk of tensor x (the largest chunk)
    int64_t src_pitch[3], src_off[3], width[3];
    const uint8_t *src[3][8];
    uint8_t *dst[3];
    uint32_t *flags_w;      // the same flags, written by the stagers
    uint32_t *cnt;          // [2][R * split] slice counters (epoch parity)
};

struct Maps {
    CUtensorMap q, k, v;
};

__device__ __forceinline__ void raise(const Params &p, int code, int where, int info) {
    if (atomicCAS(p.err, 0, code) == 0) {
        p.err[1] = where;
        p.err[2] = (int)blockIdx.x;
        p.err[3] = info;
    }
}

// Bounded wait on a shared-memory barrier phase; false on abort or timeout.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort, const Params &p) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if ((n & 63u) == 0u) {
            if (*reinterpret_cast<volatile int32_t *>(p.err) != 0) {
                *abort = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > limit) {
                raise(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)bar);
                *abort = 1;
                return false;
            }
        }
    }
}

// Wait used while draining on the way out: ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, const Params &p) {
    const uint64_t t0 = ptx::globaltimer();
    const uint64_t limit = p.timeout_ns * 4ull + 200000000ull;
    for (uint32_t n = 0;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return;
        if ((n & 63u) == 63u && ptx::globaltimer() - t0 > limit) {
            raise(p, SYN_ERR_TIMEOUT, WHERE_PIPE, (int)bar);
            return;
        }
    }
}

// Acquire-wait until chunk `code`'s flag carries this call's epoch.
__device__ __forceinline__ bool wait_chunk(const Params &p, int code, volatile int *abort) {
    const uint32_t *f = p.flags + code;
    if (flag_ready(ptx::ld_acquire_gpu(f), p.epoch)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        __nanosleep(64);
        if (flag_ready(ptx::ld_acquire_gpu(f), p.epoch)) return true;
        if (*abort) return false;
        if ((n & 15u) == 0u) {
            if (*reinterpret_cast<volatile int32_t *>(p.err) != 0) {
                *abort = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > p.timeout_ns) {
                raise(p, SYN_ERR_TIMEOUT, WHERE_FLAG, code);
                *abort = 1;
                return false;
            }
        }
    }
}

// Source rank and chunk of staging transfer a (arrival order: the local shard
// when it is not in place, then ranks r+1, r+2, ..., chunks ascending).
__device__ __forceinline__ void transfer_of(const Params &p, int a, int &q, int &j) {
    const int idx = a / p.split;
    j = a - idx * p.split;
    q = (p.rank + idx + (p.local_inplace ? 1 : 0)) % p.R;
}

// Stager warp `worker` of `n_workers`: slices worker, worker + n_workers, ...
// of the transfer list (per transfer: slices_of[0] slices of tensor 0, then
// tensor 1's, ...), each a warp-wide copy of up to slice_rows rows of one
// tensor of a chunk; the warp that completes a transfer's last slice
// publishes its flag (release) once every slice's bytes are visible.
__device__ void stage_chunks(const Params &p, int worker, int n_workers, int lane) {
    int spt = 0;
    for (int x = 0; x < p.n_tensors; ++x) spt += p.slices_of[x];
    const int nf = p.R * p.split;
    uint32_t *cnt = p.cnt + (size_t)counter_half(p.epoch) * nf;
    const int total = p.n_transfers * spt;
    for (int g = worker; g < total; g += n_workers) {
        const int a = g / spt;
        int sl = g - a * spt, x = 0;
        while (sl >= p.slices_of[x]) sl -= p.slices_of[x++];
        int q, j;
        transfer_of(p, a, q, j);
        const int64_t lo = ((int64_t)j * p.S_r + p.split - 1) / p.split;
        const int64_t hi = ((int64_t)(j + 1) * p.S_r + p.split - 1) / p.split;
        const int64_t r0 = lo + (int64_t)sl * p.slice_rows[x];
        const int64_t r1 = r0 + p.slice_rows[x] < hi ? r0 + p.slice_rows[x] : hi;
        const int64_t w = p.width[x];
        const int vpr = (int)(w / 16);  // 16-byte vectors per row
        const uint8_t *src = p.src[x][q] + p.src_off[x] + r0 * p.src_pitch[x];
        uint8_t *dst = p.dst[x] + ((int64_t)q * p.S_r + r0) * w;
        const int nvec = r0 < r1 ? (int)(r1 - r0) * vpr : 0;
        if (p.src_pitch[x] == w) {  // whole rows: one contiguous span
            const int64_t len = (int64_t)nvec * 16;
            for (int64_t b = (int64_t)lane * 16; b < len; b += 32 * 16 * 8) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (b + u * 512 < len) v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + b + u * 512));
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (b + u * 512 < len) *reinterpret_cast<uint4 *>(dst + b + u * 512) = v[u];
            }
        } else
        // eight 16-byte vectors in flight per lane (4 KB per warp round); a
        // lane's vectors are 32 apart, so its (row, column) advances by adds
        for (int b = lane; b < nvec; b += 32 * 8) {
            const int row0 = b / vpr, col0 = b - row0 * vpr;
            uint4 v[8];
            int row = row0, col = col0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b + u * 32 < nvec)
                    v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)row * p.src_pitch[x] + col * 16));
                col += 32;
                while (col >= vpr) {
                    col -= vpr;
                    ++row;
                }
            }
            row = row0;
            col = col0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b + u * 32 < nvec) *reinterpret_cast<uint4 *>(dst + (int64_t)row * w + col * 16) = v[u];
                col += 32;
                while (col >= vpr) {
                    col -= vpr;
                    ++row;
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            ptx::fence_acq_rel_gpu();  // the warp's stores, observed through the barrier, before the count
            const int code = q * p.split + j;
            const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt + code, 1u);
            if (completes_transfer(old, (uint32_t)spt) && a != p.drop_transfer)
                ptx::st_release_gpu(p.flags_w + code, p.epoch);
        }
        __syncwarp();
    }
}

// Acquire (once per call and CTA: `seen` is the producer's bitmap) the flags
// of the chunks holding gathered rows [row0, row0 + 128); false on timeout.
__device__ __forceinline__ bool acquire_rows(const Params &p, int row0, uint32_t *seen, volatile int *abort) {
    const int src = row0 / p.S_r;
    if (!p.waits || (p.local_inplace && src == p.rank)) return true;
    const int lr0 = row0 - src * p.S_r;
    const int lo = (int)(((int64_t)lr0 * p.split) / p.S_r);
    const int hi = (int)(((int64_t)(lr0 + kBK - 1) * p.split) / p.S_r);
    bool fresh = false;
    for (int c = lo; c <= hi; ++c) {
        const int code = src * p.split + c;
        if (seen[code >> 5] & (1u << (code & 31))) continue;
        if (!wait_chunk(p, code, abort)) return false;
        seen[code >> 5] |= 1u << (code & 31);
        fresh = true;
    }
    if (fresh) ptx::fence_proxy_async();  // generic acquire -> async-proxy (TMA) reads
    return true;
}

// The KV blocks a query tile visits, in chunk-arrival order: the shards of
// ranks r, r+1, ..., r-1, each shard's blocks in ascending order.  Causal:
// a block whose first key lies after the tile's last query is skipped (and
// so are the shard's later blocks).
struct KvIter {
    int t, b, nb, last;
    __device__ __forceinline__ void init(const Params &p, int q_row0) {
        t = 0;
        b = 0;
        nb = p.S_r / kBK;
        last = p.causal ? p.q_pos0 + q_row0 + kTiles * kBQ - 1 : 0x7fffffff;
    }
    // first global key row of the next block, -1 past the end
    __device__ __forceinline__ int next(const Params &p) {
        while (t < p.R) {
            const int q = (p.rank + t) % p.R;
            if (b < nb) {
                const int kv0 = q * p.S_r + b * kBK;
                ++b;
                if (kv0 <= last) return kv0;
                b = nb;
                continue;
            }
            ++t;
            b = 0;
        }
        return -1;
    }
};

// One step of a CTA's persistent walk: work item (query head, query tile)
// item = blockIdx.x, + gridDim.x, ... (head-major, so concurrently running
// CTAs share KV heads in L2), and the KV blocks of each item in order.
struct Blk {
    int h, q_row0, kv0;
    bool first, last;
};
struct Walk {
    int item, nxt;
    bool fresh;  // the next block is its item's first
    KvIter it;
    __device__ __forceinline__ void start(const Params &p) {
        fresh = true;
        nxt = -1;
        if (item < p.n_items) {
            it.init(p, (item % p.n_qtiles) * kTiles * kBQ);
            nxt = it.next(p);
        }
    }
    __device__ __forceinline__ void init(const Params &p) {
        item = (int)blockIdx.x;
        start(p);
    }
    __device__ __forceinline__ bool next(const Params &p, Blk &b) {
        while (item < p.n_items && nxt < 0) {  // (every item has a block: its diagonal one)
            item += (int)gridDim.x;
            start(p);
        }
        if (item >= p.n_items) return false;
        b.h = item / p.n_qtiles;
        b.q_row0 = (item - b.h * p.n_qtiles) * kTiles * kBQ;
        b.kv0 = nxt;
        b.first = fresh;
        fresh = false;
        nxt = it.next(p);
        b.last = nxt < 0;
        if (b.last) {
            item += (int)gridDim.x;
            start(p);
        }
        return true;
    }
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (f32x2 arithmetic: one instruction for two lanes of work)
// and a three-input max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unf2(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Descriptors of a 128 x 128 bf16 tile held as two 64-wide, 128-byte-swizzled
// boxes.  K-major (Q, K, P): 16-element slice kk lies in box kk/4, 32 bytes
// per slice inside the swizzled row; 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return ptx::sdesc(tile + (uint32_t)(kk >> 2) * kBoxBytes + (uint32_t)(kk & 3) * 32u, 16, 1024,
                      ptx::kSwizzle128B);
}
// MN-major (V as the B operand: K = keys along rows, N = d across the two
// boxes): slice kk is rows 16kk..16kk+15 (2048 bytes on), the boxes kBoxBytes apart.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return ptx::sdesc(tile + (uint32_t)kk * 2048u, kBoxBytes, 1024, ptx::kSwizzle128B);
}

constexpr float kRescale = 8.f;  // how far (log2 units) the reference max may lag

// The finished output row: the accumulator read from TMEM, normalised by l,
// stored as bf16; and its log-sum-exp.
__device__ __forceinline__ void store_row(const Params &p, uint32_t to, float m, float l, int h, int row_g) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((int64_t)row_g * p.H_q + h) * kD);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(to + (uint32_t)(c * 32), v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 o;
            o.x = pack_bf16(__uint_as_float(v[8 * k + 0]) * inv, __uint_as_float(v[8 * k + 1]) * inv);
            o.y = pack_bf16(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv);
            o.z = pack_bf16(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv);
            o.w = pack_bf16(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv);
            dst[c * 4 + k] = o;
        }
    }
    if (p.lse != nullptr)  // natural log: (m + log2 l) * ln 2, m in log2-scaled units
        p.lse[(int64_t)row_g * p.H_q + h] = (m + log2f(l)) * 0.69314718055994531f;
}

// Register split (setmaxnreg): the launch gives 168 registers per thread
// (384 threads); the producer, MMA and staging warps give theirs down to 96
// and the two softmax warpgroups take 200: 128 * 96 + 256 * 200 = 63,488 of
// the 64,512 launched.
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 96;"); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 200;"); }

__global__ void __launch_bounds__(NTHREADS, 1) ring_attn_kernel(const __grid_constant__ Params p,
                                                                const __grid_constant__ Maps m) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(sm);
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        *abort = 0;
        ptx::mbar_init(bar(B_QF), 1);
        ptx::mbar_init(bar(B_QE), kTiles);  // each tile's issuer commits once
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(B_KF + s), 1);
            ptx::mbar_init(bar(B_KE + s), kTiles);
            ptx::mbar_init(bar(B_VF + s), 1);
            ptx::mbar_init(bar(B_VE + s), kTiles);
            ptx::mbar_init(bar(B_SF + s), 1);
            ptx::mbar_init(bar(B_PF + s), 4);  // the tile's four softmax warps
            ptx::mbar_init(bar(B_PV + s), 1);
            ptx::mbar_init(bar(B_OE + s), 4);
            ptx::mbar_init(bar(B_DRAIN + s), 1);
            ptx::mbar_init(bar(B_XD + s), 4);  // the tile's four softmax warps
            ptx::mbar_init(bar(B_SL + s), 4);
        }
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // CTA 0 clears the slice counters of the other epoch parity for the next call
    if (p.stage && blockIdx.x == 0)
        for (int i = (int)threadIdx.x; i < p.R * p.split; i += (int)blockDim.x)
            p.cnt[(size_t)spare_half(p.epoch) * p.R * p.split + i] = 0u;
    if (warp < 4) {
        regs_dec();
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            const uint32_t sQ = sbase + OFF_Q, sK = sbase + OFF_K, sV = sbase + OFF_V;
            uint32_t *seen = reinterpret_cast<uint32_t *>(sm + OFF_SEEN);
            for (int i = 0; i < 16; ++i) seen[i] = 0u;
            Walk wk;
            wk.init(p);
            Blk b;
            uint32_t g = 0, ic = 0, nk = 0, nv = 0;
            for (; wk.next(p, b); ++g) {
                const int hk = b.h / p.G;
                if (b.first) {
                    // the item's Q tiles (gathered queries: once their chunks are in)
                    // replace the previous ones once that item's last Q.K^T completed
                    bool ok = true;
                    for (int t = 0; ok && p.head_mode && t < kTiles; ++t)
                        ok = acquire_rows(p, b.q_row0 + t * kBQ, seen, abort);
                    if (!ok || !wait_bar(bar(B_QE), (ic & 1u) ^ 1u, abort, p)) break;
                    ptx::mbar_arrive_expect_tx(bar(B_QF), kTiles * kTileBytes);
                    for (int t = 0; t < kTiles; ++t) {
                        ptx::tma_load_2d(sQ + t * kTileBytes, &m.q, bar(B_QF), b.h * kD, b.q_row0 + t * kBQ);
                        ptx::tma_load_2d(sQ + t * kTileBytes + kBoxBytes, &m.q, bar(B_QF), b.h * kD + 64,
                                         b.q_row0 + t * kBQ);
                    }
                    ++ic;
                }
                if (!acquire_rows(p, b.kv0, seen, abort)) break;
                const int s = (int)(g & 1u);
                const uint32_t ph = (g >> 1) & 1u;
                if (!wait_bar(bar(B_KE + s), ph ^ 1u, abort, p)) break;
                ptx::mbar_arrive_expect_tx(bar(B_KF + s), kTileBytes);
                ptx::tma_load_2d(sK + s * kTileBytes, &m.k, bar(B_KF + s), hk * kD, b.kv0);
                ptx::tma_load_2d(sK + s * kTileBytes + kBoxBytes, &m.k, bar(B_KF + s), hk * kD + 64, b.kv0);
                ++nk;
                if (!wait_bar(bar(B_VE + s), ph ^ 1u, abort, p)) break;
                ptx::mbar_arrive_expect_tx(bar(B_VF + s), kTileBytes);
                ptx::tma_load_2d(sV + s * kTileBytes, &m.v, bar(B_VF + s), hk * kD, b.kv0);
                ptx::tma_load_2d(sV + s * kTileBytes + kBoxBytes, &m.v, bar(B_VF + s), hk * kD + 64, b.kv0);
                ++nv;
            }
            // every load issued must land before the CTA exits
            if (ic > 0) drain_bar(bar(B_QF), (ic - 1u) & 1u, p);
            for (uint32_t s = 0; s < 2; ++s) {
                if (nk > s) drain_bar(bar(B_KF + (int)s), ((s + ((nk - 1u - s) / 2u) * 2u) >> 1) & 1u, p);
                if (nv > s) drain_bar(bar(B_VF + (int)s), ((s + ((nv - 1u - s) / 2u) * 2u) >> 1) & 1u, p);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ================= MMA issuers: warp 1 for tile 0, warp 3 for tile 1 =================
        // Tile t's chain is Q.K^T(g) -> softmax -> P.V(g) -> Q.K^T(g+1) (the
        // probabilities live in the tile's score buffer).  Each tile has its own
        // issuing thread, so neither tile's next MMA queues behind the other
        // tile's waits; a K or V slot is free once both issuers have committed it.
        if (lane == 0) {
            const int t = warp == 1 ? 0 : 1;
            const uint32_t sQ = sbase + OFF_Q, sK = sbase + OFF_K, sV = sbase + OFF_V;
            const uint32_t d_s = tmem + (uint32_t)(t * 128);         // S_t, then P_t
            const uint32_t d_o = tmem + 256u + (uint32_t)(t * 128);  // O_t
            const uint32_t q_t = sQ + (uint32_t)(t * kTileBytes);
            // S_t = Q_t . K_g^T (K slot g & 1) in two halves of 64 keys: the lower
            // half (score columns 0-63) once the softmax has loaded S(g-1), the
            // upper half (columns 64-127, where P(g-1) lives) once P.V(g-1) read it
            auto qk_half = [&](uint32_t g, int half) -> bool {
                const int s = (int)(g & 1u);
                if (half == 0) {
                    if (!wait_bar(bar(B_KF + s), (g >> 1) & 1u, abort, p)) return false;
                    if (g > 0 && !wait_bar(bar(B_SL + t), (g - 1u) & 1u, abort, p)) return false;
                } else if (g > 0 && !wait_bar(bar(B_PV + t), (g - 1u) & 1u, abort, p)) {
                    return false;
                }
                ptx::tc_fence_after();
                const uint32_t k_h = sK + s * kTileBytes + (uint32_t)half * 8192u;  // key rows 64*half..
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    ptx::umma_bf16(d_s + (uint32_t)(half * 64), kmajor_desc(q_t, kk), kmajor_desc(k_h, kk), IDESC_QK,
                                   kk != 0 ? 1u : 0u);
                if (half == 1) {
                    ptx::umma_commit(bar(B_SF + t));
                    ptx::umma_commit(bar(B_KE + s));
                }
                return true;
            };
            // O_t (+)= P_t . V_g, P_t from TMEM (8 columns per 16 keys); an item's
            // first product overwrites O_t once the previous item (`item` - 1)
            // has been read out
            auto pv = [&](uint32_t g, bool first, uint32_t item) -> bool {
                const int s = (int)(g & 1u);
                if (!wait_bar(bar(B_PF + t), g & 1u, abort, p)) return false;
                if (!wait_bar(bar(B_VF + s), (g >> 1) & 1u, abort, p)) return false;
                if (first && item > 0 && !wait_bar(bar(B_OE + t), (item - 1u) & 1u, abort, p)) return false;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    ptx::umma_bf16_ts(d_o, d_s + 64u + (uint32_t)(kk * 8), mnmajor_desc(sV + s * kTileBytes, kk), IDESC_PV,
                                      (kk != 0 || !first) ? 1u : 0u);
                ptx::umma_commit(bar(B_PV + t));
                ptx::umma_commit(bar(B_VE + s));
                return true;
            };
            Walk wk;
            wk.init(p);
            Blk cur, nxt;
            bool ok = true, has = wk.next(p, cur);
            uint32_t g = 0, ic = 0, item_cur = 0;
            if (has) {  // prologue: the first block's Q.K^T
                ok = wait_bar(bar(B_QF), 0u, abort, p);
                ic = 1;
                if (ok) ok = qk_half(0, 0);
                if (ok) ok = qk_half(0, 1);
                if (ok && cur.last) ptx::umma_commit(bar(B_QE));
            }
            while (ok && has) {
                const bool has_next = wk.next(p, nxt);
                if (has_next && nxt.first) {  // a new item: its Q tiles
                    if (!wait_bar(bar(B_QF), ic & 1u, abort, p)) break;
                    ++ic;
                }
                if (has_next) ok = qk_half(g + 1u, 0);
                if (ok) ok = pv(g, cur.first, item_cur);
                if (ok && has_next) ok = qk_half(g + 1u, 1);
                if (!ok) break;
                if (has_next && nxt.last) ptx::umma_commit(bar(B_QE));  // the item's Q tile is no longer read
                if (has_next && nxt.first) ++item_cur;
                cur = nxt;
                has = has_next;
                ++g;
            }
            // every MMA issued must complete before TMEM is released
            ptx::umma_commit(bar(B_DRAIN + t));
            drain_bar(bar(B_DRAIN + t), 0, p);
        }
    } else {
        // ================= stager (warp 2) =================
        if (p.stage) stage_chunks(p, (int)blockIdx.x, (int)gridDim.x, lane);
    }
    } else {
        regs_inc();
        // ================= softmax of tile t, output rescaling, epilogue =================
        const int t = (warp - 4) >> 2;
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        const uint32_t ts = tl + (uint32_t)(t * 128);         // the tile's scores (then probabilities)
        const uint32_t to = tl + 256u + (uint32_t)(t * 128);  // the tile's output accumulator
        float mref = -INFINITY, lrow = 0.f;  // reference max (log2-scaled units), running sum
        Walk wk;
        wk.init(p);
        Blk b;
        for (uint32_t g = 0; wk.next(p, b); ++g) {
            if (b.first) {
                mref = -INFINITY;
                lrow = 0.f;
            }
            bool w = wait_bar(bar(B_SF + t), g & 1u, abort, p);
            if (!__all_sync(0xffffffffu, w)) break;
            ptx::tc_fence_after();
            const int qrow = b.q_row0 + t * kBQ;                      // the tile's first query row
            const int qpos0 = p.q_pos0 + qrow;                        // its global position
            const int qpos = qpos0 + row;                             // this row's
            const bool masked = p.causal && b.kv0 + kBK - 1 > qpos0;  // the block crosses the diagonal
            uint32_t v[kBK];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                ptx::tmem_ld_32x32b_x32(ts + (uint32_t)(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
            ptx::tmem_ld_wait();
            // the scores are in registers: the next block's lower half may overwrite them
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_SL + t));
            if (masked) {
#pragma unroll
                for (int k = 0; k < kBK; ++k)
                    if (b.kv0 + k > qpos) v[k] = __float_as_uint(-INFINITY);
            }
            // row max: eight interleaved partials, two new scores per three-input max
            float mp[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mp[k] = __uint_as_float(v[k]);
#pragma unroll
            for (int k = 8; k < kBK; k += 2)
                mp[(k >> 1) & 7] = max3(mp[(k >> 1) & 7], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
            const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
            const float mcand = mx * p.scale_log2;  // (scale > 0: the max commutes with it)
            // a new reference max: the item's first block, or a rise of more than kRescale
            const bool need = !b.first && mcand > mref + kRescale;
            const float alpha = need ? ex2(mref - mcand) : 1.f;
            if (b.first || need) mref = mcand;
            if (__any_sync(0xffffffffu, need)) {
                // P.V(g-1) completed before this block's Q.K^T could overwrite the
                // scores, so the accumulator is stable: rescale it
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(to + (uint32_t)(c * 32), o);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    ptx::tmem_st_32x32b_x32(to + (uint32_t)(c * 32), o);
                }
            }
            // the tiles take turns at the exponentials (tile 1's of block g after tile
            // 0's, tile 0's of block g+1 after tile 1's of block g), so each runs them
            // alone while the other tile's products run on the tensor pipe
            if (t == 1 || g > 0) {
                w = wait_bar(bar(B_XD + (1 - t)), (t == 1 ? g : g - 1u) & 1u, abort, p);
                if (!__all_sync(0xffffffffu, w)) break;
            }
            const float base = mref == -INFINITY ? 0.f : mref;
            // probabilities: the exponent arguments and the running sums two keys at
            // a time (f32x2), four interleaved pair-sums
            const uint64_t scale2 = f2(p.scale_log2, p.scale_log2), nbase2 = f2(-base, -base);
            uint64_t sp[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) sp[k] = f2(0.f, 0.f);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // probabilities of 64 keys, as bf16 pairs in 32 columns
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 64; k += 2) {
                    float x0, x1;
                    unf2(fma2(f2(__uint_as_float(v[hh * 64 + k]), __uint_as_float(v[hh * 64 + k + 1])), scale2, nbase2),
                         x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    sp[(k >> 1) & 3] = add2(sp[(k >> 1) & 3], f2(p0, p1));
                    pk[k >> 1] = pack_bf16(p0, p1);
                }
                ptx::tmem_st_32x32b_x32(ts + 64u + (uint32_t)(hh * 32), pk);
            }
            float s0, s1, s2, s3, s4, s5, s6, s7;
            unf2(sp[0], s0, s1);
            unf2(sp[1], s2, s3);
            unf2(sp[2], s4, s5);
            unf2(sp[3], s6, s7);
            const float sum = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
            lrow = lrow * alpha + sum;
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bar(B_PF + t));
                ptx::mbar_arrive(bar(B_XD + t));
            }
            if (b.last) {  // the item's output, after the tile's last P.V
                w = wait_bar(bar(B_PV + t), g & 1u, abort, p);
                if (!__all_sync(0xffffffffu, w)) break;
                ptx::tc_fence_after();
                store_row(p, to, mref, lrow, b.h, qrow + row);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_OE + t));
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace attn
}  // namespace syn

using namespace syn;
using namespace syn::attn;

struct syn_attn_plan_s {
    syn_attn_cfg_t cfg;
    int device = 0, num_sms = 0;
    int n_qtiles = 0, grid = 0;
    uint32_t epoch = 0;
    uint32_t *d_flags = nullptr;
    uint32_t *d_cnt = nullptr;
    int32_t *d_err = nullptr;
    Maps maps;
    std::vector<const void *> map_key;
};

namespace {

void free_attn(syn_attn_plan_s *pl) {
    if (pl == nullptr) return;
    cudaFree(pl->d_flags);
    cudaFree(pl->d_cnt);
    cudaFree(pl->d_err);
    delete pl;
}

bool al16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }


}  // namespace

#define ATT_CK(call)                                                                                  \
    do {                                                                                              \
        cudaError_t e__ = (call);                                                                     \
        if (e__ != cudaSuccess) return host_fail(SYN_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e__)); \
    } while (0)

extern "C" {

int syn_attn_cfg_default(syn_attn_cfg_t *c) {
    if (c == nullptr) return host_fail(SYN_ERR_INVALID, "null cfg");
    std::memset(c, 0, sizeof(*c));
    c->R = 1;
    c->S_r = 256;
    c->H_q = c->H_kv = 1;
    c->d = 128;
    c->split = 1;
    c->backend = SYN_BACKEND_TMA_COLOCATED;
    c->debug_drop_chunk = -1;
    c->head_parallel = 0;
    return SYN_OK;
}

int syn_attn_plan_create(syn_attn_plan_t *out, const syn_attn_cfg_t *cfg) {
    if (out == nullptr || cfg == nullptr) return host_fail(SYN_ERR_INVALID, "null argument");
    *out = nullptr;
    syn_attn_cfg_t c = *cfg;
    if (c.split == 0) c.split = 1;
    if (c.R < 1 || c.rank < 0 || c.rank >= c.R) return host_fail(SYN_ERR_INVALID, "need 0 <= rank < R");
    if (c.R > 8) return host_fail(SYN_ERR_UNSUPPORTED, "R > 8");
    if (c.d != kD) return host_fail(SYN_ERR_UNSUPPORTED, "head dimension must be 128");
    if (c.S_r < kTiles * kBQ || c.S_r % (kTiles * kBQ) != 0)
        return host_fail(SYN_ERR_UNSUPPORTED, "S_r must be a positive multiple of 256");
    if (c.S_r > (1 << 20)) return host_fail(SYN_ERR_UNSUPPORTED, "S_r > 2^20");
    if (c.H_q < 1 || c.H_kv < 1 || c.H_q % c.H_kv != 0) return host_fail(SYN_ERR_INVALID, "need H_q % H_kv == 0");
    if (c.H_q > 1024) return host_fail(SYN_ERR_UNSUPPORTED, "H_q > 1024");
    if (c.causal != 0 && c.causal != 1) return host_fail(SYN_ERR_INVALID, "causal must be 0 or 1");
    if (c.split < 1 || c.split > 64 || c.split > c.S_r / kBK)  // (R * split <= 512 chunk bits)
        return host_fail(SYN_ERR_INVALID, "split must be in [1, min(64, S_r/128)]");
    if (c.backend != SYN_BACKEND_TMA_COLOCATED && c.backend != SYN_BACKEND_UNFUSED)
        return host_fail(SYN_ERR_UNSUPPORTED,
                         "ring attention stages with SYN_BACKEND_TMA_COLOCATED or SYN_BACKEND_UNFUSED");
    if (!(c.scale >= 0.f) || !std::isfinite(c.scale)) return host_fail(SYN_ERR_INVALID, "bad scale");
    int rc = host_load_driver();
    if (rc != SYN_OK) return rc;
    syn_attn_plan_s *pl = new syn_attn_plan_s();
    pl->cfg = c;
    if (pl->cfg.scale == 0.f) pl->cfg.scale = 1.f / std::sqrt((float)kD);
    if (pl->cfg.timeout_ns == 0) pl->cfg.timeout_ns = host_timeout_ns();
    if (c.head_parallel != 0 && c.head_parallel != 1) return host_fail(SYN_ERR_INVALID, "head_parallel must be 0 or 1");
    if (c.head_parallel && (c.H_q % c.R != 0 || c.H_kv % c.R != 0))
        return host_fail(SYN_ERR_INVALID, "head-parallel attention needs H_q and H_kv divisible by R");
    pl->n_qtiles = (int)((c.head_parallel ? c.R * c.S_r : c.S_r) / kBQ);
    auto bail = [&](int code, const std::string &msg) {
        free_attn(pl);
        return host_fail(code, msg);
    };
#define PL_CK(call)                                                                                 \
    do {                                                                                            \
        cudaError_t e__ = (call);                                                                   \
        if (e__ != cudaSuccess) return bail(SYN_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e__)); \
    } while (0)
    PL_CK(cudaGetDevice(&pl->device));
    PL_CK(cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device));
    PL_CK(cudaFuncSetAttribute(ring_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    int per_sm = 0;
    PL_CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_attn_kernel, NTHREADS, SMEM_BYTES));
    if (per_sm < 1) return bail(SYN_ERR_UNSUPPORTED, "the attention kernel cannot be resident");
    // persistent: one CTA per SM (all co-resident: a cooperative launch), at
    // most one per work item
    pl->grid = std::min(pl->n_qtiles / kTiles * (c.head_parallel ? c.H_q / c.R : c.H_q), pl->num_sms * per_sm);
    const size_t nf = (size_t)c.R * c.split;
    PL_CK(cudaMalloc(&pl->d_flags, nf * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_flags, 0, nf * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_cnt, 2 * nf * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_cnt, 0, 2 * nf * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_err, 4 * sizeof(int32_t)));
    PL_CK(cudaMemset(pl->d_err, 0, 4 * sizeof(int32_t)));
    PL_CK(cudaDeviceSynchronize());
#undef PL_CK
    *out = pl;
    return SYN_OK;
}

int syn_attn_plan_destroy(syn_attn_plan_t plan) {
    free_attn(plan);
    return SYN_OK;
}

}  // extern "C"

namespace {

// One call of either mode.  Ring: Q local [S_r, H_q, d], K/V shards staged
// whole; head: Q/K/V shards [S_r, H, d] of which the local heads' columns
// are staged into gathered [R*S_r, H_loc, d] buffers.
int attn_call(syn_attn_plan_s *pl, bool head, const void *Q, const void *const *Q_shards,
              const void *const *K_shards, const void *const *V_shards, void *Q_gathered, void *K_gathered,
              void *V_gathered, void *O, float *lse, void *stream) {
    if (pl == nullptr) return host_fail(SYN_ERR_INVALID, "null plan");
    const syn_attn_cfg_t &c = pl->cfg;
    if ((c.head_parallel != 0) != head)
        return host_fail(SYN_ERR_INVALID, "the plan was made for the other attention layout");
    const void *Qk = head ? Q_gathered : Q;  // the queries the kernel reads
    if (Qk == nullptr || K_shards == nullptr || V_shards == nullptr || K_gathered == nullptr ||
        V_gathered == nullptr || O == nullptr || (head && Q_shards == nullptr))
        return host_fail(SYN_ERR_INVALID, "null operand");
    if (!al16(Qk) || !al16(K_gathered) || !al16(V_gathered) || !al16(O) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return host_fail(SYN_ERR_INVALID, "operand not 16-byte aligned");
    for (int q = 0; q < c.R; ++q)
        if (K_shards[q] == nullptr || V_shards[q] == nullptr || !al16(K_shards[q]) || !al16(V_shards[q]) ||
            (head && (Q_shards[q] == nullptr || !al16(Q_shards[q]))))
            return host_fail(SYN_ERR_INVALID, "shard pointer null or not 16-byte aligned");
    const int hq = head ? c.H_q / c.R : c.H_q;    // query heads the kernel computes
    const int hkv = head ? c.H_kv / c.R : c.H_kv;  // KV heads in the gathered buffers
    const int64_t n_qrows = head ? (int64_t)c.R * c.S_r : c.S_r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t kv_w = (int64_t)hkv * kD * 2;      // gathered K/V row bytes
    const int64_t shard_bytes = c.S_r * kv_w;
    uint8_t *kg = static_cast<uint8_t *>(K_gathered), *vg = static_cast<uint8_t *>(V_gathered);
    const bool inplace = !head && K_shards[c.rank] == kg + c.rank * shard_bytes &&
                         V_shards[c.rank] == vg + c.rank * shard_bytes;
    std::vector<const void *> key = {Qk, K_gathered, V_gathered};
    if (key != pl->map_key) {
        int rc;
        if ((rc = host_encode_2d(&pl->maps.q, Qk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)hq * kD,
                                 (uint64_t)n_qrows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != SYN_OK ||
            (rc = host_encode_2d(&pl->maps.k, K_gathered, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)hkv * kD,
                                 (uint64_t)c.R * c.S_r, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != SYN_OK ||
            (rc = host_encode_2d(&pl->maps.v, V_gathered, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)hkv * kD,
                                 (uint64_t)c.R * c.S_r, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != SYN_OK)
            return rc;
        pl->map_key = key;
    }
    pl->epoch += 1;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.R = c.R;
    p.rank = c.rank;
    p.S_r = (int32_t)c.S_r;
    p.H_q = hq;
    p.G = hq / hkv;
    p.causal = c.causal;
    p.split = c.split;
    p.n_qtiles = pl->n_qtiles / kTiles;  // (the kernel's items per head: tile pairs)
    p.n_items = p.n_qtiles * hq;
    p.head_mode = head ? 1 : 0;
    p.q_pos0 = head ? 0 : c.rank * (int32_t)c.S_r;
    p.local_inplace = inplace ? 1 : 0;
    p.scale_log2 = c.scale * 1.4426950408889634f;
    p.epoch = pl->epoch;
    p.timeout_ns = c.timeout_ns;
    p.flags = pl->d_flags;
    p.flags_w = pl->d_flags;
    p.cnt = pl->d_cnt;
    p.out = static_cast<uint16_t *>(O);
    p.lse = lse;
    p.err = pl->d_err;
    p.n_transfers = (c.R - (inplace ? 1 : 0)) * c.split;
    p.drop_transfer = c.debug_drop_chunk;
    // staged tensors: K, V (and Q in head mode); a source row holds every head,
    // the gathered row only the local ones
    const void *const *srcs[3] = {K_shards, V_shards, Q_shards};
    void *dsts[3] = {K_gathered, V_gathered, Q_gathered};
    const int heads_src[3] = {c.H_kv, c.H_kv, c.H_q}, heads_loc[3] = {hkv, hkv, hq};
    p.n_tensors = head ? 3 : 2;
    const int64_t max_rows = (c.S_r + c.split - 1) / c.split;
    for (int x = 0; x < p.n_tensors; ++x) {
        p.width[x] = (int64_t)heads_loc[x] * kD * 2;
        p.src_pitch[x] = (int64_t)heads_src[x] * kD * 2;
        p.src_off[x] = head ? (int64_t)c.rank * heads_loc[x] * kD * 2 : 0;
        p.slice_rows[x] = (int32_t)std::max<int64_t>(1, (64 * 1024) / p.width[x]);
        p.slices_of[x] = (int32_t)((max_rows + p.slice_rows[x] - 1) / p.slice_rows[x]);
        for (int q = 0; q < c.R; ++q) p.src[x][q] = static_cast<const uint8_t *>(srcs[x][q]);
        p.dst[x] = static_cast<uint8_t *>(dsts[x]);
    }
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    lc.gridDim = dim3((unsigned)pl->grid, 1, 1);
    lc.blockDim = dim3(NTHREADS, 1, 1);
    lc.dynamicSmemBytes = SMEM_BYTES;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: stagers and waiters coexist
    attr[0].val.cooperative = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (c.backend == SYN_BACKEND_TMA_COLOCATED) {
        p.stage = 1;
        p.waits = 1;
    } else {  // unfused: every copy first (in stream order), then the kernel without waits
        for (int t = 0; t < c.R; ++t) {
            const int q = (c.rank + t) % c.R;
            if (q == c.rank && inplace) continue;
            for (int x = 0; x < p.n_tensors; ++x)
                ATT_CK(cudaMemcpy2DAsync(static_cast<uint8_t *>(dsts[x]) + (int64_t)q * c.S_r * p.width[x],
                                         (size_t)p.width[x], p.src[x][q] + p.src_off[x], (size_t)p.src_pitch[x],
                                         (size_t)p.width[x], (size_t)c.S_r, cudaMemcpyDeviceToDevice, st));
        }
        p.stage = 0;
        p.waits = 0;
    }
    ATT_CK(cudaLaunchKernelEx(&lc, ring_attn_kernel, p, pl->maps));
    return SYN_OK;
}

}  // namespace

extern "C" {

int syn_ring_attention(syn_attn_plan_t pl, const void *Q, const void *const *K_shards,
                       const void *const *V_shards, void *K_gathered, void *V_gathered, void *O, float *lse,
                       void *stream) {
    return attn_call(pl, false, Q, nullptr, K_shards, V_shards, nullptr, K_gathered, V_gathered, O, lse, stream);
}

int syn_head_attention(syn_attn_plan_t pl, const void *const *Q_shards, const void *const *K_shards,
                       const void *const *V_shards, void *Q_gathered, void *K_gathered, void *V_gathered,
                       void *O, float *lse, void *stream) {
    return attn_call(pl, true, nullptr, Q_shards, K_shards, V_shards, Q_gathered, K_gathered, V_gathered, O,
                     lse, stream);
}

int syn_attn_sync_status(syn_attn_plan_t pl, void *stream) {
    if (pl == nullptr) return host_fail(SYN_ERR_INVALID, "null plan");
    ATT_CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int32_t e[4] = {0, 0, 0, 0};
    ATT_CK(cudaMemcpy(e, pl->d_err, sizeof(e), cudaMemcpyDeviceToHost));
    if (e[0] == 0) return SYN_OK;
    ATT_CK(cudaMemset(pl->d_err, 0, 4 * sizeof(int32_t)));
    ATT_CK(cudaMemset(pl->d_flags, 0, (size_t)pl->cfg.R * pl->cfg.split * sizeof(uint32_t)));
    ATT_CK(cudaMemset(pl->d_cnt, 0, 2 * (size_t)pl->cfg.R * pl->cfg.split * sizeof(uint32_t)));
    ATT_CK(cudaDeviceSynchronize());
    return host_fail(e[0], std::string("device error ") + syn_status_string(e[0]) + " at site " +
                               std::to_string(e[1]) + " in CTA " + std::to_string(e[2]) + " (info " +
                               std::to_string(e[3]) + ")");
}

int syn_attn_plan_query(syn_attn_plan_t pl, syn_attn_info_t *info) {
    if (pl == nullptr || info == nullptr) return host_fail(SYN_ERR_INVALID, "null argument");
    std::memset(info, 0, sizeof(*info));
    const syn_attn_cfg_t &c = pl->cfg;
    info->R = c.R;
    info->rank = c.rank;
    info->H_q = c.H_q;
    info->H_kv = c.H_kv;
    info->d = c.d;
    info->causal = c.causal;
    info->split = c.split;
    info->backend = c.backend;
    info->S_r = c.S_r;
    info->n_qtiles = pl->n_qtiles;
    info->grid = pl->grid;
    info->n_transfers = (c.head_parallel ? c.R : c.R - 1) * c.split;  // (ring: the local shard in place)
    info->smem_bytes = SMEM_BYTES;
    info->epoch = pl->epoch;
    return SYN_OK;
}

int syn_attn_plan_flags(syn_attn_plan_t pl, uint32_t *flags) {
    if (pl == nullptr || flags == nullptr) return host_fail(SYN_ERR_INVALID, "null argument");
    ATT_CK(cudaDeviceSynchronize());
    ATT_CK(cudaMemcpy(flags, pl->d_flags, (size_t)pl->cfg.R * pl->cfg.split * sizeof(uint32_t),
                      cudaMemcpyDeviceToHost));
    return SYN_OK;
}

}  // extern "C"
