// fused.h -- parameter block of the fused persistent kernels, shared by the
// host launcher and the device code, plus the address rule of a staging
// transfer (used identically by the copy-engine, dedicated-SM and co-located
// stagers).
#pragma once

#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

#include "protocol.h"
#include "schedule.h"

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD inline
#endif

namespace syn {

enum : int { OP_AG = 0, OP_RS = 1, OP_AR = 2 };

// Device-side failure sites recorded in err[1] (for diagnostics).
enum : int {
    WHERE_AG_FLAG = 1,      // producer waiting for a gathered chunk
    WHERE_PEER_FLAG = 2,    // peer loader waiting for a staged peer chunk
    WHERE_PIPE = 3,         // a shared-memory pipeline barrier
    WHERE_STAGER = 4,       // a stager's own copy barrier
    WHERE_BOUNDS = 5        // an index check
};

struct TensorMaps {  // CUtensorMap carries its own alignment
    CUtensorMap a;                 // AG: gathered [M,K]; RS/AR: A [M,K]   (bf16, box 64x128)
    CUtensorMap b;                 // B [K,N]                               (bf16, box 64x64)
    CUtensorMap peer[kMaxRanks];   // RS/AR: peer q partial rows            (fp32, box 32x128)
                                   // AG with direct_fetch: shard q [rows_q, K] (bf16, as `a`)
    CUtensorMap f32out;            // RS/AR: send / publish [M,N]           (fp32, box 32x32)
    CUtensorMap c;                 // AG: C [M,N]                           (bf16, box 32x32)
    CUtensorMap red;               // RED: partials of reducing tiles       (fp32, box 32x32)
    CUtensorMap push_src;          // dedicated push: push_buf [M,N]        (fp32, box 256x32, no swizzle)
    CUtensorMap push_dst;          // dedicated push: send [M,N]            (fp32, box 256x32, no swizzle)
};

// Dedicated push CTAs move boxes of kPushBoxCols x 32 fp32 (the host encodes
// the push tensor maps with the same box, no swizzle).
constexpr int kPushBoxCols = 256;

struct KernelParams {
    int32_t op, R, rank;
    int32_t M, N, K, M_r, cr, split, n_rc;  // cr: rows of the largest chunk
    int32_t ldst;                  // staging copies by warps with vector loads/stores
    RowBlocks rb;                  // row blocks and chunk geometry
    int32_t tiles_m, tiles_n;
    int32_t t_begin, t_end;        // range of tile_list this launch runs
    int32_t G;                     // GEMM CTAs: blockIdx.x < G
    int32_t n_comm;                // dedicated staging CTAs: blockIdx.x >= G
    int32_t colocated;             // GEMM CTAs run the staging warp
    int32_t waits;                 // consumers wait on in_flags
    int32_t local_inplace;         // AG: local shard aliases its gathered slot
    int32_t direct_fetch;          // AG: tiles whose chunks have not arrived read the source shard
                                   // through tm.peer[q] instead of waiting
    int32_t drop_transfer;         // fault injection: arrival index never published
    int32_t delay_transfer;        // fault injection: arrival index published late (device stagers)
    uint32_t delay_ns;             //   by this long
    int32_t peer_row_off;          // row coordinate offset of the peer tensor maps
    uint32_t epoch;
    uint64_t timeout_ns;
    const int32_t *tile_list;
    const int32_t *transfers;      // rc * R + q, arrival order
    int32_t n_transfers;
    int32_t slice_bytes;           // device stagers: bytes per slice
    int32_t slices_per_transfer;
    uint32_t *in_flags;            // [n_rc * R]
    uint32_t *in_cnt;              // [2][n_rc * R] slice counters (epoch parity)
    uint32_t *out_flags;           // [n_rc]
    uint32_t *out_cnt;             // [2][n_rc] producer counters (epoch parity)
    int32_t *err;                  // [4] code, site, cta, info
    unsigned long long *stats;     // [2] flag-wait ns, CTA-busy ns (nullable)
    unsigned long long *trace;     // [n_tiles][5] per tile-list entry: MMA start, MMA end
                                   // (last commit issued), epilogue start, end, walker (nullable)
    const uint8_t *stage_src[kMaxRanks];  // AG: shard q; RS/AR: peer q partial
    uint8_t *stage_dst;            // AG: gathered; RS/AR: receive buffer
    int64_t row_bytes;             // bytes of one row of a transfer
    int64_t recv_slot_rows;        // RS/AR: rows per peer slot of the receive buffer
    uint16_t *out;                 // AG: C; RS: out_r; AR: out   (bf16)
    float *f32_out;                // RS: send; AR: publish  (nullable)
    int32_t send_push;             // GEMM-RS push mode: send rows are added into `send`
    int32_t epi_tma;               // the f32out / red / c tensor maps are encoded: instances
                                   // with staging room store the epilogue through TMA
    float *red_buf;                // RED instances: fp32 partials of the reducing tiles,
    int32_t red_row_off;           // row r stored at row r - red_row_off
    // GEMM-RS push mode with dedicated push CTAs (blockIdx.x >= G): the
    // epilogue stores send rows into push_buf [M, N] and counts them as
    // produced; the push CTAs add each produced chunk into f32_out (`send`)
    const int32_t *push_list;      // send row chunks in production order
    int32_t n_push;
    int32_t push_dedicated;
    float *push_buf;
};

// Receive-buffer slot of source rank q (the local rank has none).
SYN_HD int recv_slot(int q, int rank) { return recv_slot_of(q, rank); }

// Source, destination and size of staging transfer `code` (transfer_rows in
// protocol.h gives the rows).
SYN_HD void transfer_span(const KernelParams &p, int code, const uint8_t *&src, uint8_t *&dst,
                          int64_t &bytes) {
    const TransferRows t = transfer_rows(p.op, p.rank, p.rb, p.recv_slot_rows, code);
    bytes = t.rows * p.row_bytes;
    src = p.stage_src[t.q] + t.src_row * p.row_bytes;
    dst = p.stage_dst + t.dst_row * p.row_bytes;
}

// Which compiled kernel instance a launch uses, and its grid.
struct LaunchCfg {
    int tile_n;   // 128 or 256
    int tile_k;   // k-block depth: 64 or 32
    int stages;   // GEMM pipeline stages
    bool stg;     // CTA carries the co-located staging buffers
    bool pair;    // 2-CTA clusters share 256-row tiles (tile_m 256)
    int grid;     // CTAs
    bool red = false;  // RS/AR, resident peers: reducer warps stream the peer sum
    bool overlap_prev = false;  // CTA pairs: programmatic launch after the previous kernel
};

// Host launchers (one translation unit per operator).  cudaErrorInvalidValue
// if (tile_n, tile_k, stages, stg) is not a compiled combination.
cudaError_t launch_fused_ag(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                            cudaStream_t st);
cudaError_t launch_fused_rs(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                            cudaStream_t st);
cudaError_t launch_fused_ar(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                            cudaStream_t st);
// Dynamic shared memory of a combination (-1 if not compiled).
int fused_smem_bytes(int op, const LaunchCfg &lc);
// Default pipeline depth of a (tile_n, tile_k, stg, pair, red) choice.
inline int default_stages(int op, int tile_n, int tile_k, bool stg, bool pair, bool red = false) {
    if (red) return pair ? (op == OP_AR ? 4 : 6) : (op == OP_AR ? 3 : 4);
    if (pair) return op == OP_AG ? (stg ? 5 : 7) : 4;
    if (tile_k == 32) return op == OP_AG ? (stg ? 8 : 9) : 6;
    if (op == OP_AG) return tile_n == 256 ? 4 : 6;
    return tile_n == 256 ? 3 : 4;
}
// Co-resident 2-CTA clusters for a pair instance (0 if unknown / not a pair).
int fused_max_clusters(int op, const LaunchCfg &lc);
// GEMM-RS: 1 if the instance stores its epilogue through TMA (needed by the
// push mode), 0 if not, -1 if not compiled.
int epi_tma_rs(const LaunchCfg &lc);

// Record the message syn_last_error() returns on this thread.
void set_last_error(const std::string &msg);

}  // namespace syn
