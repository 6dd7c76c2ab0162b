/*
 * syn.h -- C ABI of libsyn: chunk-scheduled compute/communication overlap for
 * tensor-parallel GEMMs on one GB300 (sm_103a).
 *
 * Source of the method: "Syncopate: Efficient Multi-GPU AI Kernels via
 * Automatic Chunk-Centric Compute-Communication Overlap" (OSDI 2026 summary
 * page and arXiv abstract), with Entwine (arXiv 2609.11562 abstract) as
 * related work.  Communication is expressed as transfers of *chunks* -- a block
 * of a logical tensor holding one or more compute tiles (summary page, method
 * ¶1, paper §5.1).  A chunk->tile dependency graph says which chunks each tile
 * consumes or produces and where waits go (method ¶2).  The tile scheduler is
 * rewritten to walk chunks in communication order while keeping locality
 * inside a chunk (method ¶4, paper §5.2, Fig. 6).  One plan lowers to several
 * staging backends: copy engine, TMA on dedicated SMs, TMA co-located with
 * compute (method ¶3, paper §5.2, Fig. 7).  The three operators are the
 * summary page's GEMM workloads (Experiments, paper §6.1): AG-GEMM, GEMM-RS,
 * GEMM-AR.
 *
 * Ranks.  All R tensor-parallel ranks live in one GPU: the R-1 peers are
 * simulated by buffers in the same HBM, and "communication" is the staging of
 * those buffers into the local rank's buffers.
 *
 * Conventions for every call:
 *  - Every function returns an int status: SYN_OK (0) or a negative SYN_ERR_*.
 *    No C++ exception crosses this boundary.  syn_last_error() gives a message
 *    for the most recent failure on the calling thread.
 *  - Device pointers are plain CUDA device addresses, 16-byte aligned, owned by
 *    the caller.  Arrays of device pointers (shards, peer partials) are HOST
 *    arrays of length R.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Operator calls are asynchronous on it; check completion and device-side
 *    errors with syn_sync_status().  One plan must not run on two streams at
 *    once.
 *  - Matrices are row-major.  bf16 operands are IEEE bfloat16; partials fp32.
 *  - The plan owns its flags, counters, error word, tables, staging receive
 *    buffers and helper streams; syn_plan_destroy() frees them.
 *  - Limits of this version: 1 <= R <= 8; K % 8 == 0 and N % 8 == 0 (every
 *    bf16 row and fp32 partial row starts on a 16-byte boundary); dense
 *    layouts (ld* == 0 or equal to the row length); GEMM-RS needs
 *    (M/R) % 32 == 0 (a tile may hold rows of several rank blocks, sent and
 *    reduced ones; each 32-row warp group lies in one block).  M may have a
 *    tail (M % tile_m != 0).  K need not be a multiple of the 64-element
 *    k-block nor N of tile_n: the TMA operand loads read zeros past K and N,
 *    so the last k-block and the last column of tiles are partial, and no
 *    store reaches past column N.
 */
#ifndef SYN_H
#define SYN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define SYN_OK 0
#define SYN_ERR_INVALID (-1)     /* bad argument, shape, alignment or split     */
#define SYN_ERR_UNSUPPORTED (-2) /* valid but outside this version's limits     */
#define SYN_ERR_CUDA (-3)        /* a CUDA runtime/driver call failed          */
#define SYN_ERR_TIMEOUT (-4)     /* a device wait on a chunk flag or pipeline
                                    barrier ran past the plan's timeout         */
#define SYN_ERR_BOUNDS (-5)      /* a device-side index check failed           */

typedef struct syn_plan_s *syn_plan_t; /* opaque, owned by the library */

/* The three operators (summary page, Experiments, paper §6.1). */
typedef enum {
    SYN_OP_AG_GEMM = 0, /* C = concat_q(shard_q) . B                          */
    SYN_OP_GEMM_RS = 1, /* out_r = rows_r(A.B) + sum_{q!=r} rows_r(peer_q)    */
    SYN_OP_GEMM_AR = 2  /* out = A.B + sum_{q!=r} peer_q                      */
} syn_op_t;

/* Tile traversal inside a chunk (method ¶4, paper §5.2, Fig. 6: keep or
 * adjust the traversal to trade arrival time against locality). */
typedef enum {
    SYN_ORDER_ROW_MAJOR = 0, /* tile rows in order, columns fastest             */
    SYN_ORDER_COL_MAJOR = 1, /* tile columns in order, rows fastest             */
    SYN_ORDER_GROUPED = 2,   /* group_m tile rows at a time, column by column   */
    SYN_ORDER_BANDED = 3     /* AG-GEMM / A2A-GEMM only: bands of group_m tile
                                rows, each keyed by the latest chunk any of its
                                rows reads; bands in key order, each column by
                                column.  Coarser than the chunk order, so each
                                band reads the whole of B once from HBM and
                                keeps its A rows in L2 (B larger than L2)   */
} syn_order_t;

/* Staging backends for one plan (method ¶3, paper §5.2, Fig. 7), plus the two
 * comparison paths of paper Fig. 2(b). */
typedef enum {
    SYN_BACKEND_CE = 0,             /* copy engine: cudaMemcpyAsync on a side
                                       stream + a stream-ordered flag write per
                                       chunk                                      */
    SYN_BACKEND_TMA_DEDICATED = 1,  /* comm_sms extra CTAs of the same persistent
                                       grid copy chunks with TMA bulk copies     */
    SYN_BACKEND_TMA_COLOCATED = 2,  /* one staging warp in every GEMM CTA copies
                                       chunk slices with TMA bulk copies (mbarrier
                                       pipelined), slice ownership by CTA index  */
    SYN_BACKEND_TMA_COLOCATED_SMEM = 3, /* GEMM-RS/AR only: the peers' partials are
                                       resident and read in place, no global
                                       staging: by reducer warps with plain
                                       loads (default at tile_n 256, see
                                       knobs.reduce_warps) or through a TMA ring
                                       of peer tiles in the epilogue            */
    SYN_BACKEND_UNFUSED = 4,        /* baseline: whole staging copy first, then
                                       the same GEMM kernel without waits         */
    SYN_BACKEND_DECOMPOSED = 5,     /* baseline: one GEMM launch per chunk group,
                                       each after its chunks' copies (Fig. 2(b)) */
    SYN_BACKEND_LDST_DEDICATED = 6, /* as TMA_DEDICATED, but every warp of the
                                       staging CTAs copies slices with 16-byte
                                       vector loads and stores                   */
    SYN_BACKEND_LDST_COLOCATED = 7  /* one warp of every GEMM CTA copies slices
                                       with 16-byte vector loads and stores (no
                                       shared-memory staging buffers, so the
                                       GEMM keeps its deepest pipeline)          */
} syn_backend_t;

/* Shapes.  M = rows of the gathered / full output space (all ranks),
 * K = contraction, N = output columns.  Rank q owns rows [q*M/R, (q+1)*M/R).
 * ld* are leading dimensions in elements; 0 means dense row-major. */
typedef struct {
    int64_t M, N, K;
    int64_t lda, ldb, ldc;
} syn_layout_t;

/* Tuning knobs (the search space of paper §6.3, Fig. 11, and Entwine's
 * communication-SM allocation). */
typedef struct {
    syn_backend_t backend;
    int comm_sms;          /* TMA_DEDICATED: CTAs (SMs) given to staging, 1..32  */
    int tile_m;            /* rows per output tile: 128 (one CTA per tile) or
                              256 (a 2-CTA cluster shares the tile with
                              cta_group::2 UMMAs); 0 = 128                    */
    int tile_n;            /* 128 or 256 (0 = 256)                               */
    int group_m;           /* SYN_ORDER_GROUPED group height in tiles (0 = 8)   */
    int slice_kb;          /* device stagers: KiB per slice of a chunk (0 = 128) */
    uint64_t timeout_ns;   /* bound on every device wait (0 = 2 s, or the
                              SYN_TIMEOUT_NS environment variable)              */
    int debug_drop_chunk;  /* fault injection: arrival index of a staging
                              transfer whose ready flag is never published
                              (-1 = off); the call then ends in SYN_ERR_TIMEOUT */
    int trace;             /* 1 = accumulate flag-wait and CTA-busy nanoseconds
                              (read with syn_plan_stats); 2 = also record four
                              global-timer stamps and the walker per tile of
                              the last call (read with syn_plan_trace)        */
    int stages;            /* GEMM shared-memory pipeline depth; 0 = the
                              default of the chosen instance:
                                tile_m 256: AG 5 (co-located stagers) / 7;
                                  RS / AR with reducer warps 6 / 4, with the
                                  epilogue peer ring 4;
                                tile_m 128: reducer warps RS 4, AR 3; AG 4 / 6
                                  (tile_n 256 / 128); RS, AR 3 / 4;
                                tile_k 32: AG 8 (co-located) / 9, RS, AR 6.
                              Other compiled depths: tile_m 256 AG 4-7, RS
                              3-7, AR 3-7 (with reducer warps 3-5); tile_m
                              128 RS / AR 2-6 (the peer ring takes the memory
                              the stages leave).  A depth that is not
                              compiled is SYN_ERR_UNSUPPORTED.               */
    int tile_k;            /* k-block depth per pipeline stage: 64 or 32
                              (0 = 64).  32 halves each stage, so twice as
                              many fit and more loads are in flight.         */
    int reduce_spread;     /* GEMM-RS with TMA_COLOCATED_SMEM only: where the
                              reduce tiles (the ones that stream the resident
                              peer partials) go in the tile order.
                              -1 = all first; n > 0 = one per persistent tile
                              walker of a grid of n walkers (CTAs, or CTA
                              pairs at tile_m 256), in evenly spaced rounds;
                              0 = default: syn_plan_create spreads them over
                              its own grid, syn_schedule_build (which knows no
                              grid) keeps them first.                         */
    int reduce_warps;      /* GEMM-RS/AR with TMA_COLOCATED_SMEM, tile_n 256,
                              tile_k 64: 0 = default: extra warps per CTA add
                              the peer partials with plain loads.  GEMM-RS:
                              the epilogue stores each reducing tile's fp32
                              partial into a (M/R) x N plan buffer and frees
                              the accumulator at once; four reducer warps
                              then add the peers to it.  GEMM-AR: from the
                              start of the kernel, fourteen reducer warps sum
                              the peers of the CTA's tiles in walk order into
                              a M x N plan buffer, and the epilogue adds that
                              sum to the accumulator.  Same additions in the
                              same order as -1, bit for bit.
                              -1 = the epilogue adds the peers itself through a
                              shared-memory ring of peer tiles.              */
    int ce_streams;        /* CE: side streams the chunk copies are spread over
                              round-robin in arrival order, so several copy
                              engines run at once (0 = 4; at most 16)        */
    int rs_push;           /* GEMM-RS, TMA_COLOCATED_SMEM with reducer warps:
                              0 = pull mode (send rows stored for the peers to
                              pull); 1 = push mode: each send row is added
                              (fp32, TMA reduce-add at the destination) into
                              `send`, which then holds the destination ranks'
                              receive accumulators that all ranks add into;
                              SYN_ERR_UNSUPPORTED elsewhere                   */
    int debug_delay_chunk; /* fault injection (device stagers: TMA_DEDICATED,
                              TMA_COLOCATED): arrival index of a staging
                              transfer whose ready flag is published
                              debug_delay_us late; the call only waits longer
                              unless that exceeds timeout_ns                  */
    int debug_delay_us;    /* (0 = off)                                        */
    int debug_corrupt_entry; /* fault injection for the kernel's bounds checks
                              (0 = off): n > 0 gives the device copy of
                              tile-list entry n - 1 (and of transfer-list
                              entry (n - 1) mod n_transfers) an out-of-range
                              value at plan creation; every call then ends in
                              SYN_ERR_BOUNDS, with no out-of-range access     */
    int direct_fetch;      /* AG-GEMM / A2A-GEMM with device stagers: 1 = a
                              tile whose chunks have not arrived when the
                              producer reaches it, and whose rows all come
                              from one source rank, reads them in place
                              from that rank's shard (TMA, the pages'
                              in-place lowering) instead of waiting; tiles
                              whose chunks have arrived read the staged
                              copy.  The stagers still fill `gathered`
                              completely.  0 = off: every tile waits for its
                              chunks (default)                                */
    int push_sms;          /* GEMM-RS push mode (rs_push = 1): 0 = the epilogue
                              warps add each send tile into `send` with TMA
                              tile reduce-adds; n > 0 = n dedicated push CTAs
                              (SMs) of the same grid do it instead: the
                              epilogue stores send rows into a plan buffer and
                              counts each row chunk produced, and the push
                              CTAs, as each chunk's produced flag arrives (in
                              production order: destinations in ring order),
                              add it into `send` with TMA tile reduce-adds and
                              publish its delivered flag (syn_plan_flags:
                              in_flags[rc * R + rank]).  The compute grid
                              shrinks by n SMs: the communication-SM balance
                              of the Entwine abstract.  1..32             */
} syn_knobs_t;

/* Everything a caller or a test may want to know about a plan. */
typedef struct {
    int op, R, rank, backend, order;
    int64_t M, N, K, M_r;
    int64_t chunk_rows;    /* rows of the largest chunk, ceil((M/R) / split)    */
    int split;             /* chunks per rank row block                         */
    int n_row_chunks;      /* chunks over the whole row space = R * split       */
    int n_transfers;       /* staging transfers (row chunk, source rank)        */
    int tile_m, tile_n, tiles_m, tiles_n, n_tiles;
    int grid_compute;      /* GEMM CTAs (0 before a device plan exists)          */
    int grid_comm;         /* dedicated staging CTAs                             */
    int smem_bytes;        /* dynamic shared memory per CTA                      */
    int num_sms;
    uint32_t epoch;        /* calls issued so far                               */
    uint64_t recv_bytes;   /* plan-owned staging receive buffer                 */
    int a2a;               /* 1: an A2A-GEMM plan (op is SYN_OP_AG_GEMM over
                              per-source row blocks; M_r is 0)                 */
} syn_plan_info_t;

/* Host-only schedule builder: no CUDA call, usable without a GPU.
 * Builds the chunk partition, the arrival order of the staging transfers and
 * the rewritten tile order exactly as syn_plan_create does (method ¶2 and ¶4,
 * paper §5.2, Fig. 6).  Any output array may be NULL; call once with NULLs to
 * learn the sizes from *info.
 *   tile_list[i]  = tile id (tile_row * tiles_n + tile_col) of the i-th tile
 *                   in execution order; persistent CTA c runs entries
 *                   c, c + G, c + 2G, ...
 *   tile_key[i]   = the chunk-arrival key the order is sorted by (the latest
 *                   arrival index among the chunks the tile consumes; negative
 *                   for GEMM-RS tiles that only produce send chunks)
 *   transfers[a]  = row_chunk * R + source_rank of the a-th staging transfer
 *                   in arrival order
 * Returns SYN_ERR_INVALID / SYN_ERR_UNSUPPORTED for shapes outside the limits. */
int syn_schedule_build(syn_op_t op, int R, int rank, const syn_layout_t *layout,
                       int64_t chunk_rows, int split, syn_order_t order,
                       const syn_knobs_t *knobs, syn_plan_info_t *info,
                       int32_t *tile_list, int32_t *tile_key, int32_t *transfers);

/* Fill *knobs with the defaults: TMA_COLOCATED staging (the chunks are copied
 * by a warp inside every GEMM CTA, so progress never depends on another
 * engine running beside the kernel), 128x256 tiles, 2 s timeout. */
int syn_knobs_default(syn_knobs_t *knobs);

/* Build a plan on the current CUDA device: validates, builds the schedule,
 * allocates and uploads flags, counters, tables and (for backends that stage
 * through global memory in GEMM-RS/AR) the receive buffer.
 * chunk_rows and split: chunks per rank row block; give either (the other 0)
 * or both with chunk_rows * split == M/R; both 0 means split = 1.  A split
 * that does not divide M/R (1 <= split <= M/R) cuts each rank block into
 * chunks of floor or ceil((M/R)/split) rows: chunk j holds local rows
 * [ceil(j*(M/R)/split), ceil((j+1)*(M/R)/split)).
 * knobs may be NULL (defaults).  On success *out owns device memory. */
int syn_plan_create(syn_plan_t *out, syn_op_t op, int R, int rank,
                    const syn_layout_t *layout, int64_t chunk_rows, int split,
                    syn_order_t order, const syn_knobs_t *knobs);

/* Free a plan (synchronises its helper stream first).  NULL is a no-op. */
int syn_plan_destroy(syn_plan_t plan);

/* AllGather-GEMM (summary page, Experiments, paper §6.1).
 *   shards   : host array of R device pointers, bf16 [M/R, K] each; shards[r]
 *              may alias gathered + r*(M/R)*K (in-place local slot, not copied)
 *   gathered : bf16 [M, K] output; gathered[q*M/R + i] = shards[q][i] bit for bit
 *   B        : bf16 [K, N]
 *   C        : bf16 [M, N] output, C = gathered . B, fp32 accumulation, one
 *              round-to-nearest-even
 * Tiles of C start as soon as the chunks of gathered they read have arrived. */
int syn_ag_gemm(syn_plan_t plan, const void *const *shards, void *gathered,
                const void *B, void *C, void *stream);

/* GEMM-ReduceScatter for the plan's rank r (summary page, Experiments, paper
 * §6.1).
 *   A             : bf16 [M, K], B : bf16 [K, N]
 *   peer_partials : host array of R device pointers, fp32 [M, N] each: peer q's
 *                   partial product; entry r is ignored (may be NULL); only
 *                   rows_r (rows [r*M/R, (r+1)*M/R)) of each affect the
 *                   result (a tile straddling that block's edge may load,
 *                   but does not use, the rows next to it)
 *   send          : nullable fp32 [M, N]; rows of every rank q != r receive
 *                   the local partial P = A.B (the chunks peers would pull);
 *                   rows of rank r are not written
 *   out_r         : bf16 [M/R, N] = rne(P[rows_r] + S), S = the peers' rows
 *                   summed first, sum_{q != r, ascending} peer_q[rows_r]
 * Send tiles run first (in ring order of their destination), reduce tiles last
 * when peers are staged; with resident peers (TMA_COLOCATED_SMEM) the reduce
 * tiles are spread over the walk (knobs.reduce_spread). */
int syn_gemm_rs(syn_plan_t plan, const void *A, const void *B,
                const float *const *peer_partials, float *send, void *out_r,
                void *stream);

/* GEMM-AllReduce for the plan's rank r (summary page, Experiments, paper §6.1).
 *   out     : bf16 [M, N] = rne(A.B + S), S = sum_{q != r, ascending} peer_q
 *             (every GEMM-RS / GEMM-AR path adds the peers first, then the
 *             local partial: the same bits whatever the backend)
 *   publish : nullable fp32 [M, N] = A.B (the local partial peers would pull)
 * Other arguments as for syn_gemm_rs. */
int syn_gemm_ar(syn_plan_t plan, const void *A, const void *B,
                const float *const *peer_partials, float *publish, void *out,
                void *stream);

/* A2A-GEMM: the MoE-style all-to-all followed by the expert GEMM (the
 * operator pair the Syncopate paper's sensitivity study, §6.3 / Fig. 11,
 * tunes beside AG-GEMM, GEMM-RS and GEMM-AR).  Rank r hosts one expert; every
 * rank q (r included) sends it rows_from[q] token rows of K bf16 values.  The
 * rows are gathered in source-rank order and multiplied by the expert weight:
 *   gathered rows [off[q], off[q] + rows_from[q]) = part q, off[q] = sum_{p<q} rows_from[p]
 *   C = gathered . B
 * This is the AG-GEMM plan with row blocks of unequal size: block q is cut
 * into `split` chunks of near-equal size (chunk j holds block rows
 * [ceil(j*m/split), ceil((j+1)*m/split)), m = rows_from[q]; a block smaller
 * than split has empty chunks, which still publish their flags); tiles wait
 * only on the chunks they read, and the arrival order starts at the local
 * block, then r+1, r+2, ... as in AG-GEMM.
 *   rows_from : host int64 [R], each >= 0, sum M >= 1 (an expert that gets no
 *               rows has nothing to compute: SYN_ERR_INVALID)
 *   split     : 1 <= split <= 64 (0 means 1)
 *   knobs     : as syn_plan_create (TMA_COLOCATED_SMEM is GEMM-RS/AR only)
 * Every staging backend works as for AG-GEMM.  The plan reports a2a = 1. */
int syn_plan_create_a2a(syn_plan_t *out, int R, int rank, const int64_t *rows_from,
                        int64_t N, int64_t K, int split, syn_order_t order,
                        const syn_knobs_t *knobs);

/* Host-only A2A-GEMM schedule (no CUDA call), as syn_schedule_build. */
int syn_schedule_build_a2a(int R, int rank, const int64_t *rows_from, int64_t N, int64_t K,
                           int split, syn_order_t order, const syn_knobs_t *knobs,
                           syn_plan_info_t *info, int32_t *tile_list, int32_t *tile_key,
                           int32_t *transfers);

/* Run an A2A-GEMM plan (asynchronous on `stream`).
 *   parts    : host array of R device pointers, bf16 [rows_from[q], K] each
 *              (NULL allowed where rows_from[q] == 0); parts[r] may alias
 *              gathered + off[r]*K (in place, not copied)
 *   gathered : bf16 [M, K] output, gathered[off[q] + i] = parts[q][i] bit for bit
 *   B        : bf16 [K, N];  C : bf16 [M, N] = gathered . B (fp32 accumulation,
 *              one round-to-nearest-even)
 * Returns SYN_ERR_INVALID for a plan made by syn_plan_create (and syn_ag_gemm
 * does for an A2A-GEMM plan). */
int syn_a2a_gemm(syn_plan_t plan, const void *const *parts, void *gathered,
                 const void *B, void *C, void *stream);

/* Synchronise `stream`, then read and clear the plan's device error word.
 * Returns SYN_OK, SYN_ERR_TIMEOUT or SYN_ERR_BOUNDS (device side) or
 * SYN_ERR_CUDA.  After a device error the plan's flag/counter state is reset,
 * so the next call starts clean. */
int syn_sync_status(syn_plan_t plan, void *stream);

/* Plan facts (sizes, grid, epoch). */
int syn_plan_query(syn_plan_t plan, syn_plan_info_t *info);

/* Copy the plan's host schedule tables out (same meaning as in
 * syn_schedule_build; each pointer may be NULL). */
int syn_plan_tables(syn_plan_t plan, int32_t *tile_list, int32_t *tile_key,
                    int32_t *transfers);

/* Copy the device ready flags out (synchronous).  in_flags has
 * n_row_chunks * R entries (row_chunk * R + source_rank) and holds the epoch
 * of the call that last published that transfer; out_flags has n_row_chunks
 * entries and holds the epoch of the call whose tiles last finished producing
 * that row chunk of `send` (GEMM-RS) or `publish` (GEMM-AR). */
int syn_plan_flags(syn_plan_t plan, uint32_t *in_flags, uint32_t *out_flags);

/* Trace counters (knobs.trace = 1): total nanoseconds the GEMM CTAs spent in
 * chunk-flag waits, and total nanoseconds they were resident, summed over CTAs
 * since the plan was created.  Synchronous. */
int syn_plan_stats(syn_plan_t plan, uint64_t *flag_wait_ns, uint64_t *cta_busy_ns);

/* Per-tile timeline of the plan's most recent call (knobs.trace = 2), as
 * global-timer nanoseconds: for tile-list entry i, out[5i+0] = the MMA issuer
 * starts the tile, out[5i+1] = its last MMA commit is issued, out[5i+2] = the
 * epilogue sees the accumulator ready, out[5i+3] = the epilogue has released
 * it; out[5i+4] = the index of the tile walker (CTA, or CTA pair) that ran it.
 * out has 5 * n_tiles entries (host memory).  Synchronous.
 * SYN_ERR_INVALID if the plan was created without trace = 2. */
int syn_plan_trace(syn_plan_t plan, uint64_t *out);

/* Enumerate-and-measure autotuner (summary page, method ¶4 and paper §6.3,
 * Fig. 11; Entwine's communication-SM balance).  Allocates its own scratch
 * operands of the given shape and searches staging placement (backend and
 * comm_sms), tile shape, split, tile order with group_m, pipeline depth,
 * reduce_warps (GEMM-RS/AR) and direct_fetch (AG-GEMM) by coordinate descent:
 * each dimension swept with the others held at the best point so far, every
 * candidate timed over two back-to-back calls (CUDA events), the fastest
 * tenth (at least two) re-timed over ten, the best re-timed mean kept;
 * passes repeat until one finds nothing faster.  Candidates run
 * with a 50 ms wait bound and are dropped on their first error.  budget_s
 * bounds the wall time (0 = 60 s).  If the SYN_TUNE_CACHE environment
 * variable names a file, results are cached there as JSON lines keyed by
 * (op, R, rank, M, N, K) and a cache hit returns without measuring; if
 * SYN_TUNE_LOG names a file, every candidate is appended to it (phase
 * "quick" or "final" with its time; "dropped" when its plan cannot be made,
 * "failed" when a call failed, both with us = -1).  *best_us is the winner's re-timed mean, the smallest "final"
 * timing of the search.  best_us may be NULL.
 * *best is also read on input for one field: best->rs_push != 0 with
 * SYN_OP_GEMM_RS tunes push mode (a different computation, cached under its
 * own key) and adds push_sms (0, 4, 8, 16, 32) to the search. */
int syn_autotune(syn_op_t op, int R, int rank, const syn_layout_t *layout,
                 double budget_s, syn_knobs_t *best, int *best_split,
                 syn_order_t *best_order, double *best_us);

/* ---- AG-GEMM without any device allocation ------------------------------
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: plug-in hosts (inference-server
 * backends, framework custom ops under a caching allocator) that give an
 * operator only its input and output tensors, and serving loops that forbid
 * cudaMalloc/cudaFree after start-up because those calls can synchronise the
 * device and can fail mid-step.  syn_plan_create allocates; this does not.
 *
 * Same operation and arguments as syn_ag_gemm (co-located TMA staging, tile
 * order `order`, `split` chunks per shard), without a plan.  Its scratch (tile
 * and transfer lists, ready flags, counters, error word) lives in one static
 * device array of SYN_NOALLOC_SCRATCH_BYTES that every GPU loading libsyn
 * keeps until the process exits.  The first call on a device looks up that
 * array's address (cudaGetSymbolAddress) with the device current; make that
 * first call before any stream capture.  Every call writes its schedule into
 * the array with a small kernel that takes the tables as its parameters (no
 * host buffer outlives the call), then launches the GEMM; device waits are
 * bounded as for plans (SYN_TIMEOUT_NS, else 2 s).  Shapes beyond SYN_NOALLOC_MAX_TILES
 * output tiles (128 x tile_n, tile_n = 256 if N % 256 == 0 else 128) or
 * SYN_NOALLOC_MAX_ROW_CHUNKS chunks return SYN_ERR_UNSUPPORTED with a
 * message in syn_last_error().  No cudaMalloc, cudaFree or allocating library
 * routine is called.  Every call clears the flags, counters and error word it
 * needs, but all calls on a device share the one array: calls that overlap on
 * the GPU (other streams, other host threads) race and give undefined results.
 *   status_dev : nullable device int32[4]; receives {code, site, CTA, info} of
 *                this call's device error word (code 0 = no error) once the
 *                call completes on `stream`
 * Returns after enqueuing on `stream` (SYN_OK) or a SYN_ERR_* host error. */
#define SYN_NOALLOC_MAX_TILES 4096
#define SYN_NOALLOC_MAX_ROW_CHUNKS 64
#define SYN_NOALLOC_SCRATCH_BYTES 32768
int syn_ag_gemm_noalloc(int R, int rank, const syn_layout_t *layout, int split,
                        syn_order_t order, const void *const *shards, void *gathered,
                        const void *B, void *C, int32_t *status_dev, void *stream);

/* Number of SMs of the current device (0 and SYN_ERR_CUDA without a GPU). */
int syn_device_sms(int *num_sms);

/* Static description of a status code. */
const char *syn_status_string(int status);

/* Message for the most recent failing call on this thread ("" if none). */
const char *syn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SYN_H */
