/*
 * syn_attn.h -- fused ring attention with chunk-scheduled KV exchange
 * (libsyn.so; status codes and backends as in syn.h).
 *
 * The Syncopate summary page evaluates head-parallel / sequence-parallel
 * attention and RingAttention beside its GEMM operators (Experiments, paper
 * §6.1; results in Fig. 9).  This is the sequence-parallel (ring) forward:
 * R ranks each hold S_r consecutive tokens of Q, K and V; rank r computes
 * attention of its own queries over the keys of every rank.  One persistent
 * kernel (a cooperative launch, one CTA per SM) both stages the other ranks'
 * KV shards into gathered buffers chunk by chunk -- a staging warp in every
 * CTA, ranks r+1, r+2, ... in turn as in the GEMM plans, each chunk
 * publishing a ready flag once its bytes have landed -- and computes: each
 * (query tile, head) work item visits the KV blocks in that arrival order
 * (local shard first), waiting only for the chunk its next block reads
 * (method ¶2-¶4 of the summary: waits per chunk, tiles ordered by arrival).
 *
 *   O[i][h][:] = sum_j softmax_j(scale * Q[i][h] . K[j][hk]) V[j][hk][:]
 *   hk = h / (H_q / H_kv) (grouped-query attention), j over the R*S_r keys
 *   in global order; causal: keys with global position j > r*S_r + i are
 *   excluded.  lse[i][h] = log sum_j exp(scale * Q[i][h] . K[j][hk]).
 *
 * Head-parallel layout (head_parallel = 1; the all-to-all form): every rank
 * holds S_r tokens of all heads; rank r computes the full-sequence attention
 * of its heads h in [r*H_q/R, (r+1)*H_q/R) (KV heads [r*H_kv/R, ...)) for the
 * queries of every rank.  The kernel stages Q, K and V columns of those heads
 * from every rank into gathered buffers chunk by chunk (the local rank's too)
 * and each query tile waits for its own chunk as well as the KV blocks'.
 *
 * Precision: bf16 inputs; Q.K^T accumulated in fp32 by the tensor cores;
 * softmax in fp32 with exp2 (scores scaled by scale * log2(e)); the
 * probabilities are rounded to bf16 for the P.V product (fp32
 * accumulation); the running output is kept in fp32 and rounded once
 * (round-to-nearest-even) to bf16.
 */
#ifndef SYN_ATTN_H
#define SYN_ATTN_H

#include <stdint.h>

#include "syn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct syn_attn_plan_s *syn_attn_plan_t; /* opaque, owned by the library */

typedef struct {
    int R, rank;          /* simulated ranks (1..8) and the local rank          */
    int64_t S_r;          /* tokens per rank, a multiple of 256 (work items
                             take two 128-row query tiles)                     */
    int H_q, H_kv;        /* query and KV heads, H_q % H_kv == 0                */
    int d;                /* head dimension: 128                                */
    int causal;           /* 0 or 1 (global positions)                          */
    int split;            /* chunks per rank's KV shard, 1..S_r/128 (0 = 1);
                             chunk j of a shard holds its rows
                             [ceil(j*S_r/split), ceil((j+1)*S_r/split))        */
    int backend;          /* SYN_BACKEND_TMA_COLOCATED (a staging warp inside the
                             attention kernel, the default) or
                             SYN_BACKEND_UNFUSED (every copy first with
                             cudaMemcpyAsync, then the kernel without waits).
                             Copy-engine staging beside a waiting kernel is not
                             offered: the attention kernel holds every SM's
                             whole register file, and at full size the copies
                             did not progress while its CTAs waited          */
    float scale;          /* 0 = 1/sqrt(d)                                      */
    uint64_t timeout_ns;  /* bound on every device wait (0 = SYN_TIMEOUT_NS or
                             2 s); a wait that runs out ends the call in
                             SYN_ERR_TIMEOUT                                    */
    int debug_drop_chunk; /* -1 = off; else the arrival index of a chunk whose
                             flag is never written (fault injection: the call
                             must end in SYN_ERR_TIMEOUT)                       */
    int head_parallel;    /* 0: ring (sequence-parallel) layout, run with
                             syn_ring_attention; 1: head-parallel layout, run
                             with syn_head_attention (H_q and H_kv divisible
                             by R)                                              */
} syn_attn_cfg_t;

/* Plan facts. */
typedef struct {
    int R, rank, H_q, H_kv, d, causal, split, backend;
    int64_t S_r;
    int n_qtiles;         /* query tiles: S_r / 128 (ring), R*S_r / 128 (head)  */
    int grid;             /* persistent CTAs: min(n_qtiles / 2 * heads, resident
                             CTAs), heads = H_q (ring) or H_q / R (head);
                             work item (head h, tile pair t) = h * n_qtiles / 2
                             + t (query tiles 2t and 2t+1) runs on CTA item mod
                             grid                                              */
    int n_transfers;      /* staged chunks (R-1, or R when the local shard is
                             not in place, times split)                        */
    int smem_bytes;
    uint32_t epoch;       /* calls issued so far                               */
} syn_attn_info_t;

/* Defaults: R 1, rank 0, S_r 256, 1 head, d 128, not causal, split 1,
 * SYN_BACKEND_TMA_COLOCATED. */
int syn_attn_cfg_default(syn_attn_cfg_t *cfg);

/* Validate and build a plan on the current device (flags, slice counters,
 * error word).  SYN_ERR_INVALID / SYN_ERR_UNSUPPORTED for shapes outside
 * the limits above, with syn_last_error() saying which. */
int syn_attn_plan_create(syn_attn_plan_t *out, const syn_attn_cfg_t *cfg);

/* Free a plan (no call of it may still be running).  NULL is a no-op. */
int syn_attn_plan_destroy(syn_attn_plan_t plan);

/* One ring-attention forward of the plan's rank (asynchronous on `stream`).
 *   Q          : bf16 [S_r, H_q, d] (token-major), the local queries
 *   K_shards   : host array of R device pointers, bf16 [S_r, H_kv, d] each:
 *                rank q's keys; entry rank may alias K_gathered + rank*S_r*H_kv*d
 *                (in place, not copied)
 *   V_shards   : the same for the values
 *   K_gathered, V_gathered : bf16 [R*S_r, H_kv, d] outputs: row q*S_r + i =
 *                shard q row i, bit for bit (the staging destination)
 *   O          : bf16 [S_r, H_q, d] output
 *   lse        : nullable fp32 [S_r, H_q] output (natural log)
 * Every pointer 16-byte aligned.  Returns after enqueuing (SYN_OK) or a host
 * error; device errors surface in syn_attn_sync_status. */
int syn_ring_attention(syn_attn_plan_t plan, const void *Q, const void *const *K_shards,
                       const void *const *V_shards, void *K_gathered, void *V_gathered, void *O,
                       float *lse, void *stream);

/* One head-parallel attention forward of the plan's rank (asynchronous).
 *   Q_shards, K_shards, V_shards : host arrays of R device pointers, rank q's
 *                tokens of all heads: bf16 [S_r, H_q, d] and [S_r, H_kv, d]
 *   Q_gathered : bf16 [R*S_r, H_q/R, d] output: row q*S_r + i holds rank q's
 *                token i, heads r*H_q/R .. (r+1)*H_q/R - 1, bit for bit
 *   K_gathered, V_gathered : bf16 [R*S_r, H_kv/R, d] outputs, likewise
 *   O          : bf16 [R*S_r, H_q/R, d]: the local heads' attention for every
 *                token (global positions: causal excludes later tokens)
 *   lse        : nullable fp32 [R*S_r, H_q/R]
 * 16-byte alignment as for syn_ring_attention; a ring plan returns
 * SYN_ERR_INVALID here and a head-parallel plan in syn_ring_attention. */
int syn_head_attention(syn_attn_plan_t plan, const void *const *Q_shards, const void *const *K_shards,
                       const void *const *V_shards, void *Q_gathered, void *K_gathered,
                       void *V_gathered, void *O, float *lse, void *stream);

/* Synchronise `stream`, then read and clear
 * the device error word: SYN_OK, SYN_ERR_TIMEOUT, SYN_ERR_BOUNDS or
 * SYN_ERR_CUDA.  After a device error the flags are reset. */
int syn_attn_sync_status(syn_attn_plan_t plan, void *stream);

int syn_attn_plan_query(syn_attn_plan_t plan, syn_attn_info_t *info);

/* Copy the chunk ready flags out (synchronous): R*split epochs, index
 * source_rank * split + chunk. */
int syn_attn_plan_flags(syn_attn_plan_t plan, uint32_t *flags);

#ifdef __cplusplus
}
#endif

#endif /* SYN_ATTN_H */
