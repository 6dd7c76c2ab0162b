/*
 * syn_proto.h -- CPU emulation of the chunk ready-flag protocol (test
 * harness, libsynproto.so; no CUDA).
 *
 * Runs the plan builder's real schedule (arrival order, tile order) and the
 * protocol's shared logic (protocol.h: epoch flags, double-buffered slice
 * counters, last-arriver publication, the persistent tile walk, chunk ranges,
 * transfer rows) with host threads in place of the GPU's stagers and tile
 * walkers (Syncopate summary page, method ¶2-¶3: tiles wait only on the chunks
 * they consume; stagers publish a chunk once its bytes have landed).  Flags
 * and counters are std::atomic with release/acquire, the copies are memcpy of
 * byte rows, and every consumer checks the bytes of every row it waits for.
 * Faults are injected on the host: a transfer whose flag is never published
 * (the call must end in SYN_ERR_TIMEOUT, never hang) or published late.
 */
#ifndef SYN_PROTO_H
#define SYN_PROTO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Returned per call besides SYN_OK / SYN_ERR_TIMEOUT (syn.h): a consumer saw
 * bytes that did not match the source after its wait succeeded. */
#define SYN_PROTO_STALE_DATA (-100)

typedef struct {
    int op;               /* 0 AG-GEMM, 1 GEMM-RS, 2 GEMM-AR                  */
    int R, rank;
    int64_t M, N, K;      /* shapes of the plan (bytes per row: AG K*2, RS/AR N*4) */
    int split;            /* chunks per rank row block                        */
    int order;            /* syn_order_t                                      */
    int tile_m, tile_n;   /* 128 or 256; 128 or 256                           */
    int walkers;          /* persistent tile walkers (threads)                */
    int stagers;          /* staging workers (threads)                        */
    int64_t slice_bytes;  /* bytes per staged slice (>= 16)                   */
    int calls;            /* calls run back to back (epochs 1..calls)         */
    int drop_transfer;    /* arrival index whose flag is never published, -1  */
    int drop_call;        /* the call (1-based) that drops it                 */
    int delay_transfer;   /* arrival index whose flag is published late, -1   */
    int delay_us;         /* how late                                         */
    int timeout_us;       /* bound on every wait                              */
    int jitter_us;        /* stagers sleep up to this long before each slice  */
    uint64_t seed;        /* jitter and data seed                             */
    int mutation;         /* 0; 1 = a deliberately broken protocol for testing
                             the harness: the last stager of a transfer
                             publishes its flag before its own copy and only
                             then copies (after a 2 ms pause), so consumers
                             must report SYN_PROTO_STALE_DATA                 */
    const int64_t *rows_from; /* NULL, or (op 0 only) the A2A-GEMM row count
                             each source sends, R entries; M is then ignored
                             and taken as their sum                           */
} syn_proto_cfg_t;

/* Run cfg->calls calls.  status[c] receives the status of call c + 1; after a
 * failed call the protocol state is reset as syn_sync_status does.
 * tiles_checked[c] counts the tiles whose waited-for rows were verified.
 * Returns SYN_OK, or SYN_ERR_INVALID for a configuration the plan builder
 * rejects (syn_proto_last_error() says why). */
int syn_proto_emulate(const syn_proto_cfg_t *cfg, int *status, int64_t *tiles_checked);

const char *syn_proto_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SYN_PROTO_H */
