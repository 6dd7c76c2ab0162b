/*
 * syn_oracle.c -- plain CPU oracle for the chunk-overlapped operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it computes.  The Syncopate summary page (OSDI 2026, "Experiments",
 * paper §6.1) evaluates three GEMM operators, AG-GEMM, GEMM-RS and GEMM-AR,
 * taken in their standard tensor-parallel meaning.  Its method section (paper
 * §5.1-§5.2, Figs. 6-7) and the pith review's falsification test ("run the
 * fused kernel beside the original ... outputs match") say that chunk-level
 * overlap changes only WHEN data moves and in which order tiles run, never
 * WHAT is computed.  So this oracle is the plain definition of each operator:
 *
 *   AG-GEMM  : G = concat_q(shard_q)          (bit copy, R shards of M_r rows)
 *              C = bf16_rne(G . B)
 *   GEMM-RS  : P = A . B                       (fp32, never rounded)
 *              send[rows_q] = P[rows_q], q != r
 *              out_r = bf16_rne(P[rows_r] + sum_{q != r, ascending q} peer_q[rows_r])
 *   GEMM-AR  : out = bf16_rne(P + sum_{q != r, ascending q} peer_q);  publish = P
 *   ring attention (sequence parallel, the pages' RingAttention workload):
 *              O_r = softmax(scale . Q_r K^T [+ causal mask]) V over the keys of
 *              all R ranks, in fp64 (see oracle_ring_attention)
 *   A2A-GEMM : G = concat_q(part_q), parts of rows_from[q] rows (bit copy),
 *              C = bf16_rne(G . B)   -- the MoE-style all-to-all + expert
 *              GEMM that the paper's sensitivity study (§6.3, Fig. 11)
 *              tunes beside the other three
 *
 * Arithmetic.  bf16 inputs are widened exactly (bits << 16).  Every dot
 * product accumulates in fp32, sequentially in k, starting from +0.0.  The
 * peers are added in fp32 in ascending q, skipping the local rank, after the
 * dot product.  The result is rounded once, round-to-nearest-even, to bf16.
 * A bf16 x bf16 product has at most 16 significant bits and is therefore
 * exact in fp32, so fused multiply-add and multiply-then-add agree bit for
 * bit; the file is still built with -ffp-contract=off.
 *
 * Threading.  OpenMP over output rows only; the per-element operation order is
 * fixed, so every thread count gives the same bits.
 *
 * Row ranges.  Every entry point computes a half-open row range [row0, row1)
 * and writes its outputs compactly: output row i goes to index (i - row0).
 * This lets callers sample rows of a large problem.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float widen_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a float to the nearest bf16, ties to even (IEEE 754 roundTiesToEven
 * applied to the 8-bit significand).  Overflow rounds to infinity.  NaN stays
 * a (quiet) NaN. */
uint16_t oracle_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Element-wise oracle_bf16_rne over an array. */
void oracle_bf16_rne_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(x[i]);
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One output row of the plain GEMM: acc[j] = sum_k a[k] * B[k][j] in fp32,
 * sequential in k.  B is row-major [K, N] with row stride ldb elements. */
static void dot_row(const uint16_t *a, const uint16_t *B, int64_t ldb,
                    int64_t K, int64_t N, float *acc)
{
    for (int64_t j = 0; j < N; ++j)
        acc[j] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        const float ak = widen_bf16(a[k]);
        const uint16_t *bk = B + k * ldb;
        for (int64_t j = 0; j < N; ++j)
            acc[j] = acc[j] + ak * widen_bf16(bk[j]);
    }
}

/* AllGather: gathered[q*M_r + i][k] = shard_q[i][k].  Pure bit copy. */
void oracle_gather(int R, int64_t M_r, int64_t K,
                   const uint16_t *const *shards, uint16_t *gathered)
{
    for (int q = 0; q < R; ++q)
        memcpy(gathered + (int64_t)q * M_r * K, shards[q],
               (size_t)(M_r * K) * sizeof(uint16_t));
}

/* P[i - row0][j] = sum_k A[i][k] * B[k][j], fp32, not rounded.
 * A is row-major [*, K] (lda = K), B row-major [K, N]. */
void oracle_gemm_f32(const uint16_t *A, const uint16_t *B, int64_t K, int64_t N,
                     int64_t row0, int64_t row1, float *P)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = row0; i < row1; ++i)
        dot_row(A + i * K, B, N, K, N, P + (i - row0) * N);
}

/* AG-GEMM over rows [row0, row1) of the gathered row space.
 * The A row for gathered row i is row (i mod M_r) of shard (i / M_r): that is
 * the definition of the gathered matrix.  C is written compactly.
 * If `gathered` is not NULL the full gathered buffer [R*M_r, K] is also
 * written (independently of the row range). */
void oracle_ag_gemm(int R, int64_t M_r, int64_t K, int64_t N,
                    const uint16_t *const *shards, const uint16_t *B,
                    int64_t row0, int64_t row1,
                    uint16_t *gathered, uint16_t *C)
{
    if (gathered)
        oracle_gather(R, M_r, K, shards, gathered);
#pragma omp parallel
    {
        float *acc = (float *)malloc((size_t)N * sizeof(float));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = row0; i < row1; ++i) {
            const uint16_t *a = shards[i / M_r] + (i % M_r) * K;
            dot_row(a, B, N, K, N, acc);
            uint16_t *c = C + (i - row0) * N;
            for (int64_t j = 0; j < N; ++j)
                c[j] = oracle_bf16_rne(acc[j]);
        }
        free(acc);
    }
}

/* A2A-GEMM over rows [row0, row1) of the received row space.
 * The all-to-all hands rank r one part per source rank q (rows_from[q] rows,
 * possibly none); the expert's input is those parts stacked in ascending q:
 *   G[off_q + i] = part_q[i],  off_q = rows_from[0] + ... + rows_from[q-1]
 *   C = bf16_rne(G . B)
 * The part holding row i is found by walking the parts in order.  If
 * `gathered` is not NULL the whole stacked matrix [sum rows_from, K] is
 * written too (independently of the row range). */
void oracle_a2a_gemm(int R, const int64_t *rows_from, int64_t K, int64_t N,
                     const uint16_t *const *parts, const uint16_t *B,
                     int64_t row0, int64_t row1,
                     uint16_t *gathered, uint16_t *C)
{
    if (gathered) {
        int64_t off = 0;
        for (int q = 0; q < R; ++q) {
            if (rows_from[q] > 0)
                memcpy(gathered + off * K, parts[q],
                       (size_t)(rows_from[q] * K) * sizeof(uint16_t));
            off += rows_from[q];
        }
    }
#pragma omp parallel
    {
        float *acc = (float *)malloc((size_t)N * sizeof(float));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = row0; i < row1; ++i) {
            int q = 0;
            int64_t off = 0;
            while (i >= off + rows_from[q]) {
                off += rows_from[q];
                ++q;
            }
            dot_row(parts[q] + (i - off) * K, B, N, K, N, acc);
            uint16_t *c = C + (i - row0) * N;
            for (int64_t j = 0; j < N; ++j)
                c[j] = oracle_bf16_rne(acc[j]);
        }
        free(acc);
    }
}

/* Reduction step shared by the definitions of GEMM-RS and GEMM-AR, written
 * out for one element: ((p + peer_{q1}) + peer_{q2}) + ..., ascending q,
 * skipping the local rank r, all in fp32. */
static float reduce_peers(float p, int R, int r, const float *const *peers,
                          int64_t offset)
{
    float s = p;
    for (int q = 0; q < R; ++q)
        if (q != r)
            s = s + peers[q][offset];
    return s;
}

/* GEMM-RS, reduced part: out_r rows [i0, i1) of the local M_r = M/R rows.
 * out_r[i][j] = rne(P[r*M_r + i][j] + sum_{q != r} peer_q[r*M_r + i][j]).
 * peers[q] is fp32 [M, N]; peers[r] is never read. */
void oracle_gemm_rs_out(int R, int r, int64_t M, int64_t K, int64_t N,
                        const uint16_t *A, const uint16_t *B,
                        const float *const *peers,
                        int64_t i0, int64_t i1, uint16_t *out_r)
{
    const int64_t M_r = M / R;
#pragma omp parallel
    {
        float *acc = (float *)malloc((size_t)N * sizeof(float));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = i0; i < i1; ++i) {
            const int64_t g = (int64_t)r * M_r + i;
            dot_row(A + g * K, B, N, K, N, acc);
            uint16_t *o = out_r + (i - i0) * N;
            for (int64_t j = 0; j < N; ++j)
                o[j] = oracle_bf16_rne(reduce_peers(acc[j], R, r, peers, g * N + j));
        }
        free(acc);
    }
}

/* GEMM-RS, send part: for global rows g in [row0, row1) that belong to a rank
 * q != r, send[g - row0][j] = P[g][j] (fp32, unrounded).  Rows of rank r are
 * not written. */
void oracle_gemm_rs_send(int R, int r, int64_t M, int64_t K, int64_t N,
                         const uint16_t *A, const uint16_t *B,
                         int64_t row0, int64_t row1, float *send)
{
    const int64_t M_r = M / R;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t g = row0; g < row1; ++g) {
        if (g / M_r == r)
            continue;
        dot_row(A + g * K, B, N, K, N, send + (g - row0) * N);
    }
}

/* GEMM-AR over global rows [row0, row1):
 * out[g][j] = rne(P[g][j] + sum_{q != r} peer_q[g][j]); publish = P if given. */
void oracle_gemm_ar(int R, int r, int64_t M, int64_t K, int64_t N,
                    const uint16_t *A, const uint16_t *B,
                    const float *const *peers,
                    int64_t row0, int64_t row1,
                    uint16_t *out, float *publish)
{
    (void)M;
#pragma omp parallel
    {
        float *acc = (float *)malloc((size_t)N * sizeof(float));
#pragma omp for schedule(dynamic, 1)
        for (int64_t g = row0; g < row1; ++g) {
            dot_row(A + g * K, B, N, K, N, acc);
            if (publish)
                memcpy(publish + (g - row0) * N, acc, (size_t)N * sizeof(float));
            uint16_t *o = out + (g - row0) * N;
            for (int64_t j = 0; j < N; ++j)
                o[j] = oracle_bf16_rne(reduce_peers(acc[j], R, r, peers, g * N + j));
        }
        free(acc);
    }
}

/* Ring attention forward of rank r (sequence parallelism: every rank holds
 * S_r consecutive tokens; rank q's tokens have global positions
 * [q*S_r, (q+1)*S_r)).  Layouts are token-major: Q [S_r, H_q, d],
 * K[q] and V[q] [S_r, H_kv, d], bf16.  Query head h reads KV head
 * h / (H_q / H_kv).  For query row i (global position r*S_r + i) and head h,
 * over the R*S_r keys j in global order:
 *   s_j   = scale * sum_k Q[i][h][k] * K[j][hk][k]        (fp64)
 *   causal: keys with j > r*S_r + i take no part
 *   O[i][h][:] = sum_j exp(s_j - m) V[j][hk][:] / sum_j exp(s_j - m),  m = max_j s_j
 *   lse[i][h]  = m + log(sum_j exp(s_j - m))               (natural log)
 * Rows [row0, row1) of the rank's queries are computed and written compactly
 * (O [(row1-row0), H_q, d], lse [(row1-row0), H_q], both fp64; lse may be
 * NULL).  Subtracting m changes nothing mathematically; it keeps exp finite. */
void oracle_ring_attention(int R, int r, int64_t S_r, int H_q, int H_kv, int d, int causal,
                           double scale, const uint16_t *Q, const uint16_t *const *K,
                           const uint16_t *const *V, int64_t row0, int64_t row1,
                           double *O, double *lse)
{
    const int G = H_q / H_kv;
    const int64_t S = (int64_t)R * S_r;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)S * sizeof(double));
        double *q = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (int64_t i = row0; i < row1; ++i) {
            for (int h = 0; h < H_q; ++h) {
                const int hk = h / G;
                const int64_t pos = (int64_t)r * S_r + i;
                const int64_t nkeys = causal ? pos + 1 : S;
                for (int k = 0; k < d; ++k)
                    q[k] = (double)widen_bf16(Q[(i * H_q + h) * d + k]);
                double m = -INFINITY;
                for (int64_t j = 0; j < nkeys; ++j) {
                    const uint16_t *kr = K[j / S_r] + ((j % S_r) * H_kv + hk) * d;
                    double acc = 0.0;
                    for (int k = 0; k < d; ++k)
                        acc += q[k] * (double)widen_bf16(kr[k]);
                    s[j] = scale * acc;
                    if (s[j] > m)
                        m = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < nkeys; ++j) {
                    s[j] = exp(s[j] - m);
                    l += s[j];
                }
                double *o = O + ((i - row0) * H_q + h) * d;
                for (int k = 0; k < d; ++k)
                    o[k] = 0.0;
                for (int64_t j = 0; j < nkeys; ++j) {
                    const uint16_t *vr = V[j / S_r] + ((j % S_r) * H_kv + hk) * d;
                    for (int k = 0; k < d; ++k)
                        o[k] += s[j] * (double)widen_bf16(vr[k]);
                }
                for (int k = 0; k < d; ++k)
                    o[k] /= l;
                if (lse)
                    lse[(i - row0) * H_q + h] = m + log(l);
            }
        }
        free(s);
        free(q);
    }
}
