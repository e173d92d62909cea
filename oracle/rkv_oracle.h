/*
 * CPU oracle for the R-KV compression event (TEST INFRASTRUCTURE ONLY).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library. The CUDA library never includes, links or calls it.
 *
 * Sources (page title, then section):
 *   [RKV-review]  "R-KV: Redundancy-Aware KV Cache Compression for Reasoning
 *                  Models" (hysenlabs project review), section "How R-KV
 *                  decides what to drop: budget, buffer and cross-layer scoring";
 *                  flag values in "Installing R-KV and running a first math
 *                  evaluation".
 *   [RKV-blog]    hotdry.top blog "KV缓存压缩三剑客：R-KV、EvolKV与Ada-KV的工程实践",
 *                  R-KV section (three steps: redundancy from key cosine
 *                  similarity, importance from multi-head attention, eviction
 *                  by high importance + low redundancy, lambda about 0.1) and
 *                  Ada-KV section (paged blocks of 16 or 32 tokens).
 *   [RKV-abstract] R-KV abstract entry on the fugumt "RedKnot" listing.
 *
 * Readings taken where the pages are silent:
 *   R1 softmax scale 1/sqrt(d); the window queries attend to all N cached keys,
 *      no causal mask.
 *   R2 GQA: query head q belongs to KV head floor(q / G), G = Hq / Hkv.
 *   R3 importance I_j = mean over the w*G (window position, query head) rows of
 *      the softmax probability of key j.
 *   R4 redundancy R_i = mean over j != i of cos(k_i, k_j); divisor N-1; keys
 *      only; a zero-norm key has cosine 0 with everything; N = 1 gives R = 0.
 *   R5 min-max over all N tokens of the head; a constant vector maps to 0.
 *   R6 S = lambda * I_hat - (1 - lambda) * R_hat; larger S is kept.
 *   R7 the last w positions are always kept and count toward the budget; from
 *      [0, N-w) the (budget - w) largest S are kept, equal S -> lower index;
 *      the kept list is ascending. N <= budget keeps everything.
 *   R8 compaction: slot j of the head receives token keep[j] (K and V), in
 *      logical-slot space; rows at and past the new length keep their old bytes.
 *   R9 paged layout [L][num_blocks][16][Hkv][d]: logical token t of sequence b
 *      lives in block block_table[b][t/16], row t%16. Blocks past
 *      ceil(k_b/16) up to ceil(N_b/16) are freed, in table order, sequences in
 *      batch order (CSR: freed_off[B+1], freed_ids[]). The table is not changed.
 *   R10 contiguous layout [L][B][Hkv][Nmax][d] frees no blocks.
 *
 * Arithmetic: bf16 inputs are widened exactly; every score is fp64.
 */
#ifndef RKV_ORACLE_H
#define RKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int layers, batch, kv_heads, q_heads, head_dim, max_seq_len;
    int paged;          /* 0: contiguous, 1: paged */
    int block_size;     /* paged only */
    int num_blocks;     /* paged only: pool blocks per layer */
    int max_blocks;     /* paged only: block_table row length */
    int budget, window;
    double mix_lambda;
} orc_problem;

/* Per-head definitions (one layer, one sequence, one KV head). */
void orc_importance(const uint16_t *q, int rows, const uint16_t *k, int n, int d, double *imp);
void orc_redundancy(const uint16_t *k, int n, int d, double *red);
/* R by the exact rank-one identity sum_{j!=i} cos = u_i.(sum_j u_j) - u_i.u_i,
 * u = k/|k| (two passes over the keys; equal to orc_redundancy up to fp64
 * rounding). */
void orc_redundancy_closed(const uint16_t *k, int n, int d, double *red);
void orc_minmax(const double *x, int n, double *out);
void orc_mix(const double *imp_hat, const double *red_hat, int n, double lam, double *s);
int  orc_select(const double *s, int n, int budget, int window, int32_t *keep);

/* Whole event over all (layer, sequence, KV head). scores (or NULL) receives
 * five planes [5][L][B][Hkv][Nmax]: I, R, I_hat, R_hat, S (zero past N_b).
 * Returns 0 on success, a negative code on invalid input. */
int orc_compress(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                 const uint16_t *q_window, const int32_t *seq_lens, const int32_t *block_table,
                 int32_t *keep_idx, int32_t *freed_off, int32_t *freed_ids,
                 int32_t *new_seq_lens, double *scores);

/* orc_compress with orc_redundancy_closed in place of the pairwise sum. */
int orc_compress_closed(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                        const uint16_t *q_window, const int32_t *seq_lens, const int32_t *block_table,
                        int32_t *keep_idx, int32_t *freed_off, int32_t *freed_ids,
                        int32_t *new_seq_lens, double *scores);

/* Compaction alone, with given kept indices [L][B][Hkv][budget] (-1 past k_b). */
int orc_compact(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                const int32_t *seq_lens, const int32_t *block_table, const int32_t *keep_idx);

/* Freed-block CSR and new lengths. */
int orc_freed_blocks(const orc_problem *p, const int32_t *seq_lens, const int32_t *block_table,
                     int32_t *freed_off, int32_t *freed_ids, int32_t *new_seq_lens);

#ifdef __cplusplus
}
#endif
#endif
