/*
 * Oracle for paged decode attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously-correct CPU loops in double precision.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library.  It shares no code, header or constant with the CUDA
 * library in paged_kv_cache_253_gb300/csrc, and must never be used by it.
 *
 * What it computes (kgptalkie "Day 28: PagedAttention / vLLM"):
 *   - "Follow One Token Address": a token position p of a request lives in
 *     logical block p / block_size at offset p % block_size, and the block
 *     table maps that logical block to a physical block id.
 *   - "The Block Table Is the Map" / "Batching Becomes More Flexible": the
 *     decode query of each request scores every cached key of that request,
 *     found through its own block table in logical (token) order, applies
 *     softmax and mixes the matching values.  Paging changes only where the
 *     keys live, never the result (the tutorial's verification recipe under
 *     "A Tiny Block-Table Example": the output must not move when the
 *     physical blocks do).
 *
 * Readings taken where the pages are silent:
 *   - grouped-query attention: query head h reads KV head h / (Hq / Hkv);
 *   - the decode query sees every position 0 .. L-1 of its request (its own
 *     freshly appended token included); no other mask exists in decode;
 *   - a request with L == 0 yields an all-zero output row.
 *
 * Pool layout used by the oracle (its own, the plain logical one):
 *   K[num_blocks][Hkv][block_size][D] and V likewise, stored as raw float32
 *   (kind 0), raw bfloat16 bits (kind 1) or double (kind 2: e.g. fp8 codes
 *   already multiplied by their scale); every element is widened exactly to
 *   double before use, and all arithmetic is double.
 *
 * Softmax is the textbook two-pass form: max, then exp-sum, then the
 * weighted sum of values — no online rescaling, no blocking.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_BLOCK (-2)

/* Address translation, "Follow One Token Address": divmod(pos, block_size),
 * then a table lookup.  Returns the physical block, writes the offset. */
int oracle_translate(int64_t pos, int block_size, const int32_t *table,
                     int table_len, int64_t *offset_out) {
    if (block_size <= 0 || pos < 0) return ORACLE_BAD_ARG;
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    if (logical_block >= table_len) return ORACLE_BAD_ARG;
    *offset_out = offset;
    return table[logical_block];
}

/* One stored element as a double.  bfloat16 is the upper half of an IEEE
 * float32, so its bits shifted left by 16 are that float32 exactly. */
static double elem(const void *base, size_t i, int kind) {
    float f;
    if (kind == 2) return ((const double *)base)[i];
    if (kind == 0) {
        f = ((const float *)base)[i];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        memcpy(&f, &bits, sizeof f);
    }
    return (double)f;
}

/* Attention of one query row over n keys/values given as element offsets.
 * x_j = scale * <q, k_j>;  p_j = exp(x_j - max) / sum;  out = sum_j p_j v_j. */
static void attend_rows(int n, int D, const double *q, const void *k_base,
                        const void *v_base, int kind, const size_t *rows, double scale,
                        double *scores, double *out) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return;
    double max_score = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * elem(k_base, rows[j] + d, kind);
        scores[j] = scale * dot;
        if (scores[j] > max_score) max_score = scores[j];
    }
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        scores[j] = exp(scores[j] - max_score);
        denom += scores[j];
    }
    for (int j = 0; j < n; ++j) {
        double w = scores[j] / denom;
        for (int d = 0; d < D; ++d) out[d] += w * elem(v_base, rows[j] + d, kind);
    }
}

/* Paged decode attention: one query per sequence and query head; keys and
 * values found through the sequence's block table.
 *   q            [S][Hq][D]                   (double)
 *   k_pool,v_pool[num_blocks][Hkv][B][D]       (raw elements of `kind`)
 *   block_tables [S][max_blocks_per_seq]      (int32 physical block ids)
 *   context_lens [S]                          (tokens visible to the query)
 *   out          [S][Hq][D]                   (double)
 * Sequences are processed in [seq_begin, seq_end) so a caller may split the
 * batch over threads; each call touches only its own rows of out. */
int oracle_paged_decode_range(int seq_begin, int seq_end, int Hq, int Hkv, int D,
                              int B, const double *q, const void *k_pool,
                              const void *v_pool, int kind, int num_blocks,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, double scale,
                              double *out) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || B <= 0) return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    int max_len = 0;
    for (int s = seq_begin; s < seq_end; ++s) {
        if (context_lens[s] < 0 || context_lens[s] > (int64_t)max_blocks_per_seq * B)
            return ORACLE_BAD_ARG;
        if (context_lens[s] > max_len) max_len = context_lens[s];
    }
    size_t *rows = malloc(sizeof(size_t) * (size_t)(max_len + 1));
    double *scores = malloc(sizeof(double) * (size_t)(max_len + 1));
    if (!rows || !scores) {
        free(rows); free(scores);
        return ORACLE_BAD_ARG;
    }
    int rc = ORACLE_OK;
    for (int s = seq_begin; s < seq_end && rc == ORACLE_OK; ++s) {
        int L = context_lens[s];
        const int32_t *table = block_tables + (size_t)s * max_blocks_per_seq;
        for (int h = 0; h < Hq && rc == ORACLE_OK; ++h) {
            int kv = h / G;
            for (int j = 0; j < L; ++j) {
                int64_t offset;
                int phys = oracle_translate(j, B, table, max_blocks_per_seq, &offset);
                if (phys < 0 || phys >= num_blocks) { rc = ORACLE_BAD_BLOCK; break; }
                rows[j] = (((size_t)phys * Hkv + kv) * B + (size_t)offset) * D;
            }
            if (rc != ORACLE_OK) break;
            attend_rows(L, D, q + ((size_t)s * Hq + h) * D, k_pool, v_pool, kind, rows,
                        scale, scores, out + ((size_t)s * Hq + h) * D);
        }
    }
    free(rows); free(scores);
    return rc;
}

int oracle_paged_decode(int S, int Hq, int Hkv, int D, int B, const double *q,
                        const void *k_pool, const void *v_pool, int kind, int num_blocks,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, double scale, double *out) {
    return oracle_paged_decode_range(0, S, Hq, Hkv, D, B, q, k_pool, v_pool, kind, num_blocks,
                                     block_tables, max_blocks_per_seq, context_lens,
                                     scale, out);
}

/* Contiguous reference: each sequence's keys and values stored back to back.
 *   k_seq, v_seq [sum_s L_s][Hkv][D] raw elements of `kind`; sequence s occupies rows
 *   seq_start[s] .. seq_start[s] + L_s - 1. */
int oracle_contiguous_decode(int S, int Hq, int Hkv, int D, const double *q,
                             const void *k_seq, const void *v_seq, int kind,
                             const int64_t *seq_start, const int32_t *context_lens,
                             double scale, double *out) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    int max_len = 0;
    for (int s = 0; s < S; ++s) {
        if (context_lens[s] < 0) return ORACLE_BAD_ARG;
        if (context_lens[s] > max_len) max_len = context_lens[s];
    }
    size_t *rows = malloc(sizeof(size_t) * (size_t)(max_len + 1));
    double *scores = malloc(sizeof(double) * (size_t)(max_len + 1));
    if (!rows || !scores) {
        free(rows); free(scores);
        return ORACLE_BAD_ARG;
    }
    for (int s = 0; s < S; ++s) {
        for (int h = 0; h < Hq; ++h) {
            int kv = h / G;
            for (int j = 0; j < context_lens[s]; ++j) {
                rows[j] = ((size_t)(seq_start[s] + j) * Hkv + kv) * D;
            }
            attend_rows(context_lens[s], D, q + ((size_t)s * Hq + h) * D, k_seq, v_seq,
                        kind, rows, scale, scores, out + ((size_t)s * Hq + h) * D);
        }
    }
    free(rows); free(scores);
    return ORACLE_OK;
}
