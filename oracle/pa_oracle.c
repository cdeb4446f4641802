/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged-attention decode and the
 * slot-mapping cache write.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The CUDA library never
 * includes, links or calls this file, and the two share no source: this file
 * restates the method from the pages it cites, nothing more.
 *
 * Sources (page title, section):
 *   [P1] "vLLM PagedAttention: from memory fragmentation to slot mapping"
 *        §2 (block count, tail waste), §3 (logical block / offset / slot),
 *        §4 (the address formula under the minimal allocator).
 *   [P2] "PagedAttention" (LLM glossary), section "contiguous vs page-table
 *        reference": K/V are gathered by table into contiguous rows
 *        (gather_paged), then plain attention runs on them (attend_one);
 *        query heads are grouped with repeat_interleave (expand_kv).
 *   [P3] PagedAttention engineering notes (nxmr.cn) §4.2: copy-on-write
 *        copies a shared, partly filled block before it is written.
 *   [P4] "vLLM source walkthrough: PagedAttention and Continuous Batching"
 *        §1.8: the V2 kernel splits a sequence's blocks into partitions and
 *        a reduce step merges them.
 *   [P5] "Efficient Memory Management for LLM Serving with PagedAttention"
 *        (paper notes), the 10-token worked example: per-block raw scores,
 *        one global softmax over all of them, weighted V per block.
 *
 * Precision: every score, weight and accumulator is a double.  Inputs are
 * fp32 or bf16; a bf16 value is widened exactly (its 16 bits are the top half
 * of an IEEE binary32).  exp() is the C library's.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): query head h uses kv head floor(h / (Hq/Hkv)); a sequence of length
 * 0 yields a zero output row; a negative slot in slot_mapping means "skip";
 * a table entry that a needed position maps to must lie in [0, num_blocks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* ---- element access ---------------------------------------------------- */

static double widen(const void* base, int64_t index, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[index];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[index] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---- addressing [P1 §2, §3, §4] ---------------------------------------- */

/* n = ceil(S / B) blocks hold S tokens [P1 §2]. */
int64_t oracle_blocks_needed(int64_t num_tokens, int32_t block_size) {
    return (num_tokens + block_size - 1) / block_size;
}

/* w = n*B - S slots of the last block stay empty, 0 <= w < B [P1 §2]. */
int64_t oracle_tail_waste(int64_t num_tokens, int32_t block_size) {
    return oracle_blocks_needed(num_tokens, block_size) * block_size - num_tokens;
}

/* b_l = floor(p/B), o = p mod B, b_p = table[b_l], slot = b_p*B + o
 * [P1 §3, §4].  Returns -1 when the table entry is negative (padding). */
int64_t oracle_slot(const int32_t* table, int32_t block_size, int64_t position) {
    int64_t logical = position / block_size;
    int64_t offset = position % block_size;
    int64_t physical = table[logical];
    if (physical < 0) return -1;
    return physical * block_size + offset;
}

/* ---- gather [P2, gather_paged] ----------------------------------------- */

/* Copy the T logically contiguous K (or V) rows of kv head g of one sequence
 * into dst[T][D] (fp64), reading each position through the table.  The cache
 * is [num_blocks][Hkv][B][D]: the slot's block is slot / B and its row within
 * the block is slot % B.  Returns 0, or -1 if a needed entry is outside
 * [0, num_blocks). */
static int gather_rows(const void* cache, int dtype, int32_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                       const int32_t* table, int64_t T, int32_t g, double* dst) {
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = oracle_slot(table, block_size, t);
        if (slot < 0) return -1;
        int64_t block = slot / block_size;
        int64_t row = slot % block_size;
        if (block >= num_blocks) return -1;
        int64_t base = ((block * num_kv_heads + g) * block_size + row) * head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            dst[t * head_dim + d] = widen(cache, base + d, dtype);
    }
    return 0;
}

/* ---- dense attention for one query row [P2, attend_one; P1 §7] ---------- */

/* out = softmax(scale * K q) V over T contiguous rows; max-subtracted. */
void oracle_attend(const double* q, const double* K, const double* V, int64_t T,
                   int32_t D, double scale, double* out) {
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (T <= 0) return;
    double* s = (double*)malloc(sizeof(double) * (size_t)T);
    double m = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += q[d] * K[t * D + d];
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int64_t t = 0; t < T; ++t)
        for (int32_t d = 0; d < D; ++d) out[d] += s[t] * V[t * D + d];
    for (int32_t d = 0; d < D; ++d) out[d] /= l;
    free(s);
}

/* ---- decode: gather, then dense attention ------------------------------ */

/*
 * out[i][h][:] for the requested (i, h) pairs (pairs == NULL: all N*Hq).
 * q is [N][Hq][D], caches are [num_blocks][Hkv][B][D], block_tables is
 * [N][max_blocks], seq_lens is [N]; out is [N][Hq][D] fp64 and only the
 * requested rows are written.  Returns 0, or the number of pairs whose
 * gather met an invalid table entry (their rows are NaN).
 */
int64_t oracle_decode(const void* q, const void* k_cache, const void* v_cache, int dtype,
                      int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                      int32_t head_dim, const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                      double scale, const int64_t* pairs, int64_t num_pairs, double* out) {
    int32_t group = num_q_heads / num_kv_heads;
    int64_t total = pairs ? num_pairs : (int64_t)num_seqs * num_q_heads;
    int64_t bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
    for (int64_t u = 0; u < total; ++u) {
        int64_t i = pairs ? pairs[2 * u] : u / num_q_heads;
        int64_t h = pairs ? pairs[2 * u + 1] : u % num_q_heads;
        int64_t T = seq_lens[i];
        int32_t g = (int32_t)(h / group);
        double* row = out + (i * num_q_heads + h) * head_dim;
        size_t rows = (size_t)(T > 0 ? T : 1) * (size_t)head_dim;
        double* K = (double*)malloc(sizeof(double) * rows);
        double* V = (double*)malloc(sizeof(double) * rows);
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t* table = block_tables + i * (int64_t)max_blocks;
        int ok = gather_rows(k_cache, dtype, num_blocks, block_size, num_kv_heads,
                             head_dim, table, T, g, K) == 0 &&
                 gather_rows(v_cache, dtype, num_blocks, block_size, num_kv_heads,
                             head_dim, table, T, g, V) == 0;
        if (ok) {
            for (int32_t d = 0; d < head_dim; ++d)
                qv[d] = widen(q, (i * num_q_heads + h) * head_dim + d, dtype);
            oracle_attend(qv, K, V, T, head_dim, scale, row);
        } else {
            for (int32_t d = 0; d < head_dim; ++d) row[d] = NAN;
            bad += 1;
        }
        free(K);
        free(V);
        free(qv);
    }
    return bad;
}

/* ---- partitioned decode and merge [P4 §1.8 V2; P5 blockwise example] ---- */

/*
 * Split each sequence's T tokens into partitions of P tokens (the last one
 * shorter) and, for partition p of pair (i, h), return
 *   m_p   = max over its tokens of s_t = scale * q.k_t      (natural log units)
 *   l_p   = sum over its tokens of exp(s_t - m_p)
 *   acc_p = sum over its tokens of exp(s_t - m_p) * v_t      ([D])
 * Outputs are [N][Hq][max_parts] for m, l and [N][Hq][max_parts][D] for acc;
 * partitions at or beyond ceil(T/P) are left untouched.  Returns the number
 * of pairs that met an invalid table entry.
 */
int64_t oracle_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                               int dtype, int32_t num_blocks, int32_t block_size,
                               int32_t num_kv_heads, int32_t head_dim,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t num_seqs,
                               int32_t num_q_heads, double scale, int32_t partition_tokens,
                               int32_t max_parts, double* m_out, double* l_out,
                               double* acc_out) {
    int32_t group = num_q_heads / num_kv_heads;
    int64_t total = (int64_t)num_seqs * num_q_heads;
    int64_t bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
    for (int64_t u = 0; u < total; ++u) {
        int64_t i = u / num_q_heads, h = u % num_q_heads;
        int64_t T = seq_lens[i];
        int32_t g = (int32_t)(h / group);
        size_t rows = (size_t)(T > 0 ? T : 1) * (size_t)head_dim;
        double* K = (double*)malloc(sizeof(double) * rows);
        double* V = (double*)malloc(sizeof(double) * rows);
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t* table = block_tables + i * (int64_t)max_blocks;
        if (gather_rows(k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim,
                        table, T, g, K) != 0 ||
            gather_rows(v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim,
                        table, T, g, V) != 0) {
            bad += 1;
        } else {
            for (int32_t d = 0; d < head_dim; ++d)
                qv[d] = widen(q, (i * num_q_heads + h) * head_dim + d, dtype);
            int64_t parts = (T + partition_tokens - 1) / partition_tokens;
            for (int64_t p = 0; p < parts && p < max_parts; ++p) {
                int64_t t0 = p * partition_tokens;
                int64_t t1 = t0 + partition_tokens < T ? t0 + partition_tokens : T;
                int64_t cell = u * max_parts + p;
                double m = -INFINITY;
                for (int64_t t = t0; t < t1; ++t) {
                    double dot = 0.0;
                    for (int32_t d = 0; d < head_dim; ++d) dot += qv[d] * K[t * head_dim + d];
                    if (scale * dot > m) m = scale * dot;
                }
                double l = 0.0;
                double* acc = acc_out + cell * head_dim;
                for (int32_t d = 0; d < head_dim; ++d) acc[d] = 0.0;
                for (int64_t t = t0; t < t1; ++t) {
                    double dot = 0.0;
                    for (int32_t d = 0; d < head_dim; ++d) dot += qv[d] * K[t * head_dim + d];
                    double w = exp(scale * dot - m);
                    l += w;
                    for (int32_t d = 0; d < head_dim; ++d) acc[d] += w * V[t * head_dim + d];
                }
                m_out[cell] = m;
                l_out[cell] = l;
            }
        }
        free(K);
        free(V);
        free(qv);
    }
    return bad;
}

/* Log-sum-exp merge of n partials: M = max m_p,
 * out = sum_p e^(m_p - M) acc_p / sum_p e^(m_p - M) l_p. */
void oracle_merge(int32_t num_parts, const double* m, const double* l, const double* acc,
                  int32_t head_dim, double* out) {
    double M = -INFINITY;
    for (int32_t p = 0; p < num_parts; ++p)
        if (m[p] > M) M = m[p];
    double L = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (num_parts <= 0) return;
    for (int32_t p = 0; p < num_parts; ++p) {
        double w = exp(m[p] - M);
        L += w * l[p];
        for (int32_t d = 0; d < head_dim; ++d) out[d] += w * acc[(int64_t)p * head_dim + d];
    }
    for (int32_t d = 0; d < head_dim; ++d) out[d] /= L;
}

/* ---- cache write through slot_mapping [P1 §6; P5 block lifecycle] ------ */

/*
 * For each new token j in index order, with s = slot_mapping[j] >= 0:
 * block = s / B, row = s % B, and for every kv head h the D elements of
 * k[j][h][:] are stored bit for bit at k_cache[block][h][row][:] (same for v).
 * Negative slots are skipped.  Slots at or beyond num_blocks*B are skipped
 * and counted; the count is returned.
 */
int64_t oracle_write_kv(const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, void* k_cache, void* v_cache,
                        int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                        int32_t head_dim, int32_t elem_bytes) {
    int64_t rejected = 0;
    size_t row_bytes = (size_t)head_dim * (size_t)elem_bytes;
    for (int64_t j = 0; j < num_tokens; ++j) {
        int64_t s = slot_mapping[j];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) {
            rejected += 1;
            continue;
        }
        int64_t block = s / block_size;
        int64_t row = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            size_t src = (size_t)(j * num_kv_heads + h) * row_bytes;
            size_t dst = (size_t)((block * num_kv_heads + h) * block_size + row) * row_bytes;
            memcpy((char*)k_cache + dst, (const char*)k + src, row_bytes);
            memcpy((char*)v_cache + dst, (const char*)v + src, row_bytes);
        }
    }
    return rejected;
}

/* ---- multi-query (chunked prefill) attention ---------------------------- */

/*
 * Sequence i owns the packed query rows [query_start[i], query_start[i+1]):
 * its last L_i = query_start[i+1] - query_start[i] positions, so row r sits
 * at position p = T_i - L_i + (r - query_start[i]) and attends to keys
 * 0..p of its sequence (causal).  Prefill and decode rows share one batch,
 * a decode row being a sequence with L_i = 1 ("vLLM source walkthrough"
 * §2.8: chunked prefill processes part of a prompt per step, decode one
 * token; "vLLM PagedAttention: from memory fragmentation to slot mapping"
 * §6: query start locations slice the flat tokens per request, positions set
 * the causal boundary).  q and out are [total_q][Hq][D].  For each row and
 * head: gather keys 0..p through the table, then dense attention.  Returns
 * the number of (row, head) results left NaN because L_i > T_i or a needed
 * table entry was invalid.
 */
int64_t oracle_prefill(const void* q, const int32_t* query_start, const void* k_cache,
                       const void* v_cache, int dtype, int32_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                       int32_t max_blocks, const int32_t* seq_lens, int32_t num_seqs,
                       int32_t num_q_heads, double scale, double* out) {
    int32_t group = num_q_heads / num_kv_heads;
    int64_t total_rows = query_start[num_seqs];
    int64_t bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
    for (int64_t u = 0; u < total_rows * num_q_heads; ++u) {
        int64_t r = u / num_q_heads, h = u % num_q_heads;
        int64_t i = 0;
        while (i + 1 < num_seqs && query_start[i + 1] <= r) ++i;
        int64_t L = query_start[i + 1] - query_start[i];
        int64_t T = seq_lens[i];
        double* row = out + (r * num_q_heads + h) * head_dim;
        int64_t p = T - L + (r - query_start[i]);
        if (L > T || p < 0) {
            for (int32_t d = 0; d < head_dim; ++d) row[d] = NAN;
            bad += 1;
            continue;
        }
        int64_t n = p + 1;
        int32_t g = (int32_t)(h / group);
        double* K = (double*)malloc(sizeof(double) * (size_t)n * (size_t)head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)n * (size_t)head_dim);
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t* table = block_tables + i * (int64_t)max_blocks;
        if (gather_rows(k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, table,
                        n, g, K) == 0 &&
            gather_rows(v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, table,
                        n, g, V) == 0) {
            for (int32_t d = 0; d < head_dim; ++d)
                qv[d] = widen(q, (r * num_q_heads + h) * head_dim + d, dtype);
            oracle_attend(qv, K, V, n, head_dim, scale, row);
        } else {
            for (int32_t d = 0; d < head_dim; ++d) row[d] = NAN;
            bad += 1;
        }
        free(K);
        free(V);
        free(qv);
    }
    return bad;
}

/* ---- block copy for copy-on-write and swap ------------------------------ */

/*
 * For each pair (src, dst) in index order, every byte of physical block src
 * of the source K and V caches is copied to block dst of the destination
 * caches.  A block is block_bytes contiguous bytes of a [num_blocks][...]
 * cache.  This is the copy a copy-on-write performs before a shared, partly
 * filled block is written (nxmr.cn article §4.2: take a new block, copy the
 * old block's K/V into it, point the table at it), and the copy that swaps a
 * preempted sequence's blocks between GPU and CPU memory (paper notes,
 * swapping).  Pairs naming a block outside either cache are skipped and
 * counted; the count is returned.
 */
int64_t oracle_copy_blocks(const void* src_k, const void* src_v, int32_t src_blocks,
                           void* dst_k, void* dst_v, int32_t dst_blocks, const int64_t* pairs,
                           int64_t num_pairs, int64_t block_bytes) {
    int64_t rejected = 0;
    for (int64_t j = 0; j < num_pairs; ++j) {
        int64_t s = pairs[2 * j], d = pairs[2 * j + 1];
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
            rejected += 1;
            continue;
        }
        memcpy((char*)dst_k + d * block_bytes, (const char*)src_k + s * block_bytes,
               (size_t)block_bytes);
        memcpy((char*)dst_v + d * block_bytes, (const char*)src_v + s * block_bytes,
               (size_t)block_bytes);
    }
    return rejected;
}

/* ---- slots from (sequence, position) ------------------------------------ */

/*
 * slot of token j = table[seq_ids[j]][positions[j] / B] * B + positions[j] % B
 * ("vLLM PagedAttention: from memory fragmentation to slot mapping" §3, §6:
 * positions plus the block table give the slot mapping).  -1 when the
 * sequence id or position is negative or outside the table, or the entry is
 * negative.
 */
void oracle_slots_from_positions(const int32_t* seq_ids, const int32_t* positions,
                                 int64_t num_tokens, const int32_t* block_tables,
                                 int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                                 int64_t* slots) {
    for (int64_t j = 0; j < num_tokens; ++j) {
        int64_t s = seq_ids[j], p = positions[j];
        if (s < 0 || s >= num_seqs || p < 0 || p >= (int64_t)max_blocks * block_size) {
            slots[j] = -1;
            continue;
        }
        slots[j] = oracle_slot(block_tables + s * max_blocks, block_size, p);
    }
}

/* ---- threading --------------------------------------------------------- */

void oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int32_t oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
