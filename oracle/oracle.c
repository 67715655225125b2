/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the paged-KV-cache
 * hot path computes, in fp64.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may call it; the product library never
 * links, loads or calls anything in this directory, and this file includes no
 * header of the product.
 *
 * Sources (three web pages, cited by title and section):
 *   [P1] "Makale Bulteni -- vAttention" (cmlonder.com), section
 *        "Iddia ve Gerceklik: vAttention".
 *   [P2] "Makale Bulteni -- PagedAttention ve vLLM" (cmlonder.com), section
 *        "Iddia ve Gerceklik: PagedAttention ve vLLM".
 *   [P3] "PagedAttention Nedir?" (bitcanli.com), sections "PagedAttention
 *        Nedir?", "PagedAttention Nasil Calisir?", "FlashAttention ile Ayni mi?",
 *        "Sik Sorulan Sorular".
 *
 * What the pages fix: the KV cache is split into fixed-size token blocks that
 * may sit anywhere in memory [P3 "PagedAttention Nedir?"]; a per-sequence
 * block (page) table maps logical blocks to physical ones [P2; P3 "Nasil
 * Calisir?" step 3]; attention reads the blocks through the table [P3 step 4];
 * the logical token order is preserved while physical placement is free
 * [P3 "PagedAttention Nedir?"].  Paging therefore does not change the maths:
 * the result is ordinary softmax attention over each sequence's logical K/V
 * [P3 FAQ "Yanitlarin dogrulugunu artirir mi?": only small numerical
 * differences].  The oracle follows that reading literally: it first
 * reassembles each sequence's logical K and V from the pool through the block
 * table, converts them exactly to fp64, and then evaluates
 *     s_j = scale * <q, k_j>,  w_j = exp(s_j - max s),  o = sum_j w_j v_j / sum_j w_j
 * with lse = max s + log(sum_j w_j).  No blocking, tiling, online softmax or
 * split of the key range is used here.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes):
 *   - pool layout [num_blocks][num_kv_heads][block_size][head_dim], separate
 *     K and V pools; slot s of the pool is block s / block_size, offset
 *     s % block_size;
 *   - grouped-query attention: query head hq reads kv head hq / (Hq / Hkv);
 *   - prefill is causal with the new chunk placed after the cached tokens:
 *     query i of a chunk of T tokens in a sequence of total length L sits at
 *     absolute position (L - T) + i and attends keys 0 .. (L - T) + i;
 *   - an empty context gives o = 0 and lse = -infinity.
 *
 * Element types: dtype 0 = IEEE fp32, dtype 1 = bfloat16 (upper half of an
 * fp32 bit pattern), dtype 2 = IEEE binary16 (half precision).  All three
 * convert exactly to fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

static int elem_size(int dtype) { return dtype == OR_F32 ? 4 : 2; }

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent field 0: subnormal, value = fraction * 2^-24; 31: infinity
 * (fraction 0) or NaN; otherwise (1024 + fraction) * 2^(exponent - 25). */
static double half_to_double(uint16_t h) {
    const int sign = h >> 15, expo = (h >> 10) & 0x1f, frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Exact widening of one stored element to fp64. */
static double load_elem(const void *base, int64_t idx, int dtype) {
    if (dtype == OR_F16) {
        uint16_t h;
        memcpy(&h, (const char *)base + 2 * idx, 2);
        return half_to_double(h);
    }
    if (dtype == OR_BF16) {
        uint16_t h;
        memcpy(&h, (const char *)base + 2 * idx, 2);
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
    float f;
    memcpy(&f, (const char *)base + 4 * idx, 4);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Block accounting.  [P2 "Iddia ve Gerceklik"]: KV is cut into fixed-size
 * blocks (16 tokens in the example); only the last block of a sequence can
 * hold unused slots.  [P3 "Nasil Calisir?"]: 35 tokens at 16 per block need
 * three blocks and leave 13 slots unused.
 * ---------------------------------------------------------------------- */
int64_t oracle_blocks_needed(int64_t n_tokens, int64_t block_size) {
    if (n_tokens <= 0) return 0;
    int64_t blocks = 0, covered = 0;
    while (covered < n_tokens) { /* one more block whenever the last is full */
        blocks += 1;
        covered += block_size;
    }
    return blocks;
}

int64_t oracle_unused_slots(int64_t n_tokens, int64_t block_size) {
    return oracle_blocks_needed(n_tokens, block_size) * block_size - n_tokens;
}

/* Build block tables the way the pages describe allocation: sequences are
 * served in order, and every time a sequence's current block is full the
 * next free block is taken from the pool [P2 "Iddia ve Gerceklik"; P3 "Nasil
 * Calisir?" step 2].  The pool's free blocks are handed out in the order
 * `free_order` lists them.  Unused table entries hold -1.  Returns 0, or -1
 * when the pool runs out or a table row is too short. */
int oracle_build_block_tables(int batch, const int32_t *lens, int block_size,
                              const int32_t *free_order, int64_t n_free,
                              int max_blocks, int32_t *tables) {
    int64_t next_free = 0;
    for (int b = 0; b < batch; ++b) {
        int32_t *row = tables + (int64_t)b * max_blocks;
        for (int i = 0; i < max_blocks; ++i) row[i] = -1;
        int used = 0;
        for (int64_t t = 0; t < lens[b]; ++t) {
            if (t % block_size == 0) { /* token t opens a new block */
                if (next_free >= n_free || used >= max_blocks) return -1;
                row[used++] = free_order[next_free++];
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * KV append: the new token's K and V go into its slot of the block
 * [P3 "Nasil Calisir?" steps 1-3; P2 "Iddia ve Gerceklik"].  Pure byte copy;
 * a negative slot means "no write".
 * ---------------------------------------------------------------------- */
void oracle_append(void *pool_k, void *pool_v, int64_t num_blocks,
                   int num_kv_heads, int block_size, int head_dim,
                   int elem_bytes, const void *k_new, const void *v_new,
                   const int64_t *slot_mapping, int64_t num_tokens) {
    const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t block = slot / block_size, offset = slot % block_size;
        if (block >= num_blocks) continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * row_bytes;
            int64_t src = (t * num_kv_heads + h) * row_bytes;
            memcpy((char *)pool_k + dst, (const char *)k_new + src, (size_t)row_bytes);
            memcpy((char *)pool_v + dst, (const char *)v_new + src, (size_t)row_bytes);
        }
    }
}

/* ------------------------------------------------------------------------
 * Reassembly of one sequence's logical K (or V) through its block table
 * [P3 "PagedAttention Nedir?": blocks found through a mapping table, logical
 * order kept].  out is [len][num_kv_heads][head_dim] in fp64.
 * ---------------------------------------------------------------------- */
void oracle_gather_logical(const void *pool, int dtype, int num_kv_heads,
                           int block_size, int head_dim, const int32_t *table,
                           int64_t len, double *out) {
    for (int64_t j = 0; j < len; ++j) {
        int64_t block = table[j / block_size];
        int64_t offset = j % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((block * num_kv_heads + h) * block_size + offset) * head_dim;
            double *dst = out + (j * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) dst[d] = load_elem(pool, src + d, dtype);
        }
    }
}

/* The contiguous (vAttention) layout [P1 "Iddia ve Gerceklik: vAttention"]:
 * one linear buffer per request, here [num_kv_heads][max_ctx][head_dim]. */
void oracle_gather_linear(const void *base, int dtype, int num_kv_heads,
                          int64_t max_ctx, int head_dim, int64_t len, double *out) {
    for (int64_t j = 0; j < len; ++j)
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)h * max_ctx + j) * head_dim;
            double *dst = out + (j * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) dst[d] = load_elem(base, src + d, dtype);
        }
}

/* ------------------------------------------------------------------------
 * Softmax attention of one query vector over the first n_keys logical keys
 * of kv head h.  Two passes over the keys, fp64 throughout.
 * ---------------------------------------------------------------------- */
void oracle_attend(const double *q, const double *K, const double *V,
                   int64_t n_keys, int num_kv_heads, int h, int head_dim,
                   double scale, double *o, double *lse) {
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (n_keys <= 0) {
        *lse = -INFINITY;
        return;
    }
    double *s = (double *)malloc((size_t)n_keys * sizeof(double));
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double *k = K + (j * num_kv_heads + h) * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += q[d] * k[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        double w = exp(s[j] - m);
        l += w;
        const double *v = V + (j * num_kv_heads + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] += w * v[d];
    }
    for (int d = 0; d < head_dim; ++d) o[d] /= l;
    *lse = m + log(l);
    free(s);
}

/* ------------------------------------------------------------------------
 * Paged decode attention: one query token per sequence, attending all
 * lens[b] tokens of its cache [P3 "Nasil Calisir?" step 4].
 *
 * q is [batch][num_q_heads][head_dim] (q_dtype); pools are
 * [num_blocks][num_kv_heads][block_size][head_dim] (kv_dtype).
 * Work items: either all (b, hq) pairs (n_items < 0; outputs laid out
 * [batch][num_q_heads][...]) or the listed pairs item_b[i], item_h[i]
 * (outputs laid out [n_items][...]).  Outputs fp64.
 * ---------------------------------------------------------------------- */
void oracle_paged_decode(const void *pool_k, const void *pool_v, int kv_dtype,
                         int num_kv_heads, int block_size, int head_dim,
                         const int32_t *tables, int max_blocks,
                         const int32_t *lens, int batch, const void *q,
                         int q_dtype, int num_q_heads, double scale,
                         int64_t n_items, const int32_t *item_b,
                         const int32_t *item_h, double *out, double *lse) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t total = n_items < 0 ? (int64_t)batch * num_q_heads : n_items;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < total; ++it) {
        int b = n_items < 0 ? (int)(it / num_q_heads) : item_b[it];
        int hq = n_items < 0 ? (int)(it % num_q_heads) : item_h[it];
        int64_t len = lens[b];
        double *K = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
        double *V = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
        double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
        oracle_gather_logical(pool_k, kv_dtype, num_kv_heads, block_size, head_dim,
                              tables + (int64_t)b * max_blocks, len, K);
        oracle_gather_logical(pool_v, kv_dtype, num_kv_heads, block_size, head_dim,
                              tables + (int64_t)b * max_blocks, len, V);
        for (int d = 0; d < head_dim; ++d)
            qd[d] = load_elem(q, ((int64_t)b * num_q_heads + hq) * head_dim + d, q_dtype);
        oracle_attend(qd, K, V, len, num_kv_heads, hq / group, head_dim, scale,
                      out + it * head_dim, lse + it);
        free(K);
        free(V);
        free(qd);
    }
}

/* Decode over the contiguous (vAttention-style) layout: request r's K lives
 * in k_bases[r] as [num_kv_heads][max_ctx][head_dim] (same for V).  Sequence b
 * uses request req_ids[b].  Same maths as the paged decode
 * [P1 "Iddia ve Gerceklik": the kernel sees one contiguous tensor]. */
void oracle_linear_decode(const void *const *k_bases, const void *const *v_bases,
                          int kv_dtype, int num_kv_heads, int64_t max_ctx,
                          int head_dim, const int32_t *req_ids,
                          const int32_t *lens, int batch, const void *q,
                          int q_dtype, int num_q_heads, double scale,
                          int64_t n_items, const int32_t *item_b,
                          const int32_t *item_h, double *out, double *lse) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t total = n_items < 0 ? (int64_t)batch * num_q_heads : n_items;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < total; ++it) {
        int b = n_items < 0 ? (int)(it / num_q_heads) : item_b[it];
        int hq = n_items < 0 ? (int)(it % num_q_heads) : item_h[it];
        int64_t len = lens[b];
        int r = req_ids[b];
        double *K = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
        double *V = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
        double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
        oracle_gather_linear(k_bases[r], kv_dtype, num_kv_heads, max_ctx, head_dim, len, K);
        oracle_gather_linear(v_bases[r], kv_dtype, num_kv_heads, max_ctx, head_dim, len, V);
        for (int d = 0; d < head_dim; ++d)
            qd[d] = load_elem(q, ((int64_t)b * num_q_heads + hq) * head_dim + d, q_dtype);
        oracle_attend(qd, K, V, len, num_kv_heads, hq / group, head_dim, scale,
                      out + it * head_dim, lse + it);
        free(K);
        free(V);
        free(qd);
    }
}

/* ------------------------------------------------------------------------
 * Chunked causal paged prefill.  Sequence b holds seq_lens[b] tokens in its
 * cache, the last T_b = cu_q[b+1] - cu_q[b] of which are the new chunk (its
 * K/V already written).  Query row r = cu_q[b] + i sits at absolute position
 * c_b + i with c_b = seq_lens[b] - T_b and attends keys 0 .. c_b + i.
 * q is [sum T][num_q_heads][head_dim].  Work items: all (r, hq) pairs
 * (n_items < 0; outputs [rows][num_q_heads][...]) or the listed
 * item_r[i], item_h[i].  Prefill is where the pages place the cost of paged
 * kernels [P1 "Iddia ve Gerceklik"]; the maths is the same attention.
 * ---------------------------------------------------------------------- */
void oracle_paged_prefill(const void *pool_k, const void *pool_v, int kv_dtype,
                          int num_kv_heads, int block_size, int head_dim,
                          const int32_t *tables, int max_blocks,
                          const int32_t *seq_lens, const int32_t *cu_q,
                          int batch, const void *q, int q_dtype,
                          int num_q_heads, double scale, int64_t n_items,
                          const int32_t *item_r, const int32_t *item_h,
                          double *out, double *lse) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t rows = cu_q[batch];
    const int64_t total = n_items < 0 ? rows * num_q_heads : n_items;
    /* Work items are grouped per sequence so each sequence's logical K/V is
     * reassembled once per thread-chunk rather than once per item. */
#pragma omp parallel
    {
        int cur_b = -1;
        double *K = NULL, *V = NULL;
        double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
#pragma omp for schedule(dynamic, 16)
        for (int64_t it = 0; it < total; ++it) {
            int64_t r = n_items < 0 ? it / num_q_heads : item_r[it];
            int hq = n_items < 0 ? (int)(it % num_q_heads) : item_h[it];
            int b = 0;
            while (b + 1 < batch && cu_q[b + 1] <= r) ++b;
            int64_t len = seq_lens[b];
            if (b != cur_b) {
                free(K);
                free(V);
                K = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
                V = (double *)malloc((size_t)(len > 0 ? len : 1) * num_kv_heads * head_dim * sizeof(double));
                oracle_gather_logical(pool_k, kv_dtype, num_kv_heads, block_size, head_dim,
                                      tables + (int64_t)b * max_blocks, len, K);
                oracle_gather_logical(pool_v, kv_dtype, num_kv_heads, block_size, head_dim,
                                      tables + (int64_t)b * max_blocks, len, V);
                cur_b = b;
            }
            int64_t chunk = cu_q[b + 1] - cu_q[b];
            int64_t pos = (len - chunk) + (r - cu_q[b]); /* absolute position of the query */
            for (int d = 0; d < head_dim; ++d)
                qd[d] = load_elem(q, (r * num_q_heads + hq) * head_dim + d, q_dtype);
            oracle_attend(qd, K, V, pos + 1, num_kv_heads, hq / group, head_dim, scale,
                          out + it * head_dim, lse + it);
        }
        free(K);
        free(V);
        free(qd);
    }
}

/* Attention over explicit logical K/V given in fp64 ([n_keys][Hkv][D]);
 * used by the pins to evaluate hand-built cases without any pool. */
void oracle_attend_logical(const double *q, const double *K, const double *V,
                           int64_t n_keys, int num_kv_heads, int h, int head_dim,
                           double scale, double *o, double *lse) {
    oracle_attend(q, K, V, n_keys, num_kv_heads, h, head_dim, scale, o, lse);
}

int oracle_elem_size(int dtype) { return elem_size(dtype); }

/* The exact fp64 value of each of n binary16 bit patterns (for the pins). */
void oracle_half_to_double(const uint16_t *h, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = half_to_double(h[i]);
}
