/*
 * Oracle for the PagedAttention decode hot path: a plain, slow, obviously
 * correct fp64 CPU restatement of what the path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it, and it shares no code, header, table or helper with the CUDA
 * library: it has its own element decoders, its own slot arithmetic and its
 * own loops, written straight from the definitions below.
 *
 * Sources (web pages on PagedAttention; cited by title and section):
 *  [P1] "第4章 PagedAttention：虚拟内存的启示" (vLLM source-reading book):
 *       §4.3.1 block shape (2, num_blocks, block_size, num_kv_heads,
 *       head_size), index 0 = K, index 1 = V; §4.4.1 block table;
 *       §4.4.3 slot mapping (slot = table[pos / B] * B + pos % B);
 *       §4.5 write-then-read call chain; §4.6 online-softmax recurrence.
 *  [P3] "PagedAttention: virtual memory for the KV cache" digest:
 *       "写时复制" paragraph (clone the whole block on write);
 *       "常见误解" (paging does not change the attention result).
 *  [P4] CSDN beginner article, §三.1 `page_attention`: gather the valid
 *       K/V of every block in logical order, softmax(q k^T / sqrt(d)), x V.
 *  [P5] "PagedAttention原理（下）" lecture, §4.3: COW copies block P into
 *       a new block Q before the write.
 *
 * Precision: inputs are 16-bit (fp16 or bf16) bit patterns, decoded exactly
 * to double; every sum, max, exp and division is done in double.
 *
 * FP8 cache (a reading: the book names a lower-precision KV cache only as a
 * capacity lever, §4.8): K and V are stored as OCP E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 fraction bits; no infinities; S.1111.111 is
 * NaN; largest finite 448) of value / scale, one scale for K and one for V.
 * A stored code c stands for decode(c) * scale.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#ifdef __GLIBC__
#include <malloc.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* ---- threads ----
 * The batch-level functions below (decode, its sampled and FP8 forms, and
 * prefill) hand whole output rows, one (sequence or query row, q-head) at a
 * time, to OpenMP threads. Each row is computed by the same single-threaded
 * code whatever the thread count, so results do not depend on it. Built
 * without OpenMP, everything runs on the calling thread. */
void oracle_set_threads(int n)
{
#ifdef __GLIBC__
    /* Rows allocate their gathered K/V (up to tens of MB) and free them again.
     * Served by mmap, every row would fault its pages in afresh, and the
     * threads would queue on the kernel's memory map; from the heap the
     * memory is reused. This changes only where the buffers come from. */
    static int heap_set = 0;
    if (!heap_set) {
        mallopt(M_MMAP_THRESHOLD, 1 << 30);
        mallopt(M_TRIM_THRESHOLD, 1 << 30);
        heap_set = 1;
    }
#endif
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

/* Threads the next batch-level call will use (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- exact 16-bit float decoders (IEEE 754 binary16, bfloat16) ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);             /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 value. */
double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -133);            /* subnormal: frac * 2^-126 / 128 */
    } else if (expo == 255) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(128 + frac), expo - 134); /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -mag : mag;
}

/* Vector form of the two decoders, for tests: out[i] = value of bits[i]. */
void oracle_decode_elems(const uint16_t *bits, double *out, long long n, int dtype)
{
    for (long long i = 0; i < n; ++i)
        out[i] = dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits[i]) : oracle_f16_to_double(bits[i]);
}

/* ---- E4M3 (OCP FP8) ---- */

/* Exact value of an E4M3 code. */
double oracle_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 0xf;
    int frac = c & 7;
    double mag;
    if (expo == 15 && frac == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)frac, -9);              /* subnormal: frac/8 * 2^-6 */
    else
        mag = ldexp((double)(8 + frac), expo - 10); /* (1 + f/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Code of the E4M3 value nearest to x (ties to the even code), saturating
 * beyond +-448; NaN gives 0x7F. Found by comparing x with every finite code:
 * slow, and the plain definition of round-to-nearest-even. */
uint8_t oracle_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a > 448.0)
        return sign | 0x7E;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/* Quantise one 16-bit element for the FP8 cache: the element divided by the
 * scale in fp32 (one IEEE division, the precision the device uses, so that
 * both sides round the same quotient), then rounded to E4M3. */
uint8_t oracle_quantize_e4m3(uint16_t bits, int dtype, float scale)
{
    float v = (float)(dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits));
    float y = v / scale;
    return oracle_e4m3_from_float(y);
}

static double elem(const uint16_t *p, long long i, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(p[i]) : oracle_f16_to_double(p[i]);
}

/* Element (c, b, t, h, d) of a per-layer pool shaped
 * (2, num_blocks, block_size, num_kv_heads, head_size), row-major [P1 §4.3.1]. */
static long long pool_index(int c, int b, int t, int h, int d,
                            int num_blocks, int block_size, int num_kv_heads, int head_size)
{
    return ((((long long)c * num_blocks + b) * block_size + t) * num_kv_heads + h)
               * head_size + d;
}

/* ---- slot mapping [P1 §4.4.3] ---- */

/* Physical slot of logical token position `pos` of a sequence whose block
 * table row is `table`: the logical block pos / B is looked up, and the
 * offset inside it is pos % B. */
long long oracle_slot(const int32_t *table, int block_size, long long pos)
{
    long long logical_block = pos / block_size;
    long long offset = pos % block_size;
    return (long long)table[logical_block] * block_size + offset;
}

/* ---- write path: reshape_and_cache [P1 §4.5 step 1, §4.4.3] ----
 * For every new token t with slot >= 0: the K row [num_kv_heads][head_size]
 * goes to pool[0][slot / B][slot % B], the V row to pool[1][...]. Negative
 * slots are skipped (padding). Returns the number of rows written, or -1 if
 * a slot lies beyond the pool. */
int oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *pool,
                             const int32_t *slot_mapping, int num_tokens,
                             int num_blocks, int block_size, int num_kv_heads, int head_size)
{
    int written = 0;
    for (int t = 0; t < num_tokens; ++t) {
        long long slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (long long)num_blocks * block_size)
            return -1;
        int b = (int)(slot / block_size);
        int off = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_size; ++d) {
                long long src = ((long long)t * num_kv_heads + h) * head_size + d;
                pool[pool_index(0, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] = key[src];
                pool[pool_index(1, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] = value[src];
            }
        }
        ++written;
    }
    return written;
}

/* ---- FP8 cache write path ----
 * The same placement as oracle_reshape_and_cache, into a byte pool of the
 * same shape; every K element is stored as oracle_quantize_e4m3(k, k_scale)
 * and every V element as oracle_quantize_e4m3(v, v_scale). */
int oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value, uint8_t *pool,
                                 const int32_t *slot_mapping, int num_tokens,
                                 int num_blocks, int block_size, int num_kv_heads, int head_size,
                                 int dtype, float k_scale, float v_scale)
{
    int written = 0;
    for (int t = 0; t < num_tokens; ++t) {
        long long slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (long long)num_blocks * block_size)
            return -1;
        int b = (int)(slot / block_size);
        int off = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_size; ++d) {
                long long src = ((long long)t * num_kv_heads + h) * head_size + d;
                pool[pool_index(0, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] =
                    oracle_quantize_e4m3(key[src], dtype, k_scale);
                pool[pool_index(1, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] =
                    oracle_quantize_e4m3(value[src], dtype, v_scale);
            }
        }
        ++written;
    }
    return written;
}

/* ---- copy-on-write block copy [P3 写时复制; P5 §4.3] ----
 * For each (src, dst) pair, in order, and for every layer pool: the whole
 * physical block (all B slots, K and V, all heads) of src is copied to dst.
 * Returns 0, or -1 on an out-of-range block id (nothing after it copied). */
int oracle_copy_blocks(uint16_t *const *pools, int num_layers,
                       const int32_t *pairs, int num_pairs,
                       int num_blocks, int block_size, int num_kv_heads, int head_size)
{
    for (int i = 0; i < num_pairs; ++i) {
        int src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return -1;
        for (int layer = 0; layer < num_layers; ++layer) {
            uint16_t *pool = pools[layer];
            for (int c = 0; c < 2; ++c)
                for (int t = 0; t < block_size; ++t)
                    for (int h = 0; h < num_kv_heads; ++h)
                        for (int d = 0; d < head_size; ++d)
                            pool[pool_index(c, dst, t, h, d, num_blocks, block_size, num_kv_heads, head_size)] =
                                pool[pool_index(c, src, t, h, d, num_blocks, block_size, num_kv_heads, head_size)];
        }
    }
    return 0;
}

/* ---- read path: plain attention over a contiguous K/V [P4 §三.1] ----
 * out[d] = sum_i w_i V[i][d] / sum_i w_i, w_i = exp(x_i - max_j x_j),
 * x_i = scale * sum_d q[d] K[i][d]. K and V are [L][head_size] values. L = 0
 * gives a zero row (the pages are silent; this is the reading taken). */
static void attention_values(double *out, const double *q, const double *k, const double *v,
                             int seq_len, int head_size, double scale)
{
    for (int d = 0; d < head_size; ++d)
        out[d] = 0.0;
    if (seq_len <= 0)
        return;
    double *x = (double *)malloc(sizeof(double) * (size_t)seq_len);
    double mx = -INFINITY;
    for (int i = 0; i < seq_len; ++i) {
        double dot = 0.0;
        for (int d = 0; d < head_size; ++d)
            dot += q[d] * k[(long long)i * head_size + d];
        x[i] = scale * dot;
        if (x[i] > mx)
            mx = x[i];
    }
    double denom = 0.0;
    for (int i = 0; i < seq_len; ++i) {
        x[i] = exp(x[i] - mx);
        denom += x[i];
    }
    for (int d = 0; d < head_size; ++d) {
        double acc = 0.0;
        for (int i = 0; i < seq_len; ++i)
            acc += x[i] * v[(long long)i * head_size + d];
        out[d] = acc / denom;
    }
    free(x);
}

/* The same on 16-bit inputs: every element decoded exactly, then the
 * definition above. */
void oracle_attention_contiguous(double *out, const uint16_t *q, const uint16_t *k,
                                 const uint16_t *v, int seq_len, int head_size,
                                 double scale, int dtype)
{
    size_t n = seq_len > 0 ? (size_t)seq_len * head_size : 1;
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_size);
    double *kd = (double *)malloc(sizeof(double) * n);
    double *vd = (double *)malloc(sizeof(double) * n);
    for (int d = 0; d < head_size; ++d)
        qd[d] = elem(q, d, dtype);
    for (long long i = 0; i < (long long)(seq_len > 0 ? seq_len : 0) * head_size; ++i) {
        kd[i] = elem(k, i, dtype);
        vd[i] = elem(v, i, dtype);
    }
    attention_values(out, qd, kd, vd, seq_len, head_size, scale);
    free(qd);
    free(kd);
    free(vd);
}

/* ---- read path: paged decode for one (sequence, q-head) [P1 §4.5, §4.4.1] ----
 * Walk logical tokens 0..L-1; token i lives in physical block
 * table[i / B] at offset i % B. The q-head maps to kv-head
 * hq / (num_q_heads / num_kv_heads) (contiguous GQA groups). The K/V rows
 * are gathered in logical order and handed to the contiguous definition. */
void oracle_decode_one(double *out, const uint16_t *query, const uint16_t *pool,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *seq_lens, int seq, int q_head,
                       double scale, int num_q_heads, int num_kv_heads, int head_size,
                       int num_blocks, int block_size, int dtype)
{
    int seq_len = seq_lens[seq];
    int group = num_q_heads / num_kv_heads;
    int kv_head = q_head / group;
    const int32_t *table = block_tables + (long long)seq * max_blocks_per_seq;
    size_t n = seq_len > 0 ? (size_t)seq_len * head_size : 1;
    uint16_t *k = (uint16_t *)malloc(sizeof(uint16_t) * n);
    uint16_t *v = (uint16_t *)malloc(sizeof(uint16_t) * n);
    for (int i = 0; i < seq_len; ++i) {
        int b = table[i / block_size];
        int off = i % block_size;
        for (int d = 0; d < head_size; ++d) {
            k[(long long)i * head_size + d] =
                pool[pool_index(0, b, off, kv_head, d, num_blocks, block_size, num_kv_heads, head_size)];
            v[(long long)i * head_size + d] =
                pool[pool_index(1, b, off, kv_head, d, num_blocks, block_size, num_kv_heads, head_size)];
        }
    }
    const uint16_t *q = query + ((long long)seq * num_q_heads + q_head) * head_size;
    oracle_attention_contiguous(out, q, k, v, seq_len, head_size, scale, dtype);
    free(k);
    free(v);
}

/* Paged decode for a whole batch: out is [num_seqs][num_q_heads][head_size]. */
void oracle_decode(double *out, const uint16_t *query, const uint16_t *pool,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *seq_lens, int num_seqs,
                   double scale, int num_q_heads, int num_kv_heads, int head_size,
                   int num_blocks, int block_size, int dtype)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s)
        for (int hq = 0; hq < num_q_heads; ++hq)
            oracle_decode_one(out + ((long long)s * num_q_heads + hq) * head_size, query, pool,
                              block_tables, max_blocks_per_seq, seq_lens, s, hq, scale,
                              num_q_heads, num_kv_heads, head_size, num_blocks, block_size, dtype);
}

/* Decode for a list of sampled (seq, q_head) pairs: out is [n][head_size]. */
void oracle_decode_sampled(double *out, const int32_t *seq_ids, const int32_t *q_heads, int n,
                           const uint16_t *query, const uint16_t *pool,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, double scale, int num_q_heads,
                           int num_kv_heads, int head_size, int num_blocks, int block_size,
                           int dtype)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i)
        oracle_decode_one(out + (long long)i * head_size, query, pool, block_tables,
                          max_blocks_per_seq, seq_lens, seq_ids[i], q_heads[i], scale,
                          num_q_heads, num_kv_heads, head_size, num_blocks, block_size, dtype);
}

/* ---- FP8 cache read path ----
 * The paged decode of oracle_decode_one over a byte pool: a cached K element
 * stands for e4m3(code) * k_scale and a V element for e4m3(code) * v_scale
 * (exact in double); the query is the 16-bit input. The attention is the
 * same two-pass definition (attention_values) on those values. */
void oracle_decode_fp8_one(double *out, const uint16_t *query, const uint8_t *pool,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, int seq, int q_head,
                           double scale, int num_q_heads, int num_kv_heads, int head_size,
                           int num_blocks, int block_size, int dtype,
                           double k_scale, double v_scale)
{
    int seq_len = seq_lens[seq];
    int group = num_q_heads / num_kv_heads;
    int kv_head = q_head / group;
    const int32_t *table = block_tables + (long long)seq * max_blocks_per_seq;
    size_t n = seq_len > 0 ? (size_t)seq_len * head_size : 1;
    double *k = (double *)malloc(sizeof(double) * n);
    double *v = (double *)malloc(sizeof(double) * n);
    double *q = (double *)malloc(sizeof(double) * (size_t)head_size);
    for (int i = 0; i < seq_len; ++i) {
        int b = table[i / block_size];
        int off = i % block_size;
        for (int d = 0; d < head_size; ++d) {
            uint8_t kc = pool[pool_index(0, b, off, kv_head, d, num_blocks, block_size, num_kv_heads, head_size)];
            uint8_t vc = pool[pool_index(1, b, off, kv_head, d, num_blocks, block_size, num_kv_heads, head_size)];
            k[(long long)i * head_size + d] = oracle_e4m3_to_double(kc) * k_scale;
            v[(long long)i * head_size + d] = oracle_e4m3_to_double(vc) * v_scale;
        }
    }
    const uint16_t *qb = query + ((long long)seq * num_q_heads + q_head) * head_size;
    for (int d = 0; d < head_size; ++d)
        q[d] = elem(qb, d, dtype);
    attention_values(out, q, k, v, seq_len, head_size, scale);
    free(k);
    free(v);
    free(q);
}

/* FP8-cache decode for a whole batch: out is [num_seqs][num_q_heads][head_size]. */
void oracle_decode_fp8(double *out, const uint16_t *query, const uint8_t *pool,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *seq_lens, int num_seqs,
                       double scale, int num_q_heads, int num_kv_heads, int head_size,
                       int num_blocks, int block_size, int dtype, double k_scale, double v_scale)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s)
        for (int hq = 0; hq < num_q_heads; ++hq)
            oracle_decode_fp8_one(out + ((long long)s * num_q_heads + hq) * head_size, query, pool,
                                  block_tables, max_blocks_per_seq, seq_lens, s, hq, scale,
                                  num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                                  dtype, k_scale, v_scale);
}

/* FP8-cache decode for sampled (seq, q_head) pairs: out is [n][head_size]. */
void oracle_decode_fp8_sampled(double *out, const int32_t *seq_ids, const int32_t *q_heads, int n,
                               const uint16_t *query, const uint8_t *pool,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, double scale, int num_q_heads,
                               int num_kv_heads, int head_size, int num_blocks, int block_size,
                               int dtype, double k_scale, double v_scale)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i)
        oracle_decode_fp8_one(out + (long long)i * head_size, query, pool, block_tables,
                              max_blocks_per_seq, seq_lens, seq_ids[i], q_heads[i], scale,
                              num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                              dtype, k_scale, v_scale);
}

/* ---- read path: chunked prefill [P1 §4.5 step 2] ----
 * The FlashAttention backend hands the cache, the block table, the query
 * offsets cu_seqlens_q and the used lengths seqused_k to one varlen call.
 * Reading: sequence s brings q_len = cu_seqlens_q[s+1] - cu_seqlens_q[s]
 * query tokens, the last q_len of its seq_lens[s] cached tokens (this step's
 * tokens were written by slot first); query i sits at position
 * p = seq_lens[s] - q_len + i and attends causally to tokens 0..p. Each
 * output row is therefore the decode definition over the first p + 1 tokens
 * of the sequence, and is computed by oracle_decode_one on exactly that:
 * out is [total_q][num_q_heads][head_size], row cu_seqlens_q[s] + i. */
void oracle_prefill(double *out, const uint16_t *query, const uint16_t *pool,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *cu_seqlens_q, const int32_t *seq_lens, int num_seqs,
                    double scale, int num_q_heads, int num_kv_heads, int head_size,
                    int num_blocks, int block_size, int dtype)
{
    int total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < total_q; ++r) {
        int s = 0;
        while (cu_seqlens_q[s + 1] <= r) /* the sequence whose chunk holds row r */
            ++s;
        int q0 = cu_seqlens_q[s];
        int q_len = cu_seqlens_q[s + 1] - q0;
        int i = r - q0;
        const int32_t *table = block_tables + (long long)s * max_blocks_per_seq;
        int32_t visible = seq_lens[s] - q_len + i + 1; /* tokens 0..p */
        const uint16_t *q_row = query + (long long)r * num_q_heads * head_size;
        for (int hq = 0; hq < num_q_heads; ++hq)
            oracle_decode_one(out + ((long long)r * num_q_heads + hq) * head_size, q_row,
                              pool, table, max_blocks_per_seq, &visible, 0, hq, scale,
                              num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                              dtype);
    }
}

/* Chunked prefill over an E4M3 pool: the same rows as oracle_prefill, each
 * the FP8 decode definition (oracle_decode_fp8_one) over its first p + 1
 * tokens. */
void oracle_prefill_fp8(double *out, const uint16_t *query, const uint8_t *pool,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *cu_seqlens_q, const int32_t *seq_lens, int num_seqs,
                        double scale, int num_q_heads, int num_kv_heads, int head_size,
                        int num_blocks, int block_size, int dtype, double k_scale, double v_scale)
{
    int total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < total_q; ++r) {
        int s = 0;
        while (cu_seqlens_q[s + 1] <= r) /* the sequence whose chunk holds row r */
            ++s;
        int q0 = cu_seqlens_q[s];
        int q_len = cu_seqlens_q[s + 1] - q0;
        int i = r - q0;
        const int32_t *table = block_tables + (long long)s * max_blocks_per_seq;
        int32_t visible = seq_lens[s] - q_len + i + 1; /* tokens 0..p */
        const uint16_t *q_row = query + (long long)r * num_q_heads * head_size;
        for (int hq = 0; hq < num_q_heads; ++hq)
            oracle_decode_fp8_one(out + ((long long)r * num_q_heads + hq) * head_size, q_row,
                                  pool, table, max_blocks_per_seq, &visible, 0, hq, scale,
                                  num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                                  dtype, k_scale, v_scale);
    }
}

/* ---- the online-softmax recurrence [P1 §4.6] ----
 * The same attention, computed the way the method streams it: the logical
 * tokens are cut into consecutive parts of `part_len` tokens; each part
 * yields its local state (m', s', O' = sum_t exp(x_t - m') V_t); the
 * running state (m, s, O) absorbs it with
 *     m_new = max(m, m'),
 *     s_new = s * exp(m - m_new) + s' * exp(m' - m_new),
 *     O_new = O * exp(m - m_new) + O' * exp(m' - m_new),
 * and the result is O / s. This is the merge rule split-K decoding relies
 * on; it is kept here so that tests can pin it against the two-pass
 * definition above. */
void oracle_attention_online(double *out, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, int seq_len, int head_size,
                             double scale, int dtype, int part_len)
{
    double m = -INFINITY, s = 0.0;
    double *o = (double *)calloc((size_t)head_size, sizeof(double));
    double *op = (double *)calloc((size_t)head_size, sizeof(double));
    double *x = (double *)malloc(sizeof(double) * (size_t)(part_len > 0 ? part_len : 1));
    for (int start = 0; start < seq_len; start += part_len) {
        int end = start + part_len < seq_len ? start + part_len : seq_len;
        double mp = -INFINITY;
        for (int i = start; i < end; ++i) {
            double dot = 0.0;
            for (int d = 0; d < head_size; ++d)
                dot += elem(q, d, dtype) * elem(k, (long long)i * head_size + d, dtype);
            x[i - start] = scale * dot;
            if (x[i - start] > mp)
                mp = x[i - start];
        }
        double sp = 0.0;
        for (int d = 0; d < head_size; ++d)
            op[d] = 0.0;
        for (int i = start; i < end; ++i) {
            double p = exp(x[i - start] - mp);
            sp += p;
            for (int d = 0; d < head_size; ++d)
                op[d] += p * elem(v, (long long)i * head_size + d, dtype);
        }
        double m_new = m > mp ? m : mp;
        double a_old = exp(m - m_new); /* exp(-inf) = 0 on the first part */
        double a_new = exp(mp - m_new);
        s = s * a_old + sp * a_new;
        for (int d = 0; d < head_size; ++d)
            o[d] = o[d] * a_old + op[d] * a_new;
        m = m_new;
    }
    for (int d = 0; d < head_size; ++d)
        out[d] = seq_len > 0 ? o[d] / s : 0.0;
    free(o);
    free(op);
    free(x);
}
