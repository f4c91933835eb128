/*
 * pa_oracle.c — plain fp64 CPU oracle for the paged-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; it is written to be read
 * against the pages, not to be fast.
 *
 * Sources (page title, then section):
 *   [P1] "什么是 PagedAttention？"                      (glossary page)
 *   [P2] "PagedAttention学习笔记"                       (study notes)
 *   [P3] "KV cache 显存管理：为什么 PagedAttention 是 vLLM 的核心" (mini-vLLM)
 *
 * Storage convention (the pages leave the pool layout open; the plainest
 * reading of "slot in a flattened KV layout" is used): each of the K and V
 * pools is a row-major array [num_blocks][block_size][num_kv_heads][head_dim],
 * so element (slot, kv_head, d) lives at (slot*num_kv_heads + kv_head)*head_dim + d
 * with slot = physical_block*block_size + offset.
 * Query head h reads KV head h / (num_q_heads/num_kv_heads) (the pages never
 * mention grouped-query attention; this is the plainest reading).
 *
 * Every routine returns 0 on success and a negative count of invalid indices
 * otherwise; it never reads outside the arrays it was given.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* [P2] §2.1 PagedAttention 核心原理 and [P3] "分页思想": a sequence of length L
 * needs ceil(L / B) logical blocks. */
int64_t oracle_num_blocks(int64_t seq_len, int64_t block_size) {
    if (seq_len <= 0) return 0;
    return (seq_len + block_size - 1) / block_size;
}

/* Widen one stored element to double.  bf16 is the upper half of an IEEE
 * binary32 word, so the widening is exact. */
static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
    if (dtype == ORACLE_F64) return ((const double*)base)[idx];
    uint16_t bits = ((const uint16_t*)base)[idx];
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static int elem_bytes(int dtype) { return dtype == ORACLE_F32 ? 4 : dtype == ORACLE_F64 ? 8 : 2; }

/* [P2] 代码实现部分 › "块表与槽位映射：BlockTable" (compute_slot_mapping) and
 * [P3] "PagedAttention 改变了什么": for the new token at position pos of
 * sequence seq,
 *     logical_block = pos / B,  offset = pos % B,
 *     physical      = block_table[seq][logical_block],
 *     slot          = physical * B + offset.
 * pos < 0 marks a padding token: slot -1, no error ([P2] uses -1 for "not this
 * rank's token").  A token whose sequence, logical block or table entry is out
 * of range also gets slot -1 and is counted as an error. */
int oracle_slot_mapping(const int32_t* block_tables, int64_t num_seqs, int64_t max_blocks_per_seq,
                        const int32_t* seq_idx, const int32_t* pos, int64_t num_tokens,
                        int64_t block_size, int64_t num_blocks, int64_t* slot_mapping) {
    int errors = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        slot_mapping[t] = -1;
        int64_t p = pos[t];
        if (p < 0) continue;
        int64_t s = seq_idx[t];
        int64_t logical_block = p / block_size;
        int64_t offset = p % block_size;
        if (s < 0 || s >= num_seqs || logical_block >= max_blocks_per_seq) { ++errors; continue; }
        int64_t physical = block_tables[s * max_blocks_per_seq + logical_block];
        if (physical < 0 || physical >= num_blocks) { ++errors; continue; }
        slot_mapping[t] = physical * block_size + offset;
    }
    return -errors;
}

/* [P2] 代码实现部分 › "块表与槽位映射：BlockTable" (混合块, map_to_kernel_blocks):
 * when the block manager allocates blocks of ratio x kernel_block_size tokens,
 * each manager block is the same memory as `ratio` consecutive kernel blocks,
 * so manager block m becomes kernel blocks m*ratio, m*ratio+1, ...,
 * m*ratio+ratio-1, in order; a -1 entry becomes ratio -1 entries.  Row s of
 * the kernel table has kernel_width entries; positions past the manager
 * table's ratio*mgr_width are -1. */
void oracle_map_to_kernel_blocks(const int32_t* mgr_tables, int64_t num_seqs, int64_t mgr_width,
                                 int64_t ratio, int32_t* kernel_tables, int64_t kernel_width) {
    for (int64_t s = 0; s < num_seqs; ++s) {
        for (int64_t j = 0; j < kernel_width; ++j) {
            int64_t m = j / ratio;
            int32_t entry = -1;
            if (m < mgr_width) {
                int32_t mb = mgr_tables[s * mgr_width + m];
                if (mb >= 0) entry = (int32_t)(mb * ratio + j % ratio);
            }
            kernel_tables[s * kernel_width + j] = entry;
        }
    }
}

/* ---- fp8 KV pools: the e4m3 format (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448;
 * exponent field 0 holds the subnormals m * 2^-9).  The pages give the pool
 * formula with dtype_size as a free parameter ("KV cache 显存管理…", KV size
 * formula); an fp8 pool stores code = e4m3(x / scale) per element with one
 * scale per pool, and reads back code * scale. */

/* Value of an e4m3 code, straight from the format's definition. */
double oracle_e4m3_value(uint8_t code) {
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -v : v;
}

/* Nearest e4m3 code to x, ties to the even code, magnitudes beyond 448 held
 * at 448 (saturating), NaN to NaN: a search over all 127 non-negative finite
 * codes, so no bit manipulation has to be trusted. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    if (a > 448.0) best = 0x7E;
    return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* The fp8 pools' write: the slot-mapped copy of oracle_write_kv, each bf16
 * element x stored as e4m3(x * (1.0f / scale)), the product and the
 * reciprocal in float. */
int oracle_write_kv_fp8(const uint16_t* k_new, const uint16_t* v_new, int64_t num_tokens, int64_t num_kv_heads,
                        int64_t head_dim, uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                        int64_t block_size, const int64_t* slot_mapping, float k_scale, float v_scale) {
    int errors = 0;
    int64_t row = num_kv_heads * head_dim;
    float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++errors; continue; }
        for (int64_t i = 0; i < row; ++i) {
            float kx = (float)load_elem(k_new, ORACLE_BF16, t * row + i);
            float vx = (float)load_elem(v_new, ORACLE_BF16, t * row + i);
            k_cache[slot * row + i] = oracle_e4m3_encode(kx * k_inv);
            v_cache[slot * row + i] = oracle_e4m3_encode(vx * v_inv);
        }
    }
    return -errors;
}

/* code * scale for every element (exact in double: 4 + 24 significant bits). */
void oracle_dequant_e4m3(const uint8_t* codes, int64_t n, float scale, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]) * (double)scale;
}

/* [P3] "对 ModelRunner 的影响": the slot tells where the current token's K/V is
 * written.  A byte copy of each token's [num_kv_heads][head_dim] row into the
 * pool row at its slot; slot < 0 is skipped, slot beyond the pool is an error. */
int oracle_write_kv(const void* k_new, const void* v_new, int64_t num_tokens, int64_t num_kv_heads,
                    int64_t head_dim, int dtype, void* k_cache, void* v_cache, int64_t num_blocks,
                    int64_t block_size, const int64_t* slot_mapping) {
    int errors = 0;
    int64_t row_bytes = num_kv_heads * head_dim * elem_bytes(dtype);
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++errors; continue; }
        memcpy((char*)k_cache + slot * row_bytes, (const char*)k_new + t * row_bytes, (size_t)row_bytes);
        memcpy((char*)v_cache + slot * row_bytes, (const char*)v_new + t * row_bytes, (size_t)row_bytes);
    }
    return -errors;
}

/* Everything one attention problem needs. */
typedef struct {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    int dtype;
    int64_t num_q_heads, num_kv_heads, head_dim;
    int64_t num_blocks, block_size;
    const int32_t* block_tables;
    int64_t max_blocks_per_seq;
    double scale;
} problem_t;

/* Contiguous K/V of one (sequence, kv head), the max-length layout of
 * [P3] "最直观的做法": row j holds token j.  Built by walking the block table
 * token by token ([P3] "PagedAttention 改变了什么": token -> logical block ->
 * physical block -> offset -> address).  Returns -1 on an out-of-range entry. */
static int gather_contiguous(const problem_t* pr, int64_t seq, int64_t kv_head, int64_t len,
                             double* kc, double* vc) {
    int64_t D = pr->head_dim, B = pr->block_size;
    for (int64_t j = 0; j < len; ++j) {
        int64_t logical_block = j / B;
        int64_t offset = j % B;
        if (logical_block >= pr->max_blocks_per_seq) return -1;
        int64_t physical = pr->block_tables[seq * pr->max_blocks_per_seq + logical_block];
        if (physical < 0 || physical >= pr->num_blocks) return -1;
        int64_t slot = physical * B + offset;
        int64_t base = (slot * pr->num_kv_heads + kv_head) * D;
        for (int64_t d = 0; d < D; ++d) {
            kc[j * D + d] = load_elem(pr->k_cache, pr->dtype, base + d);
            vc[j * D + d] = load_elem(pr->v_cache, pr->dtype, base + d);
        }
    }
    return 0;
}

/* softmax(scale * q K^T) V over rows 0..len-1 of the contiguous K/V, in fp64:
 *   x_j = scale * sum_d q_d K_jd,  m = max_j x_j,  w_j = exp(x_j - m),
 *   o_d = sum_j w_j V_jd / sum_j w_j.
 * len == 0 gives a zero vector.  [P2] "与 FlashAttention 的关系" and [P3]
 * "PagedAttention 改变了什么": paging does not change this formula. */
static void attend(const double* q, const double* kc, const double* vc, int64_t len, int64_t D,
                   double scale, double* x, double* o) {
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    if (len <= 0) return;
    double m = -INFINITY;
    for (int64_t j = 0; j < len; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += q[d] * kc[j * D + d];
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < len; ++j) {
        double w = exp(x[j] - m);
        l += w;
        for (int64_t d = 0; d < D; ++d) o[d] += w * vc[j * D + d];
    }
    for (int64_t d = 0; d < D; ++d) o[d] /= l;
}

/* ---------------------------------------------------------------- decode */

typedef struct {
    problem_t pr;
    double* out;
    const int32_t* context_lens;
    int64_t num_seqs;
    int64_t next_item; /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
    int status;
} decode_job_t;

static int64_t take_item(int64_t* next, pthread_mutex_t* lock) {
    pthread_mutex_lock(lock);
    int64_t i = (*next)++;
    pthread_mutex_unlock(lock);
    return i;
}

/* One work item = one (sequence, kv head): gather its contiguous K/V once,
 * then attend for each of the query heads that read that kv head. */
static void* decode_worker(void* arg) {
    decode_job_t* job = (decode_job_t*)arg;
    const problem_t* pr = &job->pr;
    int64_t D = pr->head_dim, G = pr->num_q_heads / pr->num_kv_heads;
    int64_t items = job->num_seqs * pr->num_kv_heads;
    int64_t cap = 0;
    double *kc = NULL, *vc = NULL, *x = NULL;
    double* q = (double*)malloc(sizeof(double) * D);
    for (;;) {
        int64_t item = take_item(&job->next_item, &job->lock);
        if (item >= items) break;
        int64_t s = item / pr->num_kv_heads, kvh = item % pr->num_kv_heads;
        int64_t len = job->context_lens[s];
        if (len < 0) len = 0;
        if (len > cap) {
            cap = len;
            kc = (double*)realloc(kc, sizeof(double) * cap * D);
            vc = (double*)realloc(vc, sizeof(double) * cap * D);
            x = (double*)realloc(x, sizeof(double) * cap);
        }
        if (gather_contiguous(pr, s, kvh, len, kc, vc) != 0) {
            pthread_mutex_lock(&job->lock);
            job->status = -1;
            pthread_mutex_unlock(&job->lock);
            continue;
        }
        for (int64_t g = 0; g < G; ++g) {
            int64_t h = kvh * G + g;
            for (int64_t d = 0; d < D; ++d)
                q[d] = load_elem(pr->q, pr->dtype, (s * pr->num_q_heads + h) * D + d);
            attend(q, kc, vc, len, D, pr->scale, x, job->out + (s * pr->num_q_heads + h) * D);
        }
    }
    free(kc); free(vc); free(x); free(q);
    return NULL;
}

static void run_pool(void* (*fn)(void*), void* job, int num_threads) {
    if (num_threads < 1) num_threads = 1;
    if (num_threads == 1) { fn(job); return; }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * num_threads);
    for (int i = 0; i < num_threads; ++i) pthread_create(&th[i], NULL, fn, job);
    for (int i = 0; i < num_threads; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* Decode: one query token per sequence.  For sequence s and query head h,
 *   out[s][h] = softmax_j(scale * q[s][h] . k_j) v_j  over j < context_lens[s],
 * with k_j, v_j found through the block table ([P2] 三、算法流程与数据结构:
 * the kernel reads Q and the block table and gathers K/V by block).
 * q is [num_seqs][num_q_heads][head_dim] in the storage dtype; out is fp64. */
int oracle_decode(double* out, const void* q, int64_t num_seqs, int64_t num_q_heads,
                  int64_t num_kv_heads, int64_t head_dim, int dtype, const void* k_cache,
                  const void* v_cache, int64_t num_blocks, int64_t block_size,
                  const int32_t* block_tables, int64_t max_blocks_per_seq,
                  const int32_t* context_lens, double scale, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    decode_job_t job;
    job.pr = (problem_t){q, k_cache, v_cache, dtype, num_q_heads, num_kv_heads, head_dim,
                         num_blocks, block_size, block_tables, max_blocks_per_seq, scale};
    job.out = out;
    job.context_lens = context_lens;
    job.num_seqs = num_seqs;
    job.next_item = 0;
    job.status = 0;
    pthread_mutex_init(&job.lock, NULL);
    run_pool(decode_worker, &job, num_threads);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/* --------------------------------------------------------------- prefill */

typedef struct {
    problem_t pr;
    double* out;
    const int32_t* cu_q_lens;
    const int32_t* q_start_pos;
    const int32_t* seq_of_chunk;
    const int32_t* context_lens;
    int64_t num_chunks;
    int64_t num_seqs;
    int64_t next_item;
    pthread_mutex_t lock;
    int status;
} prefill_job_t;

/* One work item = one (chunk, kv head).  Query i of chunk c sits at absolute
 * position p = q_start_pos[c] + i and attends keys 0..p of its sequence
 * (causal), all read through the block table — the chunk's own keys included. */
static void* prefill_worker(void* arg) {
    prefill_job_t* job = (prefill_job_t*)arg;
    const problem_t* pr = &job->pr;
    int64_t D = pr->head_dim, G = pr->num_q_heads / pr->num_kv_heads;
    int64_t items = job->num_chunks * pr->num_kv_heads;
    double* q = (double*)malloc(sizeof(double) * D);
    for (;;) {
        int64_t item = take_item(&job->next_item, &job->lock);
        if (item >= items) break;
        int64_t c = item / pr->num_kv_heads, kvh = item % pr->num_kv_heads;
        int64_t s = job->seq_of_chunk[c];
        int64_t first = job->cu_q_lens[c], n = job->cu_q_lens[c + 1] - first;
        int64_t start = job->q_start_pos[c];
        int64_t len = start + n; /* keys needed by the chunk's last query */
        int bad = s < 0 || s >= job->num_seqs || n < 0 || start < 0 || len > job->context_lens[s];
        double *kc = NULL, *vc = NULL, *x = NULL;
        if (!bad && len > 0) {
            kc = (double*)malloc(sizeof(double) * len * D);
            vc = (double*)malloc(sizeof(double) * len * D);
            x = (double*)malloc(sizeof(double) * len);
            bad = gather_contiguous(pr, s, kvh, len, kc, vc) != 0;
        }
        if (bad) {
            pthread_mutex_lock(&job->lock);
            job->status = -1;
            pthread_mutex_unlock(&job->lock);
        } else {
            for (int64_t i = 0; i < n; ++i) {
                int64_t p = start + i;
                for (int64_t g = 0; g < G; ++g) {
                    int64_t h = kvh * G + g;
                    int64_t row = (first + i) * pr->num_q_heads + h;
                    for (int64_t d = 0; d < D; ++d) q[d] = load_elem(pr->q, pr->dtype, row * D + d);
                    attend(q, kc, vc, p + 1, D, pr->scale, x, job->out + row * D);
                }
            }
        }
        free(kc); free(vc); free(x);
    }
    free(q);
    return NULL;
}

/* Chunked prefill: chunk c holds queries cu_q_lens[c] .. cu_q_lens[c+1]-1 of
 * sequence seq_of_chunk[c] at positions q_start_pos[c] + i ([P1] 工作原理:
 * prefill takes blocks for the input length; the chunk's K/V are already in
 * the pool).  q and out are [total_q][num_q_heads][head_dim]; out is fp64. */
int oracle_prefill(double* out, const void* q, const int32_t* cu_q_lens, const int32_t* q_start_pos,
                   const int32_t* seq_of_chunk, int64_t num_chunks, int64_t num_seqs, int64_t num_q_heads,
                   int64_t num_kv_heads, int64_t head_dim, int dtype, const void* k_cache,
                   const void* v_cache, int64_t num_blocks, int64_t block_size,
                   const int32_t* block_tables, int64_t max_blocks_per_seq,
                   const int32_t* context_lens, double scale, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    prefill_job_t job;
    job.pr = (problem_t){q, k_cache, v_cache, dtype, num_q_heads, num_kv_heads, head_dim,
                         num_blocks, block_size, block_tables, max_blocks_per_seq, scale};
    job.out = out;
    job.cu_q_lens = cu_q_lens;
    job.q_start_pos = q_start_pos;
    job.seq_of_chunk = seq_of_chunk;
    job.context_lens = context_lens;
    job.num_chunks = num_chunks;
    job.num_seqs = num_seqs;
    job.next_item = 0;
    job.status = 0;
    pthread_mutex_init(&job.lock, NULL);
    run_pool(prefill_worker, &job, num_threads);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}
