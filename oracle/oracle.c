/*
 * Oracle for single-query decode attention: a plain, slow, fp64 CPU restatement of what the
 * decode-attention region computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg may call it; the library never links, loads or calls it, and
 * it shares no code, header or constant with the CUDA path.
 *
 * What it computes (one query row per (b, h), seq_q = 1):
 *   - "DecodeFlashSpec" (docs.rs, fuel_dispatch::decode_flash), fields q / k / v / k_len /
 *     softmax_scale / causal: q [B,Hq,1,D] attends rows [0, k_len) of the capacity buffers
 *     k, v [B,Hkv,capacity,D]; causal is a no-op because a single query row sees the whole live
 *     prefix; the output has q's shape.  The flash arm must equal arm 0, the decomposed chain
 *     scores -> softmax -> P.V, which is what this file writes out.
 *   - "DflashScratch" (docs.metrale.ai, dflash_head), field option_b_indirect_args_dev: a paged
 *     cache whose per-sequence kv_len is the first u32 of a per-sequence args record.
 *   - "AttnV41" (docs.metrale.ai, attn_v41), method decode_fixed_topk: attention over a
 *     fixed-width int32 selection in which a -1 entry adds exactly zero to the denominator and
 *     nothing to the output.
 *
 * Readings where the pages say nothing (each is also listed with the design notes):
 *   - GQA: query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *   - An empty attended set (k_len = 0, kv_len = 0, all entries masked) gives a zero row
 *     (the null-row convention of flashinfer packed_fused_kda_decode).
 *   - Paged: kv_len is clamped to max_pages_per_seq * page_size; a row whose block-table entry
 *     lies outside [0, num_pages) is skipped.
 *   - Sparse: every entry outside [0, pool_rows) (-1 and any other) is skipped; duplicates
 *     count once per entry.
 *
 * Arithmetic: every bf16 input is widened exactly to double; for each (b, h):
 *   s_j = scale * sum_d q[d] * K_j[d]            (d ascending)
 *   m   = max_j s_j
 *   w_j = exp(s_j - m),  l = sum_j w_j           (rows in attended order)
 *   out = (sum_j w_j * V_j) / l
 * No blocking, splitting or reordering beyond that.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static double widen_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Softmax-weighted average of the n rows listed in krow/vrow (element offsets into k/v). */
static void attend_rows(const uint16_t *qrow, const uint16_t *k, const uint16_t *v,
                        const int64_t *krow, const int64_t *vrow, int64_t n, int D,
                        double scale, double *out, double *s) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen_bf16(qrow[d]) * widen_bf16(k[krow[j] + d]);
        s[j] = scale * dot;
    }
    double m = s[0];
    for (int64_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < n; ++j)
        for (int d = 0; d < D; ++d) out[d] += s[j] * widen_bf16(v[vrow[j] + d]);
    for (int d = 0; d < D; ++d) out[d] /= l;
}

enum { VAR_DENSE = 0, VAR_PAGED = 1, VAR_SPARSE = 2 };

typedef struct {
    int variant;
    const uint16_t *q, *k, *v;
    double *out;
    int B, Hq, Hkv, D;
    double scale;
    /* dense */
    int64_t capacity, k_len;
    /* paged */
    const int32_t *block_table;
    int64_t max_pages, page_size, num_pages;
    const uint32_t *kv_lens;
    int64_t kv_len_stride;
    /* sparse */
    int64_t pool_rows;
    const int32_t *sel;
    int64_t width;
    /* query tokens per sequence (q, out [B, Hq, Sq, D]) and causal masking inside them */
    int Sq, causal;
    /* which (b*Hq + h) to compute */
    const int64_t *pairs;
    int64_t npairs;
    int nthreads;
    int64_t max_rows;
    int status;
} job_t;

typedef struct {
    job_t *job;
    int tid;
} worker_t;

/* The live length of sequence b (dense: k_len; paged: its kv_len, clamped). */
static int64_t live_len(const job_t *J, int b) {
    if (J->variant == VAR_DENSE) return J->k_len;
    int64_t len = (int64_t)J->kv_lens[(int64_t)b * J->kv_len_stride];
    const int64_t cap = J->max_pages * J->page_size;
    return len > cap ? cap : len;
}

/* Builds the attended row list of (b, g) in attended order, keeping only row positions j < jmax
 * (dense and paged); returns the row count. */
static int64_t gather_rows(const job_t *J, int b, int g, int64_t jmax, int64_t *krow) {
    const int64_t D = J->D;
    int64_t n = 0;
    if (J->variant == VAR_DENSE) {
        const int64_t base = ((int64_t)b * J->Hkv + g) * J->capacity;
        const int64_t len = J->k_len < jmax ? J->k_len : jmax;
        for (int64_t j = 0; j < len; ++j) krow[n++] = (base + j) * D;
    } else if (J->variant == VAR_PAGED) {
        int64_t len = live_len(J, b);
        if (len > jmax) len = jmax;
        for (int64_t j = 0; j < len; ++j) {
            const int64_t page = J->block_table[(int64_t)b * J->max_pages + j / J->page_size];
            if (page < 0 || page >= J->num_pages) continue;
            krow[n++] = ((page * J->Hkv + g) * J->page_size + j % J->page_size) * D;
        }
    } else {
        const int64_t base = ((int64_t)b * J->Hkv + g) * J->pool_rows;
        for (int64_t i = 0; i < J->width; ++i) {
            const int64_t idx = J->sel[(int64_t)b * J->width + i];
            if (idx < 0 || idx >= J->pool_rows) continue;
            krow[n++] = (base + idx) * D;
        }
    }
    return n;
}

static void *worker(void *arg) {
    worker_t *W = (worker_t *)arg;
    job_t *J = W->job;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(J->max_rows > 0 ? J->max_rows : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->max_rows > 0 ? J->max_rows : 1));
    if (!rows || !s) {
        J->status = ORACLE_ENOMEM;
        free(rows);
        free(s);
        return NULL;
    }
    const int G = J->Hq / J->Hkv;
    const int64_t total = J->pairs ? J->npairs : (int64_t)J->B * J->Hq;
    for (int64_t t = W->tid; t < total; t += J->nthreads) {
        const int64_t bh = J->pairs ? J->pairs[t] : t;
        const int b = (int)(bh / J->Hq), h = (int)(bh % J->Hq);
        const int g = h / G;
        for (int i = 0; i < J->Sq; ++i) {
            /* the Sq new tokens are the last Sq rows of the live prefix: causal token i sees rows
             * [0, len - Sq + i] */
            const int64_t jmax = J->causal ? live_len(J, b) - J->Sq + i + 1 : INT64_MAX;
            const int64_t n = jmax <= 0 ? 0 : gather_rows(J, b, g, jmax, rows);
            const int64_t row = bh * J->Sq + i;
            /* K and V share one layout, so the same element offsets address both. */
            attend_rows(J->q + row * J->D, J->k, J->v, rows, rows, n, J->D, J->scale,
                        J->out + row * J->D, s);
        }
    }
    free(rows);
    free(s);
    return NULL;
}

static int run_job(job_t *J) {
    if (!J->q || !J->k || !J->v || !J->out || J->B < 0 || J->Hq <= 0 || J->Hkv <= 0 ||
        J->D <= 0 || J->Hq % J->Hkv != 0)
        return ORACLE_EINVAL;
    if (J->pairs) {
        for (int64_t i = 0; i < J->npairs; ++i)
            if (J->pairs[i] < 0 || J->pairs[i] >= (int64_t)J->B * J->Hq) return ORACLE_EINVAL;
    }
    int nt = J->nthreads;
    if (nt <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nt = c > 0 ? (int)c : 1;
    }
    if (nt > 512) nt = 512;
    J->nthreads = nt;
    J->status = ORACLE_OK;
    pthread_t th[512];
    worker_t w[512];
    for (int i = 0; i < nt; ++i) {
        w[i].job = J;
        w[i].tid = i;
    }
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker, &w[i]) != 0) break;
        ++started;
    }
    if (started == 0) {
        /* no threads available: run every shard on the caller's thread */
        for (int i = 0; i < nt; ++i) worker(&w[i]);
        return J->status;
    }
    if (started < nt) {
        /* workers were sharded for nt threads; finish the missing shards here */
        for (int i = started; i < nt; ++i) worker(&w[i]);
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    return J->status;
}

/* Dense: q [B,Hq,D], k/v [B,Hkv,capacity,D] (bf16 bits), out [B,Hq,D] fp64. */
int oracle_dense(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out, int B,
                 int Hq, int Hkv, int D, int64_t capacity, int64_t k_len, double scale,
                 const int64_t *pairs, int64_t npairs, int nthreads) {
    if (k_len < 0 || k_len > capacity) return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.variant = VAR_DENSE;
    J.q = q; J.k = k; J.v = v; J.out = out;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.capacity = capacity; J.k_len = k_len;
    J.pairs = pairs; J.npairs = npairs; J.nthreads = nthreads;
    J.max_rows = k_len;
    J.Sq = 1;
    return run_job(&J);
}

/* Paged: pools [num_pages,Hkv,page_size,D]; block_table [B,max_pages]; kv_len of sequence b is
 * kv_lens[b * kv_len_stride] (stride 3 reads the first word of {kv_len, q_offset, q_rope_pos}). */
int oracle_paged(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool, double *out,
                 const int32_t *block_table, int64_t max_pages, int64_t page_size,
                 int64_t num_pages, const uint32_t *kv_lens, int64_t kv_len_stride, int B, int Hq,
                 int Hkv, int D, double scale, const int64_t *pairs, int64_t npairs,
                 int nthreads) {
    if (!block_table || !kv_lens || max_pages < 0 || page_size <= 0 || num_pages < 0 ||
        kv_len_stride <= 0)
        return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.variant = VAR_PAGED;
    J.q = q; J.k = k_pool; J.v = v_pool; J.out = out;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.block_table = block_table; J.max_pages = max_pages; J.page_size = page_size;
    J.num_pages = num_pages; J.kv_lens = kv_lens; J.kv_len_stride = kv_len_stride;
    J.pairs = pairs; J.npairs = npairs; J.nthreads = nthreads;
    J.max_rows = max_pages * page_size;
    J.Sq = 1;
    return run_job(&J);
}

/* Sparse: pools [B,Hkv,pool_rows,D]; sel [B,width] int32 shared by all KV heads of a sequence. */
int oracle_sparse(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool, double *out,
                  int64_t pool_rows, const int32_t *sel, int64_t width, int B, int Hq, int Hkv,
                  int D, double scale, const int64_t *pairs, int64_t npairs, int nthreads) {
    if (!sel || pool_rows < 0 || width < 0) return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.variant = VAR_SPARSE;
    J.q = q; J.k = k_pool; J.v = v_pool; J.out = out;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.pool_rows = pool_rows; J.sel = sel; J.width = width;
    J.pairs = pairs; J.npairs = npairs; J.nthreads = nthreads;
    J.max_rows = width;
    J.Sq = 1;
    return run_job(&J);
}

/* Several query tokens per sequence (a multi-token verify step): q, out [B, Hq, Sq, D].  The Sq
 * new tokens are the last Sq rows of each sequence's live prefix, so with causal != 0 token i
 * attends rows [0, len - Sq + i] (a token at or before row 0 of the prefix sees nothing: a zero
 * row); with causal = 0 every token attends the whole prefix [0, len).  Sq = 1 is the single-query
 * decode above.  "DecodeFlashSpec" (q [B,Hq,Sq,D], field causal), "AttnV41" method forward (m
 * tokens at start_pos). */
int oracle_dense_mq(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out, int B,
                    int Hq, int Hkv, int D, int Sq, int causal, int64_t capacity, int64_t k_len,
                    double scale, int nthreads) {
    if (k_len < 0 || k_len > capacity || Sq < 1) return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.variant = VAR_DENSE;
    J.q = q; J.k = k; J.v = v; J.out = out;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.capacity = capacity; J.k_len = k_len;
    J.nthreads = nthreads;
    J.max_rows = k_len;
    J.Sq = Sq; J.causal = causal;
    return run_job(&J);
}

int oracle_paged_mq(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool, double *out,
                    const int32_t *block_table, int64_t max_pages, int64_t page_size,
                    int64_t num_pages, const uint32_t *kv_lens, int64_t kv_len_stride, int B,
                    int Hq, int Hkv, int D, int Sq, int causal, double scale, int nthreads) {
    if (!block_table || !kv_lens || max_pages < 0 || page_size <= 0 || num_pages < 0 ||
        kv_len_stride <= 0 || Sq < 1)
        return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.variant = VAR_PAGED;
    J.q = q; J.k = k_pool; J.v = v_pool; J.out = out;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.block_table = block_table; J.max_pages = max_pages; J.page_size = page_size;
    J.num_pages = num_pages; J.kv_lens = kv_lens; J.kv_len_stride = kv_len_stride;
    J.nthreads = nthreads;
    J.max_rows = max_pages * page_size;
    J.Sq = Sq; J.causal = causal;
    return run_job(&J);
}

/* Dense attention of one (b, h) restricted to rows [j0, j1): the normalised output o [D] and
 * lse = m + log(l) (natural log; -inf and o = 0 for an empty range).  Used by the tests to check
 * the log-sum-exp merge identity that a split computation relies on. */
int oracle_dense_range(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                       int Hkv, int D, int64_t capacity, int b, int h, int64_t j0, int64_t j1,
                       double scale, double *o, double *lse) {
    if (!q || !k || !v || !o || !lse || Hq <= 0 || Hkv <= 0 || Hq % Hkv || b < 0 || b >= B ||
        h < 0 || h >= Hq || j0 < 0 || j1 < j0 || j1 > capacity)
        return ORACLE_EINVAL;
    const int g = h / (Hq / Hkv);
    const uint16_t *qrow = q + ((int64_t)b * Hq + h) * D;
    const int64_t base = ((int64_t)b * Hkv + g) * capacity;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (j1 == j0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(j1 - j0));
    if (!s) return ORACLE_ENOMEM;
    for (int64_t j = j0; j < j1; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen_bf16(qrow[d]) * widen_bf16(k[(base + j) * D + d]);
        s[j - j0] = scale * dot;
    }
    double m = s[0];
    for (int64_t j = 1; j < j1 - j0; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < j1 - j0; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < j1 - j0; ++j)
        for (int d = 0; d < D; ++d) o[d] += s[j] * widen_bf16(v[(base + j0 + j) * D + d]);
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
    free(s);
    return ORACLE_OK;
}

/*
 * KV append (the step before the hot path), restated from:
 *   - "DflashScratch" (docs.metrale.ai, dflash_head), field slot_mapping_dev: i64 paged-cache
 *     slot per new row, used by reshape_and_cache.  Row t of k_new / v_new ([T, Hkv, D]) goes to
 *     slot s = slot_mapping[t]: page s / page_size, position s % page_size, for every KV head.
 *     Reading: a slot outside [0, num_pages * page_size) (the usual -1 padding entry, or any
 *     other) writes nothing.
 *   - "AttnV41" (docs.metrale.ai, attn_v41), method decode_body: the window ring write at
 *     pos % window with the slot read on the device.  Row b of k_new / v_new ([B, Hkv, D]) goes to
 *     ring row positions[b] % window of sequence b's pool [B, Hkv, pool_rows, D].  Reading: a
 *     negative position writes nothing.
 * Plain element copies; later rows win when two rows name the same slot (rows in order).
 */
int oracle_append_paged(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                        uint16_t *v_pool, const int64_t *slot_mapping, int64_t T, int Hkv, int D,
                        int64_t page_size, int64_t num_pages) {
    if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping || T < 0 || Hkv <= 0 || D <= 0 ||
        page_size <= 0 || num_pages < 0)
        return ORACLE_EINVAL;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= num_pages * page_size) continue;
        const int64_t page = slot / page_size, off = slot % page_size;
        for (int g = 0; g < Hkv; ++g) {
            const int64_t src = (t * Hkv + g) * (int64_t)D;
            const int64_t dst = ((page * Hkv + g) * page_size + off) * (int64_t)D;
            for (int d = 0; d < D; ++d) {
                k_pool[dst + d] = k_new[src + d];
                v_pool[dst + d] = v_new[src + d];
            }
        }
    }
    return ORACLE_OK;
}

int oracle_append_ring(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                       uint16_t *v_pool, const int64_t *positions, int B, int Hkv, int D,
                       int64_t pool_rows, int64_t window) {
    if (!k_new || !v_new || !k_pool || !v_pool || !positions || B < 0 || Hkv <= 0 || D <= 0 ||
        window <= 0 || window > pool_rows)
        return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        const int64_t pos = positions[b];
        if (pos < 0) continue;
        const int64_t row = pos % window;
        for (int g = 0; g < Hkv; ++g) {
            const int64_t src = ((int64_t)b * Hkv + g) * D;
            const int64_t dst = (((int64_t)b * Hkv + g) * pool_rows + row) * D;
            for (int d = 0; d < D; ++d) {
                k_pool[dst + d] = k_new[src + d];
                v_pool[dst + d] = v_new[src + d];
            }
        }
    }
    return ORACLE_OK;
}
