/*
 * Plain, slow, fp64 CPU oracle for load-balanced paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the CUDA
 * library: it decodes bf16 and E4M3 by itself, from the formats' definitions.
 *
 * Sources (web pages; section titles as printed on them):
 *   [HPC-Ops x SGLang blog]  "HPC-Ops × SGLang：腾讯混元开源高性能 Attention、
 *       Router GEMM 与 MoE 算子", sections
 *       "Attention：变长 decode 的负载均衡" (static split-KV and its two forms),
 *       "围绕活跃 KV 工作进行调度" (assign kernel, budget, greedy bins,
 *       minimum-work floor, partial outputs with log-sum-exp, combine),
 *       "融合式 attention 前导" (FP8 Q with per-token/per-head scale).
 *   [Hy3 preview write-up]  section
 *       2.1.1 "Attention动态调度" (uniform tile granularity, greedy bin
 *       packing, task map built once per step, combine kernel).
 *
 * Functions and what pins them (tests/test_oracle_*.py):
 *   oracle_bf16_to_double, oracle_e4m3_to_double -- all codes vs torch's own
 *       conversions, plus spec values.
 *   oracle_plan -- invariants (exact cover, bin sizes within one tile of the
 *       budget, floor on bin size), closed forms, hand-worked examples.
 *   oracle_attention_span / oracle_attention -- numpy/scipy dense softmax,
 *       closed forms (q = 0, constant V, one token, GQA probe), page-pool
 *       permutation invariance.
 *   oracle_merge -- split/merge invariant (merged partials equal unsplit).
 *   oracle_static_split -- exact-cover and size properties of the two static
 *       split-KV forms.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* dtype codes used by the oracle's own API (independent of the library's). */
#define ORC_BF16 0
#define ORC_E4M3 1

/* ------------------------------------------------------------------------- */
/* Number formats                                                             */
/* ------------------------------------------------------------------------- */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. */
double oracle_bf16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double v;
    if (e == 0xFF) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -126 - 7); /* subnormal: 0.m * 2^-126 */
    } else {
        v = ldexp(1.0 + (double)m / 128.0, e - 127);
    }
    return sign ? -v : v;
}

/* OCP 8-bit E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448. */
double oracle_e4m3_to_double(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double v;
    if (e == 0xF && m == 0x7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -6 - 3); /* subnormal: 0.m * 2^-6 */
    } else {
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    }
    return sign ? -v : v;
}

static double load_elem(const void *base, int dtype, int64_t idx) {
    if (dtype == ORC_BF16) return oracle_bf16_to_double(((const uint16_t *)base)[idx]);
    return oracle_e4m3_to_double(((const uint8_t *)base)[idx]);
}

/* ------------------------------------------------------------------------- */
/* Task map: the assign step, walked tile by tile                             */
/* ------------------------------------------------------------------------- */

/*
 * [HPC-Ops x SGLang blog, "围绕活跃 KV 工作进行调度"]: the assign kernel cuts
 * every sequence into uniform 64-token tiles, sums the tiles over all heads and
 * requests, divides the total by the number of persistent CTAs to set a per-CTA
 * tile budget, and fills each CTA's bin up to that budget before spilling into
 * the next bin; a minimum-work floor prevents over-partitioning when the total
 * is small.  [Hy3 preview write-up, 2.1.1] calls the fill "greedy bin packing".
 *
 * Readings where the pages are silent:
 *  - unit u = (request b, KV head h), numbered u = b*Hkv + h; tiles are walked
 *    request-major, then KV head, then tile index;
 *  - the budget is the real number T / C_eff; "fill up to the budget" means a
 *    tile joins bin i while the tiles placed in bins 0..i stay <= (i+1)*T/C_eff;
 *  - the floor m caps the number of bins: C_eff = min(C, max(1, floor(T/m)));
 *  - a descriptor is one maximal run of one unit's tiles inside one bin, with
 *    k its index among that unit's descriptors;
 *  - a negative length is invalid input: it counts as zero tiles and sets bit 1
 *    of the status word.
 *
 * Outputs (caller-allocated):
 *  cta_desc_begin[C+1]: descriptors of bin i are [begin[i], begin[i+1]).
 *  descs[4*max_descs]: {u, t0, t1, k}, tile indices local to the unit.
 *  unit_partial_begin[U], unit_num_partials[U]: first descriptor and count of
 *      unit u (for an empty unit, the number of descriptors before it).
 *  meta[4] = {T, C_eff, num_descs, status}.
 * Returns 0, or -1 on bad arguments, or -2 if max_descs is too small.
 */
int oracle_plan(const int32_t *seq_lens, int32_t batch, int32_t num_kv_heads,
                int32_t num_ctas, int32_t tile, int32_t min_tiles_per_split,
                int32_t max_descs, int32_t *cta_desc_begin, int32_t *descs,
                int32_t *unit_partial_begin, int32_t *unit_num_partials,
                int32_t *meta) {
    if (batch < 0 || num_kv_heads < 1 || num_ctas < 1 || tile < 1 || min_tiles_per_split < 1)
        return -1;
    int64_t U = (int64_t)batch * num_kv_heads;
    int32_t status = 0;

    /* Step 1: cut each (request, head) into tiles and sum them. */
    int64_t T = 0;
    for (int64_t u = 0; u < U; ++u) {
        int32_t len = seq_lens[u / num_kv_heads];
        if (len < 0) { status |= 1; len = 0; }
        T += ((int64_t)len + tile - 1) / tile;
    }

    /* Step 2: budget T / C_eff with the minimum-work floor. */
    int64_t C_eff = 0;
    if (T > 0) {
        int64_t by_floor = T / min_tiles_per_split;
        if (by_floor < 1) by_floor = 1;
        C_eff = by_floor < num_ctas ? by_floor : num_ctas;
    }

    for (int32_t i = 0; i <= num_ctas; ++i) cta_desc_begin[i] = -1;

    /* Step 3: greedy fill, one tile at a time. */
    int64_t bin = 0;     /* current bin */
    int64_t placed = 0;  /* tiles placed so far (all bins) */
    int32_t nd = 0;      /* descriptors emitted */
    int64_t last_bin = -1, last_unit = -1;
    for (int64_t u = 0; u < U; ++u) {
        int32_t len = seq_lens[u / num_kv_heads];
        if (len < 0) len = 0;
        int64_t n_u = ((int64_t)len + tile - 1) / tile;
        unit_partial_begin[u] = nd;
        unit_num_partials[u] = 0;
        for (int64_t t = 0; t < n_u; ++t) {
            /* spill while this tile would push the bin past its budget */
            while ((placed + 1) * C_eff > (bin + 1) * T) ++bin;
            if (bin != last_bin || u != last_unit) {
                if (nd >= max_descs) return -2;
                descs[4 * nd + 0] = (int32_t)u;
                descs[4 * nd + 1] = (int32_t)t;
                descs[4 * nd + 2] = (int32_t)(t + 1);
                descs[4 * nd + 3] = unit_num_partials[u];
                unit_num_partials[u] += 1;
                if (cta_desc_begin[bin] < 0) cta_desc_begin[bin] = nd;
                ++nd;
                last_bin = bin;
                last_unit = u;
            } else {
                descs[4 * (nd - 1) + 2] = (int32_t)(t + 1);
            }
            ++placed;
        }
    }
    /* Bins that received nothing (only bins >= C_eff) start at num_descs. */
    cta_desc_begin[num_ctas] = nd;
    for (int32_t i = num_ctas - 1; i >= 0; --i)
        if (cta_desc_begin[i] < 0) cta_desc_begin[i] = cta_desc_begin[i + 1];

    meta[0] = (int32_t)T;
    meta[1] = (int32_t)C_eff;
    meta[2] = nd;
    meta[3] = status;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Static split-KV: the two fixed-grid forms                                  */
/* ------------------------------------------------------------------------- */

/*
 * [HPC-Ops x SGLang blog, "Attention：变长 decode 的负载均衡"]: a static split-KV
 * scheduler maps work onto a fixed grid over KV heads, requests and KV chunks,
 * either (mode 0) with a fixed number of splits per request, so long requests
 * get heavy chunks, or (mode 1) with a fixed chunk size, so the grid reserves
 * enough splits for the longest request and short ones get empty chunks.
 * Reading: splits are tile-aligned; mode 0 uses c = ceil(n_u / S) tiles per
 * split with S = param; mode 1 uses c = param / tile tiles per split with
 * S = ceil(max_len / param).  Split s covers tiles [s*c, min((s+1)*c, n_u)),
 * empty when s*c >= n_u.
 *
 * oracle_static_num_splits returns S; oracle_static_split writes the tile range
 * of split s of a unit with n_tiles tiles.
 */
int32_t oracle_static_num_splits(int32_t mode, int32_t param, int32_t max_seq_len) {
    if (mode == 0) return param;
    int64_t s = ((int64_t)max_seq_len + param - 1) / param;
    return s < 1 ? 1 : (int32_t)s;
}

void oracle_static_split(int32_t mode, int32_t param, int32_t tile, int32_t num_splits,
                         int32_t n_tiles, int32_t s, int32_t *t0, int32_t *t1) {
    int64_t c;
    if (mode == 0) c = ((int64_t)n_tiles + num_splits - 1) / num_splits;
    else c = param / tile;
    int64_t a = (int64_t)s * c, b = a + c;
    if (a > n_tiles) a = n_tiles;
    if (b > n_tiles) b = n_tiles;
    *t0 = (int32_t)a;
    *t1 = (int32_t)b;
}

/* ------------------------------------------------------------------------- */
/* Attention by definition                                                    */
/* ------------------------------------------------------------------------- */

typedef struct {
    const void *q; int q_dtype; const float *q_scale;
    const void *k_pages; const void *v_pages; int kv_dtype;
    const float *k_scale; const float *v_scale;
    const int32_t *block_table; int32_t max_pages_per_req; int32_t num_pages;
    const int32_t *seq_lens; int32_t batch; int32_t num_q_heads; int32_t num_kv_heads;
    int32_t head_dim; int32_t page_size; double sm_scale; int32_t q_len;
    int32_t kv_layout;  /* 0: pages [num_pages][Hkv][P][d] (HND); 1: [num_pages][P][Hkv][d] (NHD) */
} orc_problem;

/* Element row of (page, KV head, slot) in the K/V pools; the FP8 scales are always laid out
 * [num_pages][Hkv][P] (scale_row). */
static int64_t data_row(const orc_problem *p, int64_t page, int32_t h, int64_t slot) {
    if (p->kv_layout == 1) return (page * p->page_size + slot) * p->num_kv_heads + h;
    return (page * p->num_kv_heads + h) * p->page_size + slot;
}
static int64_t scale_row(const orc_problem *p, int64_t page, int32_t h, int64_t slot) {
    return (page * p->num_kv_heads + h) * p->page_size + slot;
}

/*
 * Exact attention of the G query heads of request b that share KV head h, over
 * the tokens [tok0, tok1) of that request, for each of the request's q_len query
 * tokens.  Query token i (0 <= i < q_len) stands at position len_b - q_len + i
 * and sees the tokens t <= that position (causal within the draft of a
 * multi-token verify step: Hy3 preview write-up 2.5 "MTP与异步调度优化"; SGLang
 * Low-Latency Mode: Kernels and Runtime, section 1, a verify of 1 + 5 draft
 * tokens), so its range is
 * [tok0, min(tok1, len_b - q_len + i + 1)):
 *   s_t = sm_scale * sum_k Q[b, i, j, k] * K[t, k]          (j = h*G .. h*G+G-1)
 *   o = sum_t exp(s_t - M) V[t, :] / sum_t exp(s_t - M), M = max_t s_t
 *   lse = M + ln sum_t exp(s_t - M)
 * Output row i*G + g.  Token t of request b lives in page block_table[b][t /
 * page_size] at slot t mod page_size; a page holds [Hkv][page_size][d]
 * elements (kv_layout 0, "HND") or [page_size][Hkv][d] (kv_layout 1, "NHD";
 * the blog's integration reads the serving runtime's paged KV store without a
 * layout conversion, and both orders occur there).  FP8 values are decode(byte) * scale: Q scale per (b, i, q head),
 * K/V scale per (page, KV head, slot).  An empty range gives o = 0, lse = -inf.
 * Returns nonzero if a page id is out of range.
 */
static int span(const orc_problem *p, int32_t b, int32_t h, int64_t tok0, int64_t tok1,
                double *out /*[q_len*G*d]*/, double *lse /*[q_len*G]*/, double *scratch /*[tok1-tok0]*/) {
    const int32_t G = p->num_q_heads / p->num_kv_heads;
    const int32_t d = p->head_dim;
    const int32_t P = p->page_size;
    const int64_t len = p->seq_lens[b] > 0 ? p->seq_lens[b] : 0;
    for (int32_t qi = 0; qi < p->q_len; ++qi) {
        int64_t end = len - p->q_len + qi + 1;  /* tokens this query token sees */
        if (end > tok1) end = tok1;
        for (int32_t g = 0; g < G; ++g) {
            int32_t j = h * G + g;
            int64_t r = (int64_t)qi * G + g;
            double *o = out + r * d;
            for (int32_t k = 0; k < d; ++k) o[k] = 0.0;
            if (end <= tok0) { lse[r] = -INFINITY; continue; }
            int64_t qrow = ((int64_t)b * p->q_len + qi) * p->num_q_heads + j;
            double qs = (p->q_dtype == ORC_E4M3) ? (double)p->q_scale[qrow] : 1.0;
            int64_t qbase = qrow * d;
            /* scores */
            double M = -INFINITY;
            for (int64_t t = tok0; t < end; ++t) {
                int32_t page = p->block_table[(int64_t)b * p->max_pages_per_req + t / P];
                if (page < 0 || page >= p->num_pages) return 1;
                int64_t row = data_row(p, page, h, t % P);
                double ks = (p->kv_dtype == ORC_E4M3) ? (double)p->k_scale[scale_row(p, page, h, t % P)] : 1.0;
                double dot = 0.0;
                for (int32_t k = 0; k < d; ++k)
                    dot += load_elem(p->q, p->q_dtype, qbase + k) * qs *
                           load_elem(p->k_pages, p->kv_dtype, row * d + k) * ks;
                double sc = p->sm_scale * dot;
                scratch[t - tok0] = sc;
                if (sc > M) M = sc;
            }
            /* softmax-weighted sum of V */
            double l = 0.0;
            for (int64_t t = tok0; t < end; ++t) {
                int32_t page = p->block_table[(int64_t)b * p->max_pages_per_req + t / P];
                int64_t row = data_row(p, page, h, t % P);
                double vs = (p->kv_dtype == ORC_E4M3) ? (double)p->v_scale[scale_row(p, page, h, t % P)] : 1.0;
                double w = exp(scratch[t - tok0] - M);
                l += w;
                for (int32_t k = 0; k < d; ++k)
                    o[k] += w * load_elem(p->v_pages, p->kv_dtype, row * d + k) * vs;
            }
            for (int32_t k = 0; k < d; ++k) o[k] /= l;
            lse[r] = M + log(l);
        }
    }
    return 0;
}

static int check_problem(const orc_problem *p) {
    if (p->batch < 0 || p->num_kv_heads < 1 || p->num_q_heads < 1 || p->head_dim < 1 ||
        p->page_size < 1 || p->num_q_heads % p->num_kv_heads != 0 || p->q_len < 1 ||
        (p->kv_layout != 0 && p->kv_layout != 1))
        return -1;
    if (p->q_dtype != ORC_BF16 && p->q_dtype != ORC_E4M3) return -1;
    if (p->kv_dtype != ORC_BF16 && p->kv_dtype != ORC_E4M3) return -1;
    return 0;
}

/* One (request, KV head, token range): out [q_len*G*d], lse [q_len*G] (row i*G + g). */
int oracle_attention_span(const void *q, int32_t q_dtype, const float *q_scale,
                          const void *k_pages, const void *v_pages, int32_t kv_dtype,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                          const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size, double sm_scale,
                          int32_t q_len, int32_t kv_layout, int32_t b, int32_t h, int64_t tok0, int64_t tok1,
                          double *out, double *lse) {
    orc_problem p = {q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale,
                     block_table, max_pages_per_req, num_pages, seq_lens, batch,
                     num_q_heads, num_kv_heads, head_dim, page_size, sm_scale, q_len, kv_layout};
    if (check_problem(&p) || b < 0 || b >= batch || h < 0 || h >= num_kv_heads) return -1;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(tok1 > tok0 ? tok1 - tok0 : 1));
    if (!scratch) return -3;
    int rc = span(&p, b, h, tok0, tok1, out, lse, scratch);
    free(scratch);
    return rc;
}

typedef struct {
    const orc_problem *p;
    const int32_t *units; int64_t n_units;
    double *out; double *out_lse;
    int64_t next; pthread_mutex_t *mu; int rc;
} orc_job;

static void *attention_worker(void *arg) {
    orc_job *job = (orc_job *)arg;
    const orc_problem *p = job->p;
    const int32_t G = p->num_q_heads / p->num_kv_heads;
    int64_t cap = 1;
    for (int32_t b = 0; b < p->batch; ++b) if (p->seq_lens[b] > cap) cap = p->seq_lens[b];
    double *scratch = (double *)malloc(sizeof(double) * (size_t)cap);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)p->q_len * G * (p->head_dim + 1));
    if (!scratch || !tmp) { free(scratch); free(tmp); job->rc = -3; return NULL; }
    for (;;) {
        pthread_mutex_lock(job->mu);
        int64_t k = job->next++;
        pthread_mutex_unlock(job->mu);
        if (k >= job->n_units) break;
        int32_t u = job->units ? job->units[k] : (int32_t)k;
        int32_t b = u / p->num_kv_heads, h = u % p->num_kv_heads;
        int32_t len = p->seq_lens[b] > 0 ? p->seq_lens[b] : 0;
        double *o = tmp, *l = tmp + (int64_t)p->q_len * G * p->head_dim;
        if (span(p, b, h, 0, len, o, l, scratch)) job->rc = 1;
        for (int32_t qi = 0; qi < p->q_len; ++qi) {  /* to out[b][qi][h*G + g] */
            int64_t row = ((int64_t)b * p->q_len + qi) * p->num_q_heads + (int64_t)h * G;
            for (int32_t g = 0; g < G; ++g) {
                job->out_lse[row + g] = l[qi * G + g];
                for (int32_t k = 0; k < p->head_dim; ++k)
                    job->out[(row + g) * p->head_dim + k] = o[((int64_t)qi * G + g) * p->head_dim + k];
            }
        }
    }
    free(scratch);
    free(tmp);
    return NULL;
}

/*
 * Unsplit attention for every query token and query head of the listed units
 * (u = b*Hkv + h; units == NULL means all B*Hkv units), written at
 * out[b][i][j][:] and out_lse[b][i][j] (i < q_len; q_len = 1 is a plain decode
 * step).  n_threads <= 0 uses every online core.  Returns nonzero on a
 * bad argument or an out-of-range page id.
 */
int oracle_attention(const void *q, int32_t q_dtype, const float *q_scale,
                     const void *k_pages, const void *v_pages, int32_t kv_dtype,
                     const float *k_scale, const float *v_scale,
                     const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                     const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t page_size, double sm_scale,
                     int32_t q_len, int32_t kv_layout, const int32_t *units, int64_t n_units, int32_t n_threads,
                     double *out, double *out_lse) {
    orc_problem p = {q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale,
                     block_table, max_pages_per_req, num_pages, seq_lens, batch,
                     num_q_heads, num_kv_heads, head_dim, page_size, sm_scale, q_len, kv_layout};
    if (check_problem(&p)) return -1;
    if (!units) n_units = (int64_t)batch * num_kv_heads;
    if (n_threads <= 0) n_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_units) n_threads = n_units > 0 ? (int32_t)n_units : 1;
    pthread_mutex_t mu;
    pthread_mutex_init(&mu, NULL);
    orc_job job = {&p, units, n_units, out, out_lse, 0, &mu, 0};
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int32_t i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, attention_worker, &job);
    for (int32_t i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&mu);
    return job.rc;
}

/* Number of threads oracle_attention uses for n_threads <= 0. */
int32_t oracle_default_threads(void) { return (int32_t)sysconf(_SC_NPROCESSORS_ONLN); }

/* ------------------------------------------------------------------------- */
/* Merge of partial results under the global softmax                         */
/* ------------------------------------------------------------------------- */

/*
 * [HPC-Ops x SGLang blog, "围绕活跃 KV 工作进行调度"]: each partial output comes
 * with its log-sum-exp; the combine step merges the actual number of partials
 * of a (request, head) under the global softmax normalisation:
 *   L = ln sum_k exp(lse_k),   o = sum_k exp(lse_k - L) o_k.
 * Partials with lse = -inf contribute nothing; if every lse is -inf (or n = 0)
 * the result is o = 0, L = -inf.  o: [n][rows][d], lse: [n][rows].
 */
void oracle_merge(const double *o, const double *lse, int32_t n, int32_t rows, int32_t d,
                  double *out /*[rows*d]*/, double *out_lse /*[rows]*/) {
    for (int32_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int32_t k = 0; k < n; ++k) if (lse[(int64_t)k * rows + r] > M) M = lse[(int64_t)k * rows + r];
        for (int32_t i = 0; i < d; ++i) out[(int64_t)r * d + i] = 0.0;
        if (M == -INFINITY) { out_lse[r] = -INFINITY; continue; }
        double s = 0.0;
        for (int32_t k = 0; k < n; ++k) s += exp(lse[(int64_t)k * rows + r] - M);
        double L = M + log(s);
        for (int32_t k = 0; k < n; ++k) {
            double w = exp(lse[(int64_t)k * rows + r] - L);
            if (w == 0.0) continue;
            for (int32_t i = 0; i < d; ++i)
                out[(int64_t)r * d + i] += w * o[((int64_t)k * rows + r) * d + i];
        }
        out_lse[r] = L;
    }
}
