/*
 * Seeded synthetic inputs for the sparse KV assembly path.
 *
 * This module produces INPUTS only: KV row contents for the host pool and the
 * per-step Top-k index rows.  It holds none of the method's arithmetic (no
 * residency probe, no LRU rule, no slot assignment), so both the CPU oracle and
 * the CUDA library can be fed from it without sharing any method code.
 *
 * Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants as published by
 * Vigna), used as a counter-based generator: output c of stream `key` is
 * mix(key + (c + 1) * golden).  Streams are keyed on (seed, fields...) by
 * chaining mix().  Every draw therefore depends only on its key and counter,
 * never on thread scheduling.
 *
 * Workload shapes follow the pages' evaluation: 16K-1M token contexts, 20% and
 * 40% Top-k miss rates and per-GPU batches up to 192 ("XM-Sparse: Netpreme
 * X-Mem ...", TL;DR and the test-platform section); the Top-k rows model the
 * per-layer token selection of DeepSeek-style sparse attention ("SGLang и Tair
 * представили иерархичную Sparse Attention ...", paragraph 2).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number c (0-based) of the SplitMix64 sequence started at `key`. */
static inline uint64_t sm64_at(uint64_t key, uint64_t c) { return mix64(key + (c + 1) * GOLDEN); }

static inline uint64_t key_add(uint64_t k, uint64_t field) { return mix64(k + GOLDEN + field); }

uint64_t skvw_splitmix64_at(uint64_t key, uint64_t c) { return sm64_at(key, c); }
uint64_t skvw_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t d)
{
    return key_add(key_add(key_add(key_add(seed, a), b), c), d);
}

/* A sequential stream: draw n = counter++. */
typedef struct { uint64_t key, ctr; } stream_t;
static inline uint64_t next64(stream_t *s) { return sm64_at(s->key, s->ctr++); }
/* Uniform integer in [0, n) by the multiply-high method (Lemire); the tiny
 * bias for n far below 2^64 is irrelevant for synthetic inputs. */
static inline uint64_t below(stream_t *s, uint64_t n)
{
    return (uint64_t)(((unsigned __int128)next64(s) * (unsigned __int128)n) >> 64);
}
/* Uniform double in [0, 1) with 53 random bits. */
static inline double unit01(stream_t *s) { return (double)(next64(s) >> 11) * (1.0 / 9007199254740992.0); }

/* ------------------------------------------------------------------------ */
/* KV row contents                                                            */
/* ------------------------------------------------------------------------ */

/* float32 -> bf16 with round-to-nearest-even, written from the IEEE 754
 * definition: add half an ulp of the bf16 result (minus one when the kept
 * least significant bit is 0, so exact ties round to even) and truncate.
 * Inputs here are finite values in [-1, 1). */
static inline uint16_t f32_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Element e of the KV row of token t, layer l of the request with key
 * `req_key`: bits16 = lane (e % 4) of SplitMix64 output (e / 4) of the row's
 * stream, x = (bits16 - 32768) / 32768 in [-1, 1), stored as bf16. */
void skvw_fill_rows(uint8_t *dst, int64_t dst_stride, uint64_t seed, uint64_t req_key,
                    int32_t layer, int64_t t0, int64_t n, int32_t row_elems)
{
    for (int64_t j = 0; j < n; ++j) {
        uint16_t *row = (uint16_t *)(dst + j * dst_stride);
        uint64_t key = skvw_key(seed, 0x504F4F4CULL /* "POOL" */, req_key, (uint64_t)layer,
                                (uint64_t)(t0 + j));
        for (int32_t w = 0; w * 4 < row_elems; ++w) {
            uint64_t h = sm64_at(key, (uint64_t)w);
            for (int q = 0; q < 4 && w * 4 + q < row_elems; ++q) {
                int32_t bits = (int32_t)((h >> (16 * q)) & 0xFFFFu);
                float x = (float)(bits - 32768) * (1.0f / 32768.0f);
                row[w * 4 + q] = f32_to_bf16_rne(x);
            }
        }
    }
}

/* Fill the pool region of one request: rows [0, T) of each of its L layers,
 * laid out [L][T_max][row_elems] starting at `req_base`.  Parallel over
 * (layer, token blocks); the result does not depend on the thread count. */
void skvw_fill_request(uint8_t *req_base, int32_t L, int64_t T_max, int64_t T, int32_t row_elems,
                       uint64_t seed, uint64_t req_key, int32_t nthreads)
{
    const int64_t row_bytes = (int64_t)row_elems * 2;
    const int64_t blk = 4096;
    const int64_t nblk = (T + blk - 1) / blk;
    const int64_t total = (int64_t)L * nblk;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t w = 0; w < total; ++w) {
        int32_t l = (int32_t)(w / nblk);
        int64_t t0 = (w % nblk) * blk;
        int64_t n = T - t0 < blk ? T - t0 : blk;
        skvw_fill_rows(req_base + ((int64_t)l * T_max + t0) * row_bytes, row_bytes, seed, req_key, l, t0,
                       n, row_elems);
    }
}

/* ------------------------------------------------------------------------ */
/* Top-k index rows                                                           */
/* ------------------------------------------------------------------------ */

enum { DIST_UNIFORM = 0, DIST_RECENCY = 1, DIST_ZIPF = 2 };
enum { ORDER_SORTED = 0, ORDER_SHUFFLED = 1 };

typedef struct {
    int32_t B, L, k, n_fresh, n_pad, dist, order;
    int32_t window;       /* recency: window length (last `window` positions) */
    double p_window;      /* recency: probability that a fresh pick uses the window */
    int32_t block;        /* zipf: tokens per block */
    int32_t nblocks;      /* zipf: number of ranked blocks */
    double zipf_s;        /* zipf exponent */
    uint64_t seed;
    int64_t max_len;      /* upper bound of any len passed to step() */
    int32_t *prev;        /* [B][L][kv] previous valid set */
    int32_t *prev_n;      /* [B][L] size of previous set (0 = none yet: next step is cold) */
    double *zipf_cdf;     /* [nblocks] */
    int32_t *zipf_perm;   /* [B][L][nblocks] rank -> block, per unit */
} skvw_topk;

static void unit_perm(skvw_topk *g, int32_t b, int32_t l, int32_t *perm)
{
    stream_t s = {skvw_key(g->seed, 0x5045524DULL /* "PERM" */, (uint64_t)b, (uint64_t)l, 0), 0};
    for (int32_t i = 0; i < g->nblocks; ++i) perm[i] = i;
    for (int32_t i = g->nblocks - 1; i > 0; --i) {
        int32_t j = (int32_t)below(&s, (uint64_t)i + 1);
        int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    }
}

skvw_topk *skvw_topk_create(int32_t B, int32_t L, int32_t k, int32_t n_fresh, int32_t n_pad, int32_t dist,
                            int32_t order, int32_t window, double p_window, int32_t block, int32_t nblocks,
                            double zipf_s, uint64_t seed, int64_t max_len)
{
    if (B < 1 || L < 1 || k < 1 || n_pad < 0 || n_pad >= k || n_fresh < 0 || n_fresh > k - n_pad) return NULL;
    skvw_topk *g = (skvw_topk *)calloc(1, sizeof(skvw_topk));
    if (!g) return NULL;
    g->B = B; g->L = L; g->k = k; g->n_fresh = n_fresh; g->n_pad = n_pad; g->dist = dist; g->order = order;
    g->window = window; g->p_window = p_window; g->block = block; g->nblocks = nblocks; g->zipf_s = zipf_s;
    g->seed = seed; g->max_len = max_len;
    const int32_t kv = k - n_pad;
    g->prev = (int32_t *)calloc((size_t)B * L * kv, sizeof(int32_t));
    g->prev_n = (int32_t *)calloc((size_t)B * L, sizeof(int32_t));
    if (!g->prev || !g->prev_n) goto fail;
    if (dist == DIST_ZIPF) {
        if (nblocks < 1 || block < 1) goto fail;
        g->zipf_cdf = (double *)malloc(sizeof(double) * (size_t)nblocks);
        g->zipf_perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * L * nblocks);
        if (!g->zipf_cdf || !g->zipf_perm) goto fail;
        double acc = 0.0;
        for (int32_t r = 0; r < nblocks; ++r) { acc += pow((double)(r + 1), -zipf_s); g->zipf_cdf[r] = acc; }
        for (int32_t r = 0; r < nblocks; ++r) g->zipf_cdf[r] /= acc;
        for (int32_t b = 0; b < B; ++b)
            for (int32_t l = 0; l < L; ++l) unit_perm(g, b, l, g->zipf_perm + ((size_t)b * L + l) * nblocks);
    }
    return g;
fail:
    free(g->prev); free(g->prev_n); free(g->zipf_cdf); free(g->zipf_perm); free(g);
    return NULL;
}

void skvw_topk_destroy(skvw_topk *g)
{
    if (!g) return;
    free(g->prev); free(g->prev_n); free(g->zipf_cdf); free(g->zipf_perm); free(g);
}

/* The next step for batch entry b starts cold (used after a request is
 * released and a fresh one published in its place). */
void skvw_topk_reset(skvw_topk *g, int32_t b)
{
    for (int32_t l = 0; l < g->L; ++l) g->prev_n[(size_t)b * g->L + l] = 0;
}

static inline int bm_test(const uint64_t *bm, int64_t t) { return (int)((bm[t >> 6] >> (t & 63)) & 1u); }
static inline void bm_set(uint64_t *bm, int64_t t) { bm[t >> 6] |= 1ULL << (t & 63); }
static inline void bm_clear(uint64_t *bm, int64_t t) { bm[t >> 6] &= ~(1ULL << (t & 63)); }

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* One fresh candidate token in [0, len) from the configured distribution. */
static int64_t draw_fresh(const skvw_topk *g, stream_t *s, int64_t len, const int32_t *perm)
{
    if (g->dist == DIST_RECENCY) {
        if (unit01(s) < g->p_window) {
            int64_t lo = len - g->window < 0 ? 0 : len - g->window;
            return lo + (int64_t)below(s, (uint64_t)(len - lo));
        }
        return (int64_t)below(s, (uint64_t)len);
    }
    if (g->dist == DIST_ZIPF) {
        double u = unit01(s);
        int32_t lo = 0, hi = g->nblocks - 1; /* first rank with cdf > u */
        while (lo < hi) {
            int32_t mid = (lo + hi) / 2;
            if (g->zipf_cdf[mid] > u) hi = mid; else lo = mid + 1;
        }
        int64_t blk = perm[lo];
        return blk * g->block + (int64_t)below(s, (uint64_t)g->block);
    }
    return (int64_t)below(s, (uint64_t)len);
}

/* Generate one unit's row.  Returns 0 on success, -1 if len is too small. */
static int unit_step(skvw_topk *g, int32_t b, int32_t l, int32_t step, int64_t len, int32_t *out, uint64_t *bm,
                     int32_t *tmp)
{
    const int32_t k = g->k, kv = k - g->n_pad;
    if (len < (int64_t)kv || len > g->max_len) return -1;
    int32_t *prev = g->prev + ((size_t)b * g->L + l) * kv;
    int32_t *pn = g->prev_n + (size_t)b * g->L + l;
    const int32_t *perm = g->zipf_perm ? g->zipf_perm + ((size_t)b * g->L + l) * g->nblocks : NULL;
    stream_t s = {skvw_key(g->seed, 0x544F504BULL /* "TOPK" */, (uint64_t)b, (uint64_t)l, (uint64_t)step), 0};
    int32_t n = 0;
    if (*pn == kv) {
        /* keep a uniform random subset of size kv - n_fresh of the previous set
         * (partial Fisher-Yates on a copy), dropping kept tokens that fall
         * outside [0, len) (never happens while len only grows) */
        memcpy(tmp, prev, sizeof(int32_t) * (size_t)kv);
        const int32_t keep = kv - g->n_fresh;
        for (int32_t i = 0; i < keep; ++i) {
            int32_t j = i + (int32_t)below(&s, (uint64_t)(kv - i));
            int32_t t = tmp[i]; tmp[i] = tmp[j]; tmp[j] = t;
        }
        for (int32_t i = 0; i < keep; ++i)
            if (tmp[i] < len) { out[n++] = tmp[i]; bm_set(bm, tmp[i]); }
    }
    /* fresh tokens, distinct from the kept ones and from each other (rejection) */
    int64_t tries = 0;
    while (n < kv) {
        int64_t t = draw_fresh(g, &s, len, perm);
        if (++tries > 64 * (int64_t)kv + 1000000) {
            /* distribution exhausted near its mass: fall back to uniform */
            t = (int64_t)below(&s, (uint64_t)len);
        }
        if (t < 0 || t >= len || bm_test(bm, t)) continue;
        bm_set(bm, t);
        out[n++] = (int32_t)t;
    }
    for (int32_t i = 0; i < n; ++i) bm_clear(bm, out[i]);
    memcpy(prev, out, sizeof(int32_t) * (size_t)kv);
    *pn = kv;
    /* order of the emitted row */
    if (g->order == ORDER_SORTED) {
        qsort(out, (size_t)kv, sizeof(int32_t), cmp_i32);
        if (g->n_pad > 0) {
            /* scatter -1 entries at random positions, keeping the tokens' order:
             * choose which of the k positions are padding */
            memcpy(tmp, out, sizeof(int32_t) * (size_t)kv);
            for (int32_t i = 0; i < k; ++i) out[i] = 0;
            int32_t placed = 0;
            while (placed < g->n_pad) {
                int32_t p = (int32_t)below(&s, (uint64_t)k);
                if (out[p] == 0) { out[p] = 1; ++placed; }
            }
            int32_t j = 0;
            for (int32_t i = 0; i < k; ++i) out[i] = out[i] ? -1 : tmp[j++];
        }
    } else {
        for (int32_t i = kv; i < k; ++i) out[i] = -1;
        for (int32_t i = k - 1; i > 0; --i) {
            int32_t j = (int32_t)below(&s, (uint64_t)i + 1);
            int32_t t = out[i]; out[i] = out[j]; out[j] = t;
        }
    }
    return 0;
}

/* One step for all B x L units: out is [B][L][k]; lens[b] is the current
 * context length of batch entry b.  Returns 0, or -1 on a bad length. */
int32_t skvw_topk_step(skvw_topk *g, int32_t step, const int64_t *lens, int32_t *out, int32_t nthreads)
{
    const int64_t units = (int64_t)g->B * g->L;
    const int64_t bm_words = (g->max_len + 63) / 64;
    int32_t bad = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
    {
        uint64_t *bm = (uint64_t *)calloc((size_t)bm_words, sizeof(uint64_t));
        int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)g->k);
        if (!bm || !tmp) bad = 1;
#pragma omp for schedule(dynamic, 4)
        for (int64_t u = 0; u < units; ++u) {
            if (!bm || !tmp) continue;
            int32_t b = (int32_t)(u / g->L), l = (int32_t)(u % g->L);
            if (unit_step(g, b, l, step, lens[b], out + u * g->k, bm, tmp) != 0) bad = 1;
        }
        free(bm);
        free(tmp);
    }
    return bad ? -1 : 0;
}
