/*
 * csm_oracle.c -- plain fp64 CPU oracle for online KV-cache clustering.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code,
 * header, table or helper with the CUDA path, and the product never calls it.
 *
 * Sources (web pages on arXiv 2506.11418; shorthand used below):
 *   [Chelsea]    "Chelsea: Efficient Long-Context LLM Inference via KV Cache
 *                Clustering" (xllm-io paper review).
 *   [CentroidKV] "CentroidKV: Efficient Long-Context LLM Inference via KV Cache
 *                Clustering" (gist.science explainer), section 技术摘要.
 *
 * What is computed, step by step, in the pages' order:
 *   Chunked Soft Matching, one round on one (sequence, KV head) cache
 *     [Chelsea §三 分块软匹配算法, steps 1-4; CentroidKV 核心组件 / 分块软匹配 (CSM), 聚合]
 *     1. keep the first n1 (attention sinks) and last n2 (recent) tokens;
 *        split the middle into floor((s-n1-n2)/c) full chunks of c tokens,
 *        starting at row n1; a shorter remainder is left as it is;
 *     2. alternating partition inside a chunk: A = even offsets, B = odd
 *        offsets (Theorem 6.1's A0 = {1,3,...} in 1-based numbering);
 *     3. cosine similarity of the current (centroid) keys, cos = 0 when
 *        either norm is 0;
 *     4. every A token takes its most similar B token (lowest B on ties);
 *     5. the candidate edges are sorted by similarity and only the first m
 *        are merged (ties: lowest A index);
 *     6. each B token with incoming edges becomes the degree-weighted mean of
 *        itself and its A tokens, k = sum n_i k_i / sum n_i (same for v),
 *        n = sum n_i, all from pre-round values; it keeps the B token's slot;
 *     7. merged-away A rows are removed and the rest keeps its order.
 *   Degree-aware attention [Chelsea §三 核心公式]:
 *        O = softmax(q K^T / sqrt(d) + log N) V, computed literally with the
 *        log-degree bias and a max shift.
 *   Prefill attention [Chelsea §三 算法流程, Algorithm 1]: the prompt's causal
 *        softmax attention with every degree 1, before the first round.
 *
 * Arithmetic is fp64 throughout; degrees and lengths are int32.
 * Parallelism: OpenMP over independent (sequence, KV head) units or over an
 * explicit list of independent chunks, nothing else.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- step 2: the partition the oracle uses (exported for the Theorem 6.1 test) */
void oracle_partition(int32_t c, int32_t* a_offsets, int32_t* b_offsets)
{
    for (int32_t i = 0; i < c / 2; ++i) {
        a_offsets[i] = 2 * i;     /* even offsets -> A */
        b_offsets[i] = 2 * i + 1; /* odd offsets  -> B */
    }
}

/* ---- step 3 */
static double cosine(const double* x, const double* y, int32_t d)
{
    double dot = 0.0, nx = 0.0, ny = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        dot += x[i] * y[i];
        nx += x[i] * x[i];
        ny += y[i] * y[i];
    }
    if (nx == 0.0 || ny == 0.0) return 0.0;
    return dot / (sqrt(nx) * sqrt(ny));
}

typedef struct {
    double sim;
    int32_t a;
} edge_t;

/* step 5 ordering: larger similarity first, then lower A index */
static int edge_cmp(const void* p, const void* q)
{
    const edge_t* x = (const edge_t*)p;
    const edge_t* y = (const edge_t*)q;
    if (x->sim > y->sim) return -1;
    if (x->sim < y->sim) return 1;
    return (x->a < y->a) ? -1 : (x->a > y->a ? 1 : 0);
}

/*
 * One chunk of c rows (pre-round values Kc, Vc [c][d], Nc [c]).
 * Writes the c - m surviving rows to Ko, Vo [c-m][d], No [c-m] in original
 * order. match[a] = B index (0..c/2-1) that A token a merged into, or -1.
 * best_sim[a] = cos(a, best B); margin[a] = best minus second-best cos;
 * *cut_margin = (m-th largest edge sim) - ((m+1)-th), +inf when undefined.
 * forced (may be NULL): decisions to apply instead of steps 4-5 (the replay
 * used when the GPU took a near-tie the other way); similarities are still
 * reported. origin/merged (may be NULL): per output row, the chunk offset it
 * comes from and whether it is a merged centroid (bookkeeping for tests).
 * Returns 0, or -1 if forced does not hold exactly m edges or points outside B.
 */
int oracle_csm_chunk(const double* Kc, const double* Vc, const int32_t* Nc,
                     int32_t c, int32_t d, int32_t m, const int32_t* forced,
                     double* Ko, double* Vo, int32_t* No, int32_t* match,
                     double* best_sim, double* margin, double* cut_margin,
                     int32_t* origin, uint8_t* merged)
{
    const int32_t h = c / 2;
    int32_t* best = (int32_t*)malloc(sizeof(int32_t) * h);
    edge_t* edges = (edge_t*)malloc(sizeof(edge_t) * h);
    int rc = 0;

    /* steps 3-4: A row a sits at offset 2a, B row b at offset 2b+1 */
    for (int32_t a = 0; a < h; ++a) {
        const double* ka = Kc + (size_t)(2 * a) * d;
        double top = -INFINITY, second = -INFINITY;
        int32_t arg = 0;
        for (int32_t b = 0; b < h; ++b) {
            double s = cosine(ka, Kc + (size_t)(2 * b + 1) * d, d);
            if (s > top) { /* strict: an equal later b never replaces -> lowest b */
                second = top;
                top = s;
                arg = b;
            } else if (s > second) {
                second = s;
            }
        }
        best[a] = arg;
        best_sim[a] = top;
        margin[a] = (h > 1) ? (top - second) : INFINITY;
        edges[a].sim = top;
        edges[a].a = a;
    }

    /* step 5 */
    qsort(edges, (size_t)h, sizeof(edge_t), edge_cmp);
    *cut_margin = (m > 0 && m < h) ? (edges[m - 1].sim - edges[m].sim) : INFINITY;
    for (int32_t a = 0; a < h; ++a) match[a] = -1;
    if (forced) {
        int32_t cnt = 0;
        for (int32_t a = 0; a < h; ++a) {
            if (forced[a] >= 0) {
                if (forced[a] >= h) rc = -1;
                match[a] = forced[a];
                ++cnt;
            }
        }
        if (cnt != m) rc = -1;
    } else {
        for (int32_t i = 0; i < m; ++i) match[edges[i].a] = best[edges[i].a];
    }

    /* steps 6-7: walk the chunk in order, drop merged A rows, merge into B */
    int32_t out = 0;
    for (int32_t o = 0; o < c && rc == 0; ++o) {
        if ((o & 1) == 0) {
            if (match[o / 2] >= 0) continue; /* merged away */
            memcpy(Ko + (size_t)out * d, Kc + (size_t)o * d, sizeof(double) * d);
            memcpy(Vo + (size_t)out * d, Vc + (size_t)o * d, sizeof(double) * d);
            No[out] = Nc[o];
            if (origin) origin[out] = o;
            if (merged) merged[out] = 0;
            ++out;
            continue;
        }
        const int32_t b = o / 2;
        int incoming = 0;
        for (int32_t a = 0; a < h; ++a) incoming |= (match[a] == b);
        if (origin) origin[out] = o;
        if (merged) merged[out] = (uint8_t)(incoming != 0);
        if (!incoming) { /* a singleton keeps its exact values */
            memcpy(Ko + (size_t)out * d, Kc + (size_t)o * d, sizeof(double) * d);
            memcpy(Vo + (size_t)out * d, Vc + (size_t)o * d, sizeof(double) * d);
            No[out] = Nc[o];
            ++out;
            continue;
        }
        double* kk = Ko + (size_t)out * d;
        double* vv = Vo + (size_t)out * d;
        int64_t nsum = Nc[o];
        for (int32_t i = 0; i < d; ++i) {
            kk[i] = (double)Nc[o] * Kc[(size_t)o * d + i];
            vv[i] = (double)Nc[o] * Vc[(size_t)o * d + i];
        }
        for (int32_t a = 0; a < h; ++a) {
            if (match[a] != b) continue;
            const int32_t oa = 2 * a;
            nsum += Nc[oa];
            for (int32_t i = 0; i < d; ++i) {
                kk[i] += (double)Nc[oa] * Kc[(size_t)oa * d + i];
                vv[i] += (double)Nc[oa] * Vc[(size_t)oa * d + i];
            }
        }
        for (int32_t i = 0; i < d; ++i) {
            kk[i] /= (double)nsum;
            vv[i] /= (double)nsum;
        }
        No[out] = (int32_t)nsum;
        ++out;
    }
    free(best);
    free(edges);
    return rc;
}

/* number of full chunks of a cache of length s (step 1) */
int32_t oracle_num_chunks(int32_t s, int32_t n1, int32_t n2, int32_t c)
{
    int32_t mid = s - n1 - n2;
    return mid > 0 ? mid / c : 0;
}

/*
 * One CSM round on one (sequence, KV head) cache, in place.
 * K, V: [cap][d]; N: [cap]; *len: current length s, updated.
 * Per-chunk records (may be NULL) are indexed [j][a] with row stride h=c/2
 * for up to maxch chunks.
 * limit > 0 processes only the first (oldest) min(limit, chunks) full chunks;
 * every later row, unprocessed chunks included, moves down unchanged
 * (budget-exact compression; the pages' Algorithm 1 compresses every chunk).
 */
static int csm_unit(double* K, double* V, int32_t* N, int32_t* len, int32_t cap,
                    int32_t d, int32_t n1, int32_t n2, int32_t c, int32_t m,
                    const int32_t* forced, int32_t* match, double* sim,
                    double* margin, double* cut, int32_t maxch,
                    int32_t* origin, uint8_t* merged, int32_t limit)
{
    /* origin/merged (may be NULL): [cap], per output row the pre-round row it
     * comes from and whether it is a merged centroid; identity when nothing merges */
    if (origin)
        for (int32_t t = 0; t < *len; ++t) origin[t] = t;
    if (merged)
        for (int32_t t = 0; t < *len; ++t) merged[t] = 0;
    const int32_t s = *len;
    const int32_t h = c / 2;
    const int32_t ch_all = oracle_num_chunks(s, n1, n2, c);
    if (ch_all > maxch) return -2;
    const int32_t ch = (limit > 0 && limit < ch_all) ? limit : ch_all;
    if (ch == 0 || m == 0) return 0;

    /* pre-round copy of everything from the first chunk on */
    const int32_t start = n1;
    const int32_t count = s - n1;
    double* K0 = (double*)malloc(sizeof(double) * (size_t)count * d);
    double* V0 = (double*)malloc(sizeof(double) * (size_t)count * d);
    int32_t* N0 = (int32_t*)malloc(sizeof(int32_t) * (size_t)count);
    memcpy(K0, K + (size_t)start * d, sizeof(double) * (size_t)count * d);
    memcpy(V0, V + (size_t)start * d, sizeof(double) * (size_t)count * d);
    memcpy(N0, N + start, sizeof(int32_t) * (size_t)count);

    int32_t* mt = (int32_t*)malloc(sizeof(int32_t) * h);
    double* bs = (double*)malloc(sizeof(double) * h);
    double* mg = (double*)malloc(sizeof(double) * h);
    int32_t* og = (int32_t*)malloc(sizeof(int32_t) * c);
    uint8_t* mf = (uint8_t*)malloc((size_t)c);
    int rc = 0;
    int32_t w = start; /* next output row */
    for (int32_t j = 0; j < ch && rc == 0; ++j) {
        double cm;
        const size_t base = (size_t)j * c;
        rc = oracle_csm_chunk(K0 + base * d, V0 + base * d, N0 + base, c, d, m,
                              forced ? forced + (size_t)j * h : NULL,
                              K + (size_t)w * d, V + (size_t)w * d, N + w, mt, bs, mg, &cm,
                              og, mf);
        for (int32_t o = 0; o < c - m; ++o) {
            if (origin) origin[w + o] = start + j * c + og[o];
            if (merged) merged[w + o] = mf[o];
        }
        if (match) memcpy(match + (size_t)j * h, mt, sizeof(int32_t) * h);
        if (sim) memcpy(sim + (size_t)j * h, bs, sizeof(double) * h);
        if (margin) memcpy(margin + (size_t)j * h, mg, sizeof(double) * h);
        if (cut) cut[j] = cm;
        w += c - m;
    }
    if (rc == 0) {
        /* unprocessed chunks, remainder and recent window follow in order */
        const int32_t tail0 = ch * c; /* index into the pre-round copy */
        const int32_t tail = count - tail0;
        memcpy(K + (size_t)w * d, K0 + (size_t)tail0 * d, sizeof(double) * (size_t)tail * d);
        memcpy(V + (size_t)w * d, V0 + (size_t)tail0 * d, sizeof(double) * (size_t)tail * d);
        memcpy(N + w, N0 + tail0, sizeof(int32_t) * (size_t)tail);
        for (int32_t t = 0; t < tail; ++t) {
            if (origin) origin[w + t] = start + tail0 + t;
            if (merged) merged[w + t] = 0;
        }
        *len = s - ch * m;
    }
    free(K0);
    free(V0);
    free(N0);
    free(mt);
    free(bs);
    free(mg);
    free(og);
    free(mf);
    (void)cap;
    return rc;
}

/*
 * One CSM round over BH = batch * h_kv independent caches.
 * K, V: [BH][cap][d] fp64; N: [BH][cap]; len: [BH]. skip[u] != 0 leaves unit
 * u untouched (outlier head, or a sequence not compressed this round).
 * limits[u] > 0 (limits may be NULL) caps unit u at its first limits[u] chunks.
 * Records: match/sim/margin [BH][maxch][c/2], cut [BH][maxch], origin and
 * merged [BH][cap], all optional; forced [BH][maxch][c/2] optional. Returns 0 on success, else the first
 * failing unit's code (-1 bad forced decisions, -2 maxch too small).
 */
int oracle_csm_round(double* K, double* V, int32_t* N, int32_t* len,
                     int32_t BH, int32_t cap, int32_t d, int32_t n1, int32_t n2,
                     int32_t c, int32_t m, const uint8_t* skip,
                     const int32_t* forced, int32_t* match, double* sim,
                     double* margin, double* cut, int32_t maxch,
                     int32_t* origin, uint8_t* merged, const int32_t* limits, int32_t nthreads)
{
    int rc_all = 0;
    const size_t rec = (size_t)maxch * (c / 2);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int32_t u = 0; u < BH; ++u) {
        if (skip && skip[u]) { /* untouched: every row stays where it is */
            for (int32_t t = 0; t < len[u]; ++t) {
                if (origin) origin[(size_t)u * cap + t] = t;
                if (merged) merged[(size_t)u * cap + t] = 0;
            }
            continue;
        }
        int rc = csm_unit(K + (size_t)u * cap * d, V + (size_t)u * cap * d,
                          N + (size_t)u * cap, len + u, cap, d, n1, n2, c, m,
                          forced ? forced + u * rec : NULL,
                          match ? match + u * rec : NULL,
                          sim ? sim + u * rec : NULL,
                          margin ? margin + u * rec : NULL,
                          cut ? cut + (size_t)u * maxch : NULL, maxch,
                          origin ? origin + (size_t)u * cap : NULL,
                          merged ? merged + (size_t)u * cap : NULL, limits ? limits[u] : 0);
        if (rc != 0) {
#pragma omp critical
            if (rc_all == 0) rc_all = rc;
        }
    }
    return rc_all;
}

/*
 * A list of independent chunks (pre-round values), as used for sampled checks
 * at full size. Kc, Vc: [n][c][d]; Nc: [n][c]. Outputs: Ko, Vo [n][c-m][d],
 * No [n][c-m]; match/sim/margin [n][c/2]; cut [n]; origin/merged [n][c-m].
 * forced optional [n][c/2].
 */
int oracle_csm_chunks(const double* Kc, const double* Vc, const int32_t* Nc,
                      int32_t n, int32_t c, int32_t d, int32_t m,
                      const int32_t* forced, double* Ko, double* Vo, int32_t* No,
                      int32_t* match, double* sim, double* margin, double* cut,
                      int32_t* origin, uint8_t* merged, int32_t nthreads)
{
    int rc_all = 0;
    const int32_t h = c / 2;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
    for (int32_t i = 0; i < n; ++i) {
        int rc = oracle_csm_chunk(Kc + (size_t)i * c * d, Vc + (size_t)i * c * d,
                                  Nc + (size_t)i * c, c, d, m,
                                  forced ? forced + (size_t)i * h : NULL,
                                  Ko + (size_t)i * (c - m) * d, Vo + (size_t)i * (c - m) * d,
                                  No + (size_t)i * (c - m), match + (size_t)i * h,
                                  sim + (size_t)i * h, margin + (size_t)i * h, cut + i,
                                  origin + (size_t)i * (c - m), merged + (size_t)i * (c - m));
        if (rc != 0) {
#pragma omp critical
            if (rc_all == 0) rc_all = rc;
        }
    }
    return rc_all;
}

/*
 * Decode append [Chelsea §三 算法流程, Algorithm 1 decode update]:
 * K=[K,k], V=[V,v], N=[N,1], s=s+1, for every unit u with len[u] < cap.
 * k_new, v_new: [BH][d]. Returns the number of units that were full.
 */
int32_t oracle_append(double* K, double* V, int32_t* N, int32_t* len, int32_t BH,
                      int32_t cap, int32_t d, const double* k_new, const double* v_new,
                      const uint8_t* skip)
{
    int32_t full = 0;
    for (int32_t u = 0; u < BH; ++u) {
        if (skip && skip[u]) continue;
        const int32_t s = len[u];
        if (s >= cap) { ++full; continue; }
        memcpy(K + ((size_t)u * cap + s) * d, k_new + (size_t)u * d, sizeof(double) * d);
        memcpy(V + ((size_t)u * cap + s) * d, v_new + (size_t)u * d, sizeof(double) * d);
        N[(size_t)u * cap + s] = 1;
        len[u] = s + 1;
    }
    return full;
}

/*
 * Degree-aware decode attention [Chelsea §三 核心公式; CentroidKV 聚合]:
 *   o_h = softmax(q_h K^T * scale + log N) V over the first len rows of the
 *   KV head that serves q head h. Query head h of sequence b reads KV head
 *   floor(h / G), G = Hq / Hkv (contiguous groups).
 * q: [B][Hq][d]; K, V: [B][Hkv][cap][d]; N: [B][Hkv][cap]; len: [B][Hkv];
 * out: [B][Hq][d]. A head with len 0 gets a zero output.
 */
void oracle_decode_attn_logn(const double* q, const double* K, const double* V,
                             const int32_t* N, const int32_t* len, int32_t B,
                             int32_t Hkv, int32_t Hq, int32_t cap, int32_t d,
                             double scale, double* out, int32_t nthreads)
{
    const int32_t G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int32_t bh = 0; bh < B * Hq; ++bh) {
        const int32_t b = bh / Hq, h = bh % Hq, kv = h / G;
        const size_t u = (size_t)b * Hkv + kv;
        const double* qh = q + (size_t)bh * d;
        const double* Ku = K + u * cap * d;
        const double* Vu = V + u * cap * d;
        const int32_t* Nu = N + u * cap;
        const int32_t s = len[u];
        double* o = out + (size_t)bh * d;
        for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
        if (s <= 0) continue;
        double* logit = (double*)malloc(sizeof(double) * (size_t)s);
        double mx = -INFINITY;
        for (int32_t t = 0; t < s; ++t) {
            double dot = 0.0;
            for (int32_t i = 0; i < d; ++i) dot += qh[i] * Ku[(size_t)t * d + i];
            logit[t] = dot * scale + log((double)Nu[t]);
            if (logit[t] > mx) mx = logit[t];
        }
        double den = 0.0;
        for (int32_t t = 0; t < s; ++t) {
            const double w = exp(logit[t] - mx);
            den += w;
            for (int32_t i = 0; i < d; ++i) o[i] += w * Vu[(size_t)t * d + i];
        }
        for (int32_t i = 0; i < d; ++i) o[i] /= den;
        free(logit);
    }
}

/*
 * Prefill attention [Chelsea §三 算法流程, Algorithm 1, 预填充 / 输出 O = FlashAttn(Q,K,V)]:
 *   the prompt's own causal softmax attention before any compression, every
 *   degree still 1 (N = [1]*n, so the log-degree term is 0 and left out):
 *   o_{h,i} = softmax_{t <= i}(q_{h,i} . k_t * scale) V over rows 0..i of the
 *   KV head that serves q head h (contiguous groups, G = Hq / Hkv).
 * q: [B][Hq][n][d]; K, V: [B][Hkv][cap][d] (rows 0..n-1 hold the prompt);
 * rows: nrows query positions to evaluate (NULL: all n, nrows = n);
 * out: [B][Hq][nrows][d].
 */
void oracle_prefill_attn(const double* q, const double* K, const double* V, int32_t B,
                         int32_t Hkv, int32_t Hq, int32_t n, int32_t cap, int32_t d,
                         double scale, const int32_t* rows, int32_t nrows, double* out,
                         int32_t nthreads)
{
    const int32_t G = Hq / Hkv;
    const long long total = (long long)B * Hq * nrows;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads > 0 ? nthreads : 1)
    for (long long job = 0; job < total; ++job) {
        const int32_t r = (int32_t)(job % nrows);
        const int32_t bh = (int32_t)(job / nrows);
        const int32_t b = bh / Hq, h = bh % Hq, kv = h / G;
        const int32_t i = rows ? rows[r] : r;
        const double* qi = q + ((size_t)bh * n + i) * d;
        const double* Ku = K + ((size_t)b * Hkv + kv) * cap * d;
        const double* Vu = V + ((size_t)b * Hkv + kv) * cap * d;
        double* o = out + ((size_t)bh * nrows + r) * d;
        for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
        double* logit = (double*)malloc(sizeof(double) * (size_t)(i + 1));
        double mx = -INFINITY;
        for (int32_t t = 0; t <= i; ++t) {
            double dot = 0.0;
            for (int32_t e = 0; e < d; ++e) dot += qi[e] * Ku[(size_t)t * d + e];
            logit[t] = dot * scale;
            if (logit[t] > mx) mx = logit[t];
        }
        double den = 0.0;
        for (int32_t t = 0; t <= i; ++t) {
            const double w = exp(logit[t] - mx);
            den += w;
            for (int32_t e = 0; e < d; ++e) o[e] += w * Vu[(size_t)t * d + e];
        }
        for (int32_t e = 0; e < d; ++e) o[e] /= den;
        free(logit);
    }
}

int32_t oracle_max_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}
