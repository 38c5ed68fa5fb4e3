/*
 * MSA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of MiniMax Sparse Attention (MSA) as the page
 * "MiniMax M3 算力省 20 倍" defines it (section 二, Index Branch and Main Branch; section 三 item 4,
 * the forced local block), with the deployment budget B = 128, k = 16 of the same section (also
 * "MiniMax M3.1 Flash 开放权重与部署要点", the paragraph on MSA).  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this file; the product path never does.
 *
 * Every sum is accumulated in fp64.  bf16 inputs are widened exactly (bf16 is the top half of an
 * IEEE binary32).  No blocking, fusion or reordering beyond the definition:
 *
 *  Index branch, for GQA group g and query position i, with b_i = floor(i / B):
 *    s[j]   = sum_d q_idx[i,g,d] * k_idx[j,d]            (raw dot product, no exp, no scale)
 *    S[b]   = max over the B tokens j of block b of s[j]  (max-pooling), for every b < b_i
 *    sel    = {b_i} U first min(k-1, b_i) candidates ranked by (S desc, b asc)
 *             (the local block is always kept and occupies one of the k slots)
 *    stored ascending, padded with -1 to k entries.
 *  Main branch, for query head h of group g = h / (Hq/G):
 *    T(i)   = union over b in sel of [b*B, min(b*B+B, i+1))  (causal inside the local block)
 *    z_j    = scale * sum_d q[i,h,d] * k[j,g,d]
 *    m      = max_j z_j,  l = sum_j exp(z_j - m)
 *    o      = sum_j exp(z_j - m) v[j,g,:] / l,   lse = m + ln(l)
 *  Decode: the same rules for one query per sequence at position n-1 (n = context length, the
 *  new token already in the cache), keys/values read through the page table.
 *  Exported block scores (section 三 item 1, the indexer's KL alignment needs them): S[b] for
 *  every b < b_i, +inf at b_i, -inf after it.
 *
 * Readings where the pages are silent: ties rank the lower block id first; the local block is
 * never scored (every other candidate block lies wholly in the causal past); the score is the raw
 * dot product; the natural log is used for lse; the softmax scale is a parameter.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    double score;
    int32_t block;
} cand_t;

/* (score desc, block asc) */
static int cand_cmp(const void* a, const void* b) {
    const cand_t* x = (const cand_t*)a;
    const cand_t* y = (const cand_t*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->block < y->block) ? -1 : (x->block > y->block);
}

static int int_cmp(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Key row j of the index keys, contiguous ([L][di]) or paged ([P][B][di] through page_row). */
static const uint16_t* idx_key_row(const uint16_t* base, const int32_t* page_row, int B, int di,
                                   int64_t j) {
    if (!page_row) return base + (size_t)j * di;
    int64_t page = page_row[j / B];
    return base + ((size_t)page * B + (size_t)(j % B)) * di;
}

/*
 * Select the blocks of one (query, group).  q: di bf16 values; keys through idx_key_row.
 * Writes k ids (ascending, -1 padded) to sel and, if score != NULL, the pooled score of each
 * selected block (the local block gets +inf, padding -inf).
 */
static void select_one(const uint16_t* q, const uint16_t* kbase, const int32_t* page_row, int di,
                       int B, int k, int64_t i, cand_t* cand, int32_t* sel, double* score) {
    const int32_t bi = (int32_t)(i / B);
    for (int32_t b = 0; b < bi; ++b) {
        double best = -INFINITY;
        for (int t = 0; t < B; ++t) {
            const uint16_t* kr = idx_key_row(kbase, page_row, B, di, (int64_t)b * B + t);
            double s = 0.0;
            for (int d = 0; d < di; ++d) s += bf(q[d]) * bf(kr[d]);
            if (s > best) best = s;
        }
        cand[b].score = best;
        cand[b].block = b;
    }
    qsort(cand, (size_t)bi, sizeof(cand_t), cand_cmp);
    int take = (k - 1 < bi) ? k - 1 : bi;
    int n = 0;
    for (int r = 0; r < take; ++r) sel[n++] = cand[r].block;
    sel[n++] = bi;
    qsort(sel, (size_t)n, sizeof(int32_t), int_cmp);
    for (int r = n; r < k; ++r) sel[r] = -1;
    if (score) {
        for (int r = 0; r < k; ++r) {
            if (sel[r] < 0) score[r] = -INFINITY;
            else if (sel[r] == bi) score[r] = INFINITY;
            else {
                for (int c = 0; c < take; ++c)
                    if (cand[c].block == sel[r]) score[r] = cand[c].score;
            }
        }
    }
}

/*
 * Prefill index branch.  q_idx [L][G][di], k_idx [L][di] (bf16 bits).  For each of the nrows
 * query positions rows[r] and each group g: sel[(g*nrows + r)*k + .] and score likewise.
 */
void oracle_select_prefill(const uint16_t* q_idx, const uint16_t* k_idx, int64_t L, int G, int di,
                           int B, int k, const int64_t* rows, int64_t nrows, int32_t* sel,
                           double* score) {
    (void)L;
    #pragma omp parallel
    {
        cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(L / B + 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t rg = 0; rg < nrows * G; ++rg) {
            int64_t r = rg / G;
            int g = (int)(rg % G);
            int64_t i = rows[r];
            select_one(q_idx + ((size_t)i * G + g) * di, k_idx, NULL, di, B, k, i, cand,
                       sel + ((size_t)g * nrows + r) * k,
                       score ? score + ((size_t)g * nrows + r) * k : NULL);
        }
        free(cand);
    }
}

/*
 * Every block's pooled index score for one (query, group), as exported for the indexer's KL
 * alignment ("MiniMax M3 算力省 20 倍", section 三 item 1, which fits the indexer's block scores to
 * the main branch's attention): out[c] = max over the B tokens j of block c of the raw dot
 * product q . k_idx[j] for c < b_i; +inf at c = b_i (the forced local block, never scored);
 * -inf for b_i < c < nb (not causal).
 */
static void block_scores_one(const uint16_t* q, const uint16_t* kbase, const int32_t* page_row,
                             int di, int B, int64_t i, int64_t nb, double* out) {
    const int64_t bi = i / B;
    for (int64_t c = 0; c < nb; ++c) {
        if (c == bi) { out[c] = INFINITY; continue; }
        if (c > bi) { out[c] = -INFINITY; continue; }
        double best = -INFINITY;
        for (int t = 0; t < B; ++t) {
            const uint16_t* kr = idx_key_row(kbase, page_row, B, di, c * B + t);
            double s = 0.0;
            for (int d = 0; d < di; ++d) s += bf(q[d]) * bf(kr[d]);
            if (s > best) best = s;
        }
        out[c] = best;
    }
}

/* Prefill: out [G][nrows][nb] for the query positions rows[r], nb = ceil(L / B). */
void oracle_block_scores_prefill(const uint16_t* q_idx, const uint16_t* k_idx, int64_t L, int G,
                                 int di, int B, const int64_t* rows, int64_t nrows, double* out) {
    const int64_t nb = (L + B - 1) / B;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rg = 0; rg < nrows * G; ++rg) {
        int64_t r = rg / G;
        int g = (int)(rg % G);
        block_scores_one(q_idx + ((size_t)rows[r] * G + g) * di, k_idx, NULL, di, B, rows[r], nb,
                         out + ((size_t)g * nrows + r) * nb);
    }
}

/* Decode: out [G][batch][max_pages], keys through the page table; query at seq_lens[s]-1. */
void oracle_block_scores_decode(const uint16_t* q_idx, const uint16_t* k_idx_pool,
                                const int32_t* page_table, int64_t max_pages,
                                const int32_t* seq_lens, int64_t batch, int G, int di, int B,
                                double* out) {
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t sg = 0; sg < batch * G; ++sg) {
        int64_t s = sg / G;
        int g = (int)(sg % G);
        block_scores_one(q_idx + ((size_t)s * G + g) * di, k_idx_pool,
                         page_table + (size_t)s * max_pages, di, B, (int64_t)seq_lens[s] - 1,
                         max_pages, out + ((size_t)g * batch + s) * max_pages);
    }
}

/*
 * Main branch for one (query, head) over an explicit token set: q holds d values, krows/vrows
 * point at the ntok key/value rows; writes o[d] and lse.
 */
static void attend_one(const uint16_t* q, const uint16_t* const* krows,
                       const uint16_t* const* vrows, int64_t ntok, int d, double scale,
                       double* z, double* o, double* lse) {
    double m = -INFINITY;
    for (int64_t t = 0; t < ntok; ++t) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += bf(q[c]) * bf(krows[t][c]);
        z[t] = scale * s;
        if (z[t] > m) m = z[t];
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < ntok; ++t) {
        double p = exp(z[t] - m);
        l += p;
        for (int c = 0; c < d; ++c) o[c] += p * bf(vrows[t][c]);
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
}

/*
 * Prefill main branch.  q [L][Hq][d] (or, when q_compact is set, [nrows][Hq][d] holding only
 * the listed rows), k/v [L][G][d].  For the nrows positions rows[r] and every head h, with
 * sel [G][nrows][k] the selection of those positions (the layout the index branch above writes
 * for the same rows): o[(r*Hq + h)*d + .] and lse[h*nrows + r].
 */
void oracle_attn_prefill(const uint16_t* q, const uint16_t* kk, const uint16_t* vv, int64_t L,
                         int Hq, int G, int d, int B, int k, double scale, const int32_t* sel,
                         const int64_t* rows, int64_t nrows, double* o, double* lse,
                         int q_compact) {
    const int hpg = Hq / G;
    const int64_t cap = (int64_t)k * B;
    (void)L;
    #pragma omp parallel
    {
        const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
        double* z = (double*)malloc(sizeof(double) * (size_t)cap);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t rh = 0; rh < nrows * Hq; ++rh) {
            int64_t r = rh / Hq;
            int h = (int)(rh % Hq);
            int g = h / hpg;
            int64_t i = rows[r];
            const int32_t* s = sel + ((size_t)g * nrows + r) * k;
            int64_t n = 0;
            for (int slot = 0; slot < k; ++slot) {
                if (s[slot] < 0) continue;
                int64_t lo = (int64_t)s[slot] * B, hi = lo + B;
                if (hi > i + 1) hi = i + 1;
                for (int64_t j = lo; j < hi; ++j) {
                    kr[n] = kk + ((size_t)j * G + g) * d;
                    vr[n] = vv + ((size_t)j * G + g) * d;
                    ++n;
                }
            }
            const int64_t qi = q_compact ? r : i;  /* compact q holds only the listed rows */
            attend_one(q + ((size_t)qi * Hq + h) * d, kr, vr, n, d, scale, z,
                       o + ((size_t)r * Hq + h) * d, lse + (size_t)h * nrows + r);
        }
        free(kr);
        free(vr);
        free(z);
    }
}

/*
 * Decode index branch.  q_idx [batch][G][di]; k_idx_pool [P][B][di]; page_table [batch][max_pages];
 * seq_lens [batch].  sel [G][batch][k], score likewise.
 */
void oracle_select_decode(const uint16_t* q_idx, const uint16_t* k_idx_pool,
                          const int32_t* page_table, int64_t max_pages, const int32_t* seq_lens,
                          int64_t batch, int G, int di, int B, int k, int32_t* sel, double* score) {
    #pragma omp parallel
    {
        cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(max_pages + 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t sg = 0; sg < batch * G; ++sg) {
            int64_t s = sg / G;
            int g = (int)(sg % G);
            int64_t i = (int64_t)seq_lens[s] - 1;
            select_one(q_idx + ((size_t)s * G + g) * di, k_idx_pool,
                       page_table + (size_t)s * max_pages, di, B, k, i, cand,
                       sel + ((size_t)g * batch + s) * k,
                       score ? score + ((size_t)g * batch + s) * k : NULL);
        }
        free(cand);
    }
}

/*
 * Decode main branch.  q [batch][Hq][d]; k_pool/v_pool [P][G][B][d]; sel [G][batch][k].
 * o [batch][Hq][d], lse [Hq][batch].
 */
void oracle_attn_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                        const int32_t* page_table, int64_t max_pages, const int32_t* seq_lens,
                        int64_t batch, int Hq, int G, int d, int B, int k, double scale,
                        const int32_t* sel, double* o, double* lse) {
    const int hpg = Hq / G;
    const int64_t cap = (int64_t)k * B;
    #pragma omp parallel
    {
        const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
        double* z = (double*)malloc(sizeof(double) * (size_t)cap);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t sh = 0; sh < batch * Hq; ++sh) {
            int64_t s = sh / Hq;
            int h = (int)(sh % Hq);
            int g = h / hpg;
            int64_t i = (int64_t)seq_lens[s] - 1;
            const int32_t* sl = sel + ((size_t)g * batch + s) * k;
            const int32_t* pt = page_table + (size_t)s * max_pages;
            int64_t n = 0;
            for (int slot = 0; slot < k; ++slot) {
                if (sl[slot] < 0) continue;
                int64_t lo = (int64_t)sl[slot] * B, hi = lo + B;
                if (hi > i + 1) hi = i + 1;
                for (int64_t j = lo; j < hi; ++j) {
                    size_t page = (size_t)pt[j / B];
                    size_t off = ((page * G + g) * B + (size_t)(j % B)) * d;
                    kr[n] = k_pool + off;
                    vr[n] = v_pool + off;
                    ++n;
                }
            }
            attend_one(q + ((size_t)s * Hq + h) * d, kr, vr, n, d, scale, z,
                       o + ((size_t)s * Hq + h) * d, lse + (size_t)h * batch + s);
        }
        free(kr);
        free(vr);
        free(z);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
