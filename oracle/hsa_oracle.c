/*
 * hsa_oracle.c -- plain, slow CPU oracle for hybrid compressed/sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Every value is read exactly (bf16 and fp32 widen exactly to double) and all
 * arithmetic is done in double precision, in the order the method states, with
 * no blocking, fusion or reordering.  OpenMP only distributes independent
 * output rows over host threads; it does not change any arithmetic.
 *
 * Sources (web pages on the DeepSeek-V4 technical report; cited by title and
 * section):
 *   [QbitAI]  "DeepSeek V4报告太详尽了！484天换代之路全公开" (QbitAI news
 *             article), section 混合注意力机制 ("hybrid attention").
 *   [Blog]    "DeepSeek V4是怎麼訓練出來的？58頁論文深入解讀", section
 *             "CSA + HCA：讀一本800頁的書，先翻目錄再精讀".
 *   [Essay]   yage.ai essay "deepseek-v4-agentic-workload", the three-layer
 *             description (HCA / CSA top-k 512 and 1024 / 128-token window).
 *   [Wiki]    "DeepSeek-V4 Preview — 开源模型旗舰", vision note (4x CSA
 *             compression: 324 -> 81 entries).
 *
 * Readings fixed where the pages leave a step open (the plainest reading the
 * pages support):
 *   - a compressed entry is a fixed weighted sum of its block's m tokens,
 *     weights w[0..m-1] shared by all blocks and channels, same for K and V,
 *     blocks do not overlap (the pages' learned compressor needs weights);
 *   - entry j covers tokens j*m .. j*m+m-1 and is visible to a query at
 *     position p iff (j+1)*m-1 <= p, i.e. E(p) = floor((p+1)/m) entries
 *     (strict causality of compressed attention, [QbitAI] sliding-window
 *     paragraph);
 *   - the indexer score is the int32 dot product of one int8 vector per query
 *     and one per entry; top-k orders by (score desc, index asc) and keeps
 *     min(k, E(p)) entries, reported in ascending index order, padded with -1;
 *   - the attended set is the multiset {selected entries} + {raw tokens
 *     max(0,p-W+1) .. p}, with one softmax over it and logit scale 1/sqrt(d)
 *     (supplied by the caller); an empty set gives output 0 and lse = -inf.
 *
 * Parity pins for each function live in the CPU test-suite; see the function
 * comments for what pins them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

enum {
    ORC_OK = 0,
    ORC_ERR_RANGE = -1,    /* a block/entry/token lies outside its buffer */
    ORC_ERR_OVERFLOW = -2, /* an indexer score does not fit in int32 */
    ORC_ERR_INDEX = -3,    /* a selected index is not a visible entry */
    ORC_ERR_ARG = -4,      /* bad size or dtype */
    ORC_ERR_NOMEM = -5
};

/* Exact widening of one stored element to double. */
static double orc_load(const void *p, int dt, int64_t i)
{
    if (dt == ORC_F32)
        return (double)((const float *)p)[i];
    if (dt == ORC_BF16) {
        uint32_t u = ((uint32_t)((const uint16_t *)p)[i]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return ((const double *)p)[i];
}

static void orc_store(void *p, int dt, int64_t i, double v)
{
    if (dt == ORC_F32)
        ((float *)p)[i] = (float)v;
    else
        ((double *)p)[i] = v;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* E(p): the number of complete blocks of m tokens that end at or before
 * position p ([QbitAI] "compressed attention guarantees strict causality").
 * Pinned by the closed-form counts the pages print (1M tokens / 4 and / 128,
 * 324 tokens / 4 = 81 in [Wiki]). */
int64_t orc_num_entries(int64_t p, int m)
{
    if (p < 0 || m <= 0)
        return 0;
    return (p + 1) / m;
}

/* KV compression ([QbitAI] CSA step 1 "every m tokens' KV entries are merged
 * into one"; HCA "every m'=128 tokens into one, with no overlap"):
 *     C[b, j, c] = sum_{r<m} w[r] * X[b, j*m + r, c]
 * for every block j in [tok_begin[b]/m, tok_end[b]/m) (integer division).
 * x: [B, N_cap, d] (dtype x_dt), out: [B, E_cap, d] (dtype out_dt, f32/f64).
 * Pinned by: one-hot w copies token r exactly; w = 1/m gives the block mean;
 * m = 1, w = [1] is the identity; linearity in X. */
int orc_compress(const void *x, int x_dt, int B, int64_t N_cap, int d,
                 const int64_t *tok_begin, const int64_t *tok_end,
                 const float *w, int m, void *out, int out_dt, int64_t E_cap)
{
    if (B < 0 || d <= 0 || m <= 0 || (out_dt != ORC_F32 && out_dt != ORC_F64))
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int64_t j0 = tok_begin[b] / m, j1 = tok_end[b] / m;
        if (tok_begin[b] < 0 || tok_end[b] > N_cap || j1 > E_cap)
            return ORC_ERR_RANGE;
        (void)j0;
    }
    int err = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int64_t j0 = tok_begin[b] / m, j1 = tok_end[b] / m;
#pragma omp parallel for schedule(static)
        for (int64_t j = j0; j < j1; ++j) {
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int r = 0; r < m; ++r) {
                    int64_t t = j * m + r;
                    acc += (double)w[r] * orc_load(x, x_dt, ((int64_t)b * N_cap + t) * d + c);
                }
                orc_store(out, out_dt, ((int64_t)b * E_cap + j) * d + c, acc);
            }
        }
    }
    return err;
}

typedef struct {
    int64_t s; /* indexer score */
    int32_t j; /* entry index */
} orc_scored;

/* (score desc, index asc): the strict total order that makes selection exact. */
static int orc_cmp_scored(const void *a, const void *b)
{
    const orc_scored *x = (const orc_scored *)a, *y = (const orc_scored *)b;
    if (x->s != y->s)
        return x->s > y->s ? -1 : 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int orc_cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Lightning indexer + top-k ([QbitAI] CSA step 2, "for each query token a
 * light indexer scores it against every compressed block ... keep the top-k";
 * k = 512 Flash / 1024 Pro in [Essay]).
 * Rows are independent queries: row r belongs to sequence row_b[r] and sits
 * at position row_p[r].  q: [n_rows, DI] int8, kI: [B, E_cap, DI] int8.
 *   s_j = sum_c q[c] * kI[b, j, c]      (exact, int64, checked to fit int32)
 * over j < E(p); order by (s desc, j asc); keep n = min(topk, E(p)); report
 * them in ascending j, padded with -1 to topk; cnt = n.
 * Pinned by: brute-force set characterisation on tiny inputs, numpy integer
 * matmul for the scores, all-equal scores -> 0..k-1, k >= E -> all,
 * planted winners, heavy ties. */
int orc_index_topk_rows(int64_t n_rows, const int8_t *q, const int64_t *row_b,
                        const int64_t *row_p, const int8_t *kI, int B, int64_t E_cap,
                        int DI, int m, int topk, int32_t *idx_out, int32_t *cnt_out)
{
    if (n_rows < 0 || DI <= 0 || m <= 0 || topk < 0)
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (row_b[r] < 0 || row_b[r] >= B || orc_num_entries(row_p[r], m) > E_cap)
            return ORC_ERR_RANGE;
    }
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = row_b[r];
        int64_t E = orc_num_entries(row_p[r], m);
        orc_scored *all = (orc_scored *)malloc(sizeof(orc_scored) * (size_t)(E > 0 ? E : 1));
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)(topk > 0 ? topk : 1));
        if (!all || !sel) {
#pragma omp critical
            err = ORC_ERR_NOMEM;
            free(all);
            free(sel);
            continue;
        }
        for (int64_t j = 0; j < E; ++j) {
            int64_t s = 0;
            for (int c = 0; c < DI; ++c)
                s += (int64_t)q[r * DI + c] * (int64_t)kI[((int64_t)b * E_cap + j) * DI + c];
            if (s > INT32_MAX || s < INT32_MIN) {
#pragma omp critical
                err = ORC_ERR_OVERFLOW;
            }
            all[j].s = s;
            all[j].j = (int32_t)j;
        }
        qsort(all, (size_t)E, sizeof(orc_scored), orc_cmp_scored);
        int64_t n = E < topk ? E : topk;
        for (int64_t i = 0; i < n; ++i)
            sel[i] = all[i].j;
        qsort(sel, (size_t)n, sizeof(int32_t), orc_cmp_i32);
        for (int64_t i = 0; i < topk; ++i)
            idx_out[r * topk + i] = i < n ? sel[i] : -1;
        cnt_out[r] = (int32_t)n;
        free(all);
        free(sel);
    }
    return err;
}

/* Core attention over the hybrid set ([QbitAI] CSA step 3 "Multi-Query
 * Attention over the selected top-k compressed KV blocks"; HCA "dense
 * attention over all compressed KV"; sliding-window paragraph "each query also
 * sees the uncompressed KV of the most recent 128 tokens").
 * Row r (sequence b = row_b[r], position p = row_p[r]) with query heads
 * q[r, h, :] attends, with one softmax per head, to the multiset
 *     S = {kc/vc[b, j] : j selected} + {k_raw/v_raw[b, t] : max(0,p-W+1) <= t <= p}
 * where "selected" is idx[r, :] (entries < 0 skipped; every other entry must
 * be < E(p)) or, when idx is NULL, every j < E(p) (dense, HCA).
 *   l_x = scale * <q, k_x>,  M = max l,  L = sum exp(l - M),
 *   out = sum exp(l_x - M) v_x / L,  lse = M + ln L.
 * Empty S gives out = 0 and lse = -inf.
 * Layouts: q [n_rows, H, d]; kc, vc [B, E_cap, d]; k_raw, v_raw [B, N_cap, d];
 * out [n_rows, H, d] f64; lse [n_rows, H] f64 (may be NULL).
 * Pinned by: m = 1 and every entry selected with W = 0 equals textbook causal
 * attention; W > 0 then adds a +ln 2 bias on the window keys; no entries gives
 * sliding-window attention; q = 0 gives the mean of V; one-hot V exposes the
 * probabilities (sum to 1, equal a library softmax). */
int orc_attn_rows(int64_t n_rows, const void *q, int q_dt, const int64_t *row_b,
                  const int64_t *row_p, int H, int d, const void *kc, const void *vc,
                  int c_dt, int64_t E_cap, int m, const int32_t *idx, int topk,
                  const void *k_raw, const void *v_raw, int r_dt, int64_t N_cap,
                  int window, double scale, double *out, double *lse)
{
    if (n_rows < 0 || H <= 0 || d <= 0 || m <= 0 || window < 0 || (idx && topk < 0))
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t p = row_p[r];
        if (p < 0 || p >= N_cap || orc_num_entries(p, m) > E_cap)
            return ORC_ERR_RANGE;
    }
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = row_b[r], p = row_p[r];
        int64_t E = orc_num_entries(p, m);
        int64_t t0 = p - window + 1 < 0 ? 0 : p - window + 1;
        int64_t n_win = window > 0 ? p - t0 + 1 : 0;
        int64_t n_ent = idx ? topk : E;
        /* the multiset S as (source, row) pairs: source 0 = compressed, 1 = raw */
        int64_t n_max = n_ent + n_win;
        const void **krow_base = (const void **)malloc(sizeof(void *) * (size_t)(n_max + 1));
        const void **vrow_base = (const void **)malloc(sizeof(void *) * (size_t)(n_max + 1));
        int *rdt = (int *)malloc(sizeof(int) * (size_t)(n_max + 1));
        int64_t *roff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_max + 1));
        double *logit = (double *)malloc(sizeof(double) * (size_t)(n_max + 1));
        if (!krow_base || !vrow_base || !rdt || !roff || !logit) {
#pragma omp critical
            err = ORC_ERR_NOMEM;
            free(krow_base); free(vrow_base); free(rdt); free(roff); free(logit);
            continue;
        }
        int64_t n = 0;
        for (int64_t i = 0; i < n_ent; ++i) {
            int64_t j = idx ? (int64_t)idx[r * topk + i] : i;
            if (j < 0)
                continue;
            if (j >= E) {
#pragma omp critical
                err = ORC_ERR_INDEX;
                continue;
            }
            krow_base[n] = kc;
            vrow_base[n] = vc;
            rdt[n] = c_dt;
            roff[n] = (b * E_cap + j) * d;
            ++n;
        }
        for (int64_t t = t0; t < t0 + n_win; ++t) {
            krow_base[n] = k_raw;
            vrow_base[n] = v_raw;
            rdt[n] = r_dt;
            roff[n] = (b * N_cap + t) * d;
            ++n;
        }
        for (int h = 0; h < H; ++h) {
            const int64_t qoff = (r * H + h) * (int64_t)d;
            double *o = out + qoff;
            if (n == 0) {
                for (int c = 0; c < d; ++c)
                    o[c] = 0.0;
                if (lse)
                    lse[r * H + h] = -INFINITY;
                continue;
            }
            double M = -INFINITY;
            for (int64_t x = 0; x < n; ++x) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += orc_load(q, q_dt, qoff + c) * orc_load(krow_base[x], rdt[x], roff[x] + c);
                logit[x] = scale * dot;
                if (logit[x] > M)
                    M = logit[x];
            }
            double L = 0.0;
            for (int64_t x = 0; x < n; ++x)
                L += exp(logit[x] - M);
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int64_t x = 0; x < n; ++x)
                    acc += exp(logit[x] - M) * orc_load(vrow_base[x], rdt[x], roff[x] + c);
                o[c] = acc / L;
            }
            if (lse)
                lse[r * H + h] = M + log(L);
        }
        free(krow_base); free(vrow_base); free(rdt); free(roff); free(logit);
    }
    return err;
}

/* Merging attention results computed over disjoint parts of one set (the
 * split-KV step of decode; the pages give no formula, this is the standard
 * log-sum-exp identity):
 *     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * out_s.
 * Parts with lse_s = -inf (empty) contribute nothing; all parts empty gives
 * out = 0, lse = -inf.  o_parts [n_parts, H, d], lse_parts [n_parts, H].
 * Pinned by: merging the oracle's attention over any partition of S equals
 * its attention over S. */
int orc_lse_merge(int n_parts, const double *o_parts, const double *lse_parts, int H, int d,
                  double *out, double *lse)
{
    if (n_parts < 0 || H <= 0 || d <= 0)
        return ORC_ERR_ARG;
    for (int h = 0; h < H; ++h) {
        double M = -INFINITY;
        for (int s = 0; s < n_parts; ++s)
            if (lse_parts[s * H + h] > M)
                M = lse_parts[s * H + h];
        double *o = out + (int64_t)h * d;
        if (M == -INFINITY) {
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            if (lse)
                lse[h] = -INFINITY;
            continue;
        }
        double L = 0.0;
        for (int s = 0; s < n_parts; ++s)
            L += exp(lse_parts[s * H + h] - M);
        double total = M + log(L);
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < n_parts; ++s) {
                double ls = lse_parts[s * H + h];
                if (ls == -INFINITY)
                    continue;
                acc += exp(ls - total) * o_parts[((int64_t)s * H + h) * d + c];
            }
            o[c] = acc;
        }
        if (lse)
            lse[h] = total;
    }
    return ORC_OK;
}

/* V4's per-layer attention details ([QbitAI] section 混合注意力机制, the paragraphs after
 * the CSA/HCA description):
 *   - Q/KV normalisation: before core attention the query and every KV entry go
 *     through RMSNorm, N(x)_c = gamma_c * x_c / sqrt(mean_c(x_c^2) + eps);
 *   - partial RoPE: only the last `rd` channels of the query and of the KV entries
 *     are rotated; channel pair k (channels d-rd+2k, d-rd+2k+1) of a vector at
 *     position t turns by the angle t * theta^(-2k/rd);
 *   - a KV entry is both key and value, so the output also gets the rotation of
 *     position -i (i = the query's position) on the same channels, which leaves
 *     only relative position;
 *   - a learnable sink logit z_h joins the softmax denominator.
 * For query row r (sequence b, position p) and head h, over the same multiset S as
 * orc_attn_rows (selected or all visible entries, plus raw tokens p-W+1 .. p),
 * with position t_x = (j+1)*m - 1 for entry j (its block's last token; reading)
 * and t for raw token t:
 *   q~ = R(p) N_q(q[r, h]),   e~_x = R(t_x) N_kv(e_x)
 *   logit_x = scale * <q~, e~_x>,   L = ln(sum_x exp(logit_x) + exp(z_h))
 *   out = R(-p) sum_x exp(logit_x - L) e~_x,   lse = L.
 * With S empty and no sink: out = 0, lse = -inf.  ent: [B, E_cap, d] (the shared
 * K=V entries), raw: [B, N_cap, d]; gamma_q, gamma_kv: [d] or NULL (all ones);
 * sink: [H] or NULL.
 * Pinned by: with rd = 0 and unit gamma it equals orc_attn_rows on normalised
 * inputs; one item gives out = R(t - p) N(e) in closed form; shifting every
 * position by the same amount leaves the output unchanged; the sink's weight on
 * one item is exp(l) / (exp(l) + exp(z)). */
static void orc_norm_rope(const void *x, int dt, int64_t off, int d, const double *gamma, double eps,
                          int rd, double theta, int64_t pos, double *y)
{
    double ss = 0.0;
    for (int c = 0; c < d; ++c) {
        double v = orc_load(x, dt, off + c);
        ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / d + eps);
    for (int c = 0; c < d; ++c)
        y[c] = (gamma ? gamma[c] : 1.0) * orc_load(x, dt, off + c) * inv;
    for (int k = 0; k < rd / 2; ++k) {
        int c0 = d - rd + 2 * k;
        double ang = (double)pos * pow(theta, -2.0 * k / rd);
        double u = y[c0], v = y[c0 + 1];
        y[c0] = u * cos(ang) - v * sin(ang);
        y[c0 + 1] = u * sin(ang) + v * cos(ang);
    }
}

int orc_attn_v4_rows(int64_t n_rows, const void *q, int q_dt, const int64_t *row_b,
                     const int64_t *row_p, int H, int d, const void *ent, int e_dt, int64_t E_cap,
                     int m, const int32_t *idx, int topk, const void *raw, int r_dt, int64_t N_cap,
                     int window, double scale, const double *gamma_q, const double *gamma_kv,
                     double eps, int rd, double theta, const double *sink, double *out, double *lse)
{
    if (n_rows < 0 || H <= 0 || d <= 0 || m <= 0 || window < 0 || (idx && topk < 0) || rd < 0 ||
        rd > d || rd % 2)
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t p = row_p[r];
        if (p < 0 || p >= N_cap || orc_num_entries(p, m) > E_cap)
            return ORC_ERR_RANGE;
    }
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = row_b[r], p = row_p[r];
        int64_t E = orc_num_entries(p, m);
        int64_t t0 = p - window + 1 < 0 ? 0 : p - window + 1;
        int64_t n_win = window > 0 ? p - t0 + 1 : 0;
        int64_t n_ent = idx ? topk : E;
        int64_t n_max = n_ent + n_win;
        double *items = (double *)malloc(sizeof(double) * (size_t)((n_max + 1) * d));
        double *logit = (double *)malloc(sizeof(double) * (size_t)(n_max + 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        if (!items || !logit || !qv) {
#pragma omp critical
            err = ORC_ERR_NOMEM;
            free(items); free(logit); free(qv);
            continue;
        }
        /* the multiset, each item normalised and rotated to its own position */
        int64_t n = 0;
        for (int64_t i = 0; i < n_ent; ++i) {
            int64_t j = idx ? (int64_t)idx[r * topk + i] : i;
            if (j < 0)
                continue;
            if (j >= E) {
#pragma omp critical
                err = ORC_ERR_INDEX;
                continue;
            }
            orc_norm_rope(ent, e_dt, (b * E_cap + j) * d, d, gamma_kv, eps, rd, theta, (j + 1) * m - 1,
                          items + n * d);
            ++n;
        }
        for (int64_t t = t0; t < t0 + n_win; ++t) {
            orc_norm_rope(raw, r_dt, (b * N_cap + t) * d, d, gamma_kv, eps, rd, theta, t, items + n * d);
            ++n;
        }
        for (int h = 0; h < H; ++h) {
            orc_norm_rope(q, q_dt, (r * H + h) * (int64_t)d, d, gamma_q, eps, rd, theta, p, qv);
            double z = sink ? sink[h] : -INFINITY;
            double M = z;
            for (int64_t x = 0; x < n; ++x) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += qv[c] * items[x * d + c];
                logit[x] = scale * dot;
                if (logit[x] > M)
                    M = logit[x];
            }
            double *o = out + (r * H + h) * (int64_t)d;
            if (M == -INFINITY) {
                for (int c = 0; c < d; ++c)
                    o[c] = 0.0;
                if (lse)
                    lse[r * H + h] = -INFINITY;
                continue;
            }
            double Lsum = z == -INFINITY ? 0.0 : exp(z - M);
            for (int64_t x = 0; x < n; ++x)
                Lsum += exp(logit[x] - M);
            double L = M + log(Lsum);
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int64_t x = 0; x < n; ++x)
                    acc += exp(logit[x] - L) * items[x * d + c];
                o[c] = acc;
            }
            /* the rotation of position -p on the same channels */
            for (int k = 0; k < rd / 2; ++k) {
                int c0 = d - rd + 2 * k;
                double ang = -(double)p * pow(theta, -2.0 * k / rd);
                double u = o[c0], v = o[c0 + 1];
                o[c0] = u * cos(ang) - v * sin(ang);
                o[c0 + 1] = u * sin(ang) + v * cos(ang);
            }
            if (lse)
                lse[r * H + h] = L;
        }
        free(items); free(logit); free(qv);
    }
    return err;
}

/* Learned, attention-like compression ([QbitAI] 混合注意力机制, CSA step 1: every m
 * tokens' KV entries are merged into one by an attention-like mechanism with learned
 * weights; the HCA paragraph: m' = 128 and, unlike CSA, no overlap).  The pages give
 * no formula; reading: entry j pools the L tokens t_r = (j+1)*m - L + r, r = 0..L-1
 * (L = 2m for CSA: the block and the one before it; L = m for HCA), dropping t_r < 0,
 * with weights from a learned scoring vector u [d] and position bias bias [L]:
 *     s_r = <u, K[b, t_r]> + bias[r],   a = softmax_r(s),
 *     Kc[b, j] = sum_r a_r K[b, t_r],   Vc[b, j] = sum_r a_r V[b, t_r].
 * Entry j still ends at token (j+1)*m - 1, so visibility E(p) is unchanged.  Blocks
 * j in [tok_begin[b]/m, tok_end[b]/m) are written (out dtype f32/f64).
 * Pinned by: u = 0, bias = 0, L = m gives the block mean (orc_compress with
 * w = 1/m); a bias of -inf everywhere but r copies token t_r; adding a constant to
 * bias changes nothing; L = 2m with the first m biases at -inf equals L = m. */
int orc_compress_learned(const void *k, const void *v, int x_dt, int B, int64_t N_cap, int d,
                         const double *u, const double *bias, int m, int L,
                         const int64_t *tok_begin, const int64_t *tok_end,
                         void *kc, void *vc, int out_dt, int64_t E_cap)
{
    if (B < 0 || d <= 0 || m <= 0 || L < 1 || (out_dt != ORC_F32 && out_dt != ORC_F64))
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        if (tok_begin[b] < 0 || tok_end[b] > N_cap || tok_begin[b] > tok_end[b])
            return ORC_ERR_RANGE;
        if (tok_end[b] / m > E_cap)
            return ORC_ERR_RANGE;
    }
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *sc = (double *)malloc(sizeof(double) * (size_t)L);
        if (!sc) {
#pragma omp critical
            err = ORC_ERR_NOMEM;
            continue;
        }
        for (int64_t j = tok_begin[b] / m; j < tok_end[b] / m; ++j) {
            int64_t t0 = (j + 1) * m - L;
            double M = -INFINITY;
            for (int r = 0; r < L; ++r) {
                int64_t t = t0 + r;
                sc[r] = -INFINITY;
                if (t < 0)
                    continue;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += u[c] * orc_load(k, x_dt, ((int64_t)b * N_cap + t) * d + c);
                sc[r] = dot + bias[r];
                if (sc[r] > M)
                    M = sc[r];
            }
            double Z = 0.0;
            for (int r = 0; r < L; ++r)
                if (sc[r] != -INFINITY)
                    Z += exp(sc[r] - M);
            for (int c = 0; c < d; ++c) {
                double ak = 0.0, av = 0.0;
                for (int r = 0; r < L; ++r) {
                    if (sc[r] == -INFINITY)
                        continue;
                    double a = exp(sc[r] - M) / Z;
                    int64_t t = t0 + r;
                    ak += a * orc_load(k, x_dt, ((int64_t)b * N_cap + t) * d + c);
                    av += a * orc_load(v, x_dt, ((int64_t)b * N_cap + t) * d + c);
                }
                orc_store(kc, out_dt, ((int64_t)b * E_cap + j) * d + c, ak);
                orc_store(vc, out_dt, ((int64_t)b * E_cap + j) * d + c, av);
            }
        }
        free(sc);
    }
    return err;
}

