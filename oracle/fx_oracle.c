/*
 * fx_oracle.c -- plain, slow, fp64 reference for importance-scored KV token selection feeding
 * sparse GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the bench's CPU baseline
 * may load this file.  It shares no code, header, table or helper with the CUDA library: every
 * function here is the definition written out as loops in double precision.
 *
 * Sources (pages and sections):
 *   FastOCR: Dynamic Visual Fixation via KV Cache Pruning for Efficient Document Parsing
 *     (gist.science/paper/2605.17447), Methodology, "Focal-Guided Pruning" (focal layers attend over
 *     the full cache and pick the top-attended image tokens at a kept ratio; the other layers attend
 *     only to the pruned set) and "Cross-Step Fixation Reuse" (the previous step's set warm-starts the
 *     next step).
 *   FastKV: Decoupling of Context Reduction and KV Cache Compression for Prefill-Decoding Acceleration
 *     (gist.science/paper/2502.01068), section 2.A "Token-Selective Propagation" (saliency = attention
 *     weights from a recent window of queries to all context tokens) and 2.B "Decoupled KV Retention"
 *     (a chosen subset of KV entries is kept for decoding).
 *   HPD-Parsing (zwcih.github.io/ocr-research-wiki/wiki/sources/hpd-parsing), method part 2
 *     "Shared-Prefix KV Reuse + Context Isolation" (a branch attends to the shared context, its own
 *     prefix and its own history) and part 3 "P-MTP" (several drafted tokens verified in one step).
 *
 * Conventions shared with the library's public header (restated, not included):
 *   - bf16 values arrive as their 16-bit patterns and are decoded exactly to double;
 *   - a KV cache element (b, h, t, c) lives at base + b*sb + h*sh + t*st + c (strides in elements);
 *   - query head g belongs to KV head g / G with G = Hq / Hkv;
 *   - query row r of KV head h is (gi, i) = (r / Mq, r % Mq): query head h*G + gi, position i;
 *     q and out are [B, Hq, Mq, d];
 *   - the importance of token j for KV head h is the softmax probability of j summed over every
 *     query row of the group (all G heads and all Mq positions);
 *   - top-k order is score descending, then index ascending; the chosen set is written ascending;
 *   - an empty key set gives an all-zero output row.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------------------ */
/* small helpers                                                                               */

static double bf(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int g_threads = 0;

/* Number of worker threads the oracle uses (0 or negative: every online core).  Returns the count. */
int oracle_set_threads(int n)
{
    if (n <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n = c > 0 ? (int)c : 1;
    }
    g_threads = n;
    return n;
}

int oracle_get_threads(void)
{
    if (g_threads <= 0) oracle_set_threads(0);
    return g_threads;
}

typedef void (*work_fn)(void* ctx, int item, double* scratch);

typedef struct {
    work_fn fn;
    void* ctx;
    int n_items;
    int next;
    size_t scratch_doubles;
} pool_t;

static void* pool_worker(void* arg)
{
    pool_t* p = (pool_t*)arg;
    double* scratch = (double*)malloc((p->scratch_doubles ? p->scratch_doubles : 1) * sizeof(double));
    for (;;) {
        int it = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

/* Run fn(ctx, item, scratch) for item in [0, n_items) on the worker threads. */
static void parallel_for(int n_items, work_fn fn, void* ctx, size_t scratch_doubles)
{
    pool_t p = {fn, ctx, n_items, 0, scratch_doubles};
    int nt = oracle_get_threads();
    if (nt > n_items) nt = n_items;
    if (nt <= 1) {
        pool_worker(&p);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
}

/*
 * Scaled dot-product attention of one query row over an explicit list of n key/value rows:
 *   l_j = scale * sum_c q_c k_jc,   p_j = exp(l_j - max l) / sum_i exp(l_i - max l),
 *   out_c = sum_j p_j v_jc.
 * p receives the probabilities.  n == 0 gives out = 0.
 */
static void attend(const double* q, int d, double scale, int n, const uint16_t* const* kr,
                   const uint16_t* const* vr, double* p, double* out)
{
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double l = 0.0;
        for (int c = 0; c < d; ++c) l += q[c] * bf(kr[j][c]);
        l *= scale;
        p[j] = l;
        if (l > m) m = l;
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        p[j] = exp(p[j] - m);
        z += p[j];
    }
    for (int j = 0; j < n; ++j) p[j] /= z;
    for (int j = 0; j < n; ++j) {
        const uint16_t* v = vr[j];
        for (int c = 0; c < d; ++c) out[c] += p[j] * bf(v[c]);
    }
}

static void load_q(const uint16_t* q, int64_t off, int d, double* dst)
{
    for (int c = 0; c < d; ++c) dst[c] = bf(q[off + c]);
}

/* ------------------------------------------------------------------------------------------ */
/* Focal layer: full attention over the whole cache plus per-token importance.                 */
/* FastOCR Methodology, Focal-Guided Pruning ("Cross-Layer Propagation"): focal layers attend    */
/* over the full KV cache; FastKV 2.A: saliency from a window of recent queries, which are       */
/* causal (query i at position q_pos0 + i sees tokens j <= q_pos0 + i).                         */

typedef struct {
    const uint16_t *k, *v;
    const int32_t* len;
    int64_t sb, sh, st;
    int B, Hkv, Tcap, d;
    const uint16_t* q;
    int Hq, Mq, q_pos0;
    double scale;
    int cand_lo, cand_hi;
    double *out, *scores;
} focal_ctx;

static void focal_item(void* vctx, int item, double* scratch)
{
    focal_ctx* c = (focal_ctx*)vctx;
    int b = item / c->Hkv, h = item % c->Hkv;
    int G = c->Hq / c->Hkv, d = c->d;
    int n = c->len[b];
    int ncand = c->cand_hi - c->cand_lo;
    const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
    const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
    double* p = scratch;             /* n doubles */
    double* qrow = scratch + n;      /* d doubles */
    double* orow = qrow + d;         /* d doubles */
    double* s = c->scores ? c->scores + ((int64_t)b * c->Hkv + h) * ncand : NULL;
    if (s)
        for (int j = 0; j < ncand; ++j) s[j] = 0.0;
    for (int j = 0; j < n; ++j) {
        kr[j] = c->k + b * c->sb + h * c->sh + (int64_t)j * c->st;
        vr[j] = c->v + b * c->sb + h * c->sh + (int64_t)j * c->st;
    }
    for (int gi = 0; gi < G; ++gi) {
        int g = h * G + gi;
        for (int i = 0; i < c->Mq; ++i) {
            int visible = n;
            if (c->q_pos0 >= 0) {
                int lim = c->q_pos0 + i + 1; /* tokens 0 .. q_pos0 + i */
                if (lim < visible) visible = lim;
            }
            if (visible < 0) visible = 0;
            int64_t qoff = (((int64_t)b * c->Hq + g) * c->Mq + i) * d;
            load_q(c->q, qoff, d, qrow);
            attend(qrow, d, c->scale, visible, kr, vr, p, orow);
            if (c->out)
                for (int e = 0; e < d; ++e) c->out[qoff + e] = orow[e];
            if (s)
                for (int j = 0; j < visible; ++j)
                    if (j >= c->cand_lo && j < c->cand_hi) s[j - c->cand_lo] += p[j];
        }
    }
    free(kr);
    free(vr);
}

/*
 * out    [B, Hq, Mq, d]              attention output (nullable)
 * scores [B, Hkv, cand_hi - cand_lo] importance of tokens cand_lo .. cand_hi-1 (nullable)
 * q_pos0 < 0: every query sees all len[b] tokens; otherwise query i sees tokens 0 .. q_pos0 + i.
 */
void oracle_focal(const uint16_t* k, const uint16_t* v, const int32_t* len, int64_t sb, int64_t sh,
                  int64_t st, int B, int Hkv, int Tcap, int d, const uint16_t* q, int Hq, int Mq,
                  int q_pos0, double scale, int cand_lo, int cand_hi, double* out, double* scores)
{
    focal_ctx c = {k, v, len, sb, sh, st, B, Hkv, Tcap, d, q, Hq, Mq, q_pos0, scale,
                   cand_lo, cand_hi, out, scores};
    int nmax = 0;
    for (int b = 0; b < B; ++b)
        if (len[b] > nmax) nmax = len[b];
    parallel_for(B * Hkv, focal_item, &c, (size_t)nmax + 2 * (size_t)d);
}

/* ------------------------------------------------------------------------------------------ */
/* Top-k selection.  FastOCR FGP: keep the top-attended tokens at a kept ratio; ties go to the   */
/* lower index and the kept set is reported in ascending token order.                          */

typedef struct {
    double s;
    int j;
} sj_t;

static int cmp_desc(const void* a, const void* b)
{
    const sj_t* x = (const sj_t*)a;
    const sj_t* y = (const sj_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_int(const void* a, const void* b)
{
    int x = *(const int*)a, y = *(const int*)b;
    return (x > y) - (x < y);
}

/* scores [rows, n] -> idx_out [rows, k]: the k best by (score desc, index asc), ascending. */
void oracle_topk(const double* scores, int rows, int n, int k, int32_t* idx_out)
{
    sj_t* buf = (sj_t*)malloc(sizeof(sj_t) * (size_t)(n > 0 ? n : 1));
    int* sel = (int*)malloc(sizeof(int) * (size_t)(k > 0 ? k : 1));
    for (int r = 0; r < rows; ++r) {
        for (int j = 0; j < n; ++j) {
            buf[j].s = scores[(int64_t)r * n + j];
            buf[j].j = j;
        }
        qsort(buf, (size_t)n, sizeof(sj_t), cmp_desc);
        for (int i = 0; i < k; ++i) sel[i] = buf[i].j;
        qsort(sel, (size_t)k, sizeof(int), cmp_int);
        for (int i = 0; i < k; ++i) idx_out[(int64_t)r * k + i] = sel[i];
    }
    free(buf);
    free(sel);
}

/* ------------------------------------------------------------------------------------------ */
/* Sparse GQA decode: a non-focal layer attends only over the pruned set (FastOCR FGP) plus a     */
/* dense tail [tail_lo, len) (text tokens, or every token of a compacted cache).  The softmax is  */
/* normalised over that set.  One query position per sequence.                                  */

typedef struct {
    const uint16_t *k, *v;
    const int32_t* len;
    int64_t sb, sh, st;
    int B, Hkv, d;
    const uint16_t* q;
    int Hq;
    const int32_t* idx;
    int kk, tail_lo;
    double scale;
    double* out;
} sparse_ctx;

static void sparse_item(void* vctx, int item, double* scratch)
{
    sparse_ctx* c = (sparse_ctx*)vctx;
    int b = item / c->Hkv, h = item % c->Hkv;
    int G = c->Hq / c->Hkv, d = c->d;
    int n_tail = c->len[b] - c->tail_lo;
    if (n_tail < 0) n_tail = 0;
    int n = c->kk + n_tail;
    const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
    const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
    int m = 0;
    const int32_t* row_idx = c->idx ? c->idx + ((int64_t)b * c->Hkv + h) * c->kk : NULL;
    for (int p = 0; p < c->kk; ++p, ++m) {
        int t = row_idx[p];
        kr[m] = c->k + b * c->sb + h * c->sh + (int64_t)t * c->st;
        vr[m] = c->v + b * c->sb + h * c->sh + (int64_t)t * c->st;
    }
    for (int t = c->tail_lo; t < c->len[b]; ++t, ++m) {
        kr[m] = c->k + b * c->sb + h * c->sh + (int64_t)t * c->st;
        vr[m] = c->v + b * c->sb + h * c->sh + (int64_t)t * c->st;
    }
    double* p = scratch;
    double* qrow = scratch + n;
    double* orow = qrow + d;
    for (int gi = 0; gi < G; ++gi) {
        int64_t qoff = ((int64_t)b * c->Hq + h * G + gi) * d;
        load_q(c->q, qoff, d, qrow);
        attend(qrow, d, c->scale, m, kr, vr, p, orow);
        for (int e = 0; e < d; ++e) c->out[qoff + e] = orow[e];
    }
    free(kr);
    free(vr);
}

/* q, out: [B, Hq, 1, d]; idx: [B, Hkv, k] (may be NULL when k == 0). */
void oracle_sparse_decode(const uint16_t* k, const uint16_t* v, const int32_t* len, int64_t sb,
                          int64_t sh, int64_t st, int B, int Hkv, int d, const uint16_t* q, int Hq,
                          const int32_t* idx, int kk, int tail_lo, double scale, double* out)
{
    sparse_ctx c = {k, v, len, sb, sh, st, B, Hkv, d, q, Hq, idx, kk, tail_lo, scale, out};
    int nmax = 0;
    for (int b = 0; b < B; ++b) {
        int n = kk + (len[b] > tail_lo ? len[b] - tail_lo : 0);
        if (n > nmax) nmax = n;
    }
    parallel_for(B * Hkv, sparse_item, &c, (size_t)nmax + 2 * (size_t)d);
}

/* ------------------------------------------------------------------------------------------ */
/* KV compaction (FastKV 2.B, decoupled KV retention): the retained entries of one layer are     */
/* copied, in ascending source order, into a contiguous cache: rows idx[0..k) then the tail      */
/* [tail_lo, len).  dst_len[b] = k + max(0, len[b] - tail_lo).                                   */

void oracle_kv_compact(const uint16_t* sk, const uint16_t* sv, const int32_t* len, int64_t sb,
                       int64_t sh, int64_t st, int B, int Hkv, int d, const int32_t* idx, int kk,
                       int tail_lo, uint16_t* dk, uint16_t* dv, int64_t db, int64_t dh, int64_t dt,
                       int32_t* dst_len)
{
    for (int b = 0; b < B; ++b) {
        int n_tail = len[b] > tail_lo ? len[b] - tail_lo : 0;
        dst_len[b] = kk + n_tail;
        for (int h = 0; h < Hkv; ++h) {
            for (int r = 0; r < kk + n_tail; ++r) {
                int t = r < kk ? idx[((int64_t)b * Hkv + h) * kk + r] : tail_lo + (r - kk);
                for (int c = 0; c < d; ++c) {
                    dk[b * db + h * dh + (int64_t)r * dt + c] = sk[b * sb + h * sh + (int64_t)t * st + c];
                    dv[b * db + h * dh + (int64_t)r * dt + c] = sv[b * sb + h * sh + (int64_t)t * st + c];
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Shared-prefix draft verification (HPD-Parsing parts 2 and 3).  Branch b's draft position i    */
/* attends over: the shared prefix it forked from -- its first pre_len[b] rows (all P without     */
/* pre_len), or the rows prefix_idx[b, h, 0..kp) when given -- then its own suffix rows off[b] ..  */
/* off[b]+L_b-1 (L_b = suf_len[b], or off[b+1]-off[b] without suf_len), then its own draft rows    */
/* 0 .. i (causal).                                                                                */

typedef struct {
    const uint16_t *pk, *pv;
    int64_t p_sh, p_st;
    int P;
    const uint16_t *sk, *sv;
    int64_t s_sh, s_st;
    const int32_t* off;
    const uint16_t *dk, *dv;
    int64_t d_sb, d_si, d_sh;
    const uint16_t* q;
    int Br, Hkv, Hq, Mq, d;
    const int32_t* pidx;
    int kp;
    const int32_t* pre_len;
    const int32_t* suf_len;
    double scale;
    double* out;
} prefix_ctx;

static void prefix_item(void* vctx, int item, double* scratch)
{
    prefix_ctx* c = (prefix_ctx*)vctx;
    int b = item / c->Hkv, h = item % c->Hkv;
    int G = c->Hq / c->Hkv, d = c->d;
    int np = c->pidx ? c->kp : (c->pre_len ? c->pre_len[b] : c->P);
    int s0 = c->off[b];
    int ns = c->suf_len ? c->suf_len[b] : c->off[b + 1] - c->off[b];
    int nmax = np + ns + c->Mq;
    const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)nmax);
    const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)nmax);
    int m = 0;
    for (int p = 0; p < np; ++p, ++m) {
        int t = c->pidx ? c->pidx[((int64_t)b * c->Hkv + h) * c->kp + p] : p;
        kr[m] = c->pk + h * c->p_sh + (int64_t)t * c->p_st;
        vr[m] = c->pv + h * c->p_sh + (int64_t)t * c->p_st;
    }
    for (int t = s0; t < s0 + ns; ++t, ++m) {
        kr[m] = c->sk + h * c->s_sh + (int64_t)t * c->s_st;
        vr[m] = c->sv + h * c->s_sh + (int64_t)t * c->s_st;
    }
    for (int i = 0; i < c->Mq; ++i) {
        kr[m + i] = c->dk + b * c->d_sb + (int64_t)i * c->d_si + h * c->d_sh;
        vr[m + i] = c->dv + b * c->d_sb + (int64_t)i * c->d_si + h * c->d_sh;
    }
    double* p = scratch;
    double* qrow = scratch + nmax;
    double* orow = qrow + d;
    for (int gi = 0; gi < G; ++gi) {
        for (int i = 0; i < c->Mq; ++i) {
            int64_t qoff = (((int64_t)b * c->Hq + h * G + gi) * c->Mq + i) * d;
            load_q(c->q, qoff, d, qrow);
            attend(qrow, d, c->scale, m + i + 1, kr, vr, p, orow);
            for (int e = 0; e < d; ++e) c->out[qoff + e] = orow[e];
        }
    }
    free(kr);
    free(vr);
}

/*
 * prefix: rows (h, t) at pk + h*p_sh + t*p_st, t < P;   suffix: rows (h, t) at sk + h*s_sh + t*s_st
 * with branch b owning t in [off[b], off[b] + L_b);  draft: rows (b, i, h) at dk + b*d_sb + i*d_si + h*d_sh;
 * q, out: [Br, Hq, Mq, d];  prefix_idx: [Br, Hkv, kp] or NULL (dense prefix);
 * pre_len: [Br] visible prefix rows per branch (its fork position) or NULL (all P);
 * suf_len: [Br] suffix rows per branch or NULL (L_b = off[b+1] - off[b]).
 */
void oracle_shared_prefix(const uint16_t* pk, const uint16_t* pv, int64_t p_sh, int64_t p_st, int P,
                          const uint16_t* sk, const uint16_t* sv, int64_t s_sh, int64_t s_st,
                          const int32_t* off, const uint16_t* dk, const uint16_t* dv, int64_t d_sb,
                          int64_t d_si, int64_t d_sh, const uint16_t* q, int Br, int Hkv, int Hq,
                          int Mq, int d, const int32_t* prefix_idx, int kp, const int32_t* pre_len,
                          const int32_t* suf_len, double scale, double* out)
{
    prefix_ctx c = {pk, pv, p_sh, p_st, P, sk, sv, s_sh, s_st, off, dk, dv, d_sb, d_si, d_sh,
                    q, Br, Hkv, Hq, Mq, d, prefix_idx, kp, pre_len, suf_len, scale, out};
    int nmax = 0;
    for (int b = 0; b < Br; ++b) {
        int np = prefix_idx ? kp : (pre_len ? pre_len[b] : P);
        int n = np + (suf_len ? suf_len[b] : off[b + 1] - off[b]) + Mq;
        if (n > nmax) nmax = n;
    }
    parallel_for(Br * Hkv, prefix_item, &c, (size_t)nmax + 2 * (size_t)d);
}
