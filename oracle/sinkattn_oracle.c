/*
 * sinkattn_oracle.c -- the oracle for the sink-bias attention forward pass.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may load this library.  It
 * shares no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it.
 *
 * What it computes is the plain definition of the attention layer in the
 * "MiMo-V2-Flash Technical Report" (full Chinese translation,
 * garden.houmin.site/digest/mimo-v2-flash), evaluated directly in fp64:
 *
 *   §2.1, Table 1 and the paragraph after it: grouped-query attention, QK head
 *       dim 192, V head dim 128, RoPE applied to the first 64 dims of q and k
 *       only; SWA layers use a 128-token window, GA layers attend globally.
 *   §2.2, eq. (1): a_ij = q_i . k_j / sqrt(d)
 *   §2.2, eq. (2): s_ij = exp(a_ij - m_i) / (exp(sink - m_i) + sum_j' exp(a_ij' - m_i)),
 *                  m_i = max(max_j a_ij, sink), one learnable sink per head
 *   §2.2, eq. (3): o_i = sum_j s_ij v_j
 *   §3.2 "long-context extension": RoPE base 10,000 for SWA, 640,000 then
 *       5,000,000 for GA.
 *
 * There is no tiling, no online softmax and no reordering beyond the order in
 * which the definition is written: (1) convert every input to fp64, (2) rotate
 * q and k, (3) form every logit of a row, (4) take the max including the sink,
 * (5) the denominator, (6) the weighted sum of values and the log-sum-exp.
 *
 * Readings taken where the pages are silent:
 *   - d in eq. (1) is the QK head dim; callers pass scale = 1/sqrt(192).
 *   - one sink per query head, in the units of the scaled logit, with no value
 *     vector (eq. (3) sums over keys only).
 *   - window W: key j is visible to query i iff i - W < j <= i (W = 0: global).
 *   - RoPE: theta_t = base^(-2t/drot) for pair t; pair t is dims (2t, 2t+1)
 *     (style 0, RoFormer) or (t, t + drot/2) (style 1); positions are 0-based
 *     per sequence in prefill and the absolute cache index in decode; the
 *     decode K cache holds raw (unrotated) keys unless cfg->k_rotated says it
 *     holds keys already rotated at their positions (then only q is rotated).
 *   - log-sum-exp output: lse_i = m_i + ln(exp(sink - m_i) + sum_j exp(a_ij - m_i)),
 *     natural log, sink included.
 *   - an empty visible set gives o = 0, lse = sink.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

typedef struct {
    int32_t dqk;        /* head dim of q and k */
    int32_t dv;         /* head dim of v */
    int32_t drot;       /* rotated dims at the start of q and k; 0 = no RoPE */
    int32_t rope_style; /* 0: pairs (2t, 2t+1); 1: pairs (t, t + drot/2) */
    int32_t window;     /* 0 = global causal; W > 0: i - W < j <= i */
    int32_t dtype;      /* 0: q/k/v hold bf16 bit patterns; 1: q/k/v hold fp64 */
    double rope_base;   /* <= 0 disables RoPE */
    double scale;       /* the factor applied to q.k (1/sqrt(d) in eq. (1)) */
    int32_t k_rotated;  /* 1: the keys passed in are already rotated at their own
                           positions (a cache that stores rotated keys); only q is
                           rotated here */
} oracle_cfg;

/* bf16 is the top half of an IEEE binary32; every bf16 value is exact in fp64. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void *base, int32_t dtype, int64_t idx)
{
    if (dtype == 1) return ((const double *)base)[idx];
    return oracle_bf16_to_f64(((const uint16_t *)base)[idx]);
}

/* Rotary position embedding on the first drot dims of a d-vector (§2.1:
 * "RoPE is applied only to the first 64 dims of query and key"; RoFormer
 * rotation of each dim pair by pos * theta_t). */
void oracle_rope(const double *x, int32_t d, int32_t drot, int32_t style,
                 double base, double pos, double *y)
{
    for (int32_t e = 0; e < d; ++e) y[e] = x[e];
    if (drot <= 0 || base <= 0.0) return;
    const int32_t half = drot / 2;
    for (int32_t t = 0; t < half; ++t) {
        const double theta = pow(base, -2.0 * (double)t / (double)drot);
        const double phi = pos * theta;
        const double c = cos(phi), s = sin(phi);
        const int32_t ia = style == 0 ? 2 * t : t;
        const int32_t ib = style == 0 ? 2 * t + 1 : t + half;
        y[ia] = x[ia] * c - x[ib] * s;
        y[ib] = x[ia] * s + x[ib] * c;
    }
}

/* The rotation above applied to n rows of d values, row r at position pos[r]
 * (x and y are [n, d] fp64; used to build caches that hold rotated keys). */
void oracle_rope_rows(const double *x, int64_t n, int32_t d, int32_t drot, int32_t style,
                      double base, const double *pos, double *y)
{
    for (int64_t r = 0; r < n; ++r)
        oracle_rope(x + r * d, d, drot, style, base, pos[r], y + r * d);
}

/* One requested output row: which query, which head, which keys it sees. */
typedef struct {
    int64_t slot;    /* index into out/lse */
    int64_t q_off;   /* element offset of the query vector */
    int64_t kv_base; /* storage row of key position 0 for this sequence */
    int64_t lo, hi;  /* visible key positions [lo, hi]; empty if lo > hi */
    double pos;      /* query position for RoPE */
    int32_t head;    /* query head h */
    int32_t group;   /* kv head g = h / (Hq / Hkv) */
    int64_t gkey;    /* grouping key: (sequence, kv head) */
} row_t;

static int cmp_row(const void *a, const void *b)
{
    const row_t *ra = (const row_t *)a, *rb = (const row_t *)b;
    if (ra->gkey != rb->gkey) return ra->gkey < rb->gkey ? -1 : 1;
    return ra->slot < rb->slot ? -1 : (ra->slot > rb->slot);
}

/* Evaluate eqs. (1)-(3) for every row of one (sequence, kv head) group.
 * k_stride/v_stride: elements between consecutive key rows of this kv head. */
static int run_group(row_t *rows, int64_t n, const void *q, const void *k,
                     const void *v, const float *sink, int32_t Hkv,
                     const oracle_cfg *cfg, double *out, double *lse, int nthreads)
{
    const int32_t dqk = cfg->dqk, dv = cfg->dv;
    int64_t lo = INT64_MAX, hi = INT64_MIN;
    for (int64_t r = 0; r < n; ++r) {
        if (rows[r].lo > rows[r].hi) continue;
        if (rows[r].lo < lo) lo = rows[r].lo;
        if (rows[r].hi > hi) hi = rows[r].hi;
    }
    const int64_t nk = hi >= lo ? hi - lo + 1 : 0;
    const int32_t g = rows[0].group;
    const int64_t kv_base = rows[0].kv_base;

    /* Step (2) for the keys: every key this group can see, rotated once at its
     * own position (the definition rotates each k_j before any product). */
    double *kr = NULL;
    if (nk > 0) {
        kr = (double *)malloc((size_t)nk * (size_t)dqk * sizeof(double));
        if (!kr) return -1;
    }
    int err = 0;
#pragma omp parallel num_threads(nthreads)
    {
        double *tmp = (double *)malloc((size_t)dqk * sizeof(double));
        if (!tmp) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t j = 0; j < nk; ++j) {
            if (!tmp) continue;
            const int64_t off = ((kv_base + lo + j) * Hkv + g) * (int64_t)dqk;
            for (int32_t e = 0; e < dqk; ++e) tmp[e] = load(k, cfg->dtype, off + e);
            if (cfg->k_rotated)
                memcpy(kr + j * dqk, tmp, (size_t)dqk * sizeof(double));
            else
                oracle_rope(tmp, dqk, cfg->drot, cfg->rope_style, cfg->rope_base,
                            (double)(lo + j), kr + j * dqk);
        }
        free(tmp);
    }
    if (err) { free(kr); return -1; }

#pragma omp parallel num_threads(nthreads)
    {
        double *qx = (double *)malloc((size_t)dqk * sizeof(double));
        double *qr = (double *)malloc((size_t)dqk * sizeof(double));
        double *a = (double *)malloc((size_t)(nk > 0 ? nk : 1) * sizeof(double));
        double *o = (double *)malloc((size_t)dv * sizeof(double));
        if (!qx || !qr || !a || !o) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            if (!qx || !qr || !a || !o) continue;
            const row_t *rw = &rows[r];
            const double sk = (double)sink[rw->head];
            /* (1) inputs to fp64, (2) rotate q at its own position */
            for (int32_t e = 0; e < dqk; ++e) qx[e] = load(q, cfg->dtype, rw->q_off + e);
            oracle_rope(qx, dqk, cfg->drot, cfg->rope_style, cfg->rope_base, rw->pos, qr);
            /* (3) eq. (1): every visible logit */
            const int64_t cnt = rw->lo <= rw->hi ? rw->hi - rw->lo + 1 : 0;
            for (int64_t j = 0; j < cnt; ++j) {
                const double *kj = kr + (rw->lo - lo + j) * dqk;
                double acc = 0.0;
                for (int32_t e = 0; e < dqk; ++e) acc += qr[e] * kj[e];
                a[j] = acc * cfg->scale;
            }
            /* (4) eq. (2): m_i = max(max_j a_ij, sink) */
            double m = sk;
            for (int64_t j = 0; j < cnt; ++j) if (a[j] > m) m = a[j];
            for (int32_t e = 0; e < dv; ++e) o[e] = 0.0;
            if (m == -INFINITY) {
                /* no visible key and sink = -inf: the empty sum */
                for (int32_t e = 0; e < dv; ++e) out[rw->slot * dv + e] = 0.0;
                lse[rw->slot] = -INFINITY;
                continue;
            }
            /* (5) the denominator: the sink term once, then every visible key */
            double den = exp(sk - m);
            for (int64_t j = 0; j < cnt; ++j) den += exp(a[j] - m);
            /* (6) eq. (3): o_i = sum_j s_ij v_j, and the log-sum-exp */
            for (int64_t j = 0; j < cnt; ++j) {
                const double s = exp(a[j] - m) / den;
                const int64_t voff = ((kv_base + rw->lo + j) * Hkv + rw->group) * (int64_t)dv;
                for (int32_t e = 0; e < dv; ++e) o[e] += s * load(v, cfg->dtype, voff + e);
            }
            for (int32_t e = 0; e < dv; ++e) out[rw->slot * dv + e] = o[e];
            lse[rw->slot] = m + log(den);
        }
        free(qx); free(qr); free(a); free(o);
    }
    free(kr);
    return err ? -1 : 0;
}

static int run_rows(row_t *rows, int64_t n, const void *q, const void *k, const void *v,
                    const float *sink, int32_t Hkv, const oracle_cfg *cfg,
                    double *out, double *lse, int nthreads)
{
    qsort(rows, (size_t)n, sizeof(row_t), cmp_row);
    int64_t i = 0;
    while (i < n) {
        int64_t e = i;
        while (e < n && rows[e].gkey == rows[i].gkey) ++e;
        if (run_group(rows + i, e - i, q, k, v, sink, Hkv, cfg, out, lse, nthreads)) return -1;
        i = e;
    }
    return 0;
}

static int check_cfg(const oracle_cfg *cfg, int32_t Hq, int32_t Hkv)
{
    if (!cfg || cfg->dqk <= 0 || cfg->dv <= 0 || cfg->window < 0) return -2;
    if (cfg->drot < 0 || cfg->drot > cfg->dqk || (cfg->drot & 1)) return -2;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return -2;
    return 0;
}

/* Prefill over packed variable-length sequences.
 * q [total, Hq, dqk], k [total, Hkv, dqk], v [total, Hkv, dv], sink [Hq];
 * cu_seqlens [batch+1] (host), sequence b holds tokens cu[b] .. cu[b+1]-1 at
 * positions 0 .. L_b-1.  rows: flat indices token*Hq + h to evaluate, or NULL
 * for every (token, head) in order.  out [nrows, dv], lse [nrows].
 * Returns 0, -1 on allocation failure, -2 on bad arguments. */
int oracle_prefill(const void *q, const void *k, const void *v, const float *sink,
                   const int32_t *cu_seqlens, int32_t batch, int32_t Hq, int32_t Hkv,
                   const oracle_cfg *cfg, const int64_t *rows, int64_t nrows,
                   double *out, double *lse, int nthreads)
{
    if (check_cfg(cfg, Hq, Hkv) || batch < 0) return -2;
    const int64_t total = cu_seqlens[batch];
    const int64_t n = rows ? nrows : total * Hq;
    if (n == 0) return 0;
    row_t *rl = (row_t *)malloc((size_t)n * sizeof(row_t));
    if (!rl) return -1;
    const int32_t G = Hq / Hkv;
    for (int64_t r = 0; r < n; ++r) {
        const int64_t flat = rows ? rows[r] : r;
        const int64_t tok = flat / Hq;
        const int32_t h = (int32_t)(flat % Hq);
        if (flat < 0 || tok >= total) { free(rl); return -2; }
        int32_t b = 0;
        while (b + 1 < batch && cu_seqlens[b + 1] <= tok) ++b;
        const int64_t p = tok - cu_seqlens[b];
        row_t *w = &rl[r];
        w->slot = r;
        w->q_off = flat * cfg->dqk;
        w->kv_base = cu_seqlens[b];
        w->hi = p;
        w->lo = cfg->window > 0 ? (p - cfg->window + 1 > 0 ? p - cfg->window + 1 : 0) : 0;
        w->pos = (double)p;
        w->head = h;
        w->group = h / G;
        w->gkey = (int64_t)b * Hkv + w->group;
    }
    const int rc = run_rows(rl, n, q, k, v, sink, Hkv, cfg, out, lse, nthreads);
    free(rl);
    return rc;
}

/* Multi-token (MTP-verify) decode against a KV cache.
 * q [B, T, Hq, dqk]; kcache [B, S_cap, Hkv, dqk] (raw, unrotated keys);
 * vcache [B, S_cap, Hkv, dv]; seqlens [B] (host) counts cached tokens
 * including the T new ones, so query t of sequence b sits at position
 * seqlens[b] - T + t and sees cache positions j <= that position (causal
 * among the T drafts) and, with a window, j > position - W.
 * rows: flat indices (b*T + t)*Hq + h, or NULL for all.  Returns as above. */
int oracle_decode(const void *q, const void *kcache, const void *vcache,
                  const int32_t *seqlens, const float *sink, int32_t B, int32_t T,
                  int32_t S_cap, int32_t Hq, int32_t Hkv, const oracle_cfg *cfg,
                  const int64_t *rows, int64_t nrows, double *out, double *lse,
                  int nthreads)
{
    if (check_cfg(cfg, Hq, Hkv) || B < 0 || T < 0 || S_cap < 0) return -2;
    const int64_t n = rows ? nrows : (int64_t)B * T * Hq;
    if (n == 0) return 0;
    row_t *rl = (row_t *)malloc((size_t)n * sizeof(row_t));
    if (!rl) return -1;
    const int32_t G = Hq / Hkv;
    for (int64_t r = 0; r < n; ++r) {
        const int64_t flat = rows ? rows[r] : r;
        const int64_t bt = flat / Hq;
        const int32_t h = (int32_t)(flat % Hq);
        const int32_t b = (int32_t)(bt / (T > 0 ? T : 1));
        const int32_t t = (int32_t)(bt % (T > 0 ? T : 1));
        if (flat < 0 || b >= B || seqlens[b] > S_cap) { free(rl); return -2; }
        const int64_t p = (int64_t)seqlens[b] - T + t;
        row_t *w = &rl[r];
        w->slot = r;
        w->q_off = flat * cfg->dqk;
        w->kv_base = (int64_t)b * S_cap;
        w->hi = p < (int64_t)seqlens[b] - 1 ? p : (int64_t)seqlens[b] - 1;
        w->lo = cfg->window > 0 ? (p - cfg->window + 1 > 0 ? p - cfg->window + 1 : 0) : 0;
        if (p < 0) { w->lo = 1; w->hi = 0; }
        w->pos = (double)p;
        w->head = h;
        w->group = h / G;
        w->gkey = (int64_t)b * Hkv + w->group;
    }
    const int rc = run_rows(rl, n, q, kcache, vcache, sink, Hkv, cfg, out, lse, nthreads);
    free(rl);
    return rc;
}

int oracle_max_threads(void) { return omp_get_max_threads(); }

/* The inverse rotation: R(pos)^T y, i.e. each dim pair turned by -pos*theta_t.
 * A gradient with respect to a rotated vector comes back to the raw vector's
 * coordinates this way (the rotation is orthogonal). */
static void rope_transpose(const double *y, int32_t d, int32_t drot, int32_t style,
                           double base, double pos, double *x)
{
    oracle_rope(y, d, drot, style, base, -pos, x);
}

/* Backward pass of the prefill forward above, for the loss L = sum_i dO_i . o_i,
 * by the chain rule through eqs. (1)-(3) (the pages give the forward only; the
 * gradient is the plain derivative of that definition):
 *   s_ij = exp(a_ij - lse_i), s_sink,i = exp(sink_h - lse_i)      (eq. (2))
 *   D_i = dO_i . o_i,  dP_ij = dO_i . v_j
 *   dL/dv_j    += s_ij dO_i                                         (eq. (3))
 *   dL/da_ij    = s_ij (dP_ij - D_i)                                (eq. (2))
 *   dL/dq~_i   += scale * dL/da_ij k~_j,  dL/dk~_j += scale * dL/da_ij q~_i  (eq. (1))
 *   dL/dsink_h += -s_sink,i D_i        (the sink's term in the denominator)
 * where q~, k~ are the rotated vectors; dq, dk are turned back by R^T.
 * Inputs as oracle_prefill, plus dout [total, Hq, dv] (cfg->dtype).  Outputs
 * dq [total, Hq, dqk], dk [total, Hkv, dqk], dv [total, Hkv, dv], dsink [Hq],
 * all fp64 and fully written.  Returns 0, -1 on allocation failure, -2 on bad
 * arguments.  Parallel over (sequence, kv head) groups; each group's rows are
 * walked in order, so the result does not depend on the thread count except
 * for the order of dsink's per-group sums (added in group order). */
int oracle_prefill_backward(const void *q, const void *k, const void *v, const float *sink,
                            const int32_t *cu_seqlens, int32_t batch, int32_t Hq,
                            int32_t Hkv, const oracle_cfg *cfg, const void *dout,
                            double *dq, double *dk, double *dvo, double *dsink, int nthreads)
{
    if (check_cfg(cfg, Hq, Hkv) || batch < 0) return -2;
    const int64_t total = cu_seqlens[batch];
    const int32_t dqk = cfg->dqk, dv = cfg->dv, G = Hq / Hkv;
    memset(dq, 0, (size_t)(total * Hq * dqk) * sizeof(double));
    memset(dk, 0, (size_t)(total * Hkv * dqk) * sizeof(double));
    memset(dvo, 0, (size_t)(total * Hkv * dv) * sizeof(double));
    for (int32_t h = 0; h < Hq; ++h) dsink[h] = 0.0;
    const int64_t ngroups = (int64_t)batch * Hkv;
    double *ds_part = (double *)calloc((size_t)(ngroups > 0 ? ngroups : 1) * (size_t)G, sizeof(double));
    if (!ds_part) return -1;
    int err = 0;
#pragma omp parallel num_threads(nthreads)
    {
        double *qr = (double *)malloc((size_t)dqk * sizeof(double));
        double *tmp = (double *)malloc((size_t)dqk * sizeof(double));
        double *dqr = (double *)malloc((size_t)dqk * sizeof(double));
        double *o = (double *)malloc((size_t)dv * sizeof(double));
        double *dO = (double *)malloc((size_t)dv * sizeof(double));
        if (!qr || !tmp || !dqr || !o || !dO) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t gi = 0; gi < ngroups; ++gi) {
            if (!qr || !tmp || !dqr || !o || !dO) continue;
            const int32_t b = (int32_t)(gi / Hkv), g = (int32_t)(gi % Hkv);
            const int64_t s0 = cu_seqlens[b], L = cu_seqlens[b + 1] - s0;
            if (L <= 0) continue;
            /* the rotated keys of this sequence and kv head, and their gradients */
            double *kr = (double *)malloc((size_t)L * (size_t)dqk * sizeof(double));
            double *dkr = (double *)calloc((size_t)L * (size_t)dqk, sizeof(double));
            double *a = (double *)malloc((size_t)L * sizeof(double));
            if (!kr || !dkr || !a) {
                free(kr); free(dkr); free(a);
#pragma omp atomic write
                err = 1;
                continue;
            }
            for (int64_t j = 0; j < L; ++j) {
                const int64_t off = ((s0 + j) * Hkv + g) * (int64_t)dqk;
                for (int32_t e = 0; e < dqk; ++e) tmp[e] = load(k, cfg->dtype, off + e);
                oracle_rope(tmp, dqk, cfg->drot, cfg->rope_style, cfg->rope_base, (double)j,
                            kr + j * dqk);
            }
            for (int64_t p = 0; p < L; ++p) {
                const int64_t lo = cfg->window > 0 ? (p - cfg->window + 1 > 0 ? p - cfg->window + 1 : 0) : 0;
                for (int32_t hh = 0; hh < G; ++hh) {
                    const int32_t h = g * G + hh;
                    const double sk = (double)sink[h];
                    const int64_t row = (s0 + p) * Hq + h;
                    for (int32_t e = 0; e < dqk; ++e) tmp[e] = load(q, cfg->dtype, row * dqk + e);
                    oracle_rope(tmp, dqk, cfg->drot, cfg->rope_style, cfg->rope_base, (double)p, qr);
                    for (int32_t e = 0; e < dv; ++e) dO[e] = load(dout, cfg->dtype, row * dv + e);
                    /* forward again: logits, max with the sink, denominator, o */
                    double m = sk;
                    for (int64_t j = lo; j <= p; ++j) {
                        double acc = 0.0;
                        for (int32_t e = 0; e < dqk; ++e) acc += qr[e] * kr[j * dqk + e];
                        a[j] = acc * cfg->scale;
                        if (a[j] > m) m = a[j];
                    }
                    if (m == -INFINITY) continue; /* nothing visible, no sink: o = 0, no gradient */
                    double den = exp(sk - m);
                    for (int64_t j = lo; j <= p; ++j) den += exp(a[j] - m);
                    const double lse_i = m + log(den);
                    for (int32_t e = 0; e < dv; ++e) o[e] = 0.0;
                    for (int64_t j = lo; j <= p; ++j) {
                        const double s = exp(a[j] - lse_i);
                        const int64_t voff = ((s0 + j) * Hkv + g) * (int64_t)dv;
                        for (int32_t e = 0; e < dv; ++e) o[e] += s * load(v, cfg->dtype, voff + e);
                    }
                    double D = 0.0;
                    for (int32_t e = 0; e < dv; ++e) D += dO[e] * o[e];
                    /* the sink's gradient, per head of this group */
                    ds_part[gi * G + hh] += -exp(sk - lse_i) * D;
                    for (int32_t e = 0; e < dqk; ++e) dqr[e] = 0.0;
                    for (int64_t j = lo; j <= p; ++j) {
                        const double s = exp(a[j] - lse_i);
                        const int64_t voff = ((s0 + j) * Hkv + g) * (int64_t)dv;
                        double dP = 0.0;
                        for (int32_t e = 0; e < dv; ++e) dP += dO[e] * load(v, cfg->dtype, voff + e);
                        for (int32_t e = 0; e < dv; ++e) dvo[voff + e] += s * dO[e];
                        const double dS = s * (dP - D);
                        for (int32_t e = 0; e < dqk; ++e) {
                            dqr[e] += cfg->scale * dS * kr[j * dqk + e];
                            dkr[j * dqk + e] += cfg->scale * dS * qr[e];
                        }
                    }
                    rope_transpose(dqr, dqk, cfg->drot, cfg->rope_style, cfg->rope_base, (double)p,
                                   dq + row * dqk);
                }
            }
            for (int64_t j = 0; j < L; ++j)
                rope_transpose(dkr + j * dqk, dqk, cfg->drot, cfg->rope_style, cfg->rope_base,
                               (double)j, dk + ((s0 + j) * Hkv + g) * (int64_t)dqk);
            free(kr); free(dkr); free(a);
        }
        free(qr); free(tmp); free(dqr); free(o); free(dO);
    }
    /* dsink: the per-group sums in group order */
    for (int64_t gi = 0; gi < ngroups; ++gi)
        for (int32_t hh = 0; hh < G; ++hh) dsink[(gi % Hkv) * G + hh] += ds_part[gi * G + hh];
    free(ds_part);
    return err ? -1 : 0;
}
