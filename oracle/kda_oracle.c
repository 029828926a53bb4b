/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for the packed (varlen) Kimi
 * Delta Attention forward.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline use it. It shares no code, header, table or helper with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Sources (web pages):
 *   [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss"
 *              方案 §1 "segment_ids → cu_seqlens 转换" (conversion and its
 *              worked examples), 方案 §3 "ShortConvolution segment 边界 mask".
 *   [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）"
 *              背景 "KDA 状态泄漏问题" (the recurrence), §3.1.1 API contract
 *              (segment-id reset semantics, 0 = padding).
 *   [Drill]    "Drill: Sequence Packing from scratch", 数学 / The math
 *              (cu_seqlens definition, doc(s)).
 *
 * Every floating-point quantity is double. Inputs arrive already widened from
 * their stored dtype. Nothing here is blocked, fused or reordered beyond the
 * definitions written out below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* O1: segment ids -> padded cu_seqlens                                      */
/* ------------------------------------------------------------------------ */
/*
 * [RFC-0025] 方案 §1: a position starts a segment when its id is non-zero and
 * differs from the previous position's id; padding (id 0) never starts one.
 * cu_seqlens has max_segs+1 entries: cu[0] = 0, cu[i] = end of segment i in
 * the cumulative (FLA) convention, where the end of a segment is the start of
 * the next one; segments beyond the real count ("phantoms") have zero length.
 * If there are more real segments than max_segs, the last slot ends at B*T
 * and swallows the overflow (the page warns that this leaks across documents).
 *
 * Two readings are parameters so that the page's own behaviour can be
 * compared with the amended one:
 *   force_row_starts = 1: position p with p % T == 0 also starts a segment
 *     ([RFC-0026] §3.1.1: t = 0 is always a new segment in every row);
 *     0: only p == 0 does (the page's flat scan over [B*T]).
 *   end_rule = 1: the end of the last real segment is one past the last
 *     non-padding position; 0: the number of non-padding positions (the
 *     page's count, which equals the former when padding only trails).
 *
 * Writes cu[0..max_segs] and *n_segs. Returns 0, or -1 on bad arguments.
 */
int oracle_cu_seqlens(const int32_t *seg, int64_t B, int64_t T, int32_t max_segs,
                      int force_row_starts, int end_rule,
                      int32_t *cu, int64_t *n_segs)
{
    if (!seg || !cu || !n_segs || B < 0 || T < 0 || max_segs < 1)
        return -1;
    const int64_t N = B * T;
    int64_t count = 0, last_real = -1, n_real = 0;
    /* starts[r] = position of the (r+1)-th segment start, for r < max_segs+1 */
    int64_t *starts = (int64_t *)malloc(sizeof(int64_t) * ((size_t)max_segs + 1));
    if (!starts)
        return -1;
    for (int64_t p = 0; p < N; ++p) {
        const int is_row_start = force_row_starts ? (p % T == 0) : (p == 0);
        const int is_start = seg[p] != 0 && (is_row_start || seg[p] != seg[p - 1]);
        if (seg[p] != 0) {
            last_real = p;
            n_real += 1;
        }
        if (is_start) {
            if (count < (int64_t)max_segs + 1)
                starts[count] = p;
            count += 1;
        }
    }
    const int64_t last_end = end_rule ? (last_real + 1) : n_real;
    cu[0] = 0;
    for (int64_t i = 1; i <= max_segs; ++i) {
        int64_t e;
        if (i < count)
            e = (i < max_segs) ? starts[i] : N; /* start of segment i+1, or the overflow slot */
        else
            e = last_end;                        /* last real segment, then phantoms */
        cu[i] = (int32_t)e;
    }
    *n_segs = count;
    free(starts);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O2: segment-masked causal depthwise short convolution                      */
/* ------------------------------------------------------------------------ */
/*
 * [RFC-0025] 方案 §3: y[b,t,f] = sum_{j=0}^{K-1} w[j,f] * x[b,t-j,f], where a
 * tap contributes only if t-j >= 0 (the left padding holds x = 0, id 0) and
 * the source id equals the destination id. Tap j multiplies the token j steps
 * back, so w[0] weighs the current token. With seg == NULL no id test is made.
 * The sum is exact-order fp64; the caller rounds once to the output dtype.
 * x, y: [B, T, F]; w: [K, F].
 */
int oracle_short_conv(const double *x, const double *w, const int32_t *seg,
                      int64_t B, int64_t T, int64_t F, int32_t K, double *y)
{
    if (!x || !w || !y || B < 0 || T < 0 || F < 0 || K < 1)
        return -1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t f = 0; f < F; ++f) {
                double acc = 0.0;
                for (int32_t j = 0; j < K; ++j) {
                    const int64_t s = t - j;
                    if (s < 0)
                        continue;
                    if (seg && seg[b * T + s] != seg[b * T + t])
                        continue;
                    acc += w[(int64_t)j * F + f] * x[(b * T + s) * F + f];
                }
                y[(b * T + t) * F + f] = acc;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O3: token-by-token KDA recurrence                                          */
/* ------------------------------------------------------------------------ */
/*
 * [RFC-0026] 背景 "KDA 状态泄漏问题": per head, with S in R^{Dk x Dv},
 *     S'_t = S_{t-1} * exp(g_t)            (g_t in R^{Dk} scales the rows)
 *     S_t  = S'_t + beta_t * k_t (x) v_t
 * read out as o_t = scale * S_t^T q_t. [RFC-0026] §3.1.1: S is reset to zero
 * where segment_ids[:, t] != segment_ids[:, t-1] and at t = 0 of every row;
 * id 0 is padding: it contributes nothing and its output is 0 (the state is
 * cleared there too; the next real token is a segment start anyway).
 * seg == NULL: every row is one segment.
 *
 * Layouts (flattened batch): q, k, g: [B*T, H, Dk]; v, o: [B*T, H, Dv];
 * beta: [B*T, H]; seg: [B, T].
 */
typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int32_t *seg;
    int64_t B, T, H, Dk, Dv;
    double scale;
    double *o;
    /* per-segment state, [n_state, H, Dk, Dv]; either may be NULL */
    const double *init;
    double *fin;
    int64_t n_state;
    /* work units: (row, head, first token, one-past-last token, segment rank) */
    const int64_t *units;
    int64_t n_units;
    int64_t next; /* shared counter */
    int delta;    /* 1: the delta-rule update (oracle_kda_fwd_delta) */
} kda_job_t;

static void run_unit(const kda_job_t *J, int64_t b, int64_t h, int64_t t0, int64_t t1,
                     int64_t r, double *S, double *W)
{
    const int64_t H = J->H, Dk = J->Dk, Dv = J->Dv;
    /* the segment's state before its first token: its initial state, or zero */
    const int64_t slot = (r * H + h) * Dk * Dv;
    if (J->init && r < J->n_state)
        memcpy(S, J->init + slot, sizeof(double) * (size_t)(Dk * Dv));
    else
        memset(S, 0, sizeof(double) * (size_t)(Dk * Dv));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t p = b * J->T + t;
        const double *qt = J->q + (p * H + h) * Dk;
        const double *kt = J->k + (p * H + h) * Dk;
        const double *gt = J->g + (p * H + h) * Dk;
        const double *vt = J->v + (p * H + h) * Dv;
        const double bt = J->beta[p * H + h];
        double *ot = J->o + (p * H + h) * Dv;
        if (!J->delta) {
            for (int64_t i = 0; i < Dk; ++i) {
                const double decay = exp(gt[i]);
                const double bk = bt * kt[i];
                double *row = S + i * Dv;
                for (int64_t j = 0; j < Dv; ++j)
                    row[j] = row[j] * decay + bk * vt[j];
            }
        } else {
            /* S' = S_{t-1} exp(g_t); u = S'^T k_t; S_t = S' + beta_t k_t (v_t - u)^T */
            for (int64_t i = 0; i < Dk; ++i) {
                const double ei = exp(gt[i]);
                double *row = S + i * Dv;
                for (int64_t j = 0; j < Dv; ++j)
                    row[j] *= ei;
            }
            for (int64_t j = 0; j < Dv; ++j) {
                double u = 0.0;
                for (int64_t i = 0; i < Dk; ++i)
                    u += S[i * Dv + j] * kt[i];
                W[j] = vt[j] - u;
            }
            for (int64_t i = 0; i < Dk; ++i) {
                const double wk = bt * kt[i];
                double *row = S + i * Dv;
                for (int64_t j = 0; j < Dv; ++j)
                    row[j] += wk * W[j];
            }
        }
        for (int64_t j = 0; j < Dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < Dk; ++i)
                acc += S[i * Dv + j] * qt[i];
            ot[j] = J->scale * acc;
        }
    }
    /* the segment's state after its last token */
    if (J->fin && r < J->n_state)
        memcpy(J->fin + slot, S, sizeof(double) * (size_t)(Dk * Dv));
}

static void *kda_worker(void *arg)
{
    kda_job_t *J = (kda_job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->Dk * J->Dv + J->Dv));
    if (!S)
        return NULL;
    double *W = S + J->Dk * J->Dv;     /* the delta rule's v_t - S'^T k_t */
    for (;;) {
        const int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (u >= J->n_units)
            break;
        const int64_t *U = J->units + 5 * u;
        run_unit(J, U[0], U[1], U[2], U[3], U[4], S, W);
    }
    free(S);
    return NULL;
}

/*
 * The (segment, head) work units of a packed batch: every row split into its
 * segments (maximal runs of equal non-zero ids, cut at row starts), each as
 * (row, head, first token, one-past-last token, segment rank), ranks counted in
 * flattened token order. Returns a malloc'd array of 5 * n_units entries, or
 * NULL if out of memory.
 */
static int64_t *segment_units(const int32_t *seg, int64_t B, int64_t T, int64_t H,
                              int64_t *n_units_out)
{
    /* count segments */
    int64_t n_seg = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t) {
            const int64_t p = b * T + t;
            const int32_t s = seg ? seg[p] : 1;
            if (s != 0 && (t == 0 || (seg ? seg[p - 1] : 1) != s))
                n_seg += 1;
        }
    int64_t *units = (int64_t *)malloc(sizeof(int64_t) * 5 * (size_t)(n_seg * H + 1));
    if (!units)
        return NULL;
    int64_t n_units = 0;
    int64_t rank = 0; /* segments in flattened token order */
    for (int64_t b = 0; b < B; ++b) {
        int64_t t = 0;
        while (t < T) {
            const int64_t p = b * T + t;
            const int32_t s = seg ? seg[p] : 1;
            if (s == 0) {
                ++t;
                continue;
            }
            int64_t e = t + 1;
            while (e < T && (seg ? seg[b * T + e] : 1) == s)
                ++e;
            for (int64_t h = 0; h < H; ++h) {
                units[5 * n_units + 0] = b;
                units[5 * n_units + 1] = h;
                units[5 * n_units + 2] = t;
                units[5 * n_units + 3] = e;
                units[5 * n_units + 4] = rank;
                ++n_units;
            }
            ++rank;
            t = e;
        }
    }
    *n_units_out = n_units;
    return units;
}

/*
 * Splits every row into its segments (maximal runs of equal non-zero ids,
 * cut at row starts), zeroes o, and runs one independent recurrence per
 * (segment, head) on `n_threads` threads. Starting each segment from S = 0
 * is exactly the reset rule above.
 *
 * Per-segment state ([RFC-0026] 方案, the kernel kwargs initial_state and
 * output_final_state of the FLA chunk_kda call; shapes [n_segments, H, Dk, Dv]):
 * segment r, counted in flattened token order, starts from init[r] instead of
 * zero when init is given and r < n_state, and its state after its last token
 * is written to fin[r] when fin is given and r < n_state. With init = NULL this
 * is the reset rule above. Returns 0, or -1 on bad arguments.
 */
static int kda_fwd_run(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const int32_t *seg, int64_t B, int64_t T, int64_t H,
                       int64_t Dk, int64_t Dv, double scale, const double *init, double *fin,
                       int64_t n_state, double *o, int n_threads, int delta)
{
    if (!q || !k || !v || !g || !beta || !o || B < 0 || T < 0 || H < 1 || Dk < 1 || Dv < 1 ||
        n_state < 0)
        return -1;
    const int64_t N = B * T;
    memset(o, 0, sizeof(double) * (size_t)(N * H * Dv));
    int64_t n_units = 0;
    int64_t *units = segment_units(seg, B, T, H, &n_units);
    if (!units)
        return -1;
    kda_job_t J = {q, k, v, g, beta, seg, B, T, H, Dk, Dv, scale, o,
                   init, fin, n_state, units, n_units, 0, delta};
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 256)
        n_threads = 256;
    if (n_threads == 1) {
        kda_worker(&J);
    } else {
        pthread_t th[256];
        int started = 0;
        for (int i = 0; i < n_threads; ++i)
            if (pthread_create(&th[i], NULL, kda_worker, &J) == 0)
                ++started;
        if (started == 0)
            kda_worker(&J);
        for (int i = 0; i < started; ++i)
            pthread_join(th[i], NULL);
    }
    free(units);
    return 0;
}

int oracle_kda_fwd_state(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const int32_t *seg, int64_t B, int64_t T, int64_t H,
                         int64_t Dk, int64_t Dv, double scale, const double *init, double *fin,
                         int64_t n_state, double *o, int n_threads)
{
    return kda_fwd_run(q, k, v, g, beta, seg, B, T, H, Dk, Dv, scale, init, fin, n_state, o,
                       n_threads, 0);
}

/* The recurrence with every segment starting from zero and no state written. */
int oracle_kda_fwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int32_t *seg, int64_t B, int64_t T, int64_t H,
                   int64_t Dk, int64_t Dv, double scale, double *o, int n_threads)
{
    return oracle_kda_fwd_state(q, k, v, g, beta, seg, B, T, H, Dk, Dv, scale, NULL, NULL, 0, o,
                                n_threads);
}

/*
 * The delta rule. [RFC-0026] names the method Kimi Delta Attention, but its
 * pages state only the additive update above. This is the reading the name
 * gives: the gated delta rule with a decay per key channel, which writes v_t
 * against what the decayed state already holds along k_t,
 *     S'_t = S_{t-1} * exp(g_t)
 *     S_t  = S'_t + beta_t * k_t (x) (v_t - S'_t^T k_t)
 *          = (I - beta_t k_t k_t^T) S'_t + beta_t k_t (x) v_t
 *     o_t  = scale * S_t^T q_t
 * with the same reset rule and segments. Returns 0, or -1 on bad arguments.
 */
int oracle_kda_fwd_delta(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const int32_t *seg, int64_t B, int64_t T, int64_t H,
                         int64_t Dk, int64_t Dv, double scale, double *o, int n_threads)
{
    return kda_fwd_run(q, k, v, g, beta, seg, B, T, H, Dk, Dv, scale, NULL, NULL, 0, o,
                       n_threads, 1);
}

/* ------------------------------------------------------------------------ */
/* O4: gradients of the recurrence                                           */
/* ------------------------------------------------------------------------ */
/*
 * The pages state the forward only; its gradients follow by differentiating
 * the recurrence above step by step in reverse (reverse-mode automatic
 * differentiation written out by hand). For a loss L with dL/do_t = do_t,
 * per (segment, head), keeping the forward states S_t and with S = 0 before
 * the segment's first token, going backwards over t with A = dL/dS_t (A = 0
 * after the segment's last token):
 *     A       += scale * q_t (x) do_t                 (o_t = scale S_t^T q_t)
 *     dq_t     = scale * S_t do_t
 *     dbeta_t  = k_t^T A v_t                            (S_t = S'_t + beta_t k_t v_t^T)
 *     dk_t     = beta_t * A v_t
 *     dv_t     = beta_t * A^T k_t
 *     dg_t[i]  = exp(g_t[i]) * sum_j A[i][j] S_{t-1}[i][j]   (S'_t = S_{t-1} exp(g_t))
 *     A[i][j] *= exp(g_t[i])                            (A becomes dL/dS_{t-1})
 * Padding tokens get zero gradients (they take no part in the forward).
 */
typedef struct {
    const double *q, *k, *v, *g, *beta, *d_o;
    int64_t T, H, Dk, Dv;
    double scale;
    double *dq, *dk, *dv, *dg, *dbeta;
    const int64_t *units;
    int64_t n_units;
    int64_t next;   /* shared counter */
    int failed;     /* set when a unit could not get its memory */
} kda_bwd_job_t;

static void run_bwd_unit(kda_bwd_job_t *J, int64_t b, int64_t h, int64_t t0, int64_t t1)
{
    const int64_t H = J->H, Dk = J->Dk, Dv = J->Dv, L = t1 - t0, DD = Dk * Dv;
    /* states[0] = S before the first token (zero), states[1 + u] = S after token t0 + u */
    double *states = (double *)calloc((size_t)((L + 1) * DD), sizeof(double));
    double *A = (double *)calloc((size_t)DD, sizeof(double));
    if (!states || !A) {
        free(states);
        free(A);
        __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED);
        return;
    }
    for (int64_t u = 0; u < L; ++u) {             /* forward, keeping every state */
        const int64_t row = (b * J->T + t0 + u) * H + h;   /* (token, head) */
        const double *kt = J->k + row * Dk;
        const double *gt = J->g + row * Dk;
        const double *vt = J->v + row * Dv;
        const double bt = J->beta[row];
        const double *prev = states + u * DD;
        double *cur = states + (u + 1) * DD;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j)
                cur[i * Dv + j] = prev[i * Dv + j] * exp(gt[i]) + bt * kt[i] * vt[j];
    }
    for (int64_t u = L - 1; u >= 0; --u) {        /* backward */
        const int64_t row = (b * J->T + t0 + u) * H + h;
        const double *qt = J->q + row * Dk;
        const double *kt = J->k + row * Dk;
        const double *gt = J->g + row * Dk;
        const double *vt = J->v + row * Dv;
        const double *dot = J->d_o + row * Dv;
        const double bt = J->beta[row];
        const double *S = states + (u + 1) * DD;      /* S_t */
        const double *Sp = states + u * DD;           /* S_{t-1} */
        double *dqt = J->dq + row * Dk;
        double *dkt = J->dk + row * Dk;
        double *dvt = J->dv + row * Dv;
        double *dgt = J->dg + row * Dk;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j)
                A[i * Dv + j] += J->scale * qt[i] * dot[j];
        double db = 0.0;
        for (int64_t i = 0; i < Dk; ++i) {
            double sq = 0.0, av = 0.0, sg = 0.0;
            for (int64_t j = 0; j < Dv; ++j) {
                sq += S[i * Dv + j] * dot[j];
                av += A[i * Dv + j] * vt[j];
                sg += A[i * Dv + j] * Sp[i * Dv + j];
            }
            dqt[i] = J->scale * sq;
            dkt[i] = bt * av;
            dgt[i] = exp(gt[i]) * sg;
            db += kt[i] * av;
        }
        for (int64_t j = 0; j < Dv; ++j) {
            double ak = 0.0;
            for (int64_t i = 0; i < Dk; ++i)
                ak += A[i * Dv + j] * kt[i];
            dvt[j] = bt * ak;
        }
        J->dbeta[row] = db;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j)
                A[i * Dv + j] *= exp(gt[i]);
    }
    free(states);
    free(A);
}

static void *kda_bwd_worker(void *arg)
{
    kda_bwd_job_t *J = (kda_bwd_job_t *)arg;
    for (;;) {
        const int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (u >= J->n_units)
            break;
        const int64_t *U = J->units + 5 * u;
        run_bwd_unit(J, U[0], U[1], U[2], U[3]);
    }
    return NULL;
}

/*
 * Gradients of the forward above (no per-segment state) for upstream gradient
 * d_o: dq, dk, dg [B*T, H, Dk], dv [B*T, H, Dv], dbeta [B*T, H], all written
 * (zero on padding). One independent reverse pass per (segment, head) on
 * `n_threads` threads. Returns 0, or -1 on bad arguments or out of memory.
 */
int oracle_kda_bwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int32_t *seg, int64_t B, int64_t T, int64_t H,
                   int64_t Dk, int64_t Dv, double scale, const double *d_o, double *dq,
                   double *dk, double *dv, double *dg, double *dbeta, int n_threads)
{
    if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta || B < 0 ||
        T < 0 || H < 1 || Dk < 1 || Dv < 1)
        return -1;
    const int64_t N = B * T;
    memset(dq, 0, sizeof(double) * (size_t)(N * H * Dk));
    memset(dk, 0, sizeof(double) * (size_t)(N * H * Dk));
    memset(dg, 0, sizeof(double) * (size_t)(N * H * Dk));
    memset(dv, 0, sizeof(double) * (size_t)(N * H * Dv));
    memset(dbeta, 0, sizeof(double) * (size_t)(N * H));
    int64_t n_units = 0;
    int64_t *units = segment_units(seg, B, T, H, &n_units);
    if (!units)
        return -1;
    kda_bwd_job_t J = {q, k, v, g, beta, d_o, T, H, Dk, Dv, scale,
                       dq, dk, dv, dg, dbeta, units, n_units, 0, 0};
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 256)
        n_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, kda_bwd_worker, &J) == 0)
            ++started;
    kda_bwd_worker(&J);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(units);
    return J.failed ? -1 : 0;
}
