/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the segmented ("True CP")
 * gated delta-rule forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Source of every formula: the article "flash-linear-attention 上下文并行CP
 * 从 CP2TP、Ring CP 到 True CP 的设计取舍与源码实现" (cited below as [FLA-CP]):
 *   §2.1  local (S_ext, M) per rank, one all-gather, then the merge
 *         S <- 0; for j = r-n_pre .. r-1:  S <- M_j S + S_ext,j
 *   §2.2  the chunk recurrence in WY form and the per-chunk transfer matrix
 *         M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W,  M <- M_[t] M
 *   §2.3  scalar gate (GDN) vs per-key-dim gate (KDA)
 *   §3.2  contiguous layout: rank r holds [r*T/W, (r+1)*T/W)
 *   §3.3  total tokens >= W and divisible by W, else an error
 *   §5.2  per-token comparison; the forward merge feeds a rank's FIRST
 *         local sequence; states are those entering a chunk
 * and, for the stateful-segment invariant (segmented == whole), the issue
 * comment on KDA initial_state in "hyper-parallel issue #7" (H0 -> ... -> HT,
 * chunk_kda(segment2, initial_state=state1)).
 *
 * Everything is fp64.  Inputs arrive as the exact values the GPU sees
 * (fp32 or bf16 bit patterns) and are widened per element.
 *
 * Per-token update (order 0, the order the chunk form of [FLA-CP] §2.2
 * implies -- at chunk size 1 that form is exactly this update):
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * order 1 applies the gate after the projection instead,
 *     S_t = Diag(alpha_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 * which coincides with order 0 for a scalar gate; it exists only so a test
 * can show that the two differ for a per-dimension gate.
 * alpha_t = exp(g_t), g the natural-log gate (scalar per head, or per key dim).
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force explicit matrix
 * products for T <= 16, the EMA closed form, beta = 0 => M = Diag(prod alpha)
 * and S_ext = 0, R = 1 => plain scan, segmented == serial, per-dim gate
 * constant across dims == scalar gate, chunked restatement == serial at
 * C in {1, 16, 64}, T = 1 closed form.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* problem description                                                 */
/* ------------------------------------------------------------------ */
typedef struct {
    int32_t B, H, dk, dv;
    int64_t T;                    /* tokens per row, or total tokens (varlen) */
    const int64_t *cu_seqlens;    /* NULL: B rows of T tokens; else N+1 offsets, B == 1 */
    int32_t num_seqs;             /* N */
    int32_t gate_kind;            /* 0 scalar g [B,T,H]; 1 per-dim gk [B,T,H,dk] */
    int32_t in_dtype;             /* 0 fp32, 1 bf16 (q, k, v, beta) */
    int32_t order;                /* 0 pages' order, 1 gate-after-projection */
    double scale;
    int32_t Hq;                   /* query heads (q and o): a multiple of H; 0 means H */
} oracle_problem;

/* query heads sharing each state: q head hq reads the state of head hq / G */
static int q_group(const oracle_problem *P) { return P->Hq > 0 ? P->Hq / P->H : 1; }

/* widen element i of an fp32 / bf16 array to double */
static double ld_in(const void *p, int64_t i, int dtype) {
    if (dtype == 0) return (double)((const float *)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* sequence n occupies global tokens [seq_begin, seq_end) of the [B*T] token axis */
static void seq_range(const oracle_problem *P, int n, int64_t *s, int64_t *e) {
    if (P->cu_seqlens) { *s = P->cu_seqlens[n]; *e = P->cu_seqlens[n + 1]; }
    else { *s = (int64_t)n * P->T; *e = (int64_t)(n + 1) * P->T; }
}

/* ------------------------------------------------------------------ */
/* a tiny thread pool: items 0..n-1 handed out through a shared counter */
/* ------------------------------------------------------------------ */
typedef void (*item_fn)(void *ctx, int64_t item, double *scratch);
typedef struct {
    item_fn fn; void *ctx; int64_t n; int64_t next; size_t scratch_doubles;
    pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    double *scratch = (double *)malloc(sizeof(double) * (p->scratch_doubles ? p->scratch_doubles : 1));
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->n) break;
        p->fn(p->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

static void run_pool(item_fn fn, void *ctx, int64_t n, int nthreads, size_t scratch_doubles) {
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n = n; p.next = 0; p.scratch_doubles = scratch_doubles;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    for (int i = 1; i < nthreads; i++) pthread_create(&th[i], NULL, pool_worker, &p);
    pool_worker(&p);
    for (int i = 1; i < nthreads; i++) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------ */
/* the per-token update on one head                                     */
/* ------------------------------------------------------------------ */
/*
 * Apply tokens [t0, t1) of head h to the dk x dv state S (row-major).
 * If with_v == 0 the v_t term is dropped: the update is then the linear
 * map T_t = (I - beta k k^T) Diag(alpha) alone (used to build M, whose
 * columns are states of width dk).  If o != NULL the output rows are
 * written (o is [tokens, Hq, dv] double, indexed by global token): with
 * grouped query heads (Hq = G H, the GQA mapping of [FLA-CP] §5.1) every
 * query head hq in [h G, (h+1) G) reads this head's state, o = scale S^T q_hq.
 * width = number of state columns (dv for states, dk for M).
 */
static void apply_tokens(const oracle_problem *P, const void *q, const void *k, const void *v,
                         const void *beta, const float *g, int h, int64_t t0, int64_t t1,
                         double *S, int width, int with_v, double *o, double *tmp) {
    const int dk = P->dk, dv = P->dv, H = P->H;
    double *kk = tmp, *u = tmp + dk, *alpha = tmp + dk + width, *qq = alpha + dk;
    for (int64_t t = t0; t < t1; t++) {
        const int64_t th = t * H + h;
        for (int d = 0; d < dk; d++) kk[d] = ld_in(k, th * dk + d, P->in_dtype);
        const double b = ld_in(beta, th, P->in_dtype);
        if (P->gate_kind == 0) {
            const double a = exp((double)g[th]);
            for (int d = 0; d < dk; d++) alpha[d] = a;
        } else {
            for (int d = 0; d < dk; d++) alpha[d] = exp((double)g[th * dk + d]);
        }
        if (P->order == 0) {
            /* S <- Diag(alpha) S */
            for (int d = 0; d < dk; d++)
                for (int c = 0; c < width; c++) S[d * width + c] *= alpha[d];
        }
        /* u = S^T k */
        for (int c = 0; c < width; c++) u[c] = 0.0;
        for (int d = 0; d < dk; d++)
            for (int c = 0; c < width; c++) u[c] += kk[d] * S[d * width + c];
        if (P->order == 0) {
            /* S <- S + beta k (v - u)^T */
            for (int c = 0; c < width; c++) {
                const double vc = with_v ? ld_in(v, th * dv + c, P->in_dtype) : 0.0;
                u[c] = b * (vc - u[c]);
            }
            for (int d = 0; d < dk; d++)
                for (int c = 0; c < width; c++) S[d * width + c] += kk[d] * u[c];
        } else {
            /* S <- Diag(alpha)(S - beta k u^T) + beta k v^T */
            for (int d = 0; d < dk; d++)
                for (int c = 0; c < width; c++) {
                    const double vc = with_v ? ld_in(v, th * dv + c, P->in_dtype) : 0.0;
                    S[d * width + c] = alpha[d] * (S[d * width + c] - b * kk[d] * u[c]) + b * kk[d] * vc;
                }
        }
        if (o) {
            const int G = q_group(P);
            for (int j = 0; j < G; j++) {
                const int64_t tq = t * (int64_t)(H * G) + (int64_t)h * G + j;
                for (int d = 0; d < dk; d++) qq[d] = ld_in(q, tq * dk + d, P->in_dtype);
                for (int c = 0; c < width; c++) {
                    double acc = 0.0;
                    for (int d = 0; d < dk; d++) acc += S[d * width + c] * qq[d];
                    o[tq * dv + c] = P->scale * acc;
                }
            }
        }
    }
}

static size_t tmp_doubles(const oracle_problem *P) {
    int w = P->dk > P->dv ? P->dk : P->dv;
    return (size_t)(3 * P->dk + w) + (size_t)P->dk * (P->dv + P->dk) + 64;
}

/* ------------------------------------------------------------------ */
/* 1. serial scan over whole sequences                                  */
/* ------------------------------------------------------------------ */
typedef struct {
    const oracle_problem *P;
    const void *q, *k, *v, *beta; const float *g;
    const double *h0; double *o, *ht;
} scan_ctx;

static void scan_item(void *vctx, int64_t item, double *scratch) {
    scan_ctx *c = (scan_ctx *)vctx;
    const oracle_problem *P = c->P;
    const int n = (int)(item / P->H), h = (int)(item % P->H);
    const size_t sz = (size_t)P->dk * P->dv;
    double *S = scratch, *tmp = scratch + sz;
    if (c->h0) memcpy(S, c->h0 + ((size_t)n * P->H + h) * sz, sz * sizeof(double));
    else memset(S, 0, sz * sizeof(double));
    int64_t s, e;
    seq_range(P, n, &s, &e);
    apply_tokens(P, c->q, c->k, c->v, c->beta, c->g, h, s, e, S, P->dv, 1, c->o, tmp);
    if (c->ht) memcpy(c->ht + ((size_t)n * P->H + h) * sz, S, sz * sizeof(double));
}

/* o: [B*T, Hq, dv]; ht: [N, H, dk, dv] (nullable); h0: [N, H, dk, dv] (nullable) */
int oracle_scan(const oracle_problem *P, const void *q, const void *k, const void *v,
                const void *beta, const float *g, const double *h0, double *o, double *ht,
                int nthreads) {
    scan_ctx c = {P, q, k, v, beta, g, h0, o, ht};
    run_pool(scan_item, &c, (int64_t)P->num_seqs * P->H, nthreads,
             (size_t)P->dk * P->dv + tmp_doubles(P));
    return 0;
}

/* ------------------------------------------------------------------ */
/* 2. the segmented scheme of [FLA-CP] §2.1 on R contiguous segments    */
/* ------------------------------------------------------------------ */
/*
 * Segment geometry ([FLA-CP] §3.2 contiguous layout): a fixed-length row b
 * is cut into R pieces of L = T/R tokens; a packed varlen batch (B == 1) is
 * cut over its global token range with L = total/R.  Buffers indexed by
 * segment are [R, B, H, dk, *]: entry (r, b, h).
 */
typedef struct {
    const oracle_problem *P; int R; int64_t L;
    const void *q, *k, *v, *beta; const float *g;
    double *S_ext, *M, *S_init, *o, *ht;
} seg_ctx;

/* global token range of segment (r, b) */
static void seg_range(const seg_ctx *c, int r, int b, int64_t *s, int64_t *e) {
    const int64_t base = c->P->cu_seqlens ? 0 : (int64_t)b * c->P->T;
    *s = base + (int64_t)r * c->L;
    *e = *s + c->L;
}

/* sequence containing global token t */
static int seq_of(const oracle_problem *P, int64_t t) {
    if (!P->cu_seqlens) return (int)(t / P->T);
    int n = 0;
    while (n + 1 < P->num_seqs && P->cu_seqlens[n + 1] <= t) n++;
    return n;
}

/*
 * Pre-process ([FLA-CP] §2.1, §2.3): segment (r, b) contributes the state of
 * its LAST local fragment grown from zero (S_ext) and the product of that
 * fragment's per-token linear maps (M), but only when that fragment's
 * sequence continues into the next segment.  Otherwise both stay zero.
 */
static void pre_item(void *vctx, int64_t item, double *scratch) {
    seg_ctx *c = (seg_ctx *)vctx;
    const oracle_problem *P = c->P;
    const int h = (int)(item % P->H);
    const int b = (int)((item / P->H) % P->B);
    const int r = (int)(item / ((int64_t)P->H * P->B));
    const int dk = P->dk, dv = P->dv;
    const size_t idx = ((size_t)r * P->B + b) * P->H + h;
    double *Se = c->S_ext + idx * dk * dv, *Mo = c->M + idx * dk * dk;
    memset(Se, 0, sizeof(double) * dk * dv);
    memset(Mo, 0, sizeof(double) * dk * dk);
    int64_t s, e;
    seg_range(c, r, b, &s, &e);
    const int n = seq_of(P, e - 1);
    int64_t ss, se;
    seq_range(P, n, &ss, &se);
    if (se <= e) return;                      /* last fragment ends inside: nothing crosses */
    const int64_t f0 = ss > s ? ss : s;       /* trailing fragment [f0, e) */
    double *tmp = scratch;
    apply_tokens(P, c->q, c->k, c->v, c->beta, c->g, h, f0, e, Se, dv, 1, NULL, tmp);
    for (int d = 0; d < dk; d++) Mo[d * dk + d] = 1.0;
    apply_tokens(P, c->q, c->k, c->v, c->beta, c->g, h, f0, e, Mo, dk, 0, NULL, tmp);
}

/*
 * Merge ([FLA-CP] §2.1 and §5.2): segment r whose first token continues a
 * sequence that began in segment r - n_pre gets
 *     S = 0;  for j = r - n_pre .. r-1:  S = M_j S + S_ext,j
 * written out literally (one loop per segment, as the article states it).
 */
static void merge_item(void *vctx, int64_t item, double *scratch) {
    seg_ctx *c = (seg_ctx *)vctx;
    const oracle_problem *P = c->P;
    const int h = (int)(item % P->H);
    const int b = (int)((item / P->H) % P->B);
    const int r = (int)(item / ((int64_t)P->H * P->B));
    const int dk = P->dk, dv = P->dv;
    const size_t sz = (size_t)dk * dv;
    double *out = c->S_init + (((size_t)r * P->B + b) * P->H + h) * sz;
    memset(out, 0, sizeof(double) * sz);
    int64_t s, e;
    seg_range(c, r, b, &s, &e);
    const int n = seq_of(P, s);
    int64_t ss, se;
    seq_range(P, n, &ss, &se);
    if (ss >= s) return;                      /* segment starts a sequence: zero state */
    const int64_t base = P->cu_seqlens ? 0 : (int64_t)b * P->T;
    const int r0 = (int)((ss - base) / c->L); /* segment holding the sequence start */
    double *S = scratch, *nx = scratch + sz;
    memset(S, 0, sizeof(double) * sz);
    for (int j = r0; j < r; j++) {
        const size_t jdx = ((size_t)j * P->B + b) * P->H + h;
        const double *Mj = c->M + jdx * dk * dk, *Ej = c->S_ext + jdx * sz;
        for (int i = 0; i < dk; i++)
            for (int col = 0; col < dv; col++) {
                double acc = Ej[i * dv + col];
                for (int l = 0; l < dk; l++) acc += Mj[i * dk + l] * S[l * dv + col];
                nx[i * dv + col] = acc;
            }
        memcpy(S, nx, sizeof(double) * sz);
    }
    memcpy(out, S, sizeof(double) * sz);
}

/*
 * Forward per segment: each local fragment restarts from zero, except the
 * first one when it continues an earlier sequence, which starts from
 * S_init of this segment.  A fragment that ends its sequence writes the
 * final state.
 */
static void fwd_item(void *vctx, int64_t item, double *scratch) {
    seg_ctx *c = (seg_ctx *)vctx;
    const oracle_problem *P = c->P;
    const int h = (int)(item % P->H);
    const int b = (int)((item / P->H) % P->B);
    const int r = (int)(item / ((int64_t)P->H * P->B));
    const int dk = P->dk, dv = P->dv;
    const size_t sz = (size_t)dk * dv;
    double *S = scratch, *tmp = scratch + sz;
    int64_t s, e;
    seg_range(c, r, b, &s, &e);
    int64_t t = s;
    while (t < e) {
        const int n = seq_of(P, t);
        int64_t ss, se;
        seq_range(P, n, &ss, &se);
        const int64_t fe = se < e ? se : e;
        if (ss < t) memcpy(S, c->S_init + (((size_t)r * P->B + b) * P->H + h) * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        apply_tokens(P, c->q, c->k, c->v, c->beta, c->g, h, t, fe, S, dv, 1, c->o, tmp);
        if (fe == se && c->ht) memcpy(c->ht + ((size_t)n * P->H + h) * sz, S, sizeof(double) * sz);
        t = fe;
    }
}

/*
 * S_ext, S_init: [R, B, H, dk, dv]; M: [R, B, H, dk, dk]; o: [B*T, Hq, dv];
 * ht: [N, H, dk, dv].  Returns 1 when the cut rule of [FLA-CP] §3.3 fails
 * (tokens per row < R or not divisible by R).
 */
int oracle_segmented(const oracle_problem *P, int R, const void *q, const void *k, const void *v,
                     const void *beta, const float *g, double *S_ext, double *M, double *S_init,
                     double *o, double *ht, int nthreads) {
    const int64_t total = P->cu_seqlens ? P->cu_seqlens[P->num_seqs] : P->T;
    if (R < 1 || total < R || total % R != 0) return 1;
    seg_ctx c = {P, R, total / R, q, k, v, beta, g, S_ext, M, S_init, o, ht};
    const int64_t items = (int64_t)R * P->B * P->H;
    const size_t scratch = (size_t)P->dk * (P->dv + P->dk) * 2 + tmp_doubles(P);
    run_pool(pre_item, &c, items, nthreads, scratch);
    run_pool(merge_item, &c, items, nthreads, scratch);
    run_pool(fwd_item, &c, items, nthreads, scratch);
    return 0;
}

/* ------------------------------------------------------------------ */
/* 3. the chunk form of [FLA-CP] §2.2, restated in fp64                 */
/* ------------------------------------------------------------------ */
/*
 * One head, tokens [t0, t1), chunk size C, starting from S (dk x dv),
 * optionally also carrying M (dk x dk, the chained transfer matrix, which
 * starts as whatever the caller put there).  Per chunk (natural-log gates,
 * cumulative inside the chunk):
 *   G_i = sum_{s<=i} g_s            gamma_i = exp(G_i),  gamma^C = gamma_last
 *   Gamma_j = exp(G_last - G_j)
 *   A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd),  j < i   (0 otherwise)
 *   (I + A) W = diag(beta)(gamma ⊙ K),  (I + A) U = diag(beta) V
 *   Delta = U - W S                             (the "v_new" of the article)
 *   O = scale [ (gamma ⊙ Q) S + (Q K^T ⊙ Lambda) Delta ],
 *       Lambda_ij = exp(G_i - G_j) for j <= i, 0 otherwise (per dim for KDA)
 *   S <- Diag(gamma^C) S + (Gamma ⊙ K)^T Delta
 *   M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W,   M <- M_[t] M
 * The solve is plain forward substitution.  Only order 0 has this form.
 */
static void chunk_pass(const oracle_problem *P, int C, const void *q, const void *k, const void *v,
                       const void *beta, const float *g, int h, int64_t t0, int64_t t1,
                       double *S, double *Mc, double *o) {
    const int dk = P->dk, dv = P->dv, H = P->H;
    double *G = (double *)malloc(sizeof(double) * C * dk);
    double *K = (double *)malloc(sizeof(double) * C * dk);
    double *Q = (double *)malloc(sizeof(double) * C * dk);
    double *V = (double *)malloc(sizeof(double) * C * dv);
    double *bt = (double *)malloc(sizeof(double) * C);
    double *A = (double *)malloc(sizeof(double) * C * C);
    double *W = (double *)malloc(sizeof(double) * C * dk);
    double *U = (double *)malloc(sizeof(double) * C * dv);
    double *D = (double *)malloc(sizeof(double) * C * dv);
    double *MK = (double *)malloc(sizeof(double) * dk * dk);
    double *Sn = (double *)malloc(sizeof(double) * dk * (dv > dk ? dv : dk));
    for (int64_t c0 = t0; c0 < t1; c0 += C) {
        const int n = (int)((t1 - c0) < C ? (t1 - c0) : C);
        /* gather the chunk and its cumulative log gates */
        for (int i = 0; i < n; i++) {
            const int64_t th = (c0 + i) * H + h;
            for (int d = 0; d < dk; d++) {
                K[i * dk + d] = ld_in(k, th * dk + d, P->in_dtype);
                Q[i * dk + d] = q ? ld_in(q, th * dk + d, P->in_dtype) : 0.0;
                const double gi = P->gate_kind == 0 ? (double)g[th] : (double)g[th * dk + d];
                G[i * dk + d] = (i ? G[(i - 1) * dk + d] : 0.0) + gi;
            }
            for (int e = 0; e < dv; e++) V[i * dv + e] = ld_in(v, th * dv + e, P->in_dtype);
            bt[i] = ld_in(beta, th, P->in_dtype);
        }
        /* A (strictly lower) */
        for (int i = 0; i < n; i++)
            for (int j = 0; j < n; j++) {
                double a = 0.0;
                if (j < i)
                    for (int d = 0; d < dk; d++) a += K[i * dk + d] * K[j * dk + d] * exp(G[i * dk + d] - G[j * dk + d]);
                A[i * C + j] = bt[i] * a;
            }
        /* forward substitution: (I + A) W = diag(beta)(gamma ⊙ K), (I + A) U = diag(beta) V */
        for (int i = 0; i < n; i++) {
            for (int d = 0; d < dk; d++) {
                double w = bt[i] * exp(G[i * dk + d]) * K[i * dk + d];
                for (int j = 0; j < i; j++) w -= A[i * C + j] * W[j * dk + d];
                W[i * dk + d] = w;
            }
            for (int e = 0; e < dv; e++) {
                double u = bt[i] * V[i * dv + e];
                for (int j = 0; j < i; j++) u -= A[i * C + j] * U[j * dv + e];
                U[i * dv + e] = u;
            }
        }
        /* Delta = U - W S */
        for (int i = 0; i < n; i++)
            for (int e = 0; e < dv; e++) {
                double acc = U[i * dv + e];
                for (int d = 0; d < dk; d++) acc -= W[i * dk + d] * S[d * dv + e];
                D[i * dv + e] = acc;
            }
        /* O = scale [ (gamma ⊙ Q) S + (Q K^T ⊙ Lambda) Delta ] */
        if (o)
            for (int i = 0; i < n; i++) {
                const int64_t th = (c0 + i) * H + h;
                for (int e = 0; e < dv; e++) {
                    double acc = 0.0;
                    for (int d = 0; d < dk; d++) acc += exp(G[i * dk + d]) * Q[i * dk + d] * S[d * dv + e];
                    for (int j = 0; j <= i; j++) {
                        double qk = 0.0;
                        for (int d = 0; d < dk; d++) qk += Q[i * dk + d] * K[j * dk + d] * exp(G[i * dk + d] - G[j * dk + d]);
                        acc += qk * D[j * dv + e];
                    }
                    o[th * dv + e] = P->scale * acc;
                }
            }
        /* S <- Diag(gamma^C) S + (Gamma ⊙ K)^T Delta */
        const double *GC = G + (n - 1) * dk;
        for (int d = 0; d < dk; d++)
            for (int e = 0; e < dv; e++) {
                double acc = exp(GC[d]) * S[d * dv + e];
                for (int j = 0; j < n; j++) acc += exp(GC[d] - G[j * dk + d]) * K[j * dk + d] * D[j * dv + e];
                Sn[d * dv + e] = acc;
            }
        memcpy(S, Sn, sizeof(double) * dk * dv);
        /* M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W;  M <- M_[t] M */
        if (Mc) {
            for (int d = 0; d < dk; d++)
                for (int l = 0; l < dk; l++) {
                    double acc = (d == l) ? exp(GC[d]) : 0.0;
                    for (int j = 0; j < n; j++) acc -= exp(GC[d] - G[j * dk + d]) * K[j * dk + d] * W[j * dk + l];
                    MK[d * dk + l] = acc;
                }
            for (int d = 0; d < dk; d++)
                for (int l = 0; l < dk; l++) {
                    double acc = 0.0;
                    for (int m = 0; m < dk; m++) acc += MK[d * dk + m] * Mc[m * dk + l];
                    Sn[d * dk + l] = acc;
                }
            memcpy(Mc, Sn, sizeof(double) * dk * dk);
        }
    }
    free(G); free(K); free(Q); free(V); free(bt); free(A); free(W); free(U); free(D); free(MK); free(Sn);
}

/*
 * Whole sequences in chunk form from zero state (o: [B*T,H,dv], ht: [N,H,dk,dv]);
 * returns 2 for grouped query heads, which it does not cover.
 * Single-threaded: it exists to pin the chunk equations on small inputs.
 */
int oracle_chunked(const oracle_problem *P, int C, const void *q, const void *k, const void *v,
                   const void *beta, const float *g, double *o, double *ht) {
    if (q_group(P) != 1) return 2;   /* the chunk restatement covers Hq == H only */
    if (P->order != 0 || C < 1) return 1;
    const size_t sz = (size_t)P->dk * P->dv;
    double *S = (double *)malloc(sizeof(double) * sz);
    for (int n = 0; n < P->num_seqs; n++)
        for (int h = 0; h < P->H; h++) {
            int64_t s, e;
            seq_range(P, n, &s, &e);
            memset(S, 0, sizeof(double) * sz);
            chunk_pass(P, C, q, k, v, beta, g, h, s, e, S, NULL, o);
            if (ht) memcpy(ht + ((size_t)n * P->H + h) * sz, S, sizeof(double) * sz);
        }
    free(S);
    return 0;
}

/*
 * Chunk-form pre-process of one token range [t0, t1) of head h: S_ext from
 * zero and the chained M from the identity ([FLA-CP] §2.1-§2.2).
 */
int oracle_chunked_pre(const oracle_problem *P, int C, const void *k, const void *v,
                       const void *beta, const float *g, int h, int64_t t0, int64_t t1,
                       double *S_ext, double *M) {
    if (P->order != 0 || C < 1) return 1;
    memset(S_ext, 0, sizeof(double) * P->dk * P->dv);
    memset(M, 0, sizeof(double) * P->dk * P->dk);
    for (int d = 0; d < P->dk; d++) M[d * P->dk + d] = 1.0;
    chunk_pass(P, C, NULL, k, v, beta, g, h, t0, t1, S_ext, M, NULL);
    return 0;
}

/* ------------------------------------------------------------------ */
/* 4. the backward of the per-token scan (order 0)                      */
/* ------------------------------------------------------------------ */
/*
 * Gradients of L = sum_t <do_t, o_t> + sum_n <dht_n, S_final,n> with
 * respect to q, k, v, beta and the log gates, by the reverse of the
 * per-token update (the chain rule written out, no chunking):
 *   P = Diag(alpha) S_{t-1},  u = v - P^T k,  S_t = P + beta k u^T,
 *   o_t = scale S_t^T q_t.
 * With G = dL/dS_t (after adding scale q_t do_t^T from o_t):
 *   dq_t = scale S_t do_t,       g_u = beta G^T k,       dv_t = g_u,
 *   dbeta_t = k^T G u,           dk_t = beta G u - P g_u,
 *   dP = G - k g_u^T,            dalpha_d = sum_c dP_dc S_{t-1,dc},
 *   dg_t = alpha dalpha (per key dim; summed over d for a scalar gate),
 *   dL/dS_{t-1} = Diag(alpha) dP.
 * With grouped query heads (Hq = G H, [FLA-CP] §5.1) the G query heads hq of
 * state head h each read S_t: o_t,hq = scale S_t^T q_t,hq, so each has its
 * own dq_t,hq = scale S_t do_t,hq and G collects scale q_t,hq do_t,hq^T of
 * every one of them; the rest of the step is the state head's.
 * States are recomputed forward from checkpoints every 64 tokens.
 */
typedef struct {
    const oracle_problem *P;
    const void *q, *k, *v, *beta, *dout; const float *g;
    const double *dht;
    double *dq, *dk, *dv, *dbeta, *dg;
} bwd_ctx;

static void bwd_item(void *vctx, int64_t item, double *scratch) {
    (void)scratch;
    bwd_ctx *c = (bwd_ctx *)vctx;
    const oracle_problem *P = c->P;
    const int n = (int)(item / P->H), h = (int)(item % P->H);
    const int dk = P->dk, dv = P->dv, H = P->H, Gq = q_group(P), Hq = H * Gq;
    const size_t sz = (size_t)dk * dv;
    const int CK = 64;
    int64_t s, e;
    seq_range(P, n, &s, &e);
    const int64_t len = e - s;
    const int64_t nck = (len + CK - 1) / CK;
    double *ck = (double *)malloc(sizeof(double) * sz * (size_t)(nck > 0 ? nck : 1));
    double *st = (double *)malloc(sizeof(double) * sz * (CK + 1));
    double *G = (double *)malloc(sizeof(double) * sz);
    double *Pm = (double *)malloc(sizeof(double) * sz);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(8 * (dk + dv) + 64));
    double *kk = tmp, *qq = kk + dk, *al = qq + dk, *u = al + dk, *gu = u + dv, *vv = gu + dv, *dd = vv + dv;
    /* forward: checkpoints of the state before tokens s, s + CK, ... */
    double *S = st;
    memset(S, 0, sizeof(double) * sz);
    for (int64_t t = s; t < e; t++) {
        if ((t - s) % CK == 0) memcpy(ck + (size_t)((t - s) / CK) * sz, S, sizeof(double) * sz);
        apply_tokens(P, NULL, c->k, c->v, c->beta, c->g, h, t, t + 1, S, dv, 1, NULL, tmp);
    }
    if (c->dht) memcpy(G, c->dht + ((size_t)n * H + h) * sz, sizeof(double) * sz);
    else memset(G, 0, sizeof(double) * sz);
    for (int64_t m = nck - 1; m >= 0; m--) {
        const int64_t t0 = s + m * CK, t1 = (t0 + CK < e) ? t0 + CK : e;
        const int nb = (int)(t1 - t0);
        /* st[i] = state before token t0 + i, st[nb] = after the block */
        memcpy(st, ck + (size_t)m * sz, sizeof(double) * sz);
        for (int i = 0; i < nb; i++) {
            memcpy(st + (size_t)(i + 1) * sz, st + (size_t)i * sz, sizeof(double) * sz);
            apply_tokens(P, NULL, c->k, c->v, c->beta, c->g, h, t0 + i, t0 + i + 1, st + (size_t)(i + 1) * sz,
                         dv, 1, NULL, tmp + 4 * (dk + dv));
        }
        for (int i = nb - 1; i >= 0; i--) {
            const int64_t t = t0 + i, th = t * H + h;
            const double *Sp = st + (size_t)i * sz, *St = st + (size_t)(i + 1) * sz;
            for (int d = 0; d < dk; d++) {
                kk[d] = ld_in(c->k, th * dk + d, P->in_dtype);
                al[d] = exp((double)(P->gate_kind == 0 ? c->g[th] : c->g[th * dk + d]));
            }
            for (int cc = 0; cc < dv; cc++) vv[cc] = ld_in(c->v, th * dv + cc, P->in_dtype);
            const double b = ld_in(c->beta, th, P->in_dtype);
            /* per query head of this state: dq_t = scale S_t do_t; G += scale q_t do_t^T */
            for (int gq = 0; gq < Gq; gq++) {
                const int64_t tq = t * Hq + (int64_t)h * Gq + gq;
                for (int d = 0; d < dk; d++) qq[d] = ld_in(c->q, tq * dk + d, P->in_dtype);
                for (int cc = 0; cc < dv; cc++) dd[cc] = P->scale * ld_in(c->dout, tq * dv + cc, P->in_dtype);
                for (int d = 0; d < dk; d++) {
                    double acc = 0.0;
                    for (int cc = 0; cc < dv; cc++) acc += St[d * dv + cc] * dd[cc];
                    c->dq[tq * dk + d] = acc;
                    for (int cc = 0; cc < dv; cc++) G[d * dv + cc] += qq[d] * dd[cc];
                }
            }
            /* P = Diag(alpha) S_{t-1}, u = v - P^T k */
            for (int d = 0; d < dk; d++)
                for (int cc = 0; cc < dv; cc++) Pm[d * dv + cc] = al[d] * Sp[d * dv + cc];
            for (int cc = 0; cc < dv; cc++) {
                double acc = 0.0;
                for (int d = 0; d < dk; d++) acc += Pm[d * dv + cc] * kk[d];
                u[cc] = vv[cc] - acc;
            }
            /* g_u = beta G^T k */
            for (int cc = 0; cc < dv; cc++) {
                double acc = 0.0;
                for (int d = 0; d < dk; d++) acc += G[d * dv + cc] * kk[d];
                gu[cc] = b * acc;
                c->dv[th * dv + cc] = gu[cc];
            }
            /* dbeta = k^T G u; dk = beta G u - P g_u */
            double dbeta = 0.0;
            for (int d = 0; d < dk; d++) {
                double Gu = 0.0, Pg = 0.0;
                for (int cc = 0; cc < dv; cc++) {
                    Gu += G[d * dv + cc] * u[cc];
                    Pg += Pm[d * dv + cc] * gu[cc];
                }
                dbeta += kk[d] * Gu;
                c->dk[th * dk + d] = b * Gu - Pg;
            }
            c->dbeta[th] = dbeta;
            /* dP = G - k g_u^T; dalpha; G <- Diag(alpha) dP */
            double dgs = 0.0;
            for (int d = 0; d < dk; d++) {
                double da = 0.0;
                for (int cc = 0; cc < dv; cc++) {
                    const double dP = G[d * dv + cc] - kk[d] * gu[cc];
                    da += dP * Sp[d * dv + cc];
                    G[d * dv + cc] = al[d] * dP;
                }
                if (P->gate_kind == 0) dgs += al[d] * da;
                else c->dg[th * dk + d] = al[d] * da;
            }
            if (P->gate_kind == 0) c->dg[th] = dgs;
        }
    }
    free(ck); free(st); free(G); free(Pm); free(tmp);
}

/* dout: [B*T, Hq, dv] in the input dtype; dht: [N, H, dk, dv] (nullable);
 * dq: [B*T, Hq, dk]; dk: [B*T, H, dk]; dv: [B*T, H, dv]; dbeta: [B*T, H];
 * dg like the gate.  Returns 1 for order 1 (not covered). */
int oracle_backward(const oracle_problem *P, const void *q, const void *k, const void *v, const void *beta,
                    const float *g, const void *dout, const double *dht, double *dq, double *dk, double *dv,
                    double *dbeta, double *dg, int nthreads) {
    if (P->order != 0) return 1;
    bwd_ctx c = {P, q, k, v, beta, dout, g, dht, dq, dk, dv, dbeta, dg};
    run_pool(bwd_item, &c, (int64_t)P->num_seqs * P->H, nthreads, 1);
    return 0;
}
