/*
 * sffn_oracle.c -- plain, slow fp64 CPU oracle for the activation-sparse gated FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; it reads the same raw input buffers (fp32 / bf16 bits / packed
 * int4 codes + fp16 scale bits) and decodes them itself, exactly, to fp64.
 *
 * Every step is the plain definition written out with ascending-index loops:
 *   gated FFN      out = W_down . ( act(W_gate.x + b) (.) (W_up.x) )
 *                  -- denseflux ("skipping most of a dense FFN"), sec. 1 Motivation:
 *                     neuron i owns row i of W_gate, row i of W_up, column i of W_down.
 *   exact gating   skip neuron j iff act(g_j) == 0 (ReLU/ReGLU)
 *                  -- denseflux sec. 5.1/5.2 (zero activations contribute nothing).
 *   threshold      keep j iff score_j >= tau, score_j = |a_j| * ||W_down[:,j]||_2
 *                  -- WiSparse write-up (kwkr.cn/news/623085) sec. 1.2 (absolute
 *                     threshold on SiLU/GELU) and sec. 2.3 (weight-aware score, p = 2).
 *   keep ratio     k = max(1, floor(F * keep_ratio)); keep the k largest scores
 *                  -- WiSparse sec. 3.2 (select_mask) and sec. 2.2 (tier M keeps 1/M).
 *   byte model     exact gating keeps (1 + 2a)/3 of the FFN bytes
 *                  -- denseflux sec. 3 Setup (cost measure) and sec. 5.3.
 *   token select   importance = L2 norm of the attention-output row; top-P mass,
 *                  last recent_n always kept, at least min_keep, all-zero -> dense,
 *                  mass_thresh >= 1 -> dense
 *                  -- RedKnot token-selective sparse FFN (bhfrc.com/news/43276),
 *                     "Token selective sparse FFN: how importance is judged" and the
 *                     two safeguards / equivalence-switch paragraphs.
 *   prefill        S <- Select; Z[S] <- FFN(Y[S]); Z[~S] <- 0; X_next <- Y + Z
 *                  -- RedKnot, Algorithm 1 (four steps).
 *
 * Readings where the pages are silent or garbled (each is listed in the design
 * notes): ties in the keep-ratio order and in the token order go to the lower
 * index; the crossing token of the mass prefix is included; Y = bf16_rne(X + Y_attn);
 * the FFN has no normalisation; int4 groups are 64 consecutive elements along each
 * stored row, codes are two's-complement nibbles, the low nibble is the even column.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Element formats and exact decoding to fp64                                */
/* ------------------------------------------------------------------------- */

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_INT4_G64 = 2, ORC_F64 = 3 };
enum { ORC_RELU = 0, ORC_SILU = 1 };
enum { ORC_EXACT = 0, ORC_THRESHOLD = 1, ORC_KEEP_RATIO = 2 };
enum { ORC_SCORE_GATE = 0, ORC_SCORE_GATE_UP = 1 };

#define ORC_GROUP 64

/* A read-only matrix [rows, cols] in one of the stored formats. */
typedef struct {
    int fmt;
    int rows, cols;
    const void *data;        /* f32 / bf16 bits / packed int4 / f64            */
    const uint16_t *scales;  /* int4 only: fp16 bits [rows, cols / 64]         */
} orc_mat;

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 decoded from its fields (sign, 5-bit exponent, 10-bit fraction). */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* Round an fp64 value to the nearest bf16 (ties to even), returning the bits.
 * bf16 keeps 8 significant bits and the binary32 exponent range; below 2^-126
 * the quantum is fixed at 2^-133 (subnormals). */
uint16_t orc_f64_to_bf16_rne(double v) {
    if (isnan(v)) return 0x7fc0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);                               /* a = f * 2^e, f in [0.5, 1) */
        int q = e - 8;                              /* quantum exponent: 8 significant bits */
        if (q < -133) q = -133;
        double scaled = ldexp(a, -q);               /* exact (power-of-two scaling) */
        double n = nearbyint(scaled);               /* default rounding: to nearest, ties even */
        r = ldexp(n, q);
        if (r > 3.3895313892515355e38) r = INFINITY; /* above the largest finite bf16 */
    }
    float f = (float)(signbit(v) ? -r : r);         /* exact: r is representable in bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Signed int4 code of element (r, c): byte (r*cols + c)/2, low nibble = even column. */
static int orc_int4_code(const uint8_t *packed, int cols, int r, int c) {
    size_t lin = (size_t)r * (size_t)cols + (size_t)c;
    uint8_t byte = packed[lin >> 1];
    int nib = (lin & 1) ? (byte >> 4) : (byte & 0x0f);
    return nib >= 8 ? nib - 16 : nib;
}

/* Exact value of element (r, c). */
double orc_mat_at(const orc_mat *m, int r, int c) {
    size_t lin = (size_t)r * (size_t)m->cols + (size_t)c;
    switch (m->fmt) {
    case ORC_F32: return (double)((const float *)m->data)[lin];
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t *)m->data)[lin]);
    case ORC_F64: return ((const double *)m->data)[lin];
    case ORC_INT4_G64: {
        int code = orc_int4_code((const uint8_t *)m->data, m->cols, r, c);
        size_t g = (size_t)r * (size_t)(m->cols / ORC_GROUP) + (size_t)(c / ORC_GROUP);
        return (double)code * orc_f16_to_f64(m->scales[g]);
    }
    }
    return NAN;
}

/* Dequantise a whole matrix to fp64 (used by the tests to cross-check). */
void orc_mat_to_f64(const orc_mat *m, double *out) {
    for (int r = 0; r < m->rows; ++r)
        for (int c = 0; c < m->cols; ++c)
            out[(size_t)r * m->cols + c] = orc_mat_at(m, r, c);
}

/* ------------------------------------------------------------------------- */
/* Gated FFN pieces                                                          */
/* ------------------------------------------------------------------------- */

/* The FFN of one layer.  All three weight matrices are stored neuron-major:
 * w_gate[j,:], w_up[j,:] and w_downT[j,:] = W_down[:, j], each [F, d]. */
typedef struct {
    int d_model, d_ff, act;
    orc_mat w_gate, w_up, w_downT;
    const float *b_gate; /* [F] or NULL */
} orc_ffn;

double orc_act(int act, double z) {
    if (act == ORC_RELU) return z > 0.0 ? z : 0.0;
    return z / (1.0 + exp(-z));                     /* SiLU(z) = z * sigmoid(z) */
}

/* ||W_down[:, j]||_2 = sqrt(sum_i W_downT[j, i]^2), ascending i.
 * WiSparse sec. 2.3: the weight-aware prior is the L2 norm (p = 2) of the weight
 * vector tied to neuron j; the down projection's column is the one that scales
 * the neuron's contribution to the output. */
void orc_down_norms(const orc_ffn *w, double *norms) {
    for (int j = 0; j < w->d_ff; ++j) {
        double s = 0.0;
        for (int i = 0; i < w->d_model; ++i) {
            double v = orc_mat_at(&w->w_downT, j, i);
            s += v * v;
        }
        norms[j] = sqrt(s);
    }
}

/* Per-token state of the decode oracle. */
typedef struct {
    double *g;     /* [F] gate pre-activation  W_gate[j].x + b_j              */
    double *a;     /* [F] act(g)                                               */
    double *u;     /* [F] W_up[j].x (all j)                                    */
    double *score; /* [F] mode score                                           */
    double *cond;  /* [F] conditioning scale of the decision quantity          */
} orc_tok;

/* One dot product row.x in ascending k; also its absolute-value sum. */
static double orc_row_dot(const orc_mat *m, int r, const double *x, int d, double *abs_sum) {
    double s = 0.0, c = 0.0;
    for (int k = 0; k < d; ++k) {
        double p = orc_mat_at(m, r, k) * x[k];
        s += p;
        c += fabs(p);
    }
    if (abs_sum) *abs_sum = c;
    return s;
}

/* Gate, activation, up projection and the score of every neuron for one token.
 * The decision quantity is g_j for exact gating (cut 0) and score_j otherwise;
 * cond_j bounds the magnitude of its rounding error (used only for the tie band). */
static void orc_token_scores(const orc_ffn *w, const double *x, const double *norms, int mode,
                             int score_kind, orc_tok *t) {
    int d = w->d_model, F = w->d_ff;
    for (int j = 0; j < F; ++j) {
        double cg, cu;
        double g = orc_row_dot(&w->w_gate, j, x, d, &cg);
        if (w->b_gate) {
            g += (double)w->b_gate[j];
            cg += fabs((double)w->b_gate[j]);
        }
        double u = orc_row_dot(&w->w_up, j, x, d, &cu);
        double a = orc_act(w->act, g);
        t->g[j] = g;
        t->a[j] = a;
        t->u[j] = u;
        if (score_kind == ORC_SCORE_GATE) {
            t->score[j] = fabs(a) * norms[j];
            t->cond[j] = (mode == ORC_EXACT) ? cg : 1.1 * cg * norms[j];
        } else {
            t->score[j] = fabs(a * u) * norms[j];
            t->cond[j] = (fabs(u) * 1.1 * cg + fmax(fabs(a), cg) * cu) * norms[j];
        }
    }
}

/* Sort helper: indices by (score descending, index ascending). */
static const double *orc_sort_key;
static int orc_cmp_desc(const void *pa, const void *pb) {
    int a = *(const int *)pa, b = *(const int *)pb;
    double sa = orc_sort_key[a], sb = orc_sort_key[b];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (a > b) - (a < b);
}
static pthread_mutex_t orc_sort_lock = PTHREAD_MUTEX_INITIALIZER;
static void orc_order_desc(const double *key, int n, int *order) {
    for (int i = 0; i < n; ++i) order[i] = i;
    pthread_mutex_lock(&orc_sort_lock);
    orc_sort_key = key;
    qsort(order, (size_t)n, sizeof(int), orc_cmp_desc);
    pthread_mutex_unlock(&orc_sort_lock);
}

static int orc_cmp_int(const void *pa, const void *pb) {
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/* Keep-ratio budget: k = max(1, floor(F * keep_ratio)) (WiSparse sec. 3.2). */
int orc_keep_count(int F, double keep_ratio) {
    double kk = floor((double)F * keep_ratio);
    int k = kk < 1.0 ? 1 : (int)kk;
    return k > F ? F : k;
}

/* Active set of one token, ascending.  Returns |A|.
 *   exact      : a_j != 0                     (cut 0 on g_j for ReLU)
 *   threshold  : score_j >= tau               (tau = 0 keeps everything)
 *   keep_ratio : the k largest scores, ties to the lower index            */
static int orc_select(const orc_ffn *w, const orc_tok *t, int mode, double param, int32_t *idx,
                      double *cut) {
    int F = w->d_ff, n = 0;
    if (mode == ORC_EXACT) {
        for (int j = 0; j < F; ++j)
            if (t->a[j] != 0.0) idx[n++] = j;
        if (cut) *cut = 0.0;
    } else if (mode == ORC_THRESHOLD) {
        for (int j = 0; j < F; ++j)
            if (t->score[j] >= param) idx[n++] = j;
        if (cut) *cut = param;
    } else {
        int k = orc_keep_count(F, param);
        int *order = (int *)malloc(sizeof(int) * (size_t)F);
        orc_order_desc(t->score, F, order);
        for (int i = 0; i < k; ++i) idx[i] = order[i];
        if (cut) *cut = t->score[order[k - 1]];
        free(order);
        n = k;
        qsort(idx, (size_t)n, sizeof(int32_t), orc_cmp_int);
    }
    return n;
}

/* out[i] = sum over j in A (ascending) of (a_j * u_j) * W_down[i, j]. */
static void orc_ffn_on_set(const orc_ffn *w, const orc_tok *t, const int32_t *idx, int n, double *out) {
    int d = w->d_model;
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    for (int q = 0; q < n; ++q) {
        int j = idx[q];
        double h = t->a[j] * t->u[j];
        for (int i = 0; i < d; ++i) out[i] += h * orc_mat_at(&w->w_downT, j, i);
    }
}

/* Bytes of FFN weights one token reads: the gate (and, for the gate-and-up
 * score, the up projection) in full, plus the active rows of the others.
 * denseflux sec. 3: gate always read, so (F + 2|A|) rows = (1 + 2a)/3 of 3F rows. */
double orc_row_bytes(int fmt, int d) {
    switch (fmt) {
    case ORC_F32: return 4.0 * d;
    case ORC_BF16: return 2.0 * d;
    case ORC_INT4_G64: return 0.5 * d + 2.0 * (d / ORC_GROUP);
    case ORC_F64: return 8.0 * d;
    }
    return 0.0;
}
double orc_bytes_kept(int fmt, int d, int F, int score_kind, int n_active) {
    double r = orc_row_bytes(fmt, d);
    if (score_kind == ORC_SCORE_GATE_UP) return ((double)2 * F + n_active) * r;
    return ((double)F + 2.0 * n_active) * r;
}

/* ------------------------------------------------------------------------- */
/* Decode driver (optionally parallel over tokens)                           */
/* ------------------------------------------------------------------------- */

typedef struct {
    const orc_ffn *w;
    const orc_mat *x;        /* [B, d] f32 or bf16 bits */
    const double *norms;     /* [F] */
    int mode, score_kind;
    double param;
    const int32_t *given_idx; /* optional [B, F] externally chosen sets */
    const int32_t *given_n;   /* optional [B] */
    double *out;             /* [B, d] */
    int32_t *active_idx;     /* [B, F] */
    int32_t *n_active;       /* [B] */
    double *g, *a, *u, *score, *cond, *cut; /* optional [B, F] / [B] */
    int B, next;
    pthread_mutex_t lock;
} orc_decode_job;

static void orc_decode_one(orc_decode_job *job, int b) {
    const orc_ffn *w = job->w;
    int d = w->d_model, F = w->d_ff;
    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    for (int k = 0; k < d; ++k) x[k] = orc_mat_at(job->x, b, k);
    orc_tok t;
    double *buf = (double *)malloc(sizeof(double) * (size_t)F * 5);
    t.g = buf;
    t.a = buf + F;
    t.u = buf + 2 * (size_t)F;
    t.score = buf + 3 * (size_t)F;
    t.cond = buf + 4 * (size_t)F;
    orc_token_scores(w, x, job->norms, job->mode, job->score_kind, &t);
    int32_t *idx = job->active_idx + (size_t)b * F;
    double cut = 0.0;
    int n = orc_select(w, &t, job->mode, job->param, idx, &cut);
    job->n_active[b] = n;
    const int32_t *use = idx;
    int nuse = n;
    if (job->given_idx) {
        use = job->given_idx + (size_t)b * F;
        nuse = job->given_n[b];
    }
    orc_ffn_on_set(w, &t, use, nuse, job->out + (size_t)b * d);
    if (job->g) memcpy(job->g + (size_t)b * F, t.g, sizeof(double) * F);
    if (job->a) memcpy(job->a + (size_t)b * F, t.a, sizeof(double) * F);
    if (job->u) memcpy(job->u + (size_t)b * F, t.u, sizeof(double) * F);
    if (job->score) memcpy(job->score + (size_t)b * F, t.score, sizeof(double) * F);
    if (job->cond) memcpy(job->cond + (size_t)b * F, t.cond, sizeof(double) * F);
    if (job->cut) job->cut[b] = cut;
    free(buf);
    free(x);
}

static void *orc_decode_worker(void *arg) {
    orc_decode_job *job = (orc_decode_job *)arg;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int b = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (b >= job->B) break;
        orc_decode_one(job, b);
    }
    return NULL;
}

static void orc_run_workers(void *(*fn)(void *), void *job, int nthreads) {
    if (nthreads <= 1) {
        fn(job);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, fn, job) == 0) ++started;
        else break;
    if (started == 0) fn(job);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* Decode B tokens through one FFN layer.  If given_idx is non-NULL the output
 * is computed on that externally chosen active set instead of the oracle's
 * own (the oracle's own set is still returned in active_idx / n_active).
 * Returns 0, or -1 on a bad argument. */
int orc_decode(const orc_ffn *w, const orc_mat *x, int B, int mode, int score_kind, double param,
               const int32_t *given_idx, const int32_t *given_n, double *out, int32_t *active_idx,
               int32_t *n_active, double *g, double *a, double *u, double *score, double *cond,
               double *cut, double *norms_out, int nthreads) {
    if (!w || !x || B < 0 || !out || !active_idx || !n_active) return -1;
    if (mode < ORC_EXACT || mode > ORC_KEEP_RATIO) return -1;
    if (mode == ORC_KEEP_RATIO && !(param > 0.0 && param <= 1.0)) return -1;
    int F = w->d_ff;
    double *norms = (double *)malloc(sizeof(double) * (size_t)F);
    orc_down_norms(w, norms);
    if (norms_out) memcpy(norms_out, norms, sizeof(double) * F);
    orc_decode_job job;
    memset(&job, 0, sizeof job);
    job.w = w;
    job.x = x;
    job.norms = norms;
    job.mode = mode;
    job.score_kind = score_kind;
    job.param = param;
    job.given_idx = given_idx;
    job.given_n = given_n;
    job.out = out;
    job.active_idx = active_idx;
    job.n_active = n_active;
    job.g = g;
    job.a = a;
    job.u = u;
    job.score = score;
    job.cond = cond;
    job.cut = cut;
    job.B = B;
    job.next = 0;
    pthread_mutex_init(&job.lock, NULL);
    orc_run_workers(orc_decode_worker, &job, nthreads);
    pthread_mutex_destroy(&job.lock);
    free(norms);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Token selection (RedKnot)                                                 */
/* ------------------------------------------------------------------------- */

/* s_t = ||Y_attn[t, :]||_2 in ascending k. */
void orc_token_norms(const orc_mat *y_attn, double *s) {
    for (int t = 0; t < y_attn->rows; ++t) {
        double acc = 0.0;
        for (int k = 0; k < y_attn->cols; ++k) {
            double v = orc_mat_at(y_attn, t, k);
            acc += v * v;
        }
        s[t] = sqrt(acc);
    }
}

/* Selected token set S (ascending in sel_idx), from importances s[L]:
 *   - mass_thresh >= 1, or total mass 0: every token (dense fallback);
 *   - otherwise the shortest prefix of the (s desc, t asc) order whose mass
 *     reaches mass_thresh * total (the crossing token is included; none when
 *     mass_thresh <= 0);
 *   - union the last recent_n tokens;
 *   - if still fewer than min_keep, extend along the same order.
 * prefix_k (optional) receives the length of the pure mass prefix and
 * prefix_idx (optional, [L]) its members in order.  Returns |S|, or -1. */
int orc_mass_select(int L, const double *s, double mass_thresh, int recent_n, int min_keep,
                    int32_t *sel_idx, int32_t *n_sel, int32_t *prefix_k, int32_t *prefix_idx) {
    if (L < 0 || !s || !sel_idx || !n_sel || recent_n < 0 || min_keep < 1) return -1;
    double total = 0.0;
    for (int t = 0; t < L; ++t) total += s[t];
    unsigned char *in = (unsigned char *)calloc((size_t)(L > 0 ? L : 1), 1);
    int k = 0;
    int *order = (int *)malloc(sizeof(int) * (size_t)(L > 0 ? L : 1));
    orc_order_desc(s, L, order);
    if (mass_thresh >= 1.0 || total == 0.0) {
        for (int t = 0; t < L; ++t) in[t] = 1;
        k = L;
    } else if (mass_thresh > 0.0) {
        double target = mass_thresh * total, acc = 0.0;
        while (k < L && acc < target) {
            acc += s[order[k]];
            ++k;
        }
        for (int i = 0; i < k; ++i) in[order[i]] = 1;
    }
    if (prefix_k) *prefix_k = k;
    if (prefix_idx)
        for (int i = 0; i < k; ++i) prefix_idx[i] = (mass_thresh >= 1.0 || total == 0.0) ? i : order[i];
    int tail = recent_n < L ? recent_n : L;
    for (int t = L - tail; t < L; ++t) in[t] = 1;
    int cnt = 0;
    for (int t = 0; t < L; ++t) cnt += in[t];
    int need = min_keep < L ? min_keep : L;
    for (int i = 0; i < L && cnt < need; ++i)
        if (!in[order[i]]) {
            in[order[i]] = 1;
            ++cnt;
        }
    int n = 0;
    for (int t = 0; t < L; ++t)
        if (in[t]) sel_idx[n++] = t;
    *n_sel = n;
    free(order);
    free(in);
    return n;
}

/* ------------------------------------------------------------------------- */
/* Prefill rows (RedKnot Algorithm 1)                                        */
/* ------------------------------------------------------------------------- */

/* Y[t] = bf16_rne(X[t] + Y_attn[t]) for every t: the post-attention residual
 * stream (the sum of two bf16 values is exact in fp64, then one rounding). */
void orc_residual(const orc_mat *X, const orc_mat *Y_attn, uint16_t *Y_bits) {
    for (int t = 0; t < X->rows; ++t)
        for (int k = 0; k < X->cols; ++k)
            Y_bits[(size_t)t * X->cols + k] =
                orc_f64_to_bf16_rne(orc_mat_at(X, t, k) + orc_mat_at(Y_attn, t, k));
}

typedef struct {
    const orc_ffn *w;
    const orc_mat *X, *Y_attn;
    const int32_t *rows;
    const unsigned char *selected; /* [L] */
    int n_rows, next;
    double *z;         /* [n_rows, d] FFN output (0 for unselected) */
    uint16_t *out;     /* [n_rows, d] bf16 bits of Y + Z            */
    pthread_mutex_t lock;
} orc_prefill_job;

static void orc_prefill_one(orc_prefill_job *job, int r) {
    const orc_ffn *w = job->w;
    int d = w->d_model, F = w->d_ff, t = job->rows[r];
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    double *z = job->z + (size_t)r * d;
    for (int k = 0; k < d; ++k)
        y[k] = orc_bf16_to_f64(orc_f64_to_bf16_rne(orc_mat_at(job->X, t, k) + orc_mat_at(job->Y_attn, t, k)));
    for (int i = 0; i < d; ++i) z[i] = 0.0;
    if (job->selected[t]) {
        for (int j = 0; j < F; ++j) {
            double g = orc_row_dot(&w->w_gate, j, y, d, NULL);
            double u = orc_row_dot(&w->w_up, j, y, d, NULL);
            double h = orc_act(w->act, g) * u;
            for (int i = 0; i < d; ++i) z[i] += h * orc_mat_at(&w->w_downT, j, i);
        }
    }
    for (int i = 0; i < d; ++i) job->out[(size_t)r * d + i] = orc_f64_to_bf16_rne(y[i] + z[i]);
    free(y);
}

static void *orc_prefill_worker(void *arg) {
    orc_prefill_job *job = (orc_prefill_job *)arg;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int r = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->n_rows) break;
        orc_prefill_one(job, r);
    }
    return NULL;
}

/* Prefill output rows `rows[0..n_rows)` of a length-L sequence whose selected
 * set is given by `selected[L]` (0/1).  For t in S: out = bf16(Y + FFN(Y));
 * for t not in S: Z = 0 and out = bf16(Y) = Y bit for bit. */
int orc_prefill_rows(const orc_ffn *w, const orc_mat *X, const orc_mat *Y_attn, const unsigned char *selected,
                     const int32_t *rows, int n_rows, double *z, uint16_t *out, int nthreads) {
    if (!w || !X || !Y_attn || !selected || !rows || n_rows < 0 || !z || !out) return -1;
    orc_prefill_job job;
    memset(&job, 0, sizeof job);
    job.w = w;
    job.X = X;
    job.Y_attn = Y_attn;
    job.rows = rows;
    job.selected = selected;
    job.n_rows = n_rows;
    job.z = z;
    job.out = out;
    pthread_mutex_init(&job.lock, NULL);
    orc_run_workers(orc_prefill_worker, &job, nthreads);
    pthread_mutex_destroy(&job.lock);
    return 0;
}
