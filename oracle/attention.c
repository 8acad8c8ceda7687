/*
 * ORACLE -- test infrastructure only.  A plain, slow, obviously correct fp64
 * CPU statement of what the blockwise / ring attention path computes.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never does.  It shares no code with the CUDA library.
 *
 * Sources (web pages on blockwise / ring attention):
 *  - "Attention Is All You Need" summary (#22, #15 sec. 3.2.1) and "PyTorch
 *    scaled_dot_product_attention" (#24) on ai.engineer "Transformers and
 *    Attention": O = softmax(Q K^T / sqrt(d_k)) V, softmax over source
 *    positions, excluded scores get -inf, causal keeps the diagonal and the
 *    lower triangle.
 *  - "PyTorch MultiheadAttention" (#2): key_padding_mask excludes source
 *    positions per batch item, attn_mask excludes (query, source) pairs, and
 *    the exclusions of both Boolean masks are combined.
 *  - "Sequence/context parallelism" (brunomaga), section "Ring Attention":
 *    the output of one query row is a fraction sum_i exp(s_i) v_i /
 *    sum_j exp(s_j); section "Improving numerical stability": subtract the row
 *    maximum; the per-row LSE = log sum_j exp(s_j).
 *  - "RoFormer" summary (#4): split an even-dimensional vector into coordinate
 *    pairs and rotate each pair by its positional angle.
 *
 * The attention here is the definition written out, row by row: every visible
 * score of the row, the row maximum, LSE = max + log(sum exp(s - max)), and
 * O = sum exp(s - LSE) v.  No blocking, no partitions, no merging.  Threads
 * split the list of rows only; each row is computed by one thread in order.
 *
 * Compile with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* attention                                                          */
/* ------------------------------------------------------------------ */

typedef struct {
    const float *q, *k, *v;           /* q: (B,H,L,d)  k, v: (B,H,S,d), contiguous */
    int64_t B, H, L, S, d;
    int64_t q_pos0, k_pos0;           /* global position of query row 0 / key 0 */
    const uint8_t *kpm;               /* (B, kpm_ld) at global key positions, 1 = excluded */
    int64_t kpm_ld;
    const uint8_t *am;                /* (.., am_ld) at global (query, key) positions, 1 = excluded */
    int64_t am_ld;
    int causal;
    double scale;
    const int64_t *rows;              /* flat row ids ((b*H + h)*L + i), or NULL = every row */
    int64_t nrows;
    double *out;                      /* (nrows, d) */
    double *lse;                      /* (nrows) */
    int64_t begin, end;               /* this thread's slice of the row list */
} attn_job;

/* Is key j (local index) visible from query row i (local index) of batch b? */
static int visible(const attn_job *J, int64_t b, int64_t i, int64_t j) {
    int64_t qp = J->q_pos0 + i, kp = J->k_pos0 + j;
    if (J->causal && kp > qp) return 0;
    if (J->kpm && J->kpm[b * J->kpm_ld + kp]) return 0;
    if (J->am && J->am[qp * J->am_ld + kp]) return 0;
    return 1;
}

static void *attn_worker(void *arg) {
    const attn_job *J = (const attn_job *)arg;
    const int64_t S = J->S, d = J->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    unsigned char *vis = (unsigned char *)malloc((size_t)(S > 0 ? S : 1));
    for (int64_t n = J->begin; n < J->end; ++n) {
        int64_t row = J->rows ? J->rows[n] : n;
        int64_t i = row % J->L;
        int64_t bh = row / J->L;
        int64_t b = bh / J->H;
        const float *qi = J->q + row * d;
        const float *kb = J->k + bh * S * d;
        const float *vb = J->v + bh * S * d;
        double *o = J->out + n * d;

        /* scores of the visible keys, and their maximum */
        double m = -INFINITY;
        int64_t nvis = 0;
        for (int64_t j = 0; j < S; ++j) {
            vis[j] = (unsigned char)visible(J, b, i, j);
            if (!vis[j]) continue;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += (double)qi[c] * (double)kb[j * d + c];
            s[j] = dot * J->scale;
            if (s[j] > m) m = s[j];
            ++nvis;
        }
        for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
        if (nvis == 0) {                 /* no visible key: O = 0, LSE = -inf */
            J->lse[n] = -INFINITY;
            continue;
        }
        /* LSE = log sum exp(s_j), with the maximum subtracted */
        double sum = 0.0;
        for (int64_t j = 0; j < S; ++j)
            if (vis[j]) sum += exp(s[j] - m);
        double L = m + log(sum);
        J->lse[n] = L;
        /* O = sum_j exp(s_j - LSE) v_j */
        for (int64_t j = 0; j < S; ++j) {
            if (!vis[j]) continue;
            double w = exp(s[j] - L);
            for (int64_t c = 0; c < d; ++c) o[c] += w * (double)vb[j * d + c];
        }
    }
    free(s);
    free(vis);
    return NULL;
}

/*
 * Exact (fp64) attention of the rows listed in `rows` (or of every row when
 * rows == NULL; then nrows must be B*H*L).  Inputs are float32 arrays holding
 * the exact values of the stored tensors (bf16 values are exact in float32).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention(const float *q, const float *k, const float *v,
                     int64_t B, int64_t H, int64_t L, int64_t S, int64_t d,
                     int64_t q_pos0, int64_t k_pos0,
                     const uint8_t *kpm, int64_t kpm_ld,
                     const uint8_t *am, int64_t am_ld,
                     int causal, double scale,
                     const int64_t *rows, int64_t nrows,
                     double *out, double *lse, int nthreads) {
    if (!q || !k || !v || !out || !lse || B < 0 || H < 0 || L < 0 || S < 0 || d <= 0) return -1;
    if (!rows && nrows != B * H * L) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nrows < nthreads) nthreads = nrows > 0 ? (int)nrows : 1;
    attn_job base;
    memset(&base, 0, sizeof base);
    base.q = q; base.k = k; base.v = v;
    base.B = B; base.H = H; base.L = L; base.S = S; base.d = d;
    base.q_pos0 = q_pos0; base.k_pos0 = k_pos0;
    base.kpm = kpm; base.kpm_ld = kpm_ld; base.am = am; base.am_ld = am_ld;
    base.causal = causal; base.scale = scale > 0 ? scale : 1.0 / sqrt((double)d);
    base.rows = rows; base.nrows = nrows; base.out = out; base.lse = lse;

    attn_job *jobs = (attn_job *)malloc(sizeof(attn_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = nrows * t / nthreads;
        jobs[t].end = nrows * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* ------------------------------------------------------------------ */
/* RoPE                                                               */
/* ------------------------------------------------------------------ */

/* Round a double to the nearest bfloat16 value (ties to even), returned as a
 * float (exact).  bfloat16 keeps 8 significant bits and float32's exponent
 * range; below 2^-126 its spacing is 2^-133. */
static float round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return (float)x;
    int e;
    frexp(x, &e);                     /* |x| in [2^(e-1), 2^e) */
    int qe = e - 8;                   /* spacing of 8-significant-bit values there */
    if (qe < -133) qe = -133;
    double r = nearbyint(ldexp(x, -qe));   /* default rounding mode: ties to even */
    return (float)ldexp(r, qe);
}

float oracle_round_bf16(double x) { return round_bf16(x); }

/*
 * Rotary position embedding of x (BH rows blocks of (T, d), contiguous).
 * For pair c in [0, d/2): theta_c = base^(-2c/d), angle = m * theta_c with m
 * the position of the row (positions[t], or t when positions == NULL), and
 * (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos) on coordinates (2c, 2c+1).
 * Result written as doubles to y64 (unrounded) when y64 != NULL, and rounded
 * to the storage type into y32 (round_mode 1 = float32, 2 = bfloat16) when
 * y32 != NULL.
 */
int oracle_rope(const float *x, int64_t BH, int64_t T, int64_t d,
                const int64_t *positions, double base, double pos_scale, int round_mode,
                double *y64, float *y32) {
    if (!x || d <= 0 || (d & 1)) return -1;
    for (int64_t r = 0; r < BH; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            /* Position Interpolation ("Extending Context Window of Large Language
             * Models via Position Interpolation" summary, #59): the position index is
             * rescaled before the rotary angle is formed; pos_scale = 1 is plain RoPE. */
            double m = (positions ? (double)positions[t] : (double)t) * pos_scale;
            const float *xr = x + (r * T + t) * d;
            for (int64_t c = 0; c < d / 2; ++c) {
                double theta = pow(base, -(double)(2 * c) / (double)d);
                double ang = m * theta;
                double cs = cos(ang), sn = sin(ang);
                double x0 = (double)xr[2 * c], x1 = (double)xr[2 * c + 1];
                double a = x0 * cs;
                double b = x1 * sn;
                double y0 = a - b;
                double e = x0 * sn;
                double f = x1 * cs;
                double y1 = e + f;
                int64_t o = (r * T + t) * d + 2 * c;
                if (y64) { y64[o] = y0; y64[o + 1] = y1; }
                if (y32) {
                    if (round_mode == 2) { y32[o] = round_bf16(y0); y32[o + 1] = round_bf16(y1); }
                    else { y32[o] = (float)y0; y32[o + 1] = (float)y1; }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* attention backward                                                 */
/* ------------------------------------------------------------------ */

/*
 * Gradients of the attention of the section above with respect to q, k and v,
 * contracted with dout: the plain chain rule through O_i = sum_j p_ij v_j,
 * p_ij = exp(s_ij - LSE_i), s_ij = scale q_i . k_j over the visible j.  With
 * D_i = dout_i . O_i ("Sequence/context parallelism" (brunomaga), section
 * "Ring Attention", backward pass: the per-block gradients use the saved out
 * and LSE of the whole row):
 *   dV_j += p_ij dout_i,   dp_ij = dout_i . v_j,   ds_ij = p_ij (dp_ij - D_i),
 *   dQ_i  = scale sum_j ds_ij k_j,   dK_j += scale ds_ij q_i.
 * One thread takes whole (b, h) pairs, row after row, so dK and dV of a head
 * are summed by one thread in row order.
 */
typedef struct {
    attn_job a;                       /* geometry, masks, scale (rows unused) */
    const float *dout;                /* (B,H,L,d) */
    double *dq, *dk, *dv;             /* (B,H,L,d), (B,H,S,d), (B,H,S,d), zero on entry */
    int64_t bh_begin, bh_end;
} bwd_job;

static void *bwd_worker(void *arg) {
    const bwd_job *W = (const bwd_job *)arg;
    const attn_job *J = &W->a;
    const int64_t L = J->L, S = J->S, d = J->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    unsigned char *vis = (unsigned char *)malloc((size_t)(S > 0 ? S : 1));
    for (int64_t bh = W->bh_begin; bh < W->bh_end; ++bh) {
        const int64_t b = bh / J->H;
        const float *kb = J->k + bh * S * d;
        const float *vb = J->v + bh * S * d;
        double *dkb = W->dk + bh * S * d;
        double *dvb = W->dv + bh * S * d;
        for (int64_t i = 0; i < L; ++i) {
            const int64_t row = bh * L + i;
            const float *qi = J->q + row * d;
            const float *gi = W->dout + row * d;
            double *dqi = W->dq + row * d;
            double m = -INFINITY;
            int64_t nvis = 0;
            for (int64_t j = 0; j < S; ++j) {
                vis[j] = (unsigned char)visible(J, b, i, j);
                if (!vis[j]) continue;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += (double)qi[c] * (double)kb[j * d + c];
                s[j] = dot * J->scale;
                if (s[j] > m) m = s[j];
                ++nvis;
            }
            J->lse[row] = -INFINITY;
            for (int64_t c = 0; c < d; ++c) J->out[row * d + c] = 0.0;
            if (nvis == 0) continue;   /* no visible key: out = 0 and every gradient of the row is 0 */
            double sum = 0.0;
            for (int64_t j = 0; j < S; ++j)
                if (vis[j]) sum += exp(s[j] - m);
            const double lse = m + log(sum);
            J->lse[row] = lse;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = 0; j < S; ++j) {
                if (!vis[j]) continue;
                p[j] = exp(s[j] - lse);
                for (int64_t c = 0; c < d; ++c) o[c] += p[j] * (double)vb[j * d + c];
            }
            double D = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                J->out[row * d + c] = o[c];
                D += (double)gi[c] * o[c];
            }
            for (int64_t j = 0; j < S; ++j) {
                if (!vis[j]) continue;
                double dp = 0.0;
                for (int64_t c = 0; c < d; ++c) dp += (double)gi[c] * (double)vb[j * d + c];
                const double ds = p[j] * (dp - D);
                for (int64_t c = 0; c < d; ++c) {
                    dvb[j * d + c] += p[j] * (double)gi[c];
                    dqi[c] += J->scale * ds * (double)kb[j * d + c];
                    dkb[j * d + c] += J->scale * ds * (double)qi[c];
                }
            }
        }
    }
    free(s);
    free(p);
    free(o);
    free(vis);
    return NULL;
}

/*
 * Exact (fp64) attention gradients.  dq, dk, dv, out, lse are written in full
 * (out and lse are the forward values of the same call).  Returns 0, or -1 on
 * a bad argument.
 */
int oracle_attention_bwd(const float *q, const float *k, const float *v, const float *dout,
                         int64_t B, int64_t H, int64_t L, int64_t S, int64_t d,
                         int64_t q_pos0, int64_t k_pos0,
                         const uint8_t *kpm, int64_t kpm_ld,
                         const uint8_t *am, int64_t am_ld,
                         int causal, double scale,
                         double *dq, double *dk, double *dv, double *out, double *lse, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !out || !lse) return -1;
    if (B < 0 || H < 0 || L < 0 || S < 0 || d <= 0) return -1;
    const int64_t BH = B * H;
    memset(dq, 0, sizeof(double) * (size_t)(BH * L * d));
    memset(dk, 0, sizeof(double) * (size_t)(BH * S * d));
    memset(dv, 0, sizeof(double) * (size_t)(BH * S * d));
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (BH < nthreads) nthreads = BH > 0 ? (int)BH : 1;
    bwd_job base;
    memset(&base, 0, sizeof base);
    base.a.q = q; base.a.k = k; base.a.v = v;
    base.a.B = B; base.a.H = H; base.a.L = L; base.a.S = S; base.a.d = d;
    base.a.q_pos0 = q_pos0; base.a.k_pos0 = k_pos0;
    base.a.kpm = kpm; base.a.kpm_ld = kpm_ld; base.a.am = am; base.a.am_ld = am_ld;
    base.a.causal = causal; base.a.scale = scale > 0 ? scale : 1.0 / sqrt((double)d);
    base.a.out = out; base.a.lse = lse;
    base.dout = dout; base.dq = dq; base.dk = dk; base.dv = dv;
    bwd_job *jobs = (bwd_job *)malloc(sizeof(bwd_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].bh_begin = BH * t / nthreads;
        jobs[t].bh_end = BH * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, bwd_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}
