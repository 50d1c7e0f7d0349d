/*
 * attn_oracle.c -- plain fp64 CPU oracle for softcapped / sink / masked attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the method, written out as its definition, in fp64):
 *
 *   For batch b, query head h, kv head g = h / (Hq/Hkv)        [GQA: contiguous groups]
 *   u_ij  = scale * sum_d q[b,i,h,d] k[b,j,g,d] + bias[b,h,i,j]
 *             -- post-scale additive bias ("post_scale_bias", TransformerEngine PR #3551,
 *                Greptile review "Offset Corrupts Bias Gradient Shape")
 *   t_ij  = cap * tanh(u_ij / cap)            if cap > 0, else u_ij
 *             -- tanh logit soft-capping, applied after the scale and the bias add and
 *                before masking (TransformerEngine PR #3391 intro; tokamax PR #1121 body)
 *   vis_ij = [causal => j <= i + Sk - Sq] and [W > 0 => (i + Sk - Sq) - j < W]
 *            and [segments => seg_q[b,i] == seg_k[b,j]]
 *             -- causal / sliding-window / packed-segment masks (MaxText commit message
 *                quoted on tokamax PR #1121: sliding window, packing, segment ids)
 *   Z_i   = [sink? exp(sink_h) : 0] + sum_{j vis} exp(t_ij),   LSE_i = ln Z_i
 *             -- the learnable sink is one extra softmax column with logit sink_h that
 *                enters each row exactly once (TransformerEngine PR #3551, "What changed")
 *   P_ij  = vis_ij * exp(t_ij - LSE_i),  p0_i = exp(sink_h - LSE_i)
 *   O_i   = sum_j P_ij v_j                      (the sink column carries no value)
 *
 * Backward (analytic; tokamax PR #1121 body for the cap chain rule, TransformerEngine
 * PR #3551 "What changed" for the sink gradient):
 *   D_i   = dO_i . O_i
 *   dP_ij = dO_i . v_j
 *   dT_ij = P_ij (dP_ij - D_i)
 *   dU_ij = dT_ij * (1 - tanh^2(u_ij / cap))    (factor 1 when cap == 0; taken from the
 *                                                finite pre-mask u)
 *   dQ_i  = scale * sum_j dU_ij k_j
 *   dK_j  = scale * sum_{h in group} sum_i dU_ij q_i
 *   dV_j  = sum_{h in group} sum_i P_ij dO_i
 *   dbias = dU summed over the bias's broadcast dimensions
 *   dsink_h = - sum_{b,i} p0_i D_i
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - the window W bounds how far back a key may lie: visible only if
 *     (i + Sk - Sq) - j < W, so with causal a row sees W keys including itself;
 *     the window sets no upper bound of its own (that is the causal flag's job);
 *     W <= 0 means no window;
 *   - causal alignment is bottom-right when Sq != Sk;
 *   - the sink logit is used raw: not scaled, not capped, no bias;
 *   - a row with nothing visible and no sink has LSE = -inf, O = 0 and zero gradients.
 *
 * Evaluation note: ln Z_i is evaluated as m + ln(sum exp(x - m)) with m the largest
 * term of the row; in exact arithmetic this is the same number, and in fp64 it only
 * keeps exp() from overflowing.
 *
 * All arrays are dense row-major fp64 (int32 for segment ids):
 *   q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D], O/dO/dQ [B,Sq,Hq,D], dK/dV [B,Sk,Hkv,D],
 *   LSE and Dvec [B,Hq,Sq], bias/dbias [Bb,Hb,Sq,Sk] with Bb in {1,B}, Hb in {1,Hq},
 *   seg_q [B,Sq], seg_k [B,Sk], sink/dsink [Hq].
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>

typedef struct {
    int B, Sq, Sk, Hq, Hkv, D;
    const double *q, *k, *v;
    const double *bias;   /* NULL: no bias */
    int bias_B, bias_H;   /* 1 = broadcast over that dimension, else B / Hq */
    const int32_t *seg_q, *seg_k; /* both NULL or both set */
    int causal, window;
    double softcap;       /* 0: off */
    const double *sink;   /* NULL: no sink */
    double scale;
} oracle_problem;

static const double *q_row(const oracle_problem *p, int b, int i, int h) {
    return p->q + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
}
static const double *k_row(const oracle_problem *p, int b, int j, int g) {
    return p->k + (((size_t)b * p->Sk + j) * p->Hkv + g) * p->D;
}
static const double *v_row(const oracle_problem *p, int b, int j, int g) {
    return p->v + (((size_t)b * p->Sk + j) * p->Hkv + g) * p->D;
}
static size_t bias_index(const oracle_problem *p, int b, int h, int i, int j) {
    int bb = p->bias_B == 1 ? 0 : b;
    int hb = p->bias_H == 1 ? 0 : h;
    return (((size_t)bb * p->bias_H + hb) * p->Sq + i) * p->Sk + j;
}
static int kv_head(const oracle_problem *p, int h) { return h / (p->Hq / p->Hkv); }

/* Visibility of key j to query i (causal, sliding window, packed segments). */
int oracle_visible(const oracle_problem *p, int b, int i, int j) {
    int ipos = i + p->Sk - p->Sq;          /* query position on the key axis */
    if (p->causal && j > ipos) return 0;
    if (p->window > 0 && ipos - j >= p->window) return 0;
    if (p->seg_q && p->seg_q[(size_t)b * p->Sq + i] != p->seg_k[(size_t)b * p->Sk + j]) return 0;
    return 1;
}

/* Pre-cap logit u_ij (scale * q.k + bias). */
static double logit_u(const oracle_problem *p, int b, int h, int i, int j) {
    const double *qi = q_row(p, b, i, h);
    const double *kj = k_row(p, b, j, kv_head(p, h));
    double s = 0.0;
    for (int d = 0; d < p->D; ++d) s += qi[d] * kj[d];
    double u = p->scale * s;
    if (p->bias) u += p->bias[bias_index(p, b, h, i, j)];
    return u;
}

/* Capped logit t = cap * tanh(u / cap) (identity when cap == 0). */
static double capped(const oracle_problem *p, double u) {
    return p->softcap > 0.0 ? p->softcap * tanh(u / p->softcap) : u;
}

/* d t / d u = 1 - tanh^2(u / cap), from the finite pre-mask u. */
static double cap_factor(const oracle_problem *p, double u) {
    if (!(p->softcap > 0.0)) return 1.0;
    double th = tanh(u / p->softcap);
    return 1.0 - th * th;
}

/*
 * Logits of one row: u[j] (pre-cap) and t[j] (capped) for every key j, and vis[j].
 * Buffers hold Sk entries; entries of invisible keys are still filled (u, t finite).
 */
static void row_logits(const oracle_problem *p, int b, int h, int i,
                       double *u, double *t, uint8_t *vis) {
    for (int j = 0; j < p->Sk; ++j) {
        vis[j] = (uint8_t)oracle_visible(p, b, i, j);
        u[j] = logit_u(p, b, h, i, j);
        t[j] = capped(p, u[j]);
    }
}

/* LSE_i = ln( [e^sink] + sum_{vis} e^{t_ij} ), evaluated around the row's largest term. */
static double row_lse(const oracle_problem *p, int h, const double *t, const uint8_t *vis) {
    double m = -INFINITY;
    if (p->sink) m = p->sink[h];
    for (int j = 0; j < p->Sk; ++j)
        if (vis[j] && t[j] > m) m = t[j];
    if (m == -INFINITY) return -INFINITY;           /* empty row, no sink */
    double z = p->sink ? exp(p->sink[h] - m) : 0.0;
    for (int j = 0; j < p->Sk; ++j)
        if (vis[j]) z += exp(t[j] - m);
    return m + log(z);
}

/* Row scratch: u, t (Sk doubles each) and vis (Sk bytes). */
typedef struct { double *u, *t; uint8_t *vis; } row_buf;
static row_buf row_buf_new(const oracle_problem *p) {
    row_buf r;
    r.u = (double *)malloc(sizeof(double) * (size_t)p->Sk);
    r.t = (double *)malloc(sizeof(double) * (size_t)p->Sk);
    r.vis = (uint8_t *)malloc((size_t)p->Sk);
    return r;
}
static void row_buf_free(row_buf *r) { free(r->u); free(r->t); free(r->vis); }

/*
 * Forward.  Computes O [B,Sq,Hq,D] and LSE [B,Hq,Sq] for every row i with
 * row_mask[i] != 0 (row_mask NULL: all rows); other rows are left untouched.
 */
void oracle_forward(const oracle_problem *p, const uint8_t *row_mask, double *O, double *LSE) {
    long nrows = (long)p->B * p->Hq * p->Sq;
#pragma omp parallel
    {
        row_buf rb = row_buf_new(p);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < nrows; ++r) {
            int i = (int)(r % p->Sq);
            int h = (int)((r / p->Sq) % p->Hq);
            int b = (int)(r / ((long)p->Sq * p->Hq));
            if (row_mask && !row_mask[i]) continue;
            int g = kv_head(p, h);
            row_logits(p, b, h, i, rb.u, rb.t, rb.vis);
            double lse = row_lse(p, h, rb.t, rb.vis);
            LSE[((size_t)b * p->Hq + h) * p->Sq + i] = lse;
            double *o = O + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
            for (int d = 0; d < p->D; ++d) o[d] = 0.0;
            if (lse == -INFINITY) continue;
            for (int j = 0; j < p->Sk; ++j) {
                if (!rb.vis[j]) continue;
                double pij = exp(rb.t[j] - lse);
                const double *vj = v_row(p, b, j, g);
                for (int d = 0; d < p->D; ++d) o[d] += pij * vj[d];
            }
        }
        row_buf_free(&rb);
    }
}

/* D_i = dO_i . O_i for every (b, h, i): Dvec [B,Hq,Sq].  O must hold every row. */
void oracle_rowdot(const oracle_problem *p, const double *dO, const double *O, double *Dvec) {
    long nrows = (long)p->B * p->Hq * p->Sq;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < nrows; ++r) {
        int i = (int)(r % p->Sq);
        int h = (int)((r / p->Sq) % p->Hq);
        int b = (int)(r / ((long)p->Sq * p->Hq));
        const double *o = O + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
        const double *go = dO + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
        double s = 0.0;
        for (int d = 0; d < p->D; ++d) s += go[d] * o[d];
        Dvec[((size_t)b * p->Hq + h) * p->Sq + i] = s;
    }
}

/* dP_ij = dO_i . v_j */
static double grad_p(const oracle_problem *p, const double *dO, int b, int h, int i, int j) {
    const double *go = dO + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
    const double *vj = v_row(p, b, j, kv_head(p, h));
    double dp = 0.0;
    for (int d = 0; d < p->D; ++d) dp += go[d] * vj[d];
    return dp;
}

/* dU_ij = P_ij (dP_ij - D_i) (1 - tanh^2(u_ij/cap)); 0 where not visible. */
static double grad_u(const oracle_problem *p, const double *dO, int b, int h, int i, int j,
                     double lse, double Di) {
    if (!oracle_visible(p, b, i, j) || lse == -INFINITY) return 0.0;
    double u = logit_u(p, b, h, i, j);
    double pij = exp(capped(p, u) - lse);
    return pij * (grad_p(p, dO, b, h, i, j) - Di) * cap_factor(p, u);
}

/*
 * dQ rows: dQ_i = scale * sum_j dU_ij k_j, for rows with row_mask[i] (NULL: all).
 * LSE and Dvec must be valid on those rows.
 */
void oracle_backward_dq(const oracle_problem *p, const double *dO, const double *LSE,
                        const double *Dvec, const uint8_t *row_mask, double *dQ) {
    long nrows = (long)p->B * p->Hq * p->Sq;
#pragma omp parallel
    {
        row_buf rb = row_buf_new(p);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < nrows; ++r) {
            int i = (int)(r % p->Sq);
            int h = (int)((r / p->Sq) % p->Hq);
            int b = (int)(r / ((long)p->Sq * p->Hq));
            if (row_mask && !row_mask[i]) continue;
            int g = kv_head(p, h);
            size_t ri = ((size_t)b * p->Hq + h) * p->Sq + i;
            double lse = LSE[ri], Di = Dvec[ri];
            double *dq = dQ + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
            for (int d = 0; d < p->D; ++d) dq[d] = 0.0;
            if (lse == -INFINITY) continue;
            row_logits(p, b, h, i, rb.u, rb.t, rb.vis);
            for (int j = 0; j < p->Sk; ++j) {
                if (!rb.vis[j]) continue;
                double pij = exp(rb.t[j] - lse);
                double du = pij * (grad_p(p, dO, b, h, i, j) - Di) * cap_factor(p, rb.u[j]);
                const double *kj = k_row(p, b, j, g);
                for (int d = 0; d < p->D; ++d) dq[d] += p->scale * du * kj[d];
            }
        }
        row_buf_free(&rb);
    }
}

/*
 * dK, dV columns: for every (b, g, j) with col_mask[j] (NULL: all),
 *   dK_j = scale * sum_{h in group g} sum_i dU_ij q_i,   dV_j = sum_{h,i} P_ij dO_i.
 * LSE and Dvec must be valid on every row.
 */
void oracle_backward_dkdv(const oracle_problem *p, const double *dO, const double *LSE,
                          const double *Dvec, const uint8_t *col_mask, double *dK, double *dV) {
    int G = p->Hq / p->Hkv;
    long ncols = (long)p->B * p->Hkv * p->Sk;
#pragma omp parallel for schedule(dynamic, 4)
    for (long c = 0; c < ncols; ++c) {
        int j = (int)(c % p->Sk);
        int g = (int)((c / p->Sk) % p->Hkv);
        int b = (int)(c / ((long)p->Sk * p->Hkv));
        if (col_mask && !col_mask[j]) continue;
        double *dk = dK + (((size_t)b * p->Sk + j) * p->Hkv + g) * p->D;
        double *dv = dV + (((size_t)b * p->Sk + j) * p->Hkv + g) * p->D;
        for (int d = 0; d < p->D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
        for (int h = g * G; h < (g + 1) * G; ++h)
            for (int i = 0; i < p->Sq; ++i) {
                size_t ri = ((size_t)b * p->Hq + h) * p->Sq + i;
                if (!oracle_visible(p, b, i, j) || LSE[ri] == -INFINITY) continue;
                double u = logit_u(p, b, h, i, j);
                double pij = exp(capped(p, u) - LSE[ri]);
                const double *go = dO + (((size_t)b * p->Sq + i) * p->Hq + h) * p->D;
                for (int d = 0; d < p->D; ++d) dv[d] += pij * go[d];
                double du = pij * (grad_p(p, dO, b, h, i, j) - Dvec[ri]) * cap_factor(p, u);
                const double *qi = q_row(p, b, i, h);
                for (int d = 0; d < p->D; ++d) dk[d] += p->scale * du * qi[d];
            }
    }
}

/* dbias [bias_B, bias_H, Sq, Sk] = dU summed over the broadcast dimensions. */
void oracle_backward_dbias(const oracle_problem *p, const double *dO, const double *LSE,
                           const double *Dvec, double *dbias) {
    long nrows = (long)p->bias_B * p->bias_H * p->Sq;
#pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < nrows; ++r) {
        int i = (int)(r % p->Sq);
        int hb = (int)((r / p->Sq) % p->bias_H);
        int bb = (int)(r / ((long)p->Sq * p->bias_H));
        for (int j = 0; j < p->Sk; ++j) {
            double acc = 0.0;
            for (int b = 0; b < p->B; ++b) {
                if (p->bias_B != 1 && b != bb) continue;
                for (int h = 0; h < p->Hq; ++h) {
                    if (p->bias_H != 1 && h != hb) continue;
                    size_t ri = ((size_t)b * p->Hq + h) * p->Sq + i;
                    acc += grad_u(p, dO, b, h, i, j, LSE[ri], Dvec[ri]);
                }
            }
            dbias[(((size_t)bb * p->bias_H + hb) * p->Sq + i) * p->Sk + j] = acc;
        }
    }
}

/* dsink_h = - sum_{b,i} exp(sink_h - LSE_i) D_i  (sum over every batch and row). */
void oracle_backward_dsink(const oracle_problem *p, const double *LSE, const double *Dvec,
                           double *dsink) {
    for (int h = 0; h < p->Hq; ++h) {
        double acc = 0.0;
        for (int b = 0; b < p->B; ++b)
            for (int i = 0; i < p->Sq; ++i) {
                size_t ri = ((size_t)b * p->Hq + h) * p->Sq + i;
                acc += exp(p->sink[h] - LSE[ri]) * Dvec[ri];
            }
        dsink[h] = -acc;
    }
}

/* Number of visible (i, j) pairs for one (b): brute force over the definition. */
long long oracle_count_visible(const oracle_problem *p, int b) {
    long long n = 0;
    for (int i = 0; i < p->Sq; ++i)
        for (int j = 0; j < p->Sk; ++j) n += oracle_visible(p, b, i, j);
    return n;
}

/* Visible keys of query row i of batch b (the mask definition, key by key): how many, and the
 * first and last of them (-1 when none).  Used to check the GPU's per-tile mask metadata. */
void oracle_row_visible(const oracle_problem *p, int b, int i, long long *count, int *first, int *last) {
    long long n = 0;
    int f = -1, l = -1;
    for (int j = 0; j < p->Sk; ++j) {
        if (!oracle_visible(p, b, i, j)) continue;
        if (f < 0) f = j;
        l = j;
        ++n;
    }
    *count = n;
    *first = f;
    *last = l;
}

/* The same for key j: the queries that see it. */
void oracle_col_visible(const oracle_problem *p, int b, int j, long long *count, int *first, int *last) {
    long long n = 0;
    int f = -1, l = -1;
    for (int i = 0; i < p->Sq; ++i) {
        if (!oracle_visible(p, b, i, j)) continue;
        if (f < 0) f = i;
        l = i;
        ++n;
    }
    *count = n;
    *first = f;
    *last = l;
}

/* Capped logit and its derivative factor, exposed for the pins. */
double oracle_capped(const oracle_problem *p, double u) { return capped(p, u); }
double oracle_cap_factor(const oracle_problem *p, double u) { return cap_factor(p, u); }
