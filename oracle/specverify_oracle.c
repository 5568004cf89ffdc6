/*
 * specverify_oracle.c -- plain fp64 CPU oracle of the speculative-decoding
 * verification step.
 *
 * TEST INFRASTRUCTURE ONLY (see specverify_oracle.h): the checker of the CUDA
 * library, never a fallback for it. Single-threaded, one request at a time,
 * one position at a time, in the order the pages describe the method. Every
 * logit is widened exactly to double; every probability, sum and comparison
 * is done in double. Nothing is blocked, fused or reordered: each row's
 * softmax is recomputed from its logits where the algorithm needs it.
 */
#include "specverify_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

int oracle_version(void) { return 1; }

/* Logit idx of a tensor: binary32 read as is; a bfloat16 holds the top 16
 * bits of a binary32, so it widens exactly by a 16-bit shift. */
static double logit_at(const void* base, int dtype, size_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void* base, int dtype, size_t row, int V, double* l) {
    for (int x = 0; x < V; ++x) l[x] = logit_at(base, dtype, row * (size_t)V + (size_t)x);
}

/* A row can be used when it holds no NaN, no +inf, and at least one value
 * above -inf (a row of only -inf has no distribution). Any finite logit is
 * allowed, at any T > 0: the softmax below is formed in double from the
 * differences l - max, which stay in range whatever the magnitude of l. */
static int row_usable(const double* l, int V) {
    int has_finite = 0;
    for (int x = 0; x < V; ++x) {
        if (isnan(l[x])) return 0;
        if (isinf(l[x])) {
            if (l[x] > 0) return 0;
        } else {
            has_finite = 1;
        }
    }
    return has_finite;
}

static double row_max(const double* l, int V) {
    double m = l[0];
    for (int x = 1; x < V; ++x)
        if (l[x] > m) m = l[x];
    return m;
}

/* Greedy rule of "Speculative Decoding : accélérer l'inférence des LLM",
 * §Pourquoi la qualité est préservée: the target's most likely token; on a
 * tie the lowest index (reading: the pages do not say). */
static int row_argmax(const double* l, int V) {
    int a = 0;
    for (int x = 1; x < V; ++x)
        if (l[x] > l[a]) a = x;
    return a;
}

/* Temperature softmax p(x) = exp(l(x)/T) / sum_y exp(l(y)/T), for any
 * T > 0, evaluated as exp((l(x) - m)/T) / Z with m the row max, so that no
 * term overflows; Z is summed in index order. Reports m and log Z (either
 * pointer may be NULL) and returns log sum_y exp(l(y)/T) = m/T + log Z. */
static double softmax_T2(const double* l, int V, double T, double* p, double* m_out, double* logZ_out) {
    double m = row_max(l, V);
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        p[x] = exp((l[x] - m) / T);
        Z += p[x];
    }
    for (int x = 0; x < V; ++x) p[x] /= Z;
    if (m_out) *m_out = m;
    if (logZ_out) *logZ_out = log(Z);
    return m / T + log(Z);
}

static double softmax_T(const double* l, int V, double T, double* p) {
    return softmax_T2(l, V, T, p, NULL, NULL);
}

/* alpha = min(1, p(x) / q(x)) (eq. alpha(x) of the wiki page "Speculative
 * Decoding") for softmax rows with maxima m_p, m_q and log-normalisers
 * logZ_p, logZ_q: log p(x) - log q(x) = ((l_t(x) - m_p) - (l_d(x) - m_q)) / T
 * - (logZ_p - logZ_q). The differences to the row maxima are formed first, so
 * the value stays accurate at any T > 0 and any logit magnitude, and it is
 * still defined when both probabilities lie below the fp64 range (at small T
 * they underflow together while their ratio need not be small). A softmax
 * probability is 0 only at a -inf logit: then alpha = 1 if q(x) = 0 < p(x),
 * 0 if p(x) = 0 (reading R3). */
static double accept_alpha(double lt_x, double m_p, double logZ_p, double ld_x, double m_q, double logZ_q,
                           double T) {
    if (lt_x == -INFINITY) return 0.0;
    if (ld_x == -INFINITY) return 1.0;
    const double lr = ((lt_x - m_p) - (ld_x - m_q)) / T - (logZ_p - logZ_q);
    return lr >= 0.0 ? 1.0 : exp(lr);
}

/* The acceptance test u < alpha for u in [0, 1). alpha is positive whenever
 * p(x) > 0 (a finite target logit), also where its double value underflowed
 * to 0; the only uniform below such an alpha is u = 0. */
static int accepts(double u, double alpha, int p_positive) {
    if (!p_positive) return 0;
    return u < alpha || u == 0.0;
}

/* For the checker: the measure of {t in [0, W) : |t - e| <= delta for an edge
 * e of the inverse CDF}, divided by W, with delta = ORACLE_TIE_MARGIN * W and
 * the edges 0, C_0, ..., C_{V-1} = W in index order (non-decreasing): the
 * union of the intervals [e - delta, e + delta], merged left to right and
 * clipped to [0, W]. */
static double tie_measure(const double* w, int V, double W) {
    if (!(W > 0.0)) return 1.0;
    const double delta = ORACLE_TIE_MARGIN * W;
    double lo = 0.0, hi = delta, total = 0.0, C = 0.0;
    for (int k = 0; k < V; ++k) {
        C += w[k];
        const double a = C - delta, b = C + delta;
        if (a <= hi) {
            if (b > hi) hi = b;
        } else {
            total += hi - lo;
            lo = a;
            hi = b;
        }
    }
    if (hi > W) hi = W;
    if (lo < W) total += hi - lo;
    return total / W;
}

/* Inverse-CDF draw over non-negative weights w (need not sum to one):
 * W = sum w, t = u * W, and the token is the smallest k whose inclusive
 * prefix sum C_k exceeds t, so a zero-weight token is never drawn. If
 * rounding leaves no such k, the last k with w_k > 0. Reports W and the
 * distance of t to the nearer edge of the chosen interval, divided by W. */
static int draw_inverse_cdf(const double* w, int V, double u, double* W_out,
                            double* margin_out) {
    double W = 0.0;
    for (int x = 0; x < V; ++x) W += w[x];
    *W_out = W;
    double t = u * W;
    double C = 0.0;
    for (int k = 0; k < V; ++k) {
        double before = C;
        C += w[k];
        if (C > t) {
            double lo = t - before, hi = C - t;
            *margin_out = (lo < hi ? lo : hi) / W;
            return k;
        }
    }
    *margin_out = 0.0;
    for (int k = V - 1; k >= 0; --k)
        if (w[k] > 0.0) return k;
    return 0; /* unreachable: callers pass W > 0 */
}

static void set_d(double* a, size_t i, double v) {
    if (a) a[i] = v;
}
static void set_i(int32_t* a, size_t i, int32_t v) {
    if (a) a[i] = v;
}

typedef struct {
    const void* target;
    const void* draft;
    int dtype, gamma, V;
    double *lt, *ld, *p, *q, *w;
} scratch_t;

/* Report-only pass for the checker: the max, argmax and log-normaliser of
 * every row the request reads. It does not feed the decisions. */
static void report_rows(const scratch_t* s, int b, double T, const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    for (int i = 0; i <= G; ++i) {
        size_t r = (size_t)b * (size_t)(G + 1) + (size_t)i;
        load_row(s->target, s->dtype, r, V, s->lt);
        set_d(d->max_target, r, row_max(s->lt, V));
        set_i(d->argmax_target, r, row_argmax(s->lt, V));
        if (T > 0.0) set_d(d->lse_target, r, softmax_T(s->lt, V, T, s->p));
    }
    if (T > 0.0) {
        for (int i = 0; i < G; ++i) {
            size_t r = (size_t)b * (size_t)G + (size_t)i;
            load_row(s->draft, s->dtype, r, V, s->ld);
            set_d(d->max_draft, r, row_max(s->ld, V));
            set_d(d->lse_draft, r, softmax_T(s->ld, V, T, s->q));
        }
    }
}

static void clear_detail(const oracle_detail* d, int b, int G) {
    for (int i = 0; i <= G; ++i) {
        size_t r = (size_t)b * (size_t)(G + 1) + (size_t)i;
        set_d(d->max_target, r, NAN);
        set_d(d->lse_target, r, NAN);
        set_i(d->argmax_target, r, -1);
    }
    for (int i = 0; i < G; ++i) {
        size_t r = (size_t)b * (size_t)G + (size_t)i;
        set_d(d->max_draft, r, NAN);
        set_d(d->lse_draft, r, NAN);
        set_d(d->p_x, r, NAN);
        set_d(d->q_x, r, NAN);
        set_d(d->alpha, r, NAN);
        set_d(d->accept_margin, r, NAN);
    }
    set_d(d->w_total, (size_t)b, NAN);
    set_d(d->sample_margin, (size_t)b, NAN);
    set_d(d->tie_measure, (size_t)b, NAN);
    set_i(d->kind, (size_t)b, ORACLE_KIND_ERROR);
}

/* Whether request b can be verified at all (see the header for the rule). */
static int request_valid(const scratch_t* s, int b, double T, const int32_t* tok) {
    const int G = s->gamma, V = s->V;
    if (isnan(T) || isinf(T) || T < 0.0) return 0;
    for (int i = 0; i < G; ++i)
        if (tok[i] < 0 || tok[i] >= V) return 0;
    for (int i = 0; i <= G; ++i) {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        if (!row_usable(s->lt, V)) return 0;
    }
    if (T > 0.0) {
        for (int i = 0; i < G; ++i) {
            load_row(s->draft, s->dtype, (size_t)b * (size_t)G + (size_t)i, V, s->ld);
            if (!row_usable(s->ld, V)) return 0;
        }
    }
    return 1;
}

/* Temperature zero ("Speculative Decoding : accélérer l'inférence des LLM",
 * §Pourquoi la qualité est préservée): a draft token is accepted iff it is
 * the target argmax at its position; the first mismatch is replaced by that
 * argmax and ends the scan; if all gamma match, the argmax of the last target
 * row is the extra token. Returns n. */
static int verify_greedy(const scratch_t* s, int b, const int32_t* tok, int32_t* out) {
    const int G = s->gamma, V = s->V;
    for (int i = 0; i < G; ++i) {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        int a = row_argmax(s->lt, V);
        if (tok[i] == a) {
            out[i] = tok[i];
        } else {
            out[i] = a;
            return i;
        }
    }
    load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)G, V, s->lt);
    out[G] = row_argmax(s->lt, V);
    return G;
}

/* Temperature T > 0. Left to right, draft token x_i is accepted iff
 * u_i < alpha_i = min(1, p_i(x_i) / q_i(x_i)) (eq. alpha(x) of the wiki page
 * "Speculative Decoding"); the first rejection at position n ends the scan
 * and the later draft tokens are dropped ("Il meccanismo: draft model, target
 * model, rejection sampling"). The replacement is drawn from
 * p_corr = max(p_n - q_n, 0) / sum max(p_n - q_n, 0) (eq. p_corr); if nothing
 * was rejected, the extra token is drawn from p at the last target row
 * ("Accélérer Sonar grâce à la spéculation", §Décodage spéculatif). */
static int verify_sampled(const scratch_t* s, int b, double T, const int32_t* tok,
                          const float* ua, float us, int32_t* out,
                          const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    int n = G;
    for (int i = 0; i < G; ++i) {
        size_t r = (size_t)b * (size_t)G + (size_t)i;
        int x = tok[i];
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        double m_p, logZ_p, m_q, logZ_q;
        softmax_T2(s->lt, V, T, s->p, &m_p, &logZ_p);
        load_row(s->draft, s->dtype, r, V, s->ld);
        softmax_T2(s->ld, V, T, s->q, &m_q, &logZ_q);
        double px = s->p[x], qx = s->q[x];
        double alpha = accept_alpha(s->lt[x], m_p, logZ_p, s->ld[x], m_q, logZ_q, T);
        double u = (double)ua[i];
        set_d(d->p_x, r, px);
        set_d(d->q_x, r, qx);
        set_d(d->alpha, r, alpha);
        set_d(d->accept_margin, r, alpha > 0.0 ? fabs(u - alpha) / alpha : INFINITY);
        if (accepts(u, alpha, s->lt[x] > -INFINITY)) {
            out[i] = x;
        } else {
            n = i;
            break;
        }
    }
    double W = 0.0;
    if (n < G) {
        /* s->p and s->q still hold the distributions of position n. */
        for (int x = 0; x < V; ++x) {
            double diff = s->p[x] - s->q[x];
            s->w[x] = diff > 0.0 ? diff : 0.0;
            W += s->w[x];
        }
        if (W == 0.0) /* unreachable in exact arithmetic: fall back to p_n */
            memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        set_i(d->kind, (size_t)b, ORACLE_KIND_RESIDUAL);
    } else {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)G, V, s->lt);
        softmax_T(s->lt, V, T, s->p);
        memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        set_i(d->kind, (size_t)b, ORACLE_KIND_BONUS);
    }
    double margin = 0.0;
    out[n] = draw_inverse_cdf(s->w, V, (double)us, &W, &margin);
    set_d(d->w_total, (size_t)b, W);
    set_d(d->sample_margin, (size_t)b, margin);
    if (d->tie_measure) d->tie_measure[b] = tie_measure(s->w, V, W);
    return n;
}

int oracle_spec_verify(const void* target, const void* draft, int dtype, int B, int gamma,
                       int V, const int32_t* tokens, const float* u_accept,
                       const float* u_sample, const float* temperature,
                       int32_t* out_tokens, int32_t* out_num_accepted,
                       const oracle_detail* detail) {
    if (B < 0 || gamma < 1 || V < 1) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    if (B == 0) return 0;
    if (!target || !draft || !tokens || !u_accept || !u_sample || !temperature ||
        !out_tokens || !out_num_accepted)
        return -1;
    oracle_detail none;
    memset(&none, 0, sizeof none);
    const oracle_detail* d = detail ? detail : &none;

    scratch_t s;
    s.target = target;
    s.draft = draft;
    s.dtype = dtype;
    s.gamma = gamma;
    s.V = V;
    s.lt = (double*)malloc(sizeof(double) * (size_t)V);
    s.ld = (double*)malloc(sizeof(double) * (size_t)V);
    s.p = (double*)malloc(sizeof(double) * (size_t)V);
    s.q = (double*)malloc(sizeof(double) * (size_t)V);
    s.w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s.lt || !s.ld || !s.p || !s.q || !s.w) {
        free(s.lt), free(s.ld), free(s.p), free(s.q), free(s.w);
        return -1;
    }

    for (int b = 0; b < B; ++b) {
        const int32_t* tok = tokens + (size_t)b * (size_t)gamma;
        int32_t* out = out_tokens + (size_t)b * (size_t)(gamma + 1);
        double T = (double)temperature[b];
        for (int j = 0; j <= gamma; ++j) out[j] = -1;
        clear_detail(d, b, gamma);
        if (!request_valid(&s, b, T, tok)) {
            out_num_accepted[b] = -1;
            continue;
        }
        if (detail) report_rows(&s, b, T, d);
        if (T == 0.0) {
            set_i(d->kind, (size_t)b, ORACLE_KIND_GREEDY);
            out_num_accepted[b] = verify_greedy(&s, b, tok, out);
        } else {
            out_num_accepted[b] = verify_sampled(&s, b, T, tok,
                                                 u_accept + (size_t)b * (size_t)gamma,
                                                 u_sample[b], out, d);
        }
    }
    free(s.lt), free(s.ld), free(s.p), free(s.q), free(s.w);
    return 0;
}

/* ------------------------------------------------------------------------
 * Deterministic proposals ("Speculative Decoding : accélérer l'inférence des
 * LLM", §N-gram lookup et variantes sans modèle: the draft tokens come from a
 * lookup, not from a model). Such a proposer puts all its probability on the
 * token it proposes: q_i is one-hot at x_i. The rule of §Pourquoi la qualité
 * est préservée then reads: alpha_i = min(1, p_i(x_i) / 1) = min(1, p_i(x_i));
 * the residual max(p_n - q_n, 0) is p_n with the weight of x_n set to zero.
 * Request b proposes k = num_draft[b] tokens (0 <= k <= gamma); the extra token
 * after k acceptances comes from target row k. Target rows past k are not part
 * of the request and are never read. */

static int request_valid_onehot(const scratch_t* s, int b, double T, const int32_t* tok, int k) {
    const int G = s->gamma, V = s->V;
    if (isnan(T) || isinf(T) || T < 0.0) return 0;
    if (k < 0 || k > G) return 0;
    for (int i = 0; i < k; ++i)
        if (tok[i] < 0 || tok[i] >= V) return 0;
    for (int i = 0; i <= k; ++i) {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        if (!row_usable(s->lt, V)) return 0;
    }
    return 1;
}

static void report_rows_onehot(const scratch_t* s, int b, double T, int k, const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    for (int i = 0; i <= k; ++i) {
        size_t r = (size_t)b * (size_t)(G + 1) + (size_t)i;
        load_row(s->target, s->dtype, r, V, s->lt);
        set_d(d->max_target, r, row_max(s->lt, V));
        set_i(d->argmax_target, r, row_argmax(s->lt, V));
        if (T > 0.0) set_d(d->lse_target, r, softmax_T(s->lt, V, T, s->p));
    }
}

/* T == 0: as verify_greedy, over the k proposals; the extra token is the
 * argmax of target row k. */
static int verify_greedy_onehot(const scratch_t* s, int b, const int32_t* tok, int k, int32_t* out) {
    const int G = s->gamma, V = s->V;
    for (int i = 0; i < k; ++i) {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        int a = row_argmax(s->lt, V);
        if (tok[i] == a) {
            out[i] = tok[i];
        } else {
            out[i] = a; /* the target's argmax replaces the proposal */
            return i;
        }
    }
    load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)k, V, s->lt);
    out[k] = row_argmax(s->lt, V);
    return k;
}

/* T > 0 with q_i one-hot at x_i. */
static int verify_sampled_onehot(const scratch_t* s, int b, double T, const int32_t* tok, int k,
                                 const float* ua, float us, int32_t* out, const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    int n = k;
    for (int i = 0; i < k; ++i) {
        size_t r = (size_t)b * (size_t)G + (size_t)i;
        const int x = tok[i];
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);
        softmax_T(s->lt, V, T, s->p);
        double px = s->p[x], qx = 1.0; /* q_i(x_i) of a one-hot proposal */
        double alpha = fmin(1.0, px / qx);
        double u = (double)ua[i];
        set_d(d->p_x, r, px);
        set_d(d->q_x, r, qx);
        set_d(d->alpha, r, alpha);
        set_d(d->accept_margin, r, alpha > 0.0 ? fabs(u - alpha) / alpha : INFINITY);
        if (accepts(u, alpha, s->lt[x] > -INFINITY)) {
            out[i] = x; /* accepted */
        } else {
            n = i; /* the first rejection */
            break;
        }
    }
    double W = 0.0;
    if (n < k) {
        /* s->p holds p_n; q_n is one-hot at x_n */
        for (int x = 0; x < V; ++x) {
            double diff = s->p[x] - (x == tok[n] ? 1.0 : 0.0);
            s->w[x] = diff > 0.0 ? diff : 0.0;
            W += s->w[x];
        }
        if (W == 0.0) /* unreachable in exact arithmetic: fall back to p_n */
            memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        set_i(d->kind, (size_t)b, ORACLE_KIND_RESIDUAL);
    } else {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)k, V, s->lt);
        softmax_T(s->lt, V, T, s->p);
        memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        set_i(d->kind, (size_t)b, ORACLE_KIND_BONUS);
    }
    double margin = 0.0;
    out[n] = draw_inverse_cdf(s->w, V, (double)us, &W, &margin);
    set_d(d->w_total, (size_t)b, W);
    set_d(d->sample_margin, (size_t)b, margin);
    if (d->tie_measure) d->tie_measure[b] = tie_measure(s->w, V, W);
    return n;
}

int oracle_spec_verify_onehot(const void* target, int dtype, int B, int gamma, int V,
                              const int32_t* tokens, const int32_t* num_draft,
                              const float* u_accept, const float* u_sample,
                              const float* temperature, int32_t* out_tokens,
                              int32_t* out_num_accepted, const oracle_detail* detail) {
    if (B < 0 || gamma < 1 || V < 1) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    if (B == 0) return 0;
    if (!target || !tokens || !num_draft || !u_accept || !u_sample || !temperature || !out_tokens ||
        !out_num_accepted)
        return -1;
    oracle_detail none;
    memset(&none, 0, sizeof none);
    const oracle_detail* d = detail ? detail : &none;

    scratch_t s;
    memset(&s, 0, sizeof s);
    s.target = target;
    s.dtype = dtype;
    s.gamma = gamma;
    s.V = V;
    s.lt = (double*)malloc(sizeof(double) * (size_t)V);
    s.p = (double*)malloc(sizeof(double) * (size_t)V);
    s.w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s.lt || !s.p || !s.w) {
        free(s.lt), free(s.p), free(s.w);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t* tok = tokens + (size_t)b * (size_t)gamma;
        int32_t* out = out_tokens + (size_t)b * (size_t)(gamma + 1);
        double T = (double)temperature[b];
        int k = num_draft[b];
        for (int j = 0; j < gamma + 1; ++j) out[j] = -1;
        clear_detail(d, b, gamma);
        if (!request_valid_onehot(&s, b, T, tok, k)) {
            out_num_accepted[b] = -1;
            continue;
        }
        if (detail) report_rows_onehot(&s, b, T, k, d);
        if (T == 0.0) {
            set_i(d->kind, (size_t)b, ORACLE_KIND_GREEDY);
            out_num_accepted[b] = verify_greedy_onehot(&s, b, tok, k, out);
        } else {
            out_num_accepted[b] = verify_sampled_onehot(&s, b, T, tok, k,
                                                        u_accept + (size_t)b * (size_t)gamma,
                                                        u_sample[b], out, d);
        }
    }
    free(s.lt), free(s.p), free(s.w);
    return 0;
}

/* ------------------------------------------------------------------------
 * Early exit ("Speculative Decoding — Come Accelerare l'Inferenza LLM di 2-3x
 * Senza Perdere Qualità", §Il meccanismo: after the first rejection the later
 * draft tokens are discarded; "Speculative Decoding : accélérer l'inférence
 * des LLM", §Principe et garanties mathématiques: accept left to right while
 * compatible). The decisions are those of oracle_spec_verify (or of the
 * one-hot rule when draft is NULL); the difference is which rows are read:
 * positions are taken in order and nothing after the first rejection is read,
 * so a request is invalid only when a row it reads is bad (NaN, +inf, only
 * -inf): target rows 0..n, the draft rows 0..n of the positions evaluated (T >
 * 0, model proposals), and row n again for the draw. T, the proposal count and
 * every proposed token are checked first, as before. */

static int row_ok_at(const scratch_t* s, const void* base, size_t row, double* l) {
    load_row(base, s->dtype, row, s->V, l);
    return row_usable(l, s->V);
}

/* Returns n, or -1 for an invalid request. */
static int verify_early(const scratch_t* s, int b, double T, const int32_t* tok, int k,
                        const float* ua, float us, int32_t* out, const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    const int onehot = s->draft == NULL;
    for (int i = 0; i <= k; ++i) {
        size_t tr = (size_t)b * (size_t)(G + 1) + (size_t)i;
        if (!row_ok_at(s, s->target, tr, s->lt)) return -1;
        set_d(d->max_target, tr, row_max(s->lt, V));
        set_i(d->argmax_target, tr, row_argmax(s->lt, V));
        double m_p = 0.0, logZ_p = 0.0;
        if (T > 0.0) set_d(d->lse_target, tr, softmax_T2(s->lt, V, T, s->p, &m_p, &logZ_p));
        if (i == k) break; /* the extra-token row */
        const int x = tok[i];
        size_t r = (size_t)b * (size_t)G + (size_t)i;
        if (T == 0.0) {
            const int a = row_argmax(s->lt, V);
            if (x != a) {
                out[i] = a;
                return i;
            }
            out[i] = x;
            continue;
        }
        double qx = 1.0;
        double alpha;
        const double px = s->p[x];
        if (!onehot) {
            if (!row_ok_at(s, s->draft, r, s->ld)) return -1;
            set_d(d->max_draft, r, row_max(s->ld, V));
            double m_q, logZ_q;
            set_d(d->lse_draft, r, softmax_T2(s->ld, V, T, s->q, &m_q, &logZ_q));
            qx = s->q[x];
            alpha = accept_alpha(s->lt[x], m_p, logZ_p, s->ld[x], m_q, logZ_q, T);
        } else {
            alpha = fmin(px, 1.0);  /* q one-hot at the proposal */
        }
        const double u = (double)ua[i];
        set_d(d->p_x, r, px);
        set_d(d->q_x, r, qx);
        set_d(d->alpha, r, alpha);
        set_d(d->accept_margin, r, alpha > 0.0 ? fabs(u - alpha) / alpha : INFINITY);
        if (!accepts(u, alpha, s->lt[x] > -INFINITY)) {
            /* the residual of position i: p and q of that position are still in s->p, s->q */
            double W = 0.0;
            for (int y = 0; y < V; ++y) {
                const double qy = onehot ? (y == x ? 1.0 : 0.0) : s->q[y];
                const double diff = s->p[y] - qy;
                s->w[y] = diff > 0.0 ? diff : 0.0;
                W += s->w[y];
            }
            if (W == 0.0) /* unreachable in exact arithmetic: fall back to p_i */
                memcpy(s->w, s->p, sizeof(double) * (size_t)V);
            double margin = 0.0;
            out[i] = draw_inverse_cdf(s->w, V, (double)us, &W, &margin);
            set_i(d->kind, (size_t)b, ORACLE_KIND_RESIDUAL);
            set_d(d->w_total, (size_t)b, W);
            set_d(d->sample_margin, (size_t)b, margin);
            if (d->tie_measure) d->tie_measure[b] = tie_measure(s->w, V, W);
            return i;
        }
        out[i] = x;
    }
    /* all k accepted: the extra token from target row k (in s->lt / s->p) */
    if (T == 0.0) {
        out[k] = row_argmax(s->lt, V);
        return k;
    }
    memcpy(s->w, s->p, sizeof(double) * (size_t)V);
    double W = 0.0, margin = 0.0;
    out[k] = draw_inverse_cdf(s->w, V, (double)us, &W, &margin);
    set_i(d->kind, (size_t)b, ORACLE_KIND_BONUS);
    set_d(d->w_total, (size_t)b, W);
    set_d(d->sample_margin, (size_t)b, margin);
    if (d->tie_measure) d->tie_measure[b] = tie_measure(s->w, V, W);
    return k;
}

int oracle_spec_verify_early(const void* target, const void* draft, int dtype, int B, int gamma, int V,
                             const int32_t* tokens, const int32_t* num_draft, const float* u_accept,
                             const float* u_sample, const float* temperature, int32_t* out_tokens,
                             int32_t* out_num_accepted, const oracle_detail* detail) {
    if (B < 0 || gamma < 1 || V < 1) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    if (B == 0) return 0;
    if (!target || !tokens || !u_accept || !u_sample || !temperature || !out_tokens || !out_num_accepted)
        return -1;
    if (!draft && !num_draft) return -1;
    oracle_detail none;
    memset(&none, 0, sizeof none);
    const oracle_detail* d = detail ? detail : &none;
    scratch_t s;
    memset(&s, 0, sizeof s);
    s.target = target;
    s.draft = draft;
    s.dtype = dtype;
    s.gamma = gamma;
    s.V = V;
    s.lt = (double*)malloc(sizeof(double) * (size_t)V);
    s.ld = (double*)malloc(sizeof(double) * (size_t)V);
    s.p = (double*)malloc(sizeof(double) * (size_t)V);
    s.q = (double*)malloc(sizeof(double) * (size_t)V);
    s.w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s.lt || !s.ld || !s.p || !s.q || !s.w) {
        free(s.lt), free(s.ld), free(s.p), free(s.q), free(s.w);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t* tok = tokens + (size_t)b * (size_t)gamma;
        int32_t* out = out_tokens + (size_t)b * (size_t)(gamma + 1);
        const double T = (double)temperature[b];
        const int k = draft ? gamma : num_draft[b];
        for (int j = 0; j < gamma + 1; ++j) out[j] = -1;
        clear_detail(d, b, gamma);
        int ok = !(isnan(T) || isinf(T) || T < 0.0) && k >= 0 && k <= gamma;
        for (int i = 0; ok && i < k; ++i)
            if (tok[i] < 0 || tok[i] >= V) ok = 0;
        int n = -1;
        if (ok) {
            set_i(d->kind, (size_t)b, T == 0.0 ? ORACLE_KIND_GREEDY : ORACLE_KIND_ERROR);
            n = verify_early(&s, b, T, tok, k, u_accept + (size_t)b * (size_t)gamma, u_sample[b], out, d);
        }
        if (n < 0) {
            for (int j = 0; j < gamma + 1; ++j) out[j] = -1;
            clear_detail(d, b, gamma);
        }
        out_num_accepted[b] = n;
    }
    free(s.lt), free(s.ld), free(s.p), free(s.q), free(s.w);
    return 0;
}

/* ------------------------------------------------------------------------
 * Tree verification ("Speculative Decoding : accélérer l'inférence des LLM",
 * §Medusa : plusieurs têtes de prédiction and §EAGLE: candidate continuations
 * arranged in a tree and verified in one target pass). The pages do not state
 * the rule for several candidates; this is the plainest lossless reading, the
 * rule of §Pourquoi la qualité est préservée applied candidate after candidate
 * with deterministic (one-hot) proposals:
 *  - node 0 is the root; node j in 1..m has token x_j and parent parents[j-1]
 *    in [0, j-1]; target row j holds the logits for the token after node j;
 *  - at node u, p = softmax(row u / T); u's children are tried in index
 *    order; child c is accepted with probability min(1, p'(x_c)), p' being p
 *    without the tokens of u's children rejected so far, renormalised; an
 *    accepted child becomes u and its token is emitted;
 *  - when every child is rejected (or u is a leaf) the last token is drawn
 *    from p' by inverse CDF with u_sample;
 *  - T == 0: the first child whose token is the argmax of row u is accepted;
 *    with none, the argmax is emitted and the walk ends.
 * A chain (parents[j-1] = j-1) is oracle_spec_verify_onehot. Every row 0..m is
 * read (a bad one invalidates the request), as are the parents and tokens. */

static int verify_tree_walk(const scratch_t* s, int b, double T, const int32_t* tok, const int32_t* par, int m,
                            const float* ua, float us, int32_t* out, int32_t* nodes, const oracle_detail* d) {
    const int G = s->gamma, V = s->V;
    int u = 0, n = 0;
    int excl[64];
    for (;;) {
        load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)u, V, s->lt);
        int ne = 0;
        if (T == 0.0) {
            const int a = row_argmax(s->lt, V);
            int next = -1;
            for (int c = 1; c <= m && next < 0; ++c)
                if (par[c - 1] == u && tok[c - 1] == a) next = c;
            if (next < 0) {
                out[n] = a;
                return n;
            }
            out[n] = a;
            nodes[n] = next;
            ++n;
            u = next;
            continue;
        }
        softmax_T(s->lt, V, T, s->p);
        double R = 0.0; /* probability of the children rejected so far */
        int next = -1;
        for (int c = 1; c <= m && next < 0; ++c) {
            if (par[c - 1] != u) continue;
            const int x = tok[c - 1];
            int seen = 0;
            for (int e = 0; e < ne; ++e)
                if (excl[e] == x) seen = 1;
            const double px = seen ? 0.0 : s->p[x];
            const double rest = 1.0 - R;
            const double alpha = rest > 0.0 ? fmin(1.0, px / rest) : 0.0;
            const double uc = (double)ua[c - 1];
            set_d(d->p_x, (size_t)b * (size_t)G + (size_t)(c - 1), px);
            set_d(d->q_x, (size_t)b * (size_t)G + (size_t)(c - 1), 1.0);
            set_d(d->alpha, (size_t)b * (size_t)G + (size_t)(c - 1), alpha);
            set_d(d->accept_margin, (size_t)b * (size_t)G + (size_t)(c - 1),
                  alpha > 0.0 ? fabs(uc - alpha) / alpha : INFINITY);
            if (accepts(uc, alpha, !seen && s->lt[x] > -INFINITY && rest > 0.0)) {
                next = c;
            } else if (!seen) {
                excl[ne++] = x;
                R += px;
            }
        }
        if (next >= 0) {
            out[n] = tok[next - 1];
            nodes[n] = next;
            ++n;
            u = next;
            continue;
        }
        /* the last token: p without the rejected children's tokens */
        double W = 0.0;
        for (int y = 0; y < V; ++y) {
            int ex = 0;
            for (int e = 0; e < ne; ++e)
                if (excl[e] == y) ex = 1;
            s->w[y] = ex ? 0.0 : s->p[y];
            W += s->w[y];
        }
        if (W == 0.0) /* unreachable in exact arithmetic: fall back to p */
            memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        double margin = 0.0;
        out[n] = draw_inverse_cdf(s->w, V, (double)us, &W, &margin);
        set_i(d->kind, (size_t)b, ne > 0 ? ORACLE_KIND_RESIDUAL : ORACLE_KIND_BONUS);
        set_d(d->w_total, (size_t)b, W);
        set_d(d->sample_margin, (size_t)b, margin);
        if (d->tie_measure) d->tie_measure[b] = tie_measure(s->w, V, W);
        return n;
    }
}

int oracle_spec_verify_tree(const void* target, int dtype, int B, int gamma, int V, const int32_t* tokens,
                            const int32_t* parents, const int32_t* num_nodes, const float* u_accept,
                            const float* u_sample, const float* temperature, int32_t* out_tokens,
                            int32_t* out_num_accepted, int32_t* out_nodes, const oracle_detail* detail) {
    if (B < 0 || gamma < 1 || gamma > 64 || V < 1) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    if (B == 0) return 0;
    if (!target || !tokens || !parents || !num_nodes || !u_accept || !u_sample || !temperature || !out_tokens ||
        !out_num_accepted || !out_nodes)
        return -1;
    oracle_detail none;
    memset(&none, 0, sizeof none);
    const oracle_detail* d = detail ? detail : &none;
    scratch_t s;
    memset(&s, 0, sizeof s);
    s.target = target;
    s.dtype = dtype;
    s.gamma = gamma;
    s.V = V;
    s.lt = (double*)malloc(sizeof(double) * (size_t)V);
    s.p = (double*)malloc(sizeof(double) * (size_t)V);
    s.w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s.lt || !s.p || !s.w) {
        free(s.lt), free(s.p), free(s.w);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t* tok = tokens + (size_t)b * (size_t)gamma;
        const int32_t* par = parents + (size_t)b * (size_t)gamma;
        int32_t* out = out_tokens + (size_t)b * (size_t)(gamma + 1);
        int32_t* nodes = out_nodes + (size_t)b * (size_t)gamma;
        const double T = (double)temperature[b];
        const int m = num_nodes[b];
        for (int j = 0; j < gamma + 1; ++j) out[j] = -1;
        for (int j = 0; j < gamma; ++j) nodes[j] = -1;
        clear_detail(d, b, gamma);
        int ok = !(isnan(T) || isinf(T) || T < 0.0) && m >= 0 && m <= gamma;
        for (int j = 1; ok && j <= m; ++j)
            if (par[j - 1] < 0 || par[j - 1] >= j || tok[j - 1] < 0 || tok[j - 1] >= V) ok = 0;
        for (int j = 0; ok && j <= m; ++j) {
            load_row(s.target, s.dtype, (size_t)b * (size_t)(gamma + 1) + (size_t)j, V, s.lt);
            if (!row_usable(s.lt, V)) ok = 0;
        }
        if (!ok) {
            out_num_accepted[b] = -1;
            continue;
        }
        if (detail) report_rows_onehot(&s, b, T, m, d);
        if (T == 0.0) set_i(d->kind, (size_t)b, ORACLE_KIND_GREEDY);
        out_num_accepted[b] = verify_tree_walk(&s, b, T, tok, par, m, u_accept + (size_t)b * (size_t)gamma,
                                               u_sample[b], out, nodes, d);
    }
    free(s.lt), free(s.p), free(s.w);
    return 0;
}

