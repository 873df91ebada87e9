/*
 * sc_oracle.c -- FP64 CPU oracle for score centering.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the
 * CUDA path: only the tests, the smoke check and the benchmark's CPU
 * baseline may load it.  It shares no code, header, table or constant with
 * the GPU library and must never be called by the product path.
 *
 * What it computes follows the "Score Centering" section of the Agent
 * Lightning docs page "Score Centering" (example 85):
 *
 *   P_H = sum_{v in H} p_v,   Q_H = sum_{v in H} q_v,
 *   rho = max(1 - Q_H, 1e-6) / max(1 - P_H, 1e-6),
 *   token loss = -sg(A) * [ log p_a - sum_{v in H} sg(q_v - rho p_v) log p_v ],
 *
 * where p is the trainer's softmax over the full vocabulary at the rollout
 * temperature, H the recorded candidate ids with recorded probabilities q,
 * a the sampled token and A the rollout-level advantage.  The same section
 * defines the K3 diagnostic (d = train logprob - rollout logprob,
 * k3 = exp(d) - 1 - d) and the settings table (is_mode none/tis/mis,
 * tis_max, mis_min, mis_max, centering).  The truncated importance weight
 * min(w, w_max) is the one of "Lecture 12 -- RL systems for agents", section 1
 * ("Two engines compute two probabilities").  Group-std advantages follow the
 * "Training" section of the same docs page (rollout-level advantages with
 * group standard deviation normalisation) and section 4 of the devotd.net
 * release note (mean-only variant; rewards kept fractional).
 *
 * Everything is computed in double precision, row by row, with plain
 * sequential sums in the order of the definitions.  The gradient is the
 * derivative of the token loss with respect to the raw logits z (x = z / T):
 *
 *   dloss/dz_v = (1/T) * (-A) * ( [v == a] - s p_v - [v in H] c_v ),
 *   c_v = q_v - rho p_v,   s = 1 - Q_H + rho P_H,
 *
 * obtained from d log p_u / d x_v = [u == v] - p_v with c held constant
 * (stop-gradient).  Every gradient row therefore sums to zero.
 *
 * Readings where the pages are silent:
 *   - std is the unbiased (n - 1) sample std; eps is added to it; a group
 *     whose rewards are all equal has A = 0; a group of one has A = 0.
 *   - a recorded id outside [0, V) is ignored and flagged; a repeated id is
 *     ignored after its first occurrence and flagged.
 *   - a sampled id outside [0, V), or a row whose response index is outside
 *     [0, n_resp), is an error row: zero gradient, flag set.
 *   - is_mode tis weights the token by min(w, tis_max); is_mode mis weights
 *     it by w inside [mis_min, mis_max] and by 0 outside; w = exp(d).
 *   - centering = 0 drops the centering term (c = 0, s = 1).
 *   - is_mode 3 is the clipped GRPO baseline of the page's "Training" section
 *     (the `grpo` preset: clipped objective, lower/upper clip widths 0.2/0.3,
 *     per-rollout mean loss): with the ratio w = exp(d) and its clipped copy
 *     w_c = clamp(w, 1 - clip_low, 1 + clip_high), the token loss is
 *     -min(w A, w_c A).  Its gradient is that of -A w, i.e. the policy
 *     gradient weighted by w, wherever the unclipped term is the minimum, and
 *     zero where the clipped one is (flag CLIPPED).  It has no centering term:
 *     the mode is defined with centering = 0 only.  The per-rollout mean is
 *     sco_rollout_mean_advantages below: each response's advantage divided
 *     by its number of valid tokens (0 for a response without any).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Per-row flag bits (same meaning as the library's, defined independently). */
#define SCO_FLAG_MASKED 0x1u        /* padding row (row_response < 0)        */
#define SCO_FLAG_BAD_ID 0x2u        /* a recorded id outside [0, V)           */
#define SCO_FLAG_DUP_ID 0x4u        /* a repeated recorded id                 */
#define SCO_FLAG_BAD_SAMPLED 0x8u   /* sampled id outside [0, V)              */
#define SCO_FLAG_BAD_COUNT 0x10u    /* count outside [0, K_max], clamped      */
#define SCO_FLAG_BAD_RESPONSE 0x20u /* response index >= n_resp               */
#define SCO_FLAG_CLAMP_PI 0x40u     /* 1 - P_H < 1e-6: denominator clamped    */
#define SCO_FLAG_CLAMP_MU 0x80u     /* 1 - Q_H < 1e-6: numerator clamped      */
#define SCO_FLAG_IS_TRUNC 0x100u    /* tis: weight truncated at tis_max       */
#define SCO_FLAG_IS_REJECT 0x200u   /* mis: weight outside the interval -> 0  */
#define SCO_FLAG_CLIPPED 0x400u     /* clipped GRPO: the clipped term is the minimum */

typedef struct {
    int is_mode; /* 0 none, 1 tis, 2 mis, 3 clipped GRPO */
    double tis_max, mis_min, mis_max;
    int centering; /* 1: score centering on, 0: plain importance-weighted PG */
    double inv_temperature;
    double grad_scale;
    double clip_low, clip_high; /* clipped GRPO: ratio kept in [1 - low, 1 + high] */
} sco_params;

typedef struct {
    double loss;      /* token loss of the formula above (unscaled)        */
    double logp_a;    /* log p_a at the rollout temperature                */
    double P_H;       /* sum of p over the recorded ids                    */
    double tail_pi;   /* 1 - P_H                                           */
    double Q_H;       /* sum of the recorded probabilities                 */
    double tail_mu;   /* 1 - Q_H                                           */
    double rho;       /* tail ratio with the 1e-6 clamps                   */
    double s;         /* 1 - Q_H + rho P_H                                 */
    double entropy;   /* -sum p log p                                      */
    double k3;        /* exp(d) - 1 - d, d = log p_a - rollout logprob     */
    double is_weight; /* importance weight applied to A (1 for none)       */
    double row_sum;   /* sum of the gradient row                           */
    double adv;       /* the row's advantage A                             */
    int n_valid_k;    /* recorded ids used after the range/duplicate rules */
    unsigned flags;
} sco_row_out;

/* ---- bf16 <-> double ------------------------------------------------- */

/* A bf16 value is the top 16 bits of an IEEE binary32 ("Lecture 12", section 4). */
double sco_bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, directly from the
 * double (no intermediate rounding to binary32).  NaN maps to a quiet NaN,
 * overflow past the largest finite bf16 maps to infinity. */
uint16_t sco_double_to_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    /* Normal bf16 numbers: 1.f * 2^(e-1) with 7 fraction bits, exponent
     * e - 1 >= -126.  Below that, subnormals with spacing 2^-133. */
    int exp_unbiased = e - 1;
    double spacing_exp;
    if (exp_unbiased >= -126)
        spacing_exp = exp_unbiased - 7;
    else
        spacing_exp = -126 - 7;
    double scaled = ldexp(a, -(int)spacing_exp); /* integer grid units */
    double r = nearbyint(scaled); /* default rounding mode: ties to even */
    (void)m;
    double y = ldexp(r, (int)spacing_exp);
    if (y > 3.3895313892515355e38) return (uint16_t)(sign | 0x7F80u);
    float yf = (float)y; /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &yf, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* ---- group advantages ------------------------------------------------ */

/* A_i = (r_i - mean_g) / (std_g + eps) per group of group_size responses,
 * or A_i = r_i - mean_g when normalize_std is 0.  Returns 0, or -1 on bad
 * arguments. */
int sco_group_advantages(const float* rewards, int n_groups, int group_size, int normalize_std,
                         double eps, double* adv) {
    if (n_groups < 0 || group_size < 1) return -1;
    if (n_groups > 0 && (!rewards || !adv)) return -1;
    for (int g = 0; g < n_groups; ++g) {
        const float* r = rewards + (size_t)g * group_size;
        double* out = adv + (size_t)g * group_size;
        int all_equal = 1;
        for (int i = 1; i < group_size; ++i)
            if (r[i] != r[0]) all_equal = 0;
        if (all_equal) {
            for (int i = 0; i < group_size; ++i) out[i] = 0.0;
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i < group_size; ++i) sum += (double)r[i];
        double mean = sum / group_size;
        double ss = 0.0;
        for (int i = 0; i < group_size; ++i) {
            double d = (double)r[i] - mean;
            ss += d * d;
        }
        double std = sqrt(ss / (group_size - 1));
        for (int i = 0; i < group_size; ++i) {
            double d = (double)r[i] - mean;
            out[i] = normalize_std ? d / (std + eps) : d;
        }
    }
    return 0;
}

/* Per-rollout mean: each response's advantage divided by its number of
 * valid tokens (rows whose response index is r), 0 for a response with none;
 * the counts are returned too.  Returns 0, or -1 on bad arguments. */
int sco_rollout_mean_advantages(const double* adv, const int32_t* row_response, long long T, int n_resp,
                                long long* counts, double* adv_out) {
    if (T < 0 || n_resp < 0) return -1;
    if (n_resp > 0 && (!adv || !counts || !adv_out)) return -1;
    if (T > 0 && !row_response) return -1;
    for (int r = 0; r < n_resp; ++r) counts[r] = 0;
    for (long long t = 0; t < T; ++t)
        if (row_response[t] >= 0 && row_response[t] < n_resp) ++counts[row_response[t]];
    for (int r = 0; r < n_resp; ++r) adv_out[r] = counts[r] > 0 ? adv[r] / (double)counts[r] : 0.0;
    return 0;
}

/* ---- one token row --------------------------------------------------- */

/* Score-centered forward/backward for one unmasked row.
 *   z        : V bf16 logits (raw bits)
 *   ids, lp  : `count` recorded ids and their recorded log-probabilities
 *   a        : sampled id;  rollout_lp : its rollout logprob (has_rollout)
 *   A        : the row's advantage
 *   grad     : V doubles out (d loss / d z, times grad_scale)
 *   work     : V ints of scratch (membership of H)
 * Returns the row flags. */
static unsigned sco_row_impl(const uint16_t* z, int V, const int32_t* ids, const float* lp,
                             int count, int a, double rollout_lp, int has_rollout, double A,
                             const sco_params* p, double* grad, int* in_h, double* logp,
                             sco_row_out* out) {
    unsigned flags = 0;
    memset(out, 0, sizeof *out);
    out->adv = A;
    if (a < 0 || a >= V) {
        for (int v = 0; v < V; ++v) grad[v] = 0.0;
        out->flags = SCO_FLAG_BAD_SAMPLED;
        return out->flags;
    }
    double invT = p->inv_temperature;

    /* Full-vocabulary log-softmax at the rollout temperature. */
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double x = sco_bf16_to_double(z[v]) * invT;
        if (x > m) m = x;
    }
    double l = 0.0;
    for (int v = 0; v < V; ++v) l += exp(sco_bf16_to_double(z[v]) * invT - m);
    double lse = m + log(l);
    for (int v = 0; v < V; ++v) logp[v] = sco_bf16_to_double(z[v]) * invT - lse;

    /* Recorded head H: range and duplicate rules. */
    for (int v = 0; v < V; ++v) in_h[v] = -1;
    int nk = 0;
    for (int k = 0; k < count; ++k) {
        int id = ids[k];
        if (id < 0 || id >= V) {
            flags |= SCO_FLAG_BAD_ID;
            continue;
        }
        if (in_h[id] >= 0) {
            flags |= SCO_FLAG_DUP_ID;
            continue;
        }
        in_h[id] = k;
        ++nk;
    }

    double P_H = 0.0, Q_H = 0.0;
    for (int v = 0; v < V; ++v)
        if (in_h[v] >= 0) {
            P_H += exp(logp[v]);
            Q_H += exp((double)lp[in_h[v]]);
        }
    double tail_pi = 1.0 - P_H;
    double tail_mu = 1.0 - Q_H;
    double rho = fmax(tail_mu, 1e-6) / fmax(tail_pi, 1e-6);
    if (tail_pi < 1e-6) flags |= SCO_FLAG_CLAMP_PI;
    if (tail_mu < 1e-6) flags |= SCO_FLAG_CLAMP_MU;
    double s = 1.0 - Q_H + rho * P_H;
    if (!p->centering) s = 1.0;

    /* Importance weight at the sampled token. */
    double d = has_rollout ? logp[a] - rollout_lp : 0.0;
    double w = exp(d);
    double wt = 1.0;
    if (p->is_mode == 1) {
        wt = w < p->tis_max ? w : p->tis_max;
        if (w > p->tis_max) flags |= SCO_FLAG_IS_TRUNC;
    } else if (p->is_mode == 3) {
        /* -min(w A, w_c A): the gradient is -A w where the unclipped term is
         * the minimum (equal terms included), 0 where the clipped one is */
        double wc = w < 1.0 - p->clip_low ? 1.0 - p->clip_low : (w > 1.0 + p->clip_high ? 1.0 + p->clip_high : w);
        if (wc == w || w * A < wc * A) {
            wt = w;
        } else {
            wt = 0.0;
            flags |= SCO_FLAG_CLIPPED;
        }
    } else if (p->is_mode == 2) {
        if (w >= p->mis_min && w <= p->mis_max)
            wt = w;
        else {
            wt = 0.0;
            flags |= SCO_FLAG_IS_REJECT;
        }
    }
    double A_eff = A * wt;

    /* Loss:  -A [ log p_a - sum_H c_v log p_v ]. */
    double centered = 0.0;
    if (p->centering)
        for (int v = 0; v < V; ++v)
            if (in_h[v] >= 0) {
                double c = exp((double)lp[in_h[v]]) - rho * exp(logp[v]);
                centered += c * logp[v];
            }
    double loss = -A_eff * (logp[a] - centered);
    if (p->is_mode == 3) {
        double wc = w < 1.0 - p->clip_low ? 1.0 - p->clip_low : (w > 1.0 + p->clip_high ? 1.0 + p->clip_high : w);
        loss = -fmin(w * A, wc * A);
    }

    /* Gradient: g_v = scale * (1/T) * (-A) * ([v==a] - s p_v - [v in H] c_v). */
    double coef = p->grad_scale * invT * (-A_eff);
    double row_sum = 0.0;
    for (int v = 0; v < V; ++v) {
        double pv = exp(logp[v]);
        double mu_hat = s * pv;
        if (p->centering && in_h[v] >= 0) mu_hat += exp((double)lp[in_h[v]]) - rho * pv;
        double g = coef * ((v == a ? 1.0 : 0.0) - mu_hat);
        grad[v] = g;
        row_sum += g;
    }

    double ent = 0.0;
    for (int v = 0; v < V; ++v) {
        double pv = exp(logp[v]);
        if (pv > 0.0) ent -= pv * logp[v];
    }

    out->loss = loss;
    out->logp_a = logp[a];
    out->P_H = P_H;
    out->tail_pi = tail_pi;
    out->Q_H = Q_H;
    out->tail_mu = tail_mu;
    out->rho = rho;
    out->s = s;
    out->entropy = ent;
    out->k3 = has_rollout ? exp(d) - 1.0 - d : 0.0;
    out->is_weight = wt;
    out->row_sum = row_sum;
    out->n_valid_k = nk;
    out->flags = flags;
    return flags;
}

/* One row, allocating its own scratch.  Returns flags, or ~0u on bad args. */
unsigned sco_row(const uint16_t* z, int V, const int32_t* ids, const float* lp, int count, int a,
                 double rollout_lp, int has_rollout, double A, const sco_params* p, double* grad,
                 sco_row_out* out) {
    if (!z || V <= 0 || !p || !grad || !out || count < 0 || (count > 0 && (!ids || !lp)))
        return ~0u;
    if (p->is_mode == 3 && p->centering) return ~0u; /* the clipped objective has no centering */
    int* in_h = (int*)malloc(sizeof(int) * (size_t)V);
    double* logp = (double*)malloc(sizeof(double) * (size_t)V);
    if (!in_h || !logp) {
        free(in_h);
        free(logp);
        return ~0u;
    }
    unsigned f =
        sco_row_impl(z, V, ids, lp, count, a, rollout_lp, has_rollout, A, p, grad, in_h, logp, out);
    free(in_h);
    free(logp);
    return f;
}

/* ---- a batch of rows, threaded over rows ----------------------------- */

typedef struct {
    /* batch description, laid out like the library's call */
    const uint16_t* logits;
    long long T;
    int V;
    long long row_stride;
    const int32_t* rec_ids;
    const float* rec_logprobs;
    const int32_t* rec_count; /* may be NULL: every row has K_max */
    int K_max;
    const int32_t* sampled;
    const float* rollout_lp; /* may be NULL */
    const int32_t* row_response;
    const float* adv;
    int n_resp;
    const sco_params* p;
    /* which rows, and where their results go */
    const long long* rows;
    long long n_rows;
    double* grad;   /* [n_rows, V] */
    double* logp_a; /* [n_rows]    */
    sco_row_out* out; /* [n_rows]  */
    long long next;   /* shared work index */
    pthread_mutex_t lock;
} sco_batch;

static void sco_batch_row(sco_batch* b, long long i, int* in_h, double* logp) {
    long long t = b->rows[i];
    double* g = b->grad + (size_t)i * (size_t)b->V;
    sco_row_out* o = b->out + i;
    int resp = b->row_response[t];
    if (resp < 0 || resp >= b->n_resp) {
        for (int v = 0; v < b->V; ++v) g[v] = 0.0;
        memset(o, 0, sizeof *o);
        o->flags = resp < 0 ? SCO_FLAG_MASKED : SCO_FLAG_BAD_RESPONSE;
        b->logp_a[i] = 0.0;
        return;
    }
    int count = b->rec_count ? b->rec_count[t] : b->K_max;
    unsigned extra = 0;
    if (count < 0 || count > b->K_max) {
        extra = SCO_FLAG_BAD_COUNT;
        count = count < 0 ? 0 : b->K_max;
    }
    const uint16_t* z = b->logits + (size_t)t * (size_t)b->row_stride;
    sco_row_impl(z, b->V, b->rec_ids + (size_t)t * b->K_max, b->rec_logprobs + (size_t)t * b->K_max,
                 count, b->sampled[t], b->rollout_lp ? (double)b->rollout_lp[t] : 0.0,
                 b->rollout_lp != NULL, (double)b->adv[resp], b->p, g, in_h, logp, o);
    o->flags |= extra;
    b->logp_a[i] = o->logp_a;
}

static void* sco_batch_worker(void* arg) {
    sco_batch* b = (sco_batch*)arg;
    int* in_h = (int*)malloc(sizeof(int) * (size_t)b->V);
    double* logp = (double*)malloc(sizeof(double) * (size_t)b->V);
    if (!in_h || !logp) {
        free(in_h);
        free(logp);
        return (void*)1;
    }
    for (;;) {
        pthread_mutex_lock(&b->lock);
        long long i = b->next++;
        pthread_mutex_unlock(&b->lock);
        if (i >= b->n_rows) break;
        sco_batch_row(b, i, in_h, logp);
    }
    free(in_h);
    free(logp);
    return NULL;
}

/* Rows `rows[0..n_rows)` of a batch.  nthreads <= 0 uses every online core.
 * Returns the number of threads used, or -1 on bad arguments / failure. */
int sco_rows(const uint16_t* logits, long long T, int V, long long row_stride, const int32_t* rec_ids,
             const float* rec_logprobs, const int32_t* rec_count, int K_max, const int32_t* sampled,
             const float* rollout_lp, const int32_t* row_response, const float* adv, int n_resp,
             const sco_params* p, const long long* rows, long long n_rows, double* grad,
             double* logp_a, sco_row_out* out, int nthreads) {
    if (V <= 0 || T < 0 || row_stride < V || K_max < 0 || !p || n_rows < 0) return -1;
    if (p->is_mode == 3 && p->centering) return -1;
    if (n_rows == 0) return 0;
    if (!logits || !sampled || !row_response || !adv || !rows || !grad || !logp_a || !out) return -1;
    if (K_max > 0 && (!rec_ids || !rec_logprobs)) return -1;
    for (long long i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= T) return -1;
    sco_batch b;
    memset(&b, 0, sizeof b);
    b.logits = logits;
    b.T = T;
    b.V = V;
    b.row_stride = row_stride;
    b.rec_ids = rec_ids;
    b.rec_logprobs = rec_logprobs;
    b.rec_count = rec_count;
    b.K_max = K_max;
    b.sampled = sampled;
    b.rollout_lp = rollout_lp;
    b.row_response = row_response;
    b.adv = adv;
    b.n_resp = n_resp;
    b.p = p;
    b.rows = rows;
    b.n_rows = n_rows;
    b.grad = grad;
    b.logp_a = logp_a;
    b.out = out;
    b.next = 0;
    pthread_mutex_init(&b.lock, NULL);
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if ((long long)nthreads > n_rows) nthreads = (int)n_rows;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -1;
    int started = 0, failed = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, sco_batch_worker, &b) != 0) break;
        ++started;
    }
    if (started == 0) failed = 1;
    for (int i = 0; i < started; ++i) {
        void* r = NULL;
        pthread_join(th[i], &r);
        if (r) failed = 1;
    }
    free(th);
    pthread_mutex_destroy(&b.lock);
    return failed ? -1 : started;
}

/* Every entry of x rounded to bf16 (ties to even), as bit patterns. */
void sco_round_bf16_n(const double* x, long long n, uint16_t* out) {
    for (long long i = 0; i < n; ++i) out[i] = sco_double_to_bf16_rne(x[i]);
}

int sco_row_out_size(void) { return (int)sizeof(sco_row_out); }
int sco_params_size(void) { return (int)sizeof(sco_params); }

/* ---- sampler-side top-K capture ---------------------------------------- */

/* What the sampler records per generated position (docs page "Score
 * Centering", section "Score Centering": the top K behaviour probabilities
 * of the sampling call, with their original normalisation).  The behaviour
 * distribution is mu = softmax(z * inv_t) over the V sampler logits z, or,
 * with top_p < 1, that distribution restricted to its nucleus -- the
 * smallest prefix of the entries sorted by probability whose preceding mass
 * is below top_p -- and renormalised.  Entries are sorted by z, larger
 * first, equal values by lower id.  Row t gets count = min(K, V, nucleus
 * size) ids and log mu values; the entries past the count hold id -1 and 0.
 * Plain definition: a full sort of the row, FP64 sums in sorted order. */
typedef struct {
    float z;
    int id;
} sco_entry;

static int sco_entry_cmp(const void* pa, const void* pb) {
    const sco_entry* a = (const sco_entry*)pa;
    const sco_entry* b = (const sco_entry*)pb;
    if (a->z > b->z) return -1;
    if (a->z < b->z) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

int sco_topk_capture(const float* logits, long long T, int V, long long row_stride, double inv_t, int K,
                     double top_p, int32_t* ids_out, float* lp_out, int32_t* count_out) {
    if (T < 0 || V <= 0 || row_stride < V || K < 0 || !(inv_t > 0.0) || !(top_p > 0.0 && top_p <= 1.0))
        return -1;
    if (T == 0 || K == 0) return 0;
    if (!logits || !ids_out || !lp_out) return -1;
    sco_entry* e = (sco_entry*)malloc(sizeof(sco_entry) * (size_t)V);
    if (!e) return -1;
    for (long long t = 0; t < T; ++t) {
        const float* z = logits + t * row_stride;
        for (int v = 0; v < V; ++v) {
            e[v].z = z[v];
            e[v].id = v;
        }
        qsort(e, (size_t)V, sizeof(sco_entry), sco_entry_cmp);
        /* log-sum-exp of the tempered logits, in sorted order */
        double m = (double)e[0].z * inv_t, l = 0.0;
        for (int i = 0; i < V; ++i) l += exp((double)e[i].z * inv_t - m);
        double lse = m + log(l);
        long long n_keep = V;
        double lognuc = 0.0;
        if (top_p < 1.0) {
            double cum = 0.0;
            long long i = 0;
            while (i < V && cum < top_p) {
                cum += exp((double)e[i].z * inv_t - lse);
                ++i;
            }
            n_keep = i;
            lognuc = log(cum);
        }
        int cnt = (int)(n_keep < K ? n_keep : K);
        for (int k = 0; k < K; ++k) {
            ids_out[t * K + k] = k < cnt ? e[k].id : -1;
            lp_out[t * K + k] = k < cnt ? (float)((double)e[k].z * inv_t - lse - lognuc) : 0.0f;
        }
        if (count_out) count_out[t] = cnt;
    }
    free(e);
    return 0;
}
