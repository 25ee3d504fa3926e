/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Two independent formulations, both in double precision, both written for a
 * reader to check by eye:
 *
 *  (1) kda_oracle_unit_recurrent -- the token recurrence that defines the method
 *      (gated delta rule with per-dimension decay):
 *          S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *          o_t = scale * S_t^T q_t
 *      The pages' formula sections lost their images; this is the recurrence
 *      whose chunked evaluation is printed as `naive_chunk_kda` on the page
 *      "手撕KDA" (yuyanqi.com), section "1 Naive".
 *
 *  (2) kda_oracle_unit_chunked -- the chunked (WY / UT) evaluation in the order
 *      of that same listing ("手撕KDA", section "1 Naive"): within-chunk cumsum
 *      of g, the strictly lower-triangular matrix M (beta scales ROWS), the
 *      inverse T = (I + M)^{-1} by forward substitution, A = T Diag(beta)
 *      (beta scales COLUMNS), W = A (exp(gc) * k), U = A v, then the serial
 *      chunk loop v_new = U - W S, o = (q exp(gc)) S + Aqk v_new,
 *      S <- Diag(exp(g_last)) S + (exp(g_last - gc) * k)^T v_new.
 *      Natural exp throughout: the page's C++ port ("手撕KDA", section 1.1)
 *      uses exp2 where the Python listing uses exp, and the Python listing is
 *      the one the recurrence (1) agrees with.  Exponent differences are
 *      formed before exponentiation (exp(gc_i - gc_j)), never as a product of
 *      exp(gc_i) and exp(-gc_j), so the oracle has no overflow regime of its
 *      own.  A partial last chunk simply has fewer rows.
 *
 *  (3) kda_oracle_prestage -- the activations of the gated forward (q/k L2
 *      normalisation, the bounded or softplus gate, the beta sigmoid), applied
 *      to raw projections before (1) or (2).
 *
 * Readings where the pages are silent (also listed in the design notes):
 *  - q and k of value head hv come from key head hv / (HV / H)
 *    (repeat_interleave in the listing).
 *  - no L2 normalisation, gate activation or beta sigmoid here: g is the
 *    log-space decay and beta is used as given.
 *  - an empty sequence leaves the state unchanged and produces no rows.
 *
 * Layouts (row-major, contiguous), token index tok = b*T + t (or packed):
 *   q, k  [tokens, H,  K]      v [tokens, HV, V]
 *   g     [tokens, HV, K]      beta [tokens, HV]
 * A "unit" is one (sequence, value head) pair; units are independent.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Token recurrence (definition).                                           */
/* ------------------------------------------------------------------------ */

/*
 * One unit, token by token.  Row t of q is at q + t*q_rs (K contiguous), etc.
 * s (K*V, row-major [K][V]) holds the initial state on entry and the final
 * state on exit.  o receives len rows of V values at stride o_rs.
 */
void kda_oracle_unit_recurrent(int len, int K, int V,
                               const float* q, long q_rs,
                               const float* k, long k_rs,
                               const float* v, long v_rs,
                               const float* g, long g_rs,
                               const float* beta, long beta_rs,
                               double scale, double* s,
                               double* o, long o_rs)
{
    double* u = (double*)malloc(sizeof(double) * (size_t)V);
    for (int t = 0; t < len; ++t) {
        const float* qt = q + (long)t * q_rs;
        const float* kt = k + (long)t * k_rs;
        const float* vt = v + (long)t * v_rs;
        const float* gt = g + (long)t * g_rs;
        const double bt = (double)beta[(long)t * beta_rs];

        /* P = Diag(exp g_t) S_{t-1} */
        for (int d = 0; d < K; ++d) {
            const double e = exp((double)gt[d]);
            for (int j = 0; j < V; ++j) s[(long)d * V + j] *= e;
        }
        /* u = P^T k_t */
        for (int j = 0; j < V; ++j) u[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double kd = (double)kt[d];
            for (int j = 0; j < V; ++j) u[j] += kd * s[(long)d * V + j];
        }
        /* S_t = P - beta k (k^T P) + beta k v^T = P + beta k (v - u)^T */
        for (int d = 0; d < K; ++d) {
            const double bk = bt * (double)kt[d];
            for (int j = 0; j < V; ++j) s[(long)d * V + j] += bk * ((double)vt[j] - u[j]);
        }
        /* o_t = scale S_t^T q_t */
        double* ot = o + (long)t * o_rs;
        for (int j = 0; j < V; ++j) ot[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double qd = scale * (double)qt[d];
            for (int j = 0; j < V; ++j) ot[j] += qd * s[(long)d * V + j];
        }
    }
    free(u);
}

/* ------------------------------------------------------------------------ */
/* Chunked form.                                                            */
/* ------------------------------------------------------------------------ */

/*
 * T = (I + M)^{-1} for a strictly lower-triangular n x n matrix M (row-major),
 * by forward substitution on (I + M) T = I, one row at a time:
 *     T[i][j] = delta_ij - sum_{j <= m < i} M[i][m] T[m][j].
 * T is unit lower-triangular.  ("手撕KDA", section "1 Naive": the in-place row
 * loop over the negated matrix computes the same unit lower-triangular inverse.)
 */
void kda_oracle_tri_inverse(int n, const double* M, double* Tm)
{
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < n; ++j) {
            double acc = (i == j) ? 1.0 : 0.0;
            if (j < i) {
                for (int m = j; m < i; ++m) acc -= M[(long)i * n + m] * Tm[(long)m * n + j];
            }
            Tm[(long)i * n + j] = (j <= i) ? acc : 0.0;
        }
    }
}

/*
 * One unit, chunk by chunk, with chunk size C (any C >= 1; the last chunk may
 * be shorter).  Same argument conventions as kda_oracle_unit_recurrent.
 */
void kda_oracle_unit_chunked(int len, int K, int V, int C,
                             const float* q, long q_rs,
                             const float* k, long k_rs,
                             const float* v, long v_rs,
                             const float* g, long g_rs,
                             const float* beta, long beta_rs,
                             double scale, double* s,
                             double* o, long o_rs)
{
    double* gc   = (double*)malloc(sizeof(double) * (size_t)C * K);  /* [C][K] */
    double* M    = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* Tm   = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* A    = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* Aqk  = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* W    = (double*)malloc(sizeof(double) * (size_t)C * K);
    double* U    = (double*)malloc(sizeof(double) * (size_t)C * V);
    double* vnew = (double*)malloc(sizeof(double) * (size_t)C * V);
    double* bt   = (double*)malloc(sizeof(double) * (size_t)C);

    for (int t0 = 0; t0 < len; t0 += C) {
        const int n = (len - t0 < C) ? (len - t0) : C;
#define Q(i, d) ((double)q[(long)(t0 + (i)) * q_rs + (d)])
#define KK(i, d) ((double)k[(long)(t0 + (i)) * k_rs + (d)])
#define VV(i, j) ((double)v[(long)(t0 + (i)) * v_rs + (j)])
#define G(i, d) ((double)g[(long)(t0 + (i)) * g_rs + (d)])
        for (int i = 0; i < n; ++i) bt[i] = (double)beta[(long)(t0 + i) * beta_rs];

        /* a2: within-chunk inclusive cumsum of g */
        for (int d = 0; d < K; ++d) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i) { acc += G(i, d); gc[(long)i * K + d] = acc; }
        }

        /* a4: M[i][j] = beta_i sum_d k_id k_jd exp(gc_id - gc_jd), j < i */
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double acc = 0.0;
                if (j < i)
                    for (int d = 0; d < K; ++d)
                        acc += KK(i, d) * KK(j, d) * exp(gc[(long)i * K + d] - gc[(long)j * K + d]);
                M[(long)i * n + j] = bt[i] * acc;
            }

        /* a5: T = (I + M)^{-1}; A = T Diag(beta) */
        kda_oracle_tri_inverse(n, M, Tm);
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) A[(long)i * n + j] = Tm[(long)i * n + j] * bt[j];

        /* a6: W = A (exp(gc) * k), U = A v */
        for (int i = 0; i < n; ++i) {
            for (int d = 0; d < K; ++d) {
                double acc = 0.0;
                for (int j = 0; j <= i; ++j) acc += A[(long)i * n + j] * exp(gc[(long)j * K + d]) * KK(j, d);
                W[(long)i * K + d] = acc;
            }
            for (int c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int j = 0; j <= i; ++j) acc += A[(long)i * n + j] * VV(j, c);
                U[(long)i * V + c] = acc;
            }
        }

        /* a4': Aqk[i][j] = scale sum_d q_id exp(gc_id - gc_jd) k_jd, j <= i */
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double acc = 0.0;
                if (j <= i)
                    for (int d = 0; d < K; ++d)
                        acc += Q(i, d) * exp(gc[(long)i * K + d] - gc[(long)j * K + d]) * KK(j, d);
                Aqk[(long)i * n + j] = scale * acc;
            }

        /* a7: v_new = U - W S */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < V; ++c) {
                double acc = U[(long)i * V + c];
                for (int d = 0; d < K; ++d) acc -= W[(long)i * K + d] * s[(long)d * V + c];
                vnew[(long)i * V + c] = acc;
            }

        /* a8: o = (scale q exp(gc)) S + Aqk v_new */
        for (int i = 0; i < n; ++i) {
            double* oi = o + (long)(t0 + i) * o_rs;
            for (int c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int d = 0; d < K; ++d)
                    acc += scale * Q(i, d) * exp(gc[(long)i * K + d]) * s[(long)d * V + c];
                for (int j = 0; j <= i; ++j) acc += Aqk[(long)i * n + j] * vnew[(long)j * V + c];
                oi[c] = acc;
            }
        }

        /* a7': S <- Diag(exp(g_last)) S + (exp(g_last - gc) * k)^T v_new */
        for (int d = 0; d < K; ++d) {
            const double glast = gc[(long)(n - 1) * K + d];
            const double decay = exp(glast);
            for (int c = 0; c < V; ++c) {
                double acc = decay * s[(long)d * V + c];
                for (int j = 0; j < n; ++j)
                    acc += exp(glast - gc[(long)j * K + d]) * KK(j, d) * vnew[(long)j * V + c];
                s[(long)d * V + c] = acc;
            }
        }
#undef Q
#undef KK
#undef VV
#undef G
    }
    free(gc); free(M); free(Tm); free(A); free(Aqk); free(W); free(U); free(vnew); free(bt);
}

/* ------------------------------------------------------------------------ */
/* Many units, spread over threads.                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int form, chunk, H, HV, K, V;
    const float *q, *k, *v, *g, *beta;
    double scale;
    int n_units;
    const int64_t* unit_tok0;   /* first packed token row of the unit's sequence */
    const int32_t* unit_len;    /* number of tokens in the sequence */
    const int32_t* unit_hv;     /* value head */
    const float* s0;            /* initial states, or NULL for zeros */
    const int64_t* unit_s0_off; /* element offset of the unit's K*V initial state */
    double* o_out;              /* compact outputs */
    const int64_t* unit_o_off;  /* element offset of the unit's [len][V] block */
    double* s_out;              /* [n_units][K][V] final states */
    int next;                   /* work counter */
    pthread_mutex_t lock;
} oracle_job;

static void run_unit(oracle_job* J, int u)
{
    const int G = J->HV / J->H;
    const int hv = J->unit_hv[u];
    const int hk = hv / G;
    const long tok0 = (long)J->unit_tok0[u];
    const int len = J->unit_len[u];
    const int K = J->K, V = J->V;
    double* s = J->s_out + (long)u * K * V;
    if (J->s0) {
        const float* s0 = J->s0 + J->unit_s0_off[u];
        for (long i = 0; i < (long)K * V; ++i) s[i] = (double)s0[i];
    } else {
        memset(s, 0, sizeof(double) * (size_t)K * V);
    }
    const float* q = J->q + tok0 * J->H * K + (long)hk * K;
    const float* k = J->k + tok0 * J->H * K + (long)hk * K;
    const float* v = J->v + tok0 * J->HV * V + (long)hv * V;
    const float* g = J->g + tok0 * J->HV * K + (long)hv * K;
    const float* b = J->beta + tok0 * J->HV + hv;
    double* o = J->o_out + J->unit_o_off[u];
    if (J->form == 0)
        kda_oracle_unit_recurrent(len, K, V, q, (long)J->H * K, k, (long)J->H * K,
                                  v, (long)J->HV * V, g, (long)J->HV * K, b, J->HV,
                                  J->scale, s, o, V);
    else
        kda_oracle_unit_chunked(len, K, V, J->chunk, q, (long)J->H * K, k, (long)J->H * K,
                                v, (long)J->HV * V, g, (long)J->HV * K, b, J->HV,
                                J->scale, s, o, V);
}

static void* worker(void* arg)
{
    oracle_job* J = (oracle_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int u = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->n_units) break;
        run_unit(J, u);
    }
    return NULL;
}

/*
 * Run n_units units with form 0 (recurrent) or 1 (chunked, chunk size `chunk`)
 * on `nthreads` threads.  Returns 0 on success, -1 on a bad argument.
 */
int kda_oracle_run(int form, int chunk, int H, int HV, int K, int V,
                   const float* q, const float* k, const float* v,
                   const float* g, const float* beta, double scale,
                   int n_units, const int64_t* unit_tok0, const int32_t* unit_len,
                   const int32_t* unit_hv, const float* s0, const int64_t* unit_s0_off,
                   double* o_out, const int64_t* unit_o_off, double* s_out, int nthreads)
{
    if (H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0 || n_units < 0) return -1;
    if (form == 1 && chunk < 1) return -1;
    oracle_job J;
    J.form = form; J.chunk = chunk; J.H = H; J.HV = HV; J.K = K; J.V = V;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.scale = scale;
    J.n_units = n_units; J.unit_tok0 = unit_tok0; J.unit_len = unit_len; J.unit_hv = unit_hv;
    J.s0 = s0; J.unit_s0_off = unit_s0_off; J.o_out = o_out; J.unit_o_off = unit_o_off;
    J.s_out = s_out; J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &J);
    worker(&J);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Pre-stage of the gated forward.                                          */
/* ------------------------------------------------------------------------ */

/*
 * The activations that turn raw projections into the forward's inputs, as the
 * pages apply them before the chunk computation: the CPU reference's pre-stage
 * ("手撕KDA", section 2, forward_bh: l2norm, beta sigmoid, gate activation) and
 * the bounded gate of the FlashKDA walk-through ("KDA源码剖析之FlashKDA（上）",
 * part 7, gate activation) and of "手撕KDA" section 5 (k_prepare_v8):
 *
 *   q^ = q / sqrt(sum_d q_d^2 + 1e-6)        per (token, key head); k^ likewise
 *   bounded gate  (gate_kind 0):  g = lower_bound * sigmoid(exp(A_log[hv]) * (g_raw + dt_bias[hv, d]))
 *   softplus gate (gate_kind 1):  g = -exp(A_log[hv]) * softplus(g_raw + dt_bias[hv, d])
 *   beta = sigmoid(beta_raw)
 *
 * with sigmoid(x) = 1 / (1 + exp(-x)) and softplus(x) = log(1 + exp(x)).  The
 * gate parameters belong to the value head (g is [tokens, HV, K]).  Layouts as in
 * the forward: q_raw, k_raw [n_tok, H, K]; g_raw [n_tok, HV, K]; beta_raw [n_tok, HV];
 * A_log [HV]; dt_bias [HV, K].  Everything in double precision.
 */
static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }
static double softplus_d(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

void kda_oracle_prestage(long n_tok, int H, int HV, int K,
                         const float* q_raw, const float* k_raw, const float* g_raw, const float* beta_raw,
                         const float* A_log, const float* dt_bias, int gate_kind, double lower_bound,
                         double* q_out, double* k_out, double* g_out, double* beta_out)
{
    for (long t = 0; t < n_tok; ++t) {
        for (int h = 0; h < H; ++h) {
            const float* qr = q_raw + (t * H + h) * K;
            const float* kr = k_raw + (t * H + h) * K;
            double sq = 0.0, sk = 0.0;
            for (int d = 0; d < K; ++d) {
                sq += (double)qr[d] * (double)qr[d];
                sk += (double)kr[d] * (double)kr[d];
            }
            const double nq = sqrt(sq + 1e-6), nk = sqrt(sk + 1e-6);
            for (int d = 0; d < K; ++d) {
                q_out[(t * H + h) * K + d] = (double)qr[d] / nq;
                k_out[(t * H + h) * K + d] = (double)kr[d] / nk;
            }
        }
        for (int hv = 0; hv < HV; ++hv) {
            const double a = exp((double)A_log[hv]);
            for (int d = 0; d < K; ++d) {
                const double x = (double)g_raw[(t * HV + hv) * K + d] + (double)dt_bias[hv * K + d];
                g_out[(t * HV + hv) * K + d] =
                    gate_kind == 0 ? lower_bound * sigmoid_d(a * x) : -a * softplus_d(x);
            }
            beta_out[t * HV + hv] = sigmoid_d((double)beta_raw[t * HV + hv]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Backward of the recurrence (reverse mode).                               */
/* ------------------------------------------------------------------------ */

/*
 * Gradients of one unit's token recurrence (1) with respect to its inputs, for the
 * loss sum_t <do_t, o_t> + <dS_final, S_len>.  The forward is re-run and every state
 * kept; then, from the last token back, with Sp the state before token t,
 * P = Diag(e^{g_t}) Sp, u = P^T k, r = v - u and S = P + beta k r^T:
 *     dq_t   = scale S do_t                          (o_t = scale S^T q_t)
 *     dS    += scale q_t do_t^T
 *     dbeta_t = k^T dS r,     dr = beta dS^T k,      dv_t = dr
 *     dk_t   = beta dS r - P dr                       (through r and through u = P^T k)
 *     dP     = dS - k dr^T,   dg_t,i = sum_j dP_ij P_ij,   dS <- Diag(e^{g_t}) dP
 * and dS after the first token is the initial state's gradient.  The pages' backward
 * ("手撕KDA", section 2, backward_bh; section 4) works on the chunked form; this is the
 * same derivative taken through the recurrence that form evaluates.
 * s0, dfinal: K*V (NULL: zeros).  do_: len rows of V.  Outputs are written (dq, dk per
 * token of this unit: the caller sums over value heads that share a key head).
 */
void kda_oracle_unit_backward(int len, int K, int V,
                              const float* q, long q_rs, const float* k, long k_rs,
                              const float* v, long v_rs, const float* g, long g_rs,
                              const float* beta, long beta_rs, double scale,
                              const double* s0, const double* dfinal, const double* do_, long do_rs,
                              double* dq, double* dk, double* dv, double* dg, double* dbeta, double* ds0)
{
    const size_t KV = (size_t)K * V;
    double* S = (double*)calloc((size_t)(len + 1) * KV, sizeof(double));
    double* dS = (double*)calloc(KV, sizeof(double));
    double* P = (double*)malloc(KV * sizeof(double));
    double* r = (double*)malloc((size_t)V * sizeof(double));
    double* dr = (double*)malloc((size_t)V * sizeof(double));
    if (s0) memcpy(S, s0, KV * sizeof(double));
    for (int t = 0; t < len; ++t) {   /* forward, keeping every state */
        const double* Sp = S + (size_t)t * KV;
        double* Sn = S + (size_t)(t + 1) * KV;
        const float* kt = k + (long)t * k_rs;
        const float* vt = v + (long)t * v_rs;
        const float* gt = g + (long)t * g_rs;
        const double bt = (double)beta[(long)t * beta_rs];
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j) Sn[(size_t)i * V + j] = exp((double)gt[i]) * Sp[(size_t)i * V + j];
        for (int j = 0; j < V; ++j) {
            double u = 0.0;
            for (int i = 0; i < K; ++i) u += Sn[(size_t)i * V + j] * (double)kt[i];
            r[j] = (double)vt[j] - u;
        }
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j) Sn[(size_t)i * V + j] += bt * (double)kt[i] * r[j];
    }
    if (dfinal) memcpy(dS, dfinal, KV * sizeof(double));
    for (int t = len - 1; t >= 0; --t) {
        const double* Sp = S + (size_t)t * KV;
        const double* St = S + (size_t)(t + 1) * KV;
        const float* qt = q + (long)t * q_rs;
        const float* kt = k + (long)t * k_rs;
        const float* vt = v + (long)t * v_rs;
        const float* gt = g + (long)t * g_rs;
        const double bt = (double)beta[(long)t * beta_rs];
        const double* dot = do_ + (long)t * do_rs;
        for (int i = 0; i < K; ++i) {
            const double e = exp((double)gt[i]);
            for (int j = 0; j < V; ++j) P[(size_t)i * V + j] = e * Sp[(size_t)i * V + j];
        }
        for (int j = 0; j < V; ++j) {
            double u = 0.0;
            for (int i = 0; i < K; ++i) u += P[(size_t)i * V + j] * (double)kt[i];
            r[j] = (double)vt[j] - u;
        }
        for (int i = 0; i < K; ++i) {   /* dq = scale S do; then the output's share of dS */
            double a = 0.0;
            for (int j = 0; j < V; ++j) a += St[(size_t)i * V + j] * dot[j];
            dq[(long)t * K + i] = scale * a;
            for (int j = 0; j < V; ++j) dS[(size_t)i * V + j] += scale * (double)qt[i] * dot[j];
        }
        double db = 0.0;
        for (int j = 0; j < V; ++j) {
            double a = 0.0;
            for (int i = 0; i < K; ++i) a += dS[(size_t)i * V + j] * (double)kt[i];
            dr[j] = bt * a;
            db += a * r[j];
            dv[(long)t * V + j] = dr[j];
        }
        dbeta[t] = db;
        for (int i = 0; i < K; ++i) {
            double a = 0.0, c = 0.0, d = 0.0;
            for (int j = 0; j < V; ++j) {
                a += dS[(size_t)i * V + j] * r[j];
                c += P[(size_t)i * V + j] * dr[j];
            }
            dk[(long)t * K + i] = bt * a - c;
            const double e = exp((double)gt[i]);
            for (int j = 0; j < V; ++j) {
                const double dP = dS[(size_t)i * V + j] - (double)kt[i] * dr[j];
                d += dP * P[(size_t)i * V + j];
                dS[(size_t)i * V + j] = e * dP;
            }
            dg[(long)t * K + i] = d;
        }
    }
    memcpy(ds0, dS, KV * sizeof(double));
    free(S); free(dS); free(P); free(r); free(dr);
}
