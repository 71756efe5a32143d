/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for the Kimi Delta Attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library; its only common ground with the GPU path is the seeded input data.
 *
 * What it computes (per independent (sequence, head) unit, token by token):
 *
 *   q^ = q / sqrt(sum q^2 + l2_eps),  k^ = k / sqrt(sum k^2 + l2_eps)   (optional)
 *   S  <- Diag(exp g_t) S                      decay each key channel first
 *   D  =  beta_t (v_t - S^T k^)                delta-rule write residual
 *   S  <- S + k^ D^T                           rank-one write
 *   o_t = scale * S^T q^                       read-out after the write
 *
 * Sources (page title, section):
 *  - nnterp encyclopedia "Kimi-Linear", section 03 "Kimi Delta Attention decays
 *    each key channel": KDA is a gated DeltaNet whose log decay g is per key
 *    channel, float32 and non-positive; beta is the sigmoid of b_proj; queries
 *    and keys are L2-normalised by the kernel and queries scaled by
 *    1/sqrt(key_dim); the state is [batch, heads, key_dim, value_dim].
 *  - same page, section 04 "From the family module": the state decays channel by
 *    channel before each delta-rule update; the kernels take
 *    (query, key, value, g=, beta=, initial_state=) and return
 *    (core_attn_out, last_recurrent_state); use_qk_l2norm_in_kernel.
 *  - same page, section 02 "support()" value table: layouts
 *    attention_queries/keys [batch seq heads key_dim], attention_values
 *    [batch seq heads value_dim], decays [batch seq heads key_dim],
 *    betas [batch seq heads], state_input / state_output
 *    [batch heads key_dim value_dim], states [batch seq heads key_dim value_dim].
 *  - Kimi-K3 atlas page "dense KDA layers / attention / gate-project (decode,
 *    P = 1000)", sections "Parameters" and "Code": the head outputs pass a
 *    gated RMSNorm over each head (head_dim = 128 weights shared by all heads,
 *    eps = rms_norm_eps, activation 'sigmoid') before the output projection.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *  - the L2 norm puts its epsilon inside the square root (l2_eps, 1e-6 by default);
 *  - the gated norm is y = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate);
 *  - the gate multiplies after the weight; the mean runs over value_dim of one head.
 *
 * Parity status: every function here is pinned by the CPU tests (closed forms,
 * brute-force transition products, split-halves, column independence,
 * orthonormal-key erase, norm special cases and a library RMSNorm).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_ORACLE_VERSION 1

int kda_oracle_version(void) { return KDA_ORACLE_VERSION; }

/* ------------------------------------------------------------------------- */
/* Recurrence                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    const float *q, *k, *v;               /* token-major inputs, see kda_oracle_recurrent */
    const double *g, *beta;               /* log decay and write strength (fp64) */
    const double *initial_state;          /* [N,H,K,V] or NULL (zero state) */
    double *o;                            /* [tokens,H,V] */
    double *final_state;                  /* [N,H,K,V] or NULL */
    double *states;                       /* [tokens,H,K,V] or NULL */
    const int64_t *starts;                /* per-sequence first token row, N entries */
    const int64_t *lens;                  /* per-sequence token count, N entries */
    int64_t n_units;                      /* N * H */
    int H, K, V;
    double scale, l2_eps;
    int use_qk_l2norm;
    int n_threads, tid;
} rec_job;

/* One (sequence, head) unit, token by token, in fp64. */
static void rec_unit(const rec_job *J, int64_t unit, double *S, double *qh, double *kh,
                     double *u, double *delta) {
    const int H = J->H, K = J->K, V = J->V;
    const int64_t n = unit / H;
    const int h = (int)(unit % H);
    const int64_t row0 = J->starts[n], len = J->lens[n];

    if (J->initial_state) {
        const double *s0 = J->initial_state + ((size_t)n * H + h) * (size_t)K * V;
        memcpy(S, s0, sizeof(double) * (size_t)K * V);
    } else {
        memset(S, 0, sizeof(double) * (size_t)K * V);
    }

    for (int64_t t = 0; t < len; ++t) {
        const int64_t row = row0 + t;
        const float *qt = J->q + ((size_t)row * H + h) * K;
        const float *kt = J->k + ((size_t)row * H + h) * K;
        const float *vt = J->v + ((size_t)row * H + h) * V;
        const double *gt = J->g + ((size_t)row * H + h) * K;
        const double bt = J->beta[(size_t)row * H + h];

        /* L2 normalisation of query and key over key_dim (optional). */
        double sq = 0.0, sk = 0.0;
        for (int i = 0; i < K; ++i) {
            sq += (double)qt[i] * (double)qt[i];
            sk += (double)kt[i] * (double)kt[i];
        }
        const double rq = J->use_qk_l2norm ? 1.0 / sqrt(sq + J->l2_eps) : 1.0;
        const double rk = J->use_qk_l2norm ? 1.0 / sqrt(sk + J->l2_eps) : 1.0;
        for (int i = 0; i < K; ++i) {
            qh[i] = (double)qt[i] * rq;
            kh[i] = (double)kt[i] * rk;
        }

        /* Decay each key channel (row i of S) by exp(g_t[i]) before the update. */
        for (int i = 0; i < K; ++i) {
            const double a = exp((double)gt[i]);
            double *Si = S + (size_t)i * V;
            for (int j = 0; j < V; ++j) Si[j] *= a;
        }

        /* u = S^T k^ ; delta = beta (v - u). */
        for (int j = 0; j < V; ++j) u[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double ki = kh[i];
            const double *Si = S + (size_t)i * V;
            for (int j = 0; j < V; ++j) u[j] += Si[j] * ki;
        }
        for (int j = 0; j < V; ++j) delta[j] = bt * ((double)vt[j] - u[j]);

        /* S <- S + k^ delta^T. */
        for (int i = 0; i < K; ++i) {
            const double ki = kh[i];
            double *Si = S + (size_t)i * V;
            for (int j = 0; j < V; ++j) Si[j] += ki * delta[j];
        }

        /* o_t = scale * S^T q^. */
        double *ot = J->o + ((size_t)row * H + h) * V;
        for (int j = 0; j < V; ++j) u[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double qi = qh[i];
            const double *Si = S + (size_t)i * V;
            for (int j = 0; j < V; ++j) u[j] += Si[j] * qi;
        }
        for (int j = 0; j < V; ++j) ot[j] = J->scale * u[j];

        if (J->states) {
            double *st = J->states + ((size_t)row * H + h) * (size_t)K * V;
            memcpy(st, S, sizeof(double) * (size_t)K * V);
        }
    }

    if (J->final_state) {
        double *sf = J->final_state + ((size_t)n * H + h) * (size_t)K * V;
        memcpy(sf, S, sizeof(double) * (size_t)K * V);
    }
}

static void *rec_worker(void *arg) {
    const rec_job *J = (const rec_job *)arg;
    const int K = J->K, V = J->V;
    double *S = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * K + 2 * V));
    if (!S || !buf) {
        free(S);
        free(buf);
        return (void *)1;
    }
    for (int64_t unit = J->tid; unit < J->n_units; unit += J->n_threads)
        rec_unit(J, unit, S, buf, buf + K, buf + 2 * K, buf + 2 * K + V);
    free(S);
    free(buf);
    return NULL;
}

/*
 * kda_oracle_recurrent -- run the recurrence over every (sequence, head) unit.
 *
 * Host arrays, all row-major and contiguous:
 *   q, k   [rows, H, K] float (bf16 values widened exactly to float by the caller)
 *   v      [rows, H, V] float
 *   g      [rows, H, K] float, the per-channel log decay (non-positive)
 *   beta   [rows, H]    float
 *   initial_state [N, H, K, V] double or NULL for a zero state
 *   o      [rows, H, V] double (written)
 *   final_state [N, H, K, V] double or NULL
 *   states [rows, H, K, V] double or NULL: the state after every token
 * Sequences: if cu_seqlens is NULL there are N = B sequences of T tokens each and
 * rows = B*T; otherwise N = n_seqs, sequence n covers rows
 * [cu_seqlens[n], cu_seqlens[n+1]) and rows = cu_seqlens[n_seqs].
 * Returns 0 on success, -1 on a bad argument, -2 on an allocation failure.
 */
int kda_oracle_recurrent(const float *q, const float *k, const float *v, const double *g,
                         const double *beta, const double *initial_state, double *o,
                         double *final_state, double *states, const int64_t *cu_seqlens,
                         int n_seqs, int B, int T, int H, int K, int V, double scale,
                         int use_qk_l2norm, double l2_eps, int n_threads) {
    if (!q || !k || !v || !g || !beta || !o) return -1;
    if (H <= 0 || K <= 0 || V <= 0) return -1;
    int64_t N;
    int64_t *starts, *lens;
    if (cu_seqlens) {
        if (n_seqs <= 0) return -1;
        N = n_seqs;
        starts = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        lens = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        if (!starts || !lens) {
            free(starts);
            free(lens);
            return -2;
        }
        for (int64_t n = 0; n < N; ++n) {
            if (cu_seqlens[n + 1] < cu_seqlens[n] || cu_seqlens[n] < 0) {
                free(starts);
                free(lens);
                return -1;
            }
            starts[n] = cu_seqlens[n];
            lens[n] = cu_seqlens[n + 1] - cu_seqlens[n];
        }
    } else {
        if (B <= 0 || T < 0) return -1;
        N = B;
        starts = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        lens = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        if (!starts || !lens) {
            free(starts);
            free(lens);
            return -2;
        }
        for (int64_t n = 0; n < N; ++n) {
            starts[n] = n * (int64_t)T;
            lens[n] = T;
        }
    }
    if (n_threads < 1) n_threads = 1;
    const int64_t n_units = N * H;
    if (n_threads > n_units) n_threads = (int)n_units;

    rec_job *jobs = (rec_job *)malloc(sizeof(rec_job) * (size_t)n_threads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        free(starts);
        free(lens);
        return -2;
    }
    int rc = 0;
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        rec_job J = {q, k, v, g, beta, initial_state, o, final_state, states, starts, lens,
                     n_units, H, K, V, scale, l2_eps, use_qk_l2norm, n_threads, i};
        jobs[i] = J;
    }
    for (int i = 1; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, rec_worker, &jobs[i]) != 0) {
            rc = -2;
            break;
        }
        started = i;
    }
    if (rec_worker(&jobs[0]) != NULL) rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    free(jobs);
    free(th);
    free(starts);
    free(lens);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Sigmoid-gated RMSNorm over each head                                       */
/* ------------------------------------------------------------------------- */

/*
 * kda_oracle_gated_rmsnorm -- y = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate).
 *
 * Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters" (the
 * gated RMSNorm holds 128 weights, one vector shared by all 96 heads) and "Code"
 * (o_norm(o, g) on [.., heads, head_dim] with activation 'sigmoid', then the
 * heads are flattened to [.., heads * head_dim]).
 *
 *   o    [rows, H, V] double      gate [rows, H, V] float (bf16 values widened)
 *   w    [V] float                y    [rows, H*V] double (written)
 */
int kda_oracle_gated_rmsnorm(const double *o, const float *gate, const float *w, double eps,
                             double *y, int64_t rows, int H, int V) {
    if (!o || !gate || !w || !y || rows < 0 || H <= 0 || V <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h) {
            const double *x = o + ((size_t)r * H + h) * V;
            const float *gt = gate + ((size_t)r * H + h) * V;
            double *yt = y + ((size_t)r * H + h) * V;
            double ss = 0.0;
            for (int j = 0; j < V; ++j) ss += x[j] * x[j];
            const double inv = 1.0 / sqrt(ss / (double)V + eps);
            for (int j = 0; j < V; ++j) {
                const double sig = 1.0 / (1.0 + exp(-(double)gt[j]));
                yt[j] = x[j] * inv * (double)w[j] * sig;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Short convolution                                                          */
/* ------------------------------------------------------------------------- */

/*
 * Causal depthwise convolution along the sequence with an optional SiLU, the
 * preprocessing of q, k and v.
 *
 * nnterp encyclopedia "Kimi-Linear", section "Printout": the layer's conv1d is
 * Conv1d(12288, 12288, kernel_size=(4,), stride=(1,), padding=(3,), groups=12288,
 * bias=False) -- one filter of 4 taps per channel, padded by 3 positions before
 * the first token; the first T outputs are the causal ones.  Kimi-K3 atlas
 * "gate-project (decode, P = 1000)", section "Code": q_conv1d, k_conv1d and
 * v_conv1d are ShortConvolution(hidden_size, kernel_size=short_conv_kernel_size,
 * activation='silu'), with short_conv_kernel_size = 4 in the config.
 *
 * For each sequence and channel c (cross-correlation, as Conv1d computes it):
 *   y[t][c] = act( bias[c] + sum_{w=0}^{W-1} weight[c][w] * x[t - (W-1) + w][c] )
 * A position before the sequence start takes its input from the conv state (the
 * W-1 inputs before the sequence, oldest first) or zero; act(z) = z / (1 + e^-z)
 * (SiLU) or z.  The state afterwards holds the last W-1 inputs, oldest first.
 *
 *   x         [B, T, D] float (bf16 values widened); varlen: B = 1, n_seqs > 0
 *   weight    [D, W] double        bias [D] double or NULL
 *   state_in  [N, W-1, D] double or NULL      state_out [N, W-1, D] double or NULL
 *   y         [B, T, D] double
 */
int kda_oracle_short_conv(const float *x, const double *weight, const double *bias,
                          const double *state_in, double *y, double *state_out,
                          const int64_t *cu_seqlens, int n_seqs, int B, int T, int D, int W, int act) {
    if (!weight || D <= 0 || W < 1 || W > 64 || B < 0 || T < 0) return -1;
    const int N = cu_seqlens ? n_seqs : B;
    double hist[64];
    for (int n = 0; n < N; ++n) {
        int64_t bos, len;
        if (cu_seqlens) {
            bos = cu_seqlens[n];
            len = cu_seqlens[n + 1] - cu_seqlens[n];
        } else {
            bos = (int64_t)n * T;
            len = T;
        }
        if (len < 0) return -2;
        for (int c = 0; c < D; ++c) {
            for (int w = 0; w < W - 1; ++w)
                hist[w] = state_in ? state_in[((size_t)n * (W - 1) + w) * D + c] : 0.0;
            for (int64_t t = 0; t < len; ++t) {
                const double xt = (double)x[(size_t)(bos + t) * D + c];
                double z = bias ? bias[c] : 0.0;
                for (int w = 0; w < W - 1; ++w) z += weight[(size_t)c * W + w] * hist[w];
                z += weight[(size_t)c * W + W - 1] * xt;
                y[(size_t)(bos + t) * D + c] = act ? z / (1.0 + exp(-z)) : z;
                for (int w = 0; w + 1 < W - 1; ++w) hist[w] = hist[w + 1];
                if (W > 1) hist[W - 2] = xt;
            }
            if (state_out)
                for (int w = 0; w < W - 1; ++w) state_out[((size_t)n * (W - 1) + w) * D + c] = hist[w];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Decay and write strength from their logits                                 */
/* ------------------------------------------------------------------------- */

/*
 * The layer's gate parameters, from the logits the projections produce.
 *
 * Kimi-K3 atlas "gate-project (decode, P = 1000)", section "Code" (the layer
 * holds A_log = log U(1, 16), one per head; f_a_proj / f_b_proj, the rank-128
 * pair producing one decay logit per key channel of each head; dt_bias, one bias
 * per such logit; b_proj, one write-strength logit per head; gate_lower_bound);
 * nnterp encyclopedia "Kimi-Linear", section 03 (g is per key channel, float32
 * and non-positive; beta is the sigmoid of b_proj).  The pages omit the line that
 * combines them; the reading used here (the plainest one the parameters support):
 *
 *   g[t][h][c] = max(lower_bound, -exp(A_log[h]) * softplus(z[t][h][c] + dt_bias[h][c]))
 *   beta[t][h] = 1 / (1 + exp(-b[t][h]))
 *
 * with softplus(x) = log(1 + e^x), evaluated as max(x, 0) + log1p(e^-|x|).
 *
 *   z       [rows, H, K] float (bf16 values widened)     A_log [H] float
 *   dt_bias [H, K] float or NULL (zero)                  lower_bound: -INFINITY for none
 *   b       [rows, H] float                              g [rows, H, K], beta [rows, H] double (written)
 */
int kda_oracle_gates(const float *z, const float *A_log, const float *dt_bias, double lower_bound,
                     const float *b, double *g, double *beta, int64_t rows, int H, int K) {
    if (!z || !A_log || !b || !g || !beta || rows < 0 || H <= 0 || K <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h) {
            const double a = exp((double)A_log[h]);
            for (int c = 0; c < K; ++c) {
                const size_t i = ((size_t)r * H + h) * K + c;
                const double x = (double)z[i] + (dt_bias ? (double)dt_bias[(size_t)h * K + c] : 0.0);
                const double sp = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
                const double gv = -a * sp;
                g[i] = gv > lower_bound ? gv : lower_bound;
            }
            beta[(size_t)r * H + h] = 1.0 / (1.0 + exp(-(double)b[(size_t)r * H + h]));
        }
    }
    return 0;
}
