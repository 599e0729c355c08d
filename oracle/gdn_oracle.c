/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle of the Gated-DeltaNet token mixer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the package smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header or constant with the CUDA library.
 *
 * What it follows: "qwen35moe -- Forward-Pass Design (Pantheon port)", section
 * "SSM block -- Gated-Delta-Net" (projections, decay gate, causal conv1d, the
 * per-token recurrence and the output path) and its "Correctness watch-list".
 * Every routine below cites the part of that section it restates.
 *
 * State convention here is the page's: S[i][j] with i the key index and j the
 * value index, stored row-major (i outer). The CUDA library stores the
 * transpose; the tests transpose explicitly.
 *
 * All dimensions are run-time arguments so that brute-force checks can run on
 * tiny heads (d = 2..4).  All arithmetic is double precision, scalar loops in
 * the order the page states.
 *
 * Readings taken where the page is silent (each also listed in the design
 * notes of the repository):
 *   - conv tap m multiplies the window element m, window = [3 oldest state
 *     rows, current input]; tap K-1 multiplies the current token; no bias.
 *   - L2 normalisation is x / sqrt(sum x^2 + eps_l2).
 *   - softplus(x) = x for x > 20, else log1p(exp(x)).
 *   - the gated RMSNorm runs per V-head over the value dimension with one
 *     shared weight vector, applied as w (the page says +1 is pre-baked).
 *   - the 1/sqrt(d_k) scale is applied once, to y, after the state write.
 *
 * Parity pins live in tests/test_oracle_pins.py; every routine here has at
 * least one pin that does not re-derive it from this file.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* Dimensions of one GDN layer. conv channels C = 2*Hk*dk + Hv*dv
 * (q heads | k heads | v heads, head-major inside each block). */
typedef struct {
    int Hv;   /* value heads ("time_step_rank", 32 on the page)          */
    int Hk;   /* key/query heads ("group_count", 16 on the page)          */
    int dk;   /* key head dim ("state_size", 128)                         */
    int dv;   /* value head dim (d_inner / Hv = 128)                      */
    int Kc;   /* conv kernel width ("conv_kernel", 4)                     */
} oracle_dims;

static int conv_channels(const oracle_dims *d) { return 2 * d->Hk * d->dk + d->Hv * d->dv; }

/* SiLU(x) = x * sigmoid(x): "conv ... -> SiLU", and the output gate silu(z). */
static double silu(double x) { return x / (1.0 + exp(-x)); }

/* Decay gate, section "Decay gate (scalar per V-head)":
 *   g = -exp(A_log) * softplus(alpha + dt_bias);   beta_gate = sigmoid(beta).
 * Returns g (not exp(g)); the recurrence applies exp(g). */
double oracle_softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

void oracle_gates(double A_log, double dt_bias, double alpha, double beta,
                  double *g_out, double *b_out)
{
    *g_out = -exp(A_log) * oracle_softplus(alpha + dt_bias);
    *b_out = 1.0 / (1.0 + exp(-beta));
}

/* Causal depthwise conv1d + SiLU over one token, section "Causal conv1d":
 * the conv runs over the whole q|k|v stream with the last Kc-1 inputs
 * (conv_state, oldest row first) prepended, then SiLU; afterwards the current
 * raw input is pushed into conv_state (the oldest row drops out).
 *   x      [C]        raw input of this token
 *   w      [C][Kc]    per-channel taps
 *   state  [Kc-1][C]  in/out
 *   xhat   [C]        out */
void oracle_conv_token(int C, int Kc, const double *x, const double *w,
                       double *state, double *xhat)
{
    for (int c = 0; c < C; ++c) {
        double u = 0.0;
        for (int m = 0; m < Kc - 1; ++m) u += w[(size_t)c * Kc + m] * state[(size_t)m * C + c];
        u += w[(size_t)c * Kc + (Kc - 1)] * x[c];
        xhat[c] = silu(u);
    }
    for (int m = 0; m + 1 < Kc - 1; ++m)
        for (int c = 0; c < C; ++c) state[(size_t)m * C + c] = state[(size_t)(m + 1) * C + c];
    if (Kc > 1)
        for (int c = 0; c < C; ++c) state[(size_t)(Kc - 2) * C + c] = x[c];
}

/* "L2-normalize q and k over head dim (not RMS)". */
void oracle_l2norm(int n, const double *x, double eps, double *out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * inv;
}

/* One step of the delta-rule recurrence, section "Per-token recurrence",
 * steps (a)-(d), on S[i][j] (dk x dv, row-major in i):
 *   (a) S' = exp(g) * S
 *   (b) pred_j = sum_i S'[i][j] k[i];  delta_j = (v_j - pred_j) * b
 *   (c) S[i][j] = S'[i][j] + k[i] * delta_j
 *   (d) y_j = scale * sum_i S[i][j] q[i]        (read AFTER the write) */
void oracle_delta_rule_token(int dk, int dv, double *S, const double *k, const double *v,
                             const double *q, double g, double b, double scale, double *y)
{
    double a = exp(g);
    for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= a;
    for (int j = 0; j < dv; ++j) {
        double pred = 0.0;
        for (int i = 0; i < dk; ++i) pred += S[(size_t)i * dv + j] * k[i];
        double delta = (v[j] - pred) * b;
        for (int i = 0; i < dk; ++i) S[(size_t)i * dv + j] += k[i] * delta;
    }
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * q[i];
        y[j] = scale * acc;
    }
}

/* Output path, "gated = RMSNorm(y, ssm_norm) * silu(z)" -- silu, not sigmoid;
 * plain x * rms^-1 * w since the +1 is baked into the weight. */
void oracle_gated_rmsnorm(int n, const double *y, const double *z, const double *w,
                          double eps, double *out)
{
    double ms = 0.0;
    for (int j = 0; j < n; ++j) ms += y[j] * y[j];
    ms /= (double)n;
    double r = 1.0 / sqrt(ms + eps);
    for (int j = 0; j < n; ++j) out[j] = y[j] * r * w[j] * silu(z[j]);
}

/* The whole SSM block for one sequence of T tokens, from the projected
 * streams to the gated output (the "SSM block -- Gated-Delta-Net" section in
 * page order: conv -> split -> L2 -> GQA repeat -> gates -> recurrence ->
 * gated RMSNorm).  GQA: V-head vh reads K-head vh % Hk (watch-list item on
 * the ggml_repeat interleave).
 *   qkv   [T][C]         z      [T][Hv*dv]   alpha, beta [T][Hv]
 *   conv_w[C][Kc]        A_log, dt_bias [Hv]  norm_w [dv]
 *   conv_state [Kc-1][C] in/out               S [Hv][dk][dv] in/out
 *   out   [T][Hv*dv]
 * Returns 0, or -1 on a bad argument or allocation failure. */
int oracle_gdn_sequence(const oracle_dims *d, int T,
                        const double *qkv, const double *z, const double *alpha,
                        const double *beta, const double *conv_w, const double *A_log,
                        const double *dt_bias, const double *norm_w, double l2_eps,
                        double norm_eps, double *conv_state, double *S, double *out)
{
    if (!d || T < 0 || d->Hv <= 0 || d->Hk <= 0 || d->dk <= 0 || d->dv <= 0 || d->Kc <= 0)
        return -1;
    const int C = conv_channels(d);
    const double scale = 1.0 / sqrt((double)d->dk);
    double *xhat = (double *)malloc(sizeof(double) * (size_t)C);
    double *qn = (double *)malloc(sizeof(double) * (size_t)d->dk);
    double *kn = (double *)malloc(sizeof(double) * (size_t)d->dk);
    double *y = (double *)malloc(sizeof(double) * (size_t)d->dv);
    if (!xhat || !qn || !kn || !y) { free(xhat); free(qn); free(kn); free(y); return -1; }

    for (int t = 0; t < T; ++t) {
        oracle_conv_token(C, d->Kc, qkv + (size_t)t * C, conv_w, conv_state, xhat);
        for (int vh = 0; vh < d->Hv; ++vh) {
            int kh = vh % d->Hk;
            const double *q = xhat + (size_t)kh * d->dk;
            const double *k = xhat + (size_t)d->Hk * d->dk + (size_t)kh * d->dk;
            const double *v = xhat + (size_t)2 * d->Hk * d->dk + (size_t)vh * d->dv;
            oracle_l2norm(d->dk, q, l2_eps, qn);
            oracle_l2norm(d->dk, k, l2_eps, kn);
            double g, b;
            oracle_gates(A_log[vh], dt_bias[vh], alpha[(size_t)t * d->Hv + vh],
                         beta[(size_t)t * d->Hv + vh], &g, &b);
            oracle_delta_rule_token(d->dk, d->dv, S + (size_t)vh * d->dk * d->dv, kn, v, qn,
                                    g, b, scale, y);
            oracle_gated_rmsnorm(d->dv, y, z + (size_t)t * d->Hv * d->dv + (size_t)vh * d->dv,
                                 norm_w, norm_eps, out + (size_t)t * d->Hv * d->dv + (size_t)vh * d->dv);
        }
    }
    free(xhat); free(qn); free(kn); free(y);
    return 0;
}

/* Same as oracle_gdn_sequence, restricted to the V-heads in [vh0, vh1): the
 * heads are independent chains once the conv is done, so a caller can split a
 * layer across threads or sample a few heads.  conv_state is advanced exactly
 * as in the full call (all C channels). out rows hold only the chosen heads
 * (other columns untouched). */
int oracle_gdn_sequence_heads(const oracle_dims *d, int T, int vh0, int vh1,
                              const double *qkv, const double *z, const double *alpha,
                              const double *beta, const double *conv_w, const double *A_log,
                              const double *dt_bias, const double *norm_w, double l2_eps,
                              double norm_eps, double *conv_state, double *S, double *out)
{
    if (!d || T < 0 || vh0 < 0 || vh1 > d->Hv || vh0 > vh1) return -1;
    const int C = conv_channels(d);
    const double scale = 1.0 / sqrt((double)d->dk);
    double *xhat = (double *)malloc(sizeof(double) * (size_t)C);
    double *qn = (double *)malloc(sizeof(double) * (size_t)d->dk);
    double *kn = (double *)malloc(sizeof(double) * (size_t)d->dk);
    double *y = (double *)malloc(sizeof(double) * (size_t)d->dv);
    if (!xhat || !qn || !kn || !y) { free(xhat); free(qn); free(kn); free(y); return -1; }
    for (int t = 0; t < T; ++t) {
        oracle_conv_token(C, d->Kc, qkv + (size_t)t * C, conv_w, conv_state, xhat);
        for (int vh = vh0; vh < vh1; ++vh) {
            int kh = vh % d->Hk;
            const double *q = xhat + (size_t)kh * d->dk;
            const double *k = xhat + (size_t)d->Hk * d->dk + (size_t)kh * d->dk;
            const double *v = xhat + (size_t)2 * d->Hk * d->dk + (size_t)vh * d->dv;
            oracle_l2norm(d->dk, q, l2_eps, qn);
            oracle_l2norm(d->dk, k, l2_eps, kn);
            double g, b;
            oracle_gates(A_log[vh], dt_bias[vh], alpha[(size_t)t * d->Hv + vh],
                         beta[(size_t)t * d->Hv + vh], &g, &b);
            oracle_delta_rule_token(d->dk, d->dv, S + (size_t)vh * d->dk * d->dv, kn, v, qn,
                                    g, b, scale, y);
            oracle_gated_rmsnorm(d->dv, y, z + (size_t)t * d->Hv * d->dv + (size_t)vh * d->dv,
                                 norm_w, norm_eps, out + (size_t)t * d->Hv * d->dv + (size_t)vh * d->dv);
        }
    }
    free(xhat); free(qn); free(kn); free(y);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Chunked (WY / UT-transform) form of the same recurrence, one head.
 *
 * The pages only say that prefill may be evaluated either as a token scan or
 * reorganised into blocks ("Optimizing on-device inference for Apple silicon",
 * the section on the three workload shapes).  This routine writes the block
 * form out by plain algebra from the per-token recurrence above, so the tests
 * can check that the re-association is exact in fp64 before the CUDA chunked
 * kernel relies on it.  Within a chunk of length n starting from state S0,
 * with G_r = sum_{s<=r} g_s (chunk-local) and gamma_r = exp(G_r):
 *   L[r][s]  = exp(G_r - G_s) * (k_r . k_s)          for s < r
 *   T        = (I + diag(b) L)^{-1} diag(b)          (unit lower solve)
 *   U        = T V,     W = T diag(gamma) K
 *   Vnew     = U - W S0                              (= the per-token deltas)
 *   Y        = scale * (diag(gamma) Q S0 + (Mask o Q K^T) Vnew),
 *              Mask[r][s] = exp(G_r - G_s) for s <= r, else 0
 *   S_end    = gamma_n S0 + K^T diag(exp(G_n - G_s)) Vnew
 * Every exponent used is <= 0 (r >= s), never the inverse decay.
 *   q,k [T][dk], v [T][dv], g,b [T], S [dk][dv] in/out, y [T][dv] out.
 * Returns 0 or -1. */
int oracle_delta_rule_chunked(int dk, int dv, int T, int chunk, const double *q,
                              const double *k, const double *v, const double *g,
                              const double *b, double scale, double *S, double *y)
{
    if (dk <= 0 || dv <= 0 || T < 0 || chunk <= 0) return -1;
    const int n_max = chunk;
    double *G = (double *)malloc(sizeof(double) * n_max);
    double *Lm = (double *)malloc(sizeof(double) * n_max * n_max);
    double *Tm = (double *)malloc(sizeof(double) * n_max * n_max);
    double *U = (double *)malloc(sizeof(double) * (size_t)n_max * dv);
    double *W = (double *)malloc(sizeof(double) * (size_t)n_max * dk);
    double *Vn = (double *)malloc(sizeof(double) * (size_t)n_max * dv);
    double *S0 = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    if (!G || !Lm || !Tm || !U || !W || !Vn || !S0) {
        free(G); free(Lm); free(Tm); free(U); free(W); free(Vn); free(S0);
        return -1;
    }
    for (int c0 = 0; c0 < T; c0 += chunk) {
        const int n = (T - c0 < chunk) ? (T - c0) : chunk;
        const double *Q = q + (size_t)c0 * dk, *K = k + (size_t)c0 * dk, *V = v + (size_t)c0 * dv;
        const double *gb = g + c0, *bb = b + c0;
        memcpy(S0, S, sizeof(double) * (size_t)dk * dv);
        /* chunk-local cumulative log-decay */
        double acc = 0.0;
        for (int r = 0; r < n; ++r) { acc += gb[r]; G[r] = acc; }
        /* L (strictly lower) */
        for (int r = 0; r < n; ++r)
            for (int s = 0; s < n; ++s) {
                double val = 0.0;
                if (s < r) {
                    double dot = 0.0;
                    for (int i = 0; i < dk; ++i) dot += K[(size_t)r * dk + i] * K[(size_t)s * dk + i];
                    val = exp(G[r] - G[s]) * dot;
                }
                Lm[r * n + s] = val;
            }
        /* T = (I + diag(b) L)^{-1} diag(b): forward substitution, column s of
         * T solves (I + diag(b)L) x = b_s e_s. */
        for (int s = 0; s < n; ++s) {
            for (int r = 0; r < n; ++r) {
                double rhs = (r == s) ? bb[s] : 0.0;
                double sum = 0.0;
                for (int p = 0; p < r; ++p) sum += bb[r] * Lm[r * n + p] * Tm[p * n + s];
                Tm[r * n + s] = rhs - sum;
            }
        }
        /* U = T V, W = T diag(gamma) K */
        for (int r = 0; r < n; ++r) {
            for (int j = 0; j < dv; ++j) {
                double a2 = 0.0;
                for (int s = 0; s < n; ++s) a2 += Tm[r * n + s] * V[(size_t)s * dv + j];
                U[(size_t)r * dv + j] = a2;
            }
            for (int i = 0; i < dk; ++i) {
                double a2 = 0.0;
                for (int s = 0; s < n; ++s) a2 += Tm[r * n + s] * exp(G[s]) * K[(size_t)s * dk + i];
                W[(size_t)r * dk + i] = a2;
            }
        }
        /* Vnew = U - W S0 */
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double ws = 0.0;
                for (int i = 0; i < dk; ++i) ws += W[(size_t)r * dk + i] * S0[(size_t)i * dv + j];
                Vn[(size_t)r * dv + j] = U[(size_t)r * dv + j] - ws;
            }
        /* Y = scale (diag(gamma) Q S0 + (Mask o Q K^T) Vnew) */
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double inter = 0.0;
                for (int i = 0; i < dk; ++i) inter += Q[(size_t)r * dk + i] * S0[(size_t)i * dv + j];
                double intra = 0.0;
                for (int s = 0; s <= r; ++s) {
                    double qk = 0.0;
                    for (int i = 0; i < dk; ++i) qk += Q[(size_t)r * dk + i] * K[(size_t)s * dk + i];
                    intra += exp(G[r] - G[s]) * qk * Vn[(size_t)s * dv + j];
                }
                y[(size_t)(c0 + r) * dv + j] = scale * (exp(G[r]) * inter + intra);
            }
        /* S_end = gamma_n S0 + K^T diag(exp(G_n - G_s)) Vnew */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double upd = 0.0;
                for (int s = 0; s < n; ++s)
                    upd += K[(size_t)s * dk + i] * exp(G[n - 1] - G[s]) * Vn[(size_t)s * dv + j];
                S[(size_t)i * dv + j] = exp(G[n - 1]) * S0[(size_t)i * dv + j] + upd;
            }
    }
    free(G); free(Lm); free(Tm); free(U); free(W); free(Vn); free(S0);
    return 0;
}

/* The token-scan counterpart of oracle_delta_rule_chunked on the same
 * arguments (pre-normalised q, k; gates g, b), so the two can be compared
 * head-to-head: T calls of oracle_delta_rule_token. */
int oracle_delta_rule_scan(int dk, int dv, int T, const double *q, const double *k,
                           const double *v, const double *g, const double *b, double scale,
                           double *S, double *y)
{
    if (dk <= 0 || dv <= 0 || T < 0) return -1;
    for (int t = 0; t < T; ++t)
        oracle_delta_rule_token(dk, dv, S, k + (size_t)t * dk, v + (size_t)t * dv,
                                q + (size_t)t * dk, g[t], b[t], scale, y + (size_t)t * dv);
    return 0;
}
