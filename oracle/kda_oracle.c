/*
 * KDA oracle: a plain, slow, double-precision CPU statement of what the
 * Kimi Delta Attention decode step and the KDA recurrence compute.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the bench's CPU-baseline leg
 * use it. It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [DD]  "GLM-5.3 deep dive" (gangliao.me), section 8.2:
 *           8.2.2 the delta rule and its worked example,
 *           8.2.3 Eq. 1 (the KDA update) and the per-channel gate,
 *           8.2.4 the full KDA layer (short conv + SiLU on q, k, v),
 *           8.2.6 decoding in four steps (fade, predict, correct, read) and
 *                 the implementation note on L2 normalisation (eps 1e-6).
 *   [P1]  "At the 262k cap the DSA indexer costs 12x the sparse MLA it
 *           selects for", section "Geometry" (conv kernel 4, 3 taps,
 *           weight [8192, 1, 4]) and "KDA decode step".
 *
 * Layouts (row-major, C order):
 *   conv input  x      [M][3][D]      tensors in the order q, k, v; D = H*d
 *   conv weight w      [3][D][4]      w[..][3] multiplies the current token
 *   conv cache  cache  [M][3][3][D]   tap 0 is the oldest input
 *   q, k               [M][T][H][dk]
 *   v                  [M][T][H][dv]
 *   alpha              [M][T][H][dk]  linear-space decay, one per key channel
 *   beta               [M][T][H]      one write strength per head
 *   S                  [M][H][dk][dv] S[i][j]: key channel i, value channel j
 *   o                  [M][T][H][dv]
 *
 * Readings where the pages leave a step open (each one is listed in the
 * design notes):
 *   - the conv is causal with no bias: y = w0*x[t-3] + w1*x[t-2] + w2*x[t-1]
 *     + w3*x[t], followed by SiLU, on all three of q, k and v;
 *   - L2 normalisation is x / sqrt(sum x^2 + eps), eps inside the root;
 *   - the readout uses the state after this token's update (Eq. 1), scaled by
 *     the caller's `scale` (1.0 reproduces Eq. 1; fla uses 1/sqrt(dk)).
 *
 * Parity pins: every function here is pinned by tests that do not reuse its
 * code (worked example, brute-force dense product, invariants, direct
 * convolution, chunked form).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* y = x * sigmoid(x) */
static double silu(double x) { return x / (1.0 + exp(-x)); }

/*
 * Short convolution + SiLU for one token ([P1] Geometry: depthwise, kernel 4,
 * 3 cached taps; [DD] 8.2.4 step 2). Updates the cache in place so that it
 * holds the three most recent inputs, oldest first.
 */
void kda_oracle_conv_step(const double *x, const double *w, double *cache,
                          double *y, int M, int D)
{
    for (int m = 0; m < M; ++m) {
        for (int X = 0; X < 3; ++X) {
            const double *xt = x + ((size_t)m * 3 + X) * D;
            double *c0 = cache + (((size_t)m * 3 + X) * 3 + 0) * D;
            double *c1 = cache + (((size_t)m * 3 + X) * 3 + 1) * D;
            double *c2 = cache + (((size_t)m * 3 + X) * 3 + 2) * D;
            double *yt = y + ((size_t)m * 3 + X) * D;
            for (int c = 0; c < D; ++c) {
                const double *wc = w + ((size_t)X * D + c) * 4;
                double pre = wc[0] * c0[c] + wc[1] * c1[c] + wc[2] * c2[c]
                           + wc[3] * xt[c];
                yt[c] = silu(pre);
                c0[c] = c1[c];
                c1[c] = c2[c];
                c2[c] = xt[c];
            }
        }
    }
}

/*
 * The KDA recurrence over T tokens ([DD] 8.2.3 Eq. 1, in the four-step order
 * of [DD] 8.2.6), one (stream, head) at a time:
 *   normalise q and k (if use_l2norm),
 *   fade:    S[i][j] *= alpha[i]
 *   predict: u[j] = sum_i k[i] S[i][j]
 *   correct: S[i][j] += k[i] * beta * (v[j] - u[j])
 *   read:    o[j] = scale * sum_i q[i] S[i][j]
 * S is read and updated in place.
 */
void kda_oracle_recurrent(const double *q, const double *k, const double *v,
                          const double *alpha, const double *beta,
                          double *S, double *o,
                          int M, int T, int H, int dk, int dv,
                          double scale, int use_l2norm, double eps)
{
    double *qn = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kn = (double *)malloc(sizeof(double) * (size_t)dk);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    for (int m = 0; m < M; ++m) {
        for (int h = 0; h < H; ++h) {
            double *Sh = S + ((size_t)m * H + h) * dk * dv;
            for (int t = 0; t < T; ++t) {
                size_t tk = (((size_t)m * T + t) * H + h) * dk;
                size_t tv = (((size_t)m * T + t) * H + h) * dv;
                double b = beta[((size_t)m * T + t) * H + h];
                const double *a = alpha + tk;
                /* normalise q and k ([DD] 8.2.6 implementation notes) */
                double sq = 0.0, sk = 0.0;
                for (int i = 0; i < dk; ++i) {
                    sq += q[tk + i] * q[tk + i];
                    sk += k[tk + i] * k[tk + i];
                }
                double rq = use_l2norm ? 1.0 / sqrt(sq + eps) : 1.0;
                double rk = use_l2norm ? 1.0 / sqrt(sk + eps) : 1.0;
                for (int i = 0; i < dk; ++i) {
                    qn[i] = q[tk + i] * rq;
                    kn[i] = k[tk + i] * rk;
                }
                /* 1. fade each key row by its own decay */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        Sh[(size_t)i * dv + j] *= a[i];
                /* 2. predict what the faded memory returns for k */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i)
                        acc += kn[i] * Sh[(size_t)i * dv + j];
                    u[j] = acc;
                }
                /* 3. correct: write beta * k (v - u)^T */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        Sh[(size_t)i * dv + j] += kn[i] * b * (v[tv + j] - u[j]);
                /* 4. read with q from the updated state */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i)
                        acc += qn[i] * Sh[(size_t)i * dv + j];
                    o[tv + j] = scale * acc;
                }
            }
        }
    }
    free(qn);
    free(kn);
    free(u);
}

/*
 * One full decode step of a KDA layer for M streams: short conv + SiLU on the
 * pre-conv q, k, v ([DD] 8.2.4 step 2), then the recurrence above with L2
 * normalisation of q and k ([DD] 8.2.4 step 6). Requires dk == dv == d with
 * D = H * d. Updates cache and S in place and writes o [M][H][d].
 */
void kda_oracle_decode_step(const double *x, const double *w, double *cache,
                            const double *alpha, const double *beta,
                            double *S, double *o, int M, int H, int d,
                            double scale, double eps)
{
    size_t D = (size_t)H * d;
    double *y = (double *)malloc(sizeof(double) * (size_t)M * 3 * D);
    double *qkv = (double *)malloc(sizeof(double) * (size_t)M * 3 * D);
    kda_oracle_conv_step(x, w, cache, y, M, (int)D);
    /* regroup y [M][3][D] into three [M][1][H][d] arrays */
    for (int X = 0; X < 3; ++X)
        for (int m = 0; m < M; ++m)
            memcpy(qkv + ((size_t)X * M + m) * D, y + ((size_t)m * 3 + X) * D,
                   sizeof(double) * D);
    kda_oracle_recurrent(qkv, qkv + (size_t)M * D, qkv + 2 * (size_t)M * D,
                         alpha, beta, S, o, M, 1, H, d, d, scale, 1, eps);
    free(y);
    free(qkv);
}

/*
 * KDA forget gate ([DD] 8.2.3, "The gate in GLM-5.3-Flash, as fla computes
 * it"): per stream m, head h and key channel c,
 *     g = lb * sigmoid(exp(A_h) * (f + b_{h,c})),   alpha = exp(g),
 * with lb the gate's lower bound (-5 in GLM-5.3-Flash).
 *   f [M][H][dk], A_log [H], dt_bias [H*dk] -> alpha [M][H][dk]
 */
void kda_oracle_forget_gate(const double *f, const double *A_log, const double *dt_bias,
                            double lb, double *alpha, int M, int H, int dk)
{
    for (int m = 0; m < M; ++m)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < dk; ++c) {
                size_t i = ((size_t)m * H + h) * dk + c;
                double z = exp(A_log[h]) * (f[i] + dt_bias[(size_t)h * dk + c]);
                double g = lb / (1.0 + exp(-z));
                alpha[i] = exp(g);
            }
}

/*
 * Gated RMSNorm of one head's output ([DD] 8.2.4 step 7 and its notes:
 * RMSNorm over the head's dv channels, eps 1e-5, times a sigmoid output gate):
 *     y_j = o_j / sqrt(mean_j(o^2) + eps) * w_j * sigmoid(gate_j)
 *   o, gate [M][H][dv], w [dv] -> y [M][H][dv]
 */
void kda_oracle_gated_rmsnorm(const double *o, const double *gate, const double *w, double eps,
                              double *y, int M, int H, int dv)
{
    for (int m = 0; m < M; ++m)
        for (int h = 0; h < H; ++h) {
            const double *oh = o + ((size_t)m * H + h) * dv;
            const double *gh = gate + ((size_t)m * H + h) * dv;
            double *yh = y + ((size_t)m * H + h) * dv;
            double ss = 0.0;
            for (int j = 0; j < dv; ++j) ss += oh[j] * oh[j];
            double r = 1.0 / sqrt(ss / dv + eps);
            for (int j = 0; j < dv; ++j) yh[j] = oh[j] * r * w[j] / (1.0 + exp(-gh[j]));
        }
}
