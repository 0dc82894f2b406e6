/*
 * Mamba2 mixer core — plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check of the package entry
 * file and the CPU-baseline leg of the benchmark may build, load or call this
 * code. The CUDA library never does, and this file shares nothing with it.
 *
 * What it computes (all arithmetic in fp64, on the exact values of the bf16 or
 * fp32 inputs):
 *
 *  1. Causal depthwise conv1d over the conv channels x | B | C, kernel K with
 *     bias, as a cross-correlation whose last tap multiplies the current frame,
 *     followed by SiLU. Shape facts (conv_kernel 4, use_conv_bias true,
 *     n_groups 8, mamba_num_heads 128, mamba_head_dim 80, ssm_state_size 128)
 *     come from the issue "feat(nemotron_voicechat): load the VoiceChat
 *     checkpoint and run offline duplex inference", section config.json /
 *     text_config; the weight is one K-tap row per channel (that issue,
 *     section "Network 2": conv1d.weight is [channels, 4, 1]).
 *  2. dt = softplus(dt_raw + dt_bias), A = -exp(A_log), per head.
 *  3. The Mamba-2 selective state-space recurrence, per head h with group
 *     g = h / (H/G):
 *        h_t = exp(dt_t A) h_{t-1} + dt_t x_t (outer) B_t
 *        y_t = h_t . C_t + D x_t
 *     (the standard Mamba-2 / SSD formulation, Dao & Gu 2024, restated).
 *  4. A chunked (SSD) evaluation of the same recurrence, written
 *     independently, used only to pin chunked == sequential.
 *  5. One cached step: the per-frame update of the persistent conv tail and
 *     SSM state that the VoiceChat doc ("docs/nemotron-voicechat.md", section
 *     Offline timeline, last paragraph) says must give the same result as
 *     recomputing the full history.
 *  6. The output side of the mixer and its projections (gated RMSNorm,
 *     4-bit affine group-quantized linear layers), and one cached decode
 *     position of the hybrid model's grouped-query attention layers with
 *     their KV caches (each function below cites its passage).
 *
 * Layouts (contiguous, innermost last):
 *   x [b,T,H,P]   B, C [b,T,G,N]   dt_raw [b,T,H]   y [b,T,H,P]
 *   ssm state [b,H,P,N]   conv tail [b,K-1,CH], oldest frame first,
 *   channel c: x at c = h*P+p, B at H*P + g*N+n, C at H*P + G*N + g*N+n.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int batch, T, H, P, N, G, K;
} m2o_dims;

enum { M2O_OK = 0, M2O_EINVAL = 1, M2O_ENOMEM = 2 };

static int dims_ok(const m2o_dims* d) {
    if (!d) return 0;
    if (d->batch < 0 || d->T < 0 || d->H <= 0 || d->P <= 0 || d->N <= 0 || d->G <= 0 || d->K <= 0)
        return 0;
    if (d->H % d->G) return 0;
    return 1;
}

static long chans(const m2o_dims* d) { return (long)d->H * d->P + 2L * d->G * d->N; }

/* softplus(z) = log(1 + e^z), written so that neither branch overflows:
 * for z > 0 it is z + log(1 + e^-z). */
double m2o_softplus(double z) {
    if (z > 0.0) return z + log1p(exp(-z));
    return log1p(exp(z));
}

/* SiLU(u) = u * sigmoid(u) = u / (1 + e^-u). */
double m2o_silu(double u) { return u / (1.0 + exp(-u)); }

/* Pre-conv value of conv channel c at frame t of batch row b. Frames t < 0
 * come from the initial conv tail (slot K-1+t), or are zero without one. */
static double pre_conv(const m2o_dims* d, const double* x, const double* B, const double* C,
                       const double* init_conv, int b, int t, long c) {
    const long HP = (long)d->H * d->P, GN = (long)d->G * d->N, CH = chans(d);
    if (t < 0) {
        if (!init_conv) return 0.0;
        return init_conv[((long)b * (d->K - 1) + (d->K - 1 + t)) * CH + c];
    }
    if (c < HP) return x[((long)b * d->T + t) * HP + c];
    if (c < HP + GN) return B[((long)b * d->T + t) * GN + (c - HP)];
    return C[((long)b * d->T + t) * GN + (c - HP - GN)];
}

/* Post-conv, post-SiLU value of channel c over all frames of row b. */
static void conv_silu_channel(const m2o_dims* d, const double* x, const double* B, const double* C,
                              const double* init_conv, const double* conv_w, const double* conv_b,
                              int b, long c, double* out, long out_stride) {
    for (int t = 0; t < d->T; ++t) {
        double u = conv_b ? conv_b[c] : 0.0;
        for (int k = 0; k < d->K; ++k)
            u += conv_w[c * d->K + k] * pre_conv(d, x, B, C, init_conv, b, t - (d->K - 1) + k, c);
        out[(long)t * out_stride] = m2o_silu(u);
    }
}

/* Sequential recurrence of one head over T frames, from and into h[P][N].
 * xt[T][P], Bt[T][N], Ct[T][N], dt[T]; y[T][P]. */
static void ssm_head_sequential(int T, int P, int N, const double* xt, const double* Bt,
                                const double* Ct, const double* dt, double A, double Dh,
                                double* h, double* y) {
    for (int t = 0; t < T; ++t) {
        const double decay = exp(dt[t] * A);
        for (int p = 0; p < P; ++p) {
            const double dx = dt[t] * xt[(long)t * P + p];
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                double* hs = &h[(long)p * N + n];
                *hs = decay * (*hs) + dx * Bt[(long)t * N + n];
                acc += Ct[(long)t * N + n] * (*hs);
            }
            y[(long)t * P + p] = acc + Dh * xt[(long)t * P + p];
        }
    }
}

/* Chunked (SSD) evaluation of the same recurrence with chunk length Q; the
 * last chunk may be short. Inside a chunk with cumulative log-decay
 * S_i = sum_{s<=i} dt_s A:
 *   y_i = sum_{j<=i} (C_i . B_j) exp(S_i - S_j) dt_j x_j      (intra-chunk)
 *       + exp(S_i) C_i . h_prev                               (carried state)
 *       + D x_i
 *   h   = exp(S_last) h_prev + sum_j exp(S_last - S_j) dt_j x_j (outer) B_j   */
static int ssm_head_chunked(int T, int P, int N, int Q, const double* xt, const double* Bt,
                            const double* Ct, const double* dt, double A, double Dh, double* h,
                            double* y) {
    double* S = (double*)malloc(sizeof(double) * (size_t)(Q > 0 ? Q : 1));
    double* hnew = (double*)malloc(sizeof(double) * (size_t)P * N);
    if (!S || !hnew) { free(S); free(hnew); return M2O_ENOMEM; }
    for (int c0 = 0; c0 < T; c0 += Q) {
        const int L = (T - c0 < Q) ? (T - c0) : Q;
        double run = 0.0;
        for (int i = 0; i < L; ++i) { run += dt[c0 + i] * A; S[i] = run; }
        for (int i = 0; i < L; ++i) {
            const long ti = c0 + i;
            for (int p = 0; p < P; ++p) {
                double ydiag = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const long tj = c0 + j;
                    double cb = 0.0;
                    for (int n = 0; n < N; ++n) cb += Ct[ti * N + n] * Bt[tj * N + n];
                    ydiag += cb * exp(S[i] - S[j]) * dt[tj] * xt[tj * P + p];
                }
                double ch = 0.0;
                for (int n = 0; n < N; ++n) ch += Ct[ti * N + n] * h[(long)p * N + n];
                y[ti * P + p] = ydiag + exp(S[i]) * ch + Dh * xt[ti * P + p];
            }
        }
        const double Slast = S[L - 1];
        for (int p = 0; p < P; ++p)
            for (int n = 0; n < N; ++n) {
                double s = 0.0;
                for (int j = 0; j < L; ++j) {
                    const long tj = c0 + j;
                    s += exp(Slast - S[j]) * dt[tj] * xt[tj * P + p] * Bt[tj * N + n];
                }
                hnew[(long)p * N + n] = exp(Slast) * h[(long)p * N + n] + s;
            }
        memcpy(h, hnew, sizeof(double) * (size_t)P * N);
    }
    free(S);
    free(hnew);
    return M2O_OK;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int m2o_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* SSM core on post-conv inputs: xt [b,T,H,P], Bt/Ct [b,T,G,N], dt [b,T,H]
 * (already softplus'd), A and D [H]. h [b,H,P,N] is the initial state on
 * entry and the final state on exit; y [b,T,H,P]. Heads [h_lo, h_hi) only.
 * chunk <= 0 selects the sequential recurrence, chunk >= 1 the chunked form. */
int m2o_ssm(const m2o_dims* d, const double* xt, const double* Bt, const double* Ct,
            const double* dt, const double* A, const double* D, double* h, double* y, int h_lo,
            int h_hi, int chunk, int nthreads) {
    if (!dims_ok(d) || !xt || !Bt || !Ct || !dt || !A || !D || !h || !y) return M2O_EINVAL;
    if (h_lo < 0 || h_hi > d->H || h_lo > h_hi) return M2O_EINVAL;
    const int T = d->T, H = d->H, P = d->P, N = d->N, G = d->G, R = d->H / d->G;
    const int units = d->batch * (h_hi - h_lo);
    int err = M2O_OK;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
    for (int u = 0; u < units; ++u) {
        const int b = u / (h_hi - h_lo), hh = h_lo + u % (h_hi - h_lo), g = hh / R;
        double* xs = (double*)malloc(sizeof(double) * ((size_t)T * P + 2 * (size_t)T * N + T + (size_t)T * P + 1));
        if (!xs) { err = M2O_ENOMEM; continue; }
        double *bs = xs + (size_t)T * P, *cs = bs + (size_t)T * N, *ds = cs + (size_t)T * N, *ys = ds + T;
        for (int t = 0; t < T; ++t) {
            const long bt = (long)b * T + t;
            for (int p = 0; p < P; ++p) xs[(long)t * P + p] = xt[(bt * H + hh) * P + p];
            for (int n = 0; n < N; ++n) {
                bs[(long)t * N + n] = Bt[(bt * G + g) * N + n];
                cs[(long)t * N + n] = Ct[(bt * G + g) * N + n];
            }
            ds[t] = dt[bt * H + hh];
        }
        double* hp = h + ((long)b * H + hh) * P * N;
        int rc = M2O_OK;
        if (chunk <= 0)
            ssm_head_sequential(T, P, N, xs, bs, cs, ds, A[hh], D[hh], hp, ys);
        else
            rc = ssm_head_chunked(T, P, N, chunk, xs, bs, cs, ds, A[hh], D[hh], hp, ys);
        if (rc) err = rc;
        for (int t = 0; t < T; ++t)
            for (int p = 0; p < P; ++p)
                y[(((long)b * T + t) * H + hh) * P + p] = ys[(long)t * P + p];
        free(xs);
    }
    return err;
}

/* Post-conv, post-SiLU activations of every channel: out [b,T,CH]. */
int m2o_conv_silu(const m2o_dims* d, const double* x, const double* B, const double* C,
                  const double* conv_w, const double* conv_b, const double* init_conv,
                  double* out, int nthreads) {
    if (!dims_ok(d) || !x || !B || !C || !conv_w || !out) return M2O_EINVAL;
    const long CH = chans(d);
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (long u = 0; u < (long)d->batch * CH; ++u) {
        const int b = (int)(u / CH);
        const long c = u % CH;
        conv_silu_channel(d, x, B, C, init_conv, conv_w, conv_b, b, c,
                          out + (long)b * d->T * CH + c, CH);
    }
    return M2O_OK;
}

/* The conv tail after T frames: the last K-1 pre-conv inputs, oldest first,
 * taken from the initial tail where T < K-1. out [b,K-1,CH]. */
int m2o_conv_tail(const m2o_dims* d, const double* x, const double* B, const double* C,
                  const double* init_conv, double* out) {
    if (!dims_ok(d) || !out) return M2O_EINVAL;
    const long CH = chans(d);
    for (int b = 0; b < d->batch; ++b)
        for (int k = 0; k < d->K - 1; ++k)
            for (long c = 0; c < CH; ++c)
                out[((long)b * (d->K - 1) + k) * CH + c] =
                    pre_conv(d, x, B, C, init_conv, b, d->T - (d->K - 1) + k, c);
    return M2O_OK;
}

/* Whole mixer core over a sequence (full-history recompute / prefill).
 * Inputs are the exact fp64 values of the stored activations and parameters.
 * init_ssm [b,H,P,N] and init_conv [b,K-1,CH] may be NULL (zeros).
 * Outputs for heads [h_lo, h_hi): y [b,T,H,P] and final_ssm [b,H,P,N];
 * final_conv [b,K-1,CH] for all channels (may be NULL).
 * chunk <= 0: sequential recurrence; chunk >= 1: chunked form. */
int m2o_mixer_scan(const m2o_dims* d, const double* x, const double* B, const double* C,
                   const double* dt_raw, const double* A_log, const double* D,
                   const double* dt_bias, const double* conv_w, const double* conv_b,
                   const double* init_ssm, const double* init_conv, double* y, double* final_ssm,
                   double* final_conv, int h_lo, int h_hi, int chunk, int nthreads) {
    if (!dims_ok(d) || !x || !B || !C || !dt_raw || !A_log || !D || !dt_bias || !conv_w ||
        !conv_b || !y || !final_ssm)
        return M2O_EINVAL;
    if (h_lo < 0 || h_hi > d->H || h_lo > h_hi) return M2O_EINVAL;
    const int T = d->T, H = d->H, P = d->P, N = d->N, G = d->G, R = d->H / d->G;
    const long HP = (long)H * P, GN = (long)G * N;
    const int units = d->batch * (h_hi - h_lo);
    int err = M2O_OK;
    if (final_conv) m2o_conv_tail(d, x, B, C, init_conv, final_conv);
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
    for (int u = 0; u < units; ++u) {
        const int b = u / (h_hi - h_lo), hh = h_lo + u % (h_hi - h_lo), g = hh / R;
        double* xs = (double*)malloc(sizeof(double) * ((size_t)T * P * 2 + 2 * (size_t)T * N + T + 1));
        if (!xs) { err = M2O_ENOMEM; continue; }
        double *bs = xs + (size_t)T * P, *cs = bs + (size_t)T * N, *ds = cs + (size_t)T * N, *ys = ds + T;
        for (int p = 0; p < P; ++p)
            conv_silu_channel(d, x, B, C, init_conv, conv_w, conv_b, b, (long)hh * P + p, xs + p, P);
        for (int n = 0; n < N; ++n) {
            conv_silu_channel(d, x, B, C, init_conv, conv_w, conv_b, b, HP + (long)g * N + n, bs + n, N);
            conv_silu_channel(d, x, B, C, init_conv, conv_w, conv_b, b, HP + GN + (long)g * N + n, cs + n, N);
        }
        for (int t = 0; t < T; ++t) ds[t] = m2o_softplus(dt_raw[((long)b * T + t) * H + hh] + dt_bias[hh]);
        const double A = -exp(A_log[hh]);
        double* hp = final_ssm + ((long)b * H + hh) * P * N;
        if (init_ssm)
            memmove(hp, init_ssm + ((long)b * H + hh) * P * N, sizeof(double) * (size_t)P * N);
        else
            memset(hp, 0, sizeof(double) * (size_t)P * N);
        int rc = M2O_OK;
        if (chunk <= 0)
            ssm_head_sequential(T, P, N, xs, bs, cs, ds, A, D[hh], hp, ys);
        else
            rc = ssm_head_chunked(T, P, N, chunk, xs, bs, cs, ds, A, D[hh], hp, ys);
        if (rc) err = rc;
        for (int t = 0; t < T; ++t)
            for (int p = 0; p < P; ++p)
                y[(((long)b * T + t) * H + hh) * P + p] = ys[(long)t * P + p];
        free(xs);
    }
    return err;
}

/* One cached frame for S independent sessions that share one layer's
 * weights. x [S,H,P], B/C [S,G,N], dt_raw [S,H]: this frame's pre-conv
 * inputs. ssm [S,H,P,N] and conv [S,K-1,CH] are updated in place; y [S,H,P].
 * It is one iteration of the sequential loop of m2o_mixer_scan. */
int m2o_mixer_step(const m2o_dims* d, int S, const double* x, const double* B, const double* C,
                   const double* dt_raw, const double* A_log, const double* D,
                   const double* dt_bias, const double* conv_w, const double* conv_b,
                   double* ssm, double* conv, double* y, int nthreads) {
    if (!dims_ok(d) || S < 0 || !x || !B || !C || !dt_raw || !A_log || !D || !dt_bias || !conv_w ||
        !conv_b || !ssm || !conv || !y)
        return M2O_EINVAL;
    m2o_dims one = *d;
    one.batch = 1;
    one.T = 1;
    const long CH = chans(d), HP = (long)d->H * d->P, GN = (long)d->G * d->N;
    const long PN = (long)d->P * d->N;
    int err = M2O_OK;
    for (int s = 0; s < S; ++s) {
        double* tail = conv + (long)s * (d->K - 1) * CH;
        double* hs = ssm + (long)s * d->H * PN;
        double* ys = y + (long)s * HP;
        double* newtail = (double*)malloc(sizeof(double) * (size_t)(d->K - 1) * CH);
        if (!newtail) return M2O_ENOMEM;
        int rc = m2o_mixer_scan(&one, x + (long)s * HP, B + (long)s * GN, C + (long)s * GN,
                                dt_raw + (long)s * d->H, A_log, D, dt_bias, conv_w, conv_b, hs, tail,
                                ys, hs, newtail, 0, d->H, 0, nthreads);
        if (rc) err = rc;
        memcpy(tail, newtail, sizeof(double) * (size_t)(d->K - 1) * CH);
        free(newtail);
    }
    return err;
}

/* Gated RMSNorm of the mixer output (the standard Mamba-2 output norm; the
 * VoiceChat issue, section config.json / text_config, gives rms_norm_eps
 * 1e-5). For each of `rows` positions and each of `groups` contiguous blocks
 * of width/groups channels:
 *     v   = y * silu(z)
 *     out = weight * v / sqrt(mean over the block of v^2 + eps)
 * y, z, out [rows, width]; weight [width]. */
int m2o_gated_norm(int rows, int width, int groups, const double* y, const double* z,
                   const double* weight, double eps, double* out) {
    if (rows < 0 || width <= 0 || groups <= 0 || width % groups != 0 || !y || !z || !weight || !out ||
        !(eps >= 0.0))
        return M2O_EINVAL;
    const int gw = width / groups;
    double* v = (double*)malloc(sizeof(double) * (size_t)gw);
    if (!v) return M2O_ENOMEM;
    for (long r = 0; r < rows; ++r) {
        for (int g = 0; g < groups; ++g) {
            const long base = r * width + (long)g * gw;
            double ss = 0.0;
            for (int k = 0; k < gw; ++k) {
                v[k] = y[base + k] * m2o_silu(z[base + k]);
                ss += v[k] * v[k];
            }
            const double inv = 1.0 / sqrt(ss / gw + eps);
            for (int k = 0; k < gw; ++k) out[base + k] = weight[(long)g * gw + k] * v[k] * inv;
        }
    }
    free(v);
    return M2O_OK;
}

/* Affine group-quantized linear layer: the mixer's input and output
 * projections, which the VoiceChat 4-bit checkpoint stores quantized with
 * group_size 64 and bits 4 (Nemotron VoiceChat page, config.json,
 * `quantization`). Weight element (o, i) is the 4-bit field q = bits
 * 4*(i%8) .. 4*(i%8)+3 of the 32-bit word wq[o][i/8] (the first element in
 * the lowest bits), dequantized per group of `group` consecutive inputs:
 *     W[o][i] = scale[o][i/group] * q + bias[o][i/group]
 *     y[r][o] = sum_i W[o][i] x[r][i]
 * x [rows, in]; y [rows, out]; scale, bias [out, in/group]. */
int m2o_qlinear(int rows, int in, int out, int group, const uint32_t* wq, const double* scale,
                const double* bias, const double* x, double* y) {
    if (rows < 0 || in <= 0 || out <= 0 || group <= 0 || in % group != 0 || in % 8 != 0 || !wq || !scale ||
        !bias || !x || !y)
        return M2O_EINVAL;
    const int ngroups = in / group;
    for (long r = 0; r < rows; ++r)
        for (int o = 0; o < out; ++o) y[r * out + o] = 0.0;
    /* outputs are independent: split them over threads (each y[.][o] is
     * summed by one thread, in input order) */
#pragma omp parallel for schedule(static)
    for (int o = 0; o < out; ++o) {
        for (int i = 0; i < in; ++i) {
            const uint32_t word = wq[(long)o * (in / 8) + i / 8];
            const int q = (int)((word >> (4 * (i % 8))) & 15u);
            const double w = scale[(long)o * ngroups + i / group] * q + bias[(long)o * ngroups + i / group];
            for (long r = 0; r < rows; ++r) y[r * out + o] += w * x[r * in + i];
        }
    }
    return M2O_OK;
}

/* One cached decode position of a grouped-query attention layer of the same
 * hybrid model: the Nemotron-H attention layers (num_attention_heads 40,
 * num_key_value_heads 8, head_dim 128, attention_bias false; the
 * configuration lists no positional rotation for them; VoiceChat issue,
 * section config.json / text_config, hybrid_override_pattern `*` layers),
 * whose KV caches a session keeps across positions ("docs/nemotron-voicechat.md",
 * section Online session, persistent-state table). For session s with
 * len[s] positions already cached:
 *   - each kv head's new key and value go to position len[s];
 *   - query head h reads kv head g = h / (Hq/Hkv), over positions
 *     t = 0 .. len[s] (the new position included):
 *       a_t = scale * sum_d q[h][d] k[g][t][d]
 *       w_t = exp(a_t - max_u a_u) / sum_u exp(a_u - max_u a_u)
 *       out[h] = sum_t w_t v[g][t]
 * q, out [S,Hq,D]; k_new, v_new [S,Hkv,D]; k_cache, v_cache [S,Hkv,Tmax,D].
 * Positions past len[s] are neither read nor written. A len[s] outside
 * [0, Tmax) is an error (nothing is written). */
int m2o_attn_decode(int S, int Hq, int Hkv, int D, int Tmax, const int* len, const double* q,
                    const double* k_new, const double* v_new, double* k_cache, double* v_cache,
                    double scale, double* out) {
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Tmax <= 0 || Hq % Hkv != 0 || !len || !q || !k_new ||
        !v_new || !k_cache || !v_cache || !out)
        return M2O_EINVAL;
    for (int s = 0; s < S; ++s)
        if (len[s] < 0 || len[s] >= Tmax) return M2O_EINVAL;
    const int R = Hq / Hkv;
    double* a = (double*)malloc(sizeof(double) * (size_t)Tmax);
    if (!a) return M2O_ENOMEM;
    for (int s = 0; s < S; ++s) {
        const int L = len[s];
        for (int g = 0; g < Hkv; ++g) {
            const long kv = ((long)s * Hkv + g) * Tmax;
            for (int d = 0; d < D; ++d) {
                k_cache[(kv + L) * D + d] = k_new[((long)s * Hkv + g) * D + d];
                v_cache[(kv + L) * D + d] = v_new[((long)s * Hkv + g) * D + d];
            }
            for (int r = 0; r < R; ++r) {
                const int h = g * R + r;
                const double* qh = q + ((long)s * Hq + h) * D;
                double amax = -INFINITY;
                for (int t = 0; t <= L; ++t) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qh[d] * k_cache[(kv + t) * D + d];
                    a[t] = scale * dot;
                    if (a[t] > amax) amax = a[t];
                }
                double den = 0.0;
                for (int t = 0; t <= L; ++t) {
                    a[t] = exp(a[t] - amax);
                    den += a[t];
                }
                double* oh = out + ((long)s * Hq + h) * D;
                for (int d = 0; d < D; ++d) {
                    double num = 0.0;
                    for (int t = 0; t <= L; ++t) num += a[t] * v_cache[(kv + t) * D + d];
                    oh[d] = num / den;
                }
            }
        }
    }
    free(a);
    return M2O_OK;
}

/* RMSNorm of each row, the pre-norm of every block of the hybrid model
 * (VoiceChat issue, section config.json / text_config: layer_norm_epsilon
 * 1e-5):
 *     out = weight * x / sqrt(mean over the row of x^2 + eps)
 * x, out [rows, width]; weight [width]. */
int m2o_rmsnorm(int rows, int width, const double* x, const double* weight, double eps, double* out) {
    if (rows < 0 || width <= 0 || !x || !weight || !out || !(eps >= 0.0)) return M2O_EINVAL;
    for (long r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int k = 0; k < width; ++k) ss += x[r * width + k] * x[r * width + k];
        const double inv = 1.0 / sqrt(ss / width + eps);
        for (int k = 0; k < width; ++k) out[r * width + k] = weight[k] * x[r * width + k] * inv;
    }
    return M2O_OK;
}
