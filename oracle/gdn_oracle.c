/*
 * Oracle for the Gated DeltaNet (GDN) causal core -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU code that states what the GDN core computes, one stage
 * per function, so that a reader can check each against its definition by eye.
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
 * load this library; the product path (the CUDA library) never does, and the two
 * share no code.
 *
 * Sources (pages, by title and section):
 *   [P1] "[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the head-sharded
 *        layer" (radixark/miles #3610): "What" (group-major q/k/v, GVA),
 *        "Summary of an earlier run" (fla grouped-value accumulation).
 *   [P2] prime-rl #3860 "Summary" / "Behavior change" (ZeroCenteredRMSNorm,
 *        causal_conv1d with cu_seqlens, initial_state=None /
 *        output_final_state=False defaults), "What I ran" (pure-torch
 *        reference conv / gated delta rule / gated norm).
 *   [P3] "[main] feat(moe): Support gated delta net for Qwen3-Next (1/4)"
 *        (NVIDIA/Megatron-LM #1989): "GDN args" (conv kernel 4, head dims 128,
 *        16 k-heads / 32 v-heads), "--apply-layernorm-1p" (zero-centred norm),
 *        review comment on A_log (A_log stores log A; the layer uses exp(A_log)).
 *
 * The GDN core, as implemented here (the pages name the stages; the equations
 * are the standard gated delta rule they refer to):
 *   conv:   pre[t,c] = sum_{j<K} w[c,j] * x[t-(K-1)+j, c]  (zero, or the conv
 *           cache, before the sequence start);  xc = silu(pre)
 *   l2:     q^ = q / sqrt(|q|^2 + eps) * d_k^-1/2 ;  k^ = k / sqrt(|k|^2 + eps)
 *   gates:  g = -exp(A_log[h]) * softplus(a + dt_bias[h]) ;  beta = sigmoid(b)
 *   rule:   S_t = exp(g_t) S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T
 *           o_t = S_t q^_t          (S is [d_v x d_k]; fp64 here)
 *   norm:   y = o / sqrt(mean(o^2) + eps) * (1 + w) * gate(z), gate = silu
 *           or sigmoid
 * v-head h reads the q^/k^ of k-head floor(h / (H_v/H_k)).
 *
 * Pins (tests/test_oracle_*.py): the token recurrence against the naive chunked
 * WY form below; the delta-rule memory invariant (g=0, beta=1, orthonormal keys
 * => S k_i = v_i); pure decay (beta=0 => S_T = S_0 prod exp(g)); central finite
 * differences of every backward function; the conv against a library grouped
 * convolution; the norm against a library RMS norm; gates against library
 * softplus / sigmoid; T=1 closed form; varlen = separate runs; split with
 * state + conv-cache handoff = one run.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }
/* softplus(x) = log(1 + e^x); for x > 20 the two differ by < 1e-9 relative and
 * the linear branch avoids overflow (same threshold as torch's softplus). */
static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }
static double silu(double x) { return x * sigm(x); }
/* d/dx silu(x) = s (1 + x (1 - s)), s = sigmoid(x) */
static double dsilu(double x) { double s = sigm(x); return s * (1.0 + x * (1.0 - s)); }

int gdn_ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Causal depthwise conv1d + SiLU, with cu_seqlens resets and a conv cache.  */
/* [P2] "Summary" (causal_conv1d called with cu_seqlens); [P3] "GDN args"    */
/* (--linear-conv-kernel-dim 4).                                             */
/*   x   [T, C]          w [C, K]                                            */
/*   cs_in / cs_out [N, C, K-1]: the K-1 inputs that precede the sequence    */
/*   (cs[..., m] is position start-(K-1)+m); NULL = zeros / not wanted.      */
/*   pre [T, C] (nullable) conv output before SiLU; out [T, C] after SiLU.   */
/* ------------------------------------------------------------------------ */
static double conv_input(const double *x, const double *cs_in, int64_t tau, int64_t s,
                         int n, int C, int K, int c)
{
    if (tau >= s) return x[tau * C + c];
    if (!cs_in) return 0.0;
    int64_t m = (K - 1) + (tau - s); /* 0..K-2 */
    if (m < 0) return 0.0;
    return cs_in[((int64_t)n * C + c) * (K - 1) + m];
}

void gdn_ref_conv_silu(int N, const int32_t *cu, int C, int K, const double *x,
                       const double *w, const double *cs_in, double *pre, double *out,
                       double *cs_out)
{
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        for (int n = 0; n < N; n++) {
            int64_t s = cu[n], e = cu[n + 1];
            for (int64_t t = s; t < e; t++) {
                double acc = 0.0;
                for (int j = 0; j < K; j++)
                    acc += w[c * K + j] * conv_input(x, cs_in, t - (K - 1) + j, s, n, C, K, c);
                if (pre) pre[t * C + c] = acc;
                out[t * C + c] = silu(acc);
            }
            if (cs_out)
                for (int m = 0; m < K - 1; m++)
                    cs_out[((int64_t)n * C + c) * (K - 1) + m] =
                        conv_input(x, cs_in, e - (K - 1) + m, s, n, C, K, c);
        }
    }
}

/* Backward of conv + SiLU. dout [T, C] is the gradient of the SiLU output.
 * dx [T, C]; dw [C, K]; dcs_in [N, C, K-1] (nullable). The conv cache output
 * is not differentiated. */
void gdn_ref_conv_silu_bwd(int N, const int32_t *cu, int C, int K, const double *x,
                           const double *w, const double *cs_in, const double *dout,
                           double *dx, double *dw, double *dcs_in)
{
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        for (int j = 0; j < K; j++) dw[c * K + j] = 0.0;
        for (int n = 0; n < N; n++) {
            int64_t s = cu[n], e = cu[n + 1];
            /* dpre[t] = dout[t] * silu'(pre[t]) ; recompute pre */
            for (int64_t t = s; t < e; t++) dx[t * C + c] = 0.0;
            if (dcs_in)
                for (int m = 0; m < K - 1; m++) dcs_in[((int64_t)n * C + c) * (K - 1) + m] = 0.0;
            for (int64_t t = s; t < e; t++) {
                double acc = 0.0;
                for (int j = 0; j < K; j++)
                    acc += w[c * K + j] * conv_input(x, cs_in, t - (K - 1) + j, s, n, C, K, c);
                double dpre = dout[t * C + c] * dsilu(acc);
                for (int j = 0; j < K; j++) {
                    int64_t tau = t - (K - 1) + j;
                    dw[c * K + j] += dpre * conv_input(x, cs_in, tau, s, n, C, K, c);
                    if (tau >= s)
                        dx[tau * C + c] += dpre * w[c * K + j];
                    else if (dcs_in && (K - 1) + (tau - s) >= 0)
                        dcs_in[((int64_t)n * C + c) * (K - 1) + (K - 1) + (tau - s)] +=
                            dpre * w[c * K + j];
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* L2 normalisation of one head vector: u = x / sqrt(|x|^2 + eps) * scale.   */
/* Applied per (token, k-head) to q (scale d_k^-1/2) and k (scale 1).         */
/*   x, out: [rows, d] contiguous rows.                                       */
/* ------------------------------------------------------------------------ */
void gdn_ref_l2norm(int64_t rows, int d, double eps, double scale, const double *x, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        double ss = 0.0;
        for (int i = 0; i < d; i++) ss += x[r * d + i] * x[r * d + i];
        double inv = 1.0 / sqrt(ss + eps);
        for (int i = 0; i < d; i++) out[r * d + i] = x[r * d + i] * inv * scale;
    }
}

/* Backward: dx = scale * r * (du - u (u . du)), u = x r, r = 1/sqrt(|x|^2+eps),
 * where du is the gradient of the scaled output. */
void gdn_ref_l2norm_bwd(int64_t rows, int d, double eps, double scale, const double *x,
                        const double *dout, double *dx)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        double ss = 0.0;
        for (int i = 0; i < d; i++) ss += x[r * d + i] * x[r * d + i];
        double inv = 1.0 / sqrt(ss + eps);
        double dot = 0.0;
        for (int i = 0; i < d; i++) dot += x[r * d + i] * inv * dout[r * d + i] * scale;
        for (int i = 0; i < d; i++)
            dx[r * d + i] = inv * (dout[r * d + i] * scale - x[r * d + i] * inv * dot);
    }
}

/* ------------------------------------------------------------------------ */
/* Gates. [P3] review comment on A_log: A_log holds log A; the decay rate is   */
/* exp(A_log).  g = -exp(A_log[h]) softplus(a + dt_bias[h]); beta = sigmoid(b)*/
/*   a, b, g, beta: [T, H]                                                    */
/* ------------------------------------------------------------------------ */
void gdn_ref_gates(int64_t T, int H, const double *a, const double *b, const double *A_log,
                   const double *dt_bias, double *g, double *beta)
{
    for (int64_t t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            g[t * H + h] = -exp(A_log[h]) * softplus(a[t * H + h] + dt_bias[h]);
            beta[t * H + h] = sigm(b[t * H + h]);
        }
}

/* dg/da = -exp(A_log) sigmoid(a + dt_bias); dg/dA_log = g; dbeta/db = beta (1-beta) */
void gdn_ref_gates_bwd(int64_t T, int H, const double *a, const double *b, const double *A_log,
                       const double *dt_bias, const double *dg, const double *dbeta, double *da,
                       double *db, double *dA_log, double *ddt_bias)
{
    for (int h = 0; h < H; h++) { dA_log[h] = 0.0; ddt_bias[h] = 0.0; }
    for (int64_t t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            double xa = a[t * H + h] + dt_bias[h];
            double gv = -exp(A_log[h]) * softplus(xa);
            double dadv = dg[t * H + h] * (-exp(A_log[h])) * sigm(xa);
            da[t * H + h] = dadv;
            ddt_bias[h] += dadv;
            dA_log[h] += dg[t * H + h] * gv;
            double bb = sigm(b[t * H + h]);
            db[t * H + h] = dbeta[t * H + h] * bb * (1.0 - bb);
        }
}

/* ------------------------------------------------------------------------ */
/* Gated delta rule, token by token.                                          */
/*   S' = exp(g_t) S ;  r = S' k ;  S = S' + beta (v - r) k^T ;  o = S q      */
/* which equals S_t = exp(g_t) S_{t-1} (I - beta k k^T) + beta v k^T.          */
/* GVA ([P1] "What", "Summary of an earlier run"): v-head h reads k-head      */
/* h / (hv/hk); q and k are never repeated.                                   */
/*   qh, kh [T, hk, dk]; v [T, hv, dv]; g, beta [T, hv];                      */
/*   S0 [N, hv, dv, dk] (NULL = zeros, [P2] initial_state=None);              */
/*   head_mask [hv] (NULL = all heads); o [T, hv, dv]; S_fin [N, hv, dv, dk]   */
/*   (NULL = not wanted, [P2] output_final_state=False).                      */
/* ------------------------------------------------------------------------ */
static void rule_step(double *S, int dv, int dk, double gt, double bt, const double *k,
                      const double *v)
{
    double dec = exp(gt);
    for (int i = 0; i < dv * dk; i++) S[i] *= dec;
    for (int a = 0; a < dv; a++) {
        double r = 0.0;
        for (int b = 0; b < dk; b++) r += S[a * dk + b] * k[b];
        double delta = bt * (v[a] - r);
        for (int b = 0; b < dk; b++) S[a * dk + b] += delta * k[b];
    }
}

void gdn_ref_delta_rule_fwd(int N, const int32_t *cu, int hk, int hv, int dk, int dv,
                            const double *qh, const double *kh, const double *v,
                            const double *g, const double *beta, const double *S0,
                            const uint8_t *head_mask, double *o, double *S_fin)
{
    int G = hv / hk;
    size_t sz = (size_t)dv * dk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < N * hv; p++) {
        int n = p / hv, h = p % hv;
        if (head_mask && !head_mask[h]) continue;
        double *S = (double *)malloc(sz * sizeof(double));
        if (S0) memcpy(S, S0 + (size_t)p * sz, sz * sizeof(double));
        else memset(S, 0, sz * sizeof(double));
        for (int64_t t = cu[n]; t < cu[n + 1]; t++) {
            const double *k = kh + (t * hk + h / G) * dk;
            const double *q = qh + (t * hk + h / G) * dk;
            rule_step(S, dv, dk, g[t * hv + h], beta[t * hv + h], k, v + (t * hv + h) * dv);
            for (int a = 0; a < dv; a++) {
                double acc = 0.0;
                for (int b = 0; b < dk; b++) acc += S[a * dk + b] * q[b];
                o[(t * hv + h) * dv + a] = acc;
            }
        }
        if (S_fin) memcpy(S_fin + (size_t)p * sz, S, sz * sizeof(double));
        free(S);
    }
}

/* Reverse mode through the same loop. The state before each step is
 * recomputed from checkpoints taken every SEG tokens (recomputation repeats
 * the forward arithmetic exactly, so the values are the forward's).
 * Adjoints for one step, with dS the gradient of S_t:
 *   dS += do q^T ; dq = S^T do
 *   dd = dS k ; dk = dS^T d  (d = beta (v - r)) ; dv = beta dd ; dbeta = (v-r).dd
 *   dr = -beta dd ; dS' = dS + dr k^T ; dk += S'^T dr
 *   dg = <dS', S'> ; dS_{t-1} = exp(g) dS'
 * dq_v / dk_v are per v-head [T, hv, dk]; the caller sums them over the v-heads
 * that share a k-head. dS_fin (nullable) is the gradient of the final state;
 * dS0 (nullable) receives the gradient of S0. */
#define GDN_REF_SEG 128
void gdn_ref_delta_rule_bwd(int N, const int32_t *cu, int hk, int hv, int dk, int dv,
                            const double *qh, const double *kh, const double *v,
                            const double *g, const double *beta, const double *S0,
                            const double *do_, const double *dS_fin, const uint8_t *head_mask,
                            double *dq_v, double *dk_v, double *dv_, double *dg,
                            double *dbeta, double *dS0)
{
    int G = hv / hk;
    size_t sz = (size_t)dv * dk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < N * hv; p++) {
        int n = p / hv, h = p % hv;
        if (head_mask && !head_mask[h]) continue;
        int64_t s = cu[n], e = cu[n + 1], L = e - s;
        int64_t nseg = (L + GDN_REF_SEG - 1) / GDN_REF_SEG;
        double *ck = (double *)malloc((size_t)(nseg > 0 ? nseg : 1) * sz * sizeof(double));
        double *Sb = (double *)malloc((size_t)GDN_REF_SEG * sz * sizeof(double));
        double *S = (double *)malloc(sz * sizeof(double));
        double *Sp = (double *)malloc(sz * sizeof(double));
        double *dS = (double *)malloc(sz * sizeof(double));
        double *r = (double *)malloc(dv * sizeof(double));
        double *dd = (double *)malloc(dv * sizeof(double));
        if (S0) memcpy(S, S0 + (size_t)p * sz, sz * sizeof(double));
        else memset(S, 0, sz * sizeof(double));
        for (int64_t sg = 0; sg < nseg; sg++) {
            memcpy(ck + sg * sz, S, sz * sizeof(double));
            int64_t t1 = s + (sg + 1) * GDN_REF_SEG < e ? s + (sg + 1) * GDN_REF_SEG : e;
            for (int64_t t = s + sg * GDN_REF_SEG; t < t1; t++)
                rule_step(S, dv, dk, g[t * hv + h], beta[t * hv + h], kh + (t * hk + h / G) * dk,
                          v + (t * hv + h) * dv);
        }
        if (dS_fin) memcpy(dS, dS_fin + (size_t)p * sz, sz * sizeof(double));
        else memset(dS, 0, sz * sizeof(double));
        for (int64_t sg = nseg - 1; sg >= 0; sg--) {
            int64_t t0 = s + sg * GDN_REF_SEG;
            int64_t t1 = t0 + GDN_REF_SEG < e ? t0 + GDN_REF_SEG : e;
            memcpy(S, ck + sg * sz, sz * sizeof(double));
            for (int64_t t = t0; t < t1; t++) {
                memcpy(Sb + (t - t0) * sz, S, sz * sizeof(double));
                rule_step(S, dv, dk, g[t * hv + h], beta[t * hv + h], kh + (t * hk + h / G) * dk,
                          v + (t * hv + h) * dv);
            }
            for (int64_t t = t1 - 1; t >= t0; t--) {
                const double *k = kh + (t * hk + h / G) * dk;
                const double *q = qh + (t * hk + h / G) * dk;
                const double *vt = v + (t * hv + h) * dv;
                const double *dot = do_ + (t * hv + h) * dv;
                double gt = g[t * hv + h], bt = beta[t * hv + h], dec = exp(gt);
                double *dqt = dq_v + (t * hv + h) * dk;
                double *dkt = dk_v + (t * hv + h) * dk;
                /* recompute S' , r, S for this step */
                for (size_t i = 0; i < sz; i++) Sp[i] = dec * Sb[(t - t0) * sz + i];
                for (int a = 0; a < dv; a++) {
                    double acc = 0.0;
                    for (int b = 0; b < dk; b++) acc += Sp[a * dk + b] * k[b];
                    r[a] = acc;
                }
                for (int a = 0; a < dv; a++)
                    for (int b = 0; b < dk; b++)
                        S[a * dk + b] = Sp[a * dk + b] + bt * (vt[a] - r[a]) * k[b];
                /* o = S q */
                for (int a = 0; a < dv; a++)
                    for (int b = 0; b < dk; b++) dS[a * dk + b] += dot[a] * q[b];
                for (int b = 0; b < dk; b++) {
                    double acc = 0.0;
                    for (int a = 0; a < dv; a++) acc += S[a * dk + b] * dot[a];
                    dqt[b] = acc;
                }
                /* S = S' + d k^T */
                double dbt = 0.0;
                for (int a = 0; a < dv; a++) {
                    double acc = 0.0;
                    for (int b = 0; b < dk; b++) acc += dS[a * dk + b] * k[b];
                    dd[a] = acc;
                }
                for (int b = 0; b < dk; b++) {
                    double acc = 0.0;
                    for (int a = 0; a < dv; a++) acc += dS[a * dk + b] * bt * (vt[a] - r[a]);
                    dkt[b] = acc;
                }
                for (int a = 0; a < dv; a++) {
                    dv_[(t * hv + h) * dv + a] = bt * dd[a];
                    dbt += (vt[a] - r[a]) * dd[a];
                }
                /* r = S' k : dr = -beta dd */
                for (int a = 0; a < dv; a++)
                    for (int b = 0; b < dk; b++) dS[a * dk + b] += -bt * dd[a] * k[b];
                for (int b = 0; b < dk; b++) {
                    double acc = 0.0;
                    for (int a = 0; a < dv; a++) acc += Sp[a * dk + b] * (-bt * dd[a]);
                    dkt[b] += acc;
                }
                /* S' = exp(g) S_prev */
                double dgt = 0.0;
                for (size_t i = 0; i < sz; i++) dgt += dS[i] * Sp[i];
                for (size_t i = 0; i < sz; i++) dS[i] *= dec;
                dg[t * hv + h] = dgt;
                dbeta[t * hv + h] = dbt;
            }
        }
        if (dS0) memcpy(dS0 + (size_t)p * sz, dS, sz * sizeof(double));
        free(ck); free(Sb); free(S); free(Sp); free(dS); free(r); free(dd);
    }
}

/* ------------------------------------------------------------------------ */
/* Naive chunked (WY) form of the same rule -- a second, independent way to  */
/* compute it, used only to pin the token recurrence.  Per chunk of c tokens */
/* with in-chunk cumulative gate gam_i = sum_{j<=i} g_j:                      */
/*   A_ij = beta_i exp(gam_i - gam_j) k_i.k_j  (j < i),  T = (I + A)^-1       */
/*   W = T diag(beta e^gam) K ;  U~ = T diag(beta) V ;  U = U~ - W S0^T        */
/*   O = diag(e^gam) Q S0^T + (Q K^T (.) exp(gam_i - gam_j) (.) [i>=j]) U      */
/*   S_end = e^{gam_c} S0 + U^T diag(e^{gam_c - gam}) K                        */
/* T is applied by forward substitution (solve (I + A) X = B row by row).     */
/* ------------------------------------------------------------------------ */
void gdn_ref_chunked_fwd(int N, const int32_t *cu, int hk, int hv, int dk, int dv, int chunk,
                         const double *qh, const double *kh, const double *v, const double *g,
                         const double *beta, const double *S0, double *o, double *S_fin)
{
    int G = hv / hk;
    size_t sz = (size_t)dv * dk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < N * hv; p++) {
        int n = p / hv, h = p % hv;
        int c = chunk;
        double *S = (double *)calloc(sz, sizeof(double));
        double *gam = (double *)malloc(c * sizeof(double));
        double *A = (double *)malloc((size_t)c * c * sizeof(double));
        double *W = (double *)malloc((size_t)c * dk * sizeof(double));
        double *U = (double *)malloc((size_t)c * dv * sizeof(double));
        double *Sn = (double *)malloc(sz * sizeof(double));
        if (S0) memcpy(S, S0 + (size_t)p * sz, sz * sizeof(double));
        for (int64_t cs = cu[n]; cs < cu[n + 1]; cs += c) {
            int L = (int)((cu[n + 1] - cs) < c ? (cu[n + 1] - cs) : c);
#define KR(i) (kh + ((cs + (i)) * hk + h / G) * dk)
#define QR(i) (qh + ((cs + (i)) * hk + h / G) * dk)
#define VR(i) (v + ((cs + (i)) * hv + h) * dv)
#define BE(i) (beta[(cs + (i)) * hv + h])
            double run = 0.0;
            for (int i = 0; i < L; i++) { run += g[(cs + i) * hv + h]; gam[i] = run; }
            for (int i = 0; i < L; i++)
                for (int j = 0; j < L; j++) {
                    double kk = 0.0;
                    if (j < i) {
                        for (int b = 0; b < dk; b++) kk += KR(i)[b] * KR(j)[b];
                        A[i * c + j] = BE(i) * exp(gam[i] - gam[j]) * kk;
                    } else {
                        A[i * c + j] = 0.0;
                    }
                }
            /* (I + A) W = diag(beta e^gam) K ; (I + A) U~ = diag(beta) V  */
            for (int i = 0; i < L; i++) {
                for (int b = 0; b < dk; b++) {
                    double acc = BE(i) * exp(gam[i]) * KR(i)[b];
                    for (int j = 0; j < i; j++) acc -= A[i * c + j] * W[j * dk + b];
                    W[i * dk + b] = acc;
                }
                for (int a = 0; a < dv; a++) {
                    double acc = BE(i) * VR(i)[a];
                    for (int j = 0; j < i; j++) acc -= A[i * c + j] * U[j * dv + a];
                    U[i * dv + a] = acc;
                }
            }
            /* U = U~ - W S0^T */
            for (int i = 0; i < L; i++)
                for (int a = 0; a < dv; a++) {
                    double acc = 0.0;
                    for (int b = 0; b < dk; b++) acc += W[i * dk + b] * S[a * dk + b];
                    U[i * dv + a] -= acc;
                }
            /* O */
            for (int i = 0; i < L; i++) {
                double *oi = o + ((cs + i) * hv + h) * dv;
                for (int a = 0; a < dv; a++) {
                    double acc = 0.0;
                    for (int b = 0; b < dk; b++) acc += QR(i)[b] * S[a * dk + b];
                    oi[a] = exp(gam[i]) * acc;
                }
                for (int j = 0; j <= i; j++) {
                    double qk = 0.0;
                    for (int b = 0; b < dk; b++) qk += QR(i)[b] * KR(j)[b];
                    double f = qk * exp(gam[i] - gam[j]);
                    for (int a = 0; a < dv; a++) oi[a] += f * U[j * dv + a];
                }
            }
            /* S_end */
            double gc = gam[L - 1];
            for (int a = 0; a < dv; a++)
                for (int b = 0; b < dk; b++) {
                    double acc = exp(gc) * S[a * dk + b];
                    for (int j = 0; j < L; j++)
                        acc += U[j * dv + a] * exp(gc - gam[j]) * KR(j)[b];
                    Sn[a * dk + b] = acc;
                }
            memcpy(S, Sn, sz * sizeof(double));
#undef KR
#undef QR
#undef VR
#undef BE
        }
        if (S_fin) memcpy(S_fin + (size_t)p * sz, S, sz * sizeof(double));
        free(S); free(gam); free(A); free(W); free(U); free(Sn);
    }
}

/* ------------------------------------------------------------------------ */
/* Zero-centred gated RMSNorm ([P2] "Summary": ZeroCenteredRMSNorm; [P3]      */
/* --apply-layernorm-1p), per (token, v-head) over d_v, weight shared by all  */
/* heads:  y = o / sqrt(mean(o^2) + eps) * (1 + w) * gate(z)                  */
/* gate: 0 = silu, 1 = sigmoid ([P2] "Summary": the shared GatedDeltaNet      */
/* takes output_gate_type; Qwen3.8 passes "sigmoid").                         */
/*   o, z, y [rows, d]; w [d]; rstd [rows] (nullable)                         */
/* ------------------------------------------------------------------------ */
static double out_gate(double z, int gate) { return gate ? sigm(z) : silu(z); }
/* d/dz sigmoid(z) = s (1 - s) */
static double dout_gate(double z, int gate)
{
    if (gate) { double s = sigm(z); return s * (1.0 - s); }
    return dsilu(z);
}

void gdn_ref_gated_rmsnorm(int64_t rows, int d, double eps, int gate, const double *o,
                           const double *z, const double *w, double *y, double *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        double ss = 0.0;
        for (int i = 0; i < d; i++) ss += o[r * d + i] * o[r * d + i];
        double rs = 1.0 / sqrt(ss / d + eps);
        if (rstd) rstd[r] = rs;
        for (int i = 0; i < d; i++)
            y[r * d + i] = o[r * d + i] * rs * (1.0 + w[i]) * out_gate(z[r * d + i], gate);
    }
}

/* Backward: with n = o rs, dn = dy (1+w) gate(z):
 *   do = rs (dn - n mean(dn n)) ; dz = dy n (1+w) gate'(z) ; dw = sum_rows dy n gate(z) */
void gdn_ref_gated_rmsnorm_bwd(int64_t rows, int d, double eps, int gate, const double *o,
                               const double *z, const double *w, const double *dy, double *do_,
                               double *dz, double *dw)
{
    for (int i = 0; i < d; i++) dw[i] = 0.0;
    for (int64_t r = 0; r < rows; r++) {
        double ss = 0.0;
        for (int i = 0; i < d; i++) ss += o[r * d + i] * o[r * d + i];
        double rs = 1.0 / sqrt(ss / d + eps);
        double m = 0.0;
        for (int i = 0; i < d; i++) {
            double nn = o[r * d + i] * rs;
            double dn = dy[r * d + i] * (1.0 + w[i]) * out_gate(z[r * d + i], gate);
            m += dn * nn;
        }
        m /= d;
        for (int i = 0; i < d; i++) {
            double nn = o[r * d + i] * rs;
            double zz = z[r * d + i];
            double dn = dy[r * d + i] * (1.0 + w[i]) * out_gate(zz, gate);
            do_[r * d + i] = rs * (dn - nn * m);
            dz[r * d + i] = dy[r * d + i] * nn * (1.0 + w[i]) * dout_gate(zz, gate);
            dw[i] += dy[r * d + i] * nn * out_gate(zz, gate);
        }
    }
}
