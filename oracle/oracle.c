/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the YOCO token-mixing path
 * computes ("You Only Cache Once: Decoder-Decoder Architectures for Language
 * Models", arXiv:2405.05254v2).  Only tests/, the smoke check and the bench's
 * CPU-baseline arm may call it.  It shares no code, header, table or helper
 * with the CUDA library; the product never links or loads it.
 *
 * Every routine takes fp64 arrays holding exactly the values the GPU path
 * consumes (bf16 / fp32 inputs widened without rounding) and accumulates in
 * fp64.  Nothing here is blocked, fused or reordered beyond what the cited
 * definition states.
 *
 * Layouts (row-major, last index fastest):
 *   q, k      [B, N, H, dk]      v, o [B, N, H, dv]
 *   logits    [B, N, H]          state [B, H, dk, dv]
 *   M         [R, dm]            W    [dm, n]          out [R, n]
 *   Q, O      [B, T, Hq, d]      cache K, V [B, Hkv, cap, d]
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ gate */

/* log(sigmoid(x)), written so that neither branch overflows.
 * Gate definition: gamma = sigmoid(X W_gamma)^(1/tau)  (paper Section 3.1,
 * Eq. 4); the Appendix F pseudocode takes it in log space as
 * logsigmoid(logit) / tau.  +inf gives 0 (gamma = 1), -inf gives -inf
 * (gamma = 0). */
static double log_sigmoid(double x)
{
    if (x >= 0.0)
        return -log1p(exp(-x));
    return x - log1p(exp(x));
}

/* Threads the OpenMP loops below may use (n > 0); the checker's own knob, used to
 * time it on one core as well as on all of them.  Without OpenMP it does nothing. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

double oracle_gate(double logit, double tau)
{
    return exp(log_sigmoid(logit) / tau);
}

/* ------------------------------------------------- gated retention forms */

/*
 * Recurrent form (paper Section 3.1, Eq. 5; Appendix F RecurrentRetention):
 *     S_n = gamma_n * S_{n-1} + k_n^T v_n,     o_n = q_n S_n
 * with q, k, v row vectors, S in R^{dk x dv}.  S0 (nullable = zeros) is the
 * state before token 0; the state after the last token goes to S_out
 * (nullable).
 */
void oracle_gret_recurrent(int B, int N, int H, int dk, int dv,
                           const double *q, const double *k, const double *v,
                           const double *logits, double tau, const double *S0,
                           double *o, double *S_out)
{
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
            if (S0)
                memcpy(S, S0 + ((size_t)b * H + h) * dk * dv, sizeof(double) * (size_t)dk * dv);
            else
                memset(S, 0, sizeof(double) * (size_t)dk * dv);
            for (int n = 0; n < N; ++n) {
                size_t row = ((size_t)b * N + n) * H + h;
                const double *qn = q + row * dk;
                const double *kn = k + row * dk;
                const double *vn = v + row * dv;
                double gamma = oracle_gate(logits[row], tau);
                /* S_n = gamma_n S_{n-1} + k_n^T v_n */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = gamma * S[(size_t)i * dv + j] + kn[i] * vn[j];
                /* o_n = q_n S_n */
                double *on = o + row * dv;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i)
                        acc += qn[i] * S[(size_t)i * dv + j];
                    on[j] = acc;
                }
            }
            if (S_out)
                memcpy(S_out + ((size_t)b * H + h) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
            free(S);
        }
    }
}

/*
 * Parallel form (paper Section 3.1, Eq. 4):
 *     D_nm = prod_{i=m+1..n} gamma_i  (n >= m),  0  (n < m)
 *     O    = (Q K^T (.) D) V
 * Starts from a zero state.  O(N^2 d) -- for small N only.  D_nm is formed as
 * the literal product, walked from m = n (empty product = 1) downwards.
 */
void oracle_gret_parallel(int B, int N, int H, int dk, int dv,
                          const double *q, const double *k, const double *v,
                          const double *logits, double tau, double *o)
{
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            for (int n = 0; n < N; ++n) {
                size_t rn = ((size_t)b * N + n) * H + h;
                double *on = o + rn * dv;
                for (int j = 0; j < dv; ++j)
                    on[j] = 0.0;
                double D = 1.0; /* D_nn */
                for (int m = n; m >= 0; --m) {
                    size_t rm = ((size_t)b * N + m) * H + h;
                    if (m < n) /* D_{n,m} = D_{n,m+1} * gamma_{m+1} */
                        D *= oracle_gate(logits[((size_t)b * N + (m + 1)) * H + h], tau);
                    double qk = 0.0;
                    for (int i = 0; i < dk; ++i)
                        qk += q[rn * dk + i] * k[rm * dk + i];
                    for (int j = 0; j < dv; ++j)
                        on[j] += qk * D * v[rm * dv + j];
                }
            }
        }
    }
}

/*
 * Chunkwise recurrent form, with the row/column convention made consistent
 * (re-derivation of the paper's Eq. 6 / Appendix B printed in the close-
 * reading notes Section 2.3 and the slides' backup "chunkwise recurrence with
 * consistent indices"; agrees with the Appendix F ChunkwiseRetention steps).
 * For chunk i starting at token a with length Bc (the last chunk may be
 * shorter), and beta_j = prod_{t=1..j} gamma_{a+t}:
 *     D_jk  = beta_j / beta_k  for k <= j, else 0
 *     O_[i] = (Q_[i] K_[i]^T (.) D) V_[i]  +  diag(beta) Q_[i] R_{i-1}
 *     R_i   = beta_Bc R_{i-1} + sum_k (beta_Bc / beta_k) K_{a+k}^T V_{a+k}
 * The ratio beta_j / beta_k is the product of the gammas strictly after
 * token k up to token j; it is evaluated as that product (no division), which
 * is the same number where beta_k != 0 and stays defined when a gate is 0.
 * S0 / S_out as in the recurrent form.
 */
void oracle_gret_chunkwise(int B, int N, int H, int dk, int dv, int C,
                           const double *q, const double *k, const double *v,
                           const double *logits, double tau, const double *S0,
                           double *o, double *S_out)
{
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *R = (double *)malloc(sizeof(double) * (size_t)dk * dv);
            double *Rn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
            double *g = (double *)malloc(sizeof(double) * (size_t)C);
            if (S0)
                memcpy(R, S0 + ((size_t)b * H + h) * dk * dv, sizeof(double) * (size_t)dk * dv);
            else
                memset(R, 0, sizeof(double) * (size_t)dk * dv);
            for (int a = 0; a < N; a += C) {
                int Bc = (N - a < C) ? (N - a) : C;
                for (int t = 0; t < Bc; ++t)
                    g[t] = oracle_gate(logits[((size_t)b * N + a + t) * H + h], tau);
                /* ratio(j, k) = beta_j / beta_k = prod_{t=k+1..j} g[t] (0-based) */
                for (int j = 0; j < Bc; ++j) {
                    size_t rj = ((size_t)b * N + a + j) * H + h;
                    double *oj = o + rj * dv;
                    /* beta_j = prod_{t=0..j} g[t] */
                    double beta_j = 1.0;
                    for (int t = 0; t <= j; ++t)
                        beta_j *= g[t];
                    /* cross-chunk: beta_j * q_j R_{i-1} */
                    for (int c = 0; c < dv; ++c) {
                        double acc = 0.0;
                        for (int i = 0; i < dk; ++i)
                            acc += q[rj * dk + i] * R[(size_t)i * dv + c];
                        oj[c] = beta_j * acc;
                    }
                    /* inner-chunk: sum_{k<=j} (q_j . k_k) D_jk v_k */
                    for (int kk = 0; kk <= j; ++kk) {
                        size_t rk = ((size_t)b * N + a + kk) * H + h;
                        double D = 1.0;
                        for (int t = kk + 1; t <= j; ++t)
                            D *= g[t];
                        double qk = 0.0;
                        for (int i = 0; i < dk; ++i)
                            qk += q[rj * dk + i] * k[rk * dk + i];
                        for (int c = 0; c < dv; ++c)
                            oj[c] += qk * D * v[rk * dv + c];
                    }
                }
                /* R_i = beta_Bc R_{i-1} + sum_k (beta_Bc / beta_k) k_k^T v_k */
                double beta_B = 1.0;
                for (int t = 0; t < Bc; ++t)
                    beta_B *= g[t];
                for (size_t e = 0; e < (size_t)dk * dv; ++e)
                    Rn[e] = beta_B * R[e];
                for (int kk = 0; kk < Bc; ++kk) {
                    size_t rk = ((size_t)b * N + a + kk) * H + h;
                    double w = 1.0;
                    for (int t = kk + 1; t < Bc; ++t)
                        w *= g[t];
                    for (int i = 0; i < dk; ++i)
                        for (int c = 0; c < dv; ++c)
                            Rn[(size_t)i * dv + c] += w * k[rk * dk + i] * v[rk * dv + c];
                }
                double *tmp = R; R = Rn; Rn = tmp;
            }
            if (S_out)
                memcpy(S_out + ((size_t)b * H + h) * dk * dv, R, sizeof(double) * (size_t)dk * dv);
            free(R);
            free(Rn);
            free(g);
        }
    }
}

/* ------------------------------------------------------------- shared KV */

/*
 * Shared K/V projection (paper Section 2.2, Eq. 2):
 *     K^ = LN(M) W_K,   V^ = LN(M) W_V,   LN = RMSNorm
 * RMSNorm of a row m: m * r * g with r = 1 / sqrt(mean(m^2) + eps) and an
 * optional gain g (NULL = ones).  One call projects with one weight matrix
 * W [dm, n]; the caller runs it for W_K and for W_V.
 */
void oracle_rmsnorm_proj(int R, int dm, int n, const double *M, const double *g,
                         double eps, const double *W, double *out)
{
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        const double *m = M + (size_t)r * dm;
        double ss = 0.0;
        for (int i = 0; i < dm; ++i)
            ss += m[i] * m[i];
        double rinv = 1.0 / sqrt(ss / dm + eps);
        for (int c = 0; c < n; ++c) {
            double acc = 0.0;
            for (int i = 0; i < dm; ++i)
                acc += (m[i] * rinv * (g ? g[i] : 1.0)) * W[(size_t)i * n + c];
            out[(size_t)r * n + c] = acc;
        }
    }
}

/*
 * Round an fp64 value to the nearest bfloat16 (ties to even), returning the
 * bf16 bit pattern.  bf16 = 1 sign, 8 exponent, 7 fraction bits (the float32
 * exponent range).  Written from the format definition: scale the magnitude
 * so that one bf16 unit in the last place is 1, round to the nearest integer
 * with ties to even, scale back.
 */
uint16_t oracle_round_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);             /* a = f * 2^e, f in [0.5, 1) => a in [2^(e-1), 2^e) */
    int ulp_exp = (e - 1) - 7; /* 7 fraction bits */
    if (ulp_exp < -126 - 7)
        ulp_exp = -126 - 7;   /* subnormal quantum 2^-133 */
    double m = ldexp(a, -ulp_exp);
    double mr = nearbyint(m); /* default rounding mode: to nearest, ties to even */
    double r = ldexp(mr, ulp_exp);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max)
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

/*
 * Append T projected tokens to the shared cache (paper Section 2.2: the
 * cache is produced once and reused by every cross-decoder layer).
 *   kv_new [B, T, Hkv*d]  (fp64 projection output, head-major within a row)
 *   cache  [B, Hkv, cap, d] as bf16 bits (round_bf16 != 0) or fp64 values
 * Row t of sequence b goes to slot len + t of every head; nothing else of the
 * cache changes.
 */
void oracle_kv_append_bf16(int B, int T, int Hkv, int d, int64_t cap, int64_t len,
                           const double *kv_new, uint16_t *cache)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < Hkv; ++h)
                for (int c = 0; c < d; ++c)
                    cache[(((size_t)b * Hkv + h) * cap + (size_t)(len + t)) * d + c] =
                        oracle_round_bf16(kv_new[((size_t)b * T + t) * Hkv * d + (size_t)h * d + c]);
}

/* ------------------------------------------------------- cross attention */

/*
 * Cross-decoder attention (paper Section 2.2, Eq. 3): causal softmax
 * attention of each layer's queries against the one shared K^/V^, with
 * grouped-query heads.  Query row t sits at position p0 + t and reads cache
 * slots m <= p0 + t.  Query head h reads kv head h / (Hq / Hkv).
 *     s_m = scale * q . k_m,    o = sum_m softmax(s)_m v_m
 * evaluated as the plain masked softmax (maximum subtracted for range).
 */
void oracle_cross_attn(int B, int T, int Hq, int Hkv, int d, int64_t cap,
                       const double *Q, const double *Kc, const double *Vc,
                       int64_t p0, double scale, double *O)
{
    int group = Hq / Hkv;
    #pragma omp parallel for collapse(3) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            for (int h = 0; h < Hq; ++h) {
                int64_t pos = p0 + t;
                int hk = h / group;
                const double *qv = Q + (((size_t)b * T + t) * Hq + h) * d;
                const double *Kb = Kc + ((size_t)b * Hkv + hk) * (size_t)cap * d;
                const double *Vb = Vc + ((size_t)b * Hkv + hk) * (size_t)cap * d;
                double *ov = O + (((size_t)b * T + t) * Hq + h) * d;
                double *s = (double *)malloc(sizeof(double) * (size_t)(pos + 1));
                double mx = -INFINITY;
                for (int64_t m = 0; m <= pos; ++m) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += qv[c] * Kb[(size_t)m * d + c];
                    s[m] = scale * acc;
                    if (s[m] > mx)
                        mx = s[m];
                }
                double den = 0.0;
                for (int64_t m = 0; m <= pos; ++m) {
                    s[m] = exp(s[m] - mx);
                    den += s[m];
                }
                for (int c = 0; c < d; ++c)
                    ov[c] = 0.0;
                for (int64_t m = 0; m <= pos; ++m)
                    for (int c = 0; c < d; ++c)
                        ov[c] += (s[m] / den) * Vb[(size_t)m * d + c];
                free(s);
            }
        }
    }
}

/*
 * Sliding-window attention of the self-decoder (paper Section 3.2, Eq. 8):
 *   head_i = softmax(Q K^T + B) V,  B_nm = 0 for n - C < m <= n, -inf otherwise,
 * i.e. the query at position n sees the C most recent keys including its own.
 * The formula prints no scale; the score is q . k times `scale` (the caller's
 * reading, 1 / sqrt(d) by default).  Query head h reads kv head h / (Hq / Hkv).
 * q [B, N, Hq, d], k, v [B, N, Hkv, d], o [B, N, Hq, d] (token-major, as the
 * projections write them).
 */
void oracle_swa_attn(int B, int N, int Hq, int Hkv, int d, int64_t window,
                     const double *Q, const double *K, const double *V,
                     double scale, double *O)
{
    int group = Hq / Hkv;
    #pragma omp parallel for collapse(3) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int n = 0; n < N; ++n) {
            for (int h = 0; h < Hq; ++h) {
                int hk = h / group;
                int64_t m0 = (int64_t)n - window + 1;
                if (m0 < 0)
                    m0 = 0;
                const double *qv = Q + (((size_t)b * N + n) * Hq + h) * d;
                double *ov = O + (((size_t)b * N + n) * Hq + h) * d;
                int64_t cnt = (int64_t)n - m0 + 1;
                double *s = (double *)malloc(sizeof(double) * (size_t)cnt);
                double mx = -INFINITY;
                for (int64_t m = m0; m <= n; ++m) {
                    const double *kv = K + (((size_t)b * N + m) * Hkv + hk) * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += qv[c] * kv[c];
                    s[m - m0] = scale * acc;
                    if (s[m - m0] > mx)
                        mx = s[m - m0];
                }
                double den = 0.0;
                for (int64_t i = 0; i < cnt; ++i) {
                    s[i] = exp(s[i] - mx);
                    den += s[i];
                }
                for (int c = 0; c < d; ++c)
                    ov[c] = 0.0;
                for (int64_t m = m0; m <= n; ++m) {
                    const double *vv = V + (((size_t)b * N + m) * Hkv + hk) * d;
                    for (int c = 0; c < d; ++c)
                        ov[c] += (s[m - m0] / den) * vv[c];
                }
                free(s);
            }
        }
    }
}

/*
 * Output of multi-head gated retention (paper Section 3.1, Eq. 7):
 *   Y = GroupNorm_h(Concat(head_1..head_H)),  out = swish(X W_G) (.) Y
 * GroupNorm with one group per head: each token's head vector is centred and
 * divided by sqrt(variance + eps) (variance over the head's d channels, divided
 * by d), then scaled and shifted per channel by w, b (w = 1, b = 0 when absent).
 * swish(x) = x * sigmoid(x).  `gpre` is X W_G (the projection itself is outside
 * this library).  o, gpre, z [B, N, H, d].
 */
void oracle_group_norm_gate(int B, int N, int H, int d, const double *o, const double *gpre,
                            const double *w, const double *bias, double eps, double *z)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int n = 0; n < N; ++n) {
            for (int h = 0; h < H; ++h) {
                size_t base = (((size_t)b * N + n) * H + h) * d;
                double mean = 0.0;
                for (int c = 0; c < d; ++c)
                    mean += o[base + c];
                mean /= d;
                double var = 0.0;
                for (int c = 0; c < d; ++c)
                    var += (o[base + c] - mean) * (o[base + c] - mean);
                var /= d;
                double inv = 1.0 / sqrt(var + eps);
                for (int c = 0; c < d; ++c) {
                    double y = (o[base + c] - mean) * inv;
                    if (w)
                        y *= w[(size_t)h * d + c];
                    if (bias)
                        y += bias[(size_t)h * d + c];
                    double g = gpre[base + c];
                    z[base + c] = g / (1.0 + exp(-g)) * y;
                }
            }
        }
    }
}

/*
 * Rotary position encoding (paper Section 3.1: Q = (X W_Q) (.) Theta,
 * K = (X W_K) (.) conj(Theta), Theta_n = e^{i n theta}; the notes: the shared K^
 * is rotated once in the cross-decoder's projection and every cross layer
 * rotates its own Q).  Real-valued form: channel pair (2i, 2i+1) of the vector at
 * position p is turned by the angle p * base^(-2i/d):
 *   x'_2i   = x_2i cos a - x_2i+1 sin a,   x'_2i+1 = x_2i sin a + x_2i+1 cos a.
 * Turning q and k each by its own position makes q'.k' depend on the positions
 * only through their difference, which is what the complex product of Theta and
 * conj(Theta) expresses.  x [rows, d] with row r at position pos[r]; in place.
 */
void oracle_rope(int64_t rows, int d, const int64_t *pos, double base, double *x)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int i = 0; i < d / 2; ++i) {
            double theta = pow(base, -2.0 * i / d);
            double a = (double)pos[r] * theta;
            double c = cos(a), s = sin(a);
            double x0 = x[r * d + 2 * i], x1 = x[r * d + 2 * i + 1];
            x[r * d + 2 * i] = x0 * c - x1 * s;
            x[r * d + 2 * i + 1] = x0 * s + x1 * c;
        }
    }
}
