/*
 * CPU oracle for one DSpark speculative-decoding round.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The CUDA
 * product path shares no code, header, table or helper with this file.
 *
 * Plain, single-threaded, fp64.  Each function follows the passage it cites in
 * the order the pages state it; nothing is blocked, fused or reordered.
 *
 * Pages cited:
 *   [DSpark]   "DSpark" (rainlin-net.pages.dev, llm-inference/dspark)
 *   [Handbook] "投机解码的新做法：整块草稿、按负载验证与 PD 分离"
 *              (anrans.github.io ai-infra-handbooks, serving/frontier/spec-next)
 *   [Summary]  "DSpark: Speculative decodingを活用したLLM推論の高速化" (ja.news.hada.io)
 *
 * Readings where the pages are silent:
 *   - temperature T divides the combined logits (U + bias) for draft and target
 *     alike; T == 0 means greedy argmax with the lowest index winning ties;
 *   - greedy decisions are taken on fp32 logits (the kernel's precision): the
 *     exact fp64 value U + bias is rounded once to fp32 before the argmax;
 *   - the accept rule is the textbook rejection test u < p_t(x) / p_d(x) with
 *     u in [0,1); the residual is max(0, p_t - p_d) renormalised, and when its
 *     mass is zero the token is drawn from p_t; the bonus comes from target
 *     row len (0-based);
 *   - the confidence head has no bias term; w = [w_h ; w_e] follows [h ; W1[x]];
 *   - scheduler keys sort by (a descending, position ascending, request
 *     ascending); sums of a use Q.40 fixed point (int64) so that every
 *     summation order gives the same S_b; Theta(b) = (R + S_b 2^-40) * SPS[R + b]
 *     in fp64; early stop = the first b with Theta(b+1) <= Theta(b).
 *   - uniforms: Philox4x64-10 (Salmon et al., SC'11), key = (seed, 0),
 *     counter = (round, request, position, purpose); u = (out[0] >> 40) * 2^-24.
 *     purpose 0 = draft sample, 1 = accept test, 2 = residual or bonus sample.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_MEM (-2)

/* ------------------------------------------------------------------------- */
/* bf16 storage: the upper 16 bits of an IEEE binary32.                       */
/* ------------------------------------------------------------------------- */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Philox4x64-10, from its published definition (Salmon, Moraes, Dror, Shaw,  */
/* "Parallel random numbers: as easy as 1, 2, 3", SC'11): ten rounds of two    */
/* 64x64->128 multiplies with multipliers M0, M1, key bumped by the Weyl       */
/* constants W0 (golden ratio) and W1 (sqrt(3) - 1) between rounds.           */
/* ------------------------------------------------------------------------- */
static void mul_64x64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    /* schoolbook product on 32-bit halves: portable to every host */
    uint64_t a0 = a & 0xffffffffu, a1 = a >> 32;
    uint64_t b0 = b & 0xffffffffu, b1 = b >> 32;
    uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
    *lo = (p00 & 0xffffffffu) | (mid << 32);
    *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t hi0, lo0, hi1, lo1;
        mul_64x64(M0, x0, &hi0, &lo0);
        mul_64x64(M1, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* u in [0,1) with 24 random bits, exactly representable in binary32. */
double oracle_uniform(uint64_t seed, uint64_t round, uint64_t request, uint64_t position,
                      uint64_t purpose)
{
    uint64_t ctr[4] = {round, request, position, purpose};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------- */
/* [DSpark §2.3 "Markov Head"]: B(x_{k-1}, .) = W1[x_{k-1}] W2 with           */
/* W1 in R^{V x r} and W2 in R^{r x V}.  Exact fp64 sum of bf16 products.     */
/* ------------------------------------------------------------------------- */
void oracle_markov_bias(const uint16_t *W1, const uint16_t *W2, int V, int rank, int32_t prev,
                        double *bias)
{
    for (int v = 0; v < V; ++v) bias[v] = 0.0;
    const uint16_t *e = W1 + (size_t)prev * (size_t)rank;
    for (int i = 0; i < rank; ++i) {
        double ei = bf16_value(e[i]);
        const uint16_t *row = W2 + (size_t)i * (size_t)V;
        for (int v = 0; v < V; ++v) bias[v] += ei * bf16_value(row[v]);
    }
}

/* Softmax in fp64.  Returns log Z = m + ln(sum exp(z - m)). */
static double softmax64(const double *z, int V, double *p)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) if (z[v] > m) m = z[v];
    double s = 0.0;
    for (int v = 0; v < V; ++v) { p[v] = exp(z[v] - m); s += p[v]; }
    for (int v = 0; v < V; ++v) p[v] /= s;
    return m + log(s);
}

/* Inverse CDF: the first v whose cumulative probability exceeds u.  If
 * rounding leaves the total just under u, the last v with p > 0 is taken. */
int32_t oracle_inverse_cdf(const double *p, int V, double u)
{
    double c = 0.0;
    int32_t last = 0;
    for (int v = 0; v < V; ++v) {
        if (p[v] > 0.0) last = v;
        c += p[v];
        if (c > u) return v;
    }
    return last;
}

/* argmax on fp32 values, lowest index on ties. */
static int32_t argmax_f32(const float *z, int V)
{
    int32_t best = 0;
    for (int v = 1; v < V; ++v) if (z[v] > z[best]) best = v;
    return best;
}

/* [DSpark §2.2, eq. p_k]: the draft distribution at one position.
 * z(v) = (U_k(v) + B(x_{k-1}, v)) / T in fp64; p = softmax(z).
 * Returns log Z.  Writes p[V] (fp64).  T must be > 0. */
double oracle_draft_probs(const float *U_row, const uint16_t *W1, const uint16_t *W2, int32_t prev,
                          int V, int rank, float temperature, double *p)
{
    double *bias = (double *)malloc(sizeof(double) * (size_t)V);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    if (!bias || !z) { free(bias); free(z); return NAN; }
    oracle_markov_bias(W1, W2, V, rank, prev, bias);
    for (int v = 0; v < V; ++v) z[v] = ((double)U_row[v] + bias[v]) / (double)temperature;
    double logZ = softmax64(z, V, p);
    free(bias);
    free(z);
    return logZ;
}

/* Greedy logits at one position: fl32(U_k(v) + B(x_{k-1}, v)). */
void oracle_draft_logits_f32(const float *U_row, const uint16_t *W1, const uint16_t *W2,
                             int32_t prev, int V, int rank, float *zf)
{
    double *bias = (double *)malloc(sizeof(double) * (size_t)V);
    if (!bias) return;
    oracle_markov_bias(W1, W2, V, rank, prev, bias);
    for (int v = 0; v < V; ++v) zf[v] = (float)((double)U_row[v] + bias[v]);
    free(bias);
}

/* Target distribution of one verify row: softmax(T_row / T) in fp64. */
double oracle_target_probs(const float *T_row, int V, float temperature, double *p)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    if (!z) return NAN;
    for (int v = 0; v < V; ++v) z[v] = (double)T_row[v] / (double)temperature;
    double logZ = softmax64(z, V, p);
    free(z);
    return logZ;
}

/* ------------------------------------------------------------------------- */
/* [DSpark §2.2-2.3] and the sequential loop of [DSpark §6.2]: starting from  */
/* prev = anchor, for k = 1..gamma add the Markov bias of prev to U_k, draw   */
/* x_k from the explicit softmax, keep p_k^d(x_k), set prev = x_k.            */
/* One request; U_r is [gamma, V].  Uniform for position j (0-based) is        */
/* Philox(seed; round, request, j, 0).                                         */
/* ------------------------------------------------------------------------- */
int oracle_draft_request(const float *U_r, const uint16_t *W1, const uint16_t *W2, int32_t anchor,
                         int gamma, int V, int rank, float temperature, uint64_t seed,
                         uint64_t round, uint64_t request, int32_t *tokens, float *pd_tok,
                         float *logZ)
{
    if (gamma < 0 || V <= 0 || rank <= 0 || anchor < 0 || anchor >= V) return ORACLE_ERR_ARG;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    float *zf = (float *)malloc(sizeof(float) * (size_t)V);
    if (!p || !zf) { free(p); free(zf); return ORACLE_ERR_MEM; }
    int32_t prev = anchor;
    for (int j = 0; j < gamma; ++j) {
        const float *U_row = U_r + (size_t)j * (size_t)V;
        int32_t x;
        if (temperature > 0.0f) {
            double lz = oracle_draft_probs(U_row, W1, W2, prev, V, rank, temperature, p);
            double u = oracle_uniform(seed, round, request, (uint64_t)j, 0);
            x = oracle_inverse_cdf(p, V, u);
            pd_tok[j] = (float)p[x];
            logZ[j] = (float)lz;
        } else {
            oracle_draft_logits_f32(U_row, W1, W2, prev, V, rank, zf);
            x = argmax_f32(zf, V);
            pd_tok[j] = 1.0f;
            logZ[j] = zf[x];
        }
        tokens[j] = x;
        prev = x;
    }
    free(p);
    free(zf);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* [DSpark §3.1, eq. c_k] c_k = sigma(w^T [h_k ; W1[x_{k-1}]]) and            */
/* [DSpark §1.1, eq. a_j] a_j = prod_{i<=j} c_i, left to right in fp32.       */
/* One request; h_r is bf16 [gamma, d]; w is fp32 [d + rank].                 */
/* ------------------------------------------------------------------------- */
/* a_j = fl32(a_{j-1} * c_j), a_0 = c_0: one fp32 rounding per factor. */
void oracle_survival(const float *c, int gamma, float *a)
{
    float run = 1.0f;
    for (int j = 0; j < gamma; ++j) {
        run = run * c[j];
        a[j] = run;
    }
}

/* [DSpark §3.2, STS]: with sequential temperature scaling the confidence of
 * position j is sigma(s_j / t_j) for per-position temperatures t_j > 0
 * (sts_temp == NULL: no scaling). */
int oracle_confidence_request(const uint16_t *h_r, const uint16_t *W1, const float *w,
                              int32_t anchor, const int32_t *tokens, int gamma, int d, int rank,
                              int V, const float *sts_temp, float *c, float *a)
{
    for (int j = 0; j < gamma; ++j) {
        int32_t prev = (j == 0) ? anchor : tokens[j - 1];
        if (prev < 0 || prev >= V) return ORACLE_ERR_ARG;
        if (sts_temp && !(sts_temp[j] > 0.0f && sts_temp[j] <= 3.4e38f)) return ORACLE_ERR_ARG;
        double s = 0.0;
        const uint16_t *hj = h_r + (size_t)j * (size_t)d;
        for (int i = 0; i < d; ++i) s += (double)w[i] * bf16_value(hj[i]);
        const uint16_t *e = W1 + (size_t)prev * (size_t)rank;
        for (int i = 0; i < rank; ++i) s += (double)w[d + i] * bf16_value(e[i]);
        if (sts_temp) s /= (double)sts_temp[j];
        c[j] = (float)(1.0 / (1.0 + exp(-s)));
    }
    oracle_survival(c, gamma, a);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* [DSpark §4.1-4.3] hardware-aware prefix scheduler.                         */
/* All (r, j) pairs sorted by a_{r,j} descending; S_b = sum of the top b      */
/* values; B = R + b tokens; Theta(b) = (R + S_b) * SPS(R + b).               */
/* mode 0: early stop (first b with Theta(b+1) <= Theta(b), else R*gamma);    */
/* mode 1: Top-K with a budget K from two rounds earlier (min(K, R*gamma));   */
/* mode 2: fixed length (every position verified).                            */
/* argmax_b is the global argmax of Theta (lowest b on ties), the budget the  */
/* caller keeps for round t+2 [Summary, "スケジューラの実運用適用"].          */
/* ------------------------------------------------------------------------- */
typedef struct {
    float a;
    int32_t j;
    int32_t r;
} sched_entry;

static int sched_cmp(const void *pa, const void *pb)
{
    const sched_entry *x = (const sched_entry *)pa, *y = (const sched_entry *)pb;
    if (x->a > y->a) return -1;
    if (x->a < y->a) return 1;
    if (x->j != y->j) return (x->j < y->j) ? -1 : 1;
    if (x->r != y->r) return (x->r < y->r) ? -1 : 1;
    return 0;
}

int oracle_schedule(const float *a, int R, int gamma, const double *sps, int sps_len, int mode,
                    int budget_K, int32_t *lens, int32_t *total_b, int32_t *argmax_b,
                    double *theta, double *theta_all /* optional [R*gamma+1] */)
{
    int n = R * gamma;
    if (R < 0 || gamma < 0 || sps_len < R + n + 1) return ORACLE_ERR_ARG;
    sched_entry *e = (sched_entry *)malloc(sizeof(sched_entry) * (size_t)(n > 0 ? n : 1));
    int64_t *S = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n + 1));
    double *th = (double *)malloc(sizeof(double) * (size_t)(n + 1));
    if (!e || !S || !th) { free(e); free(S); free(th); return ORACLE_ERR_MEM; }
    for (int r = 0; r < R; ++r)
        for (int j = 0; j < gamma; ++j) {
            e[r * gamma + j].a = a[(size_t)r * gamma + j];
            e[r * gamma + j].j = j;
            e[r * gamma + j].r = r;
        }
    qsort(e, (size_t)n, sizeof(sched_entry), sched_cmp);
    S[0] = 0;
    for (int b = 0; b < n; ++b) S[b + 1] = S[b] + (int64_t)llrint((double)e[b].a * 0x1p40);
    for (int b = 0; b <= n; ++b) {
        double tau = (double)R + (double)S[b] * 0x1p-40;
        th[b] = tau * sps[R + b];
    }
    int bstar;
    if (mode == 0) {
        bstar = n;
        for (int b = 0; b < n; ++b)
            if (th[b + 1] <= th[b]) { bstar = b; break; }
    } else if (mode == 1) {
        bstar = budget_K < 0 ? 0 : (budget_K > n ? n : budget_K);
    } else {
        bstar = n;
    }
    int best = 0;
    for (int b = 1; b <= n; ++b) if (th[b] > th[best]) best = b;
    for (int r = 0; r < R; ++r) lens[r] = 0;
    for (int b = 0; b < bstar; ++b) lens[e[b].r] += 1;
    *total_b = bstar;
    *argmax_b = best;
    *theta = th[bstar];
    if (theta_all) for (int b = 0; b <= n; ++b) theta_all[b] = th[b];
    free(e);
    free(S);
    free(th);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Standard speculative verification by rejection sampling [DSpark intro and   */
/* §2.2; Summary, "問題定義"].  One request, explicit uniforms:               */
/* u_acc[j] for the accept test at position j, u_res[n] for the residual or   */
/* bonus draw at position n.  T_r is [gamma+1, V]: row j holds the target     */
/* logits for draft position j, row gamma the bonus row.                      */
/* ------------------------------------------------------------------------- */
int oracle_verify_request_u(const float *T_r, const float *U_r, const uint16_t *W1,
                            const uint16_t *W2, int32_t anchor, const int32_t *tokens, int len,
                            int gamma, int V, int rank, float temperature, const double *u_acc,
                            const double *u_res, int32_t *n_accept, int32_t *next_token)
{
    if (len < 0 || len > gamma || V <= 0) return ORACLE_ERR_ARG;
    if (temperature <= 0.0f) {
        int n = len;
        for (int j = 0; j < len; ++j) {
            if (tokens[j] != argmax_f32(T_r + (size_t)j * V, V)) { n = j; break; }
        }
        *n_accept = n;
        *next_token = argmax_f32(T_r + (size_t)n * V, V);
        return ORACLE_OK;
    }
    double *pt = (double *)malloc(sizeof(double) * (size_t)V);
    double *pd = (double *)malloc(sizeof(double) * (size_t)V);
    if (!pt || !pd) { free(pt); free(pd); return ORACLE_ERR_MEM; }
    int n = len;
    for (int j = 0; j < len; ++j) {
        int32_t x = tokens[j];
        int32_t prev = (j == 0) ? anchor : tokens[j - 1];
        oracle_target_probs(T_r + (size_t)j * V, V, temperature, pt);
        oracle_draft_probs(U_r + (size_t)j * V, W1, W2, prev, V, rank, temperature, pd);
        double ratio = pt[x] / pd[x];
        if (!(u_acc[j] < ratio)) {
            /* residual max(0, p_t - p_d), renormalised */
            double s = 0.0;
            for (int v = 0; v < V; ++v) {
                double q = pt[v] - pd[v];
                pd[v] = q > 0.0 ? q : 0.0;
                s += pd[v];
            }
            int32_t y;
            if (s > 0.0) {
                for (int v = 0; v < V; ++v) pd[v] /= s;
                y = oracle_inverse_cdf(pd, V, u_res[j]);
            } else {
                y = oracle_inverse_cdf(pt, V, u_res[j]);
            }
            n = j;
            *next_token = y;
            break;
        }
    }
    if (n == len) {
        oracle_target_probs(T_r + (size_t)len * V, V, temperature, pt);
        *next_token = oracle_inverse_cdf(pt, V, u_res[len]);
    }
    *n_accept = n;
    free(pt);
    free(pd);
    return ORACLE_OK;
}

/* The same with Philox uniforms: purpose 1 for the accept tests, purpose 2
 * for the residual or bonus draw at the position where it happens. */
int oracle_verify_request(const float *T_r, const float *U_r, const uint16_t *W1,
                          const uint16_t *W2, int32_t anchor, const int32_t *tokens, int len,
                          int gamma, int V, int rank, float temperature, uint64_t seed,
                          uint64_t round, uint64_t request, int32_t *n_accept,
                          int32_t *next_token)
{
    if (len < 0 || len > gamma) return ORACLE_ERR_ARG;
    double u_acc[64], u_res[65];
    if (gamma > 64) return ORACLE_ERR_ARG;
    for (int j = 0; j < gamma; ++j) u_acc[j] = oracle_uniform(seed, round, request, (uint64_t)j, 1);
    for (int j = 0; j <= gamma; ++j) u_res[j] = oracle_uniform(seed, round, request, (uint64_t)j, 2);
    return oracle_verify_request_u(T_r, U_r, W1, W2, anchor, tokens, len, gamma, V, rank,
                                   temperature, u_acc, u_res, n_accept, next_token);
}

/* Rejection-sampling building block on explicit distributions (used by the
 * brute-force tests on tiny vocabularies): accept x with u_acc < pt[x]/pd[x],
 * else draw from the renormalised residual with u_res. */
int oracle_verify_position(const double *pt, const double *pd, int V, int32_t x, double u_acc,
                           double u_res, int32_t *accepted, int32_t *token)
{
    double ratio = pt[x] / pd[x];
    if (u_acc < ratio) { *accepted = 1; *token = x; return ORACLE_OK; }
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    if (!q) return ORACLE_ERR_MEM;
    double s = 0.0;
    for (int v = 0; v < V; ++v) { double d = pt[v] - pd[v]; q[v] = d > 0.0 ? d : 0.0; s += q[v]; }
    if (s > 0.0) {
        for (int v = 0; v < V; ++v) q[v] /= s;
        *token = oracle_inverse_cdf(q, V, u_res);
    } else {
        *token = oracle_inverse_cdf(pt, V, u_res);
    }
    *accepted = 0;
    free(q);
    return ORACLE_OK;
}

/* [DSpark §3.1, eq. c_k*]: analytic acceptance 1 - 0.5 * ||p_d - p_t||_1. */
double oracle_overlap(const double *pd, const double *pt, int V)
{
    double l1 = 0.0;
    for (int v = 0; v < V; ++v) l1 += fabs(pd[v] - pt[v]);
    return 1.0 - 0.5 * l1;
}

/* [DSpark §3.1, eq. c_k*] over the rows one verification reads: for every
 * position j <= len that has a draft distribution (j < gamma), c*[j] is the
 * overlap of the draft distribution at j (conditioned on x_{j-1}, x_{-1} =
 * anchor) with the target distribution of row j; positions j > len get NaN.
 * T == 0: both distributions are point masses, the draft's at its token x_j
 * and the target's at the first argmax of row j, so c*[j] is 1 or 0. */
int oracle_c_star_request(const float *T_r, const float *U_r, const uint16_t *W1,
                          const uint16_t *W2, int32_t anchor, const int32_t *tokens, int len,
                          int gamma, int V, int rank, float temperature, double *c_star)
{
    if (len < 0 || len > gamma || V <= 0) return ORACLE_ERR_ARG;
    for (int j = 0; j < gamma; ++j) c_star[j] = NAN;
    int last = len < gamma ? len : gamma - 1;
    if (temperature <= 0.0f) {
        for (int j = 0; j <= last; ++j)
            c_star[j] = tokens[j] == argmax_f32(T_r + (size_t)j * V, V) ? 1.0 : 0.0;
        return ORACLE_OK;
    }
    double *pt = (double *)malloc(sizeof(double) * (size_t)V);
    double *pd = (double *)malloc(sizeof(double) * (size_t)V);
    if (!pt || !pd) { free(pt); free(pd); return ORACLE_ERR_MEM; }
    for (int j = 0; j <= last; ++j) {
        int32_t prev = (j == 0) ? anchor : tokens[j - 1];
        if (prev < 0 || prev >= V) { free(pt); free(pd); return ORACLE_ERR_ARG; }
        oracle_target_probs(T_r + (size_t)j * V, V, temperature, pt);
        oracle_draft_probs(U_r + (size_t)j * V, W1, W2, prev, V, rank, temperature, pd);
        c_star[j] = oracle_overlap(pd, pt, V);
    }
    free(pt);
    free(pd);
    return ORACLE_OK;
}
