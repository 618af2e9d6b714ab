/*
 * CPU oracle for the quantised MoE layer forward (router logits, top-k with
 * softmax renormalisation, token-to-expert grouping, group-wise INT4/2-bit
 * dequantised expert FFN with SwiGLU, weighted combine plus residual and an
 * optional sigmoid-gated shared expert).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call this library.  It shares no code,
 * header, table or helper with the CUDA path; it reads the canonical packed
 * buffers through its own unpacker.  Plain, slow and obviously correct:
 * fp64 arithmetic for the FFN, exact integer arithmetic for the router.
 *
 * Sources of each step (page title, section):
 *   - router scores every expert from the token's hidden state and keeps the
 *     top-k: "12GB显卡跑68GB大模型：Betelgeuse引擎实测22 tok/s", MoE background;
 *     top-2 of 64 experts: "Strata" article, section 1.1; top-4 of 512:
 *     "Flash-MoE" article, section 1.
 *   - group-wise INT4 with one scale and one zero point per 128 weights:
 *     "Strata" article, section 2.2; w = (q - zero) * scale and the packed
 *     weight block layout: "为什么12G显存笔记本能跑MoE-16B", section 4.2;
 *     2-bit dequant matvec: "Flash-MoE" article, section 3.
 *   - per-expert aggregation of the requests routed to it
 *     (Map{expert_id: Vec(request_id, ...)}): "为什么12G显存笔记本能跑MoE-16B",
 *     section 2.3.
 *   - fused SwiGLU, and MoE combine + residual + sigmoid gate:
 *     "Flash-MoE" article, section 3.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - router logit = exact sum of the exact fp16 x fp16 products, rounded
 *     once to fp32 (round to nearest even), then one fp32 add of the bias;
 *   - top-k order: logit descending, ties to the lower expert id;
 *   - weights: softmax over the k selected biased logits, in fp64;
 *   - grouping: stable counting sort of the flat pair ids p = t*k + j;
 *   - SwiGLU: h = silu(g) * u with silu(g) = g / (1 + exp(-g));
 *   - shared expert gate: sigmoid(x . wg), no bias;
 *   - output: x + sum_j w_j y_j + gate * y_shared in fp64, rounded once to
 *     fp16 (round to nearest even).
 *   - RMSNorm in front of the router (two-pass RMSNorm, "Flash-MoE" article,
 *     section 3): the plain definition in fp64, rounded once to fp16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

/* ---------------------------------------------------------------- fp16 */

/* IEEE binary16 bit pattern -> exact double. */
double oracle_half_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return s ? -v : v;
}

/* double -> IEEE binary16, round to nearest, ties to even. */
uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (isinf(v))
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the quantum is 2^-24 */
        double r = nearbyint(a * 16777216.0);
        return sign | (uint16_t)r; /* r == 1024 is the smallest normal */
    }
    int e;
    double m = frexp(a, &e);    /* a = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 11)); /* 11-bit significand in [1024, 2048] */
    if (r == 2048.0) {
        r = 1024.0;
        e += 1;
    }
    int E = e - 1 + 15;
    if (E >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(E << 10) | (uint16_t)((int)r - 1024);
}

/* --------------------------------------------------------- code unpack */

static inline int code_at(const uint8_t *row, int k, int wbits)
{
    if (wbits == 4) {
        uint8_t b = row[k >> 1];
        return (k & 1) ? (b >> 4) : (b & 0xF);
    }
    uint8_t b = row[k >> 2];
    return (b >> (2 * (k & 3))) & 0x3;
}

int oracle_unpack_codes(const uint8_t *codes, int64_t rows, int K, int wbits, uint8_t *q)
{
    if (!codes || !q || rows < 0 || K <= 0 || (wbits != 4 && wbits != 2) || (K * wbits) % 8)
        return -1;
    int64_t rb = (int64_t)K * wbits / 8;
    for (int64_t r = 0; r < rows; r++)
        for (int k = 0; k < K; k++)
            q[r * K + k] = (uint8_t)code_at(codes + r * rb, k, wbits);
    return 0;
}

/* w[r][k] = (q - zero[r][k/G]) * scale[r][k/G], exactly in double. */
static void dequant_row(const uint8_t *crow, const uint16_t *srow, const uint8_t *zrow,
                        int K, int wbits, int group, double *w)
{
    for (int k = 0; k < K; k++) {
        int g = k / group;
        w[k] = ((double)code_at(crow, k, wbits) - (double)zrow[g]) * oracle_half_to_double(srow[g]);
    }
}

int oracle_dequant(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                   int64_t rows, int K, int wbits, int group, double *w)
{
    if (!codes || !scales || !zeros || !w || rows < 0 || K <= 0 || group <= 0 || K % group ||
        (wbits != 4 && wbits != 2))
        return -1;
    int64_t rb = (int64_t)K * wbits / 8, gb = K / group;
    for (int64_t r = 0; r < rows; r++)
        dequant_row(codes + r * rb, scales + r * gb, zeros + r * gb, K, wbits, group, w + r * K);
    return 0;
}

/* ------------------------------------------------------- router logits */

/* fp16 value = M * 2^(sh - 24), M a signed integer with |M| < 2^11, sh in [0, 29]. */
static inline void half_split(uint16_t h, int64_t *M, int *sh)
{
    int e = (h >> 10) & 0x1f, f = h & 0x3ff;
    int64_t m = e ? (f | 0x400) : f;
    *M = (h & 0x8000) ? -m : m;
    *sh = (e ? e : 1) - 1;
}

/* |c * 2^48 - s| for a finite fp32 c, as an exact integer at the common
 * scale 2^sh (sh <= 0 when c has bits below 2^-48): the distance of a
 * candidate from the exact sum, compared between candidates of one sum. */
static unsigned __int128 scaled_distance(float c, __int128 s, int sh)
{
    int e;
    const float m = frexpf(c, &e);            /* c = m * 2^e, |m| in [0.5, 1) */
    const int64_t M = (int64_t)ldexpf(m, 24); /* integer significand: c = M * 2^(e - 24) */
    /* c * 2^48 = M * 2^(e + 24); bring both sides to the scale 2^sh */
    const int up = e + 24 - sh;               /* >= 0 by the choice of sh */
    const __int128 a = (__int128)M * ((__int128)1 << up);
    const __int128 b = s * ((__int128)1 << (-sh));
    const __int128 d = a - b;
    return d < 0 ? (unsigned __int128)(-d) : (unsigned __int128)d;
}

/* s * 2^-48 rounded once to fp32, to nearest, ties to the even significand.
 * A first guess through double lies within one fp32 step of the answer, so
 * the answer is the guess or one of its two neighbours: the one nearest to
 * the exact value, compared exactly in 128-bit integers. */
static float nearest_f32_of_scaled(__int128 s)
{
    if (s == 0)
        return 0.0f;
    const float guess = (float)ldexp((double)s, -48);
    const float cand[3] = {nextafterf(guess, -INFINITY), guess, nextafterf(guess, INFINITY)};
    int sh = 0;                               /* common scale: the finest candidate's bit */
    for (int i = 0; i < 3; i++) {
        int e;
        frexpf(cand[i], &e);
        if (e + 24 < sh)
            sh = e + 24;
    }
    float best = cand[0];
    unsigned __int128 bd = scaled_distance(cand[0], s, sh);
    for (int i = 1; i < 3; i++) {
        const unsigned __int128 d = scaled_distance(cand[i], s, sh);
        uint32_t bits;
        memcpy(&bits, &cand[i], sizeof bits);
        if (d < bd || (d == bd && (bits & 1u) == 0)) {
            best = cand[i];
            bd = d;
        }
    }
    return best;
}

/* Exact dot product of two fp16 vectors, rounded once to fp32. */
static float exact_dot_f32(const uint16_t *a, const uint16_t *b, int n)
{
    __int128 acc = 0;
    for (int i = 0; i < n; i++) {
        int64_t ma, mb;
        int sa, sb;
        half_split(a[i], &ma, &sa);
        half_split(b[i], &mb, &sb);
        acc += (__int128)(ma * mb) << (sa + sb);
    }
    return nearest_f32_of_scaled(acc);
}

int oracle_router_logits(const uint16_t *x, int n, int H, const uint16_t *router_w,
                         const float *bias, int E, float *logits)
{
    if (!x || !router_w || !logits || n < 0 || H <= 0 || E <= 0)
        return -1;
#pragma omp parallel for schedule(static) collapse(2)
    for (int t = 0; t < n; t++)
        for (int e = 0; e < E; e++) {
            float l = exact_dot_f32(x + (int64_t)t * H, router_w + (int64_t)e * H, H);
            if (bias) {
                volatile float lb = l + bias[e]; /* one IEEE fp32 add */
                l = lb;
            }
            logits[(int64_t)t * E + e] = l;
        }
    return 0;
}

/* -------------------------------------------------------- top-k, softmax */

int oracle_topk(const float *logits, int n, int E, int k, int32_t *idx, float *w32, double *w64)
{
    if (!logits || !idx || n < 0 || E <= 0 || k < 1 || k > E)
        return -1;
    char *taken = (char *)malloc((size_t)E);
    if (!taken)
        return -2;
    for (int t = 0; t < n; t++) {
        const float *l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])  /* strict: ties keep the lower id */
                    best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
        }
        double mx = l[idx[(int64_t)t * k]], den = 0.0;
        for (int j = 0; j < k; j++)
            den += exp((double)l[idx[(int64_t)t * k + j]] - mx);
        for (int j = 0; j < k; j++) {
            double wj = exp((double)l[idx[(int64_t)t * k + j]] - mx) / den;
            if (w64)
                w64[(int64_t)t * k + j] = wj;
            if (w32)
                w32[(int64_t)t * k + j] = (float)wj;
        }
    }
    free(taken);
    return 0;
}

/* ---------------------------------------------------------- grouping */

int oracle_group(const int32_t *idx, int n, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm)
{
    if (!idx || !counts || !offsets || !perm || n < 0 || k < 1 || E < 1)
        return -1;
    int64_t P = (int64_t)n * k;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t p = 0; p < P; p++) {
        if (idx[p] < 0 || idx[p] >= E)
            return -1;
        counts[idx[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!next)
        return -2;
    memcpy(next, offsets, sizeof(int32_t) * (size_t)E);
    for (int64_t p = 0; p < P; p++) /* in pair order: stable */
        perm[next[idx[p]]++] = (int32_t)p;
    free(next);
    return 0;
}

/* ------------------------------------------------------- expert FFN */

/* One expert (matrices given by pointers to its gate/up/down slices) on T
 * token vectors xs [T][H] (double): y [T][H] = W_down (silu(W_gate x) * (W_up x)). */
static int expert_ffn(const uint8_t *const codes[3], const uint16_t *const scales[3],
                      const uint8_t *const zeros[3], int H, int I, int wbits, int group,
                      const double *xs, int T, double *y)
{
    if (T == 0)
        return 0;
    double *h = (double *)malloc(sizeof(double) * (size_t)T * I);
    if (!h)
        return -2;
    int64_t rb_gu = (int64_t)H * wbits / 8, gb_gu = H / group;
    int64_t rb_d = (int64_t)I * wbits / 8, gb_d = I / group;
    int err = 0;
#pragma omp parallel
    {
        double *wg = (double *)malloc(sizeof(double) * (size_t)H);
        double *wu = (double *)malloc(sizeof(double) * (size_t)H);
        double *wd = (double *)malloc(sizeof(double) * (size_t)I);
        if (!wg || !wu || !wd) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(static)
            for (int i = 0; i < I; i++) {
                dequant_row(codes[0] + i * rb_gu, scales[0] + i * gb_gu, zeros[0] + i * gb_gu, H,
                            wbits, group, wg);
                dequant_row(codes[1] + i * rb_gu, scales[1] + i * gb_gu, zeros[1] + i * gb_gu, H,
                            wbits, group, wu);
                for (int t = 0; t < T; t++) {
                    const double *x = xs + (int64_t)t * H;
                    double g = 0.0, u = 0.0;
                    for (int c = 0; c < H; c++) {
                        g += wg[c] * x[c];
                        u += wu[c] * x[c];
                    }
                    h[(int64_t)t * I + i] = g / (1.0 + exp(-g)) * u;
                }
            }
#pragma omp for schedule(static)
            for (int r = 0; r < H; r++) {
                dequant_row(codes[2] + r * rb_d, scales[2] + r * gb_d, zeros[2] + r * gb_d, I,
                            wbits, group, wd);
                for (int t = 0; t < T; t++) {
                    const double *hv = h + (int64_t)t * I;
                    double acc = 0.0;
                    for (int c = 0; c < I; c++)
                        acc += wd[c] * hv[c];
                    y[(int64_t)t * H + r] = acc;
                }
            }
        }
        free(wg);
        free(wu);
        free(wd);
    }
    free(h);
    return err;
}

/* Pointers to expert e's slices of the stacked matrices. */
static void expert_slices(const oracle_layer_t *L, int e, int shared, const uint8_t *c[3],
                          const uint16_t *s[3], const uint8_t *z[3], int *inter)
{
    int I = shared ? L->shared_inter : L->inter, H = L->hidden;
    *inter = I;
    for (int m = 0; m < 3; m++) {
        int rows = m < 2 ? I : H, K = m < 2 ? H : I;
        int64_t cb = (int64_t)rows * K * L->wbits / 8, gb = (int64_t)rows * (K / L->group);
        if (shared) {
            c[m] = L->sh_codes[m];
            s[m] = L->sh_scales[m];
            z[m] = L->sh_zeros[m];
        } else {
            c[m] = L->codes[m] + (int64_t)e * cb;
            s[m] = L->scales[m] + (int64_t)e * gb;
            z[m] = L->zeros[m] + (int64_t)e * gb;
        }
    }
}

int oracle_expert_ffn(const oracle_layer_t *L, int e, const uint16_t *x, int T, double *y)
{
    if (!L || !x || !y || T < 0 || (e < 0 && !L->has_shared) || e >= L->n_experts)
        return -1;
    const uint8_t *c[3], *z[3];
    const uint16_t *s[3];
    int I;
    expert_slices(L, e < 0 ? 0 : e, e < 0, c, s, z, &I);
    int H = L->hidden;
    double *xs = (double *)malloc(sizeof(double) * (size_t)T * H + 8);
    if (!xs)
        return -2;
    for (int64_t i = 0; i < (int64_t)T * H; i++)
        xs[i] = oracle_half_to_double(x[i]);
    int rc = expert_ffn(c, s, z, H, I, L->wbits, L->group, xs, T, y);
    free(xs);
    return rc;
}

static int check_layer(const oracle_layer_t *L)
{
    if (!L || L->hidden <= 0 || L->inter <= 0 || L->n_experts <= 0 || L->top_k < 1 ||
        L->top_k > L->n_experts || L->group <= 0 || L->hidden % L->group ||
        L->inter % L->group || (L->wbits != 4 && L->wbits != 2) || !L->router_w)
        return -1;
    for (int m = 0; m < 3; m++)
        if (!L->codes[m] || !L->scales[m] || !L->zeros[m])
            return -1;
    if (L->has_shared) {
        if (L->shared_inter <= 0 || L->shared_inter % L->group || !L->sh_gate_w)
            return -1;
        for (int m = 0; m < 3; m++)
            if (!L->sh_codes[m] || !L->sh_scales[m] || !L->sh_zeros[m])
                return -1;
    }
    return 0;
}

/* --------------------------------------------------------- forward */

int oracle_forward(const oracle_layer_t *L, const uint16_t *x, int n, const int32_t *tokens,
                   int n_sel, float *logits, int32_t *idx, float *w32, int32_t *counts,
                   int32_t *offsets, int32_t *perm, double *out64, uint16_t *out16)
{
    if (check_layer(L) || !x || n < 0 || (n_sel > 0 && !tokens && n_sel != n))
        return -1;
    const int H = L->hidden, E = L->n_experts, k = L->top_k;
    const int64_t P = (int64_t)n * k;
    int rc = 0;
    float *lg = (float *)malloc(sizeof(float) * ((size_t)n * E + 1));
    int32_t *id = (int32_t *)malloc(sizeof(int32_t) * ((size_t)P + 1));
    double *w = (double *)malloc(sizeof(double) * ((size_t)P + 1));
    int32_t *cnt = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * ((size_t)E + 1));
    int32_t *pm = (int32_t *)malloc(sizeof(int32_t) * ((size_t)P + 1));
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * ((size_t)n + 1));
    if (!lg || !id || !w || !cnt || !off || !pm || !sel) {
        rc = -2;
        goto done;
    }
    /* router, top-k, weights, grouping for every token */
    if ((rc = oracle_router_logits(x, n, H, L->router_w, L->router_bias, E, lg)))
        goto done;
    if ((rc = oracle_topk(lg, n, E, k, id, NULL, w)))
        goto done;
    if ((rc = oracle_group(id, n, k, E, cnt, off, pm)))
        goto done;
    if (logits)
        memcpy(logits, lg, sizeof(float) * (size_t)n * E);
    if (idx)
        memcpy(idx, id, sizeof(int32_t) * (size_t)P);
    if (w32)
        for (int64_t p = 0; p < P; p++)
            w32[p] = (float)w[p];
    if (counts)
        memcpy(counts, cnt, sizeof(int32_t) * (size_t)E);
    if (offsets)
        memcpy(offsets, off, sizeof(int32_t) * ((size_t)E + 1));
    if (perm)
        memcpy(perm, pm, sizeof(int32_t) * (size_t)P);
    if (!out64 && !out16)
        goto done;

    /* expert FFNs for the selected tokens, expert by expert */
    int ns = n_sel > 0 ? n_sel : 0;
    for (int i = 0; i < ns; i++) {
        sel[i] = tokens ? tokens[i] : i;
        if (sel[i] < 0 || sel[i] >= n) {
            rc = -1;
            goto done;
        }
    }
    double *acc = (double *)calloc((size_t)ns * H + 1, sizeof(double));
    double *xs = (double *)malloc(sizeof(double) * ((size_t)ns * H + 1));
    double *ys = (double *)malloc(sizeof(double) * ((size_t)ns * H + 1));
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * ((size_t)ns + 1));
    double *wt = (double *)malloc(sizeof(double) * ((size_t)ns + 1));
    /* contributions per selected token and slot, summed in slot order below */
    double *yslot = (double *)malloc(sizeof(double) * ((size_t)ns * k * H + 1));
    if (!acc || !xs || !ys || !rows || !wt || !yslot) {
        rc = -2;
        goto ffn_done;
    }
    for (int e = 0; e < E && !rc; e++) {
        int T = 0;
        for (int i = 0; i < ns; i++)
            for (int j = 0; j < k; j++)
                if (id[(int64_t)sel[i] * k + j] == e) {
                    rows[T] = i * k + j;
                    for (int c = 0; c < H; c++)
                        xs[(int64_t)T * H + c] =
                            oracle_half_to_double(x[(int64_t)sel[i] * H + c]);
                    T++;
                }
        if (!T)
            continue;
        const uint8_t *c3[3], *z3[3];
        const uint16_t *s3[3];
        int I;
        expert_slices(L, e, 0, c3, s3, z3, &I);
        rc = expert_ffn(c3, s3, z3, H, I, L->wbits, L->group, xs, T, ys);
        for (int r = 0; r < T && !rc; r++)
            memcpy(yslot + (int64_t)rows[r] * H, ys + (int64_t)r * H, sizeof(double) * H);
    }
    if (rc)
        goto ffn_done;
    /* out = x + sum_j w_j y_j (+ gate * y_shared) */
    for (int i = 0; i < ns; i++)
        for (int c = 0; c < H; c++) {
            double v = oracle_half_to_double(x[(int64_t)sel[i] * H + c]);
            for (int j = 0; j < k; j++)
                v += w[(int64_t)sel[i] * k + j] * yslot[((int64_t)i * k + j) * H + c];
            acc[(int64_t)i * H + c] = v;
        }
    if (L->has_shared) {
        for (int i = 0; i < ns; i++) {
            double z = 0.0;
            for (int c = 0; c < H; c++) {
                xs[(int64_t)i * H + c] = oracle_half_to_double(x[(int64_t)sel[i] * H + c]);
                z += xs[(int64_t)i * H + c] * oracle_half_to_double(L->sh_gate_w[c]);
            }
            wt[i] = 1.0 / (1.0 + exp(-z));
        }
        const uint8_t *c3[3], *z3[3];
        const uint16_t *s3[3];
        int I;
        expert_slices(L, 0, 1, c3, s3, z3, &I);
        rc = expert_ffn(c3, s3, z3, H, I, L->wbits, L->group, xs, ns, ys);
        for (int i = 0; i < ns && !rc; i++)
            for (int c = 0; c < H; c++)
                acc[(int64_t)i * H + c] += wt[i] * ys[(int64_t)i * H + c];
    }
    if (!rc)
        for (int64_t i = 0; i < (int64_t)ns * H; i++) {
            if (out64)
                out64[i] = acc[i];
            if (out16)
                out16[i] = oracle_double_to_half(acc[i]);
        }
ffn_done:
    free(acc);
    free(xs);
    free(ys);
    free(rows);
    free(wt);
    free(yslot);
done:
    free(lg);
    free(id);
    free(w);
    free(cnt);
    free(off);
    free(pm);
    free(sel);
    return rc;
}

/* ------------------------------------------------------------- RMSNorm */

/* Two-pass RMSNorm of rows r [n][H] with gain g [H] ("Flash-MoE" article,
 * section 3: a two-pass RMSNorm in front of the router): pass 1 the mean
 * square of the row, pass 2 the scaled row,
 *   xn_h = fp16( r_h * g_h / sqrt(mean_h(r_h^2) + eps) ).
 * [reading] The pages give no precision: this is the plain definition in
 * fp64, rounded once to fp16 (nearest even). */
int oracle_rmsnorm(const uint16_t *r, const uint16_t *g, float eps, int n, int H, uint16_t *xn)
{
    if (!r || !g || !xn || n < 0 || H <= 0)
        return -1;
    for (int t = 0; t < n; t++) {
        const uint16_t *row = r + (int64_t)t * H;
        double sq = 0.0;
        for (int h = 0; h < H; h++) {
            const double v = oracle_half_to_double(row[h]);
            sq += v * v;
        }
        const double rs = 1.0 / sqrt(sq / H + (double)eps);
        for (int h = 0; h < H; h++)
            xn[(int64_t)t * H + h] = oracle_double_to_half(
                oracle_half_to_double(row[h]) * rs * oracle_half_to_double(g[h]));
    }
    return 0;
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
