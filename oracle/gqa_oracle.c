/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for the forward pass of a
 * grouped-query attention layer whose head_dim is set independently of
 * hidden / num_heads (Qwen3-style attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  The product (the CUDA
 * library) neither links nor calls it, and this file shares no code, header
 * or table with it.
 *
 * Conventions
 *   - Every tensor input is bf16 (IEEE binary32 with the low 16 bits
 *     dropped), passed as uint16_t bit patterns, and widened to double
 *     exactly.  All arithmetic is double; nothing is rounded in between.
 *   - Loops follow the definitions in the order the pages state them; the
 *     only liberty taken is running independent output rows on OpenMP
 *     threads, which does not change any single row's arithmetic.
 *   - Sources are cited as: page title, section.
 *       [NeoX]  "Support explicit attention head_dim independent of
 *                hidden_size / num_attention_heads" (GPT-NeoX issue 1434)
 *       [T07]   "Tutorial 07: Multi-Head and Grouped-Query Attention (Full Layer)"
 *       [Knob]  "num_heads Is Not a Capacity Knob"
 *       [Part]  "Attention head partitions: keep each head's dependencies intact"
 *
 * Readings taken where the pages are silent (each is pinned by a test in
 * tests/test_oracle_pins.py, and listed with its reason in the design notes):
 *   R1 fused weight row order: all Q heads, then all K heads, then all V heads
 *      ([NeoX] "Fused QKV projection": the fused output is
 *      query_hidden_size + 2*kv_hidden_size; [NeoX] "Checkpoint conversion"
 *      gives q_proj/k_proj/v_proj as separate [out, hidden] matrices).
 *   R2 query head j uses KV head g = j / (Hq/Hkv) (contiguous groups;
 *      [NeoX] "Qwen3-0.6B example": each KV head serves 2 query heads).
 *   R3 RMSNorm(v) = v * w / sqrt(mean(v^2) + eps), mean over head_dim.
 *   R4 RoPE pairs element i with element i + d/2 ("rotate half"), angle
 *      pos * theta^(-2i/d), applied to Q and K only ([T07] §3-§4).
 *   R5 causal: query at position t sees keys u <= t, the diagonal included.
 *   R6 out = x + o_proj(attn) ([NeoX] "Qwen3-0.6B example": residual addition).
 *   R16 partial rotary: with rotary_dim rd (even, 0 <= rd <= d) the rotation
 *      of R4 acts on the first rd features only, pairing i with i + rd/2 at
 *      angle pos * theta^(-2i/rd); features [rd, d) pass unchanged; rd = d is
 *      R4 ([NeoX] "Scaling and RoPE": RoPE is built from the effective
 *      head_dim, subject to the rotary_pct setting and an even dimension).
 *      The functions named *_rd take rd; the others use rd = d.
 *   R17 FP8 KV cache (decode): one OCP FP8 E4M3 code per cached element times
 *      one scale per tensor (k_scale, v_scale); a value enters as the nearest
 *      code to value / scale, ties to even, saturating at +-448; the new
 *      token's key and value are appended as codes and attended like the
 *      rest ("Head Dimension" article, §5.2: FP8 for the K, V cache).
 *   R21 a bf16 KV cache (decode, prefill into a cache): the new tokens' keys
 *      and values are stored in the cache as bf16 (nearest value, ties to
 *      even) and attention reads them back from it, as it reads the earlier
 *      entries ([T07] §4 step 5: the cache's update-and-fetch returns what the
 *      cache holds and the attention of step 6 consumes that; R17 does the
 *      same for an FP8 cache).
 *   R19 backward: the gradients are the derivatives of the forward steps
 *      above in reverse order (the pages print none); a KV head's K and V
 *      gradients sum over the query heads of its group.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EARG (-1)
#define ORACLE_ENOMEM (-2)

/* bf16 bit pattern -> double.  Exact: a bf16 value is a binary32 value. */
static double bf(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* x rounded to the nearest bf16 value (8 significant bits, ties to even).
 * bf16 has binary32's exponent range: below 2^-126 the spacing stays 2^-133
 * (subnormals), and values rounding past the largest finite bf16,
 * (2 - 2^-7) * 2^127, become infinite (R21). */
static double round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                   /* |x| in [2^(e-1), 2^e) */
    if (e < -125) e = -125;
    double q = ldexp(1.0, e - 8);   /* spacing of 8 significant bits */
    double r = nearbyint(x / q) * q;
    if (fabs(r) > 0x1.fep127) return copysign(INFINITY, x);
    return r;
}

int oracle_round_bf16(const double *x, long n, double *out)
{
    if (!x || !out || n < 0) return ORACLE_EARG;
    for (long i = 0; i < n; ++i) out[i] = round_bf16(x[i]);
    return ORACLE_OK;
}

/* IEEE binary16 bit pattern -> double, exact (subnormals, infinities, NaN). */
static double h16(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* 16-bit pattern of either format -> double. */
static double w16(uint16_t h, int f16) { return f16 ? h16(h) : bf(h); }

/* Exported for the pin against numpy's float16 conversion. */
void oracle_f16_to_double(const uint16_t *h, long n, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = h16(h[i]);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* ------------------------------------------------------------------------ */
/* Shape and cost arithmetic ([NeoX] "Proposed implementation",
 * [Knob] "Why the cost does not move", "Where the invariance breaks").     */
/* ------------------------------------------------------------------------ */

/* Effective head width: explicit value, else hidden // heads
 * ([NeoX] "Proposed configuration behavior").  Returns -1 when it has to be
 * derived and hidden is not divisible by heads. */
long oracle_effective_head_dim(long hidden, long heads, long head_dim_or_0)
{
    if (head_dim_or_0 > 0) return head_dim_or_0;
    if (heads <= 0 || hidden % heads != 0) return -1;
    return hidden / heads;
}

/* Widths of the projections ([NeoX] "Proposed implementation", "Fused QKV
 * projection", "Output projection"):
 *   out[0] = query_hidden = Hq*d, out[1] = kv_hidden = Hkv*d,
 *   out[2] = fused QKV output width = Hq*d + 2*Hkv*d,
 *   out[3] = o_proj input width = Hq*d, out[4] = o_proj output = hidden. */
void oracle_widths(long hidden, long Hq, long Hkv, long d, long *out)
{
    out[0] = Hq * d;
    out[1] = Hkv * d;
    out[2] = Hq * d + 2 * Hkv * d;
    out[3] = Hq * d;
    out[4] = hidden;
}

/* Weight count of q_proj, k_proj, v_proj and o_proj
 * ([Knob] "Why the cost does not move": 4*d_model^2 when d = d_model/h;
 * "Where the invariance breaks": more when d is pinned). */
long long oracle_attn_param_count(long hidden, long Hq, long Hkv, long d)
{
    long long h = hidden;
    return h * (long long)(Hq * d) + 2 * h * (long long)(Hkv * d) + (long long)(Hq * d) * h;
}

/* Projection multiply-accumulates per token: every weight is used once per
 * token ([Knob] "Why the cost does not move", the 1,048,576 at d_model 512). */
long long oracle_proj_macs_per_token(long hidden, long Hq, long Hkv, long d)
{
    return oracle_attn_param_count(hidden, Hq, Hkv, d);
}

/* Score + value multiply-accumulates per query token over n keys: each
 * query head does n*d for the scores and n*d for the value average
 * ([Knob] "Why the cost does not move": 2*n*h*d_k). */
long long oracle_score_value_macs_per_token(long n, long Hq, long d)
{
    return 2LL * n * Hq * d;
}

/* ------------------------------------------------------------------------ */
/* The steps of the layer, one function each.                                */
/* ------------------------------------------------------------------------ */

/* y[n] = sum_k xrow[k] * W[n][k]  for n in [n0, n0+nn): one row of x @ W^T
 * (W stored [out, in]: [NeoX] "Checkpoint conversion"; [T07] §4 step 1,
 * "Each projection is a linear layer: x @ W^T"). */
static void linear_row(const uint16_t *xrow, const uint16_t *W, long n0, long nn,
                       long K, double *y)
{
    for (long n = 0; n < nn; ++n) {
        const uint16_t *w = W + (n0 + n) * K;
        double s = 0.0;
        for (long k = 0; k < K; ++k) s += bf(xrow[k]) * bf(w[k]);
        y[n] = s;
    }
}

/* RMSNorm over one head vector of length d, in place (reading R3):
 * v <- v * w / sqrt(mean(v^2) + eps)   ([T07] §3 "QK-Norm"). */
static void rmsnorm_head(double *v, long d, const uint16_t *w, double eps)
{
    double ms = 0.0;
    for (long i = 0; i < d; ++i) ms += v[i] * v[i];
    ms /= (double)d;
    double r = 1.0 / sqrt(ms + eps);
    for (long i = 0; i < d; ++i) v[i] = v[i] * r * bf(w[i]);
}

/* RoPE on the first rd features of one head vector at position pos, in
 * place (readings R4, R16): for i < rd/2, angle f = pos * theta^(-2i/rd),
 *   (v[i], v[i+rd/2]) <- (v[i] cos f - v[i+rd/2] sin f, v[i+rd/2] cos f + v[i] sin f);
 * features from rd on are not touched.
 * ([T07] §4 "Set up RoPE" from (head_dim, max_position, rope_theta);
 *  [NeoX] "Scaling and RoPE": built from the effective head_dim). */
static void rope_head(double *v, long rd, double pos, double theta)
{
    long half = rd / 2;
    for (long i = 0; i < half; ++i) {
        double f = pos * pow(theta, -2.0 * (double)i / (double)rd);
        double c = cos(f), s = sin(f);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

/* Exported single-row helpers so the pins can test each step alone. */
int oracle_rmsnorm_rows(const double *in, long nrows, long d, const uint16_t *w,
                        double eps, double *out)
{
    if (!in || !out || !w || nrows < 0 || d <= 0) return ORACLE_EARG;
    for (long r = 0; r < nrows; ++r) {
        memcpy(out + r * d, in + r * d, (size_t)d * sizeof(double));
        rmsnorm_head(out + r * d, d, w, eps);
    }
    return ORACLE_OK;
}

int oracle_rope_rows_rd(const double *in, long nrows, long d, long rd, const double *pos,
                        double theta, double *out)
{
    if (!in || !out || !pos || nrows < 0 || d <= 0 || (d & 1)) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    for (long r = 0; r < nrows; ++r) {
        memcpy(out + r * d, in + r * d, (size_t)d * sizeof(double));
        rope_head(out + r * d, rd, pos[r], theta);
    }
    return ORACLE_OK;
}

int oracle_rope_rows(const double *in, long nrows, long d, const double *pos,
                     double theta, double *out)
{
    return oracle_rope_rows_rd(in, nrows, d, d, pos, theta, out);
}

int oracle_linear(const uint16_t *x, const uint16_t *W, long M, long N, long K,
                  double *y, int nthreads)
{
    if (!x || !W || !y || M < 0 || N <= 0 || K <= 0) return ORACLE_EARG;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m) linear_row(x + m * K, W, 0, N, K, y + m * N);
    return ORACLE_OK;
}

/* One query row of grouped-query attention ([T07] §4 step 6, computed in
 * full precision; [NeoX] "Scaling and RoPE": scale head_dim^-0.5;
 * [Part]: every query head sees all permitted keys of its KV group):
 *   s_u = <q, k_u> / sqrt(d) for the visible keys u in [0, n_vis),
 *   o   = sum_u softmax(s)_u v_u.
 * kget/vget address key u of the group; q and o have length d.
 * The maximum is subtracted before exp, which leaves softmax unchanged. */
typedef struct {
    const uint16_t *kb;   /* 16-bit keys, row stride d, or NULL */
    const uint16_t *vb;
    const double *kd;     /* double keys (used for keys >= n_bf16), or NULL */
    const double *vd;
    long n_bf16;          /* keys [0, n_bf16) come from kb/vb (or k8/v8), the rest from kd/vd */
    int f16;              /* kb/vb hold binary16 (1) or bf16 (0) patterns */
    const uint8_t *k8;    /* FP8 E4M3 keys and values (used instead of kb/vb when k8 != NULL), */
    const uint8_t *v8;    /* each code worth e4m3(code) * ks (keys) or * vs (values) */
    double ks, vs;
} kv_src;

static double e4m3(uint8_t code);

static double key_at(const kv_src *s, long u, long c, long d)
{
    if (u >= s->n_bf16) return s->kd[(u - s->n_bf16) * d + c];
    return s->k8 ? e4m3(s->k8[u * d + c]) * s->ks : w16(s->kb[u * d + c], s->f16);
}
static double val_at(const kv_src *s, long u, long c, long d)
{
    if (u >= s->n_bf16) return s->vd[(u - s->n_bf16) * d + c];
    return s->v8 ? e4m3(s->v8[u * d + c]) * s->vs : w16(s->vb[u * d + c], s->f16);
}

static int attend_row(const double *q, const kv_src *src, long n_vis, long d, double *o)
{
    double *s = (double *)malloc((size_t)(n_vis > 0 ? n_vis : 1) * sizeof(double));
    if (!s) return ORACLE_ENOMEM;
    double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (long u = 0; u < n_vis; ++u) {
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += q[c] * key_at(src, u, c, d);
        s[u] = dot * scale;
        if (s[u] > mx) mx = s[u];
    }
    double den = 0.0;
    for (long u = 0; u < n_vis; ++u) {
        s[u] = exp(s[u] - mx);
        den += s[u];
    }
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    for (long u = 0; u < n_vis; ++u) {
        double p = s[u] / den;
        for (long c = 0; c < d; ++c) o[c] += p * val_at(src, u, c, d);
    }
    free(s);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Stage 1: QKV projection + QK-norm + RoPE, for every token.               */
/* ------------------------------------------------------------------------ */

/* q_out [B,Hq,S,d], k_out/v_out [B,Hkv,S,d] (head-major, [T07] §4 step 4).
 * q_norm_w/k_norm_w both NULL means no QK-norm.  Positions are 0..S-1. */
int oracle_qkv_stage_rd(const uint16_t *x, const uint16_t *Wqkv,
                     const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                     double rope_theta, double eps, long rd,
                     long B, long S, long hidden, long Hq, long Hkv, long d,
                     double *q_out, double *k_out, double *v_out, int nthreads)
{
    if (!x || !Wqkv || !q_out || !k_out || !v_out) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1)) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    long NQ = Hq * d, NKV = Hkv * d, N = NQ + 2 * NKV;
    int err = ORACLE_OK;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < B * S; ++m) {
        long b = m / S, t = m % S;
        double *row = (double *)malloc((size_t)N * sizeof(double));
        if (!row) { err = ORACLE_ENOMEM; continue; }
        /* step 1: fused projection, rows of Wqkv = [W_q; W_k; W_v] (R1) */
        linear_row(x + m * hidden, Wqkv, 0, N, hidden, row);
        for (long j = 0; j < Hq; ++j) {
            double *v = row + j * d;
            if (q_norm_w) rmsnorm_head(v, d, q_norm_w, eps);   /* step 2 */
            rope_head(v, rd, (double)t, rope_theta);             /* step 3 */
            memcpy(q_out + ((b * Hq + j) * S + t) * d, v, (size_t)d * sizeof(double));
        }
        for (long g = 0; g < Hkv; ++g) {
            double *v = row + NQ + g * d;
            if (k_norm_w) rmsnorm_head(v, d, k_norm_w, eps);
            rope_head(v, rd, (double)t, rope_theta);
            memcpy(k_out + ((b * Hkv + g) * S + t) * d, v, (size_t)d * sizeof(double));
            memcpy(v_out + ((b * Hkv + g) * S + t) * d, row + NQ + NKV + g * d,
                   (size_t)d * sizeof(double));
        }
        free(row);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Stage 2: causal grouped-query attention over 16-bit Q/K/V.               */
/* ------------------------------------------------------------------------ */

/* Q [B,Hq,S,d], K/V [B,Hkv,S,d], all bf16 (in_f16 = 0) or all IEEE binary16
 * (in_f16 = 1); either is widened to double exactly.  attn [n_sel, Hq*d] for the selected
 * tokens sel[i] = b*S + t (flattened, [T07] §4 step 7 "(batch, seq,
 * heads*head_dim)"; [NeoX] "Attention output flattening").  sel == NULL
 * means every token in order (n_sel must then be B*S). */
int oracle_attention_stage(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int in_f16,
                           long B, long S, long Hq, long Hkv, long d, int causal,
                           const long *sel, long n_sel, double *attn, int nthreads)
{
    if (!Q || !K || !V || !attn) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return ORACLE_EARG;
    if (!sel && n_sel != B * S) return ORACLE_EARG;
    long G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long i = 0; i < n_sel; ++i) {
        for (long j = 0; j < Hq; ++j) {
            long m = sel ? sel[i] : i;
            long b = m / S, t = m % S;
            long g = j / G;                                   /* R2 */
            double q[1024];
            if (d > 1024) { err = ORACLE_EARG; continue; }
            for (long c = 0; c < d; ++c) q[c] = w16(Q[((b * Hq + j) * S + t) * d + c], in_f16);
            kv_src src = {K + (b * Hkv + g) * S * d, V + (b * Hkv + g) * S * d, NULL, NULL, S, in_f16};
            long n_vis = causal ? t + 1 : S;                  /* R5 */
            int e = attend_row(q, &src, n_vis, d, attn + i * Hq * d + j * d);
            if (e) err = e;
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Stage 3: o_proj + residual.                                               */
/* ------------------------------------------------------------------------ */

/* out[i] = x[m] + attn[m] @ Wo^T for the selected tokens m = sel[i]
 * ([NeoX] "Output projection", "Qwen3-0.6B example" residual addition, R6).
 * attn [M, Hq*d] bf16, Wo [hidden, Hq*d] bf16, x [M, hidden] bf16. */
int oracle_oproj_stage(const uint16_t *attn, const uint16_t *Wo, const uint16_t *x,
                       long M, long hidden, long QW, const long *sel, long n_sel,
                       double *out, int nthreads)
{
    if (!attn || !Wo || !x || !out || M <= 0 || hidden <= 0 || QW <= 0) return ORACLE_EARG;
    if (!sel && n_sel != M) return ORACLE_EARG;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n_sel; ++i) {
        long m = sel ? sel[i] : i;
        linear_row(attn + m * QW, Wo, 0, hidden, QW, out + i * hidden);
        for (long n = 0; n < hidden; ++n) out[i * hidden + n] += bf(x[m * hidden + n]);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The whole layer, prefill.                                                 */
/* ------------------------------------------------------------------------ */

/* Keys and values for all tokens (they are needed by every later query),
 * then Q, attention and o_proj for the selected tokens only.  With
 * sel == NULL every token is computed.  Any of q_sel [n_sel,Hq,d],
 * attn_sel [n_sel,Hq*d], k_all/v_all [B,Hkv,S,d] may be NULL.
 * out_sel [n_sel, hidden] is required. */
int oracle_forward_rd(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                   const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                   double rope_theta, double eps, long rd,
                   long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                   const long *sel, long n_sel,
                   double *q_sel, double *attn_sel, double *out_sel,
                   double *k_all, double *v_all, int nthreads)
{
    if (!x || !Wqkv || !Wo || !out_sel) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1)) return ORACLE_EARG;
    if (Hq % Hkv || d > 1024) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    if (!sel && n_sel != B * S) return ORACLE_EARG;
    long NQ = Hq * d, NKV = Hkv * d, G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);

    double *Kd = k_all, *Vd = v_all;
    if (!Kd) Kd = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    if (!Vd) Vd = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    if (!Kd || !Vd) { err = ORACLE_ENOMEM; goto done; }

    /* keys and values of every token: projection rows [NQ, NQ+2*NKV) */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < B * S; ++m) {
        long b = m / S, t = m % S;
        double *row = (double *)malloc((size_t)(2 * NKV) * sizeof(double));
        if (!row) { err = ORACLE_ENOMEM; continue; }
        linear_row(x + m * hidden, Wqkv, NQ, 2 * NKV, hidden, row);
        for (long g = 0; g < Hkv; ++g) {
            double *k = row + g * d;
            if (k_norm_w) rmsnorm_head(k, d, k_norm_w, eps);
            rope_head(k, rd, (double)t, rope_theta);
            memcpy(Kd + ((b * Hkv + g) * S + t) * d, k, (size_t)d * sizeof(double));
            memcpy(Vd + ((b * Hkv + g) * S + t) * d, row + NKV + g * d, (size_t)d * sizeof(double));
        }
        free(row);
    }

    /* queries, attention and o_proj of the selected tokens */
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n_sel; ++i) {
        long m = sel ? sel[i] : i;
        long b = m / S, t = m % S;
        double *qrow = (double *)malloc((size_t)NQ * sizeof(double));
        double *arow = (double *)malloc((size_t)NQ * sizeof(double));
        if (!qrow || !arow) { err = ORACLE_ENOMEM; free(qrow); free(arow); continue; }
        linear_row(x + m * hidden, Wqkv, 0, NQ, hidden, qrow);
        for (long j = 0; j < Hq; ++j) {
            double *q = qrow + j * d;
            if (q_norm_w) rmsnorm_head(q, d, q_norm_w, eps);
            rope_head(q, rd, (double)t, rope_theta);
            long g = j / G;
            kv_src src = {NULL, NULL, Kd + (b * Hkv + g) * S * d, Vd + (b * Hkv + g) * S * d, 0, 0};
            long n_vis = causal ? t + 1 : S;
            int e = attend_row(q, &src, n_vis, d, arow + j * d);
            if (e) err = e;
        }
        if (q_sel) memcpy(q_sel + i * NQ, qrow, (size_t)NQ * sizeof(double));
        if (attn_sel) memcpy(attn_sel + i * NQ, arow, (size_t)NQ * sizeof(double));
        /* o_proj: out = x + attn @ Wo^T, attn kept in double here */
        for (long n = 0; n < hidden; ++n) {
            const uint16_t *w = Wo + n * NQ;
            double s = 0.0;
            for (long k = 0; k < NQ; ++k) s += arow[k] * bf(w[k]);
            out_sel[i * hidden + n] = bf(x[m * hidden + n]) + s;
        }
        free(qrow);
        free(arow);
    }
done:
    if (Kd && Kd != k_all) free(Kd);
    if (Vd && Vd != v_all) free(Vd);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Decode: one new token per sequence over a KV cache.                       */
/* ------------------------------------------------------------------------ */

/* Attention of one query token per sequence over keys [0, kv_len[b]) of a
 * bf16 cache laid out [B, Hkv, Lmax, d] ([T07] §4 step 5: the cache returns
 * the full history).  q [B,Hq,d] bf16 (q_f16 = 0) or binary16 (q_f16 = 1),
 * widened exactly; attn [B, Hq*d]. */
int oracle_decode_attention_stage(const uint16_t *q, int q_f16, const uint16_t *k_cache,
                                  const uint16_t *v_cache, const int *kv_len,
                                  long B, long Hq, long Hkv, long d, long Lmax,
                                  double *attn, int nthreads)
{
    if (!q || !k_cache || !v_cache || !kv_len || !attn) return ORACLE_EARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || d > 1024 || Hq % Hkv || Lmax <= 0) return ORACLE_EARG;
    for (long b = 0; b < B; ++b)
        if (kv_len[b] <= 0 || kv_len[b] > Lmax) return ORACLE_EARG;
    long G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long j = 0; j < Hq; ++j) {
            long g = j / G;
            double qv[1024];
            for (long c = 0; c < d; ++c) qv[c] = w16(q[(b * Hq + j) * d + c], q_f16);
            kv_src src = {k_cache + (b * Hkv + g) * Lmax * d, v_cache + (b * Hkv + g) * Lmax * d,
                          NULL, NULL, kv_len[b], 0};
            int e = attend_row(qv, &src, kv_len[b], d, attn + b * Hq * d + j * d);
            if (e) err = e;
        }
    }
    return err;
}

/* The whole decode step ([T07] §4 steps 1-7 with L = 1): for each sequence
 * b the new token sits at position p = cache_len[b]; its Q/K are normed and
 * rotated at p; its K/V, as the bf16 cache stores them (R21), join the
 * cached entries [0, p) (read from the bf16 cache, which this function does
 * not modify) and the query attends to all p+1 keys.  x [B, hidden];
 * out [B, hidden].  Optional outputs: q_new [B,Hq,d], k_new/v_new [B,Hkv,d]
 * (the new cache entries), attn [B,Hq*d]. */
int oracle_decode_rd(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                  const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                  double rope_theta, double eps, long rd,
                  long B, long hidden, long Hq, long Hkv, long d,
                  const uint16_t *k_cache, const uint16_t *v_cache, const int *cache_len,
                  long Lmax, double *out, double *q_new, double *k_new, double *v_new,
                  double *attn_out, int nthreads)
{
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !cache_len || !out) return ORACLE_EARG;
    if (B <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1) || d > 1024) return ORACLE_EARG;
    if (Hq % Hkv) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    for (long b = 0; b < B; ++b)
        if (cache_len[b] < 0 || cache_len[b] + 1 > Lmax) return ORACLE_EARG;
    long NQ = Hq * d, NKV = Hkv * d, N = NQ + 2 * NKV, G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
    double *rows = (double *)malloc((size_t)(B * N) * sizeof(double));
    double *arows = (double *)malloc((size_t)(B * NQ) * sizeof(double));
    if (!rows || !arows) { free(rows); free(arows); return ORACLE_ENOMEM; }

#pragma omp parallel for schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        double *row = rows + b * N;
        double p = (double)cache_len[b];
        linear_row(x + b * hidden, Wqkv, 0, N, hidden, row);
        for (long j = 0; j < Hq; ++j) {
            if (q_norm_w) rmsnorm_head(row + j * d, d, q_norm_w, eps);
            rope_head(row + j * d, rd, p, rope_theta);
        }
        for (long g = 0; g < Hkv; ++g) {
            if (k_norm_w) rmsnorm_head(row + NQ + g * d, d, k_norm_w, eps);
            rope_head(row + NQ + g * d, rd, p, rope_theta);
        }
        /* R21: the new key and value as the bf16 cache holds them */
        for (long c = NQ; c < N; ++c) row[c] = round_bf16(row[c]);
    }

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long j = 0; j < Hq; ++j) {
            long g = j / G;
            const double *row = rows + b * N;
            kv_src src = {k_cache + (b * Hkv + g) * Lmax * d, v_cache + (b * Hkv + g) * Lmax * d,
                          row + NQ + g * d, row + NQ + NKV + g * d, cache_len[b], 0};
            int e = attend_row(row + j * d, &src, cache_len[b] + 1, d, arows + b * NQ + j * d);
            if (e) err = e;
        }
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long n = 0; n < hidden; ++n) {
            const uint16_t *w = Wo + n * NQ;
            double s = 0.0;
            for (long k = 0; k < NQ; ++k) s += arows[b * NQ + k] * bf(w[k]);
            out[b * hidden + n] = bf(x[b * hidden + n]) + s;
        }
    }

    for (long b = 0; b < B; ++b) {
        const double *row = rows + b * N;
        if (q_new) memcpy(q_new + b * NQ, row, (size_t)NQ * sizeof(double));
        if (k_new) memcpy(k_new + b * NKV, row + NQ, (size_t)NKV * sizeof(double));
        if (v_new) memcpy(v_new + b * NKV, row + NQ + NKV, (size_t)NKV * sizeof(double));
        if (attn_out) memcpy(attn_out + b * NQ, arows + b * NQ, (size_t)NQ * sizeof(double));
    }
    free(rows);
    free(arows);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Prefill into a KV cache: S new tokens per sequence after p0[b] cached.     */
/* ------------------------------------------------------------------------ */

/* The layer for S new tokens of each sequence b at positions p0[b] .. p0[b]+S-1
 * ([T07] §4: RoPE at the position offsets, step 5 the cache returns the whole
 * history; [Part]: position encodings and masks use the same global token
 * positions).  Keys and values [0, p0[b]) come from the bf16 caches
 * [B, Hkv, Lmax, d] (not modified here); the new tokens' keys and values are
 * computed in double and attended as the bf16 cache stores them (R21).  Query
 * t attends to keys u <= p0[b] + t (causal) or to all p0[b] + S keys.
 * x [B, S, hidden]; out [B, S, hidden].  Optional: k_new/v_new [B, Hkv, S, d]
 * (the new cache entries) and attn [B, S, Hq*d].  With p0 = 0 this is the
 * plain prefill with K and V rounded to bf16; with S = 1 it is the decode
 * step. */
int oracle_prefill_cached_rd(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                          const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                          double rope_theta, double eps, long rd,
                          long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                          const uint16_t *k_cache, const uint16_t *v_cache, const int *p0,
                          long Lmax, double *out, double *k_new, double *v_new, double *attn_out,
                          int nthreads)
{
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !p0 || !out) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1) || d > 1024) return ORACLE_EARG;
    if (Hq % Hkv) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    for (long b = 0; b < B; ++b)
        if (p0[b] < 0 || p0[b] + S > Lmax) return ORACLE_EARG;
    long NQ = Hq * d, NKV = Hkv * d, N = NQ + 2 * NKV, G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
    double *rows = (double *)malloc((size_t)(B * S * N) * sizeof(double));
    double *Kn = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    double *Vn = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    double *arows = (double *)malloc((size_t)(B * S * NQ) * sizeof(double));
    if (!rows || !Kn || !Vn || !arows) { err = ORACLE_ENOMEM; goto done; }

    /* steps 1-3 for every new token, at its global position */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < B * S; ++m) {
        long b = m / S, t = m % S;
        double pos = (double)(p0[b] + t);
        double *row = rows + m * N;
        linear_row(x + m * hidden, Wqkv, 0, N, hidden, row);
        for (long j = 0; j < Hq; ++j) {
            if (q_norm_w) rmsnorm_head(row + j * d, d, q_norm_w, eps);
            rope_head(row + j * d, rd, pos, rope_theta);
        }
        for (long g = 0; g < Hkv; ++g) {
            double *k = row + NQ + g * d;
            if (k_norm_w) rmsnorm_head(k, d, k_norm_w, eps);
            rope_head(k, rd, pos, rope_theta);
            /* R21: the new key and value as the bf16 cache holds them */
            for (long c = 0; c < d; ++c) {
                Kn[((b * Hkv + g) * S + t) * d + c] = round_bf16(k[c]);
                Vn[((b * Hkv + g) * S + t) * d + c] = round_bf16(row[NQ + NKV + g * d + c]);
            }
        }
    }

    /* step 6: cached keys [0, p0) then the new ones */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long m = 0; m < B * S; ++m) {
        for (long j = 0; j < Hq; ++j) {
            long b = m / S, t = m % S, g = j / G;
            kv_src src = {k_cache + (b * Hkv + g) * Lmax * d, v_cache + (b * Hkv + g) * Lmax * d,
                          Kn + (b * Hkv + g) * S * d, Vn + (b * Hkv + g) * S * d, p0[b], 0};
            long n_vis = causal ? p0[b] + t + 1 : p0[b] + S;
            int e = attend_row(rows + m * N + j * d, &src, n_vis, d, arows + m * NQ + j * d);
            if (e) err = e;
        }
    }

    /* step 7: o_proj and the residual */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < B * S; ++m) {
        for (long n = 0; n < hidden; ++n) {
            const uint16_t *w = Wo + n * NQ;
            double s = 0.0;
            for (long k = 0; k < NQ; ++k) s += arows[m * NQ + k] * bf(w[k]);
            out[m * hidden + n] = bf(x[m * hidden + n]) + s;
        }
    }
    if (k_new) memcpy(k_new, Kn, (size_t)(B * Hkv * S * d) * sizeof(double));
    if (v_new) memcpy(v_new, Vn, (size_t)(B * Hkv * S * d) * sizeof(double));
    if (attn_out) memcpy(attn_out, arows, (size_t)(B * S * NQ) * sizeof(double));
done:
    free(rows);
    free(Kn);
    free(Vn);
    free(arows);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Full rotary (rd = d, reading R4): the entry points without _rd.           */
/* ------------------------------------------------------------------------ */

int oracle_qkv_stage(const uint16_t *x, const uint16_t *Wqkv,
                     const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                     double rope_theta, double eps,
                     long B, long S, long hidden, long Hq, long Hkv, long d,
                     double *q_out, double *k_out, double *v_out, int nthreads)
{
    return oracle_qkv_stage_rd(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, d, B, S, hidden, Hq, Hkv, d,
                               q_out, k_out, v_out, nthreads);
}

int oracle_forward(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                   const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                   double rope_theta, double eps,
                   long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                   const long *sel, long n_sel,
                   double *q_sel, double *attn_sel, double *out_sel,
                   double *k_all, double *v_all, int nthreads)
{
    return oracle_forward_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, d, B, S, hidden, Hq, Hkv, d,
                             causal, sel, n_sel, q_sel, attn_sel, out_sel, k_all, v_all, nthreads);
}

int oracle_decode(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                  const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                  double rope_theta, double eps,
                  long B, long hidden, long Hq, long Hkv, long d,
                  const uint16_t *k_cache, const uint16_t *v_cache, const int *cache_len,
                  long Lmax, double *out, double *q_new, double *k_new, double *v_new,
                  double *attn_out, int nthreads)
{
    return oracle_decode_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, d, B, hidden, Hq, Hkv, d,
                            k_cache, v_cache, cache_len, Lmax, out, q_new, k_new, v_new, attn_out, nthreads);
}

int oracle_prefill_cached(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                          const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                          double rope_theta, double eps,
                          long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                          const uint16_t *k_cache, const uint16_t *v_cache, const int *p0,
                          long Lmax, double *out, double *k_new, double *v_new, double *attn_out,
                          int nthreads)
{
    return oracle_prefill_cached_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, d, B, S, hidden, Hq,
                                    Hkv, d, causal, k_cache, v_cache, p0, Lmax, out, k_new, v_new, attn_out,
                                    nthreads);
}

/* ------------------------------------------------------------------------ */
/* FP8 KV cache for decode.                                                  */
/* ------------------------------------------------------------------------ */

/* The pages ask only for "FP8 precision for the K, V cache" ("Head Dimension"
 * article, §5.2).  Reading R17: every cached key and value is one OCP FP8
 * E4M3 code (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; exponent field 15 with mantissa 7 is NaN; largest finite 448;
 * subnormals m * 2^-9) times one scale per tensor (k_scale for keys, v_scale
 * for values).  A value x enters the cache as the code nearest to x / scale
 * (ties to even mantissa), values beyond 448 in magnitude saturating to
 * +-448. */

/* E4M3 code -> double (exact). */
static double e4m3(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* double -> nearest E4M3 code, ties to even, saturating at +-448. */
static uint8_t e4m3_code(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                      /* subnormal: a multiple of 2^-9 */
        double m = nearbyint(ldexp(a, 9));          /* 0..8; 8 is the smallest normal */
        return sign | (uint8_t)m;                   /* code 8 = exponent field 1, mantissa 0 */
    }
    int e;
    frexp(a, &e);                                   /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                         /* a in [2^e, 2^(e+1)) */
    double m = nearbyint((ldexp(a, -e) - 1.0) * 8.0);  /* 0..8 */
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && m > 6.0)) return sign | 0x7E;  /* rounded past 448 */
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

void oracle_e4m3_decode(const uint8_t *code, long n, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = e4m3(code[i]);
}

void oracle_e4m3_encode(const double *x, long n, uint8_t *code)
{
    for (long i = 0; i < n; ++i) code[i] = e4m3_code(x[i]);
}

/* Decode attention over keys [0, kv_len[b]) of FP8 caches [B, Hkv, Lmax, d]
 * (reading R17).  q [B,Hq,d] bf16 or binary16 (q_f16); attn [B, Hq*d]. */
int oracle_decode_attention_stage_fp8(const uint16_t *q, int q_f16, const uint8_t *k_cache,
                                      const uint8_t *v_cache, double k_scale, double v_scale,
                                      const int *kv_len, long B, long Hq, long Hkv, long d, long Lmax,
                                      double *attn, int nthreads)
{
    if (!q || !k_cache || !v_cache || !kv_len || !attn) return ORACLE_EARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || d > 1024 || Hq % Hkv || Lmax <= 0) return ORACLE_EARG;
    for (long b = 0; b < B; ++b)
        if (kv_len[b] <= 0 || kv_len[b] > Lmax) return ORACLE_EARG;
    long G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long j = 0; j < Hq; ++j) {
            long g = j / G;
            double qv[1024];
            for (long c = 0; c < d; ++c) qv[c] = w16(q[(b * Hq + j) * d + c], q_f16);
            kv_src src = {NULL, NULL, NULL, NULL, kv_len[b], 0,
                          k_cache + (b * Hkv + g) * Lmax * d, v_cache + (b * Hkv + g) * Lmax * d,
                          k_scale, v_scale};
            int e = attend_row(qv, &src, kv_len[b], d, attn + b * Hq * d + j * d);
            if (e) err = e;
        }
    }
    return err;
}

/* The decode step over FP8 caches (readings R17, R4): as oracle_decode, but
 * the cached entries [0, p) are E4M3 codes times k_scale / v_scale, and the
 * new token's key and value enter the cache as codes (e4m3_code of k / k_scale
 * and v / v_scale), so the query attends to their dequantised values like to
 * every other entry.  The caches are read, not modified.  Optional outputs:
 * q_new [B,Hq,d], k_new/v_new [B,Hkv,d] before quantisation, k_code/v_code
 * [B,Hkv,d] the codes appended, attn [B,Hq*d]. */
int oracle_decode_fp8(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                      const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                      double rope_theta, double eps,
                      long B, long hidden, long Hq, long Hkv, long d,
                      const uint8_t *k_cache, const uint8_t *v_cache, double k_scale, double v_scale,
                      const int *cache_len, long Lmax, double *out, double *q_new, double *k_new,
                      double *v_new, uint8_t *k_code, uint8_t *v_code, double *attn_out, int nthreads)
{
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !cache_len || !out) return ORACLE_EARG;
    if (B <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1) || d > 1024) return ORACLE_EARG;
    if (Hq % Hkv || !(k_scale > 0.0) || !(v_scale > 0.0)) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    for (long b = 0; b < B; ++b)
        if (cache_len[b] < 0 || cache_len[b] + 1 > Lmax) return ORACLE_EARG;
    long NQ = Hq * d, NKV = Hkv * d, N = NQ + 2 * NKV, G = Hq / Hkv;
    int err = ORACLE_OK;
    set_threads(nthreads);
    double *rows = (double *)malloc((size_t)(B * N) * sizeof(double));
    double *deq = (double *)malloc((size_t)(B * 2 * NKV) * sizeof(double));  /* new K, V dequantised */
    uint8_t *codes = (uint8_t *)malloc((size_t)(B * 2 * NKV));
    double *arows = (double *)malloc((size_t)(B * NQ) * sizeof(double));
    if (!rows || !deq || !codes || !arows) { err = ORACLE_ENOMEM; goto done; }

#pragma omp parallel for schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        double *row = rows + b * N;
        double p = (double)cache_len[b];
        linear_row(x + b * hidden, Wqkv, 0, N, hidden, row);
        for (long j = 0; j < Hq; ++j) {
            if (q_norm_w) rmsnorm_head(row + j * d, d, q_norm_w, eps);
            rope_head(row + j * d, d, p, rope_theta);
        }
        for (long g = 0; g < Hkv; ++g) {
            if (k_norm_w) rmsnorm_head(row + NQ + g * d, d, k_norm_w, eps);
            rope_head(row + NQ + g * d, d, p, rope_theta);
        }
        /* the new K and V as they enter the cache */
        for (long i = 0; i < NKV; ++i) {
            uint8_t ck = e4m3_code(row[NQ + i] / k_scale), cv = e4m3_code(row[NQ + NKV + i] / v_scale);
            codes[b * 2 * NKV + i] = ck;
            codes[b * 2 * NKV + NKV + i] = cv;
            deq[b * 2 * NKV + i] = e4m3(ck) * k_scale;
            deq[b * 2 * NKV + NKV + i] = e4m3(cv) * v_scale;
        }
    }

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long j = 0; j < Hq; ++j) {
            long g = j / G;
            kv_src src = {NULL, NULL, deq + b * 2 * NKV + g * d, deq + b * 2 * NKV + NKV + g * d,
                          cache_len[b], 0, k_cache + (b * Hkv + g) * Lmax * d,
                          v_cache + (b * Hkv + g) * Lmax * d, k_scale, v_scale};
            int e = attend_row(rows + b * N + j * d, &src, cache_len[b] + 1, d, arows + b * NQ + j * d);
            if (e) err = e;
        }
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (long b = 0; b < B; ++b) {
        for (long n = 0; n < hidden; ++n) {
            const uint16_t *w = Wo + n * NQ;
            double acc = 0.0;
            for (long k = 0; k < NQ; ++k) acc += arows[b * NQ + k] * bf(w[k]);
            out[b * hidden + n] = bf(x[b * hidden + n]) + acc;
        }
    }

    for (long b = 0; b < B; ++b) {
        const double *row = rows + b * N;
        if (q_new) memcpy(q_new + b * NQ, row, (size_t)NQ * sizeof(double));
        if (k_new) memcpy(k_new + b * NKV, row + NQ, (size_t)NKV * sizeof(double));
        if (v_new) memcpy(v_new + b * NKV, row + NQ + NKV, (size_t)NKV * sizeof(double));
        if (k_code) memcpy(k_code + b * NKV, codes + b * 2 * NKV, (size_t)NKV);
        if (v_code) memcpy(v_code + b * NKV, codes + b * 2 * NKV + NKV, (size_t)NKV);
        if (attn_out) memcpy(attn_out + b * NQ, arows + b * NQ, (size_t)NQ * sizeof(double));
    }
done:
    free(rows);
    free(deq);
    free(codes);
    free(arows);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Backward of the layer (gradients of a scalar loss L given dout = dL/dout). */
/* ------------------------------------------------------------------------ */

/* The pages ask for "the backward pass, including gradients into the shared
 * KV projections" ([NeoX] "Qwen3-0.6B example": both K and V projections serve
 * all query heads of a group; [Part]: a KV head's gradients come from every
 * query head that reads it).  They print no backward formulas; these are the
 * derivatives of the forward steps above, taken in reverse order:
 *   out = x + attn Wo^T          -> d_attn = dout Wo, dWo = dout^T attn, dx = dout
 *   o_t = sum_u p_u v_u, p = softmax(s), s_u = scale <q_t, k_u>
 *                                 -> dv_u += p_u do_t; dp_u = <do_t, v_u>;
 *                                    ds_u = p_u (dp_u - <do_t, o_t>);
 *                                    dq_t = scale sum_u ds_u k_u; dk_u += scale ds_u q_t
 *   q = RoPE(q_n)                 -> dq_n = RoPE^T(dq) (rotation by -angle)
 *   q_n = q_pre r w, r = (mean(q_pre^2) + eps)^(-1/2)
 *                                 -> dq_pre_i = r w_i dq_n_i - q_pre_i r^3 / d sum_k q_pre_k w_k dq_n_k
 *                                    dw_i += q_pre_i r dq_n_i (over every Q row; k_norm_w over K rows)
 *   qkv_pre = x Wqkv^T            -> dx += d_qkv_pre Wqkv, dWqkv = d_qkv_pre^T x
 * K and V gradients of a KV head sum over the G query heads of its group.
 * Rotary width rd (R16; oracle_backward: rd = d).  Outputs (all required): dx [B*S, hidden],
 * dWqkv [(Hq+2Hkv)*d, hidden], dWo [hidden, Hq*d], dqn/dkn [d] (zeroed
 * when there is no QK-norm).  Optional: d_attn [B*S, Hq*d] and the
 * attention-input gradients dq [B,Hq,S,d], dk/dv [B,Hkv,S,d] (after RoPE,
 * i.e. with respect to the attention's q, k, v). */

/* inverse RoPE: rotation of the first rd features by -angle */
static void rope_head_inv(double *v, long rd, double pos, double theta)
{
    long half = rd / 2;
    for (long i = 0; i < half; ++i) {
        double f = pos * pow(theta, -2.0 * (double)i / (double)rd);
        double c = cos(f), s = sin(f);
        double a = v[i], b = v[i + half];
        v[i] = a * c + b * s;
        v[i + half] = b * c - a * s;
    }
}

/* RMSNorm backward of one row: y = x r w.  dx and (accumulated) dw. */
static void rmsnorm_head_bwd(const double *x, const double *dy, long d, const uint16_t *w, double eps,
                             double *dx, double *dw)
{
    double ms = 0.0;
    for (long i = 0; i < d; ++i) ms += x[i] * x[i];
    ms /= (double)d;
    double r = 1.0 / sqrt(ms + eps);
    double dot = 0.0;
    for (long i = 0; i < d; ++i) dot += x[i] * bf(w[i]) * dy[i];
    for (long i = 0; i < d; ++i) {
        dx[i] = r * bf(w[i]) * dy[i] - x[i] * r * r * r / (double)d * dot;
        dw[i] += x[i] * r * dy[i];
    }
}

int oracle_backward_rd(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                       const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                       double rope_theta, double eps, long rd,
                       long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                       const uint16_t *dout,
                       double *dx, double *dWqkv, double *dWo, double *dqn, double *dkn,
                       double *d_attn_out, double *dq_out, double *dk_out, double *dv_out, int nthreads)
{
    if (!x || !Wqkv || !Wo || !dout || !dx || !dWqkv || !dWo || !dqn || !dkn) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1) || d > 1024) return ORACLE_EARG;
    if (rd < 0 || rd > d || (rd & 1)) return ORACLE_EARG;
    if (Hq % Hkv) return ORACLE_EARG;
    if ((q_norm_w == NULL) != (k_norm_w == NULL)) return ORACLE_EARG;
    const long M = B * S, NQ = Hq * d, NKV = Hkv * d, N = NQ + 2 * NKV, G = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)d);
    int err = ORACLE_OK;
    set_threads(nthreads);
    double *pre = (double *)malloc((size_t)(M * N) * sizeof(double));   /* qkv before norm/RoPE */
    double *Q = (double *)malloc((size_t)(B * Hq * S * d) * sizeof(double));
    double *K = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    double *V = (double *)malloc((size_t)(B * Hkv * S * d) * sizeof(double));
    double *attn = (double *)malloc((size_t)(M * NQ) * sizeof(double));
    double *dattn = (double *)malloc((size_t)(M * NQ) * sizeof(double));
    double *dQ = (double *)calloc((size_t)(B * Hq * S * d), sizeof(double));
    double *dK = (double *)calloc((size_t)(B * Hkv * S * d), sizeof(double));
    double *dV = (double *)calloc((size_t)(B * Hkv * S * d), sizeof(double));
    double *dpre = (double *)malloc((size_t)(M * N) * sizeof(double));
    if (!pre || !Q || !K || !V || !attn || !dattn || !dQ || !dK || !dV || !dpre) { err = ORACLE_ENOMEM; goto done; }

    /* forward: projections, norm, RoPE */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m) {
        long b = m / S, t = m % S;
        double *row = pre + m * N;
        linear_row(x + m * hidden, Wqkv, 0, N, hidden, row);
        double tmp[1024];
        for (long j = 0; j < Hq; ++j) {
            memcpy(tmp, row + j * d, (size_t)d * sizeof(double));
            if (q_norm_w) rmsnorm_head(tmp, d, q_norm_w, eps);
            rope_head(tmp, rd, (double)t, rope_theta);
            memcpy(Q + ((b * Hq + j) * S + t) * d, tmp, (size_t)d * sizeof(double));
        }
        for (long g = 0; g < Hkv; ++g) {
            memcpy(tmp, row + NQ + g * d, (size_t)d * sizeof(double));
            if (k_norm_w) rmsnorm_head(tmp, d, k_norm_w, eps);
            rope_head(tmp, rd, (double)t, rope_theta);
            memcpy(K + ((b * Hkv + g) * S + t) * d, tmp, (size_t)d * sizeof(double));
            memcpy(V + ((b * Hkv + g) * S + t) * d, row + NQ + NKV + g * d, (size_t)d * sizeof(double));
        }
    }
    /* forward attention (kept: attn rows) */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long m = 0; m < M; ++m)
        for (long j = 0; j < Hq; ++j) {
            long b = m / S, t = m % S, g = j / G;
            kv_src src = {NULL, NULL, K + (b * Hkv + g) * S * d, V + (b * Hkv + g) * S * d, 0, 0};
            int e = attend_row(Q + ((b * Hq + j) * S + t) * d, &src, causal ? t + 1 : S, d, attn + m * NQ + j * d);
            if (e) err = e;
        }
    /* out = x + attn Wo^T:  d_attn = dout Wo;  dWo = dout^T attn */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m)
        for (long c = 0; c < NQ; ++c) {
            double s = 0.0;
            for (long n = 0; n < hidden; ++n) s += bf(dout[m * hidden + n]) * bf(Wo[n * NQ + c]);
            dattn[m * NQ + c] = s;
        }
#pragma omp parallel for schedule(dynamic, 1)
    for (long n = 0; n < hidden; ++n)
        for (long c = 0; c < NQ; ++c) {
            double s = 0.0;
            for (long m = 0; m < M; ++m) s += bf(dout[m * hidden + n]) * attn[m * NQ + c];
            dWo[n * NQ + c] = s;
        }
    /* attention backward, one (sequence, KV head) at a time so that the
     * K/V gradient sums over the group's query heads need no locking */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b)
        for (long g = 0; g < Hkv; ++g) {
            const double *Kg = K + (b * Hkv + g) * S * d, *Vg = V + (b * Hkv + g) * S * d;
            double *dKg = dK + (b * Hkv + g) * S * d, *dVg = dV + (b * Hkv + g) * S * d;
            double *p = (double *)malloc((size_t)S * sizeof(double));
            double *dp = (double *)malloc((size_t)S * sizeof(double));
            if (!p || !dp) { err = ORACLE_ENOMEM; free(p); free(dp); continue; }
            for (long j = g * G; j < (g + 1) * G; ++j)
                for (long t = 0; t < S; ++t) {
                    const double *q = Q + ((b * Hq + j) * S + t) * d;
                    const double *o = attn + (b * S + t) * NQ + j * d;
                    const double *dO = dattn + (b * S + t) * NQ + j * d;
                    double *dq = dQ + ((b * Hq + j) * S + t) * d;
                    long n_vis = causal ? t + 1 : S;
                    double mx = -INFINITY;
                    for (long u = 0; u < n_vis; ++u) {
                        double s = 0.0;
                        for (long c = 0; c < d; ++c) s += q[c] * Kg[u * d + c];
                        p[u] = s * scale;
                        if (p[u] > mx) mx = p[u];
                    }
                    double den = 0.0;
                    for (long u = 0; u < n_vis; ++u) { p[u] = exp(p[u] - mx); den += p[u]; }
                    double Dt = 0.0;
                    for (long c = 0; c < d; ++c) Dt += dO[c] * o[c];
                    for (long u = 0; u < n_vis; ++u) {
                        p[u] /= den;
                        double s = 0.0;
                        for (long c = 0; c < d; ++c) s += dO[c] * Vg[u * d + c];
                        dp[u] = s;
                    }
                    for (long u = 0; u < n_vis; ++u) {
                        double ds = p[u] * (dp[u] - Dt);
                        for (long c = 0; c < d; ++c) {
                            dq[c] += scale * ds * Kg[u * d + c];
                            dKg[u * d + c] += scale * ds * q[c];
                            dVg[u * d + c] += p[u] * dO[c];
                        }
                    }
                }
            free(p);
            free(dp);
        }
    /* RoPE^T and QK-norm backward -> d_qkv_pre; norm-weight gradients */
    for (long i = 0; i < d; ++i) { dqn[i] = 0.0; dkn[i] = 0.0; }
    {
        double *dqn_rows = (double *)calloc((size_t)(M * d), sizeof(double));
        double *dkn_rows = (double *)calloc((size_t)(M * d), sizeof(double));
        if (!dqn_rows || !dkn_rows) { free(dqn_rows); free(dkn_rows); err = ORACLE_ENOMEM; goto done; }
#pragma omp parallel for schedule(dynamic, 1)
        for (long m = 0; m < M; ++m) {
            long b = m / S, t = m % S;
            double dy[1024];
            for (long j = 0; j < Hq; ++j) {
                memcpy(dy, dQ + ((b * Hq + j) * S + t) * d, (size_t)d * sizeof(double));
                rope_head_inv(dy, rd, (double)t, rope_theta);
                if (q_norm_w)
                    rmsnorm_head_bwd(pre + m * N + j * d, dy, d, q_norm_w, eps, dpre + m * N + j * d, dqn_rows + m * d);
                else
                    memcpy(dpre + m * N + j * d, dy, (size_t)d * sizeof(double));
            }
            for (long g = 0; g < Hkv; ++g) {
                memcpy(dy, dK + ((b * Hkv + g) * S + t) * d, (size_t)d * sizeof(double));
                rope_head_inv(dy, rd, (double)t, rope_theta);
                if (k_norm_w)
                    rmsnorm_head_bwd(pre + m * N + NQ + g * d, dy, d, k_norm_w, eps, dpre + m * N + NQ + g * d,
                                     dkn_rows + m * d);
                else
                    memcpy(dpre + m * N + NQ + g * d, dy, (size_t)d * sizeof(double));
                memcpy(dpre + m * N + NQ + NKV + g * d, dV + ((b * Hkv + g) * S + t) * d, (size_t)d * sizeof(double));
            }
        }
        for (long m = 0; m < M; ++m)
            for (long i = 0; i < d; ++i) { dqn[i] += dqn_rows[m * d + i]; dkn[i] += dkn_rows[m * d + i]; }
        free(dqn_rows);
        free(dkn_rows);
    }
    /* dx = dout + d_qkv_pre Wqkv;  dWqkv = d_qkv_pre^T x */
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m)
        for (long k = 0; k < hidden; ++k) {
            double s = bf(dout[m * hidden + k]);
            for (long n = 0; n < N; ++n) s += dpre[m * N + n] * bf(Wqkv[n * hidden + k]);
            dx[m * hidden + k] = s;
        }
#pragma omp parallel for schedule(dynamic, 1)
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < hidden; ++k) {
            double s = 0.0;
            for (long m = 0; m < M; ++m) s += dpre[m * N + n] * bf(x[m * hidden + k]);
            dWqkv[n * hidden + k] = s;
        }
    if (d_attn_out) memcpy(d_attn_out, dattn, (size_t)(M * NQ) * sizeof(double));
    if (dq_out) memcpy(dq_out, dQ, (size_t)(B * Hq * S * d) * sizeof(double));
    if (dk_out) memcpy(dk_out, dK, (size_t)(B * Hkv * S * d) * sizeof(double));
    if (dv_out) memcpy(dv_out, dV, (size_t)(B * Hkv * S * d) * sizeof(double));
done:
    free(pre); free(Q); free(K); free(V); free(attn); free(dattn); free(dQ); free(dK); free(dV); free(dpre);
    return err;
}

int oracle_backward(const uint16_t *x, const uint16_t *Wqkv, const uint16_t *Wo,
                    const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                    double rope_theta, double eps,
                    long B, long S, long hidden, long Hq, long Hkv, long d, int causal,
                    const uint16_t *dout,
                    double *dx, double *dWqkv, double *dWo, double *dqn, double *dkn,
                    double *d_attn_out, double *dq_out, double *dk_out, double *dv_out, int nthreads)
{
    return oracle_backward_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, d, B, S, hidden, Hq, Hkv, d,
                              causal, dout, dx, dWqkv, dWo, dqn, dkn, d_attn_out, dq_out, dk_out, dv_out, nthreads);
}

/* Attention backward alone, from 16-bit Q [B,Hq,S,d], K/V [B,Hkv,S,d] and
 * dO [B,S,Hq*d] (all bf16, or all binary16 with in_f16 = 1), widened exactly:
 * dq [B,Hq,S,d], dk/dv [B,Hkv,S,d] as in oracle_backward (K/V gradients sum
 * over the group's query heads). */
int oracle_attention_backward(const uint16_t *Qb, const uint16_t *Kb, const uint16_t *Vb, const uint16_t *dOb,
                              int in_f16, long B, long S, long Hq, long Hkv, long d, int causal,
                              double *dq, double *dk, double *dv, int nthreads)
{
    if (!Qb || !Kb || !Vb || !dOb || !dq || !dk || !dv) return ORACLE_EARG;
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || d > 1024 || Hq % Hkv) return ORACLE_EARG;
    const long G = Hq / Hkv, NQ = Hq * d;
    const double scale = 1.0 / sqrt((double)d);
    int err = ORACLE_OK;
    set_threads(nthreads);
    memset(dq, 0, (size_t)(B * Hq * S * d) * sizeof(double));
    memset(dk, 0, (size_t)(B * Hkv * S * d) * sizeof(double));
    memset(dv, 0, (size_t)(B * Hkv * S * d) * sizeof(double));
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (long b = 0; b < B; ++b)
        for (long g = 0; g < Hkv; ++g) {
            double *Kg = (double *)malloc((size_t)(S * d) * sizeof(double));
            double *Vg = (double *)malloc((size_t)(S * d) * sizeof(double));
            double *p = (double *)malloc((size_t)S * sizeof(double));
            double *dp = (double *)malloc((size_t)S * sizeof(double));
            double q[1024], o[1024], dO[1024];
            if (!Kg || !Vg || !p || !dp) { err = ORACLE_ENOMEM; free(Kg); free(Vg); free(p); free(dp); continue; }
            for (long i = 0; i < S * d; ++i) {
                Kg[i] = w16(Kb[(b * Hkv + g) * S * d + i], in_f16);
                Vg[i] = w16(Vb[(b * Hkv + g) * S * d + i], in_f16);
            }
            double *dKg = dk + (b * Hkv + g) * S * d, *dVg = dv + (b * Hkv + g) * S * d;
            for (long j = g * G; j < (g + 1) * G; ++j)
                for (long t = 0; t < S; ++t) {
                    for (long c = 0; c < d; ++c) {
                        q[c] = w16(Qb[((b * Hq + j) * S + t) * d + c], in_f16);
                        dO[c] = w16(dOb[(b * S + t) * NQ + j * d + c], in_f16);
                    }
                    long n_vis = causal ? t + 1 : S;
                    double mx = -INFINITY;
                    for (long u = 0; u < n_vis; ++u) {
                        double s = 0.0;
                        for (long c = 0; c < d; ++c) s += q[c] * Kg[u * d + c];
                        p[u] = s * scale;
                        if (p[u] > mx) mx = p[u];
                    }
                    double den = 0.0;
                    for (long u = 0; u < n_vis; ++u) { p[u] = exp(p[u] - mx); den += p[u]; }
                    for (long c = 0; c < d; ++c) o[c] = 0.0;
                    for (long u = 0; u < n_vis; ++u) {
                        p[u] /= den;
                        for (long c = 0; c < d; ++c) o[c] += p[u] * Vg[u * d + c];
                    }
                    double Dt = 0.0;
                    for (long c = 0; c < d; ++c) Dt += dO[c] * o[c];
                    double *dqr = dq + ((b * Hq + j) * S + t) * d;
                    for (long u = 0; u < n_vis; ++u) {
                        double s = 0.0;
                        for (long c = 0; c < d; ++c) s += dO[c] * Vg[u * d + c];
                        dp[u] = s;
                        double ds = p[u] * (dp[u] - Dt);
                        for (long c = 0; c < d; ++c) {
                            dqr[c] += scale * ds * Kg[u * d + c];
                            dKg[u * d + c] += scale * ds * q[c];
                            dVg[u * d + c] += p[u] * dO[c];
                        }
                    }
                }
            free(Kg); free(Vg); free(p); free(dp);
        }
    return err;
}
