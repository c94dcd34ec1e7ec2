/*
 * oracle.c -- the plain, slow, obviously correct CPU statement of the W2A8
 * ternary GEMV path (BitNet b1.58 linear layer at decode).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it is used by the tests, by the smoke check and by the
 * timed CPU baseline of the benchmark.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only at the byte formats that
 * the boundary header documents.
 *
 * Sources (page title, then the section used):
 *   [W2A8] "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核"
 *          (blog.gitcode.com) -- §一 model shape, §4.1 norms and fused
 *          projections, §4.2 weight scales, §5.1/§5.2 packing, §5.3 dot
 *          product and scale epilogue, §六 item 3 activation quantisation.
 *   [ESP]  "Յոթ ESP32-S3 տախտակ մեկ կլաստերում աշխատեցնում է 1,58 բիթանոց
 *          լեզվական մոդել" -- section "1,58 բիթ մեկ կշռի համար": three
 *          values per weight, four weights per byte.
 *
 * Readings taken where the pages are silent or disagree (each is listed in
 * the design notes):
 *   - canonical code = w + 1 in {0,1,2}; code 3 is invalid;
 *   - inside a canonical byte, weight 4j+t sits at bits 2t..2t+1 (LSB first);
 *   - the epilogue divides by the activation scale: y = acc / s * ws, with
 *     s = 127 / absmax as §六 item 3 defines it;
 *   - an all-zero activation row clamps absmax at 1e-5 (the same floor the
 *     weight quantiser of §4.2 uses), so it quantises to zeros;
 *   - the layer-stack glue (RMSNorm, ReLU^2 gate, one-token attention);
 *   - decode attention: RoPE on adjacent pairs with fp32 angles
 *     fl(p * fl(theta^(-2i/D))), the new key rounded to bf16 into the
 *     cache, scores scaled by 1/sqrt(D), softmax over positions 0..p.
 *
 * Precision: integer work is exact (int64 accumulators, checked against the
 * int32 range).  The pages fix fp32 for the quantiser and the epilogue, so
 * those decisions are taken in fp32 (IEEE, no contraction: build with
 * -ffp-contract=off).  RMSNorm statistics, which the pages leave open, are
 * accumulated in fp64, and so is all of the decode attention.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

enum {
    OR_OK = 0,
    OR_BAD_CODE = 1,   /* a canonical 2-bit code equal to 3            */
    OR_OVERFLOW = 2,   /* a dot product outside the int32 range         */
    OR_BAD_ARG = 3     /* shape, bounds or value outside the definition */
};

/* ------------------------------------------------------------------ */
/* Canonical ternary packing  ([W2A8] §5.2 step ③; [ESP] "1,58 բիթ")   */
/* ------------------------------------------------------------------ */

/* The 2-bit code of weight (n, k) in a canonical buffer of N rows of K/4
 * bytes.  Weight 4j+t of a row lives in byte j at bits 2t..2t+1. */
static int canon_code(const uint8_t *canon, int64_t K, int64_t n, int64_t k)
{
    int64_t row_bytes = K / 4;
    uint8_t byte = canon[n * row_bytes + k / 4];
    return (byte >> (2 * (k % 4))) & 3;
}

/* canon [N][K/4] -> w [N][K] int8 in {-1,0,1}.  Code 3 is rejected. */
int or_unpack(const uint8_t *canon, int64_t N, int64_t K, int8_t *w)
{
    if (N < 0 || K < 0 || K % 4 != 0) return OR_BAD_ARG;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t k = 0; k < K; k++) {
            int code = canon_code(canon, K, n, k);
            if (code == 3) return OR_BAD_CODE;
            w[n * K + k] = (int8_t)(code - 1);
        }
    }
    return OR_OK;
}

/* w [N][K] in {-1,0,1} -> canon [N][K/4]: code = w + 1, four per byte. */
int or_pack(const int8_t *w, int64_t N, int64_t K, uint8_t *canon)
{
    if (N < 0 || K < 0 || K % 4 != 0) return OR_BAD_ARG;
    int64_t row_bytes = K / 4;
    memset(canon, 0, (size_t)(N * row_bytes));
    for (int64_t n = 0; n < N; n++) {
        for (int64_t k = 0; k < K; k++) {
            int v = w[n * K + k];
            if (v < -1 || v > 1) return OR_BAD_ARG;
            int code = v + 1;
            canon[n * row_bytes + k / 4] |= (uint8_t)(code << (2 * (k % 4)));
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Integer dot product  ([W2A8] §5.3; §三 "exact int32 comparison")     */
/* ------------------------------------------------------------------ */

/* acc[m][n] = sum_k w[n][k] * q[m][k], exactly.
 * q: int8 [M][K] row-major; canon: [N][K/4]; acc: int32 [M][N]. */
int or_gemv_acc(const int8_t *q, const uint8_t *canon,
                int64_t M, int64_t N, int64_t K, int32_t *acc)
{
    if (M < 0 || N < 0 || K < 0 || K % 4 != 0) return OR_BAD_ARG;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            int64_t sum = 0;
            for (int64_t k = 0; k < K; k++) {
                int code = canon_code(canon, K, n, k);
                if (code == 3) return OR_BAD_CODE;
                int64_t wv = code - 1;
                sum += wv * (int64_t)q[m * K + k];
            }
            if (sum > INT32_MAX || sum < INT32_MIN) return OR_OVERFLOW;
            acc[m * N + n] = (int32_t)sum;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* bf16 rounding, from the IEEE-754 definition                          */
/* ------------------------------------------------------------------ */

/* Round an fp32 value to bf16 (the upper 16 bits of an fp32 pattern),
 * round-to-nearest, ties to even.  A NaN stays a quiet NaN. */
uint16_t or_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept_lsb = (u >> 16) & 1u;
    uint64_t r = (uint64_t)u + 0x7fffu + kept_lsb;   /* carry may reach inf */
    return (uint16_t)(r >> 16);
}

float or_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------ */
/* Scale epilogue  ([W2A8] §5.3 last paragraph; §4.2 per-matrix ws)     */
/* ------------------------------------------------------------------ */

/* Segment of output row n: the i with bounds[i] <= n < bounds[i+1]. */
static int64_t ws_segment(const int32_t *bounds, int64_t n_ws, int64_t n)
{
    for (int64_t i = 0; i < n_ws; i++)
        if (n >= bounds[i] && n < bounds[i + 1]) return i;
    return -1;
}

static int check_bounds(const int32_t *bounds, int64_t n_ws, int64_t N)
{
    if (n_ws < 1 || bounds[0] != 0 || bounds[n_ws] != N) return OR_BAD_ARG;
    for (int64_t i = 0; i < n_ws; i++)
        if (bounds[i + 1] <= bounds[i]) return OR_BAD_ARG;
    return OR_OK;
}

/* y[m][n] = bf16( ((float)acc[m][n] / s[m]) * ws[seg(n)] ), one rounding to
 * bf16 at the end, every step in IEEE fp32.
 * s: fp32 [M]; ws: bf16 bit patterns [n_ws]; bounds: [n_ws+1]; y: bf16 [M][N]. */
int or_gemv(const int8_t *q, const uint8_t *canon, const float *s,
            const uint16_t *ws, const int32_t *bounds, int64_t n_ws,
            int64_t M, int64_t N, int64_t K, uint16_t *y)
{
    if (M < 0 || N < 0) return OR_BAD_ARG;
    int rc = check_bounds(bounds, n_ws, N);
    if (rc != OR_OK) return rc;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            int32_t acc;
            rc = or_gemv_acc(q + m * K, canon + n * (K / 4), 1, 1, K, &acc);
            if (rc != OR_OK) return rc;
            int64_t seg = ws_segment(bounds, n_ws, n);
            float a = (float)acc;
            float scaled = a / s[m];
            float out = scaled * or_bf16_value(ws[seg]);
            y[m * N + n] = or_bf16_rne(out);
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Per-row absmax activation quantisation  ([W2A8] §六 item 3)          */
/* ------------------------------------------------------------------ */

/* s[m] = 127 / max(absmax_k |x[m][k]|, 1e-5); q = clamp(round_half_even(x*s),
 * -128, 127).  All fp32.  x must be finite. */
void or_quant_act(const float *x, int64_t M, int64_t K, int8_t *q, float *s)
{
    for (int64_t m = 0; m < M; m++) {
        float absmax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float a = fabsf(x[m * K + k]);
            if (a > absmax) absmax = a;
        }
        if (absmax < 1e-5f) absmax = 1e-5f;
        float scale = 127.0f / absmax;
        s[m] = scale;
        for (int64_t k = 0; k < K; k++) {
            float v = nearbyintf(x[m * K + k] * scale);  /* ties to even */
            if (v > 127.0f) v = 127.0f;
            if (v < -128.0f) v = -128.0f;
            q[m * K + k] = (int8_t)v;
        }
    }
}

/*
 * Absmean ternarisation of a weight matrix, per weight-scale segment (rows
 * [bounds[i], bounds[i+1])), as the checkpoint conversion of [W2A8] §4.2
 * states it: s = 1 / max(mean |W|, 1e-5), w = clamp(round(W * s), -1, 1),
 * ws = bf16(1 / s).  The page leaves the precision to the framework's dtype;
 * read here for fp32 weights: |W| summed in fp64 over the segment (rows in
 * order, k in order), the mean (sum / count in fp64) rounded to fp32; s,
 * W * s and 1 / s in fp32; round = nearest, ties to even; ws rounded to bf16
 * (round to nearest even).  Output: canonical pack [N][K/4] (code = w + 1,
 * element 4j+t at bits 2t of byte j) and the bf16 bit patterns of ws [n_ws].
 */
int or_quant_weight(const float *W, int64_t N, int64_t K,
                    const int32_t *bounds, int64_t n_ws, uint8_t *canon,
                    uint16_t *ws)
{
    if (N < 1 || K < 4 || K % 4 != 0) return OR_BAD_ARG;
    if (check_bounds(bounds, n_ws, N) != OR_OK) return OR_BAD_ARG;
    for (int64_t i = 0; i < n_ws; i++) {
        const int64_t r0 = bounds[i], r1 = bounds[i + 1];
        double sum = 0.0;
        for (int64_t n = r0; n < r1; n++)
            for (int64_t k = 0; k < K; k++)
                sum += fabs((double)W[n * K + k]);
        float mean = (float)(sum / (double)((r1 - r0) * K));
        if (mean < 1e-5f) mean = 1e-5f;
        const float s = 1.0f / mean;
        ws[i] = or_bf16_rne(1.0f / s);
        for (int64_t n = r0; n < r1; n++) {
            for (int64_t j = 0; j < K / 4; j++) {
                unsigned byte = 0;
                for (int t = 0; t < 4; t++) {
                    float v = nearbyintf(W[n * K + 4 * j + t] * s);
                    if (v > 1.0f) v = 1.0f;
                    if (v < -1.0f) v = -1.0f;
                    byte |= (unsigned)((int)v + 1) << (2 * t);
                }
                canon[n * (K / 4) + j] = (uint8_t)byte;
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Device weight layout, restated from the boundary header's layout    */
/* specification (element by element; independent of the CUDA code).  */
/* ------------------------------------------------------------------ */
/*
 * Rows are padded to a multiple of 8, K to a multiple of 64; padding codes
 * are 1 (weight 0).  A 16-byte chunk holds 64 weights of one row: chunk j
 * of row n covers k in [64j, 64j+64).  Word t (bytes 4t..4t+3) of a chunk
 * covers k in [64j+16t, 64j+16t+16); element e = k mod 16 of that word sits
 * in byte e mod 4 at bits 2*(e div 4) -- the word interleave of [W2A8] §5.2
 * (pattern 0,4,8,12,1,5,...; shift table 0,8,16,24,2,10,...).
 * Chunks are stored row-group by row-group (8 rows), chunk index next, then
 * the row inside the group: byte offset of chunk (n, j) =
 *   ((n/8) * C + j) * 128 + (n%8) * 16,   C = Kpad / 64.
 */
int64_t or_layout_bytes(int64_t N, int64_t K)
{
    if (N < 0 || K < 0) return -1;
    int64_t npad = (N + 7) / 8 * 8;
    int64_t chunks = (K + 63) / 64;
    return npad * chunks * 16;
}

int or_layout(const uint8_t *canon, int64_t N, int64_t K, uint8_t *dev)
{
    if (N < 0 || K < 0 || K % 4 != 0) return OR_BAD_ARG;
    int64_t npad = (N + 7) / 8 * 8;
    int64_t chunks = (K + 63) / 64;
    int64_t kpad = chunks * 64;
    memset(dev, 0, (size_t)or_layout_bytes(N, K));
    for (int64_t n = 0; n < npad; n++) {
        for (int64_t k = 0; k < kpad; k++) {
            int code = 1;
            if (n < N && k < K) {
                code = canon_code(canon, K, n, k);
                if (code == 3) return OR_BAD_CODE;
            }
            int64_t j = k / 64, t = (k % 64) / 16, e = k % 16;
            int64_t byte_off = ((n / 8) * chunks + j) * 128 + (n % 8) * 16
                               + t * 4 + (e % 4);
            dev[byte_off] |= (uint8_t)(code << (2 * (e / 4)));
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Layer-stack glue ([W2A8] §一 shape, §4.1 norms and fused projections)*/
/* ------------------------------------------------------------------ */

/* RMSNorm: out_k = x_k * (1/sqrt(mean(x^2) + eps)) * gamma_k.  The
 * statistic and the products are taken in fp64 and rounded to fp32 once. */
void or_rmsnorm(const float *x, const float *gamma, int64_t K, float eps,
                float *out)
{
    double sumsq = 0.0;
    for (int64_t k = 0; k < K; k++) sumsq += (double)x[k] * (double)x[k];
    double r = 1.0 / sqrt(sumsq / (double)K + (double)eps);
    for (int64_t k = 0; k < K; k++)
        out[k] = (float)((double)x[k] * r * (double)gamma[k]);
}

/* Squared-ReLU gate of the fused w13 output (gate rows first, then up):
 * g_i = max(gate_i, 0)^2 * up_i.  gu: bf16 [2F]; out: fp32 [F]. */
void or_relu2_gate(const uint16_t *gu, int64_t F, float *out)
{
    for (int64_t i = 0; i < F; i++) {
        double g = or_bf16_value(gu[i]);
        double u = or_bf16_value(gu[F + i]);
        double r = g > 0.0 ? g : 0.0;
        out[i] = (float)(r * r * u);
    }
}

/* Attention over a one-token context with grouped KV heads: the softmax of
 * a single score is 1, so query head h returns the value vector of KV head
 * h / (n_heads / n_kv_heads).  qkv: bf16 [(n_heads + 2 n_kv) * hd] laid out
 * q | k | v; out: fp32 [n_heads * hd]. */
int or_attn_one_token(const uint16_t *qkv, int64_t n_heads, int64_t n_kv,
                      int64_t head_dim, float *out)
{
    if (n_kv < 1 || n_heads % n_kv != 0) return OR_BAD_ARG;
    int64_t group = n_heads / n_kv;
    int64_t v_off = (n_heads + n_kv) * head_dim;
    for (int64_t h = 0; h < n_heads; h++)
        for (int64_t d = 0; d < head_dim; d++)
            out[h * head_dim + d] =
                or_bf16_value(qkv[v_off + (h / group) * head_dim + d]);
    return OR_OK;
}

/* One GEMV of the stack: RMSNorm -> absmax quantisation -> W2A8 GEMV.
 * Writes the intermediate int8 codes and scale too, for stage checks. */
static int norm_quant_gemv(const float *x, const float *gamma, int64_t K,
                           float eps, const uint8_t *canon, const uint16_t *ws,
                           const int32_t *bounds, int64_t n_ws, int64_t N,
                           float *normed, int8_t *q, float *s, uint16_t *y)
{
    or_rmsnorm(x, gamma, K, eps, normed);
    or_quant_act(normed, 1, K, q, s);
    return or_gemv(q, canon, s, ws, bounds, n_ws, 1, N, K, y);
}

/* ------------------------------------------------------------------ */
/* GQA decode attention over a KV cache ([W2A8] §一: 20 query heads,    */
/* 5 KV heads, head_dim 128; §4.1: RoPE rotates adjacent pairs of head */
/* dims; §六 item 2: a preallocated KV cache and flash attention)       */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern of the double x, rounded to nearest even in one step
 * (no fp32 intermediate).  |x| = m 2^e with m in [0.5, 1): a normal bf16
 * keeps 8 significant bits, k = m 2^8 in [128, 256), value k 2^(e-8). */
uint16_t or_bf16_rne_d(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7fc0u;
    if (a == 0.0) return sign;
    int e;
    double m = frexp(a, &e);
    int biased = e - 1 + 127;           /* exponent field of a normal */
    if (biased < 1) {                   /* subnormal: units of 2^-133 */
        double k = nearbyint(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)k);   /* k = 128 is 0x0080 */
    }
    double k = nearbyint(m * 256.0);    /* exact scaling, then RNE */
    if (k == 256.0) {
        k = 128.0;
        biased += 1;
    }
    if (biased > 254) return (uint16_t)(sign | 0x7f80u);  /* overflow */
    return (uint16_t)(sign | (uint16_t)(biased << 7) |
                      (uint16_t)((int)k - 128));
}

/* Angle of pair i of a head of D dims at position p.  Reading (the pages
 * leave the precision open): the frequency f_i = theta^(-2i/D) is taken in
 * fp64 and rounded to fp32 once, and the angle is the fp32 product
 * p * f_i (one IEEE rounding; this file is built without contraction). */
float or_rope_angle(int64_t p, int64_t i, int64_t D, float theta)
{
    float f = (float)pow((double)theta, -2.0 * (double)i / (double)D);
    float pf = (float)p;
    return pf * f;
}

/* RoPE of one head vector x (bf16 bits, D values) at position p, in fp64:
 * pair (x[2i], x[2i+1]) turns by the angle of pair i. */
int or_rope(const uint16_t *x, int64_t D, int64_t p, float theta,
            double *out)
{
    if (D < 2 || D % 2 != 0 || p < 0) return OR_BAD_ARG;
    for (int64_t i = 0; i < D / 2; i++) {
        double phi = (double)or_rope_angle(p, i, D, theta);
        double c = cos(phi), s = sin(phi);
        double x0 = or_bf16_value(x[2 * i]), x1 = or_bf16_value(x[2 * i + 1]);
        out[2 * i] = x0 * c - x1 * s;
        out[2 * i + 1] = x0 * s + x1 * c;
    }
    return OR_OK;
}

/* The cache append of one decode step: the new key of KV head g (qkv[H D +
 * g D ..]) is rotated at position p and stored at kc[g][p], rounded to bf16
 * (nearest even); the new value (qkv[(H + Hkv) D + g D ..]) is stored at
 * vc[g][p] as it is.  kc, vc: bf16 [Hkv][S][D]. */
int or_attn_append(const uint16_t *qkv, int64_t H, int64_t Hkv, int64_t D,
                   int64_t p, float theta, uint16_t *kc, uint16_t *vc,
                   int64_t S)
{
    if (H < 1 || Hkv < 1 || H % Hkv != 0 || D < 2 || D % 2 != 0 ||
        p < 0 || p >= S)
        return OR_BAD_ARG;
    const uint16_t *kn = qkv + H * D, *vn = qkv + (H + Hkv) * D;
    double *rot = malloc(sizeof(double) * (size_t)D);
    if (!rot) return OR_BAD_ARG;
    for (int64_t g = 0; g < Hkv; g++) {
        or_rope(kn + g * D, D, p, theta, rot);
        for (int64_t d = 0; d < D; d++) {
            kc[(g * S + p) * D + d] = or_bf16_rne_d(rot[d]);
            vc[(g * S + p) * D + d] = vn[g * D + d];
        }
    }
    free(rot);
    return OR_OK;
}

/* Attention of the step over the cache as it stands (rows 0..p, the new
 * token's row included): query head h (qkv[h D ..]) is rotated at p and
 * reads KV head g = h / (H / Hkv); s_j = q'.kc[g][j] / sqrt(D);
 * out[h] = sum_j softmax(s)_j vc[g][j].  fp64, the softmax subtracting the
 * largest score.  out: fp64 [H][D]. */
int or_attn_over_cache(const uint16_t *qkv, int64_t H, int64_t Hkv,
                       int64_t D, int64_t p, float theta, const uint16_t *kc,
                       const uint16_t *vc, int64_t S, double *out)
{
    if (H < 1 || Hkv < 1 || H % Hkv != 0 || D < 2 || D % 2 != 0 ||
        p < 0 || p >= S)
        return OR_BAD_ARG;
    int64_t G = H / Hkv;
    double *rot = malloc(sizeof(double) * (size_t)D);
    double *sc = malloc(sizeof(double) * (size_t)(p + 1));
    if (!rot || !sc) {
        free(rot);
        free(sc);
        return OR_BAD_ARG;
    }
    double scale = 1.0 / sqrt((double)D);
    for (int64_t h = 0; h < H; h++) {
        int64_t g = h / G;
        or_rope(qkv + h * D, D, p, theta, rot);
        double mx = -INFINITY;
        for (int64_t j = 0; j <= p; j++) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; d++)
                dot += rot[d] * or_bf16_value(kc[(g * S + j) * D + d]);
            sc[j] = dot * scale;
            if (sc[j] > mx) mx = sc[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j <= p; j++) {
            sc[j] = exp(sc[j] - mx);
            l += sc[j];
        }
        for (int64_t d = 0; d < D; d++) {
            double acc = 0.0;
            for (int64_t j = 0; j <= p; j++)
                acc += sc[j] * or_bf16_value(vc[(g * S + j) * D + d]);
            out[h * D + d] = acc / l;
        }
    }
    free(rot);
    free(sc);
    return OR_OK;
}

/* One decode step of grouped-query attention for one sequence: the append,
 * then the attention over positions 0..p.
 *   qkv  bf16 [(H + 2 Hkv) D]: q heads, then k heads, then v heads (the
 *        fused wqkv output of the layer).
 *   kc, vc  bf16 [Hkv][S][D]: the cache; positions 0..p-1 hold the earlier
 *        tokens' rotated keys and values; row p is written. */
int or_attn_decode(const uint16_t *qkv, int64_t H, int64_t Hkv, int64_t D,
                   int64_t p, float theta, uint16_t *kc, uint16_t *vc,
                   int64_t S, double *out)
{
    int rc = or_attn_append(qkv, H, Hkv, D, p, theta, kc, vc, S);
    if (rc) return rc;
    return or_attn_over_cache(qkv, H, Hkv, D, p, theta, kc, vc, S, out);
}

/* ------------------------------------------------------------------ */
/* Decoder layer with attention over a KV cache ([W2A8] §一, §4.1, §六)  */
/* ------------------------------------------------------------------ */

/*
 * One decoder layer of the stack, M = 1, in the order of the BitNet block:
 *   a = attn_norm(h) -> quant -> wqkv -> one-token attention
 *      (or attention over a KV cache, or_layer_kv)
 *   b = attn_sub_norm(attn) -> quant -> wo;          h += b
 *   c = ffn_norm(h) -> quant -> w13 -> relu(gate)^2 * up
 *   d = ffn_sub_norm(g) -> quant -> w2;              h += d
 * h (fp32, length dim) is updated in place; residual adds are fp32.
 * gammas: 4 vectors (attn_norm[dim], attn_sub[dim], ffn_norm[dim],
 * ffn_sub[ffn]) concatenated.  ws: wqkv 3 values, wo 1, w13 2, w2 1.
 * scratch must hold 4*ffn floats; the fused qkv width must not exceed 2*ffn.
 */
static int layer_impl(float *h, int64_t dim, int64_t ffn, int64_t n_heads,
                      int64_t n_kv, float eps,
                      const uint8_t *wqkv, const uint8_t *wo,
                      const uint8_t *w13, const uint8_t *w2,
                      const uint16_t *ws, const float *gammas, float *scratch,
                      uint16_t *kc, uint16_t *vc, int64_t S, int64_t p,
                      float theta)
{
    int64_t hd = dim / n_heads;
    int64_t qkv_n = (n_heads + 2 * n_kv) * hd;
    int32_t b_qkv[4] = {0, (int32_t)(n_heads * hd),
                        (int32_t)((n_heads + n_kv) * hd), (int32_t)qkv_n};
    int32_t b_o[2] = {0, (int32_t)dim};
    int32_t b_13[3] = {0, (int32_t)ffn, (int32_t)(2 * ffn)};
    int32_t b_2[2] = {0, (int32_t)dim};
    const float *g_attn = gammas, *g_asub = gammas + dim;
    const float *g_ffn = gammas + 2 * dim, *g_fsub = gammas + 3 * dim;

    float *normed = scratch;                 /* up to ffn floats   */
    float *vec = scratch + ffn;              /* up to ffn floats   */
    int8_t *q = (int8_t *)(scratch + 2 * ffn);   /* ffn bytes      */
    uint16_t *y = (uint16_t *)(scratch + 3 * ffn);  /* up to 2 ffn */
    float s;
    int rc;

    if (n_heads * hd != dim) return OR_BAD_ARG;
    if (qkv_n > 2 * ffn || dim > ffn) return OR_BAD_ARG;

    rc = norm_quant_gemv(h, g_attn, dim, eps, wqkv, ws + 0, b_qkv, 3, qkv_n,
                         normed, q, &s, y);
    if (rc) return rc;
    if (!kc) {
        rc = or_attn_one_token(y, n_heads, n_kv, hd, vec);
    } else {
        double *att = malloc(sizeof(double) * (size_t)dim);
        if (!att) return OR_BAD_ARG;
        rc = or_attn_decode(y, n_heads, n_kv, hd, p, theta, kc, vc, S, att);
        for (int64_t i = 0; i < dim && rc == OR_OK; i++)
            vec[i] = (float)att[i];
        free(att);
    }
    if (rc) return rc;
    rc = norm_quant_gemv(vec, g_asub, dim, eps, wo, ws + 3, b_o, 1, dim,
                         normed, q, &s, y);
    if (rc) return rc;
    for (int64_t i = 0; i < dim; i++) h[i] = h[i] + or_bf16_value(y[i]);

    rc = norm_quant_gemv(h, g_ffn, dim, eps, w13, ws + 4, b_13, 2, 2 * ffn,
                         normed, q, &s, y);
    if (rc) return rc;
    or_relu2_gate(y, ffn, vec);
    rc = norm_quant_gemv(vec, g_fsub, ffn, eps, w2, ws + 6, b_2, 1, dim,
                         normed, q, &s, y);
    if (rc) return rc;
    for (int64_t i = 0; i < dim; i++) h[i] = h[i] + or_bf16_value(y[i]);
    return OR_OK;
}


int or_layer(float *h, int64_t dim, int64_t ffn, int64_t n_heads,
             int64_t n_kv, float eps,
             const uint8_t *wqkv, const uint8_t *wo, const uint8_t *w13,
             const uint8_t *w2, const uint16_t *ws, const float *gammas,
             float *scratch)
{
    return layer_impl(h, dim, ffn, n_heads, n_kv, eps, wqkv, wo, w13, w2, ws,
                      gammas, scratch, NULL, NULL, 0, 0, 0.0f);
}

/* The same layer with grouped-query attention over the layer's KV cache
 * (kc, vc: bf16 [n_kv][S][hd]) at position p in place of the one-token
 * attention: the decode step of or_attn_decode on the bf16 wqkv output,
 * its fp64 result rounded to fp32 as the input of attn_sub_norm.  At p = 0
 * the attention returns the value heads exactly, so the layer equals
 * or_layer. */
int or_layer_kv(float *h, int64_t dim, int64_t ffn, int64_t n_heads,
                int64_t n_kv, float eps,
                const uint8_t *wqkv, const uint8_t *wo, const uint8_t *w13,
                const uint8_t *w2, const uint16_t *ws, const float *gammas,
                float *scratch, uint16_t *kc, uint16_t *vc, int64_t S,
                int64_t p, float theta)
{
    if (!kc || !vc) return OR_BAD_ARG;
    return layer_impl(h, dim, ffn, n_heads, n_kv, eps, wqkv, wo, w13, w2, ws,
                      gammas, scratch, kc, vc, S, p, theta);
}

