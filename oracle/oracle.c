/*
 * ORACLE -- test infrastructure, not the product.
 *
 * A plain, slow CPU statement of what the quantised-linear hot path computes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference arm may load this library.  It shares no code with the CUDA
 * library; both sides only receive the same seeded inputs from `synth`.
 *
 * Sources (web pages; section names as printed on them):
 *   [gemma.cpp tour]  pyshine.com "gemma.cpp" -- "Weights, Blobs, and the .sbs
 *                     Format", "The Forward Pass, Layer by Layer".
 *   [cpp20gemma]      README -- "Architecture & implementation", "Tests".
 *   [llama2.c]        "llama2.c -- Llama-2 Inference in One C File" -- "The
 *                     forward pass -- one token, one position" (Steps 0-6),
 *                     "matmul", "Sampling", "The generation loop".
 *   [citric]          "Gemma 3 1B at 114 tokens per second on a laptop CPU" --
 *                     "On a CPU, speed is bytes", "Step 1: a kernel for 1.6-bit
 *                     weights", "Step 2: making a ternary Gemma", "Step 3: the
 *                     output layer became the bottleneck".
 *
 * Precision: integer work is exact (int64 accumulators).  Plain linear maps
 * with no quantiser downstream (W8 linear, lm_head logits) accumulate in
 * fp64 and round once.  Everything that feeds an activation quantiser in the
 * decode step is defined in fp32 with a fixed operation order (pairwise sums,
 * a Cody-Waite exponential), because a one-ulp change in front of an int8
 * rounding changes a code and then every later token.  Compile with
 * -ffp-contract=off.
 *
 * Parity pins: every function here is pinned by tests under tests/ against
 * closed forms, hand-worked vectors, brute force or fp64 references.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL 1
#define OR_EBADBYTE 3

static const int32_t POW3[5] = {1, 3, 9, 27, 81};

/* ------------------------------------------------------------------ S1 / S3
 * Symmetric absmax int8 quantisation, [cpp20gemma] "Architecture &
 * implementation": scale = max(|w|, 1e-9)/127, w8 = clip(round(w/scale)).
 * Readings: division in fp32, round half to even (NumPy's round, which the
 * converter script uses), clip to +-127 (the -128 end of the page's clip is
 * unreachable because |w/scale| <= 127).  The same rule quantises activations
 * per row ([citric] "Step 2": inputs to each layer rounded to int8;
 * [llama2.c] "Key ideas": activations quantised dynamically, range +-127).
 */
static float absmax_scale(const float *v, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(v[i]);
        if (a > m) m = a;
    }
    if (m < 1e-9f) m = 1e-9f;
    return m / 127.0f;
}

static int8_t quant_one(float v, float scale) {
    float r = rintf(v / scale); /* default rounding mode: nearest, ties to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int8_t)r;
}

int or_w8_quantize(const float *w, int64_t n, int8_t *q, float *scale) {
    if (!w || !q || !scale || n < 1) return OR_EINVAL;
    float s = absmax_scale(w, n);
    for (int64_t i = 0; i < n; i++) q[i] = quant_one(w[i], s);
    *scale = s;
    return OR_OK;
}

int or_quant_i8(const float *x, int64_t M, int64_t K, int8_t *xq, float *xs) {
    if (!x || !xq || !xs || M < 1 || K < 1) return OR_EINVAL;
    for (int64_t m = 0; m < M; m++) {
        float s = absmax_scale(x + m * K, K);
        for (int64_t k = 0; k < K; k++) xq[m * K + k] = quant_one(x[m * K + k], s);
        xs[m] = s;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ S5
 * W8 linear: y = (x . w8) * scale, the scale applied once after the dot
 * product ([cpp20gemma] "Architecture & implementation"); rows of w8 are
 * [out][in] row-major; [llama2.c] "matmul" is the same loop over output rows.
 * Accumulated in fp64, rounded once to fp32.
 */
int or_w8_linear(const float *x, const int8_t *q, int64_t q_pitch, float s, int64_t M, int64_t N,
                 int64_t K, float *y) {
    if (!x || !q || !y || M < 1 || N < 1 || K < 1 || q_pitch < K) return OR_EINVAL;
    for (int64_t m = 0; m < M; m++) {
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) acc += (double)x[m * K + k] * (double)q[n * q_pitch + k];
            y[m * N + n] = (float)(acc * (double)s);
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ W8 with group scales
 * gemma.cpp's I8Stream ([gemma.cpp tour] "The compression formats"): int8 in
 * groups of 128 with a shared scale; runq.c's Q8_0 ([llama2.c] "Key ideas &
 * tradeoffs"): symmetric, range +-127, weights only.  Reading: the groups
 * are G consecutive weights of a row along K (the last group of a row is
 * shorter when G does not divide K), each quantised with the W8 rule above
 * (its own absmax, the 1e-9 floor, fp32 division, round half to even).
 * q: int8 [N][K]; scales: fp32 [N][ceil(K/G)].
 */
int or_w8g_quantize(const float *w, int64_t N, int64_t K, int64_t G, int8_t *q, float *scales) {
    if (!w || !q || !scales || N < 1 || K < 1 || G < 1) return OR_EINVAL;
    const int64_t ng = (K + G - 1) / G;
    for (int64_t n = 0; n < N; n++)
        for (int64_t g = 0; g < ng; g++) {
            const int64_t k0 = g * G, len = (k0 + G <= K) ? G : K - k0;
            const float s = absmax_scale(w + n * K + k0, len);
            for (int64_t k = k0; k < k0 + len; k++) q[n * K + k] = quant_one(w[n * K + k], s);
            scales[n * ng + g] = s;
        }
    return OR_OK;
}

/* y[m][n] = sum_g scale[n][g] * (sum_{k in g} x[m][k] * q[n][k]): each
 * group's dot product takes its own scale, in fp64, rounded once to fp32. */
int or_w8g_linear(const float *x, const int8_t *q, int64_t q_pitch, const float *scales, int64_t s_pitch, int64_t G,
                  int64_t M, int64_t N, int64_t K, float *y) {
    if (!x || !q || !scales || !y || M < 1 || N < 1 || K < 1 || G < 1 || q_pitch < K || s_pitch < (K + G - 1) / G)
        return OR_EINVAL;
    const int64_t ng = (K + G - 1) / G;
    for (int64_t m = 0; m < M; m++) {
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t g = 0; g < ng; g++) {
                double part = 0.0;
                for (int64_t k = g * G; k < K && k < (g + 1) * G; k++)
                    part += (double)x[m * K + k] * (double)q[n * q_pitch + k];
                acc += part * (double)scales[n * s_pitch + g];
            }
            y[m * N + n] = (float)acc;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ S2
 * T158 packing, [citric] "Step 1": five ternary weights per byte in base 3
 * (3^5 = 243 <= 256).  Digit order and row layout are not on the page; the
 * adopted reading: digit d_i = trit_{5j+i} + 1, byte j = sum_i d_i * 3^i
 * (least significant digit first), each row of a [N][K] matrix packed on its
 * own into `pitch` bytes; trits past K are zero trits (digit 1), so every byte
 * past ceil(K/5) is 121.
 */
int or_t158_pack(const int8_t *t, int64_t N, int64_t K, uint8_t *packed, int64_t pitch) {
    if (!t || !packed || N < 1 || K < 1 || pitch < (K + 4) / 5) return OR_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (t[i] < -1 || t[i] > 1) return OR_EINVAL;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t j = 0; j < pitch; j++) {
            int32_t byte = 0;
            for (int i = 0; i < 5; i++) {
                int64_t k = 5 * j + i;
                int32_t digit = (k < K) ? (int32_t)t[n * K + k] + 1 : 1;
                byte += digit * POW3[i];
            }
            packed[n * pitch + j] = (uint8_t)byte;
        }
    }
    return OR_OK;
}

/* Digit i (0..4) of a packed byte, as the trit it encodes. */
static int32_t trit_of(uint8_t byte, int i) { return ((int32_t)byte / POW3[i]) % 3 - 1; }

int or_t158_unpack(const uint8_t *packed, int64_t N, int64_t K, int64_t pitch, int8_t *t) {
    if (!packed || !t || N < 1 || K < 1 || pitch < (K + 4) / 5) return OR_EINVAL;
    for (int64_t n = 0; n < N; n++)
        for (int64_t j = 0; j < pitch; j++)
            if (packed[n * pitch + j] > 242) return OR_EBADBYTE;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) t[n * K + k] = (int8_t)trit_of(packed[n * pitch + k / 5], (int)(k % 5));
    return OR_OK;
}

/* Zero-group skipping ([citric] "What is next": a kernel that skips groups of
 * four zero inputs).  Its weights are stored by input group: group g holds
 * inputs 4g .. 4g+3, and row n of the group is one byte, sum_i (t[n][4g+i]+1)
 * * 3^i (least significant digit first, as the five-trit bytes; trits past K
 * are zero trits, digit 1), so one input group's weights are the gpitch
 * contiguous bytes [g][0 .. gpitch) and a zero group's bytes are never read.
 * Bytes of rows gpitch > n >= N are 40 (four zero trits).  The page gives no
 * layout; this is the plainest one in which skipping a group skips its bytes.
 * The linear layer itself is the T158 linear below: leaving out zero inputs
 * changes no sum.
 */
int or_t158_pack_groups(const int8_t *t, int64_t N, int64_t K, uint8_t *packed_g, int64_t gpitch) {
    if (!t || !packed_g || N < 1 || K < 1 || gpitch < N) return OR_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (t[i] < -1 || t[i] > 1) return OR_EINVAL;
    const int64_t G = (K + 3) / 4;
    for (int64_t g = 0; g < G; g++)
        for (int64_t n = 0; n < gpitch; n++) {
            int32_t byte = 0;
            for (int i = 0; i < 4; i++) {
                const int64_t k = 4 * g + i;
                const int32_t digit = (n < N && k < K) ? (int32_t)t[n * K + k] + 1 : 1;
                byte += digit * POW3[i];
            }
            packed_g[g * gpitch + n] = (uint8_t)byte;
        }
    return OR_OK;
}

int or_t158_unpack_groups(const uint8_t *packed_g, int64_t N, int64_t K, int64_t gpitch, int8_t *t) {
    if (!packed_g || !t || N < 1 || K < 1 || gpitch < N) return OR_EINVAL;
    const int64_t G = (K + 3) / 4;
    for (int64_t g = 0; g < G; g++)
        for (int64_t n = 0; n < N; n++)
            if (packed_g[g * gpitch + n] > 80) return OR_EBADBYTE;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) t[n * K + k] = (int8_t)trit_of(packed_g[(k / 4) * gpitch + n], (int)(k % 4));
    return OR_OK;
}

/* ------------------------------------------------------------------ S4 / S6
 * T158 linear: acc[m][n] = sum_k trit[n][k] * xq[m][k], exact integer
 * arithmetic ([citric] "Step 1": results do not depend on thread count or
 * batch), then y = ((float)acc * w_scale) * x_scale in fp32, left to right
 * (one scale per matrix, [citric] "Step 2"; scale applied after the dot
 * product, [cpp20gemma]).  (float)acc is exact because |acc| < 2^24 for the
 * shapes in use; the function reports EINVAL otherwise.
 */
int or_t158_linear(const int8_t *xq, const float *xs, const uint8_t *packed, int64_t pitch, float ws,
                   int64_t M, int64_t N, int64_t K, int32_t *acc_out, float *y) {
    if (!xq || !xs || !packed || M < 1 || N < 1 || K < 1 || pitch < (K + 4) / 5) return OR_EINVAL;
    if (127 * K >= (1 << 24)) return OR_EINVAL;
    for (int64_t m = 0; m < M; m++) {
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; k++)
                acc += (int64_t)trit_of(packed[n * pitch + k / 5], (int)(k % 5)) * (int64_t)xq[m * K + k];
            if (acc_out) acc_out[m * N + n] = (int32_t)acc;
            if (y) y[m * N + n] = ((float)acc * ws) * xs[m];
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ fp32 building blocks
 * Pairwise summation (Higham, "The accuracy of floating point summation",
 * SIAM J. Sci. Comput. 1993): the n terms are padded with zeros to the next
 * power of two P and summed as a balanced binary tree, sum(a[0:P]) =
 * sum(a[0:P/2]) + sum(a[P/2:P]).  This fixes the fp32 rounding of every sum
 * that feeds a quantiser.
 */
static int64_t next_pow2(int64_t n) {
    int64_t p = 1;
    while (p < n) p <<= 1;
    return p;
}

float or_psum_f32(const float *a, int64_t n) {
    if (n <= 0) return 0.0f;
    int64_t P = next_pow2(n);
    float *b = (float *)malloc((size_t)P * sizeof(float));
    for (int64_t i = 0; i < P; i++) b[i] = (i < n) ? a[i] : 0.0f;
    for (int64_t len = P; len > 1; len >>= 1)
        for (int64_t i = 0; i < len / 2; i++) b[i] = b[2 * i] + b[2 * i + 1];
    float r = b[0];
    free(b);
    return r;
}

/* exp in fp32: Cody-Waite argument reduction (Cody & Waite, "Software Manual
 * for the Elementary Functions", 1980) x = n ln2 + r with ln2 split into a
 * short high part and a low part, then the degree-7 Taylor polynomial of e^r
 * in Horner form with fused multiply-adds, then an exact scaling by 2^n
 * (two power-of-two multiplies below the normal range, so the one rounding
 * into subnormals is the IEEE one).  |r| <= 0.35, so the truncation error is
 * below 6e-9 relative. */
static float pow2i(int e) { /* 2^e for -126 <= e <= 127 */
    uint32_t u = (uint32_t)(e + 127) << 23;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

float or_exp_f32(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return INFINITY;
    if (x < -103.972084045410156f) return 0.0f;
    const float LOG2E = 1.44269502162933349609375f; /* log2(e) rounded to fp32 */
    const float LN2_HI = 0.693145751953125f;          /* 0x3F317200: ln2 with 9 low zero bits */
    const float LN2_LO = 1.4286068203094172321e-06f;  /* ln2 - LN2_HI */
    float n = rintf(x * LOG2E);
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int e = (int)n;
    if (e > 127) return (p * pow2i(127)) * 2.0f;
    if (e < -126) return (p * pow2i(e + 64)) * pow2i(-64);
    return p * pow2i(e);
}

/* tanh(z) = 1 - 2 / (e^{2z} + 1), with the exp above. */
float or_tanh_f32(float z) {
    float e = or_exp_f32(2.0f * z);
    return 1.0f - 2.0f / (e + 1.0f);
}

/* GELU, tanh form (the form Gemma uses; the pages only say "GeLU"/"GeGLU"):
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), fp32, in this order. */
float or_gelu_f32(float x) {
    float x3 = (x * x) * x;
    float inner = x + 0.044715f * x3;
    float z = 0.7978845608028654f * inner;
    float t = or_tanh_f32(z);
    return (0.5f * x) * (1.0f + t);
}

/* ------------------------------------------------------------------ S9
 * RMSNorm, [llama2.c] Step 1: o = w * (x / sqrt(mean(x^2) + eps)), computed
 * as ss = sum x^2 (pairwise); ss = ss/n + eps; r = 1/sqrtf(ss); o = g*(r*x).
 */
void or_rmsnorm(const float *x, const float *g, int64_t n, float eps, float *o) {
    float *sq = (float *)malloc((size_t)n * sizeof(float));
    for (int64_t i = 0; i < n; i++) sq[i] = x[i] * x[i];
    float ss = or_psum_f32(sq, n);
    free(sq);
    ss = ss / (float)n;
    ss = ss + eps;
    float r = 1.0f / sqrtf(ss);
    for (int64_t i = 0; i < n; i++) o[i] = g[i] * (r * x[i]);
}

/* ------------------------------------------------------------------ S11
 * RoPE.  Frequencies as in [llama2.c] Step 2: theta_i = base^(-2i/head_dim),
 * angle = pos * theta_i, in double, cos/sin rounded to fp32.  Pairing (i,
 * i + head_dim/2), the Gemma convention of [gemma.cpp tour] "The Forward
 * Pass"; k is rotated before it is cached ([cpp20gemma]).  Rotation in fp32,
 * each product rounded, then added:  x' = x c - y s,  y' = x s + y c.
 */
void or_rope_table(int64_t n_pos, int64_t head_dim, double base, float *cos_t, float *sin_t) {
    int64_t half = head_dim / 2;
    for (int64_t p = 0; p < n_pos; p++)
        for (int64_t i = 0; i < half; i++) {
            double theta = pow(base, -(double)(2 * i) / (double)head_dim);
            double ang = (double)p * theta;
            cos_t[p * half + i] = (float)cos(ang);
            sin_t[p * half + i] = (float)sin(ang);
        }
}

void or_rope_apply(float *x, int64_t n_heads, int64_t head_dim, const float *c, const float *s) {
    int64_t half = head_dim / 2;
    for (int64_t h = 0; h < n_heads; h++) {
        float *v = x + h * head_dim;
        for (int64_t i = 0; i < half; i++) {
            float a = v[i], b = v[i + half];
            float ac = a * c[i], bs = b * s[i], as = a * s[i], bc = b * c[i];
            v[i] = ac - bs;
            v[i + half] = as + bc;
        }
    }
}

/* ------------------------------------------------------------------ S12
 * Decode attention, [llama2.c] Step 4: for each query head h (KV head
 * h / (n_heads/n_kv), the GQA rule), score_t = q.k_t / sqrt(head_dim) for
 * t <= pos, softmax with the maximum subtracted, out = sum_t p_t v_t.
 * Reading (fp32 order): dot products are pairwise sums of the rounded
 * products; positions are taken in chunks of ATT_CHUNK and the softmax is
 * assembled from per-chunk maxima and sums (the online-softmax identity
 * e^{s-m} = e^{s-m_c} e^{m_c-m}), all sums pairwise; out = U / S.
 * Mathematically this is the page's softmax; the fixed grouping fixes the
 * rounding.
 */
#define ATT_CHUNK 32

void or_attention(const float *q, const float *kc, const float *vc, int64_t pos, int64_t n_heads,
                  int64_t n_kv, int64_t head_dim, float *out) {
    int64_t kv_dim = n_kv * head_dim;
    int64_t kv_mul = n_heads / n_kv;
    int64_t T = pos + 1;
    int64_t nc = (T + ATT_CHUNK - 1) / ATT_CHUNK;
    float scale_div = sqrtf((float)head_dim);
    float *prod = (float *)malloc((size_t)head_dim * sizeof(float));
    float *s = (float *)malloc((size_t)(nc * ATT_CHUNK) * sizeof(float));
    float *mc = (float *)malloc((size_t)nc * sizeof(float));
    float *Sc = (float *)malloc((size_t)nc * sizeof(float));
    float *Uc = (float *)malloc((size_t)(nc * head_dim) * sizeof(float));
    float *tmp = (float *)malloc((size_t)(nc > ATT_CHUNK ? nc : ATT_CHUNK) * sizeof(float));
    for (int64_t h = 0; h < n_heads; h++) {
        const float *qh = q + h * head_dim;
        int64_t kvh = h / kv_mul;
        for (int64_t t = 0; t < T; t++) {
            const float *k = kc + t * kv_dim + kvh * head_dim;
            for (int64_t i = 0; i < head_dim; i++) prod[i] = qh[i] * k[i];
            s[t] = or_psum_f32(prod, head_dim) / scale_div;
        }
        for (int64_t c = 0; c < nc; c++) {
            int64_t t0 = c * ATT_CHUNK, t1 = t0 + ATT_CHUNK < T ? t0 + ATT_CHUNK : T;
            float m = s[t0];
            for (int64_t t = t0 + 1; t < t1; t++)
                if (s[t] > m) m = s[t];
            mc[c] = m;
            float e[ATT_CHUNK];
            for (int64_t t = t0; t < t1; t++) e[t - t0] = or_exp_f32(s[t] - m);
            Sc[c] = or_psum_f32(e, t1 - t0);
            for (int64_t i = 0; i < head_dim; i++) {
                for (int64_t t = t0; t < t1; t++) tmp[t - t0] = e[t - t0] * vc[t * kv_dim + kvh * head_dim + i];
                Uc[c * head_dim + i] = or_psum_f32(tmp, t1 - t0);
            }
        }
        float m = mc[0];
        for (int64_t c = 1; c < nc; c++)
            if (mc[c] > m) m = mc[c];
        float *w = (float *)malloc((size_t)nc * sizeof(float));
        for (int64_t c = 0; c < nc; c++) w[c] = or_exp_f32(mc[c] - m);
        for (int64_t c = 0; c < nc; c++) tmp[c] = Sc[c] * w[c];
        float S = or_psum_f32(tmp, nc);
        for (int64_t i = 0; i < head_dim; i++) {
            for (int64_t c = 0; c < nc; c++) tmp[c] = Uc[c * head_dim + i] * w[c];
            out[h * head_dim + i] = or_psum_f32(tmp, nc) / S;
        }
        free(w);
    }
    free(prod);
    free(s);
    free(mc);
    free(Sc);
    free(Uc);
    free(tmp);
}

/* ------------------------------------------------------------------ S8 .. S16: decode step
 * Pre-norm residual block of [cpp20gemma] "Architecture & implementation"
 * (h += attn(rmsnorm(h)); h += mlp(rmsnorm(h)); logits = lm_head(rmsnorm(h)))
 * in the order of [llama2.c] "The forward pass", with every linear layer a
 * T158 linear on int8-quantised inputs ([citric] "Step 2") and a GeGLU MLP
 * (down(gelu(gate x) * (up x)), [gemma.cpp tour], [cpp20gemma]).  No position
 * bias (zeros per [cpp20gemma] "Real Gemma weights"), embedding kept in bf16
 * and tied to the lm_head ([citric] "Step 2"; [llama2.c] "four structs").
 */
typedef struct {
    int64_t n_layers, dim, n_heads, n_kv_heads, head_dim, ffn, vocab, max_pos;
    float eps;
    double rope_base;
    const uint8_t *w[7]; /* wq wk wv wo wg wu wd, each [L][N][pitch] */
    int64_t pitch[7];
    const float *scales; /* [L][7] */
    const float *g_attn, *g_ffn, *g_final; /* [L][dim], [L][dim], [dim] */
    const uint16_t *emb;                   /* bf16 bits [vocab][dim] */
} or_model;

static float bf16f(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static void mat_dims(const or_model *m, int j, int64_t *N, int64_t *K) {
    int64_t d = m->dim, q = m->n_heads * m->head_dim, kv = m->n_kv_heads * m->head_dim, f = m->ffn;
    static const int rows_sel[7] = {0, 1, 1, 2, 3, 3, 2}; /* 0:q 1:kv 2:d 3:f */
    static const int cols_sel[7] = {2, 2, 2, 0, 2, 2, 3};
    int64_t v[4] = {q, kv, d, f};
    *N = v[rows_sel[j]];
    *K = v[cols_sel[j]];
}

static void t158_layer(const or_model *m, int l, int j, const float *x, int8_t *xq, float *y) {
    int64_t N, K;
    mat_dims(m, j, &N, &K);
    float xs;
    or_quant_i8(x, 1, K, xq, &xs);
    const uint8_t *w = m->w[j] + (int64_t)l * N * m->pitch[j];
    or_t158_linear(xq, &xs, w, m->pitch[j], m->scales[l * 7 + j], 1, N, K, NULL, y);
}

/* ------------------------------------------------------------------ sketch head
 * [citric] "Step 3: the output layer became the bottleneck": candidates first,
 * exact scores only for them.  (1) the k dimensions of x with the largest
 * values are scored exactly for every word; (2) the other dimensions are
 * scored from the signs of the table only -- one XOR and one bit count per 64
 * dimensions of a word -- with the dimensions grouped by size and one weight
 * per group; (3) the n_cand words with the best approximate scores are scored
 * exactly, every other word scores minus infinity.
 * Readings (the page gives the steps, not their arithmetic):
 * - "largest values" = largest |x_d|, ties to the lower index;
 * - a group is one B-dimension block of the stored sign table (B = 64 on the
 *   page: one XOR and one bit count per block), so grouping by size is a fixed
 *   order of the dimensions chosen when the table is prepared: perm lists the
 *   dimensions by a per-dimension size s_d (largest |s_d| first, ties to the
 *   lower index; the identity without sizes), block b holds positions
 *   bB .. bB+B-1 of that order;
 * - block b's weight is w_b = (mean |x_d| over its sketched dims) * cE, cE =
 *   the mean |E| of the table, so that w_b * (agreeing - differing signs)
 *   estimates the block's part of the dot product; the exact dims are left
 *   out of every block;
 * - the sign of E is the sign bit of its bf16 value, the sign of x its sign bit;
 * - ties among approximate scores go to the lower index.
 * The fp32 arithmetic is fixed so that two implementations select the same
 * candidates: the exact part is the pairwise sum (zero-padded to a power of
 * two) of the products bf16(E[v][d]) * x[d], d ascending over the k dims; a
 * block's |x| sum is the pairwise sum over its B positions in order, exact
 * dims and positions past D counting +0; the sketch is the sum over blocks in
 * order of w_b * (n_b - 2 m_b), each product rounded, then added; approx =
 * exact part + sketch.
 */
typedef struct {
    float key;
    int64_t idx;
} or_keyidx;

static int or_cmp_desc(const void *a, const void *b) {
    const or_keyidx *p = (const or_keyidx *)a, *q = (const or_keyidx *)b;
    if (p->key > q->key) return -1;
    if (p->key < q->key) return 1;
    return p->idx < q->idx ? -1 : p->idx > q->idx ? 1 : 0;
}

static int or_cmp_i64(const void *a, const void *b) {
    const int64_t p = *(const int64_t *)a, q = *(const int64_t *)b;
    return p < q ? -1 : p > q ? 1 : 0;
}

int or_sketch_perm(const float *scale, int64_t D, int64_t *perm) {
    if (!perm || D < 1) return OR_EINVAL;
    or_keyidx *ord = (or_keyidx *)malloc((size_t)D * sizeof(or_keyidx));
    for (int64_t d = 0; d < D; d++) {
        ord[d].key = scale ? fabsf(scale[d]) : 0.0f;
        ord[d].idx = d;
    }
    qsort(ord, (size_t)D, sizeof(or_keyidx), or_cmp_desc);
    for (int64_t i = 0; i < D; i++) perm[i] = ord[i].idx;
    free(ord);
    return OR_OK;
}

int or_sketch_ce(const uint16_t *emb, int64_t V, int64_t D, float *cE) {
    if (!emb || !cE || V < 1 || D < 1) return OR_EINVAL;
    double acc = 0.0;
    for (int64_t i = 0; i < V * D; i++) acc += fabs((double)bf16f(emb[i]));
    *cE = (float)(acc / (double)(V * D));
    return OR_OK;
}

int or_sketch_head(const uint16_t *emb, int64_t V, int64_t D, const int64_t *perm, int64_t B, const float *x,
                   int64_t k, int64_t n_cand, float cE, float *approx, int32_t *cand, float *cand_logits,
                   int32_t *next) {
    if (!emb || !perm || !x || !approx || !cand || !cand_logits || !next || V < 1 || D < 1 || B < 1 || k < 0 ||
        k > D || n_cand < 1 || n_cand > V)
        return OR_EINVAL;
    char *seen = (char *)calloc((size_t)D, 1);
    for (int64_t i = 0; i < D; i++) {
        if (perm[i] < 0 || perm[i] >= D || seen[perm[i]]) {
            free(seen);
            return OR_EINVAL;
        }
        seen[perm[i]] = 1;
    }
    free(seen);
    /* (1) the exact dims */
    or_keyidx *ord = (or_keyidx *)malloc((size_t)D * sizeof(or_keyidx));
    for (int64_t d = 0; d < D; d++) {
        ord[d].key = fabsf(x[d]);
        ord[d].idx = d;
    }
    qsort(ord, (size_t)D, sizeof(or_keyidx), or_cmp_desc);
    char *exact_dim = (char *)calloc((size_t)D, 1);
    int64_t *top = (int64_t *)malloc((size_t)(k > 0 ? k : 1) * sizeof(int64_t));
    for (int64_t j = 0; j < k; j++) {
        top[j] = ord[j].idx;
        exact_dim[top[j]] = 1;
    }
    qsort(top, (size_t)k, sizeof(int64_t), or_cmp_i64);
    /* (2) the blocks: sketched dims, counts and weights */
    const int64_t G = (D + B - 1) / B;
    float *wg = (float *)malloc((size_t)G * sizeof(float));
    int64_t *ng = (int64_t *)malloc((size_t)G * sizeof(int64_t));
    float *tmp = (float *)malloc((size_t)B * sizeof(float));
    for (int64_t g = 0; g < G; g++) {
        ng[g] = 0;
        for (int64_t p = 0; p < B; p++) {
            const int64_t i = g * B + p;
            const int in = i < D && !exact_dim[perm[i]];
            tmp[p] = in ? fabsf(x[perm[i]]) : 0.0f;
            ng[g] += in;
        }
        wg[g] = ng[g] > 0 ? (or_psum_f32(tmp, B) / (float)ng[g]) * cE : 0.0f;
    }
#pragma omp parallel
    {
        float *prod = (float *)malloc((size_t)(k > 0 ? k : 1) * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t v = 0; v < V; v++) {
            const uint16_t *e = emb + v * D;
            for (int64_t j = 0; j < k; j++) prod[j] = bf16f(e[top[j]]) * x[top[j]];
            const float exact = k > 0 ? or_psum_f32(prod, k) : 0.0f;
            float sk = 0.0f;
            for (int64_t g = 0; g < G; g++) {
                int64_t mism = 0;
                for (int64_t p = 0; p < B && g * B + p < D; p++) {
                    const int64_t d = perm[g * B + p];
                    if (exact_dim[d]) continue;
                    mism += (int64_t)((e[d] >> 15) != (uint16_t)(signbit(x[d]) ? 1 : 0));
                }
                const float t = (float)(ng[g] - 2 * mism);
                sk = sk + wg[g] * t;
            }
            approx[v] = exact + sk;
        }
        free(prod);
    }
    /* (3) candidates and their exact scores */
    or_keyidx *all = (or_keyidx *)malloc((size_t)V * sizeof(or_keyidx));
    for (int64_t v = 0; v < V; v++) {
        all[v].key = approx[v];
        all[v].idx = v;
    }
    qsort(all, (size_t)V, sizeof(or_keyidx), or_cmp_desc);
    int64_t *cv = (int64_t *)malloc((size_t)n_cand * sizeof(int64_t));
    for (int64_t i = 0; i < n_cand; i++) cv[i] = all[i].idx;
    qsort(cv, (size_t)n_cand, sizeof(int64_t), or_cmp_i64);
    int32_t best = -1;
    float bv = 0.0f;
    for (int64_t i = 0; i < n_cand; i++) {
        const uint16_t *e = emb + cv[i] * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; d++) acc += (double)bf16f(e[d]) * (double)x[d];
        cand[i] = (int32_t)cv[i];
        cand_logits[i] = (float)acc;
        if (best < 0 || cand_logits[i] > bv) {
            best = (int32_t)cv[i];
            bv = cand_logits[i];
        }
    }
    *next = best;
    free(ord);
    free(exact_dim);
    free(top);
    free(wg);
    free(ng);
    free(tmp);
    free(all);
    free(cv);
    return OR_OK;
}

/* S16: logits[r] = sum_i bf16(emb[r][i]) * x[i] in fp64, rounded to fp32
 * ([llama2.c] Step 6), and the greedy token: the first maximum wins
 * ([llama2.c] "Sampling", strict > in the argmax loop). */
void or_lm_head_argmax(const uint16_t *emb, const float *x, int64_t vocab, int64_t dim, float *logits, int32_t *next) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < vocab; r++) {
        double acc = 0.0;
        const uint16_t *e = emb + r * dim;
        for (int64_t i = 0; i < dim; i++) acc += (double)bf16f(e[i]) * (double)x[i];
        logits[r] = (float)acc;
    }
    int32_t best = 0;
    for (int64_t r = 1; r < vocab; r++)
        if (logits[r] > logits[best]) best = (int32_t)r;
    if (next) *next = best;
}

/* One forward step at position pos: writes rotated k and v into the cache
 * [L][2][max_pos][kv_dim], fp32 logits [vocab] (may be NULL) and the greedy
 * token ([llama2.c] "Sampling": first maximum wins).  logits are fp64 sums
 * rounded to fp32. */
static int decode_hidden(const or_model *m, float *kv, int32_t token, int64_t pos, float *xn_out) {
    if (!m || !kv || pos < 0 || pos >= m->max_pos || token < 0 || token >= m->vocab) return OR_EINVAL;
    int64_t d = m->dim, qd = m->n_heads * m->head_dim, kvd = m->n_kv_heads * m->head_dim, f = m->ffn;
    int64_t half = m->head_dim / 2;
    int64_t big = f > qd ? f : qd;
    if (d > big) big = d;
    float *h = (float *)malloc((size_t)d * 4), *xn = (float *)malloc((size_t)d * 4);
    float *q = (float *)malloc((size_t)qd * 4), *k = (float *)malloc((size_t)kvd * 4);
    float *v = (float *)malloc((size_t)kvd * 4), *att = (float *)malloc((size_t)qd * 4);
    float *y = (float *)malloc((size_t)big * 4), *g = (float *)malloc((size_t)f * 4);
    float *u = (float *)malloc((size_t)f * 4);
    int8_t *xq = (int8_t *)malloc((size_t)big);
    float *rc = (float *)malloc((size_t)half * 4), *rs = (float *)malloc((size_t)half * 4);

    /* Step 0: embed */
    for (int64_t i = 0; i < d; i++) h[i] = bf16f(m->emb[(int64_t)token * d + i]);
    /* RoPE table row for this position */
    for (int64_t i = 0; i < half; i++) {
        double theta = pow(m->rope_base, -(double)(2 * i) / (double)m->head_dim);
        double ang = (double)pos * theta;
        rc[i] = (float)cos(ang);
        rs[i] = (float)sin(ang);
    }
    for (int64_t l = 0; l < m->n_layers; l++) {
        float *kc = kv + ((l * 2 + 0) * m->max_pos) * kvd;
        float *vc = kv + ((l * 2 + 1) * m->max_pos) * kvd;
        /* Step 1: RMSNorm, quantise, Q K V */
        or_rmsnorm(h, m->g_attn + l * d, d, m->eps, xn);
        t158_layer(m, (int)l, 0, xn, xq, q);
        t158_layer(m, (int)l, 1, xn, xq, k);
        t158_layer(m, (int)l, 2, xn, xq, v);
        /* Step 2: RoPE on q and k;  Step 3: cache write */
        or_rope_apply(q, m->n_heads, m->head_dim, rc, rs);
        or_rope_apply(k, m->n_kv_heads, m->head_dim, rc, rs);
        memcpy(kc + pos * kvd, k, (size_t)kvd * 4);
        memcpy(vc + pos * kvd, v, (size_t)kvd * 4);
        /* Step 4: attention, then output projection and residual */
        or_attention(q, kc, vc, pos, m->n_heads, m->n_kv_heads, m->head_dim, att);
        t158_layer(m, (int)l, 3, att, xq, y);
        for (int64_t i = 0; i < d; i++) h[i] = h[i] + y[i];
        /* Step 5: FFN (GeGLU) and residual */
        or_rmsnorm(h, m->g_ffn + l * d, d, m->eps, xn);
        t158_layer(m, (int)l, 4, xn, xq, g);
        t158_layer(m, (int)l, 5, xn, xq, u);
        for (int64_t i = 0; i < f; i++) g[i] = or_gelu_f32(g[i]) * u[i];
        t158_layer(m, (int)l, 6, g, xq, y);
        for (int64_t i = 0; i < d; i++) h[i] = h[i] + y[i];
    }
    /* Step 6 (first half): final norm */
    or_rmsnorm(h, m->g_final, d, m->eps, xn_out);

    free(h); free(xn); free(q); free(k); free(v); free(att); free(y); free(g); free(u); free(xq);
    free(rc); free(rs);
    return OR_OK;
}

int or_decode_step(const or_model *m, float *kv, int32_t token, int64_t pos, float *logits, int32_t *next) {
    if (!m || !next) return OR_EINVAL;
    float *xn = (float *)malloc((size_t)(m->dim > 0 ? m->dim : 1) * 4);
    const int rc = decode_hidden(m, kv, token, pos, xn);
    if (rc == OR_OK) {
        /* Step 6 (second half): classifier (tied bf16 table) */
        float *lg = logits ? logits : (float *)malloc((size_t)m->vocab * 4);
        or_lm_head_argmax(m->emb, xn, m->vocab, m->dim, lg, next);
        if (!logits) free(lg);
    }
    free(xn);
    return rc;
}

/* The same forward step up to the final norm: the hidden state the output
 * layer scores (for a sketch head in place of the full classifier). */
int or_decode_hidden(const or_model *m, float *kv, int32_t token, int64_t pos, float *xn) {
    if (!m || !xn) return OR_EINVAL;
    return decode_hidden(m, kv, token, pos, xn);
}

/* A step over M lanes ([citric] "Many users at once": a lane is one token of
 * one sequence at one position; batches of users and chunks of a prompt go
 * through the same step).  Lane i takes token[i] at position pos[i] of
 * sequence seq[i], whose KV cache is kv + seq[i] * (L * 2 * max_pos * kvd).
 * Layer by layer: every lane's k and v are written to its cache before any
 * lane attends, so a lane sees the positions <= its own that other lanes of
 * its sequence write in the same step.  Each lane's arithmetic is the single
 * token step's.  logits: fp32 [M][vocab] or NULL; next: [M]. */
int or_decode_lanes(const or_model *m, float *kv, int64_t n_seqs, int64_t M, const int32_t *token, const int32_t *pos,
                    const int32_t *seq, float *logits, int32_t *next) {
    if (!m || !kv || !token || !pos || !seq || !next || M < 1 || n_seqs < 1) return OR_EINVAL;
    for (int64_t i = 0; i < M; i++)
        if (pos[i] < 0 || pos[i] >= m->max_pos || token[i] < 0 || token[i] >= m->vocab || seq[i] < 0 ||
            seq[i] >= n_seqs)
            return OR_EINVAL;
    const int64_t d = m->dim, qd = m->n_heads * m->head_dim, kvd = m->n_kv_heads * m->head_dim, f = m->ffn;
    const int64_t half = m->head_dim / 2, L = m->n_layers;
    const int64_t per_seq = L * 2 * m->max_pos * kvd;
    int64_t big = f > qd ? f : qd;
    if (d > big) big = d;
    float *h = (float *)malloc((size_t)(M * d) * 4), *xn = (float *)malloc((size_t)d * 4);
    float *q = (float *)malloc((size_t)(M * qd) * 4), *k = (float *)malloc((size_t)kvd * 4);
    float *v = (float *)malloc((size_t)kvd * 4), *att = (float *)malloc((size_t)qd * 4);
    float *y = (float *)malloc((size_t)big * 4), *g = (float *)malloc((size_t)f * 4);
    float *u = (float *)malloc((size_t)f * 4);
    int8_t *xq = (int8_t *)malloc((size_t)big);
    float *rc = (float *)malloc((size_t)(M * half) * 4), *rs = (float *)malloc((size_t)(M * half) * 4);
    for (int64_t i = 0; i < M; i++) {
        for (int64_t e = 0; e < d; e++) h[i * d + e] = bf16f(m->emb[(int64_t)token[i] * d + e]);
        for (int64_t e = 0; e < half; e++) {
            double theta = pow(m->rope_base, -(double)(2 * e) / (double)m->head_dim);
            double ang = (double)pos[i] * theta;
            rc[i * half + e] = (float)cos(ang);
            rs[i * half + e] = (float)sin(ang);
        }
    }
    for (int64_t l = 0; l < L; l++) {
        /* every lane: norm, q k v, rotation, cache write */
        for (int64_t i = 0; i < M; i++) {
            float *kc = kv + seq[i] * per_seq + ((l * 2 + 0) * m->max_pos) * kvd;
            float *vc = kv + seq[i] * per_seq + ((l * 2 + 1) * m->max_pos) * kvd;
            or_rmsnorm(h + i * d, m->g_attn + l * d, d, m->eps, xn);
            t158_layer(m, (int)l, 0, xn, xq, q + i * qd);
            t158_layer(m, (int)l, 1, xn, xq, k);
            t158_layer(m, (int)l, 2, xn, xq, v);
            or_rope_apply(q + i * qd, m->n_heads, m->head_dim, rc + i * half, rs + i * half);
            or_rope_apply(k, m->n_kv_heads, m->head_dim, rc + i * half, rs + i * half);
            memcpy(kc + (int64_t)pos[i] * kvd, k, (size_t)kvd * 4);
            memcpy(vc + (int64_t)pos[i] * kvd, v, (size_t)kvd * 4);
        }
        /* every lane: attention, output projection, FFN */
        for (int64_t i = 0; i < M; i++) {
            const float *kc = kv + seq[i] * per_seq + ((l * 2 + 0) * m->max_pos) * kvd;
            const float *vc = kv + seq[i] * per_seq + ((l * 2 + 1) * m->max_pos) * kvd;
            float *hi = h + i * d;
            or_attention(q + i * qd, kc, vc, pos[i], m->n_heads, m->n_kv_heads, m->head_dim, att);
            t158_layer(m, (int)l, 3, att, xq, y);
            for (int64_t e = 0; e < d; e++) hi[e] = hi[e] + y[e];
            or_rmsnorm(hi, m->g_ffn + l * d, d, m->eps, xn);
            t158_layer(m, (int)l, 4, xn, xq, g);
            t158_layer(m, (int)l, 5, xn, xq, u);
            for (int64_t e = 0; e < f; e++) g[e] = or_gelu_f32(g[e]) * u[e];
            t158_layer(m, (int)l, 6, g, xq, y);
            for (int64_t e = 0; e < d; e++) hi[e] = hi[e] + y[e];
        }
    }
    float *lg = (float *)malloc((size_t)m->vocab * 4);
    for (int64_t i = 0; i < M; i++) {
        or_rmsnorm(h + i * d, m->g_final, d, m->eps, xn);
        or_lm_head_argmax(m->emb, xn, m->vocab, d, logits ? logits + i * m->vocab : lg, next + i);
    }
    free(lg);
    free(h); free(xn); free(q); free(k); free(v); free(att); free(y); free(g); free(u); free(xq);
    free(rc); free(rs);
    return OR_OK;
}

/* [llama2.c] "The generation loop": force-feed the prompt, then feed back
 * the greedy token.  Runs n_steps forwards at positions start_pos ...; out
 * receives the argmax of every forward (for prompt positions too). */
int or_decode_generate(const or_model *m, float *kv, const int32_t *prompt, int64_t n_prompt,
                       int64_t start_pos, int64_t n_steps, int32_t *out) {
    if (!prompt || n_prompt < 1 || !out) return OR_EINVAL;
    int32_t token = prompt[0];
    for (int64_t s = 0; s < n_steps; s++) {
        int32_t nx;
        int rc = or_decode_step(m, kv, token, start_pos + s, NULL, &nx);
        if (rc) return rc;
        out[s] = nx;
        token = (s + 1 < n_prompt) ? prompt[s + 1] : nx;
    }
    return OR_OK;
}
