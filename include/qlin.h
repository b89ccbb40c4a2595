/*
 * qlin -- quantised-weight linear layers and a ternary decode step for GB300
 * (sm_103a).  C ABI, no C++ or torch types.
 *
 * What is computed comes from four web pages, cited by title and section:
 *   [gemma.cpp tour]  "gemma.cpp" (pyshine.com)
 *   [cpp20gemma]      cpp20gemma README
 *   [llama2.c]        "llama2.c -- Llama-2 Inference in One C File"
 *   [citric]          "Gemma 3 1B at 114 tokens per second on a laptop CPU"
 *
 * Conventions for every call:
 *  - Matrices are row-major [out][in] ([cpp20gemma] "Architecture &
 *    implementation": each output row is contiguous).  A "pitch" is the byte
 *    distance between rows.
 *  - "device" pointers are CUDA global-memory addresses of the current
 *    device; "host" pointers are ordinary CPU memory.  The caller owns every
 *    buffer; no call allocates or frees device memory, and none keeps a
 *    pointer after it returns.
 *  - Device calls are asynchronous on `stream` (NULL = the legacy default
 *    stream).  Arguments are validated on the host before anything is
 *    launched; a rejected call launches nothing and returns a status != 0.
 *    Launch failures return QLIN_ERR_CUDA.  Faults inside a kernel surface at
 *    the caller's next synchronisation, like any CUDA work.
 *  - qlin_last_error() gives a thread-local message for the last failure.
 *  - Device pointers must be 16-byte aligned unless stated otherwise.
 */
#ifndef QLIN_H
#define QLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qlin_stream_t; /* the same type as cudaStream_t */

typedef enum {
    QLIN_OK = 0,
    QLIN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer or pitch */
    QLIN_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement */
    QLIN_ERR_BAD_PACKED = 3,  /* t158_unpack: a byte above 242 */
    QLIN_ERR_CUDA = 4,        /* a CUDA runtime call failed */
    QLIN_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see decode_step_t158) */
} qlin_status;

/* Name of a status code; never NULL. */
const char *qlin_status_str(int status);
/* Detail of the calling thread's last failed call ("" if none); valid until its next call. */
const char *qlin_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int qlin_version(void);

/* ========================================================================
 * S2  T158 packing  ([citric] "Step 1: a kernel for 1.6-bit weights": five
 * ternary weights per byte, 3^5 = 243 <= 256).  Byte j of a row holds trits
 * 5j..5j+4 as base-3 digits d_i = trit + 1, least significant first:
 * byte = sum_i d_i 3^i.  Trits past K are zero trits, so filler bytes past
 * ceil(K/5) are 121.  Host, synchronous.
 * ====================================================================== */

/* Row pitch the GPU kernels take for K trits: ceil(ceil(K/5) / 16) * 16 bytes. */
int64_t t158_pitch(int64_t K);

/* trits: host int8 [N][K] in {-1,0,+1}; packed: host uint8 [N][pitch], pitch >= ceil(K/5).
 * INVALID_ARG on a null pointer, N/K < 1, short pitch or a trit outside {-1,0,1}. */
qlin_status t158_pack(const int8_t *trits, int64_t N, int64_t K, uint8_t *packed, int64_t pitch);

/* Inverse of t158_pack; every byte of every row (filler included) is checked first:
 * BAD_PACKED if any is above 242, and then nothing is written. */
qlin_status t158_unpack(const uint8_t *packed, int64_t N, int64_t K, int64_t pitch, int8_t *trits);

/* ========================================================================
 * S1  W8 weight quantisation ([cpp20gemma] "Architecture & implementation":
 * scale = max(|w|, 1e-9)/127, w8 = clip(round(w/scale)); round half to even,
 * clip +-127).  One scale for the whole tensor.  Device, asynchronous.
 * w: device fp32 [N][K] (row stride K, 4-byte aligned); w8: device int8
 * [N][w_pitch], w_pitch >= K and a multiple of 16 (bytes past K are zeroed);
 * scale: device fp32 [1] (written last).
 * ====================================================================== */
qlin_status qlin_w8_quantize(const float *w, int64_t N, int64_t K, int8_t *w8, int64_t w_pitch,
                             float *scale, qlin_stream_t stream);

/* ========================================================================
 * S3  Activation quantisation ([citric] "Step 2": the inputs to each layer
 * are rounded to int8; [llama2.c] "Key ideas": dynamic symmetric +-127).
 * Per row m: x_scale[m] = max(max_k |x[m][k]|, 1e-9)/127, xq = clip(
 * rint(x / x_scale), +-127), fp32 division, ties to even.
 * x: device fp32 [M][K] (4-byte aligned); xq: device int8 [M][K] (any
 * alignment); x_scale: device fp32 [M] (4-byte aligned).
 * ====================================================================== */
qlin_status qlin_quant_i8(const float *x, int8_t *xq, float *x_scale, int M, int K, qlin_stream_t stream);

/* ========================================================================
 * S4 + S6 (+ S7 for large M)  T158 linear.
 *   acc[m][n] = sum_{k<K} trit[n][k] * xq[m][k]          (exact int32)
 *   y[m][n]   = ((float)acc[m][n] * w_scale) * x_scale[m] (fp32, in this order)
 * ([citric] "Step 1": exact integer arithmetic; "Step 2": one scale per
 * matrix, int8 inputs; [cpp20gemma]: scale applied once after the dot.)
 * xq: device int8 [M][K] (any alignment); x_scale: device fp32 [M];
 * w_packed: device uint8 [N][w_pitch] as written by t158_pack, w_pitch a
 * multiple of 16 and >= ceil(K/5), base 16-byte aligned; y: device fp32
 * [M][N] or NULL; acc: device int32 [M][N] or NULL (at least one non-NULL).
 * Bytes above 242 in w_packed give unspecified but memory-safe results.
 * M: 1..4096.  K: 1..131071 (so that |acc| stays below 2^24 and the fp32
 * epilogue is exact).  UNSUPPORTED outside these ranges.
 * From M = 8 tokens (prefill and batched decode, [citric] "Step 1: a kernel for 1.6-bit
 * weights": all prompt tokens through each matrix in one pass) the products run on the tensor cores as an fp16
 * matrix product with fp32 accumulation, exact for these operands (int8
 * codes and trits are fp16 integers and every partial sum stays below
 * 127 K < 2^24): the same acc and y, bit for bit.  Below 8 tokens the
 * CUDA-core kernel runs, except for rows too long for its activation planes
 * in shared memory, which take the tensor-core path as well.  Both kernels
 * are launched with programmatic stream serialisation (the tensor-core one
 * except behind a large activation-tile conversion): each may start while the
 * previous kernel on the stream finishes and begins its weight reads at once
 * (the packed weights and their scale are taken to be read-only inputs); it
 * reads the activations and their scales, and writes y and acc, only after
 * that kernel has completed.
 * ====================================================================== */
qlin_status qlin_t158_i8(const int8_t *xq, const float *x_scale, const uint8_t *w_packed, int64_t w_pitch,
                         float w_scale, float *y, int32_t *acc, int M, int N, int K, qlin_stream_t stream);

/* qlin_t158_i8 with caller scratch for the tensor-core path: the int8 codes
 * are converted once per call into fp16 activation tiles in the workspace
 * (one launch), instead of once per 128 weight rows inside the product.  The
 * same acc and y, bit for bit.  workspace: device, 16-byte aligned, at least
 * qlin_t158_i8_workspace_size(M, K) bytes (0 below the tensor-core threshold
 * of 8 tokens, where NULL is accepted), owned by the caller, overwritten; a
 * smaller or misaligned workspace is QLIN_ERR_INVALID_ARG.  Other arguments
 * and ranges as qlin_t158_i8.  qlin_t158_i8_workspace_size returns 0 for M or
 * K out of range. */
size_t qlin_t158_i8_workspace_size(int M, int K);
qlin_status qlin_t158_i8_ws(const int8_t *xq, const float *x_scale, const uint8_t *w_packed, int64_t w_pitch,
                            float w_scale, float *y, int32_t *acc, int M, int N, int K, void *workspace,
                            size_t workspace_bytes, qlin_stream_t stream);

/* T158 linear for one token that skips groups of four zero inputs ([citric]
 * "What is next": a kernel that skips groups of 4 zero inputs).  Same acc and
 * y as qlin_t158_i8 with M = 1, from weights stored by input group:
 * t158_pack_groups writes w_groups uint8 [ceil(K/4)][gpitch], byte [g][n] =
 * sum_i (trit[n][4g+i] + 1) * 3^i (trits past K zero; rows N .. gpitch-1 the
 * byte 40), so the weights of one input group are gpitch contiguous bytes and
 * a group of four zero codes costs no weight bytes.  gpitch >= N, a multiple
 * of 16 (t158_group_pitch(N)); w_groups 16-byte aligned; xq device int8 [K]
 * and x_scale device fp32 [1], 4-byte aligned.  K <= 65536.  Workspace:
 * qlin_t158_skip_workspace_size(N) bytes, zero-filled before first use; calls
 * leave it ready; calls sharing it must not overlap.  Bytes above 80 give
 * unspecified but memory-safe results. */
int64_t t158_group_pitch(int64_t N);
qlin_status t158_pack_groups(const int8_t *trits, int64_t N, int64_t K, uint8_t *w_groups, int64_t gpitch);
size_t qlin_t158_skip_workspace_size(int N);
qlin_status qlin_t158_i8_skip(const int8_t *xq, const float *x_scale, const uint8_t *w_groups, int64_t gpitch,
                              float w_scale, float *y, int32_t *acc, int N, int K, void *workspace,
                              size_t workspace_bytes, qlin_stream_t stream);

/* ========================================================================
 * S5  W8 linear: y[m][n] = (sum_k x[m][k] * w8[n][k]) * w_scale, fp32
 * activations, the scale applied once after the dot product
 * ([cpp20gemma] "Architecture & implementation"; [llama2.c] "matmul").
 * x: device fp32 [M][K] (4-byte aligned); w8: device int8 [N][w_pitch],
 * w_pitch >= K, multiple of 16, base 16-byte aligned; y: device fp32 [M][N].
 * M: 1..64.  Accuracy: within 1e-5 of max|y| (max-abs-rel against the exact
 * dot product) on the parity inputs.
 * One token (M = 1, K <= 16384): the weights stream through shared memory by
 * bulk copies and the dot products are integer: the slice of x a lane owns
 * (at most four 16-element chunks) is held as 22-bit fixed point on a
 * power-of-two scale 2^e from that slice's largest |x| (largest |x| < 2^e;
 * three int8 limbs, dp4a), i.e. every x is rounded to within 2^(e-23).  So
 * |y[n] - exact| <= w_scale * sum_k 2^(e(k)-23) |w8[n][k]| plus fp32 rounding
 * of at most 2^-19 w_scale sum_k |x[k] w8[n][k]|, e(k) the exponent of k's
 * slice.  That is within 1e-5 of max|y| when the magnitudes inside a slice
 * are alike (N(0,1) inputs, or outliers whose weights are not zero); an
 * input with a large outlier beside small values whose weights cancel the
 * outlier's row sums can exceed it, up to the bound.  A NaN or an infinity
 * in x makes every y NaN.
 * Two to 64 tokens run on the tensor cores (tcgen05.mma, fp32 accumulator
 * in tensor memory): each int8 weight is a bf16 value exactly and each x
 * enters as three bf16 terms hi + mid + lo that hold all of its 24
 * significant bits, so every product is exact and the error is the fp32
 * accumulation's: |y[n] - exact| <= about K 2^-24 w_scale sum_k |x[k]
 * w8[n][k]| in the worst case, far less on random signs.  A NaN or an
 * infinity in x, or |x| above the largest bf16 (about 3.39e38), makes the
 * outputs of its token NaN.
 * The kernels are launched with programmatic stream serialisation: they may
 * start while the previous kernel on the stream finishes.  The weights are
 * taken to be read-only inputs: the kernels start their weight copies at
 * once, and wait for the previous kernel's completion before they read x or
 * write y.
 * ====================================================================== */
qlin_status qlin_w8_f32(const float *x, const int8_t *w8, int64_t w_pitch, float w_scale, float *y, int M, int N,
                        int K, qlin_stream_t stream);

/* qlin_w8_f32 with caller scratch for 2 <= M <= 64: the activations are
 * turned into the tensor cores' operand once per call (one small launch per
 * token) instead of inside the product for every 128 weight rows, and the
 * weights enter the product as fp16.  fp16's exponent range is narrow, so
 * each token's x is scaled by a power of two, x' = x 2^(14-e) with max|x| <
 * 2^e, split into three fp16 terms (exact down to fp16's subnormal step,
 * i.e. every x to within 2^(e-39)), and the output is multiplied back by
 * 2^(e-14): the error is the fp32 accumulation's, as for qlin_w8_f32.  A
 * NaN or an infinity in x makes its token's outputs NaN.
 * workspace: device, 16-byte aligned, at least qlin_w8_f32_workspace_size(M,
 * K) bytes (0 for M = 1, where NULL is accepted and the call is
 * qlin_w8_f32's), owned by the caller and overwritten; calls sharing a
 * workspace must not overlap on the GPU (calls on one stream do not).  A
 * smaller or misaligned workspace is QLIN_ERR_INVALID_ARG.  Other arguments
 * and ranges as qlin_w8_f32.  qlin_w8_f32_workspace_size returns 0 for M
 * outside 2..64 or K < 1. */
size_t qlin_w8_f32_workspace_size(int M, int K);
qlin_status qlin_w8_f32_ws(const float *x, const int8_t *w8, int64_t w_pitch, float w_scale, float *y, int M, int N,
                           int K, void *workspace, size_t workspace_bytes, qlin_stream_t stream);

/* ========================================================================
 * W8 with one scale per group of G weights ([gemma.cpp tour] "The compression
 * formats": I8Stream, int8 groups of 128 with a shared scale; [llama2.c] "Key
 * ideas & tradeoffs": runq.c's Q8_0, symmetric +-127, weights only).  The
 * groups are G consecutive weights of a row along K (the last group of a row
 * is shorter when G does not divide K); each is quantised with the W8 rule:
 * scale = max(|w|, 1e-9) / 127 (fp32 division), codes rint(w / scale)
 * (half to even), clip +-127.
 * qlin_w8g_quantize: w device fp32 [N][K] (4-byte aligned); w8 device int8
 * [N][w_pitch] (16-byte aligned, w_pitch >= K, multiple of 16; bytes past K
 * written 0); scales device fp32 [N][s_pitch] (16-byte aligned, s_pitch >=
 * ceil(K/G), multiple of 4; slots past ceil(K/G) written 0).  G: a multiple
 * of 16, >= 16 (128 in the cited formats).
 * qlin_w8g_f32: y[m][n] = sum_g scales[n][g] * sum_{k in g} x[m][k] w8[n][k],
 * fp32 activations as qlin_w8_f32 (the same one-token kernel, each 16-weight
 * chunk's dot product taking its group's scale); x device fp32 [M][K]; y
 * device fp32 [M][N]; M: 1..64.  Accuracy as qlin_w8_f32.
 * Both asynchronous on `stream`; INVALID_ARG for bad sizes or alignment.
 * ====================================================================== */
qlin_status qlin_w8g_quantize(const float *w, int64_t N, int64_t K, int G, int8_t *w8, int64_t w_pitch, float *scales,
                              int64_t s_pitch, qlin_stream_t stream);
qlin_status qlin_w8g_f32(const float *x, const int8_t *w8, int64_t w_pitch, const float *scales, int64_t s_pitch, int G,
                         float *y, int M, int N, int K, qlin_stream_t stream);

/* ========================================================================
 * Decode-step building blocks (each also runs fused inside decode_step_t158).
 * ====================================================================== */

/* S8  Embedding lookup ([llama2.c] Step 0; no position bias, [cpp20gemma]
 * "Real Gemma weights"): h[i] = (float)emb[token][i].  emb: device bf16 bits
 * [vocab][dim]; token: device int32 [1]; h: device fp32 [dim].  An
 * out-of-range token writes zeros and sets *status_word (device int32, may be
 * NULL) to 1. */
qlin_status qlin_embed_bf16(const uint16_t *emb, int vocab, int dim, const int32_t *token, float *h,
                            int32_t *status_word, qlin_stream_t stream);

/* S9  RMSNorm ([llama2.c] Step 1): o = g * (r * x), r = 1/sqrtf(ss/n + eps),
 * ss = sum x^2 as a balanced pairwise sum (zero-padded to a power of two).
 * x, g, out: device fp32 [M][n] / [n] / [M][n]; out may alias x. */
qlin_status qlin_rmsnorm(const float *x, const float *gamma, float *out, int M, int n, float eps,
                         qlin_stream_t stream);

/* S11 (table)  RoPE tables: cos/sin[p][i] = (float)cos|sin(p * base^(-2i/head_dim)),
 * angle in double ([llama2.c] Step 2).  cos_t, sin_t: device fp32 [max_pos][head_dim/2]. */
qlin_status t158_rope_table(float *cos_t, float *sin_t, int max_pos, int head_dim, double base,
                            qlin_stream_t stream);

/* S11  RoPE with (i, i + head_dim/2) pairs ([gemma.cpp tour] "The Forward
 * Pass"), rotate-then-cache ([cpp20gemma]): q [n_heads][head_dim] is rotated
 * in place; k [n_kv][head_dim] is rotated and written with v to
 * k_cache[pos], v_cache[pos] (device fp32 [max_pos][n_kv*head_dim]).
 * Rotation in fp32, products rounded then added. */
qlin_status qlin_rope_kv_append(float *q, const float *k, const float *v, float *k_cache, float *v_cache,
                                const float *cos_t, const float *sin_t, int pos, int n_heads, int n_kv,
                                int head_dim, qlin_stream_t stream);

/* S12  Decode attention ([llama2.c] Step 4): for query head h (KV head
 * h/(n_heads/n_kv)), softmax over t <= pos of q.k_t/sqrt(head_dim), then
 * sum_t p_t v_t.  fp32 with a fixed order: dot products and every sum are
 * pairwise; positions go in chunks of 32 whose maxima and sums are merged
 * with the online-softmax identity.  q: device fp32 [n_heads][head_dim]
 * (rotated); caches as in qlin_rope_kv_append; out: device fp32
 * [n_heads][head_dim]; workspace: device scratch of
 * qlin_attention_workspace_size() bytes.  head_dim: 16..256, power of two. */
size_t qlin_attention_workspace_size(int max_pos, int n_heads, int head_dim);
qlin_status qlin_attention_decode(const float *q, const float *k_cache, const float *v_cache, int pos,
                                  int n_heads, int n_kv, int head_dim, float *out, void *workspace,
                                  size_t workspace_bytes, qlin_stream_t stream);

/* Decode attention with no workspace argument, for callers that cannot
 * allocate device memory (a plugin inside an application that owns all device
 * memory and gives it no allocator, a real-time loop that cannot risk an
 * allocation's latency or failure, a process that reserved its memory up
 * front).  The pages have no counterpart: this is the same computation as
 * qlin_attention_decode, whose chunk partials here go to a fixed array of
 * QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES inside the library instead of a
 * caller workspace.  Every GPU that loads the library holds that array until
 * the process exits.  The call allocates nothing.
 *  - Size limit: n_heads * ceil((pos+1)/32) * (head_dim + 2) * 4 bytes must fit
 *    in the array (e.g. 4 heads of 256 up to pos 2015); larger calls return
 *    QLIN_ERR_UNSUPPORTED and launch nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is cached per device ordinal
 *    and belongs to the device's primary context: after cudaDeviceReset, or
 *    from a context other than the primary one, the cached address is no
 *    longer valid, so such callers must not use this entry point.
 *  - All calls share the one array and it keeps the last call's contents
 *    (nothing in it needs to start at zero): calls whose kernels overlap on
 *    the GPU, e.g. on two streams, race on it and give wrong results.
 * Other arguments as in qlin_attention_decode. */
#define QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES 262144
qlin_status qlin_attention_decode_noalloc(const float *q, const float *k_cache, const float *v_cache, int pos,
                                          int n_heads, int n_kv, int head_dim, float *out, qlin_stream_t stream);

/* S14 (activation)  GeGLU: a = gelu(g) * u with the tanh form of GELU
 * (0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))), [gemma.cpp tour],
 * [cpp20gemma]); tanh(z) = 1 - 2/(e^{2z} + 1) with a Cody-Waite fp32 exp.
 * g, u, a: device fp32 [n]; a may alias g or u. */
qlin_status qlin_geglu(const float *g, const float *u, float *a, int n, qlin_stream_t stream);

/* S16  lm_head + greedy pick ([llama2.c] Step 6 and "Sampling"):
 * logits[v] = sum_i emb[v][i] * x[i] (bf16 table, fp32 x, fp32 accumulate),
 * next = the first index of the maximum.  emb: device bf16 [vocab][dim];
 * x: device fp32 [dim]; logits: device fp32 [vocab] or NULL; next: device
 * int32 [1]; workspace: qlin_lm_head_workspace_size() bytes of device memory,
 * zero-filled before its first use (each call leaves it zero-filled again);
 * calls sharing a workspace must not overlap on the GPU. */
size_t qlin_lm_head_workspace_size(int vocab);
qlin_status qlin_lm_head_argmax(const uint16_t *emb, const float *x, int vocab, int dim, float *logits,
                                int32_t *next, void *workspace, size_t workspace_bytes, qlin_stream_t stream);

/* Sketch head: candidates first, exact scores for them only ([citric] "Step 3:
 * the output layer became the bottleneck").  For the final hidden state x:
 *   1. the k dims with the largest |x_d| (ties: lower d) are scored exactly,
 *      exact[v] = pairwise fp32 sum over them, ascending d, of bf16(E[v][d])*x_d;
 *   2. the other dims are scored from the sign bits of the table, one 64-bit
 *      XOR and bit count per block of 64 dims: block b holds positions
 *      64b .. 64b+63 of the size order perm (fixed at preparation) minus the
 *      exact dims; n_b = its sketched dims, m_b[v] = how many of their sign
 *      bits differ between E[v] and x, w_b = (pairwise fp32 sum of |x| over
 *      the block's 64 positions, exact dims and positions past dim counting
 *      +0) / n_b * c_E; sketch[v] = sum over b in order (each product rounded)
 *      of w_b * (n_b - 2 m_b[v]); approx[v] = exact[v] + sketch[v];
 *   3. the n_cand words with the largest approx (ties: lower index) are the
 *      candidates, in ascending order in cand[]; cand_logits[i] = their exact
 *      logits with the lm_head's arithmetic (qlin_lm_head_argmax); every other
 *      word scores minus infinity; *next = the first maximum among them.
 * qlin_sketch_prepare makes, once per table (device memory, caller-owned):
 *   perm   int32 [dim]: the dims by size, largest |dim_scale[d]| first, ties
 *          to the lower index (dim_scale: device fp32 [dim], finite, or NULL
 *          for the identity order; the final norm gain of a decoder);
 *   emb_t  bf16 [dim][qlin_sketch_emb_t_pitch(vocab)]: the table by dimension,
 *          zeros past vocab;
 *   signs  qlin_sketch_signs_bytes(vocab, dim) bytes: uint64
 *          [ceil(dim/64)][qlin_sketch_emb_t_pitch(vocab)], bit p of [b][v] =
 *          sign bit of E[v][perm[64b + p]], zero past dim or vocab;
 *   c_e    device float: the mean |E| over the table (fp64 sum, rounded once).
 * qlin_sketch_prepare uses a static device buffer for the c_E partial sums:
 * calls must not overlap.  Limits: 8 <= dim <= 2048, dim % 8 == 0, 0 <= k <=
 * min(32, dim), 1 <= n_cand <= vocab; emb, emb_t, signs, x and workspace
 * 16-byte aligned.  approx (device fp32 [vocab]) may be NULL.  x must be
 * finite.  The workspace (qlin_sketch_workspace_size bytes) must be
 * zero-filled before its first use; calls leave it ready for the next; calls
 * sharing it must not overlap.  The kernel is one cooperative launch whose
 * grid barriers wait at most 2 s; qlin_sketch_head_status() (which
 * synchronises `stream`) returns QLIN_ERR_TIMEOUT if one gave up, after which
 * the workspace must be zero-filled again. */
int64_t qlin_sketch_emb_t_pitch(int vocab);
size_t qlin_sketch_signs_bytes(int vocab, int dim);
qlin_status qlin_sketch_prepare(const uint16_t *emb, int vocab, int dim, const float *dim_scale, uint16_t *emb_t,
                                uint64_t *signs, int32_t *perm, float *c_e, qlin_stream_t stream);
size_t qlin_sketch_workspace_size(int vocab);
qlin_status qlin_sketch_head(const uint16_t *emb, const uint16_t *emb_t, const uint64_t *signs, const int32_t *perm,
                             const float *c_e, int vocab, int dim, const float *x, int k, int n_cand, float *approx,
                             int32_t *cand, float *cand_logits, int32_t *next, void *workspace,
                             size_t workspace_bytes, qlin_stream_t stream);
qlin_status qlin_sketch_head_status(void *workspace, qlin_stream_t stream);

/* S16 for many lanes ([citric] "Many users at once"): the output layer and
 * greedy pick of n_lanes hidden states in one pass over the bf16 table.
 * logits[u][r] = sum_i emb[r][i] * x[u][i], next[u] = the first index of the
 * maximum.  On the tensor cores: x enters as three bf16 terms (hi, mid, lo;
 * x to 24 bits) against the bf16 table with fp32 accumulation, so the logits
 * are within fp32 rounding of the fp32 dot product but not in the order of
 * qlin_lm_head_argmax.  emb: device bf16 [vocab][dim], 16-byte aligned;
 * x: device fp32 [n_lanes][dim]; logits: device fp32 [n_lanes][vocab] or NULL;
 * next: device int32 [n_lanes].  dim % 8 == 0.  Workspace:
 * qlin_lm_head_lanes_workspace_size() bytes, zero-filled before its first
 * use; calls leave it ready; calls sharing it must not overlap.  Up to 64
 * lanes per pass over the table.  qlin_lm_head_lanes_status() (synchronises
 * `stream`) returns QLIN_ERR_TIMEOUT if a bounded device wait gave up. */
size_t qlin_lm_head_lanes_workspace_size(int vocab, int dim);
qlin_status qlin_lm_head_lanes(const uint16_t *emb, const float *x, int vocab, int dim, int n_lanes, float *logits,
                               int32_t *next, void *workspace, size_t workspace_bytes, qlin_stream_t stream);
qlin_status qlin_lm_head_lanes_status(void *workspace, qlin_stream_t stream);

/* ========================================================================
 * S8-S16 composed: one decode step of a ternary Gemma-style decoder
 * ([cpp20gemma] "Architecture & implementation": h += attn(rmsnorm(h));
 * h += mlp(rmsnorm(h)); logits = lm_head(rmsnorm(h)); layer order of
 * [llama2.c] "The forward pass"; every linear layer T158 on int8-quantised
 * inputs, [citric] "Step 2"; GeGLU MLP; bf16 embedding tied to the lm_head).
 * ====================================================================== */
#define T158_NMAT 7 /* per layer, in this order: wq wk wv wo wg wu wd */

typedef struct {
    int32_t n_layers, dim, n_heads, n_kv_heads, head_dim, ffn, vocab, max_pos;
    float eps;
    float reserved0;
    const uint8_t *w[T158_NMAT]; /* device, each [n_layers][rows][pitch[j]] packed by t158_pack */
    int64_t pitch[T158_NMAT];    /* multiples of 16, >= ceil(in/5) */
    const float *scales;         /* device fp32 [n_layers][7], one per matrix */
    const float *g_attn;         /* device fp32 [n_layers][dim] */
    const float *g_ffn;          /* device fp32 [n_layers][dim] */
    const float *g_final;        /* device fp32 [dim] */
    const uint16_t *emb;         /* device bf16 bits [vocab][dim], also the lm_head */
    const float *rope_cos;       /* device fp32 [max_pos][head_dim/2] from t158_rope_table */
    const float *rope_sin;
} t158_model;

/* Bytes of device scratch decode_step_t158 needs for this model.  The
 * workspace must be zero-filled before its first use; steps leave it ready
 * for the next one.  Steps sharing a workspace must not overlap on the GPU. */
qlin_status decode_step_t158_workspace_size(const t158_model *m, size_t *bytes);

/* One forward step at position pos (0 <= pos < max_pos) for the token in
 * device memory *token: writes rotated k and v of every layer at pos into
 * kv_cache (device fp32 [n_layers][2][max_pos][n_kv_heads*head_dim], k then
 * v), logits (device fp32 [vocab], or NULL) and the greedy next token to
 * device *next_token (which may be the same address as token, so steps
 * chain on the device).  Shapes supported: dim % 16 == 0, head_dim in
 * {16,...,256} a power of two, n_heads % n_kv_heads == 0.  The workspace
 * holds a status word: after the stream has finished the step,
 * decode_step_t158_status() returns QLIN_ERR_TIMEOUT if a bounded device wait
 * gave up and QLIN_ERR_INVALID_ARG if *token was out of range. */
qlin_status decode_step_t158(const t158_model *m, float *kv_cache, void *workspace, size_t workspace_bytes,
                             const int32_t *token, int32_t pos, float *logits, int32_t *next_token,
                             qlin_stream_t stream);

/* Number of kernel launches one decode_step_t158 call makes for this model
 * (for launch accounting); -1 if the model is invalid. */
int decode_step_t158_launches(const t158_model *m);

/* Reads (synchronously, after synchronising `stream`) and clears the status
 * word of a decode workspace.  After QLIN_ERR_TIMEOUT the workspace must be
 * zero-filled again before the next step, and that step's KV rows at pos
 * rewritten (the step that gave up may have left them half written). */
qlin_status decode_step_t158_status(void *workspace, qlin_stream_t stream);

/* The longest a step's CTAs wait for one another or for a copy before they
 * give up and the status word reports QLIN_ERR_TIMEOUT (process-wide, for
 * steps launched afterwards; 0 restores the default of 2 s).  A correct step
 * waits microseconds; a limit below about 1 ms can make a slow but correct
 * step give up. */
void decode_step_t158_set_wait_limit(uint64_t ns);

/* Test hook (process-wide, for steps launched afterwards): layer >= 0 makes
 * the CTA that owns residual row 0 skip publishing its residual rows after
 * the attention block of that layer, so every CTA's wait for them runs out
 * and the step reports QLIN_ERR_TIMEOUT; -1 (the default) turns it off.  It
 * exists so a test can exercise the bounded waits without faulting the GPU. */
void decode_step_t158_test_withhold(int layer);

/* The decode step with the sketch head as its output layer ([citric] "Step 3:
 * the output layer became the bottleneck"): decode_step_t158 up to the final
 * norm, then qlin_sketch_head over the tied table (m->emb) picks the next
 * token.  Two launches per step.  The tables come from qlin_sketch_prepare on
 * m->emb, with the final norm gain m->g_final as the per-dimension size. */
typedef struct {
    const uint16_t *emb_t;  /* dimension-major copy of m->emb */
    const uint64_t *signs;  /* sign words */
    const int32_t *perm;    /* size order of the dims */
    const float *c_e;       /* device float: mean |E| */
    int k;                  /* exact dims, 0..32 */
    int n_cand;             /* candidates, 1..vocab */
} t158_sketch;

/* Bytes of device scratch for decode_step_t158_sketch: the decode workspace,
 * the final hidden state, the candidates and the sketch head's workspace.
 * Zero-filled before first use; steps leave it ready for the next one. */
qlin_status decode_step_t158_sketch_workspace_size(const t158_model *m, const t158_sketch *s, size_t *bytes);
qlin_status decode_step_t158_sketch(const t158_model *m, const t158_sketch *s, float *kv_cache, void *workspace,
                                    size_t workspace_bytes, const int32_t *token, int32_t pos, int32_t *next_token,
                                    qlin_stream_t stream);
/* Reads and clears both status words (synchronises `stream`). */
qlin_status decode_step_t158_sketch_status(const t158_model *m, const t158_sketch *s, void *workspace,
                                           qlin_stream_t stream);

/* A decode step over lanes ([citric] "Many users at once": every step is a
 * set of lanes, a lane being one token of one sequence at one position, so
 * batches of users and chunks of a prompt share one path and each weight byte
 * is read once for all lanes).  Lane i takes tokens[i] at positions[i] of
 * sequence seqs[i] (device int32 [n_lanes] each); sequence s owns the KV cache
 * kv_caches + s * n_layers * 2 * max_pos * n_kv_heads * head_dim (device fp32,
 * the layout of decode_step_t158).  Layer by layer every lane's k and v are
 * written before any lane attends: lanes of one sequence at distinct
 * positions form a prompt chunk, in any order.  Each lane's results are those
 * of decode_step_t158 for its token (k, v bit for bit; logits and the
 * greedy pick as qlin_lm_head_lanes gives them).
 * logits: device fp32 [n_lanes][vocab] or NULL; next: device int32 [n_lanes].
 * The workspace (decode_lanes_t158_workspace_size(m, max_lanes) bytes, the
 * same max_lanes passed to every call) must be zero-filled before its first
 * use; calls leave it ready for the next.  The call issues a
 * fixed sequence of kernels (decode_lanes_t158_launches) and no host
 * synchronisation, so it can be captured in a CUDA graph once the first call
 * has run outside capture.  decode_lanes_t158_status() (synchronises
 * `stream`) returns QLIN_ERR_INVALID_ARG if a lane's token, position or
 * sequence slot was out of range (such a lane writes nothing to any cache). */
qlin_status decode_lanes_t158_workspace_size(const t158_model *m, int max_lanes, size_t *bytes);
qlin_status decode_lanes_t158(const t158_model *m, float *kv_caches, int n_seqs, int n_lanes, const int32_t *tokens,
                              const int32_t *positions, const int32_t *seqs, float *logits, int32_t *next,
                              void *workspace, size_t workspace_bytes, int max_lanes, qlin_stream_t stream);
int decode_lanes_t158_launches(const t158_model *m, int n_lanes);
qlin_status decode_lanes_t158_status(void *workspace, qlin_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QLIN_H */
