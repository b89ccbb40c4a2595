// Decode-step kernels: embedding lookup, RMSNorm, RoPE table and KV append,
// split-position decode attention, GeGLU, lm_head + greedy argmax, and the
// composed ternary decode step.
//
// Sources: llama2.c "The forward pass -- one token, one position" (Steps 0-6)
// and "Sampling"; cpp20gemma README "Architecture & implementation"; gemma.cpp
// tour "The Forward Pass, Layer by Layer"; "Gemma 3 1B at 114 tokens per
// second on a laptop CPU", "Step 2".
#include <algorithm>
#include <vector>

#include "decode_fused.cuh"

namespace qlin {

// ---------------------------------------------------------------- S8
__global__ void embed_kernel(const uint16_t *__restrict__ emb, int vocab, int dim, const int32_t *__restrict__ token,
                             float *__restrict__ h, int32_t *status) {
    const int tok = *token;
    const bool ok = tok >= 0 && tok < vocab;
    for (int i = threadIdx.x; i < dim; i += blockDim.x)
        h[i] = ok ? __uint_as_float((uint32_t)emb[(int64_t)tok * dim + i] << 16) : 0.0f;
    if (!ok && threadIdx.x == 0 && status) atomicOr(status, 1);
}

// ---------------------------------------------------------------- S9
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *x, const float *__restrict__ g, float *out, int n,
                                                      float eps) {
    extern __shared__ float buf[];
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    rmsnorm_row(x + row * n, g, out + row * n, n, eps, buf, red, whole_block());
}

// ---------------------------------------------------------------- S11
__global__ void rope_table_kernel(float *cos_t, float *sin_t, int max_pos, int head_dim, double base) {
    const int half = head_dim / 2;
    const int64_t total = (int64_t)max_pos * half;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(idx / half), i = (int)(idx % half);
        const double theta = pow(base, -(double)(2 * i) / (double)head_dim);
        const double ang = (double)p * theta;
        cos_t[idx] = (float)cos(ang);
        sin_t[idx] = (float)sin(ang);
    }
}

__global__ void rope_kv_kernel(float *q, const float *k, const float *v, float *kc, float *vc,
                               const float *__restrict__ cos_t, const float *__restrict__ sin_t, int pos, int nh,
                               int nkv, int hd) {
    extern __shared__ float kr[];  // [nkv*hd]
    const int half = hd / 2;
    const float *c = cos_t + (int64_t)pos * half;
    const float *s = sin_t + (int64_t)pos * half;
    rope_rotate(q, nh, hd, c, s, whole_block());
    for (int i = threadIdx.x; i < nkv * hd; i += blockDim.x) kr[i] = k[i];
    __syncthreads();
    rope_rotate(kr, nkv, hd, c, s, whole_block());
    __syncthreads();
    const int64_t off = (int64_t)pos * nkv * hd;
    for (int i = threadIdx.x; i < nkv * hd; i += blockDim.x) {
        kc[off + i] = kr[i];
        vc[off + i] = v[i];
    }
}

// ---------------------------------------------------------------- S12
struct AttnWs {
    float *m, *S, *U;  // [nh][ncmax], [nh][ncmax], [nh][ncmax][hd]
};

__host__ __device__ inline int att_chunks(int max_pos) { return (max_pos + 31) / 32; }

__host__ __device__ inline size_t attn_ws_floats(int max_pos, int nh, int hd) {
    const size_t nc = (size_t)att_chunks(max_pos);
    return (size_t)nh * nc * (2 + (size_t)hd);
}

__device__ __forceinline__ AttnWs attn_ws(float *base, int ncmax, int nh, int hd) {
    AttnWs w;
    w.m = base;
    w.S = base + (size_t)nh * ncmax;
    w.U = base + (size_t)2 * nh * ncmax;
    return w;
}

// grid (nchunks, nh): chunk c of head h
__global__ void __launch_bounds__(256) attn_chunk_kernel(const float *__restrict__ q, const float *__restrict__ kc,
                                                         const float *__restrict__ vc, int pos, int nh, int nkv, int hd,
                                                         float *ws, int ncmax) {
    __shared__ float qs[256];
    __shared__ float sc[32];
    const int c = blockIdx.x, h = blockIdx.y;
    const int kvh = h / (nh / nkv);
    for (int i = threadIdx.x; i < hd; i += blockDim.x) qs[i] = q[h * hd + i];
    __syncthreads();
    const int t0 = c * 32;
    const int nt = min(32, pos + 1 - t0);
    const int ld = nkv * hd;
    AttnWs w = attn_ws(ws, ncmax, nh, hd);
    attention_chunk(qs, kc + (int64_t)t0 * ld + kvh * hd, vc + (int64_t)t0 * ld + kvh * hd, ld, nt, hd,
                    w.m + h * ncmax + c, w.S + h * ncmax + c, w.U + ((int64_t)h * ncmax + c) * hd, sc, whole_block());
}

__global__ void __launch_bounds__(256) attn_merge_kernel(const float *ws, int ncmax, int nc, int nh, int hd, float *out) {
    extern __shared__ float wbuf[];
    __shared__ float red[32];
    const int h = blockIdx.x;
    AttnWs w = attn_ws(const_cast<float *>(ws), ncmax, nh, hd);
    attention_merge(w.m + h * ncmax, w.S + h * ncmax, w.U + (int64_t)h * ncmax * hd, nc, hd, out + h * hd, wbuf, red,
                    whole_block());
}

// ---------------------------------------------------------------- S14 / residual
__global__ void geglu_kernel(const float *g, const float *u, float *a, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        a[i] = __fmul_rn(gelu32(g[i]), u[i]);
}

__global__ void add_kernel(float *h, const float *y, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) h[i] = __fadd_rn(h[i], y[i]);
}

// ---------------------------------------------------------------- S16
// lm_head: logits[r] = emb[r] . x for every row of the bf16 table, and the
// greedy token.  One persistent CTA per SM owns a contiguous slice of rows
// and streams it through a ring of shared-memory tiles with TMA bulk copies
// (warp 0, lane 0 is the producer); eight consumer warps take two rows of a
// tile each (16 lanes per row, 16-byte chunks) against x in shared memory.
// Each CTA leaves its best (value, index) in part[]; the last CTA to finish
// (atomic ticket) reduces them and resets the ticket.  Ties go to the lower
// index, so the result does not depend on the schedule.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

constexpr int kLmStages = 4;
constexpr int kLmConsumers = 8;

struct LmWs {
    float2 *part;
    unsigned *ticket;
    int32_t *status;
};

__host__ __device__ inline int lm_tile_rows(int dim) {
    int r = 40960 / (2 * dim);
    r = r > 16 ? 16 : r;
    return r < 1 ? 1 : r;
}

__global__ void __launch_bounds__(288, 1) lm_head_kernel(const uint16_t *__restrict__ emb, const float *__restrict__ x,
                                                         int vocab, int dim, float *__restrict__ logits, LmWs ws,
                                                         int32_t *__restrict__ next) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int TR = lm_tile_rows(dim);
    const int tile_bytes = TR * dim * 2;
    uint8_t *slots = smem;
    float4 *xs4 = reinterpret_cast<float4 *>(smem + (size_t)kLmStages * tile_bytes);
    Ring<kLmStages> *ring = reinterpret_cast<Ring<kLmStages> *>(smem + (size_t)kLmStages * tile_bytes + (size_t)dim * 4);
    __shared__ float bv_s[kLmConsumers];
    __shared__ int bi_s[kLmConsumers];
    __shared__ int last_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)vocab * blockIdx.x / gridDim.x;
    const int64_t r1 = (int64_t)vocab * (blockIdx.x + 1) / gridDim.x;
    const int ntiles = (int)((r1 - r0 + TR - 1) / TR);
    if (threadIdx.x == 0) ring->init(kLmConsumers);
    // x as two float4 planes: xs4[c] = x[8c..8c+3], xs4[C + c] = x[8c+4..8c+7]
    const int C = dim / 8;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        xs4[c] = make_float4(x[8 * c], x[8 * c + 1], x[8 * c + 2], x[8 * c + 3]);
        xs4[C + c] = make_float4(x[8 * c + 4], x[8 * c + 5], x[8 * c + 6], x[8 * c + 7]);
    }
    __syncthreads();

    float best_v = -__int_as_float(0x7f800000);
    int best_i = 0x7fffffff;
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first();
            int t = 0;
            for (; t < ntiles; t++) {
                const int s = t % kLmStages;
                if (t >= kLmStages && !mbar_wait(&ring->empty[s], ((t / kLmStages) - 1) & 1)) {
                    raise_status(ws.status, kStatusTimeout);
                    break;
                }
                const int64_t row = r0 + (int64_t)t * TR;
                const int rows = (int)min((int64_t)TR, r1 - row);
                const uint32_t bytes = (uint32_t)rows * dim * 2;
                mbar_arrive_expect_tx(&ring->full[s], bytes);
                bulk_g2s(slots + (size_t)s * tile_bytes, emb + row * dim, bytes, &ring->full[s], pol);
            }
            // drain: every copy issued must have landed before the CTA leaves
            for (int u = max(0, t - kLmStages); u < t; u++)
                if (!mbar_wait(&ring->full[u % kLmStages], (u / kLmStages) & 1)) raise_status(ws.status, kStatusTimeout);
        }
    } else {
        const int cw = warp - 1, sub = lane & 15, rsub = lane >> 4;
        const int rit = 2 * cw + rsub;  // row within a tile
        for (int t = 0; t < ntiles; t++) {
            const int s = t % kLmStages;
            if (!mbar_wait(&ring->full[s], (t / kLmStages) & 1)) {
                raise_status(ws.status, kStatusTimeout);
                break;
            }
            const int64_t row = r0 + (int64_t)t * TR + rit;
            const bool valid = rit < TR && row < r1;
            float acc = 0.0f;
            if (valid) {
                const uint8_t *wrow = slots + (size_t)s * tile_bytes + (size_t)rit * dim * 2;
#pragma unroll 4
                for (int c = sub; c < C; c += 16) {
                    const uint4 w = lds128(wrow + (size_t)c * 16);
                    const float4 xa = xs4[c], xb = xs4[C + c];
                    acc = fmaf(__uint_as_float(w.x << 16), xa.x, acc);
                    acc = fmaf(__uint_as_float(w.x & 0xffff0000u), xa.y, acc);
                    acc = fmaf(__uint_as_float(w.y << 16), xa.z, acc);
                    acc = fmaf(__uint_as_float(w.y & 0xffff0000u), xa.w, acc);
                    acc = fmaf(__uint_as_float(w.z << 16), xb.x, acc);
                    acc = fmaf(__uint_as_float(w.z & 0xffff0000u), xb.y, acc);
                    acc = fmaf(__uint_as_float(w.w << 16), xb.z, acc);
                    acc = fmaf(__uint_as_float(w.w & 0xffff0000u), xb.w, acc);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring->empty[s]);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (sub == 0 && valid) {
                if (logits) logits[row] = acc;
                if (better(acc, (int)row, best_v, best_i)) {
                    best_v = acc;
                    best_i = (int)row;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best_v, off);
            const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
            if (better(ov, oi, best_v, best_i)) {
                best_v = ov;
                best_i = oi;
            }
        }
        if (lane == 0) {
            bv_s[cw] = best_v;
            bi_s[cw] = best_i;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float v = bv_s[0];
        int i = bi_s[0];
        for (int w = 1; w < kLmConsumers; w++)
            if (better(bv_s[w], bi_s[w], v, i)) {
                v = bv_s[w];
                i = bi_s[w];
            }
        ws.part[blockIdx.x] = make_float2(v, __int_as_float(i));
        __threadfence();
        last_s = (atomicAdd(ws.ticket, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!last_s) return;
    // the last CTA: reduce every CTA's candidate
    __threadfence();
    float v = -__int_as_float(0x7f800000);
    int i = 0x7fffffff;
    for (int j = threadIdx.x; j < (int)gridDim.x; j += blockDim.x) {
        const float2 p = __ldcg(&ws.part[j]);
        if (better(p.x, __float_as_int(p.y), v, i)) {
            v = p.x;
            i = __float_as_int(p.y);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
    __shared__ float fv[9];
    __shared__ int fi[9];
    if (lane == 0) {
        fv[warp] = v;
        fi[warp] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); w++)
            if (better(fv[w], fi[w], v, i)) {
                v = fv[w];
                i = fi[w];
            }
        *next = i;
        *ws.ticket = 0u;
    }
}

static int lm_head_blocks() { return sm_count(); }

static size_t lm_ws_bytes() { return 256 + sizeof(float2) * (size_t)lm_head_blocks(); }

static LmWs lm_ws(void *base, int32_t *status) {
    LmWs w;
    w.ticket = reinterpret_cast<unsigned *>(base);
    w.part = reinterpret_cast<float2 *>(reinterpret_cast<char *>(base) + 256);
    w.status = status;
    return w;
}

// ---------------------------------------------------------------- host wrappers
static qlin_status launch_rmsnorm(const float *x, const float *g, float *out, int M, int n, float eps, cudaStream_t st) {
    const size_t smem = (size_t)next_pow2(n) * sizeof(float);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "rmsnorm: n=%d too large", n);
    if (smem > 48 * 1024) blocks_per_sm((const void *)rmsnorm_kernel, smem);
    rmsnorm_kernel<<<M, 256, smem, st>>>(x, g, out, n, eps);
    QLIN_LAUNCHED("rmsnorm_kernel");
    return QLIN_OK;
}

qlin_status launch_attention(const float *q, const float *kc, const float *vc, int pos, int nh, int nkv, int hd,
                             float *out, float *ws, int ncmax, cudaStream_t st) {
    const int nc = pos / 32 + 1;
    attn_chunk_kernel<<<dim3(nc, nh), 256, 0, st>>>(q, kc, vc, pos, nh, nkv, hd, ws, ncmax);
    QLIN_LAUNCHED("attn_chunk_kernel");
    const size_t smem = (size_t)next_pow2(nc) * sizeof(float);
    attn_merge_kernel<<<nh, 256, smem, st>>>(ws, ncmax, nc, nh, hd, out);
    QLIN_LAUNCHED("attn_merge_kernel");
    return QLIN_OK;
}

static qlin_status launch_lm_head(const uint16_t *emb, const float *x, int vocab, int dim, float *logits, int32_t *next,
                                  void *ws, int32_t *status, cudaStream_t st) {
    const size_t smem = (size_t)kLmStages * lm_tile_rows(dim) * dim * 2 + (size_t)dim * 4 + sizeof(Ring<kLmStages>);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "lm_head: dim %d too large", dim);
    blocks_per_sm((const void *)lm_head_kernel, smem);  // raises the dynamic shared-memory limit once
    lm_head_kernel<<<lm_head_blocks(), 288, smem, st>>>(emb, x, vocab, dim, logits, lm_ws(ws, status), next);
    QLIN_LAUNCHED("lm_head_kernel");
    return QLIN_OK;
}

// ---------------------------------------------------------------- composed decode step
// The step runs as one persistent kernel (decode_fused.cu).
qlin_status launch_decode_fused(const FusedArgs &args, cudaStream_t st);
size_t fused_smem_bytes(const t158_model *m, int G);
int fused_lpt(const t158_model &m, int G);

static size_t align256(size_t b) { return (b + 255) / 256 * 256; }

struct DecodeWs {
    int32_t *status;
    unsigned *seq;
    unsigned *lm_ticket;
    float2 *lm_part;
    uint64_t *hT, *qkvT, *attT, *aT, *pmT, *pST, *pUT, *amaxT, *hAcc;
    int ncmax;
    size_t bytes;
};

// Host-side settings of the fused step (process-wide): the longest wait on
// another CTA or on a copy, and the test hook that withholds one CTA's words.
static uint64_t g_decode_wait_ns = 0;  // 0: the 2 s default
static int g_decode_withhold = -1;

// Workspace layout; every word is zero in a fresh (zero-filled) workspace,
// and a zero tagged word never matches the tag of any phase.
static DecodeWs carve(const t158_model *m, char *base) {
    DecodeWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    const int d = m->dim, qd = m->n_heads * m->head_dim, kvd = m->n_kv_heads * m->head_dim, f = m->ffn;
    w.ncmax = att_chunks(m->max_pos);
    w.status = (int32_t *)take(16);  // must stay first: decode_step_t158_status reads offset 0
    w.seq = (unsigned *)take(8);
    w.lm_ticket = (unsigned *)take(32);
    w.lm_part = (float2 *)take(sizeof(float2) * (size_t)sm_count());
    w.hT = (uint64_t *)take(8 * (size_t)d);
    w.qkvT = (uint64_t *)take(8 * (size_t)(qd + 2 * kvd));
    w.attT = (uint64_t *)take(8 * (size_t)qd);
    w.aT = (uint64_t *)take(8 * (size_t)f);
    w.pmT = (uint64_t *)take(8 * (size_t)m->n_heads * w.ncmax);
    w.pST = (uint64_t *)take(8 * (size_t)m->n_heads * w.ncmax);
    w.pUT = (uint64_t *)take(8 * (size_t)m->n_heads * w.ncmax * m->head_dim);
    w.amaxT = (uint64_t *)take(8 * (size_t)sm_count());
    w.hAcc = (uint64_t *)take(8 * 2 * (size_t)m->n_layers * d);
    w.bytes = off;
    return w;
}

static qlin_status check_model(const t158_model *m) {
    QLIN_REQUIRE(m, QLIN_ERR_INVALID_ARG, "decode_step_t158: null model");
    QLIN_REQUIRE(m->n_layers >= 1 && m->dim >= 16 && m->dim % 16 == 0 && m->n_heads >= 1 && m->n_kv_heads >= 1 &&
                     m->n_heads % m->n_kv_heads == 0 && m->ffn >= 1 && m->vocab >= 1 && m->max_pos >= 1,
                 QLIN_ERR_INVALID_ARG, "decode_step_t158: bad model dimensions");
    QLIN_REQUIRE(m->head_dim >= 16 && m->head_dim <= 256 && (m->head_dim & (m->head_dim - 1)) == 0,
                 QLIN_ERR_UNSUPPORTED, "decode_step_t158: head_dim %d not a power of two in 16..256", m->head_dim);
    const int d = m->dim, qd = m->n_heads * m->head_dim, kvd = m->n_kv_heads * m->head_dim, f = m->ffn;
    const int ins[T158_NMAT] = {d, d, d, qd, d, d, f};
    for (int j = 0; j < T158_NMAT; j++) {
        QLIN_REQUIRE(m->w[j] && aligned16(m->w[j]), QLIN_ERR_INVALID_ARG, "decode_step_t158: weight %d null/misaligned", j);
        QLIN_REQUIRE(m->pitch[j] % 16 == 0 && m->pitch[j] >= (ins[j] + 4) / 5, QLIN_ERR_INVALID_ARG,
                     "decode_step_t158: pitch[%d]=%lld", j, (long long)m->pitch[j]);
        QLIN_REQUIRE(m->pitch[j] <= kItemMax, QLIN_ERR_UNSUPPORTED, "decode_step_t158: pitch[%d]=%lld above %d", j,
                     (long long)m->pitch[j], kItemMax);
    }
    QLIN_REQUIRE(m->pitch[4] == m->pitch[5], QLIN_ERR_UNSUPPORTED,
                 "decode_step_t158: gate and up rows must have the same pitch (%lld, %lld)", (long long)m->pitch[4],
                 (long long)m->pitch[5]);
    QLIN_REQUIRE(32 * kvd * 4 <= kItemMax && d * 2 <= kItemMax, QLIN_ERR_UNSUPPORTED,
                 "decode_step_t158: kv width %d or dim %d too large for the weight ring", kvd, d);
    {
        // the down projection's tile of one CTA: its output rows and input chunks
        const int G = sm_count(), KG = down_kgroups(G), NG = G / KG;
        const int rows = (d + NG - 1) / NG, chunks = ((int)(m->pitch[6] / 16) + KG - 1) / KG;
        QLIN_REQUIRE(rows <= kFMaxRows && rows * chunks * 16 <= kItemMax && 80 * chunks <= m->ffn + 80,
                     QLIN_ERR_UNSUPPORTED, "decode_step_t158: down projection tile %d x %d chunks too large", rows,
                     chunks);
    }
    QLIN_REQUIRE(m->max_pos <= 4096, QLIN_ERR_UNSUPPORTED, "decode_step_t158: max_pos %d above 4096", m->max_pos);
    QLIN_REQUIRE(m->ffn % 4 == 0, QLIN_ERR_UNSUPPORTED, "decode_step_t158: ffn %d not a multiple of 4", m->ffn);
    QLIN_REQUIRE(m->n_layers <= 127, QLIN_ERR_UNSUPPORTED, "decode_step_t158: %d layers above 127", m->n_layers);
    QLIN_REQUIRE(m->dim <= 4096, QLIN_ERR_UNSUPPORTED, "decode_step_t158: dim %d above 4096", m->dim);
    QLIN_REQUIRE(t158_pitch(m->dim) <= 4 * 32 * kFConsumerWarps, QLIN_ERR_UNSUPPORTED,
                 "decode_step_t158: dim %d needs more than four packed bytes per thread", m->dim);
    QLIN_REQUIRE(m->scales && m->g_attn && m->g_ffn && m->g_final && m->emb && m->rope_cos && m->rope_sin,
                 QLIN_ERR_INVALID_ARG, "decode_step_t158: null model tensor");
    QLIN_REQUIRE(aligned16(m->g_attn) && aligned16(m->g_ffn) && aligned16(m->g_final), QLIN_ERR_INVALID_ARG,
                 "decode_step_t158: norm gains not 16-byte aligned");
    QLIN_REQUIRE(fused_lpt(*m, sm_count()) > 0, QLIN_ERR_UNSUPPORTED, "decode_step_t158: model too wide");
    QLIN_REQUIRE(aligned16(m->emb), QLIN_ERR_INVALID_ARG, "decode_step_t158: emb not 16-byte aligned");
    return QLIN_OK;
}

}  // namespace qlin

extern "C" {

qlin_status qlin_embed_bf16(const uint16_t *emb, int vocab, int dim, const int32_t *token, float *h,
                            int32_t *status_word, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(emb && token && h, QLIN_ERR_INVALID_ARG, "qlin_embed_bf16: null pointer");
    QLIN_REQUIRE(vocab >= 1 && dim >= 1, QLIN_ERR_INVALID_ARG, "qlin_embed_bf16: vocab=%d dim=%d", vocab, dim);
    qlin::embed_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(emb, vocab, dim, token, h, status_word);
    QLIN_LAUNCHED("embed_kernel");
    return QLIN_OK;
}

qlin_status qlin_rmsnorm(const float *x, const float *gamma, float *out, int M, int n, float eps, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(x && gamma && out, QLIN_ERR_INVALID_ARG, "qlin_rmsnorm: null pointer");
    QLIN_REQUIRE(M >= 1 && n >= 1, QLIN_ERR_INVALID_ARG, "qlin_rmsnorm: M=%d n=%d", M, n);
    return qlin::launch_rmsnorm(x, gamma, out, M, n, eps, (cudaStream_t)stream);
}

qlin_status t158_rope_table(float *cos_t, float *sin_t, int max_pos, int head_dim, double base, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(cos_t && sin_t, QLIN_ERR_INVALID_ARG, "t158_rope_table: null pointer");
    QLIN_REQUIRE(max_pos >= 1 && head_dim >= 2 && head_dim % 2 == 0 && base > 0, QLIN_ERR_INVALID_ARG,
                 "t158_rope_table: max_pos=%d head_dim=%d", max_pos, head_dim);
    qlin::rope_table_kernel<<<qlin::sm_count() * 4, 256, 0, (cudaStream_t)stream>>>(cos_t, sin_t, max_pos, head_dim, base);
    QLIN_LAUNCHED("rope_table_kernel");
    return QLIN_OK;
}

qlin_status qlin_rope_kv_append(float *q, const float *k, const float *v, float *k_cache, float *v_cache,
                                const float *cos_t, const float *sin_t, int pos, int n_heads, int n_kv, int head_dim,
                                qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(q && k && v && k_cache && v_cache && cos_t && sin_t, QLIN_ERR_INVALID_ARG, "qlin_rope_kv_append: null");
    QLIN_REQUIRE(pos >= 0 && n_heads >= 1 && n_kv >= 1 && head_dim >= 2 && head_dim % 2 == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_rope_kv_append: pos=%d n_heads=%d n_kv=%d head_dim=%d", pos, n_heads, n_kv, head_dim);
    QLIN_REQUIRE((size_t)n_kv * head_dim * sizeof(float) <= 48 * 1024, QLIN_ERR_UNSUPPORTED, "qlin_rope_kv_append: kv too wide");
    qlin::rope_kv_kernel<<<1, 256, n_kv * head_dim * sizeof(float), (cudaStream_t)stream>>>(
        q, k, v, k_cache, v_cache, cos_t, sin_t, pos, n_heads, n_kv, head_dim);
    QLIN_LAUNCHED("rope_kv_kernel");
    return QLIN_OK;
}

size_t qlin_attention_workspace_size(int max_pos, int n_heads, int head_dim) {
    if (max_pos < 1 || n_heads < 1 || head_dim < 1) return 0;
    return qlin::attn_ws_floats(max_pos, n_heads, head_dim) * sizeof(float);
}

qlin_status qlin_attention_decode(const float *q, const float *k_cache, const float *v_cache, int pos, int n_heads,
                                  int n_kv, int head_dim, float *out, void *workspace, size_t workspace_bytes,
                                  qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(q && k_cache && v_cache && out && workspace, QLIN_ERR_INVALID_ARG, "qlin_attention_decode: null");
    QLIN_REQUIRE(pos >= 0 && n_heads >= 1 && n_kv >= 1 && n_heads % n_kv == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_attention_decode: pos=%d n_heads=%d n_kv=%d", pos, n_heads, n_kv);
    QLIN_REQUIRE(head_dim >= 16 && head_dim <= 256 && (head_dim & (head_dim - 1)) == 0, QLIN_ERR_UNSUPPORTED,
                 "qlin_attention_decode: head_dim %d", head_dim);
    QLIN_REQUIRE(pos < (1 << 20), QLIN_ERR_UNSUPPORTED, "qlin_attention_decode: pos %d", pos);
    const size_t need = qlin_attention_workspace_size(pos + 1, n_heads, head_dim);
    QLIN_REQUIRE(workspace_bytes >= need, QLIN_ERR_INVALID_ARG, "qlin_attention_decode: workspace %zu < %zu",
                 workspace_bytes, need);
    return qlin::launch_attention(q, k_cache, v_cache, pos, n_heads, n_kv, head_dim, out, (float *)workspace,
                                  qlin::att_chunks(pos + 1), (cudaStream_t)stream);
}

qlin_status qlin_geglu(const float *g, const float *u, float *a, int n, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(g && u && a && n >= 1, QLIN_ERR_INVALID_ARG, "qlin_geglu: bad arguments");
    qlin::geglu_kernel<<<qlin::ceil_div(n, 256), 256, 0, (cudaStream_t)stream>>>(g, u, a, n);
    QLIN_LAUNCHED("geglu_kernel");
    return QLIN_OK;
}

size_t qlin_lm_head_workspace_size(int vocab) {
    (void)vocab;
    return qlin::lm_ws_bytes();
}

qlin_status qlin_lm_head_argmax(const uint16_t *emb, const float *x, int vocab, int dim, float *logits, int32_t *next,
                                void *workspace, size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(emb && x && next && workspace, QLIN_ERR_INVALID_ARG, "qlin_lm_head_argmax: null pointer");
    QLIN_REQUIRE(vocab >= 1 && dim >= 8 && dim % 8 == 0, QLIN_ERR_INVALID_ARG, "qlin_lm_head_argmax: vocab=%d dim=%d",
                 vocab, dim);
    QLIN_REQUIRE(qlin::aligned16(emb) && qlin::aligned16(x), QLIN_ERR_INVALID_ARG, "qlin_lm_head_argmax: misaligned");
    QLIN_REQUIRE(workspace_bytes >= qlin_lm_head_workspace_size(vocab), QLIN_ERR_INVALID_ARG,
                 "qlin_lm_head_argmax: workspace too small");
    return qlin::launch_lm_head(emb, x, vocab, dim, logits, next, workspace, nullptr, (cudaStream_t)stream);
}

qlin_status decode_step_t158_workspace_size(const t158_model *m, size_t *bytes) {
    qlin::clear_error();
    qlin_status s = qlin::check_model(m);
    if (s) return s;
    QLIN_REQUIRE(bytes, QLIN_ERR_INVALID_ARG, "decode_step_t158_workspace_size: null bytes");
    *bytes = qlin::carve(m, nullptr).bytes;
    return QLIN_OK;
}

qlin_status decode_step_t158(const t158_model *m, float *kv_cache, void *workspace, size_t workspace_bytes,
                             const int32_t *token, int32_t pos, float *logits, int32_t *next_token, qlin_stream_t stream) {
    qlin::clear_error();
    qlin_status s = qlin::check_model(m);
    if (s) return s;
    QLIN_REQUIRE(kv_cache && workspace && token && next_token, QLIN_ERR_INVALID_ARG, "decode_step_t158: null pointer");
    QLIN_REQUIRE(pos >= 0 && pos < m->max_pos, QLIN_ERR_INVALID_ARG, "decode_step_t158: pos %d outside [0, %d)", pos,
                 m->max_pos);
    QLIN_REQUIRE(qlin::aligned16(workspace) && qlin::aligned16(kv_cache), QLIN_ERR_INVALID_ARG,
                 "decode_step_t158: workspace or kv_cache not 16-byte aligned");
    const qlin::DecodeWs w = qlin::carve(m, (char *)workspace);
    QLIN_REQUIRE(workspace_bytes >= w.bytes, QLIN_ERR_INVALID_ARG, "decode_step_t158: workspace %zu < %zu bytes",
                 workspace_bytes, w.bytes);
    qlin::FusedArgs a{};
    a.m = *m;
    a.kv = kv_cache;
    a.token = token;
    a.pos = pos;
    a.logits = logits;
    a.next = next_token;
    a.hT = w.hT;
    a.qkvT = w.qkvT;
    a.attT = w.attT;
    a.aT = w.aT;
    a.pmT = w.pmT;
    a.pST = w.pST;
    a.pUT = w.pUT;
    a.amaxT = w.amaxT;
    a.hAcc = w.hAcc;
    a.ncmax = w.ncmax;
    a.lm_part = w.lm_part;
    a.lm_ticket = w.lm_ticket;
    a.seq = w.seq;
    a.status = w.status;
    a.wait_ns = qlin::g_decode_wait_ns;
    a.withhold = qlin::g_decode_withhold;
    return qlin::launch_decode_fused(a, (cudaStream_t)stream);
}

namespace {
struct SketchStepWs {
    float *final_x;
    int32_t *cand;
    float *cand_logits;
    char *sketch;
    size_t sketch_bytes, bytes;
};

SketchStepWs carve_sketch(const t158_model *m, const t158_sketch *s, char *base) {
    SketchStepWs w{};
    size_t off = qlin::align256(qlin::carve(m, nullptr).bytes);
    auto take = [&](size_t b) {
        char *p = base ? base + off : nullptr;
        off += qlin::align256(b);
        return p;
    };
    w.final_x = (float *)take(4 * (size_t)m->dim);
    w.cand = (int32_t *)take(4 * (size_t)s->n_cand);
    w.cand_logits = (float *)take(4 * (size_t)s->n_cand);
    w.sketch_bytes = qlin_sketch_workspace_size(m->vocab);
    w.sketch = take(w.sketch_bytes);
    w.bytes = off;
    return w;
}

qlin_status check_sketch(const t158_model *m, const t158_sketch *s) {
    QLIN_REQUIRE(s && s->emb_t && s->signs && s->perm && s->c_e, QLIN_ERR_INVALID_ARG,
                 "decode_step_t158_sketch: null sketch table");
    QLIN_REQUIRE(s->k >= 0 && s->k <= 32 && s->k <= m->dim && s->n_cand >= 1 && s->n_cand <= m->vocab,
                 QLIN_ERR_INVALID_ARG, "decode_step_t158_sketch: k = %d, n_cand = %d", s->k, s->n_cand);
    return QLIN_OK;
}
}  // namespace

qlin_status decode_step_t158_sketch_workspace_size(const t158_model *m, const t158_sketch *s, size_t *bytes) {
    qlin::clear_error();
    qlin_status st = qlin::check_model(m);
    if (st) return st;
    if ((st = check_sketch(m, s))) return st;
    QLIN_REQUIRE(bytes, QLIN_ERR_INVALID_ARG, "decode_step_t158_sketch_workspace_size: null bytes");
    *bytes = carve_sketch(m, s, nullptr).bytes;
    return QLIN_OK;
}

qlin_status decode_step_t158_sketch(const t158_model *m, const t158_sketch *s, float *kv_cache, void *workspace,
                                    size_t workspace_bytes, const int32_t *token, int32_t pos, int32_t *next_token,
                                    qlin_stream_t stream) {
    qlin::clear_error();
    qlin_status st = qlin::check_model(m);
    if (st) return st;
    if ((st = check_sketch(m, s))) return st;
    QLIN_REQUIRE(kv_cache && workspace && token && next_token, QLIN_ERR_INVALID_ARG,
                 "decode_step_t158_sketch: null pointer");
    QLIN_REQUIRE(pos >= 0 && pos < m->max_pos, QLIN_ERR_INVALID_ARG, "decode_step_t158_sketch: pos %d outside [0, %d)",
                 pos, m->max_pos);
    QLIN_REQUIRE(qlin::aligned16(workspace) && qlin::aligned16(kv_cache), QLIN_ERR_INVALID_ARG,
                 "decode_step_t158_sketch: workspace or kv_cache not 16-byte aligned");
    const SketchStepWs sw = carve_sketch(m, s, (char *)workspace);
    QLIN_REQUIRE(workspace_bytes >= sw.bytes, QLIN_ERR_INVALID_ARG,
                 "decode_step_t158_sketch: workspace %zu < %zu bytes", workspace_bytes, sw.bytes);
    const qlin::DecodeWs w = qlin::carve(m, (char *)workspace);
    qlin::FusedArgs a{};
    a.m = *m;
    a.kv = kv_cache;
    a.token = token;
    a.pos = pos;
    a.logits = nullptr;
    a.next = next_token;
    a.final_x = sw.final_x;
    a.hT = w.hT;
    a.qkvT = w.qkvT;
    a.attT = w.attT;
    a.aT = w.aT;
    a.pmT = w.pmT;
    a.pST = w.pST;
    a.pUT = w.pUT;
    a.amaxT = w.amaxT;
    a.hAcc = w.hAcc;
    a.ncmax = w.ncmax;
    a.lm_part = w.lm_part;
    a.lm_ticket = w.lm_ticket;
    a.seq = w.seq;
    a.status = w.status;
    a.wait_ns = qlin::g_decode_wait_ns;
    a.withhold = qlin::g_decode_withhold;
    if ((st = qlin::launch_decode_fused(a, (cudaStream_t)stream))) return st;
    return qlin_sketch_head(m->emb, s->emb_t, s->signs, s->perm, s->c_e, m->vocab, m->dim, sw.final_x, s->k, s->n_cand,
                            nullptr, sw.cand, sw.cand_logits, next_token, sw.sketch, sw.sketch_bytes, stream);
}

qlin_status decode_step_t158_sketch_status(const t158_model *m, const t158_sketch *s, void *workspace,
                                           qlin_stream_t stream) {
    qlin::clear_error();
    qlin_status st = qlin::check_model(m);
    if (st) return st;
    if ((st = check_sketch(m, s))) return st;
    QLIN_REQUIRE(workspace, QLIN_ERR_INVALID_ARG, "decode_step_t158_sketch_status: null workspace");
    if ((st = decode_step_t158_status(workspace, stream))) return st;
    return qlin_sketch_head_status(carve_sketch(m, s, (char *)workspace).sketch, stream);
}

int decode_step_t158_launches(const t158_model *m) {
    qlin::clear_error();
    if (qlin::check_model(m)) return -1;
    return 1;  // one persistent kernel per step
}

void decode_step_t158_set_wait_limit(uint64_t ns) { qlin::g_decode_wait_ns = ns; }

void decode_step_t158_test_withhold(int layer) { qlin::g_decode_withhold = layer; }

qlin_status decode_step_t158_status(void *workspace, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(workspace, QLIN_ERR_INVALID_ARG, "decode_step_t158_status: null workspace");
    int32_t st[4] = {0, 0, 0, 0};
    QLIN_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    QLIN_CUDA(cudaMemcpy(st, workspace, sizeof st, cudaMemcpyDeviceToHost));
    QLIN_CUDA(cudaMemset(workspace, 0, sizeof st));
    QLIN_REQUIRE(!(st[0] & 2), QLIN_ERR_TIMEOUT, "decode_step_t158: a device-side wait gave up");
    QLIN_REQUIRE(!(st[0] & 1), QLIN_ERR_INVALID_ARG, "decode_step_t158: token out of range");
    return QLIN_OK;
}

}  // extern "C"
