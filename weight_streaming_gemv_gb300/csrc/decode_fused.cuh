// Pieces of the fused decode step: the per-CTA schedule of weight slices
// (shared by the TMA producer and the consumer warps, so both walk the same
// items in the same order), quantise-into-planes, T158 rows from a shared
// memory slot, and the bounded grid barrier.
#pragma once

#include "decode_ops.cuh"
#include "stream.cuh"

namespace qlin {

constexpr int kFStages = 4;
constexpr int kFSlot = 36864;  // bytes per ring slot (16 bf16 rows of 1152)
constexpr int kFConsumerWarps = 7;  // + 1 producer warp = 8 warps: 2 per SM sub-partition, up to 255 registers
constexpr int kFThreads = 32 * (kFConsumerWarps + 1);

struct FusedArgs {
    t158_model m;
    float *kv;
    const int32_t *token;
    int pos;
    float *logits;
    int32_t *next;
    // workspace
    float *h, *q, *k, *v, *a, *att, *pm, *pS, *pU;
    int ncmax;
    float2 *lm_part;
    unsigned *lm_ticket;
    unsigned long long *bar_ctr;
    int32_t *status;
};

// rows [lo, hi) of n rows owned by CTA b of G
__device__ __forceinline__ void share(int n, int b, int G, int &lo, int &hi) {
    lo = (int)((int64_t)n * b / G);
    hi = (int)((int64_t)n * (b + 1) / G);
}

// A piece: up to slot-sized run of consecutive rows of one matrix.
struct Piece {
    const uint8_t *src;
    int rows, pitch, row0, mat;
};

// Calls f(piece) for every slot-sized piece of rows [lo, hi) of matrix `mat`.
template <class F>
__device__ __forceinline__ void pieces(const uint8_t *base, int64_t pitch, int lo, int hi, int mat, F &&f,
                                       int max_rows = 1 << 30) {
    int per = (int)(kFSlot / pitch) > 0 ? (int)(kFSlot / pitch) : 1;
    per = per < max_rows ? per : max_rows;
    for (int r = lo; r < hi; r += per) {
        Piece p;
        p.rows = min(per, hi - r);
        p.pitch = (int)pitch;
        p.row0 = r;
        p.mat = mat;
        p.src = base + (int64_t)r * pitch;
        f(p);
    }
}

// The items of layer l for CTA b, in consumption order.  QKV rows are the
// concatenation q | k | v; Wo and down share the residual rows this CTA owns;
// gate and up share the GeGLU rows; attention item e = chunk * n_heads + head
// (chunk = 32 positions) belongs to CTA e mod G and needs the cached rows of
// its chunk below `pos`, K then V.
template <class F>
__device__ __forceinline__ void layer_items(const FusedArgs &A, int l, int b, int G, F &&f) {
    const t158_model &m = A.m;
    const int d = m.dim, qd = m.n_heads * m.head_dim, kvd = m.n_kv_heads * m.head_dim, ff = m.ffn;
    const int rows[T158_NMAT] = {qd, kvd, kvd, d, ff, ff, d};
    // Q K V
    int lo, hi;
    share(qd + 2 * kvd, b, G, lo, hi);
    int base = 0;
#pragma unroll
    for (int j = 0; j < 3; j++) {
        const int a0 = max(lo, base), a1 = min(hi, base + rows[j]);
        if (a1 > a0)
            pieces(m.w[j] + (int64_t)l * rows[j] * m.pitch[j], m.pitch[j], a0 - base, a1 - base, j, f);
        base += rows[j];
    }
    // attention K/V prefetch (rows strictly below pos) for this CTA's (chunk, head) items
    const int nc = A.pos / 32 + 1;
    const float *kc = A.kv + (int64_t)(2 * l) * m.max_pos * kvd;
    const float *vc = A.kv + (int64_t)(2 * l + 1) * m.max_pos * kvd;
    for (int e = b; e < nc * m.n_heads; e += G) {
        const int c = e / m.n_heads;
        const int t0 = 32 * c, npre = min(t0 + 32, A.pos) - t0;
        if (npre > 0) {
            Piece p;
            p.rows = npre;
            p.pitch = kvd * 4;
            p.row0 = t0;
            p.mat = 7;
            p.src = reinterpret_cast<const uint8_t *>(kc + (int64_t)t0 * kvd);
            f(p);
            p.mat = 8;
            p.src = reinterpret_cast<const uint8_t *>(vc + (int64_t)t0 * kvd);
            f(p);
        }
    }
    share(d, b, G, lo, hi);
    pieces(m.w[3] + (int64_t)l * rows[3] * m.pitch[3], m.pitch[3], lo, hi, 3, f);
    int g0, g1;
    share(ff, b, G, g0, g1);
    pieces(m.w[4] + (int64_t)l * rows[4] * m.pitch[4], m.pitch[4], g0, g1, 4, f);
    pieces(m.w[5] + (int64_t)l * rows[5] * m.pitch[5], m.pitch[5], g0, g1, 5, f);
    pieces(m.w[6] + (int64_t)l * rows[6] * m.pitch[6], m.pitch[6], lo, hi, 6, f);
}

// lm_head tiles of CTA b
template <class F>
__device__ __forceinline__ void lm_items(const FusedArgs &A, int b, int G, F &&f) {
    const int dim = A.m.dim;
    int lo, hi;
    share(A.m.vocab, b, G, lo, hi);
    // two rows per consumer warp per tile: every warp does one pass
    pieces(reinterpret_cast<const uint8_t *>(A.m.emb), (int64_t)dim * 2, lo, hi, 9, f, 2 * kFConsumerWarps);
}

// ---------------------------------------------------------------- quantise into digit-plane order
// Absmax step of v[0..K) by the group.
__device__ __forceinline__ float group_absmax(const float *v, int K, float *red, Grp g) {
    float a = 0.0f;
    for (int i = g.tid; i < K; i += g.n) a = fmaxf(a, fabsf(v[i]));
    a = warp_max(a);
    if (g.lane() == 0) red[g.warp()] = a;
    g.sync();
    float m = red[0];
    for (int w = 1; w < (g.n >> 5); w++) m = fmaxf(m, red[w]);
    g.sync();
    return m;
}

// int8 codes of v/scale placed in the plane order of the T158 kernels
// (xr[c*5+i] word w byte b = code of element 5*(16c+4w+b)+i, 0 past K);
// returns the exact sum of the codes.  One thread per packed byte j (five
// consecutive elements); the four bytes of a word come from four consecutive
// lanes and are joined with shuffles.  The group size must be a multiple of 4.
__device__ __forceinline__ int quant_planes(const float *v, int K, float scale, int C, uint4 *xr, int *ired, Grp g) {
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const int nbytes = C * 16;
    int s = 0;
    const int lane = g.lane();
    for (int j0 = 0; j0 < nbytes; j0 += g.n) {
        const int j = j0 + g.tid;  // lanes of a warp take consecutive bytes
        uint32_t code[5];
#pragma unroll
        for (int i = 0; i < 5; i++) {
            const int k = 5 * j + i;
            const int q = (j < nbytes && k < K) ? quant_code(v[k], scale) : 0;
            s += q;
            code[i] = (uint32_t)(q & 0xff);
        }
        // word of plane i for bytes 4(j/4) .. 4(j/4)+3: gather from the four lanes
#pragma unroll
        for (int i = 0; i < 5; i++) {
            uint32_t w = code[i] << (8 * (lane & 3));
            w |= __shfl_xor_sync(0xffffffffu, w, 1);
            w |= __shfl_xor_sync(0xffffffffu, w, 2);
            if ((lane & 3) == 0 && j < nbytes) {
                const int c = j >> 4, wd = (j >> 2) & 3;
                xw[c * 20 + i * 4 + wd] = w;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (g.lane() == 0) ired[g.warp()] = s;
    g.sync();
    int t = 0;
    for (int w = 0; w < (g.n >> 5); w++) t += ired[w];
    g.sync();
    return t;
}

// Codes of v (shared memory, K elements) for step `scale` into the plane
// layout, one packed byte per thread (as quant_planes), with the sum of the
// codes accumulated into *isum (shared memory, zeroed by the caller before the
// last group barrier).  No group barrier inside: the caller syncs once after.
__device__ __forceinline__ void planes_from_smem(const float *v, int K, float scale, int C, uint4 *xr, int *isum,
                                                 Grp g) {
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const int nbytes = C * 16;
    const int lane = g.lane();
    int s = 0;
    for (int j0 = 0; j0 < nbytes; j0 += g.n) {
        const int j = j0 + g.tid;
        uint32_t code[5];
#pragma unroll
        for (int i = 0; i < 5; i++) {
            const int k = 5 * j + i;
            const int q = (j < nbytes && k < K) ? quant_code(v[k], scale) : 0;
            s += q;
            code[i] = (uint32_t)(q & 0xff);
        }
#pragma unroll
        for (int i = 0; i < 5; i++) {
            uint32_t w = code[i] << (8 * (lane & 3));
            w |= __shfl_xor_sync(0xffffffffu, w, 1);
            w |= __shfl_xor_sync(0xffffffffu, w, 2);
            if ((lane & 3) == 0 && j < nbytes) xw[(j >> 4) * 20 + i * 4 + ((j >> 2) & 3)] = w;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) atomicAdd(isum, s);
}

// RMSNorm + absmax quantisation of a d-vector (d <= 4096, d % 4 == 0) into
// the planes, with three group barriers.  load4(u) gives elements 4u..4u+3
// (from L2 or shared memory).  The first T threads (T = the largest power of
// two not above the group) load the S = next_pow2(d)/T consecutive leaves of
// their segment of the pairwise tree (S <= 32, in float4 units when S >= 4),
// square and sum them as a balanced tree, then lanes, then warps; every
// thread then finishes the tree itself from the warp sums.  Each thread
// normalises the five elements of its own packed byte(s), takes the absmax
// over the group and writes its codes into the planes.  gam and the staged x
// (xs) are in natural order in shared memory; xn receives the normalised
// vector.  Returns the step; *sumx gets the sum of the codes.  The arithmetic
// is that of rmsnorm_row and the absmax quantiser.
template <class Load4>
__device__ __forceinline__ float norm_quant(Load4 load4, const float *gam, int d, float eps, float *xs, float *xn,
                                            uint4 *xr, int C, float *red, int *isum, int *sumx, Grp g) {
    int T = 32;
    while (2 * T <= g.n) T *= 2;
    const int P = next_pow2(d);
    const int S = P >= T ? P / T : 1;
    const int t = g.tid;
    float part = 0.0f;
    if (t < T) {
        float v[32];
        if (S >= 4) {
            float4 w[8];
#pragma unroll
            for (int j = 0; j < 8; j++) w[j] = load4(min(t * S / 4 + j, d / 4 - 1));  // clamped: all in flight
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const bool ok = 4 * j < S && t * S + 4 * j < d;
                v[4 * j] = ok ? w[j].x : 0.0f;
                v[4 * j + 1] = ok ? w[j].y : 0.0f;
                v[4 * j + 2] = ok ? w[j].z : 0.0f;
                v[4 * j + 3] = ok ? w[j].w : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (4 * j < S && t * S + 4 * j < d)
                    reinterpret_cast<float4 *>(xs)[t * S / 4 + j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                                                                v[4 * j + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] = 0.0f;
            for (int i = 0; i < S; i++) {
                const int e = t * S + i;
                if (e < d) {
                    const float4 q = load4(e / 4);
                    const int c = e % 4;
                    const float xe = c == 0 ? q.x : c == 1 ? q.y : c == 2 ? q.z : q.w;
                    xs[e] = xe;
                    if (i == 0) v[0] = xe; else if (i == 1) v[1] = xe; else v[2 + (i & 1)] = xe;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = __fmul_rn(v[i], v[i]);
#pragma unroll
        for (int st = 1; st < 32; st <<= 1)
#pragma unroll
            for (int i = 0; i < 32; i += 2 * st)
                if (st < S) v[i] = __fadd_rn(v[i], v[i + st]);
        part = v[0];
    }
    part = warp_psum(part);
    if ((t & 31) == 0 && t < T) red[t >> 5] = part;
    g.sync();  // 1: warp sums and the staged vector are visible
    float ss;
    {
        const int W = T >> 5;  // a power of two <= 8
        float w8[8];
#pragma unroll
        for (int i = 0; i < 8; i++) w8[i] = i < W ? red[i] : 0.0f;
#pragma unroll
        for (int st = 1; st < 8; st <<= 1)
#pragma unroll
            for (int i = 0; i < 8; i += 2 * st)
                if (st < W) w8[i] = __fadd_rn(w8[i], w8[i + st]);
        ss = w8[0];
    }
    ss = __fdiv_rn(ss, (float)d);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    // normalised values of this thread's packed bytes j = t, t + n, ...
    const int nbytes = C * 16;
    constexpr int MAXB = 4;  // bytes per thread (nbytes <= 4 * group size)
    float o[MAXB][5];
    float amax = 0.0f;
#pragma unroll
    for (int bi = 0; bi < MAXB; bi++) {
        const int j = t + bi * g.n;
#pragma unroll
        for (int i = 0; i < 5; i++) {
            const int k = 5 * j + i;
            float val = 0.0f;
            if (j < nbytes && k < d) {
                val = __fmul_rn(gam[k], __fmul_rn(r, xs[k]));
                xn[k] = val;
                amax = fmaxf(amax, fabsf(val));
            }
            o[bi][i] = val;
        }
    }
    amax = warp_max(amax);
    if (g.lane() == 0) red[8 + g.warp()] = amax;
    if (t == 0) *isum = 0;
    g.sync();  // 2: absmax parts
    float m = red[8];
    for (int w = 1; w < (g.n >> 5); w++) m = fmaxf(m, red[8 + w]);
    const float scale = quant_scale(m);
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const int lane = g.lane();
    int sacc = 0;
#pragma unroll
    for (int bi = 0; bi < MAXB; bi++) {
        const int j0 = bi * g.n;
        if (j0 >= nbytes) break;  // uniform across the group
        const int j = t + j0;
        uint32_t code[5];
#pragma unroll
        for (int i = 0; i < 5; i++) {
            const int k = 5 * j + i;
            const int q = (j < nbytes && k < d) ? quant_code(o[bi][i], scale) : 0;
            sacc += q;
            code[i] = (uint32_t)(q & 0xff);
        }
#pragma unroll
        for (int i = 0; i < 5; i++) {
            uint32_t w = code[i] << (8 * (lane & 3));
            w |= __shfl_xor_sync(0xffffffffu, w, 1);
            w |= __shfl_xor_sync(0xffffffffu, w, 2);
            if ((lane & 3) == 0 && j < nbytes) xw[(j >> 4) * 20 + i * 4 + ((j >> 2) & 3)] = w;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, off);
    if (lane == 0) atomicAdd(isum, sacc);
    g.sync();  // 3: planes and the code sum
    *sumx = *isum;
    return scale;
}

// Absmax quantisation of a K-vector written by other CTAs (global, read
// through L2) into the planes, with two group barriers: the vector is staged
// in v (shared memory) while each thread tracks its maximum.
__device__ __forceinline__ float quant_from_l2(const float *src, int K, float *v, uint4 *xr, int C, float *red,
                                               int *isum, int *sumx, Grp g) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(v);
    float amax = 0.0f;
    const int n4 = K / 4;
    for (int i0 = 0; i0 < n4; i0 += 8 * g.n) {
        float4 t[8];
#pragma unroll
        for (int j = 0; j < 8; j++) t[j] = __ldcg(s4 + min(i0 + g.tid + j * g.n, n4 - 1));  // clamped: all in flight
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int i = i0 + g.tid + j * g.n;
            if (i < n4) {
                d4[i] = t[j];
                amax = fmaxf(fmaxf(fmaxf(amax, fabsf(t[j].x)), fmaxf(fabsf(t[j].y), fabsf(t[j].z))), fabsf(t[j].w));
            }
        }
    }
    amax = warp_max(amax);
    if (g.lane() == 0) red[g.warp()] = amax;
    if (g.tid == 0) *isum = 0;
    g.sync();
    float m = red[0];
    for (int w = 1; w < (g.n >> 5); w++) m = fmaxf(m, red[w]);
    const float scale = quant_scale(m);
    planes_from_smem(v, K, scale, C, xr, isum, g);
    g.sync();
    *sumx = *isum;
    return scale;
}

// RMSNorm of the d-vector x in global memory (written by other CTAs: read
// through L2) into xn (shared memory), also leaving x itself in xs_out
// (shared memory).  Same tree as rmsnorm_row: the first T threads (T = the
// largest power of two not above the group) hold the P/T consecutive squares
// of their segment in registers (P = next_pow2(d) <= 32 T), sum them as a
// balanced tree, then lanes, then warps.
__device__ __forceinline__ void rmsnorm_from_l2(const float *x, const float *gam, float *xs_out, float *xn, int d,
                                                float eps, float *red, Grp g) {
    int T = 32;
    while (2 * T <= g.n) T *= 2;
    const int P = next_pow2(d);
    const int S = P >= T ? P / T : 1;
    const int t = g.tid;
    float v[32];
    float part = 0.0f;
    if (t < T) {
#pragma unroll
        for (int i = 0; i < 32; i++) {
            const int k = t * S + i;
            v[i] = (i < S && k < d) ? __ldcg(x + k) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 32; i++)
            if (i < S && t * S + i < d) xs_out[t * S + i] = v[i];
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = __fmul_rn(v[i], v[i]);
#pragma unroll
        for (int st = 1; st < 32; st <<= 1)
#pragma unroll
            for (int i = 0; i < 32; i += 2 * st)
                if (st < S) v[i] = __fadd_rn(v[i], v[i + st]);
        part = (P >= T || t < P) ? v[0] : 0.0f;
    }
    part = warp_psum(part);
    if ((t & 31) == 0 && t < T) red[t >> 5] = part;
    g.sync();
    if (t == 0) {
        const int W = T >> 5;
        for (int st = 1; st < W; st <<= 1)
            for (int i = 0; i < W; i += 2 * st) red[i] = __fadd_rn(red[i], red[i + st]);
    }
    g.sync();
    float ss = red[0];
    ss = __fdiv_rn(ss, (float)d);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    for (int i = t; i < d; i += g.n) xn[i] = __fmul_rn(gam[i], __fmul_rn(r, xs_out[i]));
    g.sync();
}

// ---------------------------------------------------------------- T158 rows from a slot
// rows x pitch packed bytes at `slot` (shared memory) against the planes xr;
// f(row, acc) with the exact integer sum of d * x (digits 0..2) per row.
template <int LPR, class F>
__device__ __forceinline__ void slot_rows(const uint8_t *slot, int rows, int pitch, const uint4 *xr, Grp g, F &&f) {
    constexpr int RPS = 32 / LPR;
    const int lane = g.lane(), sub = lane % LPR, rsub = lane / LPR;
    const int C = pitch / 16;
    const int nw = g.n >> 5;
    for (int r0 = g.warp() * RPS; r0 < rows; r0 += nw * RPS) {
        const int row = r0 + rsub;
        int acc = 0;
        if (row < rows) {
            const uint8_t *wr = slot + (size_t)row * pitch;
            for (int c = sub; c < C; c += LPR) {
                const uint4 wv = lds128(wr + (size_t)c * 16);
                uint32_t D[4][5];
                t158_planes(wv.x, D[0]);
                t158_planes(wv.y, D[1]);
                t158_planes(wv.z, D[2]);
                t158_planes(wv.w, D[3]);
                const uint4 *X = xr + (size_t)c * 5;
#pragma unroll
                for (int i = 0; i < 5; i++) {
                    const uint4 xv = X[i];
                    acc = dp4a(D[0][i], xv.x, acc);
                    acc = dp4a(D[1][i], xv.y, acc);
                    acc = dp4a(D[2][i], xv.z, acc);
                    acc = dp4a(D[3][i], xv.w, acc);
                }
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (sub == 0 && row < rows) f(row, acc);
    }
}

template <class F>
__device__ __forceinline__ void slot_rows_any(const uint8_t *slot, int rows, int pitch, const uint4 *xr, Grp g, F &&f) {
    const int C = pitch / 16;
    if (C <= 8)
        slot_rows<8>(slot, rows, pitch, xr, g, f);
    else if (C <= 16)
        slot_rows<16>(slot, rows, pitch, xr, g, f);
    else
        slot_rows<32>(slot, rows, pitch, xr, g, f);
}

// ---------------------------------------------------------------- async copies of small constants
// n floats (n % 4 == 0, both pointers 16-byte aligned) global -> shared with
// cp.async; completes at cp_async_wait().
__device__ __forceinline__ void cp_async_f4(float *dst, const float *src, int n, Grp g) {
    for (int i = g.tid; i < n / 4; i += g.n)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst + 4 * i)), "l"(src + 4 * i)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait(Grp g) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    g.sync();
}

// ---------------------------------------------------------------- grid barrier
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// All CTAs of the (co-resident) grid meet here.  The counter only grows
// within a launch; barrier number k completes at k * gridDim.x arrivals.
// Bounded: on timeout the status word gets kStatusTimeout and *abort is set.
__device__ __forceinline__ bool grid_barrier(unsigned long long *ctr, unsigned long long target, int32_t *status,
                                             volatile int *abort, Grp g) {
    g.sync();  // the CTA's writes happen-before thread 0's release below (bar.sync is cumulative)
    if (g.tid == 0 && !*abort) {
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
        const uint64_t t0 = global_ns();
        uint32_t it = 0;
        while (ld_acquire_u64(ctr) < target) {  // acquire: other CTAs' writes are visible after the loop
            if ((++it & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                raise_status(status, kStatusTimeout);
                *abort = 1;
                break;
            }
        }
    }
    g.sync();
    return !*abort;
}

}  // namespace qlin
