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
constexpr int kFConsumerWarps = 11;  // + 1 producer warp = 12 warps: 3 per SM sub-partition, up to 168 registers
constexpr int kFThreads = 32 * (kFConsumerWarps + 1);
constexpr int kFMaxRows = 512;  // rows of a T158 piece (their integer sums wait in shared memory)

struct FusedArgs {
    t158_model m;
    float *kv;
    const int32_t *token;
    int pos;
    float *logits;
    int32_t *next;
    float *final_x;  // non-null: stop after the final norm and write it here (no lm_head, next untouched)
    // workspace: vectors passed between CTAs as tagged words (value | tag << 32)
    uint64_t *hT, *qkvT, *attT, *aT, *pmT, *pST, *pUT;
    int ncmax;
    float2 *lm_part;
    unsigned *lm_ticket;
    unsigned *seq;  // launch sequence number, advanced by the last CTA of every launch
    int32_t *status;
};

// ---------------------------------------------------------------- tagged words
// A float handed from one CTA to others is stored together with a tag in one
// 8-byte word (relaxed, gpu scope: single-copy atomic), so a reader that sees
// the tag of the current launch, layer and phase also sees the value.  This
// replaces grid-wide barriers: every CTA waits only for the words it reads.
__device__ __forceinline__ uint32_t make_tag(uint32_t seq, int layer, int phase) {
    return (seq << 10) | ((uint32_t)layer << 3) | (uint32_t)phase;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
    const uint64_t w = (uint64_t)__float_as_uint(v) | ((uint64_t)tag << 32);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// out[j] = value of the tagged word at ptr(j) for every j whose bit is set in
// `mask`, 0 for the others; waits (bounded) until every one of those words
// carries `tag`.  All loads of a round are in flight together; only words
// still stale are reloaded.  On timeout: status gets kStatusTimeout, *abort
// is set.
template <int N, class Ptr>
__device__ __forceinline__ void fetch_tagged_at(Ptr &&ptr, uint32_t mask, uint32_t tag, float (&out)[N],
                                                volatile int *abort, int32_t *status) {
    uint64_t w[N];
#pragma unroll
    for (int j = 0; j < N; j++) w[j] = 0;
    uint32_t pending = mask;
    uint64_t t0 = 0;
    // one block of loads serves the first pass and every retry (a small loop
    // body keeps the instruction cache free for the rest of the layer)
    for (int pass = 0;; pass++) {
#pragma unroll
        for (int j = 0; j < N; j++)
            if (pending & (1u << j)) w[j] = ld_relaxed_u64(ptr(j));
#pragma unroll
        for (int j = 0; j < N; j++)
            if ((pending & (1u << j)) && (uint32_t)(w[j] >> 32) == tag) pending &= ~(1u << j);
        if (!pending || *abort) break;
        if (pass == 0) t0 = global_ns();
        if (global_ns() - t0 > kWaitLimitNs) {
            raise_status(status, kStatusTimeout);
            *abort = 1;
            break;
        }
        __nanosleep(32);
    }
#pragma unroll
    for (int j = 0; j < N; j++) out[j] = (mask & (1u << j)) ? __uint_as_float((uint32_t)w[j]) : 0.0f;
}

// src[first + j * stride] for j < count (count <= N)
template <int N>
__device__ __forceinline__ void fetch_tagged(const uint64_t *src, int first, int stride, int count, uint32_t tag,
                                             float (&out)[N], volatile int *abort, int32_t *status) {
    const uint32_t mask = count >= 32 ? 0xffffffffu : (1u << (count > 0 ? count : 0)) - 1u;
    fetch_tagged_at<N>([&](int j) { return src + first + j * stride; }, mask, tag, out, abort, status);
}

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
            pieces(m.w[j] + (int64_t)l * rows[j] * m.pitch[j], m.pitch[j], a0 - base, a1 - base, j, f, kFMaxRows);
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
    pieces(m.w[3] + (int64_t)l * rows[3] * m.pitch[3], m.pitch[3], lo, hi, 3, f, kFMaxRows);
    int g0, g1;
    share(ff, b, G, g0, g1);
    // gate and up in pairs over the same rows (one pass computes both)
    pieces(m.w[4] + (int64_t)l * rows[4] * m.pitch[4], m.pitch[4], g0, g1, 4, [&](const Piece &p) {
        f(p);
        Piece u = p;
        u.mat = 5;
        u.src = m.w[5] + (int64_t)l * rows[5] * m.pitch[5] + (int64_t)p.row0 * m.pitch[5];
        f(u);
    }, kFMaxRows);
    pieces(m.w[6] + (int64_t)l * rows[6] * m.pitch[6], m.pitch[6], lo, hi, 6, f, kFMaxRows);
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
// Codes of v (shared memory, K elements) for step `scale` into the plane
// layout, one plane word per thread and round: word c*20 + 4i + w holds, in
// byte b, the code of element 5(16c + 4w + b) + i (0 past K).  The sum of the
// codes is added into *isum (shared memory, zeroed by the caller before the
// last group barrier).  No group barrier inside: the caller syncs once after.
__device__ __forceinline__ void planes_words(const float *v, int K, float scale, int C, uint4 *xr, int *isum, Grp g) {
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const float rinv = __fdiv_rn(1.0f, scale);
    const int nwords = C * 20;
    int s = 0;
    for (int wi = g.tid; wi < nwords; wi += g.n) {
        const int c = wi / 20, r = wi - 20 * c;
        const int base = 5 * (16 * c + 4 * (r & 3)) + (r >> 2);
        uint32_t word = 0;
#pragma unroll
        for (int bb = 0; bb < 4; bb++) {
            const int k = base + 5 * bb;
            const int q = k < K ? quant_code_r(v[k], scale, rinv) : 0;
            s += q;
            word |= (uint32_t)(q & 0xff) << (8 * bb);
        }
        xw[wi] = word;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (g.lane() == 0) atomicAdd(isum, s);
}

// Sum of squares of x[0..d) (d <= 4096) as the pairwise tree over
// next_pow2(d) zero-padded leaves.  The 32-leaf segment s of x (elements
// 32s .. 32s+31) is held by warp s mod nw, one element per lane, so the loads
// are coalesced; the warp sums the squares of a segment with the adjacent-lane
// tree (its lower five levels) and seg[s] keeps the result.  With srcT the
// vector comes from tagged words (waited for by tag) and is staged into xs;
// without, xs already holds it.  The caller syncs the group, then calls
// seg_total.
__device__ __forceinline__ void stage_segments(const uint64_t *srcT, uint32_t tag, float *xs, int d, float *seg,
                                               Grp g, volatile int *abort, int32_t *status) {
    constexpr int N = 8;
    const int nw = g.n >> 5, lane = g.lane(), w = g.warp();
    const int nseg = (d + 31) >> 5;
    for (int s0 = 0; s0 < nseg; s0 += N * nw) {
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < N; j++) {
            const int k = 32 * (s0 + w + j * nw) + lane;
            if (k < d) mask |= 1u << j;
        }
        float v[N];
        if (srcT) {
            fetch_tagged_at<N>([&](int j) { return srcT + 32 * (s0 + w + j * nw) + lane; }, mask, tag, v, abort,
                               status);
#pragma unroll
            for (int j = 0; j < N; j++)
                if (mask & (1u << j)) xs[32 * (s0 + w + j * nw) + lane] = v[j];
        } else {
#pragma unroll
            for (int j = 0; j < N; j++) v[j] = (mask & (1u << j)) ? xs[32 * (s0 + w + j * nw) + lane] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < N; j++) {
            const int sg = s0 + w + j * nw;  // uniform across the warp
            if (sg < nseg) {
                const float sq = warp_psum(__fmul_rn(v[j], v[j]));
                if (lane == 0) seg[sg] = sq;
            }
        }
    }
}

// The upper levels of the tree of stage_segments: every warp sums the
// segment sums (zero past the last segment of x) and returns the total.
__device__ __forceinline__ float seg_total(const float *seg, int d, Grp g) {
    const int nseg = (d + 31) >> 5;
    const int ns = next_pow2(d) >> 5;  // segments of the padded tree (>= 1)
    const int L = ns > 32 ? ns / 32 : 1;  // 1, 2 or 4 per lane
    const int lane = g.lane();
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int idx = lane * L + i;
        a[i] = (i < L && idx < nseg) ? seg[idx] : 0.0f;
    }
    float t = a[0];
    if (L == 2) t = __fadd_rn(a[0], a[1]);
    if (L == 4) t = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
    return warp_psum(t);
}

// RMSNorm + absmax quantisation of a d-vector (d <= 4096) into the planes,
// with three group barriers.  The vector comes from tagged words srcT (other
// CTAs' output, waited for by tag, staged into xs) or, when srcT is null, is
// already in xs (shared memory).  Sum of squares as stage_segments/seg_total;
// each thread normalises the elements k = t, t + n, ... into xn, with its
// gains (global memory, read-only) read into registers before the vector
// arrives; the group takes the absmax, and the codes are written one plane
// word per thread (planes_words).  Returns the step; *sumx gets the sum of
// the codes.  The arithmetic is that of rmsnorm_row and the
// absmax quantiser.
__device__ __forceinline__ float norm_quant(const uint64_t *srcT, uint32_t tag, float *xs, const float *gam, int d,
                                            float eps, float *xn, uint4 *xr, int C, float *red, float *seg, int *isum,
                                            int *sumx, Grp g, volatile int *abort, int32_t *status) {
    const int t = g.tid;
    constexpr int MAXE = 20;  // elements per thread (d <= 20 * group size)
    float gv[MAXE];
#pragma unroll
    for (int e = 0; e < MAXE; e++) {
        const int k = t + e * g.n;
        gv[e] = k < d ? __ldg(gam + k) : 0.0f;
    }
    stage_segments(srcT, tag, xs, d, seg, g, abort, status);
    g.sync();  // 1: segment sums and the staged vector are visible
    float ss = seg_total(seg, d, g);
    ss = __fdiv_rn(ss, (float)d);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < MAXE; e++) {
        const int k = t + e * g.n;
        if (k < d) {
            const float val = __fmul_rn(gv[e], __fmul_rn(r, xs[k]));
            xn[k] = val;
            amax = fmaxf(amax, fabsf(val));
        }
    }
    amax = warp_max(amax);
    if (g.lane() == 0) red[8 + g.warp()] = amax;
    if (t == 0) *isum = 0;
    g.sync();  // 2: the normalised vector and the absmax parts
    float m = red[8];
    for (int w = 1; w < (g.n >> 5); w++) m = fmaxf(m, red[8 + w]);
    const float scale = quant_scale(m);
    planes_words(xn, d, scale, C, xr, isum, g);
    g.sync();  // 3: planes and the code sum
    *sumx = *isum;
    return scale;
}

// Absmax quantisation of a K-vector of tagged words (other CTAs' output, waited
// for by tag) into the planes, with two group barriers: the vector is staged
// in v (shared memory) while each thread tracks its maximum.
__device__ __forceinline__ float quant_from_tagged(const uint64_t *srcT, uint32_t tag, int K, float *v, uint4 *xr, int C,
                                                   float *red, int *isum, int *sumx, Grp g, volatile int *abort,
                                                   int32_t *status) {
    float amax = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 32 * g.n) {
        const int first = k0 + g.tid;
        const int cnt = first < K ? min(32, (K - first + g.n - 1) / g.n) : 0;
        float val[32];
        fetch_tagged<32>(srcT, first < K ? first : 0, g.n, cnt, tag, val, abort, status);
#pragma unroll
        for (int j = 0; j < 32; j++)
            if (j < cnt) {
                v[first + j * g.n] = val[j];
                amax = fmaxf(amax, fabsf(val[j]));
            }
    }
    amax = warp_max(amax);
    if (g.lane() == 0) red[g.warp()] = amax;
    if (g.tid == 0) *isum = 0;
    g.sync();
    float m = red[0];
    for (int w = 1; w < (g.n >> 5); w++) m = fmaxf(m, red[w]);
    const float scale = quant_scale(m);
    planes_words(v, K, scale, C, xr, isum, g);
    g.sync();
    *sumx = *isum;
    return scale;
}

// RMSNorm of the d-vector of tagged words srcT (waited for by tag) into xn
// (shared memory), staging x in xs; gains gam in global memory.  Same tree as
// rmsnorm_row.
__device__ __forceinline__ void rmsnorm_from_tagged(const uint64_t *srcT, uint32_t tag, const float *gam, float *xs,
                                                    float *xn, int d, float eps, float *seg, Grp g,
                                                    volatile int *abort, int32_t *status) {
    stage_segments(srcT, tag, xs, d, seg, g, abort, status);
    g.sync();
    float ss = seg_total(seg, d, g);
    ss = __fdiv_rn(ss, (float)d);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    for (int i = g.tid; i < d; i += g.n) xn[i] = __fmul_rn(__ldg(gam + i), __fmul_rn(r, xs[i]));
    g.sync();
}

// attention_merge_one on tagged partials (pm/pS [chunk], pU [chunk][hd] of
// one head), waiting for each word's tag: one output element per warp.
__device__ __forceinline__ float attention_merge_tagged(const uint64_t *pm, const uint64_t *pS, const uint64_t *pU,
                                                        int nc, int hd, int i, int lane, uint32_t tag,
                                                        volatile int *abort, int32_t *status) {
    const int P = next_pow2(nc);
    const int Lf = P > 32 ? P / 32 : 1;  // leaves per lane: 1, 2 or 4 (nc <= 128)
    const int c0 = lane * Lf;
    const int cnt = c0 < nc ? min(Lf, nc - c0) : 0;
    float all[12];
    const uint32_t m4 = (1u << cnt) - 1u;
    fetch_tagged_at<12>(
        [&](int j) {
            const int c = c0 + (j & 3);
            return j < 4 ? pm + c : j < 8 ? pS + c : pU + (int64_t)c * hd + i;
        },
        m4 | (m4 << 4) | (m4 << 8), tag, all, abort, status);
    float mv[4], sv[4], uv[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        mv[j] = all[j];
        sv[j] = all[4 + j];
        uv[j] = all[8 + j];
    }
    float m = -__int_as_float(0x7f800000);
#pragma unroll
    for (int j = 0; j < 4; j++)
        if (j < cnt) m = fmaxf(m, mv[j]);
    m = warp_max(m);
    float ws[4], wu[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const bool ok = j < cnt;
        const float w = ok ? exp32(__fsub_rn(mv[j], m)) : 0.0f;
        ws[j] = ok ? __fmul_rn(sv[j], w) : 0.0f;
        wu[j] = ok ? __fmul_rn(uv[j], w) : 0.0f;
    }
    float s_l = ws[0], u_l = wu[0];
    if (Lf == 2) {
        s_l = __fadd_rn(ws[0], ws[1]);
        u_l = __fadd_rn(wu[0], wu[1]);
    } else if (Lf == 4) {
        s_l = __fadd_rn(__fadd_rn(ws[0], ws[1]), __fadd_rn(ws[2], ws[3]));
        u_l = __fadd_rn(__fadd_rn(wu[0], wu[1]), __fadd_rn(wu[2], wu[3]));
    }
    const float S = warp_psum(s_l);
    const float U = warp_psum(u_l);
    return __fdiv_rn(U, S);
}

// ---------------------------------------------------------------- T158 rows from a slot
// acc + the dot product of one 16-byte chunk of packed trits (digits 0..2)
// with its 80 activation codes in plane order X[0..5).
__device__ __forceinline__ int chunk_dot(const uint4 wv, const uint4 *X, int acc) {
    uint32_t D[4][5];
    t158_planes(wv.x, D[0]);
    t158_planes(wv.y, D[1]);
    t158_planes(wv.z, D[2]);
    t158_planes(wv.w, D[3]);
#pragma unroll
    for (int i = 0; i < 5; i++) {
        const uint4 xv = X[i];
        acc = dp4a(D[0][i], xv.x, acc);
        acc = dp4a(D[1][i], xv.y, acc);
        acc = dp4a(D[2][i], xv.z, acc);
        acc = dp4a(D[3][i], xv.w, acc);
    }
    return acc;
}

// Integer row sums of `rows` packed rows (pitch bytes each) at `slot` against
// the planes xr, added into racc[row] (shared memory, zero on entry); with
// slot2, rows rows1.. come from slot2 (two matrices of one input in one pass).  The
// rows x C chunk dot products are spread over the whole group in units of U
// chunks of one row (U <= 4, so that nearly every thread has work and keeps
// several independent chunks in flight); unit k of a row takes chunks k,
// k + upr, ... so consecutive lanes read consecutive chunks.  Partial sums
// meet through shared-memory atomics: integer addition, exact in any order.
__device__ __forceinline__ void t158_rows(const uint8_t *slot, int rows, int pitch, const uint4 *xr, int *racc, Grp g,
                                          const uint8_t *slot2 = nullptr, int rows1 = 1 << 30) {
    const int C = pitch / 16;
    int U = (rows * C + g.n - 1) / g.n;
    U = U < 1 ? 1 : U > 4 ? 4 : U;
    const int upr = (C + U - 1) / U;
    const int units = rows * upr;
    for (int u = g.tid; u < units; u += g.n) {
        const int r = u / upr, k = u - r * upr;
        const uint8_t *wr = r < rows1 ? slot + (size_t)r * pitch : slot2 + (size_t)(r - rows1) * pitch;
        int a0 = 0, a1 = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = k + j * upr;
            if (j < U && c < C) {
                const int t = chunk_dot(lds128(wr + (size_t)c * 16), xr + (size_t)c * 5, 0);
                if (j & 1)
                    a1 += t;
                else
                    a0 += t;
            }
        }
        atomicAdd(&racc[r], a0 + a1);
    }
}

}  // namespace qlin
