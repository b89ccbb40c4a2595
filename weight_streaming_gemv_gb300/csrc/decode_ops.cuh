// Device building blocks of the ternary decode step (RMSNorm, RoPE, decode
// attention, GeGLU, lm_head argmax), shared by the standalone kernels and the
// fused decode step.  Every fp32 sum that can reach an activation quantiser
// uses a fixed order: a balanced pairwise tree over the terms, zero-padded to
// a power of two.
#pragma once

#include "common.cuh"

namespace qlin {

// A group of n consecutive threads (whole warps, n >= 32) that
// synchronises on hardware barrier `bar`; tid is the thread's rank in it.
// Group{threadIdx.x, blockDim.x, 0} is the whole block (barrier 0 is the one
// __syncthreads uses).
struct Grp {
    int tid, n, bar;
    __device__ __forceinline__ void sync() const { asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory"); }
    __device__ __forceinline__ int lane() const { return tid & 31; }
    __device__ __forceinline__ int warp() const { return tid >> 5; }
};

__device__ __forceinline__ Grp whole_block() { return Grp{(int)threadIdx.x, (int)blockDim.x, 0}; }

// Pairwise sum of buf[0..P) (P a power of two, zero-padded by the caller) by
// a group of threads.  The first T threads (T = the largest power of two not
// above the group size) each reduce their own segment of P/T consecutive
// terms in place, then lanes, then warps, always adjacent subtrees first.
// `red` holds >= 32 floats.  Every thread of the group must call it.
__device__ __forceinline__ float block_psum(float *buf, int P, float *red, Grp g) {
    int T = 32;
    while (2 * T <= g.n) T *= 2;
    const int t = g.tid;
    g.sync();
    float v = 0.0f;
    if (t < T) {
        if (P >= T) {
            const int S = P / T;
            float *a = buf + t * S;
            for (int st = 1; st < S; st <<= 1)
                for (int i = 0; i < S; i += 2 * st) a[i] = __fadd_rn(a[i], a[i + st]);
            v = a[0];
        } else {
            v = (t < P) ? buf[t] : 0.0f;
        }
    }
    v = warp_psum(v);
    if ((t & 31) == 0 && t < T) red[t >> 5] = v;
    g.sync();
    if (t == 0) {
        const int W = T >> 5;  // a power of two
        for (int st = 1; st < W; st <<= 1)
            for (int i = 0; i < W; i += 2 * st) red[i] = __fadd_rn(red[i], red[i + st]);
    }
    g.sync();
    const float r = red[0];
    g.sync();
    return r;
}

// Streaming form of the same pairwise tree for one thread: push the terms in
// order; result() equals the zero-padded balanced tree over them.  Up to
// 2^MAXD terms.
template <int MAXD>
struct PairwiseStream {
    float stk[MAXD + 1];
    unsigned n = 0;
    __device__ __forceinline__ void push(float v) {
        unsigned j = n++;
        int k = 0;
#pragma unroll 1
        while (j & 1u) {
            v = __fadd_rn(stk[k], v);
            j >>= 1;
            k++;
        }
        stk[k] = v;
    }
    __device__ __forceinline__ float result() const {
        // pending subtrees are combined from the smallest (rightmost) upwards:
        // the missing right parts are zeros, and x + 0 = x.
        float acc = 0.0f;
        bool have = false;
#pragma unroll 1
        for (int k = 0; k <= MAXD; k++)
            if (n & (1u << k)) {
                acc = have ? __fadd_rn(stk[k], acc) : stk[k];
                have = true;
            }
        return acc;
    }
};

// RMSNorm of one row of n floats into out (may alias x): o = g * (r * x),
// r = 1/sqrtf(ss/n + eps), ss the pairwise sum of x^2.  buf: smem >= P
// floats (P = next_pow2(n)), red: smem >= 32 floats.
__device__ __forceinline__ void rmsnorm_row(const float *x, const float *g, float *out, int n, float eps, float *buf,
                                            float *red, Grp gr) {
    const int P = next_pow2(n);
    for (int i = gr.tid; i < P; i += gr.n) {
        const float v = (i < n) ? x[i] : 0.0f;
        buf[i] = __fmul_rn(v, v);
    }
    float ss = block_psum(buf, P, red, gr);
    ss = __fdiv_rn(ss, (float)n);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    for (int i = gr.tid; i < n; i += gr.n) out[i] = __fmul_rn(g[i], __fmul_rn(r, x[i]));
}

// RoPE on pairs (i, i + hd/2) of each head of v [nh][hd]: x' = xc - ys, y' = xs + yc.
__device__ __forceinline__ void rope_rotate(float *v, int nh, int hd, const float *c, const float *s, Grp g) {
    const int half = hd / 2;
    for (int idx = g.tid; idx < nh * half; idx += g.n) {
        const int h = idx / half, i = idx % half;
        float *p = v + h * hd;
        const float a = p[i], b = p[i + half];
        const float ci = c[i], si = s[i];
        p[i] = __fsub_rn(__fmul_rn(a, ci), __fmul_rn(b, si));
        p[i + half] = __fadd_rn(__fmul_rn(a, si), __fmul_rn(b, ci));
    }
}

// Attention over one chunk of <= 32 positions for one head.
//   q: smem [hd]; K, V: row t of the chunk at Kc + t*ld, Vc + t*ld (global or
//   smem); nt valid positions.  Writes m_c, S_c and U_c[hd] (pairwise sums
//   over the 32 slots of e_t and e_t * v_t) to out_m, out_S, out_U.
//   sc: smem >= 32 floats.  Block of 256 threads; hd a power of two <= 256.
template <int HD>
__device__ __forceinline__ void attention_chunk_t(const float *q, const float *Kc, const float *Vc, int ld, int nt,
                                                  float *out_m, float *out_S, float *out_U, float *sc, Grp g) {
    constexpr int hd = HD;
    const int lane = g.lane(), warp = g.warp(), nwarps = g.n >> 5;
    const float div = __fsqrt_rn((float)hd);
    // each lane owns the contiguous dims [lane*S, lane*S + S) (the leaves of its
    // subtree); its q values stay in registers for all positions
    constexpr int S = HD >= 32 ? HD / 32 : 1;
    float qr[S];
#pragma unroll
    for (int i = 0; i < S; i++) qr[i] = (HD >= 32 || lane < HD) ? q[lane * S + i] : 0.0f;
    for (int t = warp; t < 32; t += nwarps) {
        float part = 0.0f;
        if (t < nt) {
            const float *k = Kc + (int64_t)t * ld;
            if constexpr (HD >= 32) {
                float kr[S];
                if constexpr (S == 8) {
                    // two 16-byte loads; lanes 4..7 of each shared-memory phase read
                    // their upper half first so the 8 lanes hit distinct banks
                    const float4 *k4 = reinterpret_cast<const float4 *>(k + lane * S);
                    const int sw = (lane >> 2) & 1;
                    const float4 f = k4[sw], s2 = k4[sw ^ 1];
                    const float4 lo = sw ? s2 : f, hi = sw ? f : s2;
                    kr[0] = lo.x;
                    kr[1] = lo.y;
                    kr[2] = lo.z;
                    kr[3] = lo.w;
                    kr[4] = hi.x;
                    kr[5] = hi.y;
                    kr[6] = hi.z;
                    kr[7] = hi.w;
                } else if constexpr (S == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(k + lane * 4);
                    kr[0] = v.x;
                    kr[1] = v.y;
                    kr[2] = v.z;
                    kr[3] = v.w;
                } else {
#pragma unroll
                    for (int i = 0; i < S; i++) kr[i] = k[lane * S + i];
                }
                float p[S];
#pragma unroll
                for (int i = 0; i < S; i++) p[i] = __fmul_rn(qr[i], kr[i]);
#pragma unroll
                for (int st = 1; st < S; st <<= 1)
#pragma unroll
                    for (int i = 0; i < S; i += 2 * st) p[i] = __fadd_rn(p[i], p[i + st]);
                part = p[0];
            } else if (lane < hd) {
                part = __fmul_rn(qr[0], k[lane]);
            }
        }
        const float s = warp_psum(part);
        if (lane == 0) sc[t] = (t < nt) ? __fdiv_rn(s, div) : 0.0f;
    }
    g.sync();
    if (g.tid < 32) {
        const int t = g.tid;
        const float m = warp_max(t < nt ? sc[t] : -__int_as_float(0x7f800000));
        const float e = (t < nt) ? exp32(__fsub_rn(sc[t], m)) : 0.0f;
        __syncwarp();
        sc[t] = e;
        const float S = warp_psum(e);
        if (t == 0) {
            *out_m = m;
            *out_S = S;
        }
    }
    g.sync();
    // U: dims split so that one pass covers the head (two dims per thread when
    // the head is wider than the group)
    const int dpt = hd > g.n ? 2 : 1;
    for (int i0 = g.tid * dpt; i0 < hd; i0 += g.n * dpt) {
#pragma unroll
        for (int dd = 0; dd < 2; dd++) {
            if (dd < dpt) {
                const int i = i0 + dd;
                float p[32];
#pragma unroll
                for (int t = 0; t < 32; t++) p[t] = (t < nt) ? __fmul_rn(sc[t], Vc[(int64_t)t * ld + i]) : 0.0f;
#pragma unroll
                for (int st = 1; st < 32; st <<= 1)
#pragma unroll
                    for (int t = 0; t < 32; t += 2 * st) p[t] = __fadd_rn(p[t], p[t + st]);
                out_U[i] = p[0];
            }
        }
    }
    g.sync();
}

// head_dim dispatch (16..256, powers of two) so every per-lane array is static
__device__ __forceinline__ void attention_chunk(const float *q, const float *Kc, const float *Vc, int ld, int nt, int hd,
                                                float *out_m, float *out_S, float *out_U, float *sc, Grp g) {
    switch (hd) {
        case 16: attention_chunk_t<16>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, g); break;
        case 32: attention_chunk_t<32>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, g); break;
        case 64: attention_chunk_t<64>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, g); break;
        case 128: attention_chunk_t<128>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, g); break;
        default: attention_chunk_t<256>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, g); break;
    }
}

// Merge of nc chunk partials of one head: m = max m_c, w_c = e^{m_c - m},
// S = sum S_c w_c, out = (sum U_c w_c) / S, every sum pairwise over the
// chunks.  wbuf: smem >= next_pow2(nc) floats, red: smem >= 32 floats.
__device__ __forceinline__ void attention_merge(const float *pm, const float *pS, const float *pU, int nc, int hd,
                                                float *out, float *wbuf, float *red, Grp g) {
    // partials are written by other CTAs: read them from L2 (__ldcg), never a stale L1 line
    float m = __ldcg(pm);
    for (int c = 1; c < nc; c++) m = fmaxf(m, __ldcg(pm + c));
    const int P = next_pow2(nc);
    for (int c = g.tid; c < P; c += g.n) wbuf[c] = (c < nc) ? exp32(__fsub_rn(__ldcg(pm + c), m)) : 0.0f;
    g.sync();
    for (int i = g.tid; i < hd; i += g.n) {
        PairwiseStream<16> ps;
        for (int c = 0; c < nc; c++) ps.push(__fmul_rn(__ldcg(pU + (int64_t)c * hd + i), wbuf[c]));
        out[i] = ps.result();
    }
    g.sync();
    // S: reuse wbuf as the product buffer
    for (int c = g.tid; c < P; c += g.n) wbuf[c] = (c < nc) ? __fmul_rn(__ldcg(pS + c), wbuf[c]) : 0.0f;
    const float S = block_psum(wbuf, P, red, g);
    for (int i = g.tid; i < hd; i += g.n) out[i] = __fdiv_rn(out[i], S);
    g.sync();
}

// Copies n floats (n % 4 == 0, 16-byte aligned) written by other CTAs from
// global memory (L2, never a stale L1 line) into shared memory, every load of
// a thread in flight together.
__device__ __forceinline__ void load_l2_f4(float *dst, const float *src, int n, Grp g) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    const int n4 = n / 4;
    for (int i0 = 0; i0 < n4; i0 += 4 * g.n) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = __ldcg(s4 + min(i0 + g.tid + j * g.n, n4 - 1));  // clamped: all in flight
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = i0 + g.tid + j * g.n;
            if (i < n4) d4[i] = v[j];
        }
    }
}

// attention_merge for all heads at once, with the loads batched and no
// local memory: the same arithmetic (and so the same bits) as
// attention_merge.  nc <= 128.  Partials are
// pm/pS [nh][ncmax], pU [nh][ncmax][hd]; out [nh][hd]; wsm: smem >= nh *
// next_pow2(nc) floats; red: smem >= 32 floats.  hd % 4 == 0.
__device__ __forceinline__ void attention_merge_all(const float *pm, const float *pS, const float *pU, int nc,
                                                    int ncmax, int nh, int hd, float *out, float *wsm, float *red,
                                                    Grp g) {
    const int P = next_pow2(nc);
    // maxima and weights per head
    for (int idx = g.tid; idx < nh * P; idx += g.n) wsm[idx] = (idx % P < nc) ? __ldcg(pm + (idx / P) * ncmax + idx % P) : 0.0f;
    g.sync();
    for (int h = 0; h < nh; h++) {
        float m = wsm[h * P];
        for (int c = 1; c < nc; c++) m = fmaxf(m, wsm[h * P + c]);
        g.sync();
        for (int c = g.tid; c < P; c += g.n) wsm[h * P + c] = (c < nc) ? exp32(__fsub_rn(wsm[h * P + c], m)) : 0.0f;
        g.sync();
    }
    // U: one float4 of one head per thread.  The pairwise tree over the
    // zero-padded chunks is evaluated as 16 blocks of 8 (8 loads in flight per
    // block, a fixed 3-level tree in registers) and a fixed 4-level tree over
    // the block sums: the tree over 128 zero-padded leaves, which equals the
    // tree over next_pow2(nc) leaves because x + 0 = x.  nc <= 128.
    const int nq = nh * hd / 4;
    for (int qi = g.tid; qi < nq; qi += g.n) {
        const int h = (qi * 4) / hd, i = (qi * 4) % hd;
        const float *base = pU + (int64_t)h * ncmax * hd + i;
        const float *w = wsm + h * P;
        float4 bp[16];
#pragma unroll
        for (int kb = 0; kb < 16; kb++) {
            bp[kb] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kb * 8 < nc) {
                float4 v[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int c = kb * 8 + j;
                    if (c < nc) {
                        const float4 u = __ldcg(reinterpret_cast<const float4 *>(base + (int64_t)c * hd));
                        const float wc = w[c];
                        v[j] = make_float4(__fmul_rn(u.x, wc), __fmul_rn(u.y, wc), __fmul_rn(u.z, wc),
                                           __fmul_rn(u.w, wc));
                    } else {
                        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int st = 1; st < 8; st <<= 1)
#pragma unroll
                    for (int j = 0; j < 8; j += 2 * st)
                        v[j] = make_float4(__fadd_rn(v[j].x, v[j + st].x), __fadd_rn(v[j].y, v[j + st].y),
                                           __fadd_rn(v[j].z, v[j + st].z), __fadd_rn(v[j].w, v[j + st].w));
                bp[kb] = v[0];
            }
        }
#pragma unroll
        for (int st = 1; st < 16; st <<= 1)
#pragma unroll
            for (int j = 0; j < 16; j += 2 * st)
                bp[j] = make_float4(__fadd_rn(bp[j].x, bp[j + st].x), __fadd_rn(bp[j].y, bp[j + st].y),
                                    __fadd_rn(bp[j].z, bp[j + st].z), __fadd_rn(bp[j].w, bp[j + st].w));
        float *o = out + h * hd + i;
        o[0] = bp[0].x;
        o[1] = bp[0].y;
        o[2] = bp[0].z;
        o[3] = bp[0].w;
    }
    g.sync();
    // S per head, then divide
    for (int h = 0; h < nh; h++) {
        float *buf = wsm + h * P;
        for (int c = g.tid; c < P; c += g.n) buf[c] = (c < nc) ? __fmul_rn(__ldcg(pS + h * ncmax + c), buf[c]) : 0.0f;
        const float S = block_psum(buf, P, red, g);
        for (int i = g.tid; i < hd; i += g.n) out[h * hd + i] = __fdiv_rn(out[h * hd + i], S);
        g.sync();
    }
}

// One element o[h][i] of the merged attention output, computed by one warp
// with the same trees as attention_merge: m = max_c m_c, w_c = e^{m_c - m},
// S = pairwise sum of S_c w_c, U = pairwise sum of U_c[i] w_c over the
// zero-padded P = next_pow2(nc) chunks, o = U / S.  Lane l holds the
// consecutive leaves [l*L, l*L + L), L = max(1, P/32), so the in-lane sums
// followed by warp_psum are that balanced tree.  nc <= 128.  Returns o in
// every lane.
__device__ __forceinline__ float attention_merge_one(const float *pm, const float *pS, const float *pU, int nc,
                                                     int hd, int i, int lane) {
    const int P = next_pow2(nc);
    const int Lf = P > 32 ? P / 32 : 1;  // leaves per lane: 1, 2 or 4
    float mv[4], sv[4], uv[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = lane * Lf + j;
        const bool ok = j < Lf && c < nc;
        mv[j] = ok ? __ldcg(pm + c) : -__int_as_float(0x7f800000);
        sv[j] = ok ? __ldcg(pS + c) : 0.0f;
        uv[j] = ok ? __ldcg(pU + (int64_t)c * hd + i) : 0.0f;
    }
    float m = fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3]));
    m = warp_max(m);
    float ws[4], wu[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = lane * Lf + j;
        const bool ok = j < Lf && c < nc;
        const float w = ok ? exp32(__fsub_rn(mv[j], m)) : 0.0f;
        ws[j] = ok ? __fmul_rn(sv[j], w) : 0.0f;
        wu[j] = ok ? __fmul_rn(uv[j], w) : 0.0f;
    }
    // in-lane subtree over Lf leaves (Lf = 1, 2 or 4)
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

// Launches the chunk and merge kernels of the decode attention on `st`; `ws`
// holds n_heads * ncmax * (head_dim + 2) floats, ncmax >= pos/32 + 1.
qlin_status launch_attention(const float *q, const float *kc, const float *vc, int pos, int nh, int nkv, int hd,
                             float *out, float *ws, int ncmax, cudaStream_t st);

}  // namespace qlin
