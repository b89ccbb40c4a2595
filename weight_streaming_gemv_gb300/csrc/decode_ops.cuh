// Device building blocks of the ternary decode step (RMSNorm, RoPE, decode
// attention, GeGLU, lm_head argmax), shared by the standalone kernels and the
// fused decode step.  Every fp32 sum that can reach an activation quantiser
// uses a fixed order: a balanced pairwise tree over the terms, zero-padded to
// a power of two.
#pragma once

#include "common.cuh"

namespace qlin {

// Pairwise sum of buf[0..P) (P a power of two, zero-padded by the caller) by
// the whole block (blockDim.x a power of two >= 32).  Thread t first reduces
// its own segment of P/T consecutive terms in place (T = blockDim.x), then
// lanes, then warps, always adjacent subtrees first.  `red` holds >= 32
// floats.  Contains __syncthreads(); every thread of the block must call it.
__device__ __forceinline__ float block_psum(float *buf, int P, float *red) {
    const int T = blockDim.x, t = threadIdx.x;
    __syncthreads();
    float v;
    if (P >= T) {
        const int S = P / T;
        float *a = buf + t * S;
        for (int st = 1; st < S; st <<= 1)
            for (int i = 0; i < S; i += 2 * st) a[i] = __fadd_rn(a[i], a[i + st]);
        v = a[0];
    } else {
        v = (t < P) ? buf[t] : 0.0f;
    }
    v = warp_psum(v);
    if ((t & 31) == 0) red[t >> 5] = v;
    __syncthreads();
    if (t == 0) {
        const int W = T >> 5;
        for (int st = 1; st < W; st <<= 1)
            for (int i = 0; i < W; i += 2 * st) red[i] = __fadd_rn(red[i], red[i + st]);
    }
    __syncthreads();
    const float r = red[0];
    __syncthreads();
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
                                            float *red) {
    const int P = next_pow2(n);
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const float v = (i < n) ? x[i] : 0.0f;
        buf[i] = __fmul_rn(v, v);
    }
    float ss = block_psum(buf, P, red);
    ss = __fdiv_rn(ss, (float)n);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = __fmul_rn(g[i], __fmul_rn(r, x[i]));
}

// RoPE on pairs (i, i + hd/2) of each head of v [nh][hd]: x' = xc - ys, y' = xs + yc.
__device__ __forceinline__ void rope_rotate(float *v, int nh, int hd, const float *c, const float *s) {
    const int half = hd / 2;
    for (int idx = threadIdx.x; idx < nh * half; idx += blockDim.x) {
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
__device__ __forceinline__ void attention_chunk(const float *q, const float *Kc, const float *Vc, int ld, int nt,
                                                int hd, float *out_m, float *out_S, float *out_U, float *sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const float div = __fsqrt_rn((float)hd);
    for (int t = warp; t < 32; t += nwarps) {
        float part = 0.0f;
        if (t < nt) {
            const float *k = Kc + (int64_t)t * ld;
            if (hd >= 32) {
                const int S = hd / 32;
                float p[8];
                for (int i = 0; i < S; i++) p[i] = __fmul_rn(q[lane * S + i], k[lane * S + i]);
                for (int st = 1; st < S; st <<= 1)
                    for (int i = 0; i < S; i += 2 * st) p[i] = __fadd_rn(p[i], p[i + st]);
                part = p[0];
            } else if (lane < hd) {
                part = __fmul_rn(q[lane], k[lane]);
            }
        }
        const float s = warp_psum(part);
        if (lane == 0) sc[t] = (t < nt) ? __fdiv_rn(s, div) : 0.0f;
    }
    __syncthreads();
    float m = sc[0];
    for (int t = 1; t < nt; t++) m = fmaxf(m, sc[t]);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int t = threadIdx.x;
        const float e = (t < nt) ? exp32(__fsub_rn(sc[t], m)) : 0.0f;
        sc[t] = e;
        const float S = warp_psum(e);
        if (t == 0) {
            *out_m = m;
            *out_S = S;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < hd; i += blockDim.x) {
        float p[32];
#pragma unroll
        for (int t = 0; t < 32; t++) p[t] = (t < nt) ? __fmul_rn(sc[t], Vc[(int64_t)t * ld + i]) : 0.0f;
#pragma unroll
        for (int st = 1; st < 32; st <<= 1)
#pragma unroll
            for (int t = 0; t < 32; t += 2 * st) p[t] = __fadd_rn(p[t], p[t + st]);
        out_U[i] = p[0];
    }
    __syncthreads();
}

// Merge of nc chunk partials of one head: m = max m_c, w_c = e^{m_c - m},
// S = sum S_c w_c, out = (sum U_c w_c) / S, every sum pairwise over the
// chunks.  wbuf: smem >= next_pow2(nc) floats, red: smem >= 32 floats.
__device__ __forceinline__ void attention_merge(const float *pm, const float *pS, const float *pU, int nc, int hd,
                                                float *out, float *wbuf, float *red) {
    float m = pm[0];
    for (int c = 1; c < nc; c++) m = fmaxf(m, pm[c]);
    const int P = next_pow2(nc);
    for (int c = threadIdx.x; c < P; c += blockDim.x) wbuf[c] = (c < nc) ? exp32(__fsub_rn(pm[c], m)) : 0.0f;
    __syncthreads();
    for (int i = threadIdx.x; i < hd; i += blockDim.x) {
        PairwiseStream<16> ps;
        for (int c = 0; c < nc; c++) ps.push(__fmul_rn(pU[(int64_t)c * hd + i], wbuf[c]));
        out[i] = ps.result();
    }
    __syncthreads();
    // S: reuse wbuf as the product buffer
    for (int c = threadIdx.x; c < P; c += blockDim.x) wbuf[c] = (c < nc) ? __fmul_rn(pS[c], wbuf[c]) : 0.0f;
    const float S = block_psum(wbuf, P, red);
    for (int i = threadIdx.x; i < hd; i += blockDim.x) out[i] = __fdiv_rn(out[i], S);
    __syncthreads();
}

// Launches the chunk and merge kernels of the decode attention on `st`; `ws`
// holds n_heads * ncmax * (head_dim + 2) floats, ncmax >= pos/32 + 1.
qlin_status launch_attention(const float *q, const float *kc, const float *vc, int pos, int nh, int nkv, int hd,
                             float *out, float *ws, int ncmax, cudaStream_t st);

}  // namespace qlin
