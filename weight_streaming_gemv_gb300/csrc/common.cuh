// Shared host plumbing and device building blocks of the qlin library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/qlin.h"

namespace qlin {

// ----------------------------------------------------------------- host errors
void set_error(const char *fmt, ...);
void clear_error();

#define QLIN_REQUIRE(cond, status, ...)          \
    do {                                         \
        if (!(cond)) {                           \
            ::qlin::set_error(__VA_ARGS__);      \
            return (status);                     \
        }                                        \
    } while (0)

#define QLIN_CUDA(call)                                                                            \
    do {                                                                                           \
        cudaError_t _e = (call);                                                                   \
        if (_e != cudaSuccess) {                                                                   \
            ::qlin::set_error("%s failed: %s (%s:%d)", #call, cudaGetErrorString(_e), __FILE__, __LINE__); \
            return QLIN_ERR_CUDA;                                                                  \
        }                                                                                          \
    } while (0)

#define QLIN_LAUNCHED(what)                                                                        \
    do {                                                                                           \
        cudaError_t _e = cudaGetLastError();                                                       \
        if (_e != cudaSuccess) {                                                                   \
            ::qlin::set_error("launch of %s failed: %s", what, cudaGetErrorString(_e));            \
            return QLIN_ERR_CUDA;                                                                  \
        }                                                                                          \
    } while (0)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// SM count and opt-in shared memory of the current device (cached per device).
int sm_count();
int max_smem_optin();

// Resident blocks per SM of `kern` (blockDim 256) for `smem` dynamic bytes on
// the current device, with the kernel's dynamic shared-memory limit raised to
// the opt-in maximum on first use.  Cached per (kernel, device, smem): the
// CUDA occupancy queries run once, not on every launch.
int blocks_per_sm(const void *kern, size_t smem);

// ----------------------------------------------------------------- device helpers
// 16-byte streaming load: read-only path, no L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Base-3 digit planes of four packed bytes.  Byte j of w holds
// b_j = sum_i d_i 3^i (d_i in {0,1,2}); D[i] gets d_i of every byte, in the
// byte positions of w.  F_i = floor(b / 3^i) is built by repeated exact
// division by 3, floor(v/3) = ((v + 1) * 85) >> 8 for v <= 255, on two 16-bit
// lanes at a time; then d_i = F_i - 3 F_{i+1}, a borrow-free bytewise
// subtraction.  F_4 = floor(F_3 / 3) = (11 F_3) >> 5 fits in byte lanes.
__device__ __forceinline__ void t158_planes(uint32_t w, uint32_t D[5]) {
    const uint32_t C85 = 0x00550055u;
    uint32_t L = __byte_perm(w, 0u, 0x4240u);  // [b0, 0, b2, 0]
    uint32_t H = __byte_perm(w, 0u, 0x4341u);  // [b1, 0, b3, 0]
    uint32_t PL = L * 85u + C85, PH = H * 85u + C85;
    const uint32_t W1 = __byte_perm(PL, PH, 0x7351u);
    L = __byte_perm(PL, 0u, 0x4341u);
    H = __byte_perm(PH, 0u, 0x4341u);
    PL = L * 85u + C85;
    PH = H * 85u + C85;
    const uint32_t W2 = __byte_perm(PL, PH, 0x7351u);
    L = __byte_perm(PL, 0u, 0x4341u);
    H = __byte_perm(PH, 0u, 0x4341u);
    PL = L * 85u + C85;
    PH = H * 85u + C85;
    const uint32_t W3 = __byte_perm(PL, PH, 0x7351u);
    const uint32_t W4 = ((W3 * 11u) >> 5) & 0x03030303u;
    D[0] = w - 3u * W1;
    D[1] = W1 - 3u * W2;
    D[2] = W2 - 3u * W3;
    D[3] = W3 - 3u * W4;
    D[4] = W4;
}

// ---- fp32 definitions shared by the decode-step kernels (fixed rounding order)

// exp: Cody & Waite argument reduction (x = n ln2 + r, ln2 split in a short
// high part and a low part) and the degree-7 Taylor polynomial of e^r in
// Horner form with fused multiply-adds, then exact scaling by 2^n (two
// power-of-two products below the normal range: one IEEE rounding).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ float exp32(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return __int_as_float(0x7f800000);
    if (x < -103.972084045410156f) return 0.0f;
    const float n = rintf(__fmul_rn(x, 1.44269502162933349609375f));
    float r = __fmaf_rn(-n, 0.693145751953125f, x);
    r = __fmaf_rn(-n, 1.4286068203094172321e-06f, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int e = static_cast<int>(n);
    if (e > 127) return __fmul_rn(__fmul_rn(p, pow2i(127)), 2.0f);
    if (e < -126) return __fmul_rn(__fmul_rn(p, pow2i(e + 64)), pow2i(-64));
    return __fmul_rn(p, pow2i(e));
}

// tanh(z) = 1 - 2/(e^{2z} + 1)
__device__ __forceinline__ float tanh32(float z) {
    const float e = exp32(__fmul_rn(2.0f, z));
    return __fsub_rn(1.0f, __fdiv_rn(2.0f, __fadd_rn(e, 1.0f)));
}

// GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
__device__ __forceinline__ float gelu32(float x) {
    const float x3 = __fmul_rn(__fmul_rn(x, x), x);
    const float inner = __fadd_rn(x, __fmul_rn(0.044715f, x3));
    const float z = __fmul_rn(0.7978845608028654f, inner);
    const float t = tanh32(z);
    return __fmul_rn(__fmul_rn(0.5f, x), __fadd_rn(1.0f, t));
}

// Symmetric absmax int8 code of v for step `scale`: clip(rint(v/scale), +-127).
__device__ __forceinline__ int quant_code(float v, float scale) {
    float r = rintf(__fdiv_rn(v, scale));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

// quant_code with the division replaced by a product with rinv = RN(1/scale),
// the same code for every v whose quotient is at most 127(1+2^-23) in
// magnitude (every element of the vector the scale was taken from).  With
// r = RN(1/s), y = RN(v r) = (v/s)(1+d1)(1+d2), |d1|,|d2| <= 2^-24, so
// |y - v/s| < 2^-15.9 for |v/s| <= 128, and f = RN(v/s) is within 2^-18 of
// v/s: |y - f| < 2^-15.  When y lies farther than 0.5 - 2^-14 from its
// nearest integer k, f is strictly within 0.5 of k and rint(f) = k; otherwise
// (and for NaN) the IEEE quotient decides.
__device__ __forceinline__ int quant_code_r(float v, float scale, float rinv) {
    const float y = __fmul_rn(v, rinv);
    float r = rintf(y);
    if (!(fabsf(__fsub_rn(y, r)) < 0.49993896484375f)) r = rintf(__fdiv_rn(v, scale));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

// Step of the absmax quantiser: max(absmax, 1e-9)/127.
__device__ __forceinline__ float quant_scale(float absmax) {
    return __fdiv_rn(fmaxf(absmax, 1e-9f), 127.0f);
}

// Pairwise sum across a warp of lane partials that are already the sums of
// consecutive, equally long segments: adjacent lanes first (xor 1, 2, ...),
// which is the balanced binary tree over the segments in order.
__device__ __forceinline__ float warp_psum(float v) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Pairwise tree over a power-of-two count of values in shared memory, in
// place: at stride st, s[2 st i] += s[2 st i + st] (adjacent subtrees first).
// All threads of the block must call it.
__device__ __forceinline__ float smem_psum_pow2(float *s, int count) {
    for (int st = 1; st < count; st <<= 1) {
        __syncthreads();
        for (int i = threadIdx.x; 2 * st * i < count; i += blockDim.x)
            s[2 * st * i] = __fadd_rn(s[2 * st * i], s[2 * st * i + st]);
    }
    __syncthreads();
    return s[0];
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

__host__ __device__ inline int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace qlin
