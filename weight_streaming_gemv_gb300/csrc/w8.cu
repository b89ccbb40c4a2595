// W8 linear layers: symmetric per-tensor int8 weights, fp32 activations,
// the scale applied once after the dot product (cpp20gemma README,
// "Architecture & implementation"; llama2.c "matmul" is the same loop over
// output rows).  Weights stream with 16-byte loads; each int8 is widened to
// fp32 exactly with the 2^23 magic-number trick (one byte permute and one
// subtraction) and accumulated with fp32 FMA.
#include <algorithm>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {

// ---------------------------------------------------------------- S1
__global__ void absmax_kernel(const float *__restrict__ w, int64_t n, unsigned int *__restrict__ out) {
    float a = 0.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        a = fmaxf(a, fabsf(w[i]));
    a = warp_max(a);
    if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(a));  // non-negative floats order as uints
}

__global__ void w8_quant_kernel(const float *__restrict__ w, int64_t N, int64_t K, int8_t *__restrict__ q,
                                int64_t pitch, const unsigned int *__restrict__ absmax_bits) {
    const float s = quant_scale(__uint_as_float(*absmax_bits));
    const int64_t total = N * pitch;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / pitch, k = i % pitch;
        q[i] = (k < K) ? (int8_t)quant_code(w[n * K + k], s) : (int8_t)0;
    }
}

__global__ void w8_scale_kernel(float *scale) {
    *scale = quant_scale(__uint_as_float(*reinterpret_cast<unsigned int *>(scale)));
}

// Group quantisation: one warp per (row n, group g) of G weights; the group's
// absmax, its step (the W8 rule) and codes; the row's bytes past K and the
// scale slots past ceil(K/G) are written zero.
__global__ void w8g_quant_kernel(const float *__restrict__ w, int64_t N, int64_t K, int G, int8_t *__restrict__ q,
                                 int64_t pitch, float *__restrict__ scales, int64_t s_pitch) {
    const int64_t ng = (K + G - 1) / G;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= N * s_pitch) return;
    const int64_t n = gw / s_pitch, g = gw % s_pitch;
    if (g >= ng) {
        if (lane == 0) scales[n * s_pitch + g] = 0.0f;
        return;
    }
    const int64_t k0 = g * G, k1 = min(K, k0 + G);
    float a = 0.0f;
    for (int64_t k = k0 + lane; k < k1; k += 32) a = fmaxf(a, fabsf(w[n * K + k]));
    a = warp_max(a);
    const float sc = quant_scale(a);
    for (int64_t k = k0 + lane; k < k1; k += 32) q[n * pitch + k] = (int8_t)quant_code(w[n * K + k], sc);
    if (g == ng - 1)
        for (int64_t k = K + lane; k < pitch; k += 32) q[n * pitch + k] = 0;
    if (lane == 0) scales[n * s_pitch + g] = sc;
}

// ---------------------------------------------------------------- S5 GEMV
// int8 byte j of a (bias-flipped) word -> exact fp32 value
__device__ __forceinline__ float i8_to_f32(uint32_t flipped, uint32_t sel) {
    return __fsub_rn(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel)), 8388736.0f);  // 2^23 + 128
}

// One warp handles R rows; lanes take 16-byte chunks c = lane + 32 j; the
// fp32 activations of a chunk are read from shared memory once and used for
// all R rows.  MT tokens per block.
// scales: null for one scale s of the whole tensor, else group scales
// [N][s_pitch], one per G weights of a row (G a multiple of 16, so a chunk of
// 16 weights lies in one group): each chunk's dot product takes its scale.
template <int R, int MT>
__global__ void __launch_bounds__(256) w8_gemv_kernel(const float *__restrict__ x, const int8_t *__restrict__ w,
                                                      int64_t pitch, float s, float *__restrict__ y, int M, int N,
                                                      int K, const float *__restrict__ scales, int64_t s_pitch, int G) {
    extern __shared__ float4 xs4[];  // [MT][C*4] float4
    const int C = (K + 15) / 16;
    const int m0 = blockIdx.y * MT;
    float *xsf = reinterpret_cast<float *>(xs4);
    for (int idx = threadIdx.x; idx < MT * C * 16; idx += blockDim.x) {
        const int mm = idx / (C * 16), k = idx % (C * 16), m = m0 + mm;
        xsf[idx] = (m < M && k < K) ? x[(int64_t)m * K + k] : 0.0f;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * warps;
    for (int64_t r0 = gwarp * R; r0 < N; r0 += nwarps * R) {
        float acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int mm = 0; mm < MT; mm++) acc[r][mm] = 0.0f;
        for (int c = lane; c < C; c += 32) {
            uint4 wv[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t row = r0 + r;
                wv[r] = (row < N) ? ld_stream_v4(w + row * pitch + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
            }
            float wf[R][16];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const uint32_t u[4] = {wv[r].x ^ 0x80808080u, wv[r].y ^ 0x80808080u, wv[r].z ^ 0x80808080u,
                                       wv[r].w ^ 0x80808080u};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    wf[r][4 * q + 0] = i8_to_f32(u[q], 0x7650u);
                    wf[r][4 * q + 1] = i8_to_f32(u[q], 0x7651u);
                    wf[r][4 * q + 2] = i8_to_f32(u[q], 0x7652u);
                    wf[r][4 * q + 3] = i8_to_f32(u[q], 0x7653u);
                }
            }
            float gs[R];  // the chunk's group scale per row (1 without groups)
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t row = r0 + r;
                gs[r] = (scales && row < N) ? __ldg(scales + row * s_pitch + (16 * c) / G) : 1.0f;
            }
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                const float4 *X = xs4 + ((size_t)mm * C + c) * 4;
                float cs[R];
#pragma unroll
                for (int r = 0; r < R; r++) cs[r] = scales ? 0.0f : acc[r][mm];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float4 xv = X[q];
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        float a = cs[r];
                        a = fmaf(xv.x, wf[r][4 * q + 0], a);
                        a = fmaf(xv.y, wf[r][4 * q + 1], a);
                        a = fmaf(xv.z, wf[r][4 * q + 2], a);
                        a = fmaf(xv.w, wf[r][4 * q + 3], a);
                        cs[r] = a;
                    }
                }
#pragma unroll
                for (int r = 0; r < R; r++) acc[r][mm] = scales ? fmaf(cs[r], gs[r], acc[r][mm]) : cs[r];
            }
        }
#pragma unroll
        for (int r = 0; r < R; r++) {
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                float v = acc[r][mm];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                acc[r][mm] = v;
            }
            const int64_t row = r0 + r;
            if (lane == 0 && row < N) {
#pragma unroll
                for (int mm = 0; mm < MT; mm++)
                    if (m0 + mm < M) y[(int64_t)(m0 + mm) * N + row] = acc[r][mm] * s;
            }
        }
    }
}

// ---------------------------------------------------------------- S5 GEMV, one token, TMA streaming
// One CTA per SM over a contiguous run of rows.  Lane 0 of warp 0 streams the
// run as tiles of TR whole rows (one bulk copy each: rows are contiguous)
// through a ring of S shared-memory slots (3 or 4: the count that keeps the
// more bytes in flight within half an SM's shared memory, for the row length;
// five slots of 22 KB measured slower than four);
// an mbarrier per slot counts
// the bytes in, another counts the consumer warps out.
//
// The consumers never widen a weight.  Each lane holds its slice of x (at most
// kW8JMax chunks of 16 elements) as 22-bit fixed point on a power-of-two
// scale taken from the slice's largest |x|, X = rint(x 2^(22-E)), split into
// three signed 8-bit limbs X = 2^16 a + 2^8 b + c; a row's dot product is then
// three dp4a per 4 weights into exact int32 sums A, B, C, and the lane's
// partial is (2^16 A + 2^8 B + C) 2^(E-22) in fp32.  x is thereby rounded to
// within 2^-23 of the slice's largest |x| (an fp32 value carries 2^-24 of
// itself).  A slice holding a NaN or an infinity makes its partial, and so
// the row, NaN.
//
// The eight consumer warps are KS K-parts x (8 / KS) row groups: warp w owns
// chunks [C p / KS, C (p+1) / KS) of the rows of group g (p = w % KS,
// g = w / KS; C = pitch / 16), two rows at a time.  After every tile the
// consumers meet at a named barrier and one warp adds the KS partials of each
// row in a fixed order, so the result does not depend on timing.
constexpr int kW8Warps = 8;    // consumer warps
constexpr int kW8MinStages = 3, kW8MaxStages = 4;  // slots of <= 32 KB within half an SM: two CTAs fit on an SM
constexpr int kW8JMax = 4;     // chunks per lane: C <= 32 * 8 * 4 (K <= 16384)
constexpr int kW8MaxTR = 32;   // rows per tile

struct W8Smem {
    int slot, tr, ks, xoff, total;  // slots at 0, then (at xoff) the ring and the partials
    int stages;                     // slots in the ring
    int sslot, soff;                // group scales: a slot of sslot bytes per stage at soff (0 without groups)
};

// s_pitch: floats per row of group scales (0: one scale for the tensor)
__host__ __device__ inline W8Smem w8_stream_layout_s(int64_t pitch, int smem_optin, int64_t s_pitch, int stages) {
    W8Smem L;
    L.stages = stages;
    const int C = (int)(pitch / 16);
    L.ks = 1;  // the fewest K parts that leave at most kW8JMax chunks per lane
    while (L.ks < kW8Warps && (C + L.ks * 32 - 1) / (L.ks * 32) > kW8JMax) L.ks *= 2;
    const int rstep = 2 * (kW8Warps / L.ks);  // a tile holds whole row pairs of every group
    const int fixed = (int)(sizeof(Ring<kW8MaxStages>) + 2 * kW8MaxTR * kW8Warps * sizeof(float)) + 256;
    // weight tiles of up to 32 KB, group scales (4 s_pitch bytes a row) beside
    // them, all within half the shared memory so that two CTAs fit on an SM
    const int budget = smem_optin / 2 - 1024 - fixed;
    int slot = budget / stages;
    slot = slot > 32768 ? 32768 : slot;
    slot = slot / 128 * 128;  // so that the rounded-up tile below stays within it
    int tr = (int)(slot / pitch);
    tr = tr > kW8MaxTR ? kW8MaxTR : tr;
    tr = tr / rstep * rstep;
    while (tr > 0 && stages * (((tr * pitch + 127) / 128 + (tr * 4 * s_pitch + 127) / 128) * 128) > budget)
        tr -= rstep;
    L.tr = tr;
    L.slot = (int)((tr * pitch + 127) / 128 * 128);
    L.sslot = (int)((tr * 4 * s_pitch + 127) / 128 * 128);
    L.soff = stages * L.slot;
    L.xoff = stages * (L.slot + L.sslot);
    L.total = L.xoff + fixed;
    if ((C + L.ks * 32 - 1) / (L.ks * 32) > kW8JMax) L.tr = 0;  // K too large for this kernel
    return L;
}

// The ring with the most bytes in flight (stages x slot) that holds at least
// one row per tile; ties go to fewer stages.
inline W8Smem w8_stream_layout(int64_t pitch, int smem_optin, int64_t s_pitch = 0) {
    W8Smem best = w8_stream_layout_s(pitch, smem_optin, s_pitch, kW8MinStages);
    for (int st = kW8MinStages + 1; st <= kW8MaxStages; st++) {
        const W8Smem L = w8_stream_layout_s(pitch, smem_optin, s_pitch, st);
        if (L.tr >= 1 && (best.tr < 1 || (int64_t)st * L.slot > (int64_t)best.stages * best.slot)) best = L;
    }
    return best;
}

// 2^e for -126 <= e <= 127
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// GROUPED: group scales `scales` [N][s_pitch], one per G weights of a row;
// otherwise one scale s of the whole tensor (scales unused)
template <bool GROUPED, int S>
__global__ void __launch_bounds__(32 * (kW8Warps + 1), 2) w8_stream_kernel(const float *__restrict__ x,
                                                                         const int8_t *__restrict__ w, int64_t pitch,
                                                                         float s, float *__restrict__ y, int N, int K,
                                                                         W8Smem L, const float *__restrict__ scales,
                                                                         int64_t s_pitch, int G) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *slots = smem;
    Ring<S> *ring = reinterpret_cast<Ring<S> *>(smem + L.xoff);  // within the fixed part sized for kW8MaxStages
    float *part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ring) + sizeof(Ring<S>));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = (int)(pitch / 16), TR = L.tr, KS = L.ks;
    const int64_t r0 = (int64_t)N * blockIdx.x / gridDim.x, r1 = (int64_t)N * (blockIdx.x + 1) / gridDim.x;
    const int ntiles = (int)((r1 - r0 + TR - 1) / TR);
    // Programmatic dependent launch: the next kernel on the stream may start its
    // own set-up now.  The weights (and group scales) are read-only inputs, so
    // the first tile of their stream goes out before this kernel waits for the
    // previous one to complete (and its writes to be visible); x is read and y
    // written after the wait.  The other stages go out after the x loads, so
    // that those few loads do not queue behind the stream (issuing all of
    // them first measured 6% slower).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t pol = l2_evict_first();
    auto issue = [&](int t) {
        const int st = t % S;
        const int64_t row = r0 + (int64_t)t * TR;
        const int64_t nr = min((int64_t)TR, r1 - row);
        const uint32_t bytes = (uint32_t)(nr * pitch), sbytes = GROUPED ? (uint32_t)(nr * 4 * s_pitch) : 0u;
        mbar_arrive_expect_tx(&ring->full[st], bytes + sbytes);
        bulk_g2s(slots + (size_t)st * L.slot, w + row * pitch, bytes, &ring->full[st], pol);
        if (GROUPED) bulk_g2s(slots + L.soff + (size_t)st * L.sslot, scales + row * s_pitch, sbytes, &ring->full[st], pol);
    };
    if (threadIdx.x == 0) {
        ring->init(kW8Warps);
        if (ntiles > 0) issue(0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // consumers: this lane's x slice
    const int cw = warp - 1, p = cw % KS, grp = cw / KS;
    const int ca = C * p / KS, cb = C * (p + 1) / KS;
    // the slice straight from global memory, every load in flight at once (16-byte
    // loads when x is 16-byte aligned; a 16-byte group that crosses K element by element)
    float xv[kW8JMax][16];
    if (warp > 0) {
        const bool x16 = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
#pragma unroll
        for (int j = 0; j < kW8JMax; j++) {
            const int c = ca + lane + 32 * j;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int k0 = 16 * c + 4 * q;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c < cb) {
                    if (x16 && k0 + 3 < K) {
                        v = __ldg(reinterpret_cast<const float4 *>(x + k0));
                    } else {
                        if (k0 < K) v.x = __ldg(x + k0);
                        if (k0 + 1 < K) v.y = __ldg(x + k0 + 1);
                        if (k0 + 2 < K) v.z = __ldg(x + k0 + 2);
                        if (k0 + 3 < K) v.w = __ldg(x + k0 + 3);
                    }
                }
                xv[j][4 * q] = v.x;
                xv[j][4 * q + 1] = v.y;
                xv[j][4 * q + 2] = v.z;
                xv[j][4 * q + 3] = v.w;
            }
        }
    }
    // the loads are in flight; one barrier (the ring is initialised), then the rest of the stream
    __syncthreads();
    if (threadIdx.x == 0)
        for (int t = 1; t < min(ntiles, S); t++) issue(t);

    if (warp == 0) {
        if (lane != 0) return;
        int t = min(ntiles, S);
        for (; t < ntiles; t++) {
            if (!mbar_wait(&ring->empty[t % S], ((t / S) - 1) & 1)) break;
            issue(t);
        }
        // every copy issued must have landed before the CTA leaves
        for (int u = max(0, t - S); u < t; u++) mbar_wait(&ring->full[u % S], (u / S) & 1);
        return;
    }

    // consumers: this lane's x chunks as three limbs of 22-bit fixed point
    // largest |x| of the slice and finiteness from one integer maximum of the magnitude bits
    uint32_t mbits = 0;
#pragma unroll
    for (int j = 0; j < kW8JMax; j++)
#pragma unroll
        for (int e = 0; e < 16; e++) mbits = max(mbits, (uint32_t)__float_as_int(xv[j][e]) & 0x7fffffffu);
    const bool finite = mbits < 0x7f800000u;
    // amax < 2^E (E from the exponent bits; frexp for a subnormal amax)
    int E = 0;
    if (mbits != 0 && finite) {
        const int eb = (int)(mbits >> 23);
        if (eb != 0)
            E = eb - 126;
        else
            frexpf(__int_as_float((int)mbits), &E);
    }
    // X = rint(v 2^(22-E)) with two exact power-of-two factors (the second
    // one only matters for slices below 2^-78); |X| <= 2^22, so adding
    // 1.5 * 2^23 rounds to the integer (ties to even) and leaves it in the
    // low mantissa bits.  Y = X + 0x808080 has bytes c_i + 128 for the
    // balanced base-256 digits X = 2^16 c2 + 2^8 c1 + c0 (c_i in -128..127),
    // so each limb word is four bytes of Y with the top bit flipped.
    const int sh = 22 - E;
    const float p1 = pow2f(sh > 100 ? 100 : sh), p2 = pow2f(sh > 100 ? sh - 100 : 0);
    uint32_t la[kW8JMax][4], lb[kW8JMax][4], lc[kW8JMax][4];
#pragma unroll
    for (int j = 0; j < kW8JMax; j++) {
        const int c = ca + lane + 32 * j;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t Y[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float v = (finite && c < cb) ? xv[j][4 * q + e] : 0.0f;
                const float r = __fadd_rn(__fmul_rn(__fmul_rn(v, p1), p2), 12582912.0f);
                Y[e] = (uint32_t)__float_as_int(r) - (0x4B400000u - 0x808080u);
            }
            const uint32_t lo = __byte_perm(Y[0], Y[1], 0x5140u), hi = __byte_perm(Y[2], Y[3], 0x5140u);
            // lo = [Y0.b0, Y1.b0, Y0.b1, Y1.b1], hi likewise for Y2, Y3
            lc[j][q] = __byte_perm(lo, hi, 0x5410u) ^ 0x80808080u;
            lb[j][q] = __byte_perm(lo, hi, 0x7632u) ^ 0x80808080u;
            la[j][q] = __byte_perm(__byte_perm(Y[0], Y[1], 0x0062u), __byte_perm(Y[2], Y[3], 0x0062u), 0x5410u) ^
                       0x80808080u;
        }
    }
    if (!finite) E = 0;
    const int ush = E - 22;  // partial = (2^16 A + 2^8 B + C) 2^(E-22), in two exact steps
    const float s1 = pow2f(ush < -100 ? -100 : ush), s2 = pow2f(ush < -100 ? ush + 100 : 0);
    const float nanv = finite ? 0.0f : __int_as_float(0x7fc00000);  // a non-finite slice poisons its partials
    const int gsz = TR / (kW8Warps / KS);  // rows of a group in a full tile (even)

    bool ok = true;
    for (int t = 0; t < ntiles; t++) {
        const int st = t % S;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(&ring->full[st], (t / S) & 1))) ok = false;
        const int64_t row0 = r0 + (int64_t)t * TR;
        const int rows = (int)min((int64_t)TR, r1 - row0);
        float *pt = part + (size_t)(t & 1) * kW8MaxTR * kW8Warps;
        if (ok) {
            const uint8_t *tile = slots + (size_t)st * L.slot;
            const float *stile = reinterpret_cast<const float *>(slots + L.soff + (size_t)st * L.sslot);
            const int g0 = grp * gsz, g1 = min(rows, g0 + gsz);
            for (int r = g0; r < g1; r += 2) {
                const bool two = r + 1 < g1;
                const uint8_t *ra = tile + (size_t)r * pitch, *rb = ra + pitch;
                int Aa = 0, Ba = 0, Ca = 0, Ab = 0, Bb = 0, Cb = 0;
                float ga = 0.0f, gb = 0.0f;  // with group scales: sum of the chunks' scaled sums
#pragma unroll
                for (int j = 0; j < kW8JMax; j++) {
                    const int c = ca + lane + 32 * j;
                    if (c < cb) {
                        if (GROUPED) Aa = Ba = Ca = Ab = Bb = Cb = 0;
                        const uint4 wa = lds128(ra + (size_t)c * 16);
                        const uint4 wb = two ? lds128(rb + (size_t)c * 16) : make_uint4(0u, 0u, 0u, 0u);
                        const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w}, ub[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            Aa = dp4a(ua[q], la[j][q], Aa);
                            Ba = dp4a(ua[q], lb[j][q], Ba);
                            Ca = dp4a(ua[q], lc[j][q], Ca);
                            Ab = dp4a(ub[q], la[j][q], Ab);
                            Bb = dp4a(ub[q], lb[j][q], Bb);
                            Cb = dp4a(ub[q], lc[j][q], Cb);
                        }
                        if (GROUPED && 16 * c < K) {  // the chunk lies in group 16 c / G (G a multiple of 16)
                            const int gi = (16 * c) / G;
                            ga = fmaf(fmaf((float)Aa, 65536.0f, fmaf((float)Ba, 256.0f, (float)Ca)),
                                      stile[(size_t)r * s_pitch + gi], ga);
                            if (two)
                                gb = fmaf(fmaf((float)Ab, 65536.0f, fmaf((float)Bb, 256.0f, (float)Cb)),
                                          stile[(size_t)(r + 1) * s_pitch + gi], gb);
                        }
                    }
                }
                if (!GROUPED) {
                    ga = fmaf((float)Aa, 65536.0f, fmaf((float)Ba, 256.0f, (float)Ca));
                    gb = fmaf((float)Ab, 65536.0f, fmaf((float)Bb, 256.0f, (float)Cb));
                }
                float fa = __fmul_rn(__fmul_rn(ga, s1), s2);
                float fb = __fmul_rn(__fmul_rn(gb, s1), s2);
                fa = __fadd_rn(fa, nanv);
                fb = __fadd_rn(fb, nanv);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    fa += __shfl_xor_sync(0xffffffffu, fa, o);
                    fb += __shfl_xor_sync(0xffffffffu, fb, o);
                }
                if (lane == 0) {
                    pt[r * kW8Warps + p] = fa;
                    if (two) pt[(r + 1) * kW8Warps + p] = fb;
                }
            }
        }
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&ring->empty[st]);
        // all partials of tile t are in: one warp adds them (the other buffer
        // takes tile t+1 meanwhile)
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kW8Warps) : "memory");
        if (cw == t % kW8Warps && lane < rows) {
            float v = pt[lane * kW8Warps];
            for (int q = 1; q < KS; q++) v += pt[lane * kW8Warps + q];
            y[row0 + lane] = ok ? v * s : __int_as_float(0x7fc00000);
        }
    }
}

// the tensor-core paths for 2 <= M <= 64 (w8_tc.cu): activations split in
// the product kernel, or once per call into a workspace
qlin_status w8_linear_tensor_cores(const float *x, const int8_t *w8, int64_t pitch, float s, float *y, int M, int N,
                                   int K, cudaStream_t st);
size_t w8_tc_workspace_bytes(int M, int K);
qlin_status w8_linear_tensor_cores_ws(const float *x, const int8_t *w8, int64_t pitch, float s, float *y, int M,
                                      int N, int K, void *work, cudaStream_t st);

// The one-token stream kernel for layout L (its ring depth picks the
// instantiation), launched with programmatic stream serialisation.
template <bool GROUPED, int S>
static qlin_status launch_stream_s(const float *x, const int8_t *w, int64_t pitch, float s, float *y, int N, int K,
                                   const W8Smem &L, const float *scales, int64_t s_pitch, int G, cudaStream_t st) {
    const int per_sm = blocks_per_sm((const void *)w8_stream_kernel<GROUPED, S>, L.total);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sm_count() * std::min(per_sm, 2)));
    cfg.blockDim = dim3(32 * (kW8Warps + 1));
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, w8_stream_kernel<GROUPED, S>, x, w, pitch, s, y, N, K, L, scales, s_pitch, G));
    QLIN_LAUNCHED("w8_stream_kernel");
    return QLIN_OK;
}
template <bool GROUPED>
static qlin_status launch_stream(const float *x, const int8_t *w, int64_t pitch, float s, float *y, int N, int K,
                                 const W8Smem &L, const float *scales, int64_t s_pitch, int G, cudaStream_t st) {
    static_assert(kW8MinStages == 3 && kW8MaxStages == 4, "instantiations");
    if (L.stages == 4) return launch_stream_s<GROUPED, 4>(x, w, pitch, s, y, N, K, L, scales, s_pitch, G, st);
    return launch_stream_s<GROUPED, 3>(x, w, pitch, s, y, N, K, L, scales, s_pitch, G, st);
}

template <int R, int MT>
static qlin_status launch_w8(const float *x, const int8_t *w, int64_t pitch, float s, float *y, int M, int N, int K,
                             cudaStream_t st, const float *scales = nullptr, int64_t s_pitch = 0, int G = 0) {
    auto kern = w8_gemv_kernel<R, MT>;
    const int C = (K + 15) / 16;
    const size_t smem = (size_t)MT * C * 16 * sizeof(float);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_w8_f32: M tile x K=%d needs %zu B smem", K,
                 smem);
    const int per_sm = blocks_per_sm((const void *)kern, smem);
    const int64_t warps_needed = (N + R - 1) / R;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (blocks > cap) blocks = cap;
    dim3 grid((unsigned)blocks, (unsigned)((M + MT - 1) / MT));
    kern<<<grid, 256, smem, st>>>(x, w, pitch, s, y, M, N, K, scales, s_pitch, G);
    QLIN_LAUNCHED("w8_gemv_kernel");
    return QLIN_OK;
}

}  // namespace qlin

extern "C" {

qlin_status qlin_w8_quantize(const float *w, int64_t N, int64_t K, int8_t *w8, int64_t w_pitch, float *scale,
                             qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(w && w8 && scale, QLIN_ERR_INVALID_ARG, "qlin_w8_quantize: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1 && w_pitch >= K && w_pitch % 16 == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_w8_quantize: N=%lld K=%lld w_pitch=%lld", (long long)N, (long long)K, (long long)w_pitch);
    QLIN_REQUIRE(qlin::aligned4(w) && qlin::aligned16(w8) && qlin::aligned4(scale), QLIN_ERR_INVALID_ARG,
                 "qlin_w8_quantize: misaligned pointer");
    cudaStream_t st = (cudaStream_t)stream;
    QLIN_CUDA(cudaMemsetAsync(scale, 0, sizeof(float), st));
    const int blocks = qlin::sm_count() * 4;
    qlin::absmax_kernel<<<blocks, 256, 0, st>>>(w, N * K, reinterpret_cast<unsigned int *>(scale));
    QLIN_LAUNCHED("absmax_kernel");
    qlin::w8_quant_kernel<<<blocks, 256, 0, st>>>(w, N, K, w8, w_pitch, reinterpret_cast<unsigned int *>(scale));
    QLIN_LAUNCHED("w8_quant_kernel");
    qlin::w8_scale_kernel<<<1, 1, 0, st>>>(scale);
    QLIN_LAUNCHED("w8_scale_kernel");
    return QLIN_OK;
}

qlin_status qlin_w8_f32(const float *x, const int8_t *w8, int64_t w_pitch, float w_scale, float *y, int M, int N,
                        int K, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(x && w8 && y, QLIN_ERR_INVALID_ARG, "qlin_w8_f32: null pointer");
    QLIN_REQUIRE(M >= 1 && N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_w8_f32: M=%d N=%d K=%d", M, N, K);
    QLIN_REQUIRE(w_pitch >= K && w_pitch % 16 == 0, QLIN_ERR_INVALID_ARG, "qlin_w8_f32: w_pitch %lld",
                 (long long)w_pitch);
    QLIN_REQUIRE(qlin::aligned16(w8) && qlin::aligned4(x) && qlin::aligned4(y), QLIN_ERR_INVALID_ARG,
                 "qlin_w8_f32: misaligned pointer");
    QLIN_REQUIRE(M <= 64, QLIN_ERR_UNSUPPORTED, "qlin_w8_f32: M=%d > 64", M);
    cudaStream_t st = (cudaStream_t)stream;
    if (M == 1 && w_pitch <= 16 * 32 * qlin::kW8Warps * qlin::kW8JMax) {
        const qlin::W8Smem L = qlin::w8_stream_layout(w_pitch, qlin::max_smem_optin());
        if (L.tr >= 1)
            return qlin::launch_stream<false>(x, w8, w_pitch, w_scale, y, N, K, L, (const float *)nullptr, (int64_t)0, 0,
                                              st);
    }
    if (M == 1) return qlin::launch_w8<4, 1>(x, w8, w_pitch, w_scale, y, M, N, K, st);
    return qlin::w8_linear_tensor_cores(x, w8, w_pitch, w_scale, y, M, N, K, st);
}

size_t qlin_w8_f32_workspace_size(int M, int K) { return qlin::w8_tc_workspace_bytes(M, K); }

qlin_status qlin_w8_f32_ws(const float *x, const int8_t *w8, int64_t w_pitch, float w_scale, float *y, int M, int N,
                           int K, void *workspace, size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(x && w8 && y, QLIN_ERR_INVALID_ARG, "qlin_w8_f32_ws: null pointer");
    QLIN_REQUIRE(M >= 1 && N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_w8_f32_ws: M=%d N=%d K=%d", M, N, K);
    QLIN_REQUIRE(w_pitch >= K && w_pitch % 16 == 0, QLIN_ERR_INVALID_ARG, "qlin_w8_f32_ws: w_pitch %lld",
                 (long long)w_pitch);
    QLIN_REQUIRE(qlin::aligned16(w8) && qlin::aligned4(x) && qlin::aligned4(y), QLIN_ERR_INVALID_ARG,
                 "qlin_w8_f32_ws: misaligned pointer");
    QLIN_REQUIRE(M <= 64, QLIN_ERR_UNSUPPORTED, "qlin_w8_f32_ws: M=%d > 64", M);
    if (M == 1) return qlin_w8_f32(x, w8, w_pitch, w_scale, y, M, N, K, stream);
    const size_t need = qlin::w8_tc_workspace_bytes(M, K);
    QLIN_REQUIRE(workspace_bytes >= need && workspace && qlin::aligned16(workspace), QLIN_ERR_INVALID_ARG,
                 "qlin_w8_f32_ws: workspace %zu < %zu bytes, null or not 16-byte aligned", workspace_bytes, need);
    return qlin::w8_linear_tensor_cores_ws(x, w8, w_pitch, w_scale, y, M, N, K, workspace, (cudaStream_t)stream);
}

qlin_status qlin_w8g_quantize(const float *w, int64_t N, int64_t K, int G, int8_t *w8, int64_t w_pitch, float *scales,
                              int64_t s_pitch, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(w && w8 && scales, QLIN_ERR_INVALID_ARG, "qlin_w8g_quantize: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1 && G >= 16 && G % 16 == 0 && w_pitch >= K && w_pitch % 16 == 0 &&
                     s_pitch >= (K + G - 1) / G && s_pitch % 4 == 0,
                 QLIN_ERR_INVALID_ARG, "qlin_w8g_quantize: N=%lld K=%lld G=%d w_pitch=%lld s_pitch=%lld", (long long)N,
                 (long long)K, G, (long long)w_pitch, (long long)s_pitch);
    QLIN_REQUIRE(qlin::aligned4(w) && qlin::aligned16(w8) && qlin::aligned16(scales), QLIN_ERR_INVALID_ARG,
                 "qlin_w8g_quantize: misaligned pointer");
    const int64_t warps = N * s_pitch;
    const int64_t blocks = (warps * 32 + 255) / 256;
    QLIN_REQUIRE(blocks < ((int64_t)1 << 31), QLIN_ERR_UNSUPPORTED, "qlin_w8g_quantize: too many groups");
    qlin::w8g_quant_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(w, N, K, G, w8, w_pitch, scales,
                                                                               s_pitch);
    QLIN_LAUNCHED("w8g_quant_kernel");
    return QLIN_OK;
}

qlin_status qlin_w8g_f32(const float *x, const int8_t *w8, int64_t w_pitch, const float *scales, int64_t s_pitch, int G,
                         float *y, int M, int N, int K, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(x && w8 && scales && y, QLIN_ERR_INVALID_ARG, "qlin_w8g_f32: null pointer");
    QLIN_REQUIRE(M >= 1 && N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_w8g_f32: M=%d N=%d K=%d", M, N, K);
    QLIN_REQUIRE(G >= 16 && G % 16 == 0 && w_pitch >= K && w_pitch % 16 == 0 && s_pitch >= (K + G - 1) / G &&
                     s_pitch % 4 == 0,
                 QLIN_ERR_INVALID_ARG, "qlin_w8g_f32: G=%d w_pitch=%lld s_pitch=%lld", G, (long long)w_pitch,
                 (long long)s_pitch);
    QLIN_REQUIRE(qlin::aligned16(w8) && qlin::aligned16(scales) && qlin::aligned4(x) && qlin::aligned4(y),
                 QLIN_ERR_INVALID_ARG, "qlin_w8g_f32: misaligned pointer");
    QLIN_REQUIRE(M <= 64, QLIN_ERR_UNSUPPORTED, "qlin_w8g_f32: M=%d > 64", M);
    cudaStream_t st = (cudaStream_t)stream;
    if (M == 1 && w_pitch <= 16 * 32 * qlin::kW8Warps * qlin::kW8JMax) {
        const qlin::W8Smem L = qlin::w8_stream_layout(w_pitch, qlin::max_smem_optin(), s_pitch);
        if (L.tr >= 1) return qlin::launch_stream<true>(x, w8, w_pitch, 1.0f, y, N, K, L, scales, s_pitch, G, st);
    }
    const size_t tile8_smem = (size_t)8 * ((K + 15) / 16) * 16 * sizeof(float);
    if (M == 1) return qlin::launch_w8<4, 1>(x, w8, w_pitch, 1.0f, y, M, N, K, st, scales, s_pitch, G);
    if (M <= 4 || (int)tile8_smem > qlin::max_smem_optin())
        return qlin::launch_w8<2, 4>(x, w8, w_pitch, 1.0f, y, M, N, K, st, scales, s_pitch, G);
    return qlin::launch_w8<2, 8>(x, w8, w_pitch, 1.0f, y, M, N, K, st, scales, s_pitch, G);
}

}  // extern "C"
