// T158 linear for many tokens (prefill, batched decode) on the fifth-generation
// tensor cores.
//
// All tokens go through each weight matrix in one pass (citric, "Step 1: a
// kernel for 1.6-bit weights": batched prompt processing).  The integer dot
// products of that step run as an fp16 matrix product with fp32 accumulation,
// which is exact here: int8 codes (|x| <= 127) and trits are fp16 integers,
// every product is an integer of magnitude <= 127 and every partial sum stays
// below 127 K < 2^24, so each fp32 addition is exact and the accumulator
// equals the int32 sum.
//
// One CTA computes 128 weight rows x T tokens (T a multiple of 32, at most
// 128, so that two CTAs share an SM's tensor memory and one's output write
// overlaps the other's products) with tcgen05.mma (M = 128 weight rows, N = T tokens, K = 16 per
// instruction) into T fp32 accumulator columns of tensor memory.  K advances in
// steps of 80 elements: 16 packed bytes of every weight row.  Within a step
// both operands use the same permuted K order, K' = 16 i + j for element
// 5 j + i (digit i of packed byte j), which leaves the dot product unchanged
// and lets the trits come straight out of the digit-plane decode.
//
// The weight tile is the MMA's A operand and sits in tensor memory: eight
// converter warps decode the packed bytes (warp w: rows 32 (w % 4) .. + 31,
// half w / 4 of the step's 16 bytes) and write the fp16 trits with tcgen05.st
// into the lanes of their own rows, so decoded weights never pass through
// shared memory.  The activation tile is the B operand, in shared memory in
// the no-swizzle K-major layout of the MMA (8-row x 16-byte core matrices, 128
// bytes apart along K, kTcSBO bytes between 8-row groups), reached one of two
// ways:
//  - with a workspace, t158_act_tiles_kernel converts every token row once per
//    call into the exact image of each step's tile, and a copy warp brings a
//    step's tile in with one bulk copy (the conversion is not repeated for
//    every 128 weight rows);
//  - without one, the converter warps also convert the step's int8 rows, two
//    units of work per row (bytes 0..47 and 32..79 of the step: the first and
//    second eight packed-byte columns).
// Raw bytes run a few steps ahead through cp.async; several operand stages let
// the conversion of later steps overlap the MMAs of earlier ones; one thread
// issues each step's five MMAs and commits them to the stage's mbarrier.  The
// epilogue reads the accumulator back with tcgen05.ld: a thread holds one
// weight row for 16 tokens at a time and its warp writes 32 consecutive
// outputs of each token.  Split K: a cluster of CTAs over one tile, each over
// its own K steps, adds the partial tiles through distributed shared memory in
// rank order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "common.cuh"
#include "decode_ops.cuh"
#include "stream.cuh"
#include "tcgen05.cuh"

namespace qlin {

constexpr int kTmRows = 128;              // weight rows per CTA (MMA M, tensor-memory lanes)
constexpr int kTmMaxTok = 128;            // tokens per CTA at most (MMA N)
constexpr int kTcKS = 80;                 // K elements per step (16 packed bytes)
constexpr int kTcChunks = kTcKS / 8;      // 16-byte core-matrix columns per row and step
constexpr int kTcSBO = kTcChunks * 128;   // bytes between 8-row groups of the activation tile
constexpr int kTmConv = 256;              // converter threads (8 warps)
constexpr int kTmThreads = kTmConv + 64;  // + the warp that issues the MMAs + the warp that copies activation tiles
constexpr int kTmMaxStages = 4;
constexpr int kTmACols = kTcKS / 2;       // tensor-memory columns of one step's weight tile (fp16 pairs)
constexpr int kTmUnit = 48;               // raw bytes of one activation unit (three 16-byte copies)
constexpr int kTmCtl = 2048;              // bytes of the control block at the start of shared memory
constexpr int kTmPStride = kTmRows + 4;   // floats per token of a partial tile (split K)
constexpr int kTmMaxSplit = 8;            // CTAs of a cluster that split K
constexpr int kTmEarlyMaxItems = 16384;   // tile-conversion work items (token rows x steps) behind which the product starts early

// Two ways to the activation tile.  PRE: converted once per call by
// t158_act_tiles_kernel into a workspace, one bulk copy per stage; else
// converted by the converter warps from the int8 codes at every step.
// Stages (operand tiles) and raw stages (copies ahead) of each:
__host__ __device__ constexpr int tm_stages(bool) { return 3; }
__host__ __device__ constexpr int tm_raws(bool pre) { return pre ? 4 : 3; }

struct TmCtl {
    uint64_t full[kTmMaxStages];      // the stage is filled (converter arrivals, + the copy with PRE)
    uint64_t mma_done[kTmMaxStages];  // the MMAs reading the stage are done (tcgen05.commit)
    float xs[kTmMaxTok];              // activation scales of the tile's tokens
    uint32_t tmem;
    int abort;
    int issued;  // steps whose MMAs were issued
};
static_assert(sizeof(TmCtl) <= kTmCtl, "control block");

// Dynamic shared memory for T tokens: control block, the activation tiles of
// the stages, raw activation stages (2 T units; in-kernel conversion only),
// raw weight stages (8 bytes per converter); after the K loop the partial
// tile (split K) reuses the space behind the control block.
__host__ __device__ constexpr int tm_b_bytes(int T) { return T / 8 * kTcSBO; }
__host__ __device__ constexpr int tm_raw_a_off(int T, bool pre) { return kTmCtl + tm_stages(pre) * tm_b_bytes(T); }
__host__ __device__ constexpr int tm_raw_w_off(int T, bool pre) {
    return tm_raw_a_off(T, pre) + (pre ? 0 : tm_raws(pre) * 2 * T * kTmUnit);
}
__host__ __device__ constexpr int tm_smem_bytes(int T, bool pre) {
    return tm_raw_w_off(T, pre) + tm_raws(pre) * kTmConv * 8 > kTmCtl + T * kTmPStride * 4
               ? tm_raw_w_off(T, pre) + tm_raws(pre) * kTmConv * 8
               : kTmCtl + T * kTmPStride * 4;
}
// Tensor-memory columns: T accumulator columns, then the stages' weight
// tiles; a power of two from 32 (the allocation unit).
__host__ __device__ inline uint32_t tm_cols(int T, bool pre) {
    uint32_t c = 32;
    while ((int)c < T + tm_stages(pre) * kTmACols) c <<= 1;
    return c;
}
static_assert(tm_smem_bytes(kTmMaxTok, false) <= 227 * 1024 && tm_smem_bytes(kTmMaxTok, true) <= 227 * 1024,
              "shared memory of the largest tile");

// Shared-memory matrix descriptor of the MMA: K-major, no swizzle, leading
// byte offset 128 (next core matrix along K), stride byte offset kTcSBO (next
// 8-row group), descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(((uint32_t)kTcSBO >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = T tokens, M = kTmRows weight rows.
__device__ __forceinline__ uint32_t tm_idesc(int T) {
    return (1u << 4) | ((uint32_t)(T >> 3) << 17) | ((uint32_t)(kTmRows >> 4) << 24);
}






// Byte offset of 16-byte chunk kc of row r in an activation tile.
__device__ __forceinline__ int tc_off(int r, int kc) { return (r >> 3) * kTcSBO + kc * 128 + (r & 7) * 16; }

// Two int8 bytes (already xor 0x80, i.e. v + 128) -> fp16x2 of the two values:
// fp16 (1024 + u) has the bits 0x6400 | u, less 1152 gives v exactly.
__device__ __forceinline__ uint32_t i8pair_bits(uint32_t w0, uint32_t w1, int b0, int b1) {
    // [w0.b0, w1.b1, -, -] then [., 0x64, ., 0x64]
    const uint32_t t = __byte_perm(w0, w1, (uint32_t)b0 | ((uint32_t)(4 + b1) << 4));
    return __byte_perm(t, 0x6464u, 0x5140u);
}

__device__ __forceinline__ uint32_t h2sub(uint32_t bits, uint32_t cbits) {
    __half2 a = *reinterpret_cast<__half2 *>(&bits), c = *reinterpret_cast<__half2 *>(&cbits);
    __half2 r = __hsub2(a, c);
    return *reinterpret_cast<uint32_t *>(&r);
}

// Activation unit H of token row r: in[] holds bytes 32 H .. 32 H + 47 of the
// step (v + 128 for each value v); it fills chunks kc = 2 i + H (K' 16 i + 8 H
// .. + 7, i.e. packed-byte columns j = 8 H .. 8 H + 7 of digit i) of row r.
template <int H>
__device__ __forceinline__ void tm_put_act(uint8_t *tile, const uint32_t (&in)[12], int r) {
#pragma unroll
    for (int i = 0; i < 5; i++) {
        uint32_t h[4];
#pragma unroll
        for (int p = 0; p < 4; p++) {
            // K' = 16 i + 8 H + 2 p is element 5 (8 H + 2 p) + i, byte 8 H + 10 p + i of the unit
            const int e0 = 8 * H + 10 * p + i, e1 = e0 + 5;
            h[p] = h2sub(i8pair_bits(in[e0 >> 2], in[e1 >> 2], e0 & 3, e1 & 3), 0x64806480u);
        }
        *reinterpret_cast<uint4 *>(tile + tc_off(r, 2 * i + H)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// Eight packed bytes (v.x, v.y: packed-byte columns 8 hw .. 8 hw + 7 of the
// step) of this thread's weight row -> fp16 trits into its tensor-memory lane:
// chunk kc = 2 i + hw is the four columns 4 kc .. 4 kc + 3 from `ta`.
__device__ __forceinline__ void tm_put_w(uint32_t ta, uint2 v, int hw) {
    uint32_t D0[5], D1[5];
    t158_planes(v.x, D0);
    t158_planes(v.y, D1);
#pragma unroll
    for (int i = 0; i < 5; i++) {
        // digits d in 0..2: fp16 (1024 + d) - 1025 = d - 1
        const uint32_t h0 = h2sub(__byte_perm(D0[i], 0x6464u, 0x5140u), 0x64016401u);
        const uint32_t h1 = h2sub(__byte_perm(D0[i], 0x6464u, 0x5342u), 0x64016401u);
        const uint32_t h2 = h2sub(__byte_perm(D1[i], 0x6464u, 0x5140u), 0x64016401u);
        const uint32_t h3 = h2sub(__byte_perm(D1[i], 0x6464u, 0x5342u), 0x64016401u);
        tm_st4(ta + (uint32_t)(4 * (2 * i + hw)), h0, h1, h2, h3);
    }
}

// 1-D bulk copy global -> shared completing on `bar`; bytes and both addresses
// multiples of 16.
__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Unit h of token m at step s loaded directly (any alignment; zero past K and
// for m >= M), as bytes v + 128.
__device__ __forceinline__ void tm_load_act(uint32_t (&in)[12], const int8_t *__restrict__ xq, int M, int K, int m,
                                            int s, int h) {
    const int k0 = s * kTcKS + 32 * h;
#pragma unroll
    for (int i = 0; i < 12; i++) {
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int k = k0 + 4 * i + b;
            const uint32_t byte = (m < M && k < K) ? (uint32_t)(uint8_t)xq[(int64_t)m * K + k] : 0u;
            v |= byte << (8 * b);
        }
        in[i] = v ^ 0x80808080u;
    }
}


// One token row of one step into an activation tile: in[] holds the 80 bytes
// (v + 128 for each value v); chunk kc of row r is K' 8 kc .. 8 kc + 7.
__device__ __forceinline__ void tm_put_row(uint8_t *tile, const uint32_t (&in)[20], int r) {
#pragma unroll
    for (int kc = 0; kc < kTcChunks; kc++) {
        uint32_t h[4];
#pragma unroll
        for (int p = 0; p < 4; p++) {
            const int kp = 8 * kc + 2 * p;          // K' of the low half
            const int e0 = 5 * (kp & 15) + (kp >> 4), e1 = e0 + 5;  // elements 5 j + i
            h[p] = h2sub(i8pair_bits(in[e0 >> 2], in[e1 >> 2], e0 & 3, e1 & 3), 0x64806480u);
        }
        *reinterpret_cast<uint4 *>(tile + tc_off(r, kc)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// Activation tiles for the PRE path, converted once per call: the image of
// the shared-memory activation tile of token tile tt at step s (tokens
// tt T .. + T - 1, elements 80 s .. + 79, zero past M and K) at
// out + (tt nsteps + s) tm_b_bytes(T).  One thread per token row and step;
// a warp's 32 rows make 4 runs of 128 contiguous bytes per store.
__global__ void __launch_bounds__(256) t158_act_tiles_kernel(const int8_t *__restrict__ xq, int M, int K, int T,
                                                             int tiles_m, int nsteps, uint8_t *__restrict__ out) {
    // the product kernel after this one may start its weight decode now; the
    // codes are read only after the kernel that wrote them has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)tiles_m * T * nsteps) return;
    const int r = (int)(idx % T);
    const int64_t rest = idx / T;
    const int tt = (int)(rest % tiles_m), s = (int)(rest / tiles_m);
    const int m = tt * T + r, k0 = s * kTcKS;
    uint32_t in[20];
    if (m >= M) {
#pragma unroll
        for (int i = 0; i < 20; i++) in[i] = 0x80808080u;  // bytes v + 128 of v = 0
    } else if ((reinterpret_cast<uintptr_t>(xq) & 15) == 0 && K % 16 == 0) {
        const int8_t *row = xq + (int64_t)m * K;
#pragma unroll
        for (int c = 0; c < 5; c++) {
            // K % 16 == 0: a 16-byte chunk is wholly inside K or wholly past it
            const uint4 v = k0 + 16 * c < K ? __ldg(reinterpret_cast<const uint4 *>(row + k0 + 16 * c))
                                            : make_uint4(0, 0, 0, 0);
            in[4 * c] = v.x ^ 0x80808080u;
            in[4 * c + 1] = v.y ^ 0x80808080u;
            in[4 * c + 2] = v.z ^ 0x80808080u;
            in[4 * c + 3] = v.w ^ 0x80808080u;
        }
    } else {
        const int8_t *row = xq + (int64_t)m * K;
#pragma unroll
        for (int i = 0; i < 20; i++) {
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const int k = k0 + 4 * i + b;
                v |= (k < K ? (uint32_t)(uint8_t)row[k] : 0u) << (8 * b);
            }
            in[i] = v ^ 0x80808080u;
        }
    }
    tm_put_row(out + ((int64_t)tt * nsteps + s) * tm_b_bytes(T), in, r);
}

constexpr int kQtNormLoads = 4;  // elements per thread and round of the norm prologue (n <= 4096: one round)

// rmsnorm_row (decode_ops.cuh) for a whole block, the same sums: the squares'
// pairwise tree over next_pow2(n) zero-padded leaves, each of the T threads
// (T the largest power of two in the block) first reducing its segment of
// P / T adjacent leaves, then lanes, then warps adjacent first.  The warps'
// partials are reduced by one warp's butterfly instead of a serial loop (zero
// padding past the last warp adds exactly nothing, so the tree is the same).
// buf: shared memory >= next_pow2(n) floats, red: >= 32 floats.
__device__ __forceinline__ void qt_rmsnorm(const float *x, const float *g, float *out, int n, float eps, float *buf,
                                           float *red) {
    const int P = next_pow2(n), tid = threadIdx.x, nth = blockDim.x;
    for (int i0 = tid; i0 < P; i0 += kQtNormLoads * nth) {  // every load of a round in flight
        float v[kQtNormLoads];
#pragma unroll
        for (int j = 0; j < kQtNormLoads; j++) {
            const int i = i0 + j * nth;
            v[j] = (i < n) ? x[i] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kQtNormLoads; j++) {
            const int i = i0 + j * nth;
            if (i < P) buf[i] = __fmul_rn(v[j], v[j]);
        }
    }
    int T = 32;
    while (2 * T <= nth) T *= 2;
    __syncthreads();
    float v = 0.0f;
    if (tid < T) {
        if (P >= T) {
            const int S = P / T;
            float *a = buf + tid * S;
            for (int st = 1; st < S; st <<= 1)
                for (int i = 0; i < S; i += 2 * st) a[i] = __fadd_rn(a[i], a[i + st]);
            v = a[0];
        } else {
            v = (tid < P) ? buf[tid] : 0.0f;
        }
    }
    v = warp_psum(v);
    if ((tid & 31) == 0 && tid < T) red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
        float w = tid < (T >> 5) ? red[tid] : 0.0f;
        w = warp_psum(w);
        if (tid == 0) red[0] = w;
    }
    __syncthreads();
    float ss = red[0];
    ss = __fdiv_rn(ss, (float)n);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    for (int i0 = tid; i0 < n; i0 += kQtNormLoads * nth) {
        float gv[kQtNormLoads], xv[kQtNormLoads];
#pragma unroll
        for (int j = 0; j < kQtNormLoads; j++) {
            const int i = i0 + j * nth;
            gv[j] = i < n ? g[i] : 0.0f;
            xv[j] = i < n ? x[i] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kQtNormLoads; j++) {
            const int i = i0 + j * nth;
            if (i < n) out[i] = __fmul_rn(gv[j], __fmul_rn(r, xv[j]));
        }
    }
}

// Where the row a quantiser block quantises comes from.
enum QtMode : int {
    kQtRow = 0,   // x[m] as it is
    kQtNorm = 1,  // h[m] (+= y[m] first, written back, when y is given), then RMSNorm with gain g
    kQtGeglu = 2  // gelu(x[m]) * u[m], elementwise
};
struct QtArgs {
    const float *x;  // kQtRow, kQtGeglu: the row (gate); kQtNorm: unused
    float *h;        // kQtNorm: the residual stream
    const float *y;  // kQtNorm: added to h first, or null
    const float *g;  // kQtNorm: the RMSNorm gain
    const float *u;  // kQtGeglu: the up projection
    float eps;
    int8_t *xq;      // the codes [M][K], or null when only the tiles are wanted
    float *xs;
    uint8_t *tiles;  // activation tiles (t158_tc_workspace_bytes(M, K)), or null (then xq is required)
    int M, K, T, tiles_m, nsteps;
};

// The activation quantiser (absmax per token, as quant_i8_kernel) with the
// tile conversion of t158_act_tiles_kernel, behind an optional row prologue
// (the residual add and RMSNorm of rmsnorm_kernel, or the GeGLU product of
// geglu_kernel, the same operations in the same order): block m builds its
// row (in shared memory for the prologues), quantises it to xq and, as fp16
// in K' order, into its row of every step's tile image; blocks M ..
// tiles_m T - 1 zero the padding rows.  One thread per 16-byte chunk (eight
// K' values of one step); every input is read by exactly one chunk.
constexpr int kQtThreads = 1024;  // a whole row per block: wide blocks keep a few tokens fast
constexpr int kQtGegluLoads = 8;  // gate and up elements per thread and round of the GeGLU prologue

template <int MODE>
__global__ void __launch_bounds__(kQtThreads) t158_quant_tiles_kernel(QtArgs a) {
    extern __shared__ float qt_row[];  // prologues: [K] the row, then [next_pow2(K)] scratch (kQtNorm)
    __shared__ float red[32];
    // the product kernel after this one may start its weight decode now; the
    // inputs are read only after the kernel that wrote them has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = blockIdx.x, K = a.K;
    const bool real = m < a.M;
    const float *row = nullptr;
    if (real) {
        if (MODE == kQtRow) {
            row = a.x + (int64_t)m * K;
        } else if (MODE == kQtGeglu) {
            // rounds of kQtGegluLoads elements per thread (K <= 8192: one round), every
            // load of a round in flight before the products
            const float *gr = a.x + (int64_t)m * K, *ur = a.u + (int64_t)m * K;
            for (int k0 = threadIdx.x; k0 < K; k0 += kQtGegluLoads * blockDim.x) {
                float gv[kQtGegluLoads], uv[kQtGegluLoads];
#pragma unroll
                for (int j = 0; j < kQtGegluLoads; j++) {
                    const int k = k0 + j * blockDim.x;
                    gv[j] = k < K ? gr[k] : 0.0f;
                    uv[j] = k < K ? ur[k] : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < kQtGegluLoads; j++) {
                    const int k = k0 + j * blockDim.x;
                    if (k < K) qt_row[k] = __fmul_rn(gelu32(gv[j]), uv[j]);
                }
            }
            __syncthreads();
            row = qt_row;
        } else {
            float *hr = a.h + (int64_t)m * K;
            if (a.y) {
                const float *yr = a.y + (int64_t)m * K;
                for (int k0 = threadIdx.x; k0 < K; k0 += kQtNormLoads * blockDim.x) {
                    float hv[kQtNormLoads], yv[kQtNormLoads];
#pragma unroll
                    for (int j = 0; j < kQtNormLoads; j++) {
                        const int k = k0 + j * blockDim.x;
                        hv[j] = k < K ? hr[k] : 0.0f;
                        yv[j] = k < K ? yr[k] : 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < kQtNormLoads; j++) {
                        const int k = k0 + j * blockDim.x;
                        if (k < K) hr[k] = __fadd_rn(hv[j], yv[j]);
                    }
                }
            }
            // each thread reads back only the elements it wrote; the norm syncs before the sum
            qt_rmsnorm(hr, a.g, qt_row, K, a.eps, qt_row + K, red);
            __syncthreads();
            row = qt_row;
        }
    }
    float sc = 0.0f, rinv = 0.0f;
    if (real) {
        float am = 0.0f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) am = fmaxf(am, fabsf(row[k]));
        am = warp_max(am);
        __syncthreads();  // red is free (the prologue's sums are done with it)
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
            v = warp_max(v);
            if (threadIdx.x == 0) red[0] = v;
        }
        __syncthreads();
        sc = quant_scale(red[0]);
        rinv = __fdiv_rn(1.0f, sc);
        if (threadIdx.x == 0) a.xs[m] = sc;
    }
    if (!a.tiles) {  // codes only
        if (real)
            for (int k = threadIdx.x; k < K; k += blockDim.x) a.xq[(int64_t)m * K + k] = (int8_t)quant_code_r(row[k], sc, rinv);
        return;
    }
    const int tt = m / a.T, r = m % a.T;
    for (int c = threadIdx.x; c < a.nsteps * kTcChunks; c += blockDim.x) {
        const int s = c / kTcChunks, kc = c % kTcChunks;
        const int i = kc >> 1, jb = 8 * (kc & 1);  // digit i of packed-byte columns jb .. jb + 7
        uint32_t hh[4];
#pragma unroll
        for (int p = 0; p < 4; p++) {
            int q2[2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int k = s * kTcKS + 5 * (jb + 2 * p + e) + i;
                q2[e] = 0;
                if (real && k < K) {
                    q2[e] = quant_code_r(row[k], sc, rinv);
                    if (a.xq) a.xq[(int64_t)m * K + k] = (int8_t)q2[e];
                }
            }
            const __half2 hv = __halves2half2(__int2half_rn(q2[0]), __int2half_rn(q2[1]));
            hh[p] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        *reinterpret_cast<uint4 *>(a.tiles + ((int64_t)tt * a.nsteps + s) * tm_b_bytes(a.T) + tc_off(r, kc)) =
            make_uint4(hh[0], hh[1], hh[2], hh[3]);
    }
}

// Up to three weight matrices that share the input (and K): one launch runs
// them all, tiles 0 .. of matrix 0 first (blockIdx.x from tile0[j] on is
// matrix j).
constexpr int kTmMaxMats = 3;
struct TmMats {
    const uint8_t *w[kTmMaxMats];
    int64_t pitch[kTmMaxMats];
    const float *ws_ptr[kTmMaxMats];  // weight scale in device memory, or null (then ws_arg)
    float *y[kTmMaxMats];
    int32_t *acc[kTmMaxMats];
    int N[kTmMaxMats];
    int tile0[kTmMaxMats + 1];
    int count;
    int y_maps;  // bit j: y[j] is written through ymaps.m[j] (tile staged in shared memory, one tensor store)
};

// Tensor maps of the outputs y[j]: fp32 [M][N[j]], boxes of kTmRows outputs
// x T tokens, no swizzle.
struct TmYMaps {
    CUtensorMap m[kTmMaxMats];
};
struct TmNoMaps {  // the launches that store y directly (a K split) carry no maps
    int unused;
};

// Grid: (weight-row tiles, token tiles, split); a cluster is the `split` CTAs
// of one tile, each over its own range of K steps.  split == 1: no cluster
// reduction.  T: tokens per tile (a multiple of 32, at most kTmMaxTok).
// PRE: `tiles` holds the activation tiles written by t158_act_tiles_kernel.
template <bool PRE, bool YT>
__global__ void __launch_bounds__(kTmThreads, 1)
    t158_tm_kernel(const int8_t *__restrict__ xq, const uint8_t *__restrict__ tiles, const float *__restrict__ xs,
                   const TmMats mats, const __grid_constant__ typename std::conditional<YT, TmYMaps, TmNoMaps>::type ymaps,
                   float ws_arg, int M, int K, int T, int split) {
    constexpr int S = tm_stages(PRE), R = tm_raws(PRE);
    int mj = 0;  // this CTA's matrix
    while (mj + 1 < mats.count && (int)blockIdx.x >= mats.tile0[mj + 1]) mj++;
    const uint8_t *__restrict__ w = mats.w[mj];
    const int64_t pitch = mats.pitch[mj];
    float *__restrict__ y = mats.y[mj];
    int32_t *__restrict__ acc_out = mats.acc[mj];
    const int N = mats.N[mj];
    const float ws = mats.ws_ptr[mj] ? __ldg(mats.ws_ptr[mj]) : ws_arg;  // the weight scale, from device memory when given
    extern __shared__ __align__(128) uint8_t tm_smem[];
    TmCtl &C = *reinterpret_cast<TmCtl *>(tm_smem);
    uint8_t *const btile = tm_smem + kTmCtl;
    uint8_t *const raw_a = tm_smem + tm_raw_a_off(T, PRE);
    uint8_t *const raw_w = tm_smem + tm_raw_w_off(T, PRE);
    const int bstage = tm_b_bytes(T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = ((int)blockIdx.x - mats.tile0[mj]) * kTmRows, m0 = blockIdx.y * T;
    const int nsteps = (K + kTcKS - 1) / kTcKS;
    const int z = split > 1 ? (int)cluster_rank() : 0;
    const int s_lo = (int)((int64_t)nsteps * z / split), s_hi = (int)((int64_t)nsteps * (z + 1) / split);
    const int nst = s_hi - s_lo;  // steps of this CTA
    const int units = 2 * T;      // activation units per step (in-kernel conversion)
    // converter roles: weight rows 32 q .. + 31, packed bytes 8 hw .. + 7 of each step
    const int q = warp & 3, hw = (warp >> 2) & 1;
    const int wrow = 32 * q + lane;
    const bool a_async = !PRE && (reinterpret_cast<uintptr_t>(xq) & 15) == 0 && K % 16 == 0;

    // Raw bytes of each converter's own work run R - 1 steps ahead (zero-filled
    // past K, M and N: such products are zero or land outside the output); a
    // thread reads back only what it copied, so its own wait_group is enough.
    // Unaligned activations are loaded directly.
    auto fetch = [&](int s) {
        if (s < s_hi) {
            const int rs = (s - s_lo) % R;
            const int n = n0 + wrow;
            cp_async8(raw_w + (rs * kTmConv + tid) * 8, w + (int64_t)(n < N ? n : 0) * pitch + (int64_t)s * 16 + 8 * hw,
                      n < N ? 8 : 0);
            if (a_async) {
#pragma unroll
                for (int k = 0; k < 2; k++) {
                    const int u = tid + kTmConv * k;
                    if (u < units) {
                        const int h = u >= T, m = m0 + (h ? u - T : u);
                        const int8_t *row = xq + (int64_t)(m < M ? m : 0) * K;
#pragma unroll
                        for (int c = 0; c < 3; c++) {
                            const int kb = s * kTcKS + 32 * h + 16 * c;
                            const int nb = m < M ? max(0, min(16, K - kb)) : 0;
                            cp_async16(raw_a + (rs * units + u) * kTmUnit + 16 * c, nb > 0 ? row + kb : row, nb);
                        }
                    }
                }
            }
        }
        cp_async_commit();
    };
    // Programmatic dependent launch: the next kernel on the stream may start
    // its set-up now.  The packed weights and their scale are read-only
    // inputs, so their copies start at once; the activations (codes, tiles,
    // scales) are read, and y and acc written, only after the previous kernel
    // on the stream has completed (griddepcontrol.wait).  With the tile
    // images (PRE) only the copy warp (which also loads the scales) waits, so
    // the weight decode of the first steps overlaps the kernel that wrote the
    // tiles; otherwise the converters read the codes and wait too.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!PRE) asm volatile("griddepcontrol.wait;" ::: "memory");
    // the first copies go out before anything else
    if (tid < kTmConv) {
#pragma unroll
        for (int s = 0; s < R - 1; s++) fetch(s_lo + s);
    }
    // the tile's activation scales (without tile images): loaded now, stored for the
    // epilogue after the K loop; with them the copy warp stores them
    const float xs_own = (!PRE && tid < T && m0 + tid < M) ? xs[m0 + tid] : 0.0f;
    const uint32_t ncols = tm_cols(T, PRE);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&C.tmem)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int i = 0; i < S; i++) {
            mbar_init(&C.full[i], kTmConv + (PRE ? 1 : 0));
            mbar_init(&C.mma_done[i], 1);
        }
        C.abort = 0;
        C.issued = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = C.tmem;
    volatile int *abort = &C.abort;

    if (warp == kTmConv / 32) {
        // ---- MMA warp: lane 0 issues each step's five MMAs once the stage is
        // filled, and commits them to the stage's mma_done
        if (lane == 0) {
            const uint32_t idesc = tm_idesc(T);
            for (int i = 0; i < nst && !*abort; i++) {
                const int st = i % S;
                if (!mbar_wait(&C.full[st], (uint32_t)(i / S) & 1u)) {
                    *abort = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t bd = tc_desc(smem_addr(btile + st * bstage));
                const uint32_t a0 = tmem + (uint32_t)(T + kTmACols * st);
#pragma unroll
                for (int u = 0; u < kTcKS / 16; u++)  // K = 16: 8 weight columns, 2 activation core matrices (256 bytes)
                    tm_mma(tmem, a0 + 8u * u, bd + (uint64_t)(16 * u), idesc, (i > 0 || u > 0) ? 1u : 0u);
                tc_commit(&C.mma_done[st]);
                *reinterpret_cast<volatile int *>(&C.issued) = i + 1;
            }
        }
    } else if (warp == kTmConv / 32 + 1) {
        // ---- copy warp (PRE): lane 0 brings each step's activation tile in
        // with one bulk copy once the MMAs that read the stage before are done
        if (PRE) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the tile images and the scales are written
            for (int t = lane; t < T; t += 32) C.xs[t] = m0 + t < M ? xs[m0 + t] : 0.0f;  // read after the barriers below
        }
        if (PRE && lane == 0) {
            const uint8_t *src = tiles + ((int64_t)blockIdx.y * nsteps + s_lo) * bstage;
            for (int i = 0; i < nst && !*abort; i++) {
                const int st = i % S;
                if (i >= S && !mbar_wait(&C.mma_done[st], (uint32_t)(i / S - 1) & 1u)) {
                    *abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&C.full[st], (uint32_t)bstage);
                bulk_g2s_plain(btile + st * bstage, src + (int64_t)i * bstage, (uint32_t)bstage, &C.full[st]);
            }
        }
    } else {
        // ---- converters (whole warps: the tensor-memory stores are warp-wide)
        const uint32_t ta_row = tmem + ((uint32_t)(32 * q) << 16);
        for (int i = 0; i < nst; i++) {
            if (__any_sync(0xffffffffu, *abort != 0)) break;
            const int s = s_lo + i, st = i % S, rs = i % R;
            fetch(s + R - 1);
            cp_async_wait_pending<R - 1>();  // this thread's copies of step s have landed
            // the MMAs of step i - S read this stage: wait until they are done
            bool ok = true;
            if (i >= S) ok = mbar_wait(&C.mma_done[st], (uint32_t)(i / S - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                *abort = 1;
                break;
            }
            tc_fence_after();
            tm_put_w(ta_row + (uint32_t)(T + kTmACols * st),
                     *reinterpret_cast<const uint2 *>(raw_w + (rs * kTmConv + tid) * 8), hw);
            if (!PRE) {
                uint8_t *const bt = btile + st * bstage;
#pragma unroll
                for (int k = 0; k < 2; k++) {
                    const int u = tid + kTmConv * k;
                    if (u < units) {  // whole warps: T is a multiple of 32
                        const int h = u >= T, r = h ? u - T : u;
                        uint32_t in[12];
                        if (a_async) {
                            const uint4 *src = reinterpret_cast<const uint4 *>(raw_a + (rs * units + u) * kTmUnit);
#pragma unroll
                            for (int c = 0; c < 3; c++) {
                                const uint4 v = src[c];
                                in[4 * c] = v.x ^ 0x80808080u;
                                in[4 * c + 1] = v.y ^ 0x80808080u;
                                in[4 * c + 2] = v.z ^ 0x80808080u;
                                in[4 * c + 3] = v.w ^ 0x80808080u;
                            }
                        } else {
                            tm_load_act(in, xq, M, K, m0 + r, s, h);
                        }
                        if (h)
                            tm_put_act<1>(bt, in, r);
                        else
                            tm_put_act<0>(bt, in, r);
                    }
                }
            }
            tm_wait_st();
            // the generic-proxy writes above, visible to the tensor core (async proxy)
            if (!PRE) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&C.full[st]);
        }
        cp_async_wait_pending<0>();
    }
    if (!PRE && tid < T) C.xs[tid] = xs_own;  // read after the barriers below
    // the last commit covers every MMA issued before it
    __syncthreads();
    const int issued = C.issued;
    if (issued > 0) {
        const int i = issued - 1;
        if (!mbar_wait(&C.mma_done[i % S], (uint32_t)(i / S) & 1u)) *abort = 1;
    }
    __syncthreads();
    const bool ok = !*abort && issued == nst;
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // y and acc may be read by the previous kernel until it ends

    const float nanv = ok ? 0.0f : __int_as_float(0x7fc00000);  // a wait that gave up: the tile reads NaN
    float *const part = reinterpret_cast<float *>(tm_smem + kTmCtl);
    // Without a K split, y leaves as one tensor store of the tile, staged in
    // shared memory as [token][row] (the stages' space, free now): one 4-byte
    // shared store per value instead of a global store with its address.
    const bool y_tma = YT && split == 1 && y && ((mats.y_maps >> mj) & 1) && (smem_addr(part) & 127u) == 0;
    if (warp < kTmConv / 32) {
        // warp w: weight rows 32 (w % 4) .. + 31 (its lanes), tokens T/2 (w / 4) .. + T/2 - 1
        const int n = n0 + wrow;
        const int tb = (warp >> 2) * (T / 2);
        const int nch = T / 32;  // 16-column loads of this warp's T/2 tokens (1..4)
        // two loads go out before each wait
#pragma unroll 1
        for (int k2 = 0; k2 < nch; k2 += 2) {
        uint32_t r[2][16];
#pragma unroll
        for (int k = 0; k < 2; k++)
            if (k2 + k < nch) tm_ld16_nw(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(tb + 16 * (k2 + k)), r[k]);
#pragma unroll
        for (int k = 0; k < 2; k++)
            if (k2 + k < nch) tm_wait_ld(r[k]);
#pragma unroll
        for (int k = 0; k < 2; k++) {
            if (k2 + k >= nch) break;
            const int t0 = tb + 16 * (k2 + k);
            if (split == 1) {
                if (y_tma) {  // rows past N and tokens past M are clipped by the store
                    // the scales first: a store into the stage may alias them for the
                    // compiler, which would otherwise wait out each load in turn
                    float xk[16];
#pragma unroll
                    for (int j = 0; j < 16; j++) xk[j] = C.xs[t0 + j];
#pragma unroll
                    for (int j = 0; j < 16; j++)
                        part[(t0 + j) * kTmRows + wrow] =
                            __fadd_rn(__fmul_rn(__fmul_rn(__uint_as_float(r[k][j]), ws), xk[j]), nanv);
                }
                if (n < N && (acc_out || (y && !y_tma))) {
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int m = m0 + t0 + j;
                        if (m >= M) break;
                        const float v = __uint_as_float(r[k][j]);
                        if (acc_out) acc_out[(int64_t)m * N + n] = __float2int_rz(v);
                        if (y && !y_tma) y[(int64_t)m * N + n] = __fadd_rn(__fmul_rn(__fmul_rn(v, ws), C.xs[t0 + j]), nanv);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; j++) part[(t0 + j) * kTmPStride + wrow] = __uint_as_float(r[k][j]);
            }
        }
        }
        if (y_tma) {
            fence_proxy_async_smem();  // the staged tile, visible to the tensor store
            asm volatile("bar.sync 2, %0;" ::"n"(kTmConv) : "memory");
            if constexpr (YT) {
                if (tid == 0) {
                    tma_store_2d(&ymaps.m[mj], part, n0, m0);
                    bulk_commit_group();
                    bulk_wait_read_all();  // the shared memory is read before the CTA can leave
                }
            }
        }
    }
    if (split > 1) {
        // CTA z adds tokens [T z / split, T (z+1) / split) over the cluster in
        // rank order (integers below 2^24: exact)
        cluster_sync();
        const int t_lo = T * z / split, t_hi = T * (z + 1) / split;
        const bool vec_y = y && (reinterpret_cast<uintptr_t>(y) & 15) == 0 && N % 4 == 0;
        const bool vec_acc = acc_out && (reinterpret_cast<uintptr_t>(acc_out) & 15) == 0 && N % 4 == 0;
#pragma unroll 2
        for (int e = tid; e < (t_hi - t_lo) * (kTmRows / 4); e += kTmThreads) {
            const int t = t_lo + e / (kTmRows / 4), c4 = e % (kTmRows / 4);
            const int m = m0 + t, nb = n0 + 4 * c4;
            if (m >= M || nb >= N) continue;
            float4 u[kTmMaxSplit];
#pragma unroll
            for (int qq = 0; qq < kTmMaxSplit; qq++)
                if (qq < split) u[qq] = ld_peer_f4(&part[t * kTmPStride + 4 * c4], (uint32_t)qq);
            float4 v = u[0];
#pragma unroll
            for (int qq = 1; qq < kTmMaxSplit; qq++)
                if (qq < split) {
                    v.x = __fadd_rn(v.x, u[qq].x);
                    v.y = __fadd_rn(v.y, u[qq].y);
                    v.z = __fadd_rn(v.z, u[qq].z);
                    v.w = __fadd_rn(v.w, u[qq].w);
                }
            const float vv[4] = {v.x, v.y, v.z, v.w};
            const float xsm = C.xs[t];
            if (acc_out) {
                if (vec_acc && nb + 4 <= N) {
                    *reinterpret_cast<int4 *>(acc_out + (int64_t)m * N + nb) = make_int4(
                        __float2int_rz(vv[0]), __float2int_rz(vv[1]), __float2int_rz(vv[2]), __float2int_rz(vv[3]));
                } else {
                    for (int j = 0; j < 4; j++)
                        if (nb + j < N) acc_out[(int64_t)m * N + nb + j] = __float2int_rz(vv[j]);
                }
            }
            if (y) {
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; j++) o[j] = __fadd_rn(__fmul_rn(__fmul_rn(vv[j], ws), xsm), nanv);
                if (vec_y && nb + 4 <= N) {
                    *reinterpret_cast<float4 *>(y + (int64_t)m * N + nb) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
                    for (int j = 0; j < 4; j++)
                        if (nb + j < N) y[(int64_t)m * N + nb + j] = o[j];
                }
            }
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}

// Token tiling of M tokens: the fewest tiles of at most kTmMaxTok tokens,
// T rounded up to a multiple of 32.
static void tm_token_tiles(int M, int &tiles_m, int &T) {
    tiles_m = (M + kTmMaxTok - 1) / kTmMaxTok;
    T = ((M + tiles_m - 1) / tiles_m + 31) / 32 * 32;
}

size_t t158_tc_workspace_bytes(int M, int K) {
    int tiles_m = 0, T = 0;
    tm_token_tiles(M, tiles_m, T);
    return (size_t)tiles_m * (size_t)((K + kTcKS - 1) / kTcKS) * (size_t)tm_b_bytes(T);
}

// The tensor map of an output y: fp32 [M][N] (N a multiple of 4, y 16-byte
// aligned), boxes of kTmRows outputs x T tokens, no swizzle.  Encoded through
// the driver entry point (no link against the driver library); recent maps
// are kept for the next call on the same output.
static qlin_status tm_y_map(float *y, int M, int N, int T, CUtensorMap *out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::map<std::tuple<int, const void *, int, int, int>, CUtensorMap> cache;
    int dev = 0;
    QLIN_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_tuple(dev, (const void *)y, M, N, T);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return QLIN_OK;
    }
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        QLIN_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
        QLIN_REQUIRE(fn && q == cudaDriverEntryPointSuccess, QLIN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    const cuuint64_t gdim[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)N * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kTmRows, (cuuint32_t)T};
    const cuuint32_t estride[2] = {1, 1};
    CUtensorMap m;
    const CUresult r = encode(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, gdim, gstride, box, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    QLIN_REQUIRE(r == CUDA_SUCCESS, QLIN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    if (cache.size() >= 256) cache.clear();
    cache[key] = m;
    *out = m;
    return QLIN_OK;
}

// Clusters of `c` CTAs of this kernel with `smem` bytes each that can be
// resident at once (cached).
template <bool PRE>
static int tm_resident_clusters(int c, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, c, smem});
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, (unsigned)c);
    cfg.blockDim = dim3(kTmThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)c;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, t158_tm_kernel<PRE, false>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    cache[{dev, c, smem}] = n;
    return n;
}

// Dynamic shared memory of a launch with T tokens per tile (cached per
// device).  No more CTAs may share an SM than their tensor-memory allocations
// fit in (512 columns): a CTA beyond that would block in tcgen05.alloc, and
// with split-K clusters waiting on one another that wait might never end.
// Shared memory enforces it: each CTA takes more than 1/(fit+1) of the SM's,
// checked against the occupancy the runtime reports.
template <bool PRE>
static qlin_status tm_launch_smem(int T, size_t *out) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, size_t> cache;
    int dev = 0;
    QLIN_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, T});
    if (it != cache.end()) {
        *out = it->second;
        return QLIN_OK;
    }
    const int fit = (int)(512u / tm_cols(T, PRE));
    size_t smem = (size_t)tm_smem_bytes(T, PRE);
    int sm_smem = 0, reserved = 0;
    QLIN_CUDA(cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
    QLIN_CUDA(cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev));
    const size_t floor_smem = (size_t)(sm_smem / (fit + 1) - reserved + 16) / 16 * 16 + 16;
    if (smem < floor_smem) smem = floor_smem;
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: tensor-core tile does not fit");
    blocks_per_sm((const void *)t158_tm_kernel<PRE, false>, smem);  // raises the dynamic shared-memory limit
    blocks_per_sm((const void *)t158_tm_kernel<PRE, true>, smem);
    int resident = 0;
    QLIN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, t158_tm_kernel<PRE, false>, kTmThreads, smem));
    QLIN_REQUIRE(resident >= 1 && resident <= fit, QLIN_ERR_UNSUPPORTED,
                 "qlin_t158_i8: %d CTAs per SM would exceed tensor memory (%d fit)", resident, fit);
    cache[{dev, T}] = smem;
    *out = smem;
    return QLIN_OK;
}

// early: launch with programmatic stream serialisation, so that the weight
// decode of the first steps overlaps the kernel before (the tile
// conversion).  Measured on the decoder's shapes: a win except behind a
// large conversion (512 tokens x 6912 inputs), where the early CTAs slow the
// conversion down more than they gain.
template <bool PRE>
static qlin_status launch_tm(const int8_t *xq, const uint8_t *tiles, const float *xs, TmMats mats, float ws,
                             int M, int K, int tiles_m, int T, cudaStream_t st, bool early = true) {
    size_t smem = 0;
    if (qlin_status e = tm_launch_smem<PRE>(T, &smem)) return e;
    mats.y_maps = 0;
    mats.tile0[0] = 0;
    for (int j = 0; j < mats.count; j++) mats.tile0[j + 1] = mats.tile0[j] + (mats.N[j] + kTmRows - 1) / kTmRows;
    for (int j = mats.count + 1; j <= kTmMaxMats; j++) mats.tile0[j] = mats.tile0[mats.count];
    const int tiles_n = mats.tile0[mats.count];
    const int nsteps = (K + kTcKS - 1) / kTcKS;
    // split K over a cluster when the tiles alone leave SMs idle: the largest
    // split whose clusters (they must fit within a GPC) are all resident at once
    const int ntiles = tiles_n * tiles_m;
    int split = 1;
    for (int c = kTmMaxSplit; c >= 2; c--) {
        if (c > nsteps || ntiles * c > 2 * sm_count()) continue;
        if (tm_resident_clusters<PRE>(c, smem) >= ntiles) {
            split = c;
            break;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles_n, (unsigned)tiles_m, (unsigned)split);
    cfg.blockDim = dim3(kTmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)split;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    // without a K split no cluster is needed: a plain grid launch
    cfg.attrs = split > 1 ? attr : attr + 1;
    cfg.numAttrs = (split > 1 ? 1 : 0) + (early ? 1 : 0);
    if (split == 1) {
        // y through tensor stores where its layout allows (16-byte rows)
        TmYMaps ymaps;
        memset(&ymaps, 0, sizeof(ymaps));
        for (int j = 0; j < mats.count; j++)
            if (mats.y[j] && (reinterpret_cast<uintptr_t>(mats.y[j]) & 15) == 0 && mats.N[j] % 4 == 0) {
                if (qlin_status e = tm_y_map(mats.y[j], M, mats.N[j], T, &ymaps.m[j])) return e;
                mats.y_maps |= 1 << j;
            }
        if (mats.y_maps) {
            QLIN_CUDA(cudaLaunchKernelEx(&cfg, t158_tm_kernel<PRE, true>, xq, tiles, xs, mats, ymaps, ws, M, K, T, split));
            QLIN_LAUNCHED("t158_tm_kernel");
            return QLIN_OK;
        }
    }
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, t158_tm_kernel<PRE, false>, xq, tiles, xs, mats, TmNoMaps{0}, ws, M, K, T, split));
    QLIN_LAUNCHED("t158_tm_kernel");
    return QLIN_OK;
}

// work: device scratch of at least t158_tc_workspace_bytes(M, K) bytes,
// 16-byte aligned, or null (then the converter warps convert the activations
// at every step of every tile).  convert: write the activation tiles of xq
// into work first; false when an earlier call with the same xq, M and K on
// this stream already did.
qlin_status t158_linear_tensor_cores(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                     const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st,
                                     void *work, bool convert) {
    int tiles_m = 0, T = 0;
    tm_token_tiles(M, tiles_m, T);
    TmMats mats{};
    mats.w[0] = w, mats.pitch[0] = pitch, mats.ws_ptr[0] = ws_ptr, mats.y[0] = y, mats.acc[0] = acc, mats.N[0] = N;
    mats.count = 1;
    if (!work) return launch_tm<false>(xq, nullptr, xs, mats, ws, M, K, tiles_m, T, st);
    if (convert) {
        const int nsteps = (K + kTcKS - 1) / kTcKS;
        const int64_t threads = (int64_t)tiles_m * T * nsteps;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        // launched after the previous kernel ends; it lets the product start at once
        QLIN_CUDA(cudaLaunchKernelEx(&cfg, t158_act_tiles_kernel, xq, M, K, T, tiles_m, nsteps, (uint8_t *)work));
        QLIN_LAUNCHED("t158_act_tiles_kernel");
    }
    // behind a large tile conversion the product does not start early (see launch_tm)
    const bool early = !convert || (int64_t)tiles_m * T * ((K + kTcKS - 1) / kTcKS) <= kTmEarlyMaxItems;
    return launch_tm<true>(xq, (const uint8_t *)work, xs, mats, ws, M, K, tiles_m, T, st, early);
}

// Linears j = 0 .. count - 1 on one set of activation tiles (already in work,
// written by the quantiser for this xq, M and K): w[j] [N[j]][pitch[j]],
// weight scale in device memory at ws_ptr[j], output y[j] [M][N[j]], all in
// one launch.
qlin_status t158_linear_tiles_multi(const float *xs, int count, const uint8_t *const *w, const int64_t *pitch,
                                    const float *const *ws_ptr, float *const *y, const int *N, int M, int K,
                                    void *work, cudaStream_t st) {
    QLIN_REQUIRE(count >= 1 && count <= kTmMaxMats && work, QLIN_ERR_INVALID_ARG, "t158_linear_tiles_multi: %d", count);
    int tiles_m = 0, T = 0;
    tm_token_tiles(M, tiles_m, T);
    TmMats mats{};
    for (int j = 0; j < count; j++)
        mats.w[j] = w[j], mats.pitch[j] = pitch[j], mats.ws_ptr[j] = ws_ptr[j], mats.y[j] = y[j], mats.N[j] = N[j];
    mats.count = count;
    return launch_tm<true>(nullptr, (const uint8_t *)work, xs, mats, 0.0f, M, K, tiles_m, T, st);
}

// The quantiser kernels' launch: one block per token (per padded token row
// when tiles are written), with the row prologue's shared memory.
template <int MODE>
static qlin_status launch_qt(QtArgs a, void *work, cudaStream_t st) {
    int tiles_m = 0, T = 0;
    tm_token_tiles(a.M, tiles_m, T);
    a.T = T;
    a.tiles_m = tiles_m;
    a.nsteps = (a.K + kTcKS - 1) / kTcKS;
    a.tiles = (uint8_t *)work;
    const size_t smem = MODE == kQtRow     ? 0
                        : MODE == kQtGeglu ? (size_t)a.K * sizeof(float)
                                           : (size_t)(a.K + next_pow2(a.K)) * sizeof(float);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "quantiser: row of %d too long", a.K);
    QLIN_REQUIRE(a.xq || work, QLIN_ERR_INVALID_ARG, "quantiser: neither codes nor tiles requested");
    if (smem > 48 * 1024) blocks_per_sm((const void *)t158_quant_tiles_kernel<MODE>, smem);
    const unsigned grid = (unsigned)(work ? tiles_m * T : a.M);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kQtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // launched after the previous kernel ends; it lets the product start at once
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, t158_quant_tiles_kernel<MODE>, a));
    QLIN_LAUNCHED("t158_quant_tiles_kernel");
    return QLIN_OK;
}

// qlin_quant_i8 (the same xq and xs) that also writes the activation tiles of
// t158_linear_tensor_cores into work (t158_tc_workspace_bytes(M, K) bytes;
// null: codes only), so that the linears on this input run with convert =
// false.
qlin_status quant_i8_tiles(const float *x, int8_t *xq, float *xs, int M, int K, void *work, cudaStream_t st) {
    QtArgs a{};
    a.x = x, a.xq = xq, a.xs = xs, a.M = M, a.K = K;
    return launch_qt<kQtRow>(a, work, st);
}

// h[m] += y[m] (y may be null), then the quantiser on RMSNorm(h[m]) * gain:
// rmsnorm_kernel and quant_i8_tiles in one launch, the same values.
qlin_status norm_quant_tiles(float *h, const float *y, const float *gain, float eps, int8_t *xq, float *xs, int M,
                             int K, void *work, cudaStream_t st) {
    QtArgs a{};
    a.h = h, a.y = y, a.g = gain, a.eps = eps, a.xq = xq, a.xs = xs, a.M = M, a.K = K;
    return launch_qt<kQtNorm>(a, work, st);
}

// The quantiser on gelu(gate) * up: geglu_kernel and quant_i8_tiles in one
// launch, the same values (the product itself is not stored).
qlin_status geglu_quant_tiles(const float *gate, const float *up, int8_t *xq, float *xs, int M, int K, void *work,
                              cudaStream_t st) {
    QtArgs a{};
    a.x = gate, a.u = up, a.xq = xq, a.xs = xs, a.M = M, a.K = K;
    return launch_qt<kQtGeglu>(a, work, st);
}

}  // namespace qlin
