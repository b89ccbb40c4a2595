// W8 linear for a few tokens (2 <= M <= 64) on the fifth-generation tensor
// cores.
//
// y[m][n] = s * sum_k w8[n][k] x[m][k] (cpp20gemma README, "Architecture &
// implementation": int8 weights, one scale per tensor applied after the dot
// product; llama2.c "matmul" is the same loop over output rows) as a matrix
// product per 128 weight rows: tcgen05.mma (kind::f16: fp16 or bf16
// operands, fp32 accumulator in tensor memory), M = 128 weight rows, N = the
// tile's tokens times three terms, K = 16 per instruction.
//
// Operands.  Every int8 weight is an fp16 and a bf16 value exactly.  Each
// fp32 activation enters as three terms of the weights' type, x = hi + mid +
// lo with hi = round(x), mid = round(x - hi), lo = round(x - hi - mid): the
// differences are exact in fp32 and the three terms carry x's 24 significant
// bits, so every product w * term is exact and the only rounding is the fp32
// accumulation.  The output adds a token's three accumulators, (lo + mid) +
// hi, and applies the scale.  Two ways to the terms:
//  - in the product kernel (qlin_w8_f32): four splitter warps copy the
//    tile's x a few stages ahead with cp.async and write bf16 terms (bf16
//    has fp32's exponent range, so no scaling); the weights become bf16;
//  - once per call into a workspace (qlin_w8_f32_ws): w8_terms_kernel writes
//    each stage's operand image, fp16 terms of x' = x 2^(14 - e) with max|x| <
//    2^e (fp16's exponent range is narrow), and the product multiplies the
//    sum back by 2^(e - 14).  The product kernel then only copies each image
//    in (one bulk copy), and the weights become fp16, which costs half the
//    instructions of bf16.  fp16 terms carry x' exactly down to fp16's
//    subnormal step, i.e. every x to within 2^(e - 39).
//
// Data path, one stage of 128 K at a time.  Weights: one tensor copy (TMA,
// 2-D tile mode, 128-byte swizzle) brings 128 rows x 128 bytes into shared
// memory, four stages in flight; rows past N and bytes past K read as zeros.
// Eight converter warps, one
// thread per weight row and half stage (the tensor-memory lane of that row),
// read 64 bytes of their row, release the stage at once, and store the
// converted pairs with tcgen05.st into the stage's slot of the A operand in
// tensor memory: the converted weights never pass through shared memory.
// One thread issues each stage's eight MMAs and commits them to the slot's
// mbarrier; two slots let one stage be converted while the other is
// multiplied.
//
// Split K: a cluster of CTAs over one weight-row tile, each over its own range
// of K stages, adds the partial tiles through distributed shared memory in
// rank order, so the result does not depend on timing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "stream.cuh"
#include "tcgen05.cuh"

namespace qlin {
namespace {

constexpr int kWtRows = 128;                 // weight rows per CTA (MMA M, tensor-memory lanes)
constexpr int kWtKS = 128;                   // K per stage: one tensor copy of 128 rows x 128 bytes
constexpr int kWtRaw = 4;                    // weight stages in flight
constexpr int kWtSlots = 2;                  // A slots in tensor memory (and, splitting in the kernel, B slots)
constexpr int kWtBRing = 3;                  // B images in flight (workspace path)
constexpr int kWtXDepth = 3;                 // stages of raw activations copied ahead (splitting in the kernel)
constexpr int kWtMaxTT = 16;                 // tokens per tile at most
constexpr int kWtConvWarps = 8;              // weight converters: lane quarter w % 4, half stage w / 4
constexpr int kWtXWarps = 4;                 // activation splitters (splitting in the kernel)
constexpr int kWtXThreads = 32 * kWtXWarps;
constexpr int kWtUnits = 2;                  // (token, 8 activations) units per splitter thread and stage
constexpr int kWtMaxSplit = 8;               // CTAs of a cluster that split K
constexpr int kWtChunks = kWtKS / 8;         // 16-byte core-matrix columns of a B row per stage
constexpr int kWtSBO = kWtChunks * 128;      // bytes between 8-row groups of a B operand
constexpr int kWtBMax = 3 * kWtMaxTT / 8 * kWtSBO;               // B operand of a stage: at most 48 rows
constexpr int kWtXHalf = kWtMaxTT * kWtChunks * 16;              // raw activations: 4 of each unit, [unit][16 B]
constexpr int kWtXStage = 2 * kWtXHalf;                          // both halves of every unit of a stage
constexpr int kWtWStage = kWtRows * kWtKS;                       // 16 KB
constexpr int kWtPStride = kWtRows + 4;                          // floats per token of a partial tile
constexpr int kWtTermThreads = 1024;                             // w8_terms_kernel: threads per CTA,
constexpr int kWtTermChunks = 2;                                 // chunks a thread holds in registers,
constexpr int kWtTermMaxP = 8;                                   // CTAs per token (a cluster) at most
constexpr uint32_t kWtCols = 256;   // tensor memory: accumulators at column 0, the A slots from kWtACol
constexpr uint32_t kWtACol = 64;    // A slot s: columns kWtACol + 64 s .. + 63 (128 16-bit values per lane)
static_assert(kWtMaxTT * kWtChunks <= kWtUnits * kWtXThreads, "splitter units");
static_assert(3 * kWtMaxTT <= (int)kWtACol, "accumulator columns");
static_assert(kWtMaxTT * kWtPStride * 4 <= kWtRaw * kWtWStage, "partial tile fits in the weight stages");

// Shared memory of one CTA: the weight stages (1024-byte aligned: the
// swizzle), then the B operands (slots, or the ring of images), the raw
// activations (splitting in the kernel), the control block.
template <bool PRE>
struct WtLayout {
    static constexpr int kB = kWtRaw * kWtWStage;
    static constexpr int kBSlots = PRE ? kWtBRing : kWtSlots;
    static constexpr int kX = kB + kBSlots * kWtBMax;
    static constexpr int kCtl = kX + (PRE ? 0 : kWtXDepth * kWtXStage);
    static constexpr int kThreads = 32 * (kWtConvWarps + (PRE ? 1 : kWtXWarps) + 2);
};

struct WtCtl {
    uint64_t wfull[kWtRaw];      // the weight stage has landed (the tensor copy's bytes)
    uint64_t wempty[kWtRaw];     // the converter warps have read it
    uint64_t full[kWtSlots];     // the A slot (and the B slot when splitting in the kernel) is written
    uint64_t mma_done[kWtSlots]; // the MMAs reading the slot are done (tcgen05.commit)
    uint64_t bfull[kWtBRing];    // workspace path: the B image has landed
    uint64_t bempty[kWtBRing];   // workspace path: the MMAs reading it are done
    uint32_t tmem;
    int abort;
    int issued;  // stages whose MMAs were issued
};
template <bool PRE>
constexpr int wt_smem() {
    return WtLayout<PRE>::kCtl + (int)sizeof(WtCtl);
}
// Above a third of an SM's shared memory, so at most two CTAs share an SM and
// their tensor-memory allocations (256 columns each) always fit; two fit in
// an SM's 228 KB with the largest carveout.
static_assert(wt_smem<false>() > 228 * 1024 / 3 && 2 * (wt_smem<false>() + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(wt_smem<true>() > 228 * 1024 / 3 && 2 * (wt_smem<true>() + 1024) <= 228 * 1024, "two CTAs per SM");

// Bytes of a stage's B image for token capacity PS: 3 PS rows rounded up to
// whole 8-row groups.
__host__ __device__ constexpr int wt_img_bytes(int PS) { return (3 * PS + 7) / 8 * kWtSBO; }

// Four int8 weights (one 32-bit word) -> two bf16 pairs, exactly: the byte b
// of weight w sits under the bf16 exponent of 128 (bits 0x43bb); with bit 7
// of b cleared that is 128 + (w & 127), with only bit 7 kept it is 128 + 128
// [w < 0], and the difference w is exact.  `sel` picks bytes 0, 1 (0x4140) or
// 2, 3 (0x4342) into the low byte of each half.
__device__ __forceinline__ uint32_t wt_i8x2_bf16(uint32_t v, uint32_t sel) {
    const uint32_t t = __byte_perm(v, 0x43u, sel);
    const uint32_t a = t & 0xFF7FFF7Fu, c = t & 0xFF80FF80u;
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}

// The same into fp16 pairs from the word with every byte's top bit flipped
// (b ^ 0x80 = w + 128): under the fp16 exponent of 1024 (bits 0x64bb) that is
// 1152 + w, less 1152.
__device__ __forceinline__ uint32_t wt_i8x2_f16(uint32_t flipped, uint32_t sel) {
    const uint32_t t = __byte_perm(flipped, 0x64u, sel);
    const uint32_t c = 0x64806480u;
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&t), *reinterpret_cast<const __half2 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t *>(&v); }
__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Two activations -> their hi, mid and lo bf16 terms, two per word.
__device__ __forceinline__ void wt_split_bf16(float a, float b, uint32_t &h, uint32_t &m, uint32_t &l) {
    const __nv_bfloat162 H = __floats2bfloat162_rn(a, b);
    const float ra = __fsub_rn(a, __low2float(H)), rb = __fsub_rn(b, __high2float(H));
    const __nv_bfloat162 Mi = __floats2bfloat162_rn(ra, rb);
    const float sa = __fsub_rn(ra, __low2float(Mi)), sb = __fsub_rn(rb, __high2float(Mi));
    h = bf2_bits(H);
    m = bf2_bits(Mi);
    l = bf2_bits(__floats2bfloat162_rn(sa, sb));
}

// The same in fp16 (the caller keeps |a|, |b| < 2^14).
__device__ __forceinline__ void wt_split_f16(float a, float b, uint32_t &h, uint32_t &m, uint32_t &l) {
    const __half2 H = __floats2half2_rn(a, b);
    const float ra = __fsub_rn(a, __low2float(H)), rb = __fsub_rn(b, __high2float(H));
    const __half2 Mi = __floats2half2_rn(ra, rb);
    const float sa = __fsub_rn(ra, __low2float(Mi)), sb = __fsub_rn(rb, __high2float(Mi));
    h = h2_bits(H);
    m = h2_bits(Mi);
    l = h2_bits(__floats2half2_rn(sa, sb));
}

// 2^k as a product of two normal fp32 powers of two, for |k| <= 252.
__device__ __forceinline__ void pow2_pair(int k, float &a, float &b) {
    const int ka = k > 127 ? 127 : k < -126 ? -126 : k;
    a = __int_as_float((ka + 127) << 23);
    b = __int_as_float((k - ka + 127) << 23);
}

// Byte offset of 16-byte chunk kc of row r in a B operand.
__device__ __forceinline__ int wt_boff(int r, int kc) { return (r >> 3) * kWtSBO + kc * 128 + (r & 7) * 16; }

__device__ __forceinline__ void sts128(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Workspace path: a cluster of P CTAs per token m (cluster rank = the CTA's
// slice of K, whole 8-activation chunks) finds the largest |x| of the row
// (each CTA over its slice, then over the cluster through distributed shared
// memory), takes the power of two and writes the three fp16 terms of every
// x' into the B images of the token's tile (rows p PS + t of each stage's
// image, t = m % TT; zeros past K); tscale[m] = 2^(e - 14) as two factors.  A
// thread holds up to kWtTermChunks chunks in registers between the two
// steps (longer slices read their chunks again).  A row holding a NaN or an
// infinity gets NaN terms and a NaN scale.
template <int PS>
__global__ void __launch_bounds__(kWtTermThreads) w8_terms_kernel(const float *__restrict__ x, int M, int K, int TT,
                                                                  int nstg, uint8_t *__restrict__ imgs,
                                                                  float2 *__restrict__ tscale) {
    __shared__ uint32_t red[kWtTermThreads / 32];
    __shared__ uint32_t cta_max;
    constexpr int IMG = wt_img_bytes(PS);
    const int P = (int)gridDim.x, rank = (int)blockIdx.x;  // the cluster spans x
    const int m = blockIdx.y, tt = m / TT, t = m % TT;
    const int tid = threadIdx.x;
    const int nchunks = nstg * kWtChunks;  // up to the end of the last stage (zeros past K)
    const int c_lo = (int)((int64_t)nchunks * rank / P), c_hi = (int)((int64_t)nchunks * (rank + 1) / P);
    // the product kernel after this one may start its weight copies; the
    // workspace may still be read by the product before this one
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float *row = x + (int64_t)m * K;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    auto load = [&](int c, float (&v)[8]) {
        const int k0 = 8 * c;
        if (vec && k0 + 8 <= K) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(row + k0));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(row + k0 + 4));
            v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; q++) v[q] = k0 + q < K ? row[k0 + q] : 0.0f;
        }
    };
    float v[kWtTermChunks][8];
    uint32_t mb = 0;  // largest magnitude bits (NaN and infinity have all exponent bits set)
#pragma unroll
    for (int j = 0; j < kWtTermChunks; j++) {
        const int c = c_lo + tid + kWtTermThreads * j;
        if (c < c_hi) {
            load(c, v[j]);
#pragma unroll
            for (int q = 0; q < 8; q++) mb = max(mb, __float_as_uint(v[j][q]) & 0x7fffffffu);
        }
    }
    for (int c = c_lo + tid + kWtTermThreads * kWtTermChunks; c < c_hi; c += kWtTermThreads) {
        float u[8];
        load(c, u);
#pragma unroll
        for (int q = 0; q < 8; q++) mb = max(mb, __float_as_uint(u[q]) & 0x7fffffffu);
    }
    mb = __reduce_max_sync(0xffffffffu, mb);
    if ((tid & 31) == 0) red[tid >> 5] = mb;
    __syncthreads();
    if (tid == 0) {
        uint32_t b = 0;
#pragma unroll
        for (int w = 0; w < kWtTermThreads / 32; w++) b = max(b, red[w]);
        cta_max = b;
    }
    if (P == 1) {
        __syncthreads();
        mb = cta_max;
    } else {
        cluster_sync();  // every CTA's maximum is written
        mb = 0;
        for (int q = 0; q < P; q++) {
            uint32_t a;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(&cta_max)), "r"(q));
            uint32_t b;
            asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(b) : "r"(a) : "memory");
            mb = max(mb, b);
        }
        cluster_sync();  // no CTA leaves while another still reads its maximum
    }
    const bool finite = mb < 0x7f800000u;
    int e = 0;  // max|x| < 2^e
    if (finite && mb != 0) {
        const int eb = (int)(mb >> 23);
        if (eb != 0)
            e = eb - 126;
        else
            frexpf(__uint_as_float(mb), &e);
    }
    // x' = x 2^(14 - e) and back 2^(e - 14), each as two exact powers of two
    // (|14 - e| <= 163: beyond one fp32 normal exponent)
    float u1, u2, d1, d2;
    pow2_pair(14 - e, u1, u2);
    pow2_pair(e - 14, d1, d2);
    if (rank == 0 && tid == 0)
        tscale[m] = finite ? make_float2(d1, d2) : make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    uint8_t *const base = imgs + (int64_t)tt * nstg * IMG;
    auto emit = [&](int c, const float (&u)[8]) {
        uint32_t th[4], tm[4], tl[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (finite) {
                wt_split_f16(__fmul_rn(__fmul_rn(u[2 * q], u1), u2), __fmul_rn(__fmul_rn(u[2 * q + 1], u1), u2), th[q],
                             tm[q], tl[q]);
            } else {
                th[q] = tm[q] = tl[q] = 0x7e007e00u;  // fp16 NaN
            }
        }
        uint8_t *const img = base + (int64_t)(c / kWtChunks) * IMG;
        const int kc = c % kWtChunks;
        *reinterpret_cast<uint4 *>(img + wt_boff(t, kc)) = make_uint4(th[0], th[1], th[2], th[3]);
        *reinterpret_cast<uint4 *>(img + wt_boff(PS + t, kc)) = make_uint4(tm[0], tm[1], tm[2], tm[3]);
        *reinterpret_cast<uint4 *>(img + wt_boff(2 * PS + t, kc)) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
    };
#pragma unroll
    for (int j = 0; j < kWtTermChunks; j++) {
        const int c = c_lo + tid + kWtTermThreads * j;
        if (c < c_hi) emit(c, v[j]);
    }
    for (int c = c_lo + tid + kWtTermThreads * kWtTermChunks; c < c_hi; c += kWtTermThreads) {
        float u[8];
        load(c, u);
        emit(c, u);
    }
}

// The epilogue: warps 0 .. 3, thread = weight row (tensor-memory lane 32 warp
// + lane), add each token's three accumulators, (lo + mid) + hi, and scale by
// s (and, given `tscale`, the token's power of two as two factors).  With
// split K the partial tiles go to shared memory (the weight stages, free by
// now) and the cluster's CTAs share out (token, 4 rows) items, adding the
// partials of each in rank order.
template <int PS, int THREADS>
__device__ __forceinline__ void wt_epilogue(uint8_t *sm, uint32_t tmem, bool ok, float *__restrict__ y, float s,
                                            const float2 *__restrict__ tscale, int M, int N, int TT, int m0, int n0,
                                            int split, int z) {
    constexpr int NC = (3 * PS + 15) / 16 * 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float nanv = ok ? 0.0f : __int_as_float(0x7fc00000);  // a wait that gave up: the tile reads NaN
    float *const part = reinterpret_cast<float *>(sm);
    if (warp < 4) {
        const int rr = 32 * warp + lane, n = n0 + rr;
        uint32_t d[NC];
#pragma unroll
        for (int c = 0; c < NC; c += 16)
            tm_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, *reinterpret_cast<uint32_t(*)[16]>(d + c));
#pragma unroll
        for (int t = 0; t < PS; t++) {
            if (t >= TT) break;
            float v = __fadd_rn(__fadd_rn(__fadd_rn(__uint_as_float(d[2 * PS + t]), __uint_as_float(d[PS + t])),
                                          __uint_as_float(d[t])),
                                nanv);
            if (tscale && m0 + t < M) {
                const float2 ts = tscale[m0 + t];
                v = __fmul_rn(__fmul_rn(v, ts.x), ts.y);
            }
            if (split == 1) {
                if (m0 + t < M && n < N) y[(int64_t)(m0 + t) * N + n] = __fmul_rn(v, s);
            } else {
                part[t * kWtPStride + rr] = v;
            }
        }
    }
    if (split > 1) {
        cluster_sync();
        const int items = TT * (kWtRows / 4);
        const int e_lo = items * z / split, e_hi = items * (z + 1) / split;
        const bool vec_y = (reinterpret_cast<uintptr_t>(y) & 15) == 0 && N % 4 == 0;
        for (int e = e_lo + tid; e < e_hi; e += THREADS) {
            const int t = e / (kWtRows / 4), c4 = e % (kWtRows / 4);
            const int m = m0 + t, nb = n0 + 4 * c4;
            if (m >= M || nb >= N) continue;
            float4 u[kWtMaxSplit];
#pragma unroll
            for (int q = 0; q < kWtMaxSplit; q++)
                if (q < split) u[q] = ld_peer_f4(&part[t * kWtPStride + 4 * c4], (uint32_t)q);
            float4 v = u[0];
#pragma unroll
            for (int q = 1; q < kWtMaxSplit; q++)
                if (q < split) {
                    v.x = __fadd_rn(v.x, u[q].x);
                    v.y = __fadd_rn(v.y, u[q].y);
                    v.z = __fadd_rn(v.z, u[q].z);
                    v.w = __fadd_rn(v.w, u[q].w);
                }
            const float o[4] = {__fmul_rn(v.x, s), __fmul_rn(v.y, s), __fmul_rn(v.z, s), __fmul_rn(v.w, s)};
            float *const dst = y + (int64_t)m * N + nb;
            if (vec_y && nb + 4 <= N) {
                *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
                for (int q = 0; q < 4; q++)
                    if (nb + q < N) dst[q] = o[q];
            }
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
    }
}

// Grid: (token tiles, weight-row tiles, split); a cluster is the `split` CTAs
// of one tile.  PS: the tile's token capacity (4, 8 or 16); the B operand's
// rows are term p of token t at p PS + t, N = 3 PS rounded up to 16.  PRE:
// the B images of w8_terms_kernel in `imgs` (fp16, scaled per token by
// tscale); otherwise the splitter warps build bf16 B operands from x.
// Warps: converters 0 .. 7, then the splitters (4) or the B-copy warp (PRE),
// the MMA warp, the weight-copy warp.
template <int PS, bool PRE>
__global__ void __launch_bounds__(WtLayout<PRE>::kThreads, 2)
    w8_tm_kernel(const __grid_constant__ CUtensorMap wmap, const float *__restrict__ x, const uint8_t *__restrict__ imgs, const float2 *__restrict__ tscale,
                 float s, float *__restrict__ y, int M, int N, int K, int TT, int split) {
    using L = WtLayout<PRE>;
    constexpr int NC = (3 * PS + 15) / 16 * 16;  // MMA N: accumulator columns
    constexpr int IMG = wt_img_bytes(PS);
    constexpr int kRoleWarps = PRE ? 1 : kWtXWarps;
    constexpr int kMmaWarp = kWtConvWarps + kRoleWarps, kCopyWarp = kMmaWarp + 1;
    extern __shared__ __align__(1024) uint8_t wt_smem_buf[];
    uint8_t *const sm = wt_smem_buf;
    WtCtl &C = *reinterpret_cast<WtCtl *>(sm + L::kCtl);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * TT, n0 = blockIdx.y * kWtRows;
    if ((smem_addr(sm) & 1023u) != 0) {  // the swizzle would not match: the tile reads NaN (the same in every CTA)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int e = tid; e < TT * kWtRows; e += L::kThreads) {
            const int m = m0 + e / kWtRows, n = n0 + e % kWtRows;
            if (m < M && n < N) y[(int64_t)m * N + n] = __int_as_float(0x7fc00000);
        }
        return;
    }
    const int z = split > 1 ? (int)cluster_rank() : 0;
    const int nstg = (K + kWtKS - 1) / kWtKS;
    const int g_lo = (int)((int64_t)nstg * z / split), g_hi = (int)((int64_t)nstg * (z + 1) / split);
    const int ng = g_hi - g_lo;
    const uint64_t pol = l2_evict_first();

    // Programmatic dependent launch: the next kernel on the stream may start
    // its set-up now.  Weights are read-only inputs, so their copies start at
    // once (below, before the block's set-up is done); every read of x or of
    // the images and every write of y waits for the previous kernel.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == kCopyWarp && lane == 0) {
        for (int i = 0; i < kWtRaw; i++) {
            mbar_init(&C.wfull[i], 1);
            mbar_init(&C.wempty[i], kWtConvWarps);
        }
        for (int i = 0; i < kWtSlots; i++) {
            mbar_init(&C.full[i], kWtConvWarps + (PRE ? 0 : kWtXWarps));
            mbar_init(&C.mma_done[i], 1);
        }
        for (int i = 0; i < kWtBRing; i++) {
            mbar_init(&C.bfull[i], 1);
            mbar_init(&C.bempty[i], 1);
        }
        C.abort = 0;
        C.issued = 0;
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
        for (int g = 0; g < kWtRaw && g < ng; g++) {
            mbar_arrive_expect_tx(&C.wfull[g], (uint32_t)kWtWStage);
            tma_load_2d(sm + g * kWtWStage, &wmap, (g_lo + g) * kWtKS, n0, &C.wfull[g], pol);
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&C.tmem)),
                     "r"(kWtCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = C.tmem;
    volatile int *abort = &C.abort;

    if (warp == kCopyWarp) {
        // ---- weight-copy warp: lane 0 streams the rest of the weight stages
        if (lane == 0) {
            int g = kWtRaw;
            for (; g < ng; g++) {
                const int rs = g % kWtRaw;
                if (!mbar_wait(&C.wempty[rs], (uint32_t)(g / kWtRaw - 1) & 1u)) {
                    *abort = 1;
                    break;
                }
                if (*abort) break;
                mbar_arrive_expect_tx(&C.wfull[rs], (uint32_t)kWtWStage);
                tma_load_2d(sm + rs * kWtWStage, &wmap, (g_lo + g) * kWtKS, n0, &C.wfull[rs], pol);
            }
            // every copy issued has landed before the stages are reused or the CTA leaves
            g = g < ng ? g : ng;
            for (int u = g > kWtRaw ? g - kWtRaw : 0; u < g; u++)
                mbar_wait(&C.wfull[u % kWtRaw], (uint32_t)(u / kWtRaw) & 1u);
        }
    } else if (warp == kMmaWarp) {
        // ---- MMA warp: lane 0 issues each stage's eight MMAs once the A slot
        // (and the B operand) is ready, and commits them to the slot's mma_done
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (PRE ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)(NC >> 3) << 17) |
                                   ((uint32_t)(kWtRows >> 4) << 24);  // fp32 D, fp16 (bf16) A and B, K-major
            for (int g = 0; g < ng && !*abort; g++) {
                const int sl = g % kWtSlots, bs = PRE ? g % kWtBRing : sl;
                if (!mbar_wait(&C.full[sl], (uint32_t)(g / kWtSlots) & 1u) ||
                    (PRE && !mbar_wait(&C.bfull[bs], (uint32_t)(g / kWtBRing) & 1u))) {
                    *abort = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t bd = desc_kmajor(smem_addr(sm + L::kB + bs * kWtBMax), 128u, (uint32_t)kWtSBO);
                const uint32_t a0 = tmem + kWtACol + 64u * (uint32_t)sl;
#pragma unroll
                for (int u = 0; u < kWtKS / 16; u++)  // K = 16: 8 A columns, 2 B core matrices (256 bytes)
                    tm_mma(tmem, a0 + 8u * u, bd + (uint64_t)(16 * u), idesc, (g > 0 || u > 0) ? 1u : 0u);
                tc_commit(&C.mma_done[sl]);
                if (PRE) tc_commit(&C.bempty[bs]);
                *reinterpret_cast<volatile int *>(&C.issued) = g + 1;
            }
        }
    } else if (warp < kWtConvWarps) {
        // ---- converter warps: thread = weight row r (tensor-memory lane r),
        // bytes 64 hh .. 64 hh + 63 of each stage
        const int q4 = warp & 3, hh = warp >> 2, r = 32 * q4 + lane;
        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16) + kWtACol + 32u * (uint32_t)hh;
        const uint32_t sw = (uint32_t)(r & 7);  // the 128-byte swizzle: chunk c of row r sits at chunk c ^ (r % 8)
        for (int g = 0; g < ng; g++) {
            if (__any_sync(0xffffffffu, *abort != 0)) break;
            const int rs = g % kWtRaw, sl = g % kWtSlots;
            if (!__all_sync(0xffffffffu, mbar_wait(&C.wfull[rs], (uint32_t)(g / kWtRaw) & 1u))) {
                *abort = 1;
                break;
            }
            const uint8_t *row = sm + rs * kWtWStage + r * kWtKS;
            uint4 c[4];
#pragma unroll
            for (int j = 0; j < 4; j++) c[j] = lds128(row + (((4u * hh + j) ^ sw) << 4));
            __syncwarp();  // the stage is read: the copy warp may refill it
            if (lane == 0) mbar_arrive(&C.wempty[rs]);
            // the MMAs of stage g - kWtSlots read this A slot: wait until they are done
            if (g >= kWtSlots &&
                !__all_sync(0xffffffffu, mbar_wait(&C.mma_done[sl], (uint32_t)(g / kWtSlots - 1) & 1u))) {
                *abort = 1;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const uint32_t wv[8] = {c[2 * half].x,     c[2 * half].y,     c[2 * half].z,     c[2 * half].w,
                                        c[2 * half + 1].x, c[2 * half + 1].y, c[2 * half + 1].z, c[2 * half + 1].w};
                uint32_t h[16];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    if (PRE) {
                        const uint32_t f = wv[q] ^ 0x80808080u;
                        h[2 * q] = wt_i8x2_f16(f, 0x4140u);
                        h[2 * q + 1] = wt_i8x2_f16(f, 0x4342u);
                    } else {
                        h[2 * q] = wt_i8x2_bf16(wv[q], 0x4140u);
                        h[2 * q + 1] = wt_i8x2_bf16(wv[q], 0x4342u);
                    }
                }
                tm_st16(ta + 64u * (uint32_t)sl + 16u * (uint32_t)half, h);
            }
            tm_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[sl]);
        }
    } else if (PRE) {
        // ---- B-copy warp: lane 0 brings each stage's image in (one bulk
        // copy) once the MMAs that read its slot before are done
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the images are written
            const uint8_t *const img0 = imgs + ((int64_t)blockIdx.x * nstg + g_lo) * IMG;
            int g = 0;
            for (; g < ng && !*abort; g++) {
                const int bs = g % kWtBRing;
                if (g >= kWtBRing && !mbar_wait(&C.bempty[bs], (uint32_t)(g / kWtBRing - 1) & 1u)) {
                    *abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&C.bfull[bs], (uint32_t)IMG);
                bulk_g2s_l2(sm + L::kB + bs * kWtBMax, img0 + (int64_t)g * IMG, (uint32_t)IMG, &C.bfull[bs]);
            }
            for (int u = g > kWtBRing ? g - kWtBRing : 0; u < g; u++)
                mbar_wait(&C.bfull[u % kWtBRing], (uint32_t)(u / kWtBRing) & 1u);
        }
    } else {
        // ---- splitter warps: the tile's activations of each stage, copied
        // kWtXDepth - 1 stages ahead (each thread reads back only its own copies)
        const int xt = tid - 32 * kWtConvWarps;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && K % 4 == 0;
        const int units = TT * kWtChunks;  // (token, 8 activations) per stage
        auto fetch = [&](int g) {
            if (g < ng) {
                uint8_t *const dst0 = sm + L::kX + (g % kWtXDepth) * kWtXStage;
                const int kb = (g_lo + g) * kWtKS;
#pragma unroll
                for (int uu = 0; uu < kWtUnits; uu++) {
                    const int u = xt + kWtXThreads * uu;
                    if (u >= units) break;
                    const int t = u % TT, kc = u / TT, m = m0 + t, k = kb + 8 * kc;
                    uint8_t *const dst = dst0 + u * 16;
                    const float *src = x + (int64_t)(m < M ? m : 0) * K;
                    if (vec) {
#pragma unroll
                        for (int q = 0; q < 2; q++) {  // K % 4 == 0: four activations are all inside K or all past it
                            const int kk = k + 4 * q;
                            const bool in = m < M && kk < K;
                            cp_async16(dst + kWtXHalf * q, in ? src + kk : x, in ? 16 : 0);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const int kk = k + e;
                            const bool in = m < M && kk < K;
                            cp_async4(dst + kWtXHalf * (e >> 2) + 4 * (e & 3), in ? src + kk : x, in ? 4 : 0);
                        }
                    }
                }
            }
            cp_async_commit();
        };
#pragma unroll 1
        for (int g = 0; g < kWtXDepth - 1; g++) fetch(g);
        for (int g = 0; g < ng; g++) {
            if (__any_sync(0xffffffffu, *abort != 0)) break;
            fetch(g + kWtXDepth - 1);
            cp_async_wait_pending<kWtXDepth - 1>();  // this thread's copies of stage g have landed
            const int sl = g % kWtSlots;
            bool ok = true;
            if (g >= kWtSlots) ok = mbar_wait(&C.mma_done[sl], (uint32_t)(g / kWtSlots - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                *abort = 1;
                break;
            }
            tc_fence_after();
            const uint8_t *const src0 = sm + L::kX + (g % kWtXDepth) * kWtXStage;
            uint8_t *const bt = sm + L::kB + sl * kWtBMax;
#pragma unroll
            for (int uu = 0; uu < kWtUnits; uu++) {
                const int u = xt + kWtXThreads * uu;
                if (u >= units) break;
                const int t = u % TT, kc = u / TT;  // lanes: consecutive tokens, so the stores fill whole rows of banks
                const uint4 va = lds128(src0 + u * 16), vb = lds128(src0 + kWtXHalf + u * 16);
                const float v[8] = {__uint_as_float(va.x), __uint_as_float(va.y), __uint_as_float(va.z),
                                    __uint_as_float(va.w), __uint_as_float(vb.x), __uint_as_float(vb.y),
                                    __uint_as_float(vb.z), __uint_as_float(vb.w)};
                uint32_t th[4], tm[4], tl[4];
#pragma unroll
                for (int e = 0; e < 4; e++) wt_split_bf16(v[2 * e], v[2 * e + 1], th[e], tm[e], tl[e]);
                sts128(bt + wt_boff(t, kc), th[0], th[1], th[2], th[3]);
                sts128(bt + wt_boff(PS + t, kc), tm[0], tm[1], tm[2], tm[3]);
                sts128(bt + wt_boff(2 * PS + t, kc), tl[0], tl[1], tl[2], tl[3]);
            }
            // the generic-proxy writes above, visible to the tensor core (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[sl]);
        }
        cp_async_wait_pending<0>();
    }
    // the last commit covers every MMA issued before it
    __syncthreads();
    const int issued = C.issued;
    if (issued > 0) {
        const int i = issued - 1;
        if (!mbar_wait(&C.mma_done[i % kWtSlots], (uint32_t)(i / kWtSlots) & 1u)) *abort = 1;
    }
    __syncthreads();
    const bool ok = !*abort && issued == ng;
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // y may be read by the previous kernel until it ends
    wt_epilogue<PS, L::kThreads>(sm, tmem, ok, y, s, PRE ? tscale : nullptr, M, N, TT, m0, n0, split, z);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kWtCols) : "memory");
}

// The weights' tensor map: uint8 [N][K] with row pitch `pitch` bytes, boxes of
// 128 bytes x 128 rows, 128-byte swizzle, zeros out of range.  Encoded through
// the driver entry point (no link against the driver library); recent maps are
// kept for the next call on the same weights.
qlin_status w8_weight_map(const int8_t *w, int64_t pitch, int N, int K, CUtensorMap *out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::map<std::tuple<int, const void *, int64_t, int, int>, CUtensorMap> cache;
    int dev = 0;
    QLIN_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_tuple(dev, (const void *)w, pitch, N, K);
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
    const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)pitch};
    const cuuint32_t box[2] = {(cuuint32_t)kWtKS, (cuuint32_t)kWtRows};
    const cuuint32_t estride[2] = {1, 1};
    CUtensorMap m;
    const CUresult r = encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(w), gdim, gstride, box, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    QLIN_REQUIRE(r == CUDA_SUCCESS, QLIN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    if (cache.size() >= 256) cache.clear();
    cache[key] = m;
    *out = m;
    return QLIN_OK;
}

// Token tiling: tiles of at most kWtMaxTT tokens, capacity PS (4, 8 or 16).
void wt_tiles(int M, int &tiles_m, int &TT, int &PS) {
    tiles_m = (M + kWtMaxTT - 1) / kWtMaxTT;
    TT = (M + tiles_m - 1) / tiles_m;
    PS = TT <= 4 ? 4 : TT <= 8 ? 8 : 16;
}

// The split of K: the largest split (a cluster of at most kWtMaxSplit CTAs
// over one weight-row tile) whose CTAs all fit at once, two to an SM.  No
// cluster waits on another, so a CTA that does not fit only waits for an SM.
// (The runtime's occupancy calculator reports one CTA of these kernels per
// SM; two share an SM by their shared memory and tensor-memory sizes.)
int wt_choose_split(int ntiles, int nstg) {
    for (int c = kWtMaxSplit; c >= 2; c--)
        if (c <= nstg && ntiles * c <= 2 * sm_count()) return c;
    return 1;
}

template <int PS, bool PRE>
qlin_status launch_wt(const CUtensorMap &map, const float *x, const uint8_t *imgs,
                      const float2 *tscale, float s, float *y, int M, int N, int K, int TT, int tiles_m,
                      cudaStream_t st) {
    auto kern = w8_tm_kernel<PS, PRE>;
    constexpr int smem = wt_smem<PRE>();
    // two CTAs of this size fit on an SM only with the largest shared-memory carveout
    static std::once_flag carve;
    std::call_once(carve, [kern] {
        (void)cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
    });
    (void)blocks_per_sm((const void *)kern, smem);  // raises the dynamic shared-memory limit
    const int tiles_n = (N + kWtRows - 1) / kWtRows;
    const int nstg = (K + kWtKS - 1) / kWtKS;
    const int split = wt_choose_split(tiles_n * tiles_m, nstg);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles_m, (unsigned)tiles_n, (unsigned)split);
    cfg.blockDim = dim3(WtLayout<PRE>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)split;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, kern, map, x, imgs, tscale, s, y, M, N, K, TT, split));
    QLIN_LAUNCHED("w8_tm_kernel");
    return QLIN_OK;
}

template <int PS>
qlin_status launch_terms(const float *x, int M, int K, int TT, uint8_t *imgs, float2 *tscale, cudaStream_t st) {
    // CTAs per token: enough that each thread holds its chunks in registers
    const int nchunks = (K + kWtKS - 1) / kWtKS * kWtChunks;
    int P = (nchunks + kWtTermThreads * kWtTermChunks - 1) / (kWtTermThreads * kWtTermChunks);
    P = P < 1 ? 1 : P > kWtTermMaxP ? kWtTermMaxP : P;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, (unsigned)M);
    cfg.blockDim = dim3(kWtTermThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)P;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = P > 1 ? 2 : 1;  // one CTA per token (K <= 16384) needs no cluster
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, w8_terms_kernel<PS>, x, M, K, TT, (K + kWtKS - 1) / kWtKS, imgs, tscale));
    QLIN_LAUNCHED("w8_terms_kernel");
    return QLIN_OK;
}

}  // namespace

// Workspace of w8_linear_tensor_cores_ws: the B images of every token tile
// and stage, then the tokens' powers of two.
size_t w8_tc_workspace_bytes(int M, int K) {
    if (M < 2 || M > 64 || K < 1) return 0;
    int tiles_m = 0, TT = 0, PS = 0;
    wt_tiles(M, tiles_m, TT, PS);
    const size_t nstg = ((size_t)K + kWtKS - 1) / kWtKS;
    return ((size_t)tiles_m * nstg * wt_img_bytes(PS) + 15) / 16 * 16 + ((size_t)M * 8 + 15) / 16 * 16;
}

// y [M][N] = s * x [M][K] . w8 [N][K]^T for 2 <= M <= 64 on the tensor cores,
// the activations split in the product kernel.  Token tiles of at most 16
// tokens; the tile's capacity (4, 8 or 16) sets the MMA's N (16, 32 or 48).
qlin_status w8_linear_tensor_cores(const float *x, const int8_t *w8, int64_t pitch, float s, float *y, int M, int N,
                                   int K, cudaStream_t st) {
    QLIN_REQUIRE(M >= 2 && M <= 64, QLIN_ERR_UNSUPPORTED, "w8_linear_tensor_cores: M=%d", M);
    CUtensorMap map;
    if (qlin_status e = w8_weight_map(w8, pitch, N, K, &map)) return e;
    int tiles_m = 0, TT = 0, PS = 0;
    wt_tiles(M, tiles_m, TT, PS);
    if (PS == 4) return launch_wt<4, false>(map, x, nullptr, nullptr, s, y, M, N, K, TT, tiles_m, st);
    if (PS == 8) return launch_wt<8, false>(map, x, nullptr, nullptr, s, y, M, N, K, TT, tiles_m, st);
    return launch_wt<16, false>(map, x, nullptr, nullptr, s, y, M, N, K, TT, tiles_m, st);
}

// The same with the workspace path (w8_terms_kernel, then the product on its
// images); work: w8_tc_workspace_bytes bytes, 16-byte aligned.
qlin_status w8_linear_tensor_cores_ws(const float *x, const int8_t *w8, int64_t pitch, float s, float *y, int M,
                                      int N, int K, void *work, cudaStream_t st) {
    QLIN_REQUIRE(M >= 2 && M <= 64, QLIN_ERR_UNSUPPORTED, "w8_linear_tensor_cores_ws: M=%d", M);
    CUtensorMap map;
    if (qlin_status e = w8_weight_map(w8, pitch, N, K, &map)) return e;
    int tiles_m = 0, TT = 0, PS = 0;
    wt_tiles(M, tiles_m, TT, PS);
    const int nstg = (K + kWtKS - 1) / kWtKS;
    uint8_t *const imgs = static_cast<uint8_t *>(work);
    float2 *const tscale =
        reinterpret_cast<float2 *>(imgs + ((size_t)tiles_m * nstg * wt_img_bytes(PS) + 15) / 16 * 16);
    qlin_status e = QLIN_OK;
    if (PS == 4) {
        if ((e = launch_terms<4>(x, M, K, TT, imgs, tscale, st))) return e;
        return launch_wt<4, true>(map, x, imgs, tscale, s, y, M, N, K, TT, tiles_m, st);
    }
    if (PS == 8) {
        if ((e = launch_terms<8>(x, M, K, TT, imgs, tscale, st))) return e;
        return launch_wt<8, true>(map, x, imgs, tscale, s, y, M, N, K, TT, tiles_m, st);
    }
    if ((e = launch_terms<16>(x, M, K, TT, imgs, tscale, st))) return e;
    return launch_wt<16, true>(map, x, imgs, tscale, s, y, M, N, K, TT, tiles_m, st);
}

}  // namespace qlin
