// The greedy output layer for many lanes at once ([llama2.c] Step 6 and
// "Sampling", one token per lane of a step of [citric] "Many users at once"):
// logits[u][r] = sum_k E[r][k] x_u[k] over the bf16 table, next[u] = the first
// index of the maximum.  The table is read once for all lanes.
//
// Tensor cores: the product is a matrix product [rows x K] x [K x lanes].  One
// tcgen05.mma (kind::f16, bf16 operands, fp32 accumulator in tensor memory)
// takes 128 table rows (M) against N = 3 * Up columns: each lane's x enters as
// three bf16 terms, x = hi + mid + lo with hi = bf16(x), mid = bf16(x - hi),
// lo = bf16(x - hi - mid) (each difference exact in fp32), so the three
// partial logits carry x to 24 bits and their fp32 sum (hi + mid) + lo is
// within fp32 rounding of the fp32 dot product.  One persistent CTA per SM
// walks its row tiles: K advances 64 elements a step through four
// shared-memory stages (table rows by cp.async from 256 loader threads into
// the no-swizzle K-major core-matrix layout; the lanes' operand as one bulk
// copy of the image the split kernel prepared), one thread issues each step's
// four MMAs, and two accumulators alternate between tiles so that four
// epilogue warps reduce one tile (each lane's logits, its best row) while the
// next is multiplied.  The last CTA reduces the CTAs' bests per lane.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {
namespace {

constexpr int kLlRows = 128;              // table rows per CTA (MMA M)
constexpr int kLlKS = 64;                 // K elements per step
constexpr int kLlChunks = kLlKS / 8;      // 16-byte core-matrix columns per row and step
constexpr int kLlSBO = kLlChunks * 128;   // bytes between 8-row groups
constexpr int kLlStages = 5;
constexpr int kLlEpiWarps = 4;  // read a finished tile's accumulator (one per tensor-memory lane quarter)
constexpr int kLlThreads = 64 + 32 * kLlEpiWarps;  // the copy warp, the MMA warp, the epilogue warps
constexpr int kLlMaxLanes = 64;              // lanes per pass: 3 x 64 = 192 accumulator columns
constexpr int kLlMaxN = 3 * kLlMaxLanes;
constexpr uint32_t kLlCols = 512;            // tensor-memory columns: two accumulators, at 0 and 256
constexpr int kLlAccStride = 256;
constexpr int kLlATile = kLlRows * kLlKS * 2;     // 16 KB: 128 table rows x 64 inputs, 128-byte swizzled
constexpr int kLlBTile = kLlMaxN / 8 * kLlSBO;    // 24 KB: the lanes' operand of a step

struct LlSmem {  // 1024-byte aligned (the swizzled table tiles)
    uint8_t a[kLlStages][kLlATile];  // table rows of a step, as the tensor copy writes them
    uint8_t b[kLlStages][kLlBTile];  // the lanes' split x of a step
    uint64_t full[kLlStages];        // the stage has landed (one arrival + the bytes of both copies)
    uint64_t mma_done[kLlStages];    // the MMAs reading the stage are done (tcgen05.commit)
    uint64_t acc_full[2];            // accumulator b holds a finished tile (tcgen05.commit)
    uint64_t acc_empty[2];           // the epilogue warps have read accumulator b
    float2 wbest[kLlEpiWarps][kLlMaxLanes];  // a tile's best (value, row) per lane from each epilogue warp
    float2 cbest[kLlMaxLanes];               // this CTA's best per lane over its tiles so far
    uint32_t tmem;
    int abort;
    int last;
};

// Descriptor of a table tile: K-major, 128-byte swizzle (the layout of the
// tensor copy with CU_TENSOR_MAP_SWIZZLE_128B: row r at 128 r, its 16-byte
// chunk c at chunk c ^ (r % 8)), 8-row groups 1024 bytes apart; the start
// advances 32 bytes per 16 inputs inside the swizzle atom.
__device__ __forceinline__ uint64_t ll_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;                         // leading byte offset (unused for this layout)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // next 8-row group
    d |= (uint64_t)1 << 46;                         // descriptor version
    d |= (uint64_t)2 << 61;                         // 128-byte swizzle
    return d;
}

// 2-D tensor copy (tile mode; out-of-range rows read as zeros) completing on bar
__device__ __forceinline__ void ll_tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t ll_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 16;                // next core matrix along K
    d |= (uint64_t)(((uint32_t)kLlSBO >> 4) & 0x3FFFu) << 32;   // next 8-row group
    d |= (uint64_t)1 << 46;
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both
// K-major, N columns, M = 128 rows
__device__ __forceinline__ uint32_t ll_idesc(int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kLlRows >> 4) << 24);
}

__device__ __forceinline__ void ll_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void ll_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 8 consecutive accumulator columns of this thread's tensor-memory lane (no wait)
__device__ __forceinline__ void ll_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ int ll_off(int r, int kc) { return (r >> 3) * kLlSBO + kc * 128 + (r & 7) * 16; }

__device__ __forceinline__ bool ll_better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// x [U][K] fp32 -> the lanes' operand of every K step as the image of its
// shared-memory stage: N = 3 Up rows (row t Up + u: term t of lane u, the terms
// hi, mid, lo), step s at xs + s N 64 elements in the K-major core-matrix
// layout; zero for lanes U..Up-1 and past K.
__global__ void lm_lanes_split_kernel(const float *__restrict__ x, int U, int Up, int K, int nsteps,
                                      uint16_t *__restrict__ xs) {
    const int u = blockIdx.x, N = 3 * Up;
    for (int k = threadIdx.x; k < nsteps * kLlKS; k += blockDim.x) {
        const float v = (u < U && k < K) ? x[(int64_t)u * K + k] : 0.0f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = __fsub_rn(v, __bfloat162float(hi));
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = __fsub_rn(r1, __bfloat162float(mid));
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        const int st = k / kLlKS, kc = (k % kLlKS) / 8, e = k % 8;
        uint16_t *img = xs + (int64_t)st * N * kLlKS;
        img[(ll_off(0 * Up + u, kc) >> 1) + e] = __bfloat16_as_ushort(hi);
        img[(ll_off(1 * Up + u, kc) >> 1) + e] = __bfloat16_as_ushort(mid);
        img[(ll_off(2 * Up + u, kc) >> 1) + e] = __bfloat16_as_ushort(lo);
    }
}

// L2 policy for data every CTA reads again: keep it.
__device__ __forceinline__ uint64_t ll_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

struct LlArgs {
    const uint16_t *emb;  // [V][K]
    const uint16_t *xs;   // the split kernel's step images, [ceil(K/64)][3 Up x 64]
    int V, K, U, Up;
    float *logits;        // [U][V] or null
    int32_t *next;        // [U]
    float2 *part;         // [gridDim][kLlMaxLanes]
    unsigned *ticket;
    int32_t *status;
};

// Persistent: CTA c takes row tiles c, c + gridDim.x, ... (128 rows each).  The
// K steps of all its tiles form one sequence g = tile * nsteps + step through
// the stage ring, so the copies of the next tile start while the current one
// is multiplied.  Two accumulators alternate between tiles: the epilogue warps
// read tile i's (each lane's logits, its best row) while the MMAs of tile i + 1
// run.  Each lane's best over the CTA's tiles stays in shared memory; the last
// CTA to finish takes every lane's best over the CTAs (ties to the lower row).
__global__ void __launch_bounds__(kLlThreads, 1) lm_lanes_kernel(const __grid_constant__ CUtensorMap tmap, LlArgs A) {
    extern __shared__ uint8_t ll_smem_raw[];
    // the swizzled table tiles want a 1024-byte aligned base (the launch adds 1 KB)
    uint8_t *const ll_base = ll_smem_raw + ((1024u - (smem_addr(ll_smem_raw) & 1023u)) & 1023u);
    LlSmem &S = *reinterpret_cast<LlSmem *>(ll_base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = A.K, Up = A.Up, N = 3 * Up;
    const int nsteps = (K + kLlKS - 1) / kLlKS;
    const int ntiles = (A.V + kLlRows - 1) / kLlRows;
    const int my_tiles = ntiles > (int)blockIdx.x ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * nsteps;  // steps of this CTA
    auto tile_row0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) * kLlRows; };
    const uint32_t bbytes = (uint32_t)N * kLlKS * 2;  // the lanes' operand of one step

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(kLlCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int i = 0; i < kLlStages; i++) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.mma_done[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&S.acc_full[i], 1);
            mbar_init(&S.acc_empty[i], 32 * kLlEpiWarps);
        }
        S.abort = 0;
        fence_mbar_init();
    }
    if (tid < kLlMaxLanes) S.cbest[tid] = make_float2(-__int_as_float(0x7f800000), __int_as_float(0x7fffffff));
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = S.tmem;
    volatile int *abort = &S.abort;

    if (warp == 0) {
        // ---- copies: step g's table tile (one tensor copy) and lanes operand
        // (one bulk copy) into stage g % S once the MMAs of step g - S are done
        if (lane == 0) {
            const uint64_t keep = ll_evict_last();
            for (int g = 0; g < total && !*abort; g++) {
                const int st = g % kLlStages;
                if (g >= kLlStages && !mbar_wait(&S.mma_done[st], (uint32_t)(g / kLlStages - 1) & 1u)) {
                    *abort = 1;
                    raise_status(A.status, kStatusTimeout);
                    break;
                }
                mbar_arrive_expect_tx(&S.full[st], (uint32_t)kLlATile + bbytes);
                ll_tma_2d(S.a[st], &tmap, (g % nsteps) * kLlKS, tile_row0(g / nsteps), &S.full[st]);
                bulk_g2s(S.b[st], A.xs + (int64_t)(g % nsteps) * N * kLlKS, bbytes, &S.full[st], keep);
            }
        }
    } else if (warp == 1) {
        // ---- lane 0 issues each step's four MMAs into the tile's accumulator
        if (lane == 0) {
            const uint32_t idesc = ll_idesc(N);
            for (int g = 0; g < total && !*abort; g++) {
                const int ti = g / nsteps, t = g % nsteps, buf = ti & 1;
                // the accumulator of tile ti - 2 must have been read out
                if (t == 0 && ti >= 2 && !mbar_wait(&S.acc_empty[buf], (uint32_t)((ti >> 1) - 1) & 1u)) {
                    *abort = 1;
                    raise_status(A.status, kStatusTimeout);
                    break;
                }
                const int st = g % kLlStages;
                if (!mbar_wait(&S.full[st], (uint32_t)(g / kLlStages) & 1u)) {
                    *abort = 1;
                    raise_status(A.status, kStatusTimeout);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a0 = smem_addr(S.a[st]), b0 = smem_addr(S.b[st]);
                const uint32_t dacc = tmem + (uint32_t)(buf * kLlAccStride);
#pragma unroll
                for (int kk = 0; kk < kLlKS / 16; kk++)  // K = 16: 32 bytes of a table row, 2 core-matrix columns of x
                    ll_mma(dacc, ll_desc_sw128(a0 + 32u * kk), ll_desc(b0 + 256u * kk), idesc,
                           (t > 0 || kk > 0) ? 1u : 0u);
                ll_commit(&S.mma_done[st]);
                if (t == nsteps - 1) ll_commit(&S.acc_full[buf]);
            }
        }
    } else {
        // ---- epilogue warps: warp w reads tensor-memory lanes 32 (w % 4) .. + 31,
        // i.e. those rows of each finished tile
        const int ew = warp - 2;
        const int q = warp & 3;
        for (int ti = 0; ti < my_tiles; ti++) {
            const int buf = ti & 1;
            uint32_t fail = *abort != 0;
            if (!fail && !mbar_wait(&S.acc_full[buf], (uint32_t)(ti >> 1) & 1u)) {
                fail = 1;
                *abort = 1;
                raise_status(A.status, kStatusTimeout);
            }
            // one decision for all epilogue warps (they meet at named barriers below)
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(fail)
                : "r"(fail), "n"(32 * kLlEpiWarps)
                : "memory");
            if (fail) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int row = tile_row0(ti) + 32 * q + lane;
            const bool row_ok = row < A.V;
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kLlAccStride);
            for (int u0 = 0; u0 < Up; u0 += 8) {
                uint32_t hi[8], mid[8], lo[8];
                ll_ld8(tb + (uint32_t)u0, hi);
                ll_ld8(tb + (uint32_t)(Up + u0), mid);
                ll_ld8(tb + (uint32_t)(2 * Up + u0), lo);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                float bv[8];
                int bi[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int u = u0 + j;
                    const float v = __fadd_rn(__fadd_rn(__uint_as_float(hi[j]), __uint_as_float(mid[j])),
                                              __uint_as_float(lo[j]));
                    const bool ok = row_ok && u < A.U;
                    if (ok && A.logits) A.logits[(int64_t)u * A.V + row] = v;
                    bv[j] = ok ? v : -__int_as_float(0x7f800000);
                    bi[j] = ok ? row : 0x7fffffff;
                }
                // (value, row) is a total order: the reduction order does not matter
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv[j], off);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi[j], off);
                        if (ll_better(ov, oi, bv[j], bi[j])) bv[j] = ov, bi[j] = oi;
                    }
                if (lane == 0)
#pragma unroll
                    for (int j = 0; j < 8; j++) S.wbest[ew][u0 + j] = make_float2(bv[j], __int_as_float(bi[j]));
            }
            // the accumulator is read: the MMAs of tile ti + 2 may overwrite it
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&S.acc_empty[buf]);
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kLlEpiWarps) : "memory");
            if (ew == 0)
                for (int u = lane; u < A.U; u += 32) {
                    float2 b = S.cbest[u];
#pragma unroll
                    for (int w = 0; w < kLlEpiWarps; w++) {
                        const float2 c = S.wbest[w][u];
                        if (ll_better(c.x, __float_as_int(c.y), b.x, __float_as_int(b.y))) b = c;
                    }
                    S.cbest[u] = b;
                }
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kLlEpiWarps) : "memory");  // wbest is free for the next tile
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kLlCols) : "memory");
    if (tid < A.U) A.part[(int64_t)blockIdx.x * kLlMaxLanes + tid] = S.cbest[tid];
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        S.last = atomicAdd(A.ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!S.last) return;
    __threadfence();
    // the last CTA: every lane's best over all CTAs (ties to the lower row)
    {
        for (int u = warp; u < A.U; u += kLlThreads / 32) {
            float bv = -__int_as_float(0x7f800000);
            int bi = 0x7fffffff;
            for (int c = lane; c < (int)gridDim.x; c += 32) {
                const float2 p = __ldcg(&A.part[(int64_t)c * kLlMaxLanes + u]);
                if (ll_better(p.x, __float_as_int(p.y), bv, bi)) {
                    bv = p.x;
                    bi = __float_as_int(p.y);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ll_better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == 0) A.next[u] = bi;
        }
    }
    if (tid == 0) *A.ticket = 0u;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// The table's tensor map: bf16 [vocab][dim], boxes of 64 inputs x 128 rows,
// 128-byte swizzle, zeros out of range.  Encoded through the driver entry
// point (no link against the driver library); the last one is kept for the
// next call with the same table.
qlin_status table_map(const uint16_t *emb, int vocab, int dim, CUtensorMap *out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static CUtensorMap last;
    static const void *last_emb = nullptr;
    static int last_v = 0, last_d = 0;
    std::lock_guard<std::mutex> lk(mu);
    if (last_emb == emb && last_v == vocab && last_d == dim) {
        *out = last;
        return QLIN_OK;
    }
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        QLIN_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
        QLIN_REQUIRE(fn && q == cudaDriverEntryPointSuccess, QLIN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    const cuuint64_t gdim[2] = {(cuuint64_t)dim, (cuuint64_t)vocab};
    const cuuint64_t gstride[1] = {(cuuint64_t)dim * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kLlKS, (cuuint32_t)kLlRows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = encode(&last, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(emb), gdim, gstride, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    QLIN_REQUIRE(r == CUDA_SUCCESS, QLIN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    last_emb = emb, last_v = vocab, last_d = dim;
    *out = last;
    return QLIN_OK;
}

struct LlWs {
    int32_t *status;
    unsigned *ticket;
    uint16_t *xs;
    float2 *part;
    size_t bytes;
};

LlWs carve_ll(int vocab, int dim, char *base) {
    LlWs w{};
    size_t off = 0;
    auto take = [&](size_t b) {
        char *p = base ? base + off : nullptr;
        off += align256(b);
        return p;
    };
    w.status = (int32_t *)take(16);
    w.ticket = (unsigned *)take(4);
    w.xs = (uint16_t *)take((size_t)(dim + kLlKS - 1) / kLlKS * kLlKS * 3 * kLlMaxLanes * 2);
    w.part = (float2 *)take(sizeof(float2) * (size_t)((vocab + kLlRows - 1) / kLlRows) * kLlMaxLanes);
    w.bytes = off;
    return w;
}

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" {

size_t qlin_lm_head_lanes_workspace_size(int vocab, int dim) {
    if (vocab < 1 || dim < 1) return 0;
    return carve_ll(vocab, dim, nullptr).bytes;
}

qlin_status qlin_lm_head_lanes(const uint16_t *emb, const float *x, int vocab, int dim, int n_lanes, float *logits,
                               int32_t *next, void *workspace, size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(emb && x && next && workspace, QLIN_ERR_INVALID_ARG, "qlin_lm_head_lanes: null pointer");
    QLIN_REQUIRE(vocab >= 1 && dim >= 8 && dim % 8 == 0 && n_lanes >= 1, QLIN_ERR_INVALID_ARG,
                 "qlin_lm_head_lanes: vocab %d, dim %d, lanes %d", vocab, dim, n_lanes);
    QLIN_REQUIRE(aligned16(emb) && aligned4(x) && aligned4(next) && (!logits || aligned4(logits)) &&
                     aligned16(workspace),
                 QLIN_ERR_INVALID_ARG, "qlin_lm_head_lanes: misaligned pointer");
    const LlWs w = carve_ll(vocab, dim, (char *)workspace);
    QLIN_REQUIRE(workspace_bytes >= w.bytes, QLIN_ERR_INVALID_ARG, "qlin_lm_head_lanes: workspace %zu < %zu bytes",
                 workspace_bytes, w.bytes);
    cudaStream_t st = (cudaStream_t)stream;
    const size_t smem = sizeof(LlSmem) + 1024;  // + the alignment of the swizzled tiles
    CUtensorMap tmap;
    if (qlin_status e = table_map(emb, vocab, dim, &tmap)) return e;
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_lm_head_lanes: tile does not fit");
    blocks_per_sm((const void *)lm_lanes_kernel, smem);  // raises the dynamic shared-memory limit once
    const int grid = std::min(sm_count(), (vocab + kLlRows - 1) / kLlRows);  // persistent: one CTA per SM
    for (int u0 = 0; u0 < n_lanes; u0 += kLlMaxLanes) {  // up to 64 lanes per pass over the table
        const int U = std::min(kLlMaxLanes, n_lanes - u0);
        const int Up = (U + 15) / 16 * 16;
        lm_lanes_split_kernel<<<Up, 256, 0, st>>>(x + (int64_t)u0 * dim, U, Up, dim, (dim + kLlKS - 1) / kLlKS,
                                                  w.xs);
        QLIN_LAUNCHED("lm_lanes_split_kernel");
        LlArgs a{};
        a.emb = emb;
        a.xs = w.xs;
        a.V = vocab;
        a.K = dim;
        a.U = U;
        a.Up = Up;
        a.logits = logits ? logits + (int64_t)u0 * vocab : nullptr;
        a.next = next + u0;
        a.part = w.part;
        a.ticket = w.ticket;
        a.status = w.status;
        lm_lanes_kernel<<<grid, kLlThreads, smem, st>>>(tmap, a);
        QLIN_LAUNCHED("lm_lanes_kernel");
    }
    return QLIN_OK;
}

qlin_status qlin_lm_head_lanes_status(void *workspace, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(workspace, QLIN_ERR_INVALID_ARG, "qlin_lm_head_lanes_status: null workspace");
    int32_t stw[4] = {0, 0, 0, 0};
    QLIN_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    QLIN_CUDA(cudaMemcpy(stw, workspace, sizeof stw, cudaMemcpyDeviceToHost));
    QLIN_CUDA(cudaMemset(workspace, 0, sizeof stw));
    QLIN_REQUIRE(!(stw[0] & kStatusTimeout), QLIN_ERR_TIMEOUT, "qlin_lm_head_lanes: a device-side wait gave up");
    return QLIN_OK;
}

}  // extern "C"
