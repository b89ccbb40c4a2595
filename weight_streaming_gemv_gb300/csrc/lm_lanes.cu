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
// within fp32 rounding of the fp32 dot product.  K advances 64 elements a
// step through four shared-memory stages filled by cp.async (256 loader
// threads, 16-byte copies into the no-swizzle K-major core-matrix layout); one
// thread issues the step's four MMAs.  The accumulator goes to shared memory,
// each lane's logits are formed, written (if asked for) and reduced to the
// CTA's best row; the last CTA reduces the CTAs' bests per lane.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {
namespace {

constexpr int kLlRows = 128;              // table rows per CTA (MMA M)
constexpr int kLlKS = 64;                 // K elements per step
constexpr int kLlChunks = kLlKS / 8;      // 16-byte core-matrix columns per row and step
constexpr int kLlSBO = kLlChunks * 128;   // bytes between 8-row groups
constexpr int kLlStages = 4;
constexpr int kLlLoaders = 256;
constexpr int kLlThreads = kLlLoaders + 32;  // + the warp that issues the MMAs
constexpr int kLlMaxLanes = 64;              // lanes per pass: 3 x 64 = 192 accumulator columns
constexpr int kLlMaxN = 3 * kLlMaxLanes;
constexpr uint32_t kLlCols = 256;            // tensor-memory columns allocated
constexpr int kLlDStride = kLlMaxN + 1;      // floats per accumulator row in shared memory

struct LlSmem {
    union {
        struct {
            uint8_t a[kLlStages][kLlRows / 8 * kLlSBO];  // table rows of a step
            uint8_t b[kLlStages][kLlMaxN / 8 * kLlSBO];  // the lanes' split x of a step
        } in;
        float d[kLlRows][kLlDStride];  // after the K loop: the accumulator
    };
    uint64_t full[kLlStages];      // the stage has landed (kLlLoaders arrivals + the lanes operand's bytes)
    uint64_t mma_done[kLlStages];  // the MMAs reading the stage are done (tcgen05.commit)
    float bv[8][kLlMaxLanes];      // epilogue: each warp's best per lane
    int bi[8][kLlMaxLanes];
    uint32_t tmem;
    int abort;
    int last;
};

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

__device__ __forceinline__ void ll_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte cp.async; nbytes < 16 zero-fills the rest
__device__ __forceinline__ void ll_cp16(void *dst, const void *src, int nbytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(nbytes)
                 : "memory");
}
__device__ __forceinline__ void ll_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void ll_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

__global__ void __launch_bounds__(kLlThreads, 1) lm_lanes_kernel(LlArgs A) {
    extern __shared__ __align__(128) uint8_t ll_smem_raw[];
    LlSmem &S = *reinterpret_cast<LlSmem *>(ll_smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * kLlRows;
    const int K = A.K, N = 3 * A.Up;
    const int nsteps = (K + kLlKS - 1) / kLlKS;

    const uint32_t bbytes = (uint32_t)N * kLlKS * 2;  // the lanes' operand of one step
    const uint64_t keep = ll_evict_last();
    // step t's lanes operand: one bulk copy of its image (thread 0; the stage's
    // barrier is initialised), completing on the stage's full barrier
    auto fetch_b = [&](int t) {
        if (t < nsteps) {
            const int st = t % kLlStages;
            mbar_arrive_expect_tx(&S.full[st], bbytes);
            bulk_g2s(S.in.b[st], A.xs + (int64_t)t * N * kLlKS, bbytes, &S.full[st], keep);
        }
    };
    // step t's table rows into its stage: 1024 chunks of 16 bytes over the loaders
    auto fetch = [&](int t) {
        if (t < nsteps) {
            const int st = t % kLlStages, k0 = t * kLlKS;
            for (int idx = tid; idx < kLlRows * kLlChunks; idx += kLlLoaders) {
                const int r = idx / kLlChunks, kc = idx % kLlChunks;
                const int row = row0 + r, k = k0 + 8 * kc;
                const bool ok = row < A.V && k < K;
                ll_cp16(S.in.a[st] + ll_off(r, kc), A.emb + (ok ? (int64_t)row * K + k : 0), ok ? 16 : 0);
            }
            if (tid == 0) fetch_b(t);
        }
        ll_commit_group();
    };
    if (tid < kLlLoaders)
        for (int t = 0; t < kLlStages - 1; t++) {  // table rows only: the barriers are not yet initialised
            if (t < nsteps) {
                const int st = t % kLlStages, k0 = t * kLlKS;
                for (int idx = tid; idx < kLlRows * kLlChunks; idx += kLlLoaders) {
                    const int r = idx / kLlChunks, kc = idx % kLlChunks;
                    const int row = row0 + r, k = k0 + 8 * kc;
                    const bool ok = row < A.V && k < K;
                    ll_cp16(S.in.a[st] + ll_off(r, kc), A.emb + (ok ? (int64_t)row * K + k : 0), ok ? 16 : 0);
                }
            }
            ll_commit_group();
        }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(kLlCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == kLlLoaders) {
        for (int i = 0; i < kLlStages; i++) {
            mbar_init(&S.full[i], kLlLoaders + 1);  // the loaders, and thread 0's byte-counted arrival
            mbar_init(&S.mma_done[i], 1);
        }
        S.abort = 0;
        fence_mbar_init();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = S.tmem;
    volatile int *abort = &S.abort;
    if (tid == 0)
        for (int t = 0; t < kLlStages - 1; t++) fetch_b(t);

    if (warp == kLlLoaders / 32) {
        if (lane == 0) {  // the MMAs of each step once its stage is full
            const uint32_t idesc = ll_idesc(N);
            for (int t = 0; t < nsteps && !*abort; t++) {
                const int st = t % kLlStages;
                if (!mbar_wait(&S.full[st], (t / kLlStages) & 1)) {
                    *abort = 1;
                    raise_status(A.status, kStatusTimeout);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a0 = smem_addr(S.in.a[st]), b0 = smem_addr(S.in.b[st]);
#pragma unroll
                for (int kk = 0; kk < kLlKS / 16; kk++)  // K = 16: two core-matrix columns (256 bytes)
                    ll_mma(tmem, ll_desc(a0 + 256u * kk), ll_desc(b0 + 256u * kk), idesc, (t > 0 || kk > 0) ? 1u : 0u);
                ll_commit(&S.mma_done[st]);
            }
        }
    } else {
        for (int t = 0; t < nsteps && !*abort; t++) {
            // step t is signalled as soon as this thread's copies of it have landed
            // (one group per step; steps t + 1 and t + 2 may still be in flight) ...
            ll_wait_group<kLlStages - 2>();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&S.full[t % kLlStages]);
            // ... then stage (t - 1) % S is refilled with step t + S - 1 once the
            // MMAs of step t - 1 are done
            if (t >= 1 && t + kLlStages - 1 < nsteps &&
                !mbar_wait(&S.mma_done[(t - 1) % kLlStages], ((t - 1) / kLlStages) & 1)) {
                *abort = 1;
                raise_status(A.status, kStatusTimeout);
                break;
            }
            fetch(t + kLlStages - 1);
        }
        ll_wait_group<0>();
    }
    // the last commit covers every MMA issued before it
    if (nsteps > 0 && !*abort) {
        const int t = nsteps - 1;
        if (!mbar_wait(&S.mma_done[t % kLlStages], (t / kLlStages) & 1)) {
            *abort = 1;
            raise_status(A.status, kStatusTimeout);
        }
    }
    __syncthreads();
    const bool ok = !*abort;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // the accumulator into shared memory: warp w (< 4) reads lanes 32 w .. + 31
    if (warp < 4 && ok) {
        const int row = 32 * warp + lane;
        for (int col = 0; col < N; col += 32) {
            uint32_t r[32];
            ll_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)col, r);
#pragma unroll
            for (int j = 0; j < 32; j++)
                if (col + j < kLlMaxN) S.d[row][col + j] = __uint_as_float(r[j]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kLlCols) : "memory");
    // each lane's logits, its best row in this tile
    const int Up = A.Up;
    if (warp < 8) {
        // warp w: lanes w, w + 8, ... together (the (value, row) order is total,
        // so the reduction order does not matter)
        constexpr int LPW = kLlMaxLanes / 8;
        float bv[LPW];
        int bi[LPW];
#pragma unroll
        for (int j = 0; j < LPW; j++) bv[j] = -__int_as_float(0x7f800000), bi[j] = 0x7fffffff;
        for (int r = lane; r < kLlRows; r += 32) {
            const int row = row0 + r;
            if (row >= A.V) break;
#pragma unroll
            for (int j = 0; j < LPW; j++) {
                const int u = warp + 8 * j;
                if (u < A.U) {
                    const float v = ok ? __fadd_rn(__fadd_rn(S.d[r][u], S.d[r][Up + u]), S.d[r][2 * Up + u])
                                       : __int_as_float(0x7fc00000);
                    if (A.logits) A.logits[(int64_t)u * A.V + row] = v;
                    if (ll_better(v, row, bv[j], bi[j])) bv[j] = v, bi[j] = row;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int j = 0; j < LPW; j++) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[j], off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[j], off);
                if (ll_better(ov, oi, bv[j], bi[j])) bv[j] = ov, bi[j] = oi;
            }
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < LPW; j++)
                if (warp + 8 * j < A.U)
                    A.part[(int64_t)blockIdx.x * kLlMaxLanes + warp + 8 * j] = make_float2(bv[j], __int_as_float(bi[j]));
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        S.last = atomicAdd(A.ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!S.last) return;
    __threadfence();
    // the last CTA: every lane's best over all CTAs (ties to the lower row)
    if (warp < 8) {
        for (int u = warp; u < A.U; u += 8) {
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
    const size_t smem = sizeof(LlSmem);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_lm_head_lanes: tile does not fit");
    blocks_per_sm((const void *)lm_lanes_kernel, smem);  // raises the dynamic shared-memory limit once
    const int grid = (vocab + kLlRows - 1) / kLlRows;
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
        lm_lanes_kernel<<<grid, kLlThreads, smem, st>>>(a);
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
