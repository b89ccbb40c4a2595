// T158 linear for many tokens (prefill) on the fifth-generation tensor cores.
//
// All prompt tokens go through each weight matrix in one pass (citric, "Step 4":
// batched prompt processing).  The integer dot products of "Step 1" run as an
// fp16 matrix product with fp32 accumulation, which is exact here: int8 codes
// (|x| <= 127) and trits are fp16 integers, every product is an integer of
// magnitude <= 127 and every partial sum stays below 127 K < 2^24, so each fp32
// addition is exact and the accumulator equals the int32 sum.
//
// One CTA computes a 128-token x 128-row tile with tcgen05.mma (M = 128,
// N = 128, K = 16 per instruction) into a 128-column fp32 accumulator in tensor
// memory.  K advances in steps of 80 elements: 16 packed bytes of every weight
// row.  Within a step both operands use the same permuted K order, K' = 16 i + j
// for element 5 j + i (digit i of packed byte j), which leaves the dot product
// unchanged and lets the trits come straight out of the digit-plane decode.
// Threads 0..127 convert the step's activation rows (int8 -> fp16, gathered into
// K' order), threads 128..255 decode the weight rows (5 trits per byte ->
// fp16), both into shared memory in the no-swizzle K-major layout of the MMA
// (8-row x 16-byte core matrices, 128 bytes apart along K, kTcSBO bytes
// between 8-row groups); one thread issues the step's five MMAs and commits
// them to an mbarrier; two stages let the conversion of step s+1 overlap the
// MMAs of step s.  The epilogue reads the accumulator back with tcgen05.ld
// (warp w reads lanes 32 (w % 4) .. + 31, columns 64 (w / 4) .. + 63).
#include <cuda_fp16.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {

constexpr int kTcBM = 128;                      // tokens per CTA (MMA M)
constexpr int kTcBN = 256;                      // weight rows per CTA (MMA N)
constexpr int kTcKS = 80;                       // K elements per step (16 packed bytes)
constexpr int kTcConv = kTcBM + kTcBN;          // converter threads: one per activation row and per weight row
constexpr int kTcThreads = kTcConv + 32;        // + one warp that issues the MMAs
constexpr int kTcChunks = kTcKS / 8;            // 16-byte core-matrix columns per row and step
constexpr int kTcSBO = kTcChunks * 128;         // bytes between 8-row groups
constexpr int kTcTileA = (kTcBM / 8) * kTcSBO;  // bytes of the A tile of one step
constexpr int kTcTileB = (kTcBN / 8) * kTcSBO;  // bytes of the B tile of one step
constexpr int kTcStages = 2;                    // fp16 operand stages
constexpr int kTcRaw = 6;                       // raw (int8 / packed) stages copied ahead
constexpr uint32_t kTcCols = kTcBN;             // tensor-memory columns: the 128 x 256 fp32 accumulator
constexpr int kTcPStride = kTcBN + 4;           // floats per row of a partial tile in shared memory
constexpr int kTcMaxSplit = 8;                  // CTAs of a cluster that split K

struct TcSmem {
    union {
        struct {
            uint8_t a[kTcStages][kTcTileA];
            uint8_t b[kTcStages][kTcTileB];
            uint8_t raw_a[kTcRaw][kTcBM][kTcKS];  // each thread's own activation row, step by step
            uint8_t raw_b[kTcRaw][kTcBN][16];     // each thread's own packed weight row
        } in;
        float part[kTcBM][kTcPStride];  // after the K loop: this CTA's partial tile (split K)
    };
    uint64_t full[kTcStages];      // the converters have written the stage (kTcConv arrivals)
    uint64_t mma_done[kTcStages];  // the MMAs reading the stage are done (tcgen05.commit)
    float xs[kTcBM];               // activation scales of the tile's tokens
    uint32_t tmem;
    int abort;
};

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
// K-major, N = kTcBN, M = kTcBM.  Both tiles use the descriptor above (the same
// K step, so the same stride between 8-row groups).
constexpr uint32_t kTcIdesc =
    (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kTcBN >> 3) << 17) | ((uint32_t)(kTcBM >> 4) << 24);

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 32 consecutive accumulator columns of this thread's tensor-memory lane
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// Byte offset of 16-byte chunk kc of row r in an operand tile.
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

// 80 activation bytes of one row (words in[], byte v + 128 of each value v,
// i.e. already xor 0x80) into row r of the A tile, K' order, fp16.
__device__ __forceinline__ void tc_put_a(uint8_t *tile, const uint32_t (&in)[20], int r) {
#pragma unroll
    for (int kc = 0; kc < kTcChunks; kc++) {
        uint32_t h[4];
#pragma unroll
        for (int p = 0; p < 4; p++) {
            const int kp = 8 * kc + 2 * p;           // K' of the low half
            const int i = kp >> 4, j = kp & 15;      // digit, packed byte
            const int e0 = 5 * j + i, e1 = e0 + 5;   // element offsets within the step
            h[p] = h2sub(i8pair_bits(in[e0 >> 2], in[e1 >> 2], e0 & 3, e1 & 3), 0x64806480u);
        }
        *reinterpret_cast<uint4 *>(tile + tc_off(r, kc)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// 16 packed bytes of one weight row into row r of the B tile, K' order, fp16 trits.
__device__ __forceinline__ void tc_put_b(uint8_t *tile, const uint4 v, int r) {
    uint32_t D[4][5];
    t158_planes(v.x, D[0]);
    t158_planes(v.y, D[1]);
    t158_planes(v.z, D[2]);
    t158_planes(v.w, D[3]);
#pragma unroll
    for (int kc = 0; kc < kTcChunks; kc++) {
        const int i = kc >> 1, wa = 2 * (kc & 1);
        // digits d in 0..2: fp16 (1024 + d) - 1025 = d - 1
        const uint32_t h0 = h2sub(__byte_perm(D[wa][i], 0x6464u, 0x5140u), 0x64016401u);
        const uint32_t h1 = h2sub(__byte_perm(D[wa][i], 0x6464u, 0x5342u), 0x64016401u);
        const uint32_t h2 = h2sub(__byte_perm(D[wa + 1][i], 0x6464u, 0x5140u), 0x64016401u);
        const uint32_t h3 = h2sub(__byte_perm(D[wa + 1][i], 0x6464u, 0x5342u), 0x64016401u);
        *reinterpret_cast<uint4 *>(tile + tc_off(r, kc)) = make_uint4(h0, h1, h2, h3);
    }
}

// 16 bytes global -> shared, the bytes past src_bytes (0..16) zero.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_pending() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Activation row m (token) of step s into the A tile, K' order, fp16, loaded
// directly (any alignment).
__device__ __forceinline__ void tc_fill_a(uint8_t *tile, const int8_t *__restrict__ xq, int M, int K, int m, int r,
                                          int s, bool vec) {
    const int k0 = s * kTcKS;
    uint32_t in[20];
    if (m >= M) {
#pragma unroll
        for (int i = 0; i < 20; i++) in[i] = 0x80808080u;  // bytes v + 128 of v = 0
    } else if (vec && k0 + kTcKS <= K) {
        const uint4 *src = reinterpret_cast<const uint4 *>(xq + (int64_t)m * K + k0);
#pragma unroll
        for (int i = 0; i < 5; i++) {
            const uint4 v = __ldg(src + i);
            in[4 * i] = v.x ^ 0x80808080u;
            in[4 * i + 1] = v.y ^ 0x80808080u;
            in[4 * i + 2] = v.z ^ 0x80808080u;
            in[4 * i + 3] = v.w ^ 0x80808080u;
        }
    } else {
        const int8_t *row = xq + (int64_t)m * K;
#pragma unroll
        for (int i = 0; i < 20; i++) {
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const int k = k0 + 4 * i + b;
                const uint32_t byte = k < K ? (uint32_t)(uint8_t)row[k] : 0u;
                v |= byte << (8 * b);
            }
            in[i] = v ^ 0x80808080u;
        }
    }
    tc_put_a(tile, in, r);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// float4 at a shared address of CTA `rank` of this cluster
__device__ __forceinline__ float4 ld_peer_f4(const void *local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a)
                 : "memory");
    return v;
}

// Grid: (N tiles, M tiles, split); a cluster is the `split` CTAs of one tile,
// each over its own range of K steps.  split == 1: no cluster reduction.
__global__ void __launch_bounds__(kTcThreads, 1) t158_tc_kernel(const int8_t *__restrict__ xq,
                                                               const float *__restrict__ xs,
                                                               const uint8_t *__restrict__ w, int64_t pitch, float ws_arg,
                                                               const float *__restrict__ ws_ptr,
                                                               float *__restrict__ y, int32_t *__restrict__ acc_out,
                                                               int M, int N, int K, int split) {
    const float ws = ws_ptr ? __ldg(ws_ptr) : ws_arg;  // the weight scale, from device memory when given
    extern __shared__ __align__(128) uint8_t tc_smem_raw[];
    TcSmem &S = *reinterpret_cast<TcSmem *>(tc_smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kTcBN, m0 = blockIdx.y * kTcBM;
    const int nsteps = (K + kTcKS - 1) / kTcKS;
    const int z = split > 1 ? (int)cluster_rank() : 0;
    const int s_lo = (int)((int64_t)nsteps * z / split), s_hi = (int)((int64_t)nsteps * (z + 1) / split);

    // Converters.  Raw bytes of each thread's own row run kTcRaw - 1
    // steps ahead through cp.async (16-byte copies, zero-filled past K, M
    // and N: such products are zero or land outside the output); a thread
    // reads back only what it copied, so its own wait_group is enough.
    // Activations that are not 16-byte aligned are loaded directly.
    const bool a_async = (reinterpret_cast<uintptr_t>(xq) & 15) == 0 && K % 16 == 0;
    const bool is_a = tid < kTcBM;
    const int r_own = is_a ? tid : tid - kTcBM;
    auto fetch = [&](int s) {
        if (s < s_hi) {
            const int rs = (s - s_lo) % kTcRaw;
            if (is_a) {
                if (a_async) {
                    const int m = m0 + r_own, k0 = s * kTcKS;
                    const int8_t *row = xq + (int64_t)(m < M ? m : 0) * K;
#pragma unroll
                    for (int c = 0; c < kTcKS / 16; c++) {
                        const int kb = k0 + 16 * c;
                        const int nb = m < M ? max(0, min(16, K - kb)) : 0;
                        cp_async16(S.in.raw_a[rs][r_own] + 16 * c, nb > 0 ? row + kb : row, nb);
                    }
                }
            } else {
                const int n = n0 + r_own;
                cp_async16(S.in.raw_b[rs][r_own], w + (int64_t)(n < N ? n : 0) * pitch + (int64_t)s * 16,
                           n < N ? 16 : 0);
            }
        }
        cp_async_commit();
    };
    // the first copies go out before anything else
    if (tid < kTcConv) {
#pragma unroll
        for (int s = 0; s < kTcRaw - 1; s++) fetch(s_lo + s);
    }
    for (int i = tid; i < kTcBM; i += kTcThreads) S.xs[i] = m0 + i < M ? xs[m0 + i] : 0.0f;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int i = 0; i < kTcStages; i++) {
            mbar_init(&S.full[i], kTcConv);
            mbar_init(&S.mma_done[i], 1);
        }
        S.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    volatile int *abort = &S.abort;
    const int nst = s_hi - s_lo;  // steps of this CTA

    if (warp == kTcConv / 32) {
        // ---- MMA warp: lane 0 issues each step's five MMAs once the converters
        // have filled the stage, and commits them to the stage's mma_done
        if (lane == 0) {
            for (int i = 0; i < nst && !*abort; i++) {
                const int st = i & 1;
                if (!mbar_wait(&S.full[st], (i >> 1) & 1)) {
                    *abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(S.in.a[st]), b0 = smem_addr(S.in.b[st]);
#pragma unroll
                for (int u = 0; u < kTcKS / 16; u++)  // K = 16: two core-matrix columns (256 bytes)
                    tc_mma(tmem, tc_desc(a0 + 256u * u), tc_desc(b0 + 256u * u), (i > 0 || u > 0) ? 1u : 0u);
                tc_commit(&S.mma_done[st]);
            }
        }
    } else {
        // ---- converters
        for (int i = 0; i < nst && !*abort; i++) {
            const int s = s_lo + i, st = i & 1;
            fetch(s + kTcRaw - 1);
            cp_async_wait_pending<kTcRaw - 1>();  // this thread's copies of step s have landed
            // the MMAs of step i-2 read this stage: wait until they are done
            if (i >= 2 && !mbar_wait(&S.mma_done[st], ((i >> 1) - 1) & 1)) {
                *abort = 1;
                break;
            }
            if (is_a) {
                if (a_async) {
                    uint32_t in[20];
                    const uint4 *src = reinterpret_cast<const uint4 *>(S.in.raw_a[i % kTcRaw][r_own]);
#pragma unroll
                    for (int q = 0; q < 5; q++) {
                        const uint4 v = src[q];
                        in[4 * q] = v.x ^ 0x80808080u;
                        in[4 * q + 1] = v.y ^ 0x80808080u;
                        in[4 * q + 2] = v.z ^ 0x80808080u;
                        in[4 * q + 3] = v.w ^ 0x80808080u;
                    }
                    tc_put_a(S.in.a[st], in, r_own);
                } else {
                    tc_fill_a(S.in.a[st], xq, M, K, m0 + r_own, r_own, s, false);
                }
            } else {
                tc_put_b(S.in.b[st], *reinterpret_cast<const uint4 *>(S.in.raw_b[i % kTcRaw][r_own]), r_own);
            }
            // the generic-proxy writes above, visible to the tensor core (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&S.full[st]);
        }
        cp_async_wait_pending<0>();
    }
    // the last commit covers every MMA issued before it
    bool ok = true;
    if (nst > 0 && !*abort) {
        const int i = nst - 1;
        if (!mbar_wait(&S.mma_done[i & 1], (i >> 1) & 1)) *abort = 1;
    }
    __syncthreads();
    ok = !*abort;
    tc_fence_after();

    const float nanv = ok ? 0.0f : __int_as_float(0x7fc00000);  // a wait that gave up: the tile reads NaN
    const bool vec_out = y && (reinterpret_cast<uintptr_t>(y) & 15) == 0 && N % 4 == 0;
    // the accumulator into shared memory (warps 0..7: lanes 32 (w % 4) .. + 31,
    // columns 128 (w / 4) .. + 127), so that the output rows are written coalesced
    if (warp < 8) {
        const int q = warp & 3, cg = warp >> 2;
        const int row = 32 * q + lane;
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
            const int col = 128 * cg + 32 * c;
            uint32_t r[32];
            tc_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, r);
            float4 *dst = reinterpret_cast<float4 *>(&S.part[row][col]);
#pragma unroll
            for (int j = 0; j < 8; j++)
                dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                     __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
    }
    // split K: CTA z adds rows [128 z / split, 128 (z+1) / split) over the
    // cluster in rank order (integers below 2^24: exact); split 1: all rows
    if (split > 1)
        cluster_sync();
    else
        __syncthreads();
    const int r0 = kTcBM * z / split, r1 = kTcBM * (z + 1) / split;
#pragma unroll 4
    for (int e = tid; e < (r1 - r0) * (kTcBN / 4); e += kTcThreads) {
        const int row = r0 + e / (kTcBN / 4), c4 = e % (kTcBN / 4);
        float4 v;
        if (split == 1) {
            v = *reinterpret_cast<const float4 *>(&S.part[row][4 * c4]);
        } else {
            float4 u[kTcMaxSplit];
#pragma unroll
            for (int qq = 0; qq < kTcMaxSplit; qq++)
                if (qq < split) u[qq] = ld_peer_f4(&S.part[row][4 * c4], (uint32_t)qq);
            v = u[0];
#pragma unroll
            for (int qq = 1; qq < kTcMaxSplit; qq++)
                if (qq < split) {
                    v.x = __fadd_rn(v.x, u[qq].x);
                    v.y = __fadd_rn(v.y, u[qq].y);
                    v.z = __fadd_rn(v.z, u[qq].z);
                    v.w = __fadd_rn(v.w, u[qq].w);
                }
        }
        const int m = m0 + row, nb = n0 + 4 * c4;
        if (m >= M || nb >= N) continue;
        const float xsm = S.xs[row];
        const float vv[4] = {v.x, v.y, v.z, v.w};
        if (acc_out) {
            if ((reinterpret_cast<uintptr_t>(acc_out) & 15) == 0 && N % 4 == 0 && nb + 4 <= N) {
                *reinterpret_cast<int4 *>(acc_out + (int64_t)m * N + nb) =
                    make_int4(__float2int_rz(vv[0]), __float2int_rz(vv[1]), __float2int_rz(vv[2]), __float2int_rz(vv[3]));
            } else {
                for (int j = 0; j < 4; j++)
                    if (nb + j < N) acc_out[(int64_t)m * N + nb + j] = __float2int_rz(vv[j]);
            }
        }
        if (y) {
            if (vec_out && nb + 4 <= N) {
                *reinterpret_cast<float4 *>(y + (int64_t)m * N + nb) =
                    make_float4(__fadd_rn(__fmul_rn(__fmul_rn(vv[0], ws), xsm), nanv),
                                __fadd_rn(__fmul_rn(__fmul_rn(vv[1], ws), xsm), nanv),
                                __fadd_rn(__fmul_rn(__fmul_rn(vv[2], ws), xsm), nanv),
                                __fadd_rn(__fmul_rn(__fmul_rn(vv[3], ws), xsm), nanv));
            } else {
                for (int j = 0; j < 4; j++)
                    if (nb + j < N) y[(int64_t)m * N + nb + j] = __fadd_rn(__fmul_rn(__fmul_rn(vv[j], ws), xsm), nanv);
            }
        }
    }
    if (split > 1) cluster_sync();  // no CTA leaves while another still reads its shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
}

// Clusters of `c` CTAs of this kernel that can be resident at once (cached).
static int tc_resident_clusters(int c, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, c});
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, (unsigned)c);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)c;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, t158_tc_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    cache[{dev, c}] = n;
    return n;
}

qlin_status t158_linear_tensor_cores(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                     const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K,
                                     cudaStream_t st) {
    const size_t smem = sizeof(TcSmem);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: tensor-core tile does not fit");
    blocks_per_sm((const void *)t158_tc_kernel, smem);  // raises the dynamic shared-memory limit
    const int tiles_n = (N + kTcBN - 1) / kTcBN, tiles_m = (M + kTcBM - 1) / kTcBM;
    const int nsteps = (K + kTcKS - 1) / kTcKS;
    // split K over a cluster when the tiles alone leave SMs idle: the largest
    // split whose clusters (they must fit within a GPC) are all resident at once
    const int tiles = tiles_n * tiles_m;
    int split = 1;
    for (int c = kTcMaxSplit; c >= 2; c--) {
        if (c > nsteps || tiles * c > 2 * sm_count()) continue;
        if (tc_resident_clusters(c, smem) >= tiles) {
            split = c;
            break;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles_n, (unsigned)tiles_m, (unsigned)split);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)split;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, t158_tc_kernel, xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, split));
    QLIN_LAUNCHED("t158_tc_kernel");
    return QLIN_OK;
}

}  // namespace qlin
