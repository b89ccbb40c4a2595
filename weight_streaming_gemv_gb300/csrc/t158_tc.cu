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

#include "common.cuh"
#include "stream.cuh"

namespace qlin {

constexpr int kTcBM = 128;                      // tokens per CTA (MMA M)
constexpr int kTcBN = 128;                      // weight rows per CTA (MMA N)
constexpr int kTcKS = 80;                       // K elements per step (16 packed bytes)
constexpr int kTcThreads = 256;
constexpr int kTcChunks = kTcKS / 8;            // 16-byte core-matrix columns per row and step
constexpr int kTcSBO = kTcChunks * 128;         // bytes between 8-row groups
constexpr int kTcTile = (kTcBM / 8) * kTcSBO;   // bytes of one operand tile of one step
constexpr int kTcStages = 2;
constexpr uint32_t kTcCols = 128;               // tensor-memory columns: the 128 x 128 fp32 accumulator

static_assert(kTcBM == kTcBN, "both operand tiles share one layout");

struct TcSmem {
    uint8_t a[kTcStages][kTcTile];
    uint8_t b[kTcStages][kTcTile];
    uint64_t mma_done[kTcStages];
    uint32_t tmem;
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
// K-major, N = kTcBN, M = kTcBM.
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

// Activation row m (token) of step s into the A tile, K' order, fp16.
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

// Weight row n of step s into the B tile, K' order, fp16 trits.
__device__ __forceinline__ void tc_fill_b(uint8_t *tile, const uint8_t *__restrict__ w, int64_t pitch, int N, int n,
                                          int r, int s) {
    uint4 v = make_uint4(0x79797979u, 0x79797979u, 0x79797979u, 0x79797979u);  // byte 121: five zero trits
    if (n < N) v = __ldg(reinterpret_cast<const uint4 *>(w + (int64_t)n * pitch + (int64_t)s * 16));
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

__global__ void __launch_bounds__(kTcThreads, 1) t158_tc_kernel(const int8_t *__restrict__ xq,
                                                               const float *__restrict__ xs,
                                                               const uint8_t *__restrict__ w, int64_t pitch, float ws,
                                                               float *__restrict__ y, int32_t *__restrict__ acc_out,
                                                               int M, int N, int K) {
    extern __shared__ __align__(128) uint8_t tc_smem_raw[];
    TcSmem &S = *reinterpret_cast<TcSmem *>(tc_smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kTcBN, m0 = blockIdx.y * kTcBM;
    const int nsteps = (K + kTcKS - 1) / kTcKS;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int i = 0; i < kTcStages; i++) mbar_init(&S.mma_done[i], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    const bool a_vec = (reinterpret_cast<uintptr_t>(xq) & 15) == 0 && K % 16 == 0;

    bool ok = true;
    int issued = 0;  // steps whose MMAs were issued
    for (int s = 0; s < nsteps; s++) {
        const int st = s & 1;
        // the MMAs of step s-2 read this stage: wait until they are done
        const bool waited = s < 2 || mbar_wait(&S.mma_done[st], ((s >> 1) - 1) & 1);
        if (!__syncthreads_and(waited)) {
            ok = false;
            break;
        }
        if (tid < 128)
            tc_fill_a(S.a[st], xq, M, K, m0 + tid, tid, s, a_vec);
        else
            tc_fill_b(S.b[st], w, pitch, N, n0 + tid - 128, tid - 128, s);
        // the generic-proxy writes above, visible to the tensor core (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a0 = smem_addr(S.a[st]), b0 = smem_addr(S.b[st]);
#pragma unroll
            for (int u = 0; u < kTcKS / 16; u++)  // K = 16: two core-matrix columns (256 bytes)
                tc_mma(tmem, tc_desc(a0 + 256u * u), tc_desc(b0 + 256u * u), (s > 0 || u > 0) ? 1u : 0u);
            tc_commit(&S.mma_done[st]);
        }
        issued = s + 1;
    }
    // the last commit covers every MMA issued before it
    if (issued > 0) {
        const int s = issued - 1;
        if (!mbar_wait(&S.mma_done[s & 1], (s >> 1) & 1)) ok = false;
    }
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();

    if (ok && issued == nsteps) {
        const int q = warp & 3, hf = warp >> 2;
        const int m = m0 + 32 * q + lane;
        const float xsm = m < M ? xs[m] : 0.0f;
        const bool vec_out = y && (reinterpret_cast<uintptr_t>(y) & 15) == 0 && N % 4 == 0;
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int col = 64 * hf + 32 * c;
            uint32_t r[32];
            tc_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, r);
            if (m < M) {
                const int nb = n0 + col;
                if (acc_out)
                    for (int j = 0; j < 32; j++)
                        if (nb + j < N) acc_out[(int64_t)m * N + nb + j] = __float2int_rz(__uint_as_float(r[j]));
                if (y) {
                    if (vec_out && nb + 32 <= N) {
                        float4 *dst = reinterpret_cast<float4 *>(y + (int64_t)m * N + nb);
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            dst[j] = make_float4(__fmul_rn(__fmul_rn(__uint_as_float(r[4 * j]), ws), xsm),
                                                 __fmul_rn(__fmul_rn(__uint_as_float(r[4 * j + 1]), ws), xsm),
                                                 __fmul_rn(__fmul_rn(__uint_as_float(r[4 * j + 2]), ws), xsm),
                                                 __fmul_rn(__fmul_rn(__uint_as_float(r[4 * j + 3]), ws), xsm));
                    } else {
                        for (int j = 0; j < 32; j++)
                            if (nb + j < N)
                                y[(int64_t)m * N + nb + j] = __fmul_rn(__fmul_rn(__uint_as_float(r[j]), ws), xsm);
                    }
                }
            }
        }
    } else if (!ok && tid == 0) {
        // a wait gave up (never in a correct build): the tile reads NaN
        for (int mm = 0; mm < kTcBM && m0 + mm < M; mm++)
            for (int j = 0; j < kTcBN && n0 + j < N; j++)
                if (y) y[(int64_t)(m0 + mm) * N + n0 + j] = __int_as_float(0x7fc00000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
}

qlin_status t158_linear_tensor_cores(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                     float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    const size_t smem = sizeof(TcSmem);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: tensor-core tile does not fit");
    blocks_per_sm((const void *)t158_tc_kernel, smem);  // raises the dynamic shared-memory limit
    dim3 grid((unsigned)((N + kTcBN - 1) / kTcBN), (unsigned)((M + kTcBM - 1) / kTcBM));
    t158_tc_kernel<<<grid, kTcThreads, smem, st>>>(xq, xs, w, pitch, ws, y, acc, M, N, K);
    QLIN_LAUNCHED("t158_tc_kernel");
    return QLIN_OK;
}

}  // namespace qlin
