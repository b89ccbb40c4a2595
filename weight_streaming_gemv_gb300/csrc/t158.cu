// T158 linear layers (int8-absmax activations x ternary weights packed five
// per byte in base 3) on CUDA cores, and the per-row activation quantiser.
//
// "Gemma 3 1B at 114 tokens per second on a laptop CPU", "Step 1: a kernel
// for 1.6-bit weights": the weights are streamed packed, unpacked in
// registers, and multiplied with int8 activations in exact integer math.
// The page's CPU kernel regroups "trit number i of 4 neighbouring bytes" and
// reorders the input once per token; here the same idea runs on the
// canonical byte layout: the four bytes of a 32-bit word are decoded into
// five digit planes (one byte lane per packed byte), and the activations are
// reordered once per block into matching planes, so every plane is one
// __dp4a operand.  Digits are unsigned (d = trit + 1); the row result is
// sum(d * x) - sum(x).
#include <algorithm>

#include "common.cuh"

namespace qlin {

// ---------------------------------------------------------------- S3 quantiser
__global__ void __launch_bounds__(256) quant_i8_kernel(const float *__restrict__ x, int8_t *__restrict__ xq,
                                                       float *__restrict__ xs, int K) {
    __shared__ float red[32];
    const int m = blockIdx.x;
    const float *row = x + (int64_t)m * K;
    float a = 0.0f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) a = fmaxf(a, fabsf(row[k]));
    a = warp_max(a);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float s = quant_scale(red[0]);
    const float rinv = __fdiv_rn(1.0f, s);
    for (int k = threadIdx.x; k < K; k += blockDim.x)
        xq[(int64_t)m * K + k] = (int8_t)quant_code_r(row[k], s, rinv);
    if (threadIdx.x == 0) xs[m] = s;
}

// ---------------------------------------------------------------- activation planes
// xr[c*5 + i] (uint4) holds, in word w / byte b, the activation of trit
// 5*(16c + 4w + b) + i: digit i of byte 4w + b of chunk c.  Zero past K.
__device__ __forceinline__ void build_planes(const int8_t *__restrict__ x, int K, int C, uint4 *xr) {
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const int nwords = C * 20;
    for (int idx = threadIdx.x; idx < nwords; idx += blockDim.x) {
        const int c = idx / 20, r = idx % 20, i = r / 4, w = r % 4;
        const int byte0 = 16 * c + 4 * w;
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int k = 5 * (byte0 + b) + i;
            const uint32_t xb = (k < K) ? (uint32_t)(uint8_t)x[k] : 0u;
            v |= xb << (8 * b);
        }
        xw[idx] = v;
    }
}

// Row sum of the int8 activations (exact).
__device__ __forceinline__ int block_isum(const int8_t *__restrict__ x, int K, int *red) {
    int s = 0;
    for (int k = threadIdx.x; k < K; k += blockDim.x) s += x[k];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    int t = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); i++) t += red[i];
    __syncthreads();
    return t;
}

// ---------------------------------------------------------------- S4 / S6 GEMV
// LPR lanes share one packed row (chunk c = lane % LPR + LPR*j); 32/LPR rows
// per slot, R slots per warp pass.  MT tokens per block (grid.y tiles M).
template <int LPR, int R, int MT>
__global__ void __launch_bounds__(256) t158_gemv_kernel(const int8_t *__restrict__ xq, const float *__restrict__ xs,
                                                        const uint8_t *__restrict__ w, int64_t pitch, float ws,
                                                        const float *__restrict__ ws_ptr, float *__restrict__ y, int32_t *__restrict__ acc_out,
                                                        int M, int N, int K) {
    extern __shared__ uint4 smem[];
    const int C = (int)(pitch / 16);
    uint4 *xr = smem;                                            // [MT][C*5]
    int *sumx = reinterpret_cast<int *>(smem + (size_t)MT * C * 5);  // [MT] then 32 scratch
    const int m0 = blockIdx.y * MT;
    const float wsv = ws_ptr ? *ws_ptr : ws;
    for (int mm = 0; mm < MT; mm++) {
        const int m = m0 + mm;
        if (m < M) {
            build_planes(xq + (int64_t)m * K, K, C, xr + (size_t)mm * C * 5);
            const int s = block_isum(xq + (int64_t)m * K, K, sumx + MT);
            if (threadIdx.x == 0) sumx[mm] = s;
        } else {
            for (int idx = threadIdx.x; idx < C * 5; idx += blockDim.x) xr[(size_t)mm * C * 5 + idx] = make_uint4(0, 0, 0, 0);
            if (threadIdx.x == 0) sumx[mm] = 0;
        }
    }
    __syncthreads();

    constexpr int RPS = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int warps = blockDim.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * warps;
    constexpr int ROWS = RPS * R;

    for (int64_t r0 = gwarp * ROWS; r0 < N; r0 += nwarps * ROWS) {
        int acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int mm = 0; mm < MT; mm++) acc[r][mm] = 0;

        for (int c = sub; c < C; c += LPR) {
            uint4 wv[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t row = r0 + r * RPS + rsub;
                // wide rows: the chunk two iterations ahead toward L2 (more bytes in flight per warp)
                if (LPR == 32 && row < N && c + 2 * LPR < C)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(w + row * pitch + (int64_t)(c + 2 * LPR) * 16));
                wv[r] = (row < N) ? ld_stream_v4(w + row * pitch + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
            }
            uint32_t D[R][4][5];
#pragma unroll
            for (int r = 0; r < R; r++) {
                t158_planes(wv[r].x, D[r][0]);
                t158_planes(wv[r].y, D[r][1]);
                t158_planes(wv[r].z, D[r][2]);
                t158_planes(wv[r].w, D[r][3]);
            }
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                const uint4 *X = xr + ((size_t)mm * C + c) * 5;
#pragma unroll
                for (int i = 0; i < 5; i++) {
                    const uint4 xv = X[i];
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        int a = acc[r][mm];
                        a = dp4a(D[r][0][i], xv.x, a);
                        a = dp4a(D[r][1][i], xv.y, a);
                        a = dp4a(D[r][2][i], xv.z, a);
                        a = dp4a(D[r][3][i], xv.w, a);
                        acc[r][mm] = a;
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; r++) {
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                int v = acc[r][mm];
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                acc[r][mm] = v;
            }
            const int64_t row = r0 + r * RPS + rsub;
            if (sub == 0 && row < N) {
#pragma unroll
                for (int mm = 0; mm < MT; mm++) {
                    const int m = m0 + mm;
                    if (m < M) {
                        const int a = acc[r][mm] - sumx[mm];
                        if (acc_out) acc_out[(int64_t)m * N + row] = a;
                        if (y) y[(int64_t)m * N + row] = __fmul_rn(__fmul_rn((float)a, wsv), xs[m]);
                    }
                }
            }
        }
    }
}

qlin_status launch_quant_i8(const float *x, int8_t *xq, float *xs, int M, int K, cudaStream_t st) {
    quant_i8_kernel<<<M, 256, 0, st>>>(x, xq, xs, K);
    QLIN_LAUNCHED("quant_i8_kernel");
    return QLIN_OK;
}

template <int LPR, int R, int MT>
static qlin_status launch_t158(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                               const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    auto kern = t158_gemv_kernel<LPR, R, MT>;
    const int C = (int)(pitch / 16);
    const size_t smem = (size_t)MT * C * 5 * sizeof(uint4) + (MT + 32) * sizeof(int);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: K=%d needs %zu B of shared memory",
                 K, smem);
    const int per_sm = blocks_per_sm((const void *)kern, smem);
    constexpr int ROWS = (32 / LPR) * R;
    const int64_t warps_needed = (N + ROWS - 1) / ROWS;
    int64_t blocks = (warps_needed + 7) / 8;
    // each block builds the activation planes once: at most two blocks per SM,
    // so that they serve more rows each (the grid-stride loop takes the rest)
    const int64_t cap = (int64_t)sm_count() * std::min(per_sm, 2);
    if (blocks > cap) blocks = cap;
    dim3 grid((unsigned)blocks, (unsigned)((M + MT - 1) / MT));
    kern<<<grid, 256, smem, st>>>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K);
    QLIN_LAUNCHED("t158_gemv_kernel");
    return QLIN_OK;
}

template <int LPR>
static qlin_status dispatch_mt(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                               const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    if (M == 1) return launch_t158<LPR, 4, 1>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (M == 2) return launch_t158<LPR, 4, 2>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (M <= 4) return launch_t158<LPR, 2, 4>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (M <= 8) return launch_t158<LPR, 2, 8>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    return launch_t158<LPR, 2, 16>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
}

// Tokens from which the tensor-core kernel (a 128-token tile) takes over: its
// time hardly depends on M, and from about 8 tokens it beats the CUDA-core
// kernel on the Gemma-3-1B shapes (1152 -> 6912 and 6912 -> 1152).
constexpr int kTensorCoreMinM = 8;
// work: null, or scratch of t158_tc_workspace_bytes(M, K) bytes for the
// activation tiles; convert: write them from xq first (false: they already
// hold this xq's tiles, written by an earlier call with the same M and K).
qlin_status t158_linear_tensor_cores(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                     const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K,
                                     cudaStream_t st, void *work, bool convert);
size_t t158_tc_workspace_bytes(int M, int K);

qlin_status t158_linear_cuda_cores(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                   const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    const int C = (int)(pitch / 16);
    if (C <= 8) return dispatch_mt<8>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (C <= 16) return dispatch_mt<16>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    return dispatch_mt<32>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
}

// T158 linear for M tokens with the weight scale in device memory (the decode
// paths keep the model's scales on the device): the same dispatch as
// qlin_t158_i8, with the activation-tile scratch of t158_linear_tensor_cores.
qlin_status t158_linear_dev_scale(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch,
                                  const float *ws_ptr, float *y, int M, int N, int K, cudaStream_t st, void *work,
                                  bool convert) {
    if (M >= kTensorCoreMinM)
        return t158_linear_tensor_cores(xq, xs, w, pitch, 0.0f, ws_ptr, y, nullptr, M, N, K, st, work, convert);
    return t158_linear_cuda_cores(xq, xs, w, pitch, 0.0f, ws_ptr, y, nullptr, M, N, K, st);
}

size_t t158_workspace_bytes(int M, int K) { return M >= kTensorCoreMinM ? t158_tc_workspace_bytes(M, K) : 0; }

}  // namespace qlin

extern "C" {

qlin_status qlin_quant_i8(const float *x, int8_t *xq, float *x_scale, int M, int K, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(x && xq && x_scale, QLIN_ERR_INVALID_ARG, "qlin_quant_i8: null pointer");
    QLIN_REQUIRE(M >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_quant_i8: M=%d K=%d", M, K);
    QLIN_REQUIRE(qlin::aligned4(x) && qlin::aligned4(x_scale), QLIN_ERR_INVALID_ARG, "qlin_quant_i8: misaligned");
    return qlin::launch_quant_i8(x, xq, x_scale, M, K, (cudaStream_t)stream);
}

qlin_status qlin_t158_i8(const int8_t *xq, const float *x_scale, const uint8_t *w_packed, int64_t w_pitch,
                         float w_scale, float *y, int32_t *acc, int M, int N, int K, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(xq && x_scale && w_packed && (y || acc), QLIN_ERR_INVALID_ARG, "qlin_t158_i8: null pointer");
    QLIN_REQUIRE(M >= 1 && N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_t158_i8: M=%d N=%d K=%d", M, N, K);
    QLIN_REQUIRE(w_pitch % 16 == 0 && w_pitch >= (K + 4) / 5, QLIN_ERR_INVALID_ARG,
                 "qlin_t158_i8: w_pitch %lld must be a multiple of 16 and >= ceil(K/5)", (long long)w_pitch);
    QLIN_REQUIRE(qlin::aligned16(w_packed), QLIN_ERR_INVALID_ARG, "qlin_t158_i8: w_packed not 16-byte aligned");
    QLIN_REQUIRE(qlin::aligned4(x_scale) && (!y || qlin::aligned4(y)) && (!acc || qlin::aligned4(acc)),
                 QLIN_ERR_INVALID_ARG, "qlin_t158_i8: misaligned x_scale/y/acc");
    QLIN_REQUIRE(M <= 4096 && K <= 131071, QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: M=%d K=%d outside 1..4096 x 1..131071",
                 M, K);
    if (M >= qlin::kTensorCoreMinM)
        return qlin::t158_linear_tensor_cores(xq, x_scale, w_packed, w_pitch, w_scale, nullptr, y, acc, M, N, K,
                                              (cudaStream_t)stream, nullptr, false);
    return qlin::t158_linear_cuda_cores(xq, x_scale, w_packed, w_pitch, w_scale, nullptr, y, acc, M, N, K,
                                        (cudaStream_t)stream);
}

size_t qlin_t158_i8_workspace_size(int M, int K) {
    if (M < 1 || K < 1 || M > 4096 || K > 131071) return 0;
    return qlin::t158_workspace_bytes(M, K);
}

qlin_status qlin_t158_i8_ws(const int8_t *xq, const float *x_scale, const uint8_t *w_packed, int64_t w_pitch,
                            float w_scale, float *y, int32_t *acc, int M, int N, int K, void *workspace,
                            size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(xq && x_scale && w_packed && (y || acc), QLIN_ERR_INVALID_ARG, "qlin_t158_i8_ws: null pointer");
    QLIN_REQUIRE(M >= 1 && N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_t158_i8_ws: M=%d N=%d K=%d", M, N, K);
    QLIN_REQUIRE(w_pitch % 16 == 0 && w_pitch >= (K + 4) / 5, QLIN_ERR_INVALID_ARG,
                 "qlin_t158_i8_ws: w_pitch %lld must be a multiple of 16 and >= ceil(K/5)", (long long)w_pitch);
    QLIN_REQUIRE(qlin::aligned16(w_packed), QLIN_ERR_INVALID_ARG, "qlin_t158_i8_ws: w_packed not 16-byte aligned");
    QLIN_REQUIRE(qlin::aligned4(x_scale) && (!y || qlin::aligned4(y)) && (!acc || qlin::aligned4(acc)),
                 QLIN_ERR_INVALID_ARG, "qlin_t158_i8_ws: misaligned x_scale/y/acc");
    QLIN_REQUIRE(M <= 4096 && K <= 131071, QLIN_ERR_UNSUPPORTED,
                 "qlin_t158_i8_ws: M=%d K=%d outside 1..4096 x 1..131071", M, K);
    const size_t need = qlin::t158_workspace_bytes(M, K);
    QLIN_REQUIRE(workspace_bytes >= need && (need == 0 || (workspace && qlin::aligned16(workspace))),
                 QLIN_ERR_INVALID_ARG, "qlin_t158_i8_ws: workspace %zu < %zu bytes, null or not 16-byte aligned",
                 workspace_bytes, need);
    if (M >= qlin::kTensorCoreMinM)
        return qlin::t158_linear_tensor_cores(xq, x_scale, w_packed, w_pitch, w_scale, nullptr, y, acc, M, N, K,
                                              (cudaStream_t)stream, workspace, true);
    return qlin::t158_linear_cuda_cores(xq, x_scale, w_packed, w_pitch, w_scale, nullptr, y, acc, M, N, K,
                                        (cudaStream_t)stream);
}

}  // extern "C"
