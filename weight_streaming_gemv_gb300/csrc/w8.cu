// W8 linear layers: symmetric per-tensor int8 weights, fp32 activations,
// the scale applied once after the dot product (cpp20gemma README,
// "Architecture & implementation"; llama2.c "matmul" is the same loop over
// output rows).  Weights stream with 16-byte loads; each int8 is widened to
// fp32 exactly with the 2^23 magic-number trick (one byte permute and one
// subtraction) and accumulated with fp32 FMA.
#include "common.cuh"

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

// ---------------------------------------------------------------- S5 GEMV
// int8 byte j of a (bias-flipped) word -> exact fp32 value
__device__ __forceinline__ float i8_to_f32(uint32_t flipped, uint32_t sel) {
    return __fsub_rn(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel)), 8388736.0f);  // 2^23 + 128
}

// One warp handles R rows; lanes take 16-byte chunks c = lane + 32 j; the
// fp32 activations of a chunk are read from shared memory once and used for
// all R rows.  MT tokens per block.
template <int R, int MT>
__global__ void __launch_bounds__(256) w8_gemv_kernel(const float *__restrict__ x, const int8_t *__restrict__ w,
                                                      int64_t pitch, float s, float *__restrict__ y, int M, int N,
                                                      int K) {
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
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                const float4 *X = xs4 + ((size_t)mm * C + c) * 4;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float4 xv = X[q];
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        float a = acc[r][mm];
                        a = fmaf(xv.x, wf[r][4 * q + 0], a);
                        a = fmaf(xv.y, wf[r][4 * q + 1], a);
                        a = fmaf(xv.z, wf[r][4 * q + 2], a);
                        a = fmaf(xv.w, wf[r][4 * q + 3], a);
                        acc[r][mm] = a;
                    }
                }
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

template <int R, int MT>
static qlin_status launch_w8(const float *x, const int8_t *w, int64_t pitch, float s, float *y, int M, int N, int K,
                             cudaStream_t st) {
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
    kern<<<grid, 256, smem, st>>>(x, w, pitch, s, y, M, N, K);
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
    const size_t tile8_smem = (size_t)8 * ((K + 15) / 16) * 16 * sizeof(float);
    if (M == 1) return qlin::launch_w8<4, 1>(x, w8, w_pitch, w_scale, y, M, N, K, st);
    if (M <= 4 || (int)tile8_smem > qlin::max_smem_optin())
        return qlin::launch_w8<2, 4>(x, w8, w_pitch, w_scale, y, M, N, K, st);
    return qlin::launch_w8<2, 8>(x, w8, w_pitch, w_scale, y, M, N, K, st);
}

}  // extern "C"
