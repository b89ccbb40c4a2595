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
//
// The planes are built from a copy of the row in shared memory: the row is
// fetched with 16-byte loads (the bytes before the first and after the last
// 16-byte boundary one by one), so a block pays one L2 round trip for it.
// stage[off0 + k] = x[k] for k < K and 0 up to 80*C, where off0 = x mod 16
// keeps the 16-byte stores aligned; stage holds 80*C + 32 bytes.
__device__ __forceinline__ void stage_row(const int8_t *__restrict__ x, int K, int C, uint8_t *stage) {
    const int off0 = (int)((uintptr_t)x & 15);
    const uint8_t *base = reinterpret_cast<const uint8_t *>(x) - off0;  // 16-byte aligned
    const int j0 = off0 ? 1 : 0;            // first 16-byte block lying wholly inside the row
    const int j1 = max((off0 + K) >> 4, j0);  // one past the last such block
    for (int j = j0 + (int)threadIdx.x; j < j1; j += blockDim.x)
        reinterpret_cast<uint4 *>(stage)[j] = ld_stream_v4(base + 16 * (size_t)j);
    const int head = min(K, 16 * j0 - off0);  // bytes k < head precede the blocks
    const int tail = max(16 * j1 - off0, head);  // bytes k >= tail follow them
    for (int k = threadIdx.x; k < head; k += blockDim.x) stage[off0 + k] = (uint8_t)x[k];
    for (int k = tail + (int)threadIdx.x; k < K; k += blockDim.x) stage[off0 + k] = (uint8_t)x[k];
    for (int k = K + (int)threadIdx.x; k < 80 * C; k += blockDim.x) stage[off0 + k] = 0;
}

// One span is the 20 activations of the four packed bytes 4w..4w+3 of chunk c
// (s = 4c + w); plane i of the span takes its bytes i, i+5, i+10, i+15.
// Returns this thread's part of the row's byte sum (exact, signed).
__device__ __forceinline__ int planes_from_stage(const uint8_t *stage, int off0, int C, uint4 *xr) {
    uint32_t *xw = reinterpret_cast<uint32_t *>(xr);
    const uint32_t *sw = reinterpret_cast<const uint32_t *>(stage);
    const uint32_t sh = 8u * (uint32_t)(off0 & 3);
    int sum = 0;
    for (int sp = threadIdx.x; sp < 4 * C; sp += blockDim.x) {
        const int b0 = off0 + 20 * sp;  // stage index of the span's first byte
        const int q = b0 >> 2;
        uint32_t u[6], v[5];
#pragma unroll
        for (int t = 0; t < 6; t++) u[t] = sw[q + t];
#pragma unroll
        for (int t = 0; t < 5; t++) v[t] = __funnelshift_r(u[t], u[t + 1], sh);  // bytes 4t..4t+3 of the span
        // plane i = span bytes {i, i+5, i+10, i+15}
        const uint32_t p0 = __byte_perm(__byte_perm(v[0], v[1], 0x0050), __byte_perm(v[2], v[3], 0x0072), 0x5410);
        const uint32_t p1 = __byte_perm(__byte_perm(v[0], v[1], 0x0061), __byte_perm(v[2], v[4], 0x0043), 0x5410);
        const uint32_t p2 = __byte_perm(__byte_perm(v[0], v[1], 0x0072), __byte_perm(v[3], v[4], 0x0050), 0x5410);
        const uint32_t p3 = __byte_perm(__byte_perm(v[0], v[2], 0x0043), __byte_perm(v[3], v[4], 0x0061), 0x5410);
        const uint32_t p4 = __byte_perm(__byte_perm(v[1], v[2], 0x0050), __byte_perm(v[3], v[4], 0x0072), 0x5410);
        const int c = sp >> 2, w = sp & 3;
        uint32_t *o = xw + (size_t)c * 20 + w;
        o[0] = p0;
        o[4] = p1;
        o[8] = p2;
        o[12] = p3;
        o[16] = p4;
#pragma unroll
        for (int t = 0; t < 5; t++) sum = dp4a(v[t], 0x01010101u, sum);
    }
    return sum;
}

// ---------------------------------------------------------------- S4 / S6 GEMV
// LPR lanes share one packed row (chunk c = lane % LPR + LPR*j); 32/LPR rows
// per slot, R slots per warp pass.  MT tokens per block (grid.y tiles M).
// The weight chunks are double-buffered in registers: the next chunk's loads
// are in flight while the current one is decoded, and the first chunk of a
// warp's first rows is requested before the activation planes are built, so
// that its DRAM latency overlaps the plane build.
template <int LPR, int R, int MT>
__global__ void __launch_bounds__(256) t158_gemv_kernel(const int8_t *__restrict__ xq, const float *__restrict__ xs,
                                                        const uint8_t *__restrict__ w, int64_t pitch, float ws,
                                                        const float *__restrict__ ws_ptr, float *__restrict__ y, int32_t *__restrict__ acc_out,
                                                        int M, int N, int K) {
    extern __shared__ uint4 smem[];
    const int C = (int)(pitch / 16);
    uint4 *xr = smem;                                                    // [MT][C*5]
    uint8_t *stage = reinterpret_cast<uint8_t *>(smem + (size_t)MT * C * 5);  // 80*C + 32 bytes
    int *sumx = reinterpret_cast<int *>(stage + 80 * (size_t)C + 32);     // [MT]
    int *red = sumx + MT;                                                // [MT][8] warp partial sums
    const int m0 = blockIdx.y * MT;

    constexpr int RPS = 32 / LPR;
    constexpr int ROWS = RPS * R;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int warps = blockDim.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * warps;
    // Programmatic dependent launch: the packed weights are read-only inputs,
    // so the first chunks are requested before the wait; the activations,
    // their scales and the weight scale are read, and y written, only after
    // the previous kernel on the stream has completed (griddepcontrol.wait).
    // The next kernel may launch once every CTA has begun its last row pass
    // (below): launched at the start instead, its early reads slowed these
    // latency-bound calls down.
    uint4 nxt[R];  // the next chunk of each of the warp's R row slots
#pragma unroll
    for (int r = 0; r < R; r++) {
        const int64_t row = gwarp * ROWS + r * RPS + rsub;
        nxt[r] = (row < N && sub < C) ? ld_stream_v4(w + row * pitch + (int64_t)sub * 16) : make_uint4(0, 0, 0, 0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const float wsv = ws_ptr ? *ws_ptr : ws;
    for (int mm = 0; mm < MT; mm++) {
        const int m = m0 + mm;
        int part = 0;
        if (m < M) {
            const int8_t *xrow = xq + (int64_t)m * K;
            if (mm > 0) __syncthreads();  // the previous token's planes have been read from the stage
            stage_row(xrow, K, C, stage);
            __syncthreads();
            part = planes_from_stage(stage, (int)((uintptr_t)xrow & 15), C, xr + (size_t)mm * C * 5);
        } else {
            for (int idx = threadIdx.x; idx < C * 5; idx += blockDim.x) xr[(size_t)mm * C * 5 + idx] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) red[mm * 8 + (threadIdx.x >> 5)] = part;
    }
    __syncthreads();
    if (threadIdx.x < MT) {
        int t = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) t += red[threadIdx.x * 8 + i];
        sumx[threadIdx.x] = t;
    }
    __syncthreads();

    for (int64_t r0 = gwarp * ROWS; r0 < N; r0 += nwarps * ROWS) {
        if (r0 + nwarps * ROWS >= N) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        int acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int mm = 0; mm < MT; mm++) acc[r][mm] = 0;
        if (r0 != gwarp * ROWS) {
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t row = r0 + r * RPS + rsub;
                nxt[r] = (row < N && sub < C) ? ld_stream_v4(w + row * pitch + (int64_t)sub * 16) : make_uint4(0, 0, 0, 0);
            }
        }

        for (int c = sub; c < C; c += LPR) {
            uint4 wv[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t row = r0 + r * RPS + rsub;
                // wide rows: the chunk two iterations ahead toward L2 (more bytes in flight per warp)
                if (LPR == 32 && row < N && c + 2 * LPR < C)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(w + row * pitch + (int64_t)(c + 2 * LPR) * 16));
                wv[r] = nxt[r];
                nxt[r] = (row < N && c + LPR < C) ? ld_stream_v4(w + row * pitch + (int64_t)(c + LPR) * 16)
                                                  : make_uint4(0, 0, 0, 0);
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
    const size_t smem = (size_t)MT * C * 5 * sizeof(uint4) + 80 * (size_t)C + 32 + (size_t)MT * 9 * sizeof(int);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "qlin_t158_i8: K=%d needs %zu B of shared memory",
                 K, smem);
    const int per_sm = blocks_per_sm((const void *)kern, smem);
    constexpr int ROWS = (32 / LPR) * R;
    const int64_t warps_needed = (N + ROWS - 1) / ROWS;
    int64_t blocks = (warps_needed + 7) / 8;
    // each block builds the activation planes once: at most three blocks per
    // SM for one token (two for several), so that they serve more rows each
    // (the grid-stride loop takes the rest)
    const int64_t cap = (int64_t)sm_count() * std::min(per_sm, MT == 1 ? 3 : 2);
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, (unsigned)((M + MT - 1) / MT));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // Programmatic stream serialisation: the launch and the first weight reads
    // overlap the previous kernel's last row passes (6912 -> 1152 at one
    // token: 3.9 -> 3.4 us per call in a graph of back-to-back calls; with the
    // kernel's trigger at its start instead: 6.3 us).
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QLIN_CUDA(cudaLaunchKernelEx(&cfg, kern, xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K));
    QLIN_LAUNCHED("t158_gemv_kernel");
    return QLIN_OK;
}

// Row slots per warp: the most (up to RMAX) that still give every SM a block.
template <int LPR, int MT, int RMAX>
static qlin_status launch_slots(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                                const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    const int64_t blocks_r1 = ((int64_t)N + (32 / LPR) * 8 - 1) / ((32 / LPR) * 8);
    if constexpr (RMAX >= 4)
        if (blocks_r1 >= 4LL * sm_count()) return launch_t158<LPR, 4, MT>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (blocks_r1 >= 2LL * sm_count()) return launch_t158<LPR, 2, MT>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    return launch_t158<LPR, 1, MT>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
}

// Tokens per block: 1, 2, 4, then 8 (grid.y takes the rest; the public entry
// points send 8 tokens and more to the tensor cores).
template <int LPR>
static qlin_status dispatch_mt(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch, float ws,
                               const float *ws_ptr, float *y, int32_t *acc, int M, int N, int K, cudaStream_t st) {
    if (M == 1) return launch_slots<LPR, 1, 4>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (M == 2) return launch_slots<LPR, 2, 4>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    if (M <= 4) return launch_slots<LPR, 4, 2>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
    return launch_slots<LPR, 8, 2>(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st);
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
    // the activation planes of a block's tokens and the staged row must fit in
    // shared memory; past that (very long rows) the tensor-core kernel, which
    // streams K in steps, takes the call: the same acc and y
    const int MT = M == 1 ? 1 : M == 2 ? 2 : M <= 4 ? 4 : 8;
    if ((size_t)MT * C * 80 + 80 * (size_t)C + 32 + (size_t)MT * 9 * sizeof(int) > (size_t)max_smem_optin())
        return t158_linear_tensor_cores(xq, xs, w, pitch, ws, ws_ptr, y, acc, M, N, K, st, nullptr, true);
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
