// T158 linear for one token that skips groups of four zero inputs ([citric]
// "What is next": a kernel that skips groups of 4 zero inputs, faster when
// most groups are zero).
//
// The weights are stored by input group (t158_pack_groups): group g, row n is
// one byte holding the four trits t[n][4g .. 4g+3] in base 3, and a group's
// bytes for all rows are contiguous.  Every CTA lists the token's nonzero
// groups (a ballot over the int8 codes), then takes its share of that list
// for its 1024 rows: per group one 32-bit load gives four rows' bytes (the
// loads of 32 groups in flight per thread), a shared-memory table turns a
// byte into its four trits (int8 x 4) and one dp4a with the group's four
// codes adds the group to a row.  A zero group's
// weight bytes are never read.  Partial sums go to the workspace per group
// share; the last CTA of a row block adds them in share order (integers:
// exact) and writes acc and y = ((float)acc * w_scale) * x_scale.
#include <algorithm>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {
namespace {

constexpr int kSkThreads = 256;
constexpr int kSkRows = 4 * kSkThreads;  // rows per CTA: four per thread
constexpr int kSkMaxGroups = 16384;      // K <= 65536
constexpr int kSkMaxShares = 16;
constexpr int kSkBatch = 32;             // weight loads in flight per thread
constexpr int kSkListLoads = 16;         // code words per thread and round of the list (4096 groups)

__global__ void __launch_bounds__(kSkThreads, 2) t158_skip_kernel(const int8_t *__restrict__ xq,
                                                              const float *__restrict__ xs,
                                                              const uint8_t *__restrict__ wg, int64_t gpitch,
                                                              float w_scale, int N, int K, int32_t *part,
                                                              unsigned *tickets, int32_t *__restrict__ acc_out,
                                                              float *__restrict__ y) {
    extern __shared__ __align__(16) uint32_t sk_dyn[];
    const int G = (K + 3) / 4;
    uint32_t *xg = sk_dyn;                                        // [G] the listed groups' four codes
    uint16_t *list = reinterpret_cast<uint16_t *>(sk_dyn + G);  // [G] the nonzero groups
    __shared__ uint32_t tab[256];                                 // byte -> four trits (int8 x 4)
    __shared__ int last;
    const int tid = threadIdx.x;
    const int rb = blockIdx.x, share = blockIdx.y, shares = gridDim.y;
    const int Np = (N + 3) / 4 * 4;  // row stride of the partial sums (16-byte rows of four)
    {
        const uint32_t v = (uint32_t)tid;
        const uint32_t d0 = v % 3, d1 = (v / 3) % 3, d2 = (v / 9) % 3, d3 = (v / 27) % 3;
        tab[tid] = ((d0 - 1) & 0xffu) | (((d1 - 1) & 0xffu) << 8) | (((d2 - 1) & 0xffu) << 16) | ((d3 - 1) << 24);
    }
    // the nonzero groups, in the same order in every CTA (thread by thread, then
    // the thread's groups in turn), so that the CTAs of a row block split one list
    __shared__ unsigned wsum[kSkThreads / 32 + 1];
    const int lane = tid & 31, warp = tid >> 5;
    unsigned base = 0;
    for (int g0 = 0; g0 < G; g0 += kSkListLoads * kSkThreads) {
        uint32_t x4[kSkListLoads];
#pragma unroll
        for (int u = 0; u < kSkListLoads; u++) {  // every load of the round in flight
            const int g = g0 + u * kSkThreads + tid;
            uint32_t v = 0u;
            if (g < G) {
                if (4 * g + 4 <= K) {
                    v = __ldg(reinterpret_cast<const uint32_t *>(xq + 4 * g));
                } else {
                    for (int i = 0; i < 4 && 4 * g + i < K; i++) v |= (uint32_t)(uint8_t)xq[4 * g + i] << (8 * i);
                }
            }
            x4[u] = v;
        }
        unsigned c = 0;
#pragma unroll
        for (int u = 0; u < kSkListLoads; u++) c += x4[u] != 0u;
        unsigned inc = c;  // inclusive scan over the threads
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        if (tid == 0) {
            unsigned run = 0;
            for (int w = 0; w < kSkThreads / 32; w++) {
                const unsigned t = wsum[w];
                wsum[w] = run;
                run += t;
            }
            wsum[kSkThreads / 32] = run;
        }
        __syncthreads();
        unsigned p = base + wsum[warp] + inc - c;
#pragma unroll
        for (int u = 0; u < kSkListLoads; u++)
            if (x4[u] != 0u) {
                list[p] = (uint16_t)(g0 + u * kSkThreads + tid);
                xg[p] = x4[u];
                p++;
            }
        base += wsum[kSkThreads / 32];
        __syncthreads();
    }
    const int nnz = (int)base;
    // this CTA's share of the nonzero groups, for rows 1024 rb + 4 tid .. + 3
    const int j0 = (int)((int64_t)nnz * share / shares), j1 = (int)((int64_t)nnz * (share + 1) / shares);
    const int n0 = rb * kSkRows + 4 * tid;
    const bool rows_in = n0 < N;
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    if (rows_in) {
        const uint8_t *col = wg + n0;
        // batches of kSkBatch groups, every load of a batch in flight at once; a
        // slot past the share adds nothing (its codes are zero)
        for (int j = j0; j < j1; j += kSkBatch) {
            uint32_t w[kSkBatch];
#pragma unroll
            for (int u = 0; u < kSkBatch; u++)  // a slot past the share reloads the share's last group
                w[u] = __ldg(reinterpret_cast<const uint32_t *>(col + (int64_t)list[min(j + u, j1 - 1)] * gpitch));
#pragma unroll
            for (int u = 0; u < kSkBatch; u++) {
                const uint32_t x4 = j + u < j1 ? xg[min(j + u, j1 - 1)] : 0u;
                a0 = __dp4a((int)tab[w[u] & 0xffu], (int)x4, a0);
                a1 = __dp4a((int)tab[(w[u] >> 8) & 0xffu], (int)x4, a1);
                a2 = __dp4a((int)tab[(w[u] >> 16) & 0xffu], (int)x4, a2);
                a3 = __dp4a((int)tab[w[u] >> 24], (int)x4, a3);
            }
        }
        *reinterpret_cast<int4 *>(part + (int64_t)share * Np + n0) = make_int4(a0, a1, a2, a3);
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        last = atomicAdd(&tickets[rb], 1u) == (unsigned)shares - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (rows_in) {
        int4 s = make_int4(0, 0, 0, 0);
        for (int q = 0; q < shares; q++) {
            const int4 v = __ldcg(reinterpret_cast<const int4 *>(part + (int64_t)q * Np + n0));
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        const float xsv = __ldg(xs);
        const int av[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int n = n0 + r;
            if (n >= N) break;
            if (acc_out) acc_out[n] = av[r];
            if (y) y[n] = __fmul_rn(__fmul_rn((float)av[r], w_scale), xsv);
        }
    }
    if (tid == 0) tickets[rb] = 0u;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" {

size_t qlin_t158_skip_workspace_size(int N) {
    if (N < 1) return 0;
    const int rbs = (N + kSkRows - 1) / kSkRows;
    return align256((size_t)rbs * sizeof(unsigned)) + align256((size_t)kSkMaxShares * rbs * kSkRows * sizeof(int32_t));
}

qlin_status qlin_t158_i8_skip(const int8_t *xq, const float *x_scale, const uint8_t *w_groups, int64_t gpitch,
                              float w_scale, float *y, int32_t *acc, int N, int K, void *workspace,
                              size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(xq && x_scale && w_groups && (y || acc) && workspace, QLIN_ERR_INVALID_ARG,
                 "qlin_t158_i8_skip: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "qlin_t158_i8_skip: N=%d K=%d", N, K);
    QLIN_REQUIRE(K <= 4 * kSkMaxGroups, QLIN_ERR_UNSUPPORTED, "qlin_t158_i8_skip: K=%d above %d", K, 4 * kSkMaxGroups);
    QLIN_REQUIRE(gpitch >= N && gpitch % 16 == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_t158_i8_skip: gpitch %lld must be >= N and a multiple of 16", (long long)gpitch);
    QLIN_REQUIRE(aligned16(w_groups) && aligned4(xq) && aligned4(x_scale) && aligned16(workspace) &&
                     (!y || aligned4(y)) && (!acc || aligned4(acc)),
                 QLIN_ERR_INVALID_ARG, "qlin_t158_i8_skip: misaligned pointer");
    QLIN_REQUIRE(workspace_bytes >= qlin_t158_skip_workspace_size(N), QLIN_ERR_INVALID_ARG,
                 "qlin_t158_i8_skip: workspace %zu < %zu bytes", workspace_bytes, qlin_t158_skip_workspace_size(N));
    const int rbs = (N + kSkRows - 1) / kSkRows;
    // the groups split between CTAs of a row block, about 64 groups (16 nonzero at 75% zeros) each
    const int shares = std::max(1, std::min(kSkMaxShares, std::min(2 * sm_count() / rbs, ((K + 3) / 4 + 63) / 64)));
    unsigned *tickets = (unsigned *)workspace;
    int32_t *part = (int32_t *)((char *)workspace + align256((size_t)rbs * sizeof(unsigned)));
    const size_t smem = (size_t)6 * ((K + 3) / 4) + 16;
    if (smem > 48 * 1024) blocks_per_sm((const void *)t158_skip_kernel, smem);  // raises the limit once
    t158_skip_kernel<<<dim3(rbs, shares), kSkThreads, smem, (cudaStream_t)stream>>>(
        xq, x_scale, w_groups, gpitch, w_scale, N, K, part, tickets, acc, y);
    QLIN_LAUNCHED("t158_skip_kernel");
    return QLIN_OK;
}

}  // extern "C"
