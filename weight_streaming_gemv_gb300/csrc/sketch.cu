// Sketch head for the output layer ([citric] "Step 3: the output layer became
// the bottleneck"): pick candidate words first, score only those exactly.
//
//   1. the k dimensions of x with the largest |x_d| are scored exactly for
//      every word, from a dimension-major copy of the table (k rows of it);
//   2. the other dimensions are scored from a 1-bit copy of the table (the
//      sign bits), one XOR and one bit count per 64-dimension block of a word.
//      The blocks follow a fixed order of the dimensions by size, chosen when
//      the table is prepared; block b has its own weight w_b = (mean |x_d| over
//      its sketched dims) * c_E, and word v gets sum_b w_b (n_b - 2 m_b), m_b =
//      how many signs of block b differ between E[v] and x;
//   3. the n_cand words with the best approximate scores are scored exactly;
//      every other word scores minus infinity; next = their first maximum.
//
// GB300 mapping: one persistent cooperative kernel, one CTA per SM, each CTA
// owning a contiguous range of words.
//   * A producer warp streams the range through a ring of shared-memory
//     stages with 1-D bulk copies (TMA): per stage, the sign words of every
//     block row ([block][word], contiguous) and the k exact rows of the
//     dimension-major copy.  The sign copies of the first stages go out at
//     kernel start, while the CTA ranks the dimensions of x; the exact rows
//     follow once the k strongest dims are known.
//   * 16 consumer warps score one word per lane from shared memory: k
//     products summed as a fixed pairwise tree, then per block one 64-bit
//     XOR with x's sign bits, a mask of the sketched dims and a bit count.
//     Each word's 32-bit order key stays in shared memory; a 12-bit
//     histogram of the keys goes to global memory.
//   * One grid barrier.  Every CTA reads the histogram, finds the bin of the
//     n_cand-th largest key, and rescores (with the lm_head's arithmetic) its
//     words at or above that bin -- a superset of its candidates of about
//     n_cand plus one bin in all.  The last CTA to finish picks the exact
//     n_cand among them (a radix select over the boundary bin, ties to the
//     lower index), writes them in ascending order and reduces the argmax.
//   * If the superset is too large to resolve in one CTA (massive ties), the
//     CTAs finish the radix select together instead (two more barriers),
//     write the candidates in word order and rescore their own.
//
// fp32 order (fixed, so that any implementation picks the same candidates):
// exact part = pairwise sum of bf16(E[v][d]) * x_d over the k dims in
// ascending d, zero-padded to a power of two; a block's |x| sum = pairwise sum
// over its 64 positions in order (exact dims and positions past D count +0);
// w_b = sum / n_b * c_E; sketch = sum over b ascending of w_b * (n_b - 2 m_b)
// with every product rounded; approx = exact + sketch.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "stream.cuh"

namespace qlin {
namespace {

constexpr int kSkConsumerWarps = 16;
constexpr int kSkWarps = kSkConsumerWarps + 1;  // + the producer warp
constexpr int kSkThreads = 32 * kSkWarps;
constexpr int kSkStages = 4;  // consumer groups divide it (see the scoring loop)
constexpr int kSkRingBudget = 180 * 1024;  // bytes of shared memory for the stages
constexpr int kSkMaxDim = 2048;
constexpr int kSkMaxK = 32;
constexpr int kSkBlockDims = 64;                          // dims per sign word (one group)
constexpr int kSkMaxBlocks = kSkMaxDim / kSkBlockDims;  // sign words per table row
constexpr int kSkBins1 = 4096;  // key bits 31..20
constexpr int kSkBins2 = 1024;  // key bits 19..10
constexpr int kSkBins3 = 1024;  // key bits 9..0
constexpr int kSkHistWords = kSkBins1 + kSkBins2 + kSkBins3;
constexpr int kSkTile = 32;        // words per range unit
constexpr int kSkSub = 64;         // words per warp pass (two per lane)
constexpr int kSkCap = 4096;       // superset words one CTA resolves
constexpr int kSkMemberCap = kSkThreads;  // dims of the boundary magnitude bin ranked pairwise

// Workspace: status first (qlin_sketch_head_status reads offset 0).
struct SketchWs {
    int32_t *status;
    unsigned *bar;     // [2]: arrivals (zero between calls), generation
    unsigned *ticket;  // CTAs done (zero between calls)
    unsigned *tcount;  // superset words written (zero between calls)
    unsigned *info;    // [4] the boundary bin, words above it, superset size (written each call)
    unsigned *hist;    // [kSkHistWords] (zero between calls)
    uint2 *counts;     // [blocks] words above / equal to the threshold per CTA
    float2 *part;      // [blocks] best (logit, index) per CTA
    uint2 *segs;       // [blocks] (offset, count) of each CTA's superset words
    uint32_t *tkey;    // [kSkCap] superset: order key,
    int32_t *tidx;     //          word,
    float *tlogit;     //          exact logit
};

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

int max_blocks() { return sm_count(); }

SketchWs carve(char *base, size_t *bytes) {
    SketchWs w{};
    size_t off = 0;
    auto take = [&](size_t b) {
        char *p = base ? base + off : nullptr;
        off += align256(b);
        return p;
    };
    w.status = (int32_t *)take(16);
    w.bar = (unsigned *)take(8);
    w.ticket = (unsigned *)take(4);
    w.tcount = (unsigned *)take(4);
    w.info = (unsigned *)take(16);
    w.hist = (unsigned *)take(4 * (size_t)kSkHistWords);
    w.counts = (uint2 *)take(sizeof(uint2) * (size_t)max_blocks());
    w.part = (float2 *)take(sizeof(float2) * (size_t)max_blocks());
    w.segs = (uint2 *)take(sizeof(uint2) * (size_t)max_blocks());
    w.tkey = (uint32_t *)take(4 * (size_t)kSkCap);
    w.tidx = (int32_t *)take(4 * (size_t)kSkCap);
    w.tlogit = (float *)take(4 * (size_t)kSkCap);
    if (bytes) *bytes = off;
    return w;
}

int64_t emb_t_pitch(int V) { return ((int64_t)V + 7) / 8 * 8; }

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Every CTA of the (co-resident, cooperatively launched) grid arrives; the
// last one opens the next generation.  The wait is bounded: on timeout the
// status gets kStatusTimeout and the CTA is told to stop.
__device__ bool grid_barrier(unsigned *bar, int32_t *status, int *flag_s) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *count = bar, *gen = bar + 1;
        const unsigned g = ld_acquire_u32(gen);
        __threadfence();
        int ok = 1;
        if (atomicAdd(count, 1u) == gridDim.x - 1) {
            atomicExch(count, 0u);
            __threadfence();
            st_release_u32(gen, g + 1);
        } else {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u32(gen) == g) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    raise_status(status, kStatusTimeout);
                    ok = 0;
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        *flag_s = ok;
    }
    __syncthreads();
    return *flag_s != 0;
}

// Exclusive prefix sum over the CTA's threads in thread order; *total gets
// the sum of all.  tmp: 33 words of shared memory.
__device__ unsigned block_scan(unsigned v, unsigned *tmp, unsigned *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    unsigned inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const unsigned w = lane < nwarps ? tmp[lane] : 0u;
        unsigned wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < nwarps) tmp[lane] = wi - w;
        if (lane == nwarps - 1) tmp[32] = wi;
    }
    __syncthreads();
    const unsigned r = tmp[warp] + inc - v;
    *total = tmp[32];
    __syncthreads();
    return r;
}

// The bin of h (nbins, counted from the top) that holds the need-th largest
// key (1 <= need <= total), and how many keys lie in the bins above it.  h is
// in global memory (filled by every CTA; read through L2) or shared memory.
template <bool kGlobal>
__device__ void find_bin(const unsigned *h, int nbins, unsigned need, unsigned *tmp, int *bin_s,
                         unsigned *above_s) {
    const int per = (nbins + (int)blockDim.x - 1) / (int)blockDim.x;
    const int hi = max(0, nbins - per * (int)threadIdx.x);  // this thread owns bins [lo, hi)
    const int lo = max(0, hi - per);
    unsigned s = 0;
    for (int b = hi - 1; b >= lo; b--) s += kGlobal ? __ldcg(h + b) : h[b];
    unsigned total;
    const unsigned pre = block_scan(s, tmp, &total);
    if (pre < need && need <= pre + s) {
        unsigned acc = pre;
        for (int b = hi - 1; b >= lo; b--) {
            const unsigned c = kGlobal ? __ldcg(h + b) : h[b];
            if (acc + c >= need) {
                *bin_s = b;
                *above_s = acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

// Order-preserving map of a float to 32 bits (larger float, larger key);
// -0 and +0 share a key, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Exact logit of one row with the lm_head's arithmetic: 16 lanes per row,
// lane s takes 8-dim chunks s, s+16, ... with fused multiply-adds in
// dimension order, then a butterfly over the 16 lanes.  NCH >= the chunks of
// a lane (all its loads are issued first).  Called by whole warps; rows of the
// two half-warps may differ; invalid rows give 0.
template <int NCH>
__device__ __forceinline__ float row_logit(const uint16_t *emb, int D, int word, bool valid, const float *xv) {
    const int sub = threadIdx.x & 15, C = D / 8;
    const uint4 *row = reinterpret_cast<const uint4 *>(emb + (int64_t)word * D);
    uint4 w[NCH];
#pragma unroll
    for (int i = 0; i < NCH; i++)
        if (valid && sub + 16 * i < C) w[i] = ld_stream_v4(row + sub + 16 * i);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < NCH; i++) {
        const int c = sub + 16 * i;
        if (valid && c < C) {
            const float4 xa = *reinterpret_cast<const float4 *>(xv + 8 * c);
            const float4 xb = *reinterpret_cast<const float4 *>(xv + 8 * c + 4);
            acc = fmaf(__uint_as_float(w[i].x << 16), xa.x, acc);
            acc = fmaf(__uint_as_float(w[i].x & 0xffff0000u), xa.y, acc);
            acc = fmaf(__uint_as_float(w[i].y << 16), xa.z, acc);
            acc = fmaf(__uint_as_float(w[i].y & 0xffff0000u), xa.w, acc);
            acc = fmaf(__uint_as_float(w[i].z << 16), xb.x, acc);
            acc = fmaf(__uint_as_float(w[i].z & 0xffff0000u), xb.y, acc);
            acc = fmaf(__uint_as_float(w[i].w << 16), xb.z, acc);
            acc = fmaf(__uint_as_float(w[i].w & 0xffff0000u), xb.w, acc);
        }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

// Histogram of bits [bshift, bshift + log2 nbins) of the keys whose bits from
// `shift` up equal prefix (all keys when shift >= 32), into shared memory.
__device__ void hist_pass(const uint32_t *keys, int n, int shift, uint32_t prefix, int bshift, int nbins,
                          unsigned *h) {
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const uint32_t key = keys[i];
        if (shift >= 32 || (key >> shift) == prefix) atomicAdd(&h[(key >> bshift) & (uint32_t)(nbins - 1)], 1u);
    }
    __syncthreads();
}

// The argmax over a CTA: every thread offers (v, i); thread 0 gets the best.
__device__ void block_best(float &v, int &i, float *wbv, int *wbi) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
    __syncthreads();
    if (lane == 0) {
        wbv[warp] = v;
        wbi[warp] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int w = 1; w < (int)(blockDim.x >> 5); w++)
            if (better(wbv[w], wbi[w], v, i)) {
                v = wbv[w];
                i = wbi[w];
            }
}

struct SkSmem {
    int ring, bars, hist, xv, pv, isx, mem, topd, xt, bmx, bwn, tmp, misc, wbv, wk, sel, total;
};

// Shared-memory carve: ring_bytes of stages (the ring region is at least
// 12 * kSkCap bytes: the last CTA's copy of the superset), range_words words
// per CTA.
__host__ __device__ inline SkSmem sk_layout(int ring_bytes, int range_words) {
    SkSmem s{};
    int o = 0;
    auto take = [&](int b) {
        const int r = o;
        o += (b + 127) / 128 * 128;
        return r;
    };
    // the stages; afterwards the last CTA's copy of the superset (key, word, logit)
    s.ring = take(ring_bytes > 12 * kSkCap ? ring_bytes : 12 * kSkCap);
    s.bars = take(16 * kSkStages);
    s.hist = take(4 * kSkBins1);
    s.xv = take(4 * kSkMaxDim);
    s.pv = take(4 * kSkMaxDim);
    s.isx = take(kSkMaxDim);
    s.mem = take(4 * kSkMemberCap);
    s.topd = take(4 * kSkMaxK);
    s.xt = take(4 * kSkMaxK);
    s.bmx = take(16 * kSkMaxBlocks);  // per block: sketched-dim mask, x's sign bits (64 bits each)
    s.bwn = take(8 * kSkMaxBlocks);   // per block: weight, sketched-dim count
    s.tmp = take(4 * 40);
    s.misc = take(4 * 16);
    s.wbv = take(8 * kSkWarps);
    s.wk = take(4 * range_words);   // each word's order key
    s.sel = take(4 * range_words);  // this CTA's candidates (superset or final)
    s.total = o;
    return s;
}

struct SketchArgs {
    const uint16_t *emb;    // [V][D] bf16
    const uint16_t *emb_t;  // [D][Vt] bf16
    const uint64_t *signs;  // [nblk][Vt]
    const int32_t *perm;    // [D] the size order of the dimensions
    const float *c_e;
    const float *x;
    int V, D, Vt, nblk, k, n_cand, tiles, range_tiles, chunk;  // chunk: words per stage (multiple of 32)
    int ring_bytes;
    float *approx;
    int32_t *cand;
    float *cand_logits;
    int32_t *next;
    SketchWs ws;
};

// MAXB: sign words per table row the kernel is compiled for (>= ceil(D / 64)).
template <int MAXB>
__global__ void __launch_bounds__(kSkThreads, 1) sketch_head_kernel(SketchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int range_words = kSkTile * a.range_tiles;
    const SkSmem L = sk_layout(a.ring_bytes, range_words);
    uint8_t *ringp = smem + L.ring;
    Ring<kSkStages> *ring = reinterpret_cast<Ring<kSkStages> *>(smem + L.bars);
    unsigned *hist_s = reinterpret_cast<unsigned *>(smem + L.hist);
    float *xv = reinterpret_cast<float *>(smem + L.xv);
    int *pv = reinterpret_cast<int *>(smem + L.pv);
    uint8_t *isx = smem + L.isx;
    int *mem = reinterpret_cast<int *>(smem + L.mem);
    int *topd = reinterpret_cast<int *>(smem + L.topd);
    float *xt = reinterpret_cast<float *>(smem + L.xt);
    uint4 *bmx = reinterpret_cast<uint4 *>(smem + L.bmx);
    float2 *bwn = reinterpret_cast<float2 *>(smem + L.bwn);
    unsigned *tmp = reinterpret_cast<unsigned *>(smem + L.tmp);
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    float *wbv = reinterpret_cast<float *>(smem + L.wbv);
    int *wbi = reinterpret_cast<int *>(smem + L.wbv + 4 * kSkWarps);
    uint32_t *wkey = reinterpret_cast<uint32_t *>(smem + L.wk);
    int *sel = reinterpret_cast<int *>(smem + L.sel);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = a.V, D = a.D, k = a.k, nblk = a.nblk, W = a.chunk;
    const int t0 = (int)((int64_t)a.tiles * blockIdx.x / gridDim.x);
    const int t1 = (int)((int64_t)a.tiles * (blockIdx.x + 1) / gridDim.x);
    const int w0 = kSkTile * t0;
    const int nw = max(0, min(kSkTile * t1, V) - w0);  // words of this CTA
    const int nchunks = (nw + W - 1) / W;
    const size_t stage_bytes = (size_t)W * 8 * nblk;
    const bool producer = warp == kSkConsumerWarps;
    // Consumer warps form `groups` groups of gsize warps; group g takes the
    // chunks c = g (mod groups), one 64-word sub-tile per warp at a time.
    // groups divides kSkStages, so chunk c - kSkStages (the previous fill of
    // the stage chunk c waits on) belongs to the same group and has landed:
    // a waiter is never two phases ahead of a stage's full barrier, where
    // the parity would name an old phase.
    const int gsize = min(kSkConsumerWarps, W / kSkSub);
    const int groups = kSkConsumerWarps / gsize >= kSkStages ? kSkStages : kSkConsumerWarps / gsize >= 2 ? 2 : 1;
    // words, sign bytes and exact-row bytes of chunk c
    auto chunk_words = [&](int c) { return min(W, nw - c * W); };
    auto sign_bytes = [&](int c) { return (uint32_t)((chunk_words(c) + 1) / 2 * 16); };

    if (tid == 0) ring->init(gsize);
    for (int d = tid; d < D; d += kSkThreads) {
        xv[d] = a.x[d];
        const int pd = a.perm[d];
        pv[d] = (pd >= 0 && pd < D) ? pd : -1;  // an entry out of range (not from preparation) drops out
    }
    for (int i = tid; i < 2048; i += kSkThreads) hist_s[i] = 0u;
    __syncthreads();
    const uint64_t pol = l2_evict_first();
    if (producer) {  // the sign words of the first stages need nothing from x
        for (int c = 0; c < min(kSkStages, nchunks); c++) {
            uint8_t *st = ringp + (size_t)c * stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&ring->full[c], (uint32_t)nblk * sign_bytes(c));
            __syncwarp();
            for (int b = lane; b < nblk; b += 32)
                bulk_g2s(st + (size_t)b * W * 8, a.signs + (int64_t)b * a.Vt + w0 + c * W, sign_bytes(c),
                         &ring->full[c], pol);
        }
    }

    // ---------------------------------------------------------------- set-up
    // the k strongest dims: a histogram of the top 11 bits of |x| finds the
    // boundary bin; its members are ranked pairwise (|x| descending, ties to
    // the lower index); a very full boundary bin falls back to two more radix
    // passes and an index-ordered count of the ties.
    if (k > 0) {
        const uint32_t *xb = reinterpret_cast<const uint32_t *>(xv);
        for (int d = tid; d < D; d += kSkThreads) atomicAdd(&hist_s[(xb[d] & 0x7fffffffu) >> 20], 1u);
        __syncthreads();
        find_bin<false>(hist_s, 2048, (unsigned)k, tmp, misc + 0, (unsigned *)misc + 1);
        const uint32_t bA = (uint32_t)misc[0];
        unsigned need = (unsigned)k - (unsigned)misc[1];
        const unsigned members = hist_s[bA];
        if (tid == 0) misc[2] = 0;
        __syncthreads();
        if (members <= (unsigned)kSkMemberCap) {
            for (int d = tid; d < D; d += kSkThreads) {
                const uint32_t m = xb[d] & 0x7fffffffu;
                isx[d] = (m >> 20) > bA;
                if ((m >> 20) == bA) mem[atomicAdd(misc + 2, 1)] = d;
            }
            __syncthreads();
            if (tid < (int)members) {
                const int d = mem[tid];
                const uint32_t m = xb[d] & 0x7fffffffu;
                unsigned r = 0;
                for (int i = 0; i < (int)members; i++) {
                    const int e = mem[i];
                    const uint32_t me = xb[e] & 0x7fffffffu;
                    r += (me > m || (me == m && e < d)) ? 1u : 0u;
                }
                isx[d] = r < need;
            }
        } else {
            uint32_t prefix = bA;
#pragma unroll 1
            for (int pass = 0; pass < 2; pass++) {
                const int bshift = pass == 0 ? 10 : 0;
                for (int i = tid; i < 1024; i += kSkThreads) hist_s[i] = 0u;
                __syncthreads();
                for (int d = tid; d < D; d += kSkThreads) {
                    const uint32_t m = xb[d] & 0x7fffffffu;
                    if ((m >> (bshift + 10)) == prefix) atomicAdd(&hist_s[(m >> bshift) & 1023u], 1u);
                }
                __syncthreads();
                find_bin<false>(hist_s, 1024, need, tmp, misc + 0, (unsigned *)misc + 1);
                prefix = (prefix << 10) | (uint32_t)misc[0];
                need -= (unsigned)misc[1];
            }
            const uint32_t T = prefix;
            const int per = (D + kSkThreads - 1) / kSkThreads;
            const int d0 = min(D, per * tid), d1 = min(D, d0 + per);
            unsigned n_eq = 0;
            for (int d = d0; d < d1; d++) n_eq += (xb[d] & 0x7fffffffu) == T;
            unsigned tot;
            unsigned er = block_scan(n_eq, tmp, &tot);
            for (int d = d0; d < d1; d++) {
                const uint32_t m = xb[d] & 0x7fffffffu;
                isx[d] = m > T || (m == T && er < need);
                er += m == T;
            }
        }
    } else {
        for (int d = tid; d < D; d += kSkThreads) isx[d] = 0;
    }
    __syncthreads();
    {  // the exact dims in ascending order
        const int per = (D + kSkThreads - 1) / kSkThreads;
        const int d0 = min(D, per * tid), d1 = min(D, d0 + per);
        unsigned n_x = 0;
        for (int d = d0; d < d1; d++) n_x += isx[d];
        unsigned tot;
        unsigned pos = block_scan(n_x, tmp, &tot);
        for (int d = d0; d < d1; d++)
            if (isx[d]) {
                topd[pos] = d;
                xt[pos] = xv[d];
                pos++;
            }
    }
    // per block: sketched-dim mask, x's sign bits, count and weight
    {
        const float cE = __ldg(a.c_e);
        for (int b = warp; b < nblk; b += kSkWarps) {
            uint64_t ne = 0, xs = 0;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int i = kSkBlockDims * b + 32 * h + lane;
                const int d = i < D ? pv[i] : -1;
                const bool in = d >= 0 && !isx[d];
                const unsigned mi = __ballot_sync(0xffffffffu, in);
                const unsigned si = __ballot_sync(0xffffffffu, in && (__float_as_uint(xv[in ? d : 0]) >> 31));
                ne |= (uint64_t)mi << (32 * h);
                xs |= (uint64_t)si << (32 * h);
            }
            // pairwise sum of |x| over positions 64b .. 64b+63: lane holds 2 lane, 2 lane + 1
            const int i0 = kSkBlockDims * b + 2 * lane;
            const int d0 = i0 < D ? pv[i0] : -1;
            const int d1 = i0 + 1 < D ? pv[i0 + 1] : -1;  // pv entries are -1 or in range
            const float v0 = (d0 >= 0 && !isx[d0]) ? fabsf(xv[d0]) : 0.0f;
            const float v1 = (d1 >= 0 && !isx[d1]) ? fabsf(xv[d1]) : 0.0f;
            float s = __fadd_rn(v0, v1);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
            if (lane == 0) {
                const int n = __popcll(ne);
                bmx[b] = make_uint4((uint32_t)ne, (uint32_t)(ne >> 32), (uint32_t)xs, (uint32_t)(xs >> 32));
                bwn[b] = make_float2(n > 0 ? __fmul_rn(__fdiv_rn(s, (float)n), cE) : 0.0f, __int_as_float(n));
            }
        }
    }
    for (int i = tid; i < kSkBins1; i += kSkThreads) hist_s[i] = 0u;
    __syncthreads();

    // ---------------------------------------------------------------- approximate scores
    if (producer) {
        int c = kSkStages;
        for (; c < nchunks; c++) {
            const int s = c % kSkStages;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&ring->empty[s], ((c / kSkStages) - 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_status(a.ws.status, kStatusTimeout);
                break;
            }
            uint8_t *st = ringp + (size_t)s * stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&ring->full[s], (uint32_t)nblk * sign_bytes(c));
            __syncwarp();
            for (int b = lane; b < nblk; b += 32)
                bulk_g2s(st + (size_t)b * W * 8, a.signs + (int64_t)b * a.Vt + w0 + c * W, sign_bytes(c),
                         &ring->full[s], pol);
        }
        // every copy issued must have landed before the CTA moves on
        if (lane == 0) {
            const int issued = min(c, nchunks);
            for (int u = max(0, issued - kSkStages); u < issued; u++)
                if (!mbar_wait(&ring->full[u % kSkStages], (u / kSkStages) & 1))
                    raise_status(a.ws.status, kStatusTimeout);
        }
    } else if (warp < groups * gsize) {
        const int grp = warp / gsize, wg = warp % gsize;
#pragma unroll 1
        for (int c = grp; c < nchunks; c += groups) {
            const int s = c % kSkStages;
            const int ncw = chunk_words(c);
            // the exact rows of this warp's first sub-tile: coalesced loads issued before the stage wait
            uint32_t raw[kSkMaxK];
            {
                const int v = w0 + c * W + wg * kSkSub + 2 * lane;
                const bool any = wg * kSkSub < ncw && v < V;
#pragma unroll
                for (int j = 0; j < kSkMaxK; j++)
                    raw[j] = (any && j < k) ? __ldg(reinterpret_cast<const uint32_t *>(a.emb_t + (int64_t)topd[j] * a.Vt + v)) : 0u;
            }
            if (!mbar_wait(&ring->full[s], (c / kSkStages) & 1)) {
                raise_status(a.ws.status, kStatusTimeout);
                break;
            }
            const uint64_t *sg = reinterpret_cast<const uint64_t *>(ringp + (size_t)s * stage_bytes);
#pragma unroll 1
            for (int sub = wg; sub * kSkSub < ncw; sub += gsize) {
                const int vl = sub * kSkSub + 2 * lane;  // this lane's two words: vl, vl + 1
                if (sub != wg) {
                    const int v = w0 + c * W + vl;
#pragma unroll
                    for (int j = 0; j < kSkMaxK; j++)
                        raw[j] = (v < V && j < k) ? __ldg(reinterpret_cast<const uint32_t *>(a.emb_t + (int64_t)topd[j] * a.Vt + v)) : 0u;
                }
                // exact part: a streaming pairwise tree per word (slot l holds a
                // finished subtree of 2^l products; element j merges with the
                // slots of its trailing one bits), zero-padded up to P
                float p0[6], p1[6];
#pragma unroll
                for (int l = 0; l < 6; l++) p0[l] = p1[l] = 0.0f;
                const int P = k > 0 ? 1 << (32 - __clz(k - 1)) : 0;
#pragma unroll
                for (int j = 0; j < kSkMaxK; j++)
                    if (j < P) {
                        float c0 = 0.0f, c1 = 0.0f;
                        if (j < k) {
                            const uint32_t pr = raw[j];
                            const float xj = xt[j];
                            c0 = __fmul_rn(__uint_as_float(pr << 16), xj);
                            c1 = __fmul_rn(__uint_as_float(pr & 0xffff0000u), xj);
                        }
#pragma unroll
                        for (int l = 0; l < 6; l++) {
                            if (l < 5 && ((j >> l) & 1)) {
                                c0 = __fadd_rn(p0[l], c0);
                                c1 = __fadd_rn(p1[l], c1);
                            } else {
                                p0[l] = c0;
                                p1[l] = c1;
                                break;
                            }
                        }
                    }
                const int lv = k > 0 ? 32 - __clz(k - 1) : 0;  // the root of the P-tree sits in slot log2 P
                float exact0 = 0.0f, exact1 = 0.0f;
#pragma unroll
                for (int l = 0; l < 6; l++)
                    if (k > 0 && l == lv) {
                        exact0 = p0[l];
                        exact1 = p1[l];
                    }
                float sk0 = 0.0f, sk1 = 0.0f;
#pragma unroll
                for (int b = 0; b < MAXB; b++)
                    if (b < nblk) {
                        const uint4 sw = *reinterpret_cast<const uint4 *>(sg + (size_t)b * W + vl);
                        const uint4 mx = bmx[b];
                        const float2 wn = bwn[b];
                        const int n = __float_as_int(wn.y);
                        const int m0 = __popc((sw.x ^ mx.z) & mx.x) + __popc((sw.y ^ mx.w) & mx.y);
                        const int m1 = __popc((sw.z ^ mx.z) & mx.x) + __popc((sw.w ^ mx.w) & mx.y);
                        sk0 = __fadd_rn(sk0, __fmul_rn(wn.x, (float)(n - 2 * m0)));
                        sk1 = __fadd_rn(sk1, __fmul_rn(wn.x, (float)(n - 2 * m1)));
                    }
#pragma unroll
                for (int h = 0; h < 2; h++)
                    if (vl + h < ncw) {
                        const int v = w0 + c * W + vl + h;
                        const float ap = __fadd_rn(h ? exact1 : exact0, h ? sk1 : sk0);
                        if (a.approx) a.approx[v] = ap;
                        const uint32_t key = order_key(ap);
                        wkey[v - w0] = key;
                        atomicAdd(&hist_s[key >> 20], 1u);
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring->empty[s]);
        }
    }
    __syncthreads();
    for (int i = tid; i < kSkBins1; i += kSkThreads)
        if (hist_s[i]) atomicAdd(&a.ws.hist[i], hist_s[i]);
    // ---------------------------------------------------------------- the boundary bin
    // A grid barrier whose last arrival (every histogram is in) finds the bin
    // of the n_cand-th largest key before it opens the barrier.
    __syncthreads();
    if (tid == 0) {
        const unsigned g = ld_acquire_u32(a.ws.bar + 1);
        __threadfence();
        misc[9] = atomicAdd(a.ws.bar, 1u) == gridDim.x - 1;
        misc[10] = (int)g;
    }
    __syncthreads();
    if (misc[9]) {
        __threadfence();
        find_bin<true>(a.ws.hist, kSkBins1, (unsigned)a.n_cand, tmp, misc + 0, (unsigned *)misc + 1);
        if (tid == 0) {
            a.ws.info[0] = (unsigned)misc[0];
            a.ws.info[1] = (unsigned)misc[1];
            a.ws.info[2] = (unsigned)misc[1] + __ldcg(a.ws.hist + misc[0]);
            atomicExch(a.ws.bar, 0u);
            __threadfence();
            st_release_u32(a.ws.bar + 1, (unsigned)misc[10] + 1);
        }
    } else if (tid == 0) {
        const uint64_t tw = global_ns();
        while (ld_acquire_u32(a.ws.bar + 1) == (unsigned)misc[10]) {
            if (global_ns() - tw > kWaitLimitNs) {
                raise_status(a.ws.status, kStatusTimeout);
                misc[9] = -1;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
    }
    __syncthreads();
    if (misc[9] < 0) return;
    const uint32_t b1 = __ldcg(a.ws.info + 0);
    const unsigned above1 = __ldcg(a.ws.info + 1);
    const unsigned superset = __ldcg(a.ws.info + 2);
    const int per = (nw + kSkThreads - 1) / kSkThreads;
    const int c0 = min(nw, per * tid), c1 = min(nw, c0 + per);

    if (superset <= (unsigned)kSkCap) {
        // ------------------------------------------------------------ fast path: rescore the superset
        unsigned n_sup = 0;
        for (int i = c0; i < c1; i++) n_sup += (wkey[i] >> 20) >= b1;
        unsigned blk;
        unsigned pos = block_scan(n_sup, tmp, &blk);
        if (tid == 0) {
            const unsigned off = atomicAdd(a.ws.tcount, blk);
            a.ws.segs[blockIdx.x] = make_uint2(off, blk);
            misc[3] = (int)off;
        }
        __syncthreads();
        const unsigned off = (unsigned)misc[3];
        for (int i = c0; i < c1; i++)
            if ((wkey[i] >> 20) >= b1) {
                sel[pos] = w0 + i;
                a.ws.tkey[off + pos] = wkey[i];
                a.ws.tidx[off + pos] = w0 + i;
                pos++;
            }
        __syncthreads();
        for (int jw = 2 * warp; jw < (int)blk; jw += 2 * kSkWarps) {  // warp-uniform trip count
            const int j = jw + (lane >> 4);
            const bool valid = j < (int)blk;
            const float lg = row_logit<MAXB / 2>(a.emb, D, valid ? sel[j] : 0, valid, xv);
            if ((lane & 15) == 0 && valid) a.ws.tlogit[off + j] = lg;
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            misc[12] = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1);
        }
        __syncthreads();
        if (!misc[12]) return;
        __threadfence();
        // ------------------------------------------------------------ the last CTA picks the candidates
        const int nb = (int)gridDim.x;
        unsigned *wst = hist_s;  // [nb] walk start and [nb] tuple offset of every CTA's segment
        unsigned my = 0;
        uint2 sg = make_uint2(0u, 0u);
        if (tid < nb) {
            sg = __ldcg(&a.ws.segs[tid]);
            my = sg.y;
        }
        unsigned S;
        const unsigned start = block_scan(my, tmp, &S);
        if (tid < nb) {
            wst[tid] = start;
            wst[nb + tid] = sg.x;
        }
        __syncthreads();
        uint32_t *rk = reinterpret_cast<uint32_t *>(ringp);
        int *ri = reinterpret_cast<int *>(ringp + 4 * kSkCap);
        float *rl = reinterpret_cast<float *>(ringp + 8 * kSkCap);
        constexpr int kGather = (kSkCap + kSkThreads - 1) / kSkThreads;
        unsigned srcs[kGather];
#pragma unroll
        for (int q = 0; q < kGather; q++) {
            const int p = tid + q * kSkThreads;
            srcs[q] = 0xffffffffu;
            if (p < (int)S) {
                int lo = 0, hi = nb - 1;  // the CTA whose segment holds walk position p
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (wst[mid] <= (unsigned)p) lo = mid;
                    else hi = mid - 1;
                }
                srcs[q] = wst[nb + lo] + ((unsigned)p - wst[lo]);
            }
        }
        uint32_t gk[kGather];
        int gi[kGather];
        float gl[kGather];
#pragma unroll
        for (int q = 0; q < kGather; q++)
            if (srcs[q] != 0xffffffffu) {
                gk[q] = __ldcg(a.ws.tkey + srcs[q]);
                gi[q] = __ldcg(a.ws.tidx + srcs[q]);
                gl[q] = __ldcg(a.ws.tlogit + srcs[q]);
            }
#pragma unroll
        for (int q = 0; q < kGather; q++)
            if (srcs[q] != 0xffffffffu) {
                const int p = tid + q * kSkThreads;
                rk[p] = gk[q];
                ri[p] = gi[q];
                rl[p] = gl[q];
            }
        __syncthreads();
        // the n_cand-th largest key: the rest of the radix select inside bin b1
        unsigned need = (unsigned)a.n_cand - above1;
        uint32_t prefix = b1;
#pragma unroll 1
        for (int pass = 0; pass < 2; pass++) {
            const int shift = pass == 0 ? 20 : 10;
            hist_pass(rk, (int)S, shift, prefix, shift - 10, 1024, hist_s);
            find_bin<false>(hist_s, 1024, need, tmp, misc + 0, (unsigned *)misc + 1);
            prefix = (prefix << 10) | (uint32_t)misc[0];
            need -= (unsigned)misc[1];
        }
        const uint32_t T = prefix;
        const int pp = ((int)S + kSkThreads - 1) / kSkThreads;
        const int p0 = min((int)S, pp * tid), p1 = min((int)S, p0 + pp);
        unsigned n_eq = 0;
        for (int p = p0; p < p1; p++) n_eq += rk[p] == T;
        unsigned tot;
        unsigned er = block_scan(n_eq, tmp, &tot);
        unsigned n_s = 0;
        {
            unsigned e2 = er;
            for (int p = p0; p < p1; p++) {
                n_s += rk[p] > T || (rk[p] == T && e2 < need);
                e2 += rk[p] == T;
            }
        }
        unsigned opos = block_scan(n_s, tmp, &tot);
        float bv = -__int_as_float(0x7f800000);
        int bi = 0x7fffffff;
        for (int p = p0; p < p1; p++) {
            const bool take = rk[p] > T || (rk[p] == T && er < need);
            er += rk[p] == T;
            if (take) {
                a.cand[opos] = ri[p];
                a.cand_logits[opos] = rl[p];
                opos++;
                if (better(rl[p], ri[p], bv, bi)) {
                    bv = rl[p];
                    bi = ri[p];
                }
            }
        }
        block_best(bv, bi, wbv, wbi);
        if (tid == 0) {
            *a.next = bi;
            *a.ws.ticket = 0u;
            *a.ws.tcount = 0u;
        }
        for (int j = tid; j < kSkHistWords; j += kSkThreads) a.ws.hist[j] = 0u;
        return;
    }

    // ---------------------------------------------------------------- slow path: finish the select together
    unsigned need = (unsigned)a.n_cand - above1;
    uint32_t prefix = b1;
#pragma unroll 1
    for (int pass = 0; pass < 2; pass++) {
        const int shift = pass == 0 ? 20 : 10;
        unsigned *gh = a.ws.hist + (pass == 0 ? kSkBins1 : kSkBins1 + kSkBins2);
        hist_pass(wkey, nw, shift, prefix, shift - 10, 1024, hist_s);
        for (int i = tid; i < 1024; i += kSkThreads)
            if (hist_s[i]) atomicAdd(&gh[i], hist_s[i]);
        if (!grid_barrier(a.ws.bar, a.ws.status, misc + 8)) return;
        find_bin<true>(gh, 1024, need, tmp, misc + 0, (unsigned *)misc + 1);
        prefix = (prefix << 10) | (uint32_t)misc[0];
        need -= (unsigned)misc[1];
    }
    const uint32_t TW = prefix;      // the n_cand-th largest key
    const unsigned eq_words = need;  // words with key == TW that are kept (lowest indices first)
    unsigned n_gt = 0, n_eq = 0;
    for (int i = c0; i < c1; i++) {
        n_gt += wkey[i] > TW;
        n_eq += wkey[i] == TW;
    }
    unsigned blk_gt, blk_eq;
    block_scan(n_gt, tmp, &blk_gt);
    const unsigned eq_pre = block_scan(n_eq, tmp, &blk_eq);
    if (tid == 0) a.ws.counts[blockIdx.x] = make_uint2(blk_gt, blk_eq);
    if (!grid_barrier(a.ws.bar, a.ws.status, misc + 8)) return;
    unsigned gt_b = 0, eq_b = 0;
    for (int b = tid; b < (int)blockIdx.x; b += kSkThreads) {
        const uint2 c = __ldcg(&a.ws.counts[b]);
        gt_b += c.x;
        eq_b += c.y;
    }
    unsigned gt_before, eq_before;
    block_scan(gt_b, tmp, &gt_before);
    block_scan(eq_b, tmp, &eq_before);
    unsigned n_sel = 0;
    {
        unsigned er = eq_before + eq_pre;
        for (int i = c0; i < c1; i++) {
            const uint32_t key = wkey[i];
            n_sel += key > TW || (key == TW && er < eq_words);
            er += key == TW;
        }
    }
    unsigned blk_sel;
    const unsigned sel_pre = block_scan(n_sel, tmp, &blk_sel);
    const unsigned base = gt_before + min(eq_before, eq_words);
    {
        unsigned er = eq_before + eq_pre, j = sel_pre;
        for (int i = c0; i < c1; i++) {
            const uint32_t key = wkey[i];
            if (key > TW || (key == TW && er < eq_words)) {
                sel[j] = w0 + i;
                a.cand[base + j] = w0 + i;
                j++;
            }
            er += key == TW;
        }
    }
    __syncthreads();
    float best_v = -__int_as_float(0x7f800000);
    int best_i = 0x7fffffff;
    for (int jw = 2 * warp; jw < (int)blk_sel; jw += 2 * kSkWarps) {  // warp-uniform trip count
        const int j = jw + (lane >> 4);
        const bool valid = j < (int)blk_sel;
        const int word = valid ? sel[j] : 0;
        const float lg = row_logit<MAXB / 2>(a.emb, D, word, valid, xv);
        if ((lane & 15) == 0 && valid) {
            a.cand_logits[base + j] = lg;
            if (better(lg, word, best_v, best_i)) {
                best_v = lg;
                best_i = word;
            }
        }
    }
    block_best(best_v, best_i, wbv, wbi);
    if (tid == 0) {
        a.ws.part[blockIdx.x] = make_float2(best_v, __int_as_float(best_i));
        __threadfence();
        misc[12] = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!misc[12]) return;
    // the last CTA: the grid's argmax, then leave the workspace zeroed
    __threadfence();
    float v = -__int_as_float(0x7f800000);
    int i = 0x7fffffff;
    for (int b = tid; b < (int)gridDim.x; b += kSkThreads) {
        const float2 p = __ldcg(&a.ws.part[b]);
        if (better(p.x, __float_as_int(p.y), v, i)) {
            v = p.x;
            i = __float_as_int(p.y);
        }
    }
    block_best(v, i, wbv, wbi);
    if (tid == 0) {
        *a.next = i;
        *a.ws.ticket = 0u;
        *a.ws.tcount = 0u;
    }
    for (int j = tid; j < kSkHistWords; j += kSkThreads) a.ws.hist[j] = 0u;
}

// ---------------------------------------------------------------- preparation
// perm[r] = the dim of rank r by size: largest |s_d| first (compared as bits),
// ties to the lower index; the identity without sizes.
__global__ void sketch_perm_kernel(const float *__restrict__ scale, int D, int32_t *__restrict__ perm) {
    const int d = blockIdx.x * blockDim.x + threadIdx.x;
    if (d >= D) return;
    if (!scale) {
        perm[d] = d;
        return;
    }
    const uint32_t me = __float_as_uint(scale[d]) & 0x7fffffffu;
    int r = 0;
    for (int e = 0; e < D; e++) {
        const uint32_t o = __float_as_uint(scale[e]) & 0x7fffffffu;
        r += (o > me || (o == me && e < d)) ? 1 : 0;
    }
    perm[r] = d;
}

// emb [V][D] -> emb_t [D][Vt], zeros for words V..Vt-1.
__global__ void sketch_transpose_kernel(const uint16_t *__restrict__ emb, int V, int D, int Vt,
                                        uint16_t *__restrict__ emb_t) {
    __shared__ uint16_t tile[32][33];
    const int v0 = 32 * blockIdx.x, d0 = 32 * blockIdx.y;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int v = v0 + r, d = d0 + threadIdx.x;
        tile[r][threadIdx.x] = (v < V && d < D) ? emb[(int64_t)v * D + d] : (uint16_t)0;
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int d = d0 + r, v = v0 + threadIdx.x;
        if (d < D && v < Vt) emb_t[(int64_t)d * Vt + v] = tile[threadIdx.x][r];
    }
}

// signs[b][v] bit p = sign bit of E[v][perm[64b + p]] (zero past D or V).
__global__ void sketch_signs_kernel(const uint16_t *__restrict__ emb, const int32_t *__restrict__ perm, int V,
                                    int D, int Vt, int nblk, uint64_t *__restrict__ signs) {
    const int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= (int64_t)nblk * Vt) return;
    const int b = (int)(item / Vt), v = (int)(item % Vt);
    uint64_t w = 0;
    if (v < V) {
        const uint16_t *row = emb + (int64_t)v * D;
        for (int p = 0; p < kSkBlockDims; p++) {
            const int i = kSkBlockDims * b + p;
            if (i < D) w |= (uint64_t)(row[perm[i]] >> 15) << p;
        }
    }
    signs[item] = w;
}

constexpr int kCeBlocks = 512;
constexpr int kCeThreads = 256;  // a power of two: the in-CTA tree halves it
__device__ double g_ce_part[kCeBlocks];

// mean |E| in fp64: CTA b sums a fixed slice, a fixed tree within the CTA.
__global__ void sketch_ce_part_kernel(const uint16_t *__restrict__ emb, int64_t n) {
    __shared__ double red[kCeThreads];
    const int64_t lo = n * blockIdx.x / gridDim.x, hi = n * (blockIdx.x + 1) / gridDim.x;
    double s = 0.0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x)
        s += (double)fabsf(__uint_as_float((uint32_t)emb[i] << 16));
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) g_ce_part[blockIdx.x] = red[0];
}

__global__ void sketch_ce_final_kernel(int64_t n, float *c_e) {
    if (threadIdx.x != 0) return;
    double s = 0.0;
    for (int b = 0; b < kCeBlocks; b++) s += g_ce_part[b];
    *c_e = (float)(s / (double)n);
}

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" {

int64_t qlin_sketch_emb_t_pitch(int vocab) { return vocab >= 1 ? emb_t_pitch(vocab) : -1; }

size_t qlin_sketch_signs_bytes(int vocab, int dim) {
    if (vocab < 1 || dim < 1) return 0;
    return (size_t)((dim + kSkBlockDims - 1) / kSkBlockDims) * (size_t)emb_t_pitch(vocab) * 8u;
}

qlin_status qlin_sketch_prepare(const uint16_t *emb, int vocab, int dim, const float *dim_scale, uint16_t *emb_t,
                                uint64_t *signs, int32_t *perm, float *c_e, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(emb && emb_t && signs && perm && c_e, QLIN_ERR_INVALID_ARG, "qlin_sketch_prepare: null pointer");
    QLIN_REQUIRE(vocab >= 1 && dim >= 8 && dim <= kSkMaxDim && dim % 8 == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_sketch_prepare: vocab %d, dim %d (need vocab >= 1, 8 <= dim <= %d, dim %% 8 == 0)", vocab, dim,
                 kSkMaxDim);
    QLIN_REQUIRE(aligned16(emb) && aligned16(emb_t) && aligned16(signs) && aligned4(perm) && aligned4(c_e) &&
                     (!dim_scale || aligned4(dim_scale)),
                 QLIN_ERR_INVALID_ARG, "qlin_sketch_prepare: misaligned pointer");
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t Vt = emb_t_pitch(vocab);
    const int nblk = (dim + kSkBlockDims - 1) / kSkBlockDims;
    sketch_perm_kernel<<<(dim + 255) / 256, 256, 0, st>>>(dim_scale, dim, perm);
    QLIN_LAUNCHED("sketch_perm_kernel");
    sketch_transpose_kernel<<<dim3((unsigned)((Vt + 31) / 32), (unsigned)((dim + 31) / 32)), dim3(32, 8), 0, st>>>(
        emb, vocab, dim, (int)Vt, emb_t);
    QLIN_LAUNCHED("sketch_transpose_kernel");
    const int64_t items = (int64_t)nblk * Vt;
    sketch_signs_kernel<<<(unsigned)((items + 255) / 256), 256, 0, st>>>(emb, perm, vocab, dim, (int)Vt, nblk, signs);
    QLIN_LAUNCHED("sketch_signs_kernel");
    const int64_t n = (int64_t)vocab * dim;
    sketch_ce_part_kernel<<<kCeBlocks, kCeThreads, 0, st>>>(emb, n);
    QLIN_LAUNCHED("sketch_ce_part_kernel");
    sketch_ce_final_kernel<<<1, 32, 0, st>>>(n, c_e);
    QLIN_LAUNCHED("sketch_ce_final_kernel");
    return QLIN_OK;
}

size_t qlin_sketch_workspace_size(int vocab) {
    (void)vocab;
    size_t b = 0;
    carve(nullptr, &b);
    return b;
}

qlin_status qlin_sketch_head(const uint16_t *emb, const uint16_t *emb_t, const uint64_t *signs, const int32_t *perm,
                             const float *c_e, int vocab, int dim, const float *x, int k, int n_cand, float *approx,
                             int32_t *cand, float *cand_logits, int32_t *next, void *workspace,
                             size_t workspace_bytes, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(emb && emb_t && signs && perm && c_e && x && cand && cand_logits && next && workspace,
                 QLIN_ERR_INVALID_ARG, "qlin_sketch_head: null pointer");
    QLIN_REQUIRE(vocab >= 1 && dim >= 8 && dim <= kSkMaxDim && dim % 8 == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_sketch_head: vocab %d, dim %d (need vocab >= 1, 8 <= dim <= %d, dim %% 8 == 0)", vocab, dim,
                 kSkMaxDim);
    QLIN_REQUIRE(k >= 0 && k <= kSkMaxK && k <= dim, QLIN_ERR_INVALID_ARG, "qlin_sketch_head: k = %d (0..%d)", k,
                 kSkMaxK);
    QLIN_REQUIRE(n_cand >= 1 && n_cand <= vocab, QLIN_ERR_INVALID_ARG, "qlin_sketch_head: n_cand = %d (1..vocab)",
                 n_cand);
    QLIN_REQUIRE(aligned16(emb) && aligned16(emb_t) && aligned16(signs) && aligned4(perm) && aligned4(c_e) &&
                     aligned4(x) && aligned4(cand) && aligned4(cand_logits) && aligned4(next) &&
                     (!approx || aligned4(approx)) && aligned16(workspace),
                 QLIN_ERR_INVALID_ARG, "qlin_sketch_head: misaligned pointer");
    size_t need = 0;
    SketchWs ws = carve(static_cast<char *>(workspace), &need);
    QLIN_REQUIRE(workspace_bytes >= need, QLIN_ERR_INVALID_ARG, "qlin_sketch_head: workspace %zu < %zu bytes",
                 workspace_bytes, need);
    const int tiles = (vocab + kSkTile - 1) / kSkTile;
    const int nblk = (dim + kSkBlockDims - 1) / kSkBlockDims;
    const void *kern = nblk <= 8    ? (const void *)sketch_head_kernel<8>
                       : nblk <= 16 ? (const void *)sketch_head_kernel<16>
                       : nblk <= 18 ? (const void *)sketch_head_kernel<18>
                       : nblk <= 24 ? (const void *)sketch_head_kernel<24>
                                    : (const void *)sketch_head_kernel<32>;
    // one CTA per SM; the stages take what the per-CTA tables leave
    const int nb = std::min(sm_count(), tiles);
    const int range_tiles = (tiles + nb - 1) / nb;
    const int per_word = 8 * nblk;
    // the stages get what the opt-in limit leaves after the fixed tables (at most kSkRingBudget)
    const int fixed = sk_layout(0, kSkTile * range_tiles).total - sk_layout(0, 0).ring - 12 * kSkCap;
    const int budget = std::min(kSkRingBudget, max_smem_optin() - fixed - 1024);
    int chunk = budget / (kSkStages * per_word) / kSkSub * kSkSub;
    chunk = std::max(kSkSub, std::min(chunk, (range_tiles * kSkTile + kSkSub - 1) / kSkSub * kSkSub));
    const int ring_bytes = kSkStages * chunk * per_word;
    const size_t smem = (size_t)sk_layout(ring_bytes, kSkTile * range_tiles).total;
    QLIN_REQUIRE(smem <= (size_t)max_smem_optin(), QLIN_ERR_UNSUPPORTED,
                 "qlin_sketch_head: vocab %d needs %zu bytes of shared memory per CTA", vocab, smem);
    blocks_per_sm(kern, smem);  // raises the kernel's dynamic shared-memory limit once
    int fit = 0;
    QLIN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kern, kSkThreads, smem));
    QLIN_REQUIRE(fit >= 1, QLIN_ERR_UNSUPPORTED, "qlin_sketch_head: no CTA fits on an SM");
    SketchArgs args{};
    args.emb = emb;
    args.emb_t = emb_t;
    args.signs = signs;
    args.perm = perm;
    args.c_e = c_e;
    args.x = x;
    args.V = vocab;
    args.D = dim;
    args.Vt = (int)emb_t_pitch(vocab);
    args.nblk = nblk;
    args.k = k;
    args.n_cand = n_cand;
    args.tiles = tiles;
    args.range_tiles = range_tiles;
    args.chunk = chunk;
    args.ring_bytes = ring_bytes;
    args.approx = approx;
    args.cand = cand;
    args.cand_logits = cand_logits;
    args.next = next;
    args.ws = ws;
    void *params[] = {&args};
    QLIN_CUDA(cudaLaunchCooperativeKernel(kern, dim3(nb), dim3(kSkThreads), params, smem, (cudaStream_t)stream));
    return QLIN_OK;
}

qlin_status qlin_sketch_head_status(void *workspace, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(workspace, QLIN_ERR_INVALID_ARG, "qlin_sketch_head_status: null workspace");
    int32_t st[4] = {0, 0, 0, 0};
    QLIN_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    QLIN_CUDA(cudaMemcpy(st, workspace, sizeof st, cudaMemcpyDeviceToHost));
    QLIN_CUDA(cudaMemset(workspace, 0, sizeof st));
    QLIN_REQUIRE(!(st[0] & kStatusTimeout), QLIN_ERR_TIMEOUT, "qlin_sketch_head: a grid barrier wait gave up");
    return QLIN_OK;
}

}  // extern "C"
