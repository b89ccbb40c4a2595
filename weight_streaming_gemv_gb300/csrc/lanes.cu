// A decode step over lanes ([citric] "Many users at once": every step is a set
// of lanes, a lane being one token of one sequence at one position; batches of
// users and chunks of a prompt go through the same step, and each weight byte
// is read once for all lanes).
//
// Lane i takes tokens[i] at positions[i] of sequence seqs[i]; sequence s owns
// the KV cache kv + s * L * 2 * max_pos * kv_dim (the single-token decode
// step's layout).  Layer by layer, every lane's k and v are written before any
// lane attends, so lanes of one sequence at consecutive positions form a
// prompt chunk.  Each lane's arithmetic is the single-token step's, operation
// for operation: RMSNorm, int8 absmax quantisation, T158 linear (exact integer
// dot, fp32 epilogue), RoPE and cache write, chunked attention, GeGLU,
// residual adds, final norm and the bf16 output layer with a greedy pick
// (here for all lanes in one pass over the table, on the tensor cores, with
// fp32-accurate logits rather than the single step's exact fp32 order).
//
// GB300 mapping: the step is a fixed sequence of kernels over all lanes at
// once (19 per layer), so it can be captured in a CUDA graph; from 8 lanes
// the T158 products run on the tensor cores (one pass over each matrix for all
// lanes).  Positions and sequence slots live in device memory: attention
// grids are sized for max_pos and chunks past a lane's position exit at once.
#include <algorithm>

#include "common.cuh"
#include "decode_ops.cuh"
#include "stream.cuh"

namespace qlin {

qlin_status t158_linear_dev_scale(const int8_t *xq, const float *xs, const uint8_t *w, int64_t pitch,
                                  const float *ws_ptr, float *y, int M, int N, int K, cudaStream_t st, void *work,
                                  bool convert);
size_t t158_tc_workspace_bytes(int M, int K);
qlin_status quant_i8_tiles(const float *x, int8_t *xq, float *xs, int M, int K, void *work, cudaStream_t st);
qlin_status t158_linear_tiles_multi(const float *xs, int count, const uint8_t *const *w, const int64_t *pitch,
                                    const float *const *ws_ptr, float *const *y, const int *N, int M, int K,
                                    void *work, cudaStream_t st);
qlin_status norm_quant_tiles(float *h, const float *y, const float *gain, float eps, int8_t *xq, float *xs, int M,
                             int K, void *work, cudaStream_t st);
qlin_status geglu_quant_tiles(const float *gate, const float *up, int8_t *xq, float *xs, int M, int K, void *work,
                              cudaStream_t st);

namespace {

constexpr int kLaneStatusBad = 1;      // a lane's token, position or sequence slot out of range
constexpr int kLaneStatusTimeout = 2;  // a bounded wait inside the attention kernel gave up
// Lanes from which every linear runs on the tensor cores (on activation tiles
// the quantisers write, the linears sharing an input in one launch); below it
// the CUDA-core kernels, one launch per linear.
constexpr int kLanesTensorMin = 3;

__device__ __forceinline__ bool lane_ok(int pos, int seq, int max_pos, int n_seqs) {
    return pos >= 0 && pos < max_pos && seq >= 0 && seq < n_seqs;
}

// per lane (blockIdx.x): h = emb[token]; a token out of range gives zeros
__global__ void lanes_embed_kernel(const uint16_t *__restrict__ emb, int vocab, int dim,
                                   const int32_t *__restrict__ tokens, float *__restrict__ h, int32_t *status) {
    const int i = blockIdx.x;
    const int tok = tokens[i];
    const bool ok = tok >= 0 && tok < vocab;
    for (int e = threadIdx.x; e < dim; e += blockDim.x)
        h[(int64_t)i * dim + e] = ok ? __uint_as_float((uint32_t)emb[(int64_t)tok * dim + e] << 16) : 0.0f;
    if (!ok && threadIdx.x == 0) atomicOr(status, kLaneStatusBad);
}

// per lane: rotate q and k at the lane's position, write k and v to its cache row
__global__ void lanes_rope_kv_kernel(float *q, const float *k, const float *v, float *kv, const int32_t *pos,
                                     const int32_t *seq, int n_seqs, int layer, int L, int max_pos,
                                     const float *__restrict__ cos_t, const float *__restrict__ sin_t, int nh,
                                     int nkv, int hd, int32_t *status) {
    extern __shared__ float kr[];  // [nkv*hd]
    const int i = blockIdx.x;
    const int p = pos[i], s = seq[i];
    if (!lane_ok(p, s, max_pos, n_seqs)) {
        if (threadIdx.x == 0) atomicOr(status, kLaneStatusBad);
        return;
    }
    const int half = hd / 2, kvd = nkv * hd;
    const float *c = cos_t + (int64_t)p * half;
    const float *sn = sin_t + (int64_t)p * half;
    rope_rotate(q + (int64_t)i * nh * hd, nh, hd, c, sn, whole_block());
    for (int e = threadIdx.x; e < kvd; e += blockDim.x) kr[e] = k[(int64_t)i * kvd + e];
    __syncthreads();
    rope_rotate(kr, nkv, hd, c, sn, whole_block());
    __syncthreads();
    float *kc = kv + (((int64_t)s * L + layer) * 2 + 0) * max_pos * kvd;
    float *vc = kc + (int64_t)max_pos * kvd;
    const int64_t off = (int64_t)p * kvd;
    for (int e = threadIdx.x; e < kvd; e += blockDim.x) {
        kc[off + e] = kr[e];
        vc[off + e] = v[(int64_t)i * kvd + e];
    }
}

// chunk partials of lane i (one workspace block of nh * ncmax * (2 + hd) floats per lane)
struct LaneAttnWs {
    float *m, *S, *U;
};

__device__ __forceinline__ LaneAttnWs lane_attn_ws(float *base, int lane, int ncmax, int nh, int hd) {
    float *b = base + (size_t)lane * nh * ncmax * (2 + hd);
    LaneAttnWs w;
    w.m = b;
    w.S = b + (size_t)nh * ncmax;
    w.U = b + (size_t)2 * nh * ncmax;
    return w;
}

// 16 bytes global -> shared without a register round trip; every copy of a
// thread stays in flight until its wait.
__device__ __forceinline__ void lanes_cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void lanes_cp_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

constexpr int kAttnGroupThreads = 128;  // threads per query head in the chunk kernel
constexpr int kAttnMaxGroups = 8;        // query heads served at once (1024 threads)

// grid (ncmax, nkv, lanes), block hpar * 128 threads: chunk c of KV head g of
// lane i for every query head of the group.  The chunk's k and v rows are
// read once into shared memory (16-byte asynchronous copies, all of them in
// flight together); hpar heads then run at once,
// each on its own 128 threads and hardware barrier.  Chunks past the lane's
// position exit.
__global__ void __launch_bounds__(kAttnGroupThreads * kAttnMaxGroups)
    lanes_attn_chunk_kernel(const float *__restrict__ q, const float *__restrict__ kv, const int32_t *pos,
                            const int32_t *seq, int n_seqs, int layer, int L, int max_pos, int nh, int nkv, int hd,
                            float *ws, int ncmax) {
    extern __shared__ __align__(16) float kvs[];  // [32][hd] k rows, then [32][hd] v rows
    __shared__ float qs[kAttnMaxGroups][256];
    __shared__ float sc[kAttnMaxGroups][32];
    const int c = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
    const int p = pos[i], s = seq[i];
    if (!lane_ok(p, s, max_pos, n_seqs) || c * 32 > p) return;
    const int t0 = c * 32;
    const int nt = min(32, p + 1 - t0);
    const int ld = nkv * hd;
    const float *kc = kv + (((int64_t)s * L + layer) * 2 + 0) * max_pos * ld + (int64_t)t0 * ld + kvh * hd;
    const float *vc = kc + (int64_t)max_pos * ld;
    float *Ks = kvs, *Vs = kvs + 32 * hd;
    const int hd4 = hd / 4;
    for (int e = threadIdx.x; e < nt * hd4; e += blockDim.x) {
        const int t = e / hd4, dd = e - t * hd4;
        lanes_cp16(Ks + 4 * e, kc + (int64_t)t * ld + 4 * dd);
        lanes_cp16(Vs + 4 * e, vc + (int64_t)t * ld + 4 * dd);
    }
    lanes_cp_wait_all();  // this thread's copies have landed; the barrier below publishes them
    LaneAttnWs w = lane_attn_ws(ws, i, ncmax, nh, hd);
    const int grp = nh / nkv, hpar = blockDim.x / kAttnGroupThreads;
    const int gi = threadIdx.x / kAttnGroupThreads;
    const Grp g{(int)threadIdx.x - gi * kAttnGroupThreads, kAttnGroupThreads, 1 + gi};
    for (int h0 = 0; h0 < grp; h0 += hpar) {
        __syncthreads();  // the k/v rows are in; the previous round is done with qs
        const int h = kvh * grp + h0 + gi;
        const bool active = h0 + gi < grp;
        if (active)
            for (int e = g.tid; e < hd; e += g.n) qs[gi][e] = q[((int64_t)i * nh + h) * hd + e];
        __syncthreads();
        if (active)
            attention_chunk(qs[gi], Ks, Vs, hd, nt, hd, w.m + h * ncmax + c, w.S + h * ncmax + c,
                            w.U + ((int64_t)h * ncmax + c) * hd, sc[gi], g);
    }
}

// Persistent attention over lanes: the chunk partials of lanes_attn_chunk_kernel
// (the same arithmetic, term for term, so the same bits), with each CTA
// streaming a range of units (lane, KV head, chunk) through kAttnBufs
// shared-memory buffers that asynchronous copies fill ahead of use.  Units are
// numbered chunk fastest, so a CTA's consecutive units share a lane and KV head
// and its q rows stay in registers; units past a lane's position are skipped.
// Per unit: each warp scores positions warp and warp + 16 against every query
// head of the group (one k row read serves them all), one warp per head takes
// the softmax, and all threads form the weighted value sums.
constexpr int kAttnThreads = 512;
constexpr int kAttnBufs = 3;

template <int HD, int GRP>
__global__ void __launch_bounds__(kAttnThreads, 1)
    lanes_attn_kernel(const float *__restrict__ q, const float *__restrict__ kv, const int32_t *pos,
                      const int32_t *seq, int n_seqs, int layer, int L, int max_pos, int nh, int nkv, int M,
                      float *ws, int ncmax, int32_t *status) {
    constexpr int S = HD / 32;   // dims per lane in the scores
    constexpr int CH = 32 * HD;  // floats of a chunk's k (or v) rows
    extern __shared__ __align__(16) float abuf[];  // [kAttnBufs][2][32][HD]
    __shared__ __align__(16) float sc[GRP][32];
    __shared__ uint64_t full[kAttnBufs];  // buffer b's rows have landed (one arrival + the bytes)
    __shared__ int4 unit[kAttnBufs];      // buffer b's unit {lane, KV head, chunk, position}, lane -1: no more
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = nh / nkv;  // query heads per KV head, <= GRP
    if (tid == 0) {
        for (int b = 0; b < kAttnBufs; b++) mbar_init(&full[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = l2_evict_first();  // every KV row is read once per step
    const int ld = nkv * HD;
    const int64_t units = (int64_t)M * nkv * ncmax;
    const int64_t u_lo = units * blockIdx.x / gridDim.x;
    int64_t left = units * (blockIdx.x + 1) / gridDim.x - u_lo;  // units of this CTA not yet walked
    // unit counters, chunk fastest: lane ai, KV head ag, chunk ac
    int ac = (int)(u_lo % ncmax), ag = (int)((u_lo / ncmax) % nkv), ai = (int)(u_lo / ((int64_t)ncmax * nkv));
    const float div = __fsqrt_rn((float)HD);

    // the position and sequence slot of lane ci, loaded once per lane (units
    // of one lane are consecutive)
    int ci = -1, cpos = 0, cseq = 0;
    auto lane_info = [&](int li) {
        if (li != ci) {
            ci = li;
            cpos = pos[li];
            cseq = seq[li];
        }
    };
    // the next unit of this CTA with work as {lane, KV head, chunk, position},
    // lane -1 when none is left (every thread computes the same)
    auto advance = [&]() -> int4 {
        while (left > 0) {
            const int li = ai, g = ag, c = ac;
            left--;
            if (++ac == ncmax) {
                ac = 0;
                if (++ag == nkv) ag = 0, ai++;
            }
            lane_info(li);
            if (lane_ok(cpos, cseq, max_pos, n_seqs) && c * 32 <= cpos) return make_int4(li, g, c, cpos);
        }
        return make_int4(-1, 0, 0, 0);
    };
    auto issue = [&](int4 un, int b) {  // un's lane is the one advance() just found
        const int g = un.y, c = un.z, p = un.w, s = cseq;
        const int t0 = c * 32, nt = min(32, p + 1 - t0);
        const float *kc = kv + (((int64_t)s * L + layer) * 2 + 0) * max_pos * ld + (int64_t)t0 * ld + g * HD;
        const float *vc = kc + (int64_t)max_pos * ld;
        float *Kb = abuf + (size_t)b * 2 * CH, *Vb = Kb + CH;
        constexpr uint32_t rowb = HD * sizeof(float);
        // (the issuing warp only)
        if (ld == HD) {  // one KV head: the chunk's k rows are contiguous, and so are its v rows
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[b], 2u * (uint32_t)nt * rowb);
                bulk_g2s(Kb, kc, (uint32_t)nt * rowb, &full[b], pol);
                bulk_g2s(Vb, vc, (uint32_t)nt * rowb, &full[b], pol);
            }
        } else {  // one bulk copy per k row and per v row, lane t: row t
            if (lane == 0) mbar_arrive_expect_tx(&full[b], 2u * (uint32_t)nt * rowb);
            __syncwarp();
            if (lane < nt) {
                bulk_g2s(Kb + lane * HD, kc + (int64_t)lane * ld, rowb, &full[b], pol);
                bulk_g2s(Vb + lane * HD, vc + (int64_t)lane * ld, rowb, &full[b], pol);
            }
        }
    };
    // The last warp walks the units and issues the copies: it publishes buffer
    // b's unit in unit[b] before the buffer's barrier completes (with the bytes,
    // or with a plain arrival for the end marker), so the other warps learn
    // the unit there; it finds the next unit while the others take the softmax.
    constexpr int kIssWarp = kAttnThreads / 32 - 1;
    static_assert(kIssWarp >= GRP, "the issuing warp is not a softmax warp");
    auto publish = [&](int4 un, int b) {
        if (lane == 0) unit[b] = un;
        __syncwarp();
        if (un.x >= 0)
            issue(un, b);
        else if (lane == 0)
            mbar_arrive(&full[b]);
    };

    if (warp == kIssWarp)
        for (int b = 0; b < kAttnBufs; b++) publish(advance(), b);
    int4 nx = make_int4(-1, 0, 0, 0);  // the issuing warp: the unit found during the softmax
    float qr[GRP][S];
    int64_t cur = -1;  // lane * nkv + KV head whose q rows are in qr
    for (int k = 0;; k++) {
        const int b = k % kAttnBufs;
        // buffer b's (k / kAttnBufs)-th fill: unit[b] and, for a unit, its k and v rows
        const bool landed = mbar_wait(&full[b], (uint32_t)(k / kAttnBufs) & 1u);
        if (__syncthreads_or(!landed)) {
            if (tid == 0) atomicOr(status, kLaneStatusTimeout);
            return;
        }
        const int4 un = unit[b];
        if (un.x < 0) break;
        const int i = un.x, g = un.y, c = un.z, p = un.w;
        const int t0 = c * 32, nt = min(32, p + 1 - t0);
        const float *Kb = abuf + (size_t)b * 2 * CH, *Vb = Kb + CH;
        LaneAttnWs w = lane_attn_ws(ws, i, ncmax, nh, HD);
        if ((int64_t)i * nkv + g != cur) {
            cur = (int64_t)i * nkv + g;
#pragma unroll
            for (int h = 0; h < GRP; h++)
#pragma unroll
                for (int e = 0; e < S; e++)
                    qr[h][e] = h < grp ? q[((int64_t)i * nh + g * grp + h) * HD + lane * S + e] : 0.0f;
        }
        // scores: lane owns dims [lane S, lane S + S), a tree over them, then across lanes
        for (int t = warp; t < 32; t += kAttnThreads / 32) {
            float kr[S];
            if (t < nt) {
                const float *kt = Kb + t * HD;
                if constexpr (S == 8) {
                    // two 16-byte loads; lanes 4..7 of each phase read their upper half first
                    const float4 *k4 = reinterpret_cast<const float4 *>(kt + lane * S);
                    const int sw = (lane >> 2) & 1;
                    const float4 f = k4[sw], s2 = k4[sw ^ 1];
                    const float4 lo = sw ? s2 : f, hi = sw ? f : s2;
                    kr[0] = lo.x, kr[1] = lo.y, kr[2] = lo.z, kr[3] = lo.w;
                    kr[4] = hi.x, kr[5] = hi.y, kr[6] = hi.z, kr[7] = hi.w;
                } else if constexpr (S == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(kt + lane * 4);
                    kr[0] = v.x, kr[1] = v.y, kr[2] = v.z, kr[3] = v.w;
                } else {
#pragma unroll
                    for (int e = 0; e < S; e++) kr[e] = kt[lane * S + e];
                }
            }
            // every head's lane tree, then the warp sums level by level across
            // heads (the sums of warp_psum, interleaved)
            float part[GRP];
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                part[h] = 0.0f;
                if (t < nt) {
                    float pp[S];
#pragma unroll
                    for (int e = 0; e < S; e++) pp[e] = __fmul_rn(qr[h][e], kr[e]);
#pragma unroll
                    for (int st = 1; st < S; st <<= 1)
#pragma unroll
                        for (int e = 0; e < S; e += 2 * st) pp[e] = __fadd_rn(pp[e], pp[e + st]);
                    part[h] = pp[0];
                }
            }
            // Reduce-scatter over the heads, then a butterfly: at level off = 1,
            // 2, .. < GRP a lane keeps the half of its heads picked by lane bit
            // off, sends the other half and adds the partner's copy of the half
            // it keeps (the partner sent exactly those); once one head is left
            // (hk, from the lane's low bits) the remaining levels are those of
            // warp_psum.  Every head's sum is the same adjacent-lanes-first tree.
            int hk = 0;
#pragma unroll
            for (int off = 1, n = GRP; off < GRP; off <<= 1, n >>= 1) {
                const bool up = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < n / 2; i++) {
                    const float keep = up ? part[n / 2 + i] : part[i];
                    const float send = up ? part[i] : part[n / 2 + i];
                    part[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, off));
                }
                if (up) hk += n / 2;
            }
            float sv = part[0];
#pragma unroll
            for (int off = GRP; off < 32; off <<= 1) sv = __fadd_rn(sv, __shfl_xor_sync(0xffffffffu, sv, off));
            if (lane < GRP) sc[hk][t] = (t < nt) ? __fdiv_rn(sv, div) : 0.0f;  // lanes 0 .. GRP-1 hold every head once
        }
        __syncthreads();
        if (warp == kIssWarp) nx = advance();  // meanwhile: the unit for buffer b after this one
        if (warp < grp) {  // softmax of head `warp` over the chunk
            const int h = warp, t = lane;
            const float m = warp_max(t < nt ? sc[h][t] : -__int_as_float(0x7f800000));
            const float e = (t < nt) ? exp32(__fsub_rn(sc[h][t], m)) : 0.0f;
            __syncwarp();
            sc[h][t] = e;
            const float Ssum = warp_psum(e);
            if (t == 0) {
                const int hg = g * grp + h;
                w.m[hg * ncmax + c] = m;
                w.S[hg * ncmax + c] = Ssum;
            }
        }
        __syncthreads();
        {
            // thread: dim d, heads hb, hb + HG, ... (HG = threads / HD), two at a
            // time sharing each value load
            constexpr int HG = kAttnThreads / HD;
            const int d = tid % HD, hb = tid / HD;
            for (int h0 = hb; h0 < grp; h0 += 2 * HG) {
                const int h1 = h0 + HG;
                const bool two = h1 < grp;
                // running pairwise stacks over the 32 positions: pushing t merges
                // the completed subtrees below it, so after 32 pushes level 5 holds
                // the balanced tree (left + right at every node)
                float sa[6], sb[6];
                float4 wa = make_float4(0.f, 0.f, 0.f, 0.f), wb = wa;
#pragma unroll
                for (int t = 0; t < 32; t++) {
                    if ((t & 3) == 0) {  // the weights of positions t .. t + 3, one load per head
                        wa = *reinterpret_cast<const float4 *>(&sc[h0][t]);
                        if (two) wb = *reinterpret_cast<const float4 *>(&sc[h1][t]);
                    }
                    const float ea = (t & 3) == 0 ? wa.x : (t & 3) == 1 ? wa.y : (t & 3) == 2 ? wa.z : wa.w;
                    const float eb = (t & 3) == 0 ? wb.x : (t & 3) == 1 ? wb.y : (t & 3) == 2 ? wb.z : wb.w;
                    const float v = (t < nt) ? Vb[t * HD + d] : 0.0f;
                    float xa = (t < nt) ? __fmul_rn(ea, v) : 0.0f;
                    float xb = (t < nt && two) ? __fmul_rn(eb, v) : 0.0f;
                    int k = 0;
#pragma unroll
                    for (int jj = t; jj & 1; jj >>= 1, k++) {
                        xa = __fadd_rn(sa[k], xa);
                        xb = __fadd_rn(sb[k], xb);
                    }
                    sa[k] = xa;
                    sb[k] = xb;
                }
                w.U[((int64_t)(g * grp + h0) * ncmax + c) * HD + d] = sa[5];
                if (two) w.U[((int64_t)(g * grp + h1) * ncmax + c) * HD + d] = sb[5];
            }
        }
        __syncthreads();  // buffer b, unit[b] and sc are free again
        if (warp == kIssWarp) publish(nx, b);
    }
}

// grid (nh, lanes): merge the lane's chunks of head h
__global__ void __launch_bounds__(256) lanes_attn_merge_kernel(const float *ws, int ncmax, const int32_t *pos,
                                                               const int32_t *seq, int n_seqs, int max_pos, int nh,
                                                               int hd, float *out) {
    extern __shared__ float wbuf[];
    __shared__ float red[32];
    const int h = blockIdx.x, i = blockIdx.y;
    const int p = pos[i];
    if (!lane_ok(p, seq[i], max_pos, n_seqs)) return;
    LaneAttnWs w = lane_attn_ws(const_cast<float *>(ws), i, ncmax, nh, hd);
    attention_merge(w.m + h * ncmax, w.S + h * ncmax, w.U + (int64_t)h * ncmax * hd, p / 32 + 1, hd,
                    out + ((int64_t)i * nh + h) * hd, wbuf, red, whole_block());
}

// block_psum (decode_ops.cuh) for a whole block, the same tree: each of the T
// threads (T the largest power of two in the block) reduces its segment of
// P / T adjacent terms, then lanes, then warps adjacent first; the warps'
// partials by one warp's butterfly (zero padding adds exactly nothing).
__device__ __forceinline__ float merge_psum(float *buf, int P, float *red) {
    const int tid = threadIdx.x;
    int T = 32;
    while (2 * T <= (int)blockDim.x) T *= 2;
    __syncthreads();
    float v = 0.0f;
    if (tid < T) {
        if (P >= T) {
            const int S = P / T;
            float *a = buf + tid * S;
            for (int st = 1; st < S; st <<= 1)
                for (int i = 0; i < S; i += 2 * st) a[i] = __fadd_rn(a[i], a[i + st]);
            v = a[0];
        } else {
            v = (tid < P) ? buf[tid] : 0.0f;
        }
    }
    v = warp_psum(v);
    if ((tid & 31) == 0 && tid < T) red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
        float w = tid < (T >> 5) ? red[tid] : 0.0f;
        w = warp_psum(w);
        if (tid == 0) red[0] = w;
    }
    __syncthreads();
    return red[0];
}

// grid (nh, lanes): lanes_attn_merge_kernel with the lane's partials of head h
// staged in shared memory first (4-byte asynchronous copies, all in flight
// together), then the same maximum, weights, pairwise sums and division.
// Shared memory: [ncmax hd] U, [ncmax] m, [ncmax] S, [next_pow2(ncmax)]
// weights, [hd] outputs.
__global__ void __launch_bounds__(256) lanes_attn_merge_smem_kernel(const float *ws, int ncmax, const int32_t *pos,
                                                                    const int32_t *seq, int n_seqs, int max_pos,
                                                                    int nh, int hd, float *out) {
    extern __shared__ __align__(16) float msm[];
    __shared__ float red[32];
    const int h = blockIdx.x, i = blockIdx.y;
    const int p = pos[i];
    if (!lane_ok(p, seq[i], max_pos, n_seqs)) return;
    const int nc = p / 32 + 1, P = next_pow2(nc);
    LaneAttnWs w = lane_attn_ws(const_cast<float *>(ws), i, ncmax, nh, hd);
    const float *pU = w.U + (int64_t)h * ncmax * hd, *pm = w.m + h * ncmax, *pS = w.S + h * ncmax;
    float *U = msm, *Mc = U + (size_t)ncmax * hd, *Sc = Mc + ncmax, *wb = Sc + ncmax, *o = wb + next_pow2(ncmax);
    // a lane's U rows start 16-byte aligned when nh ncmax is even (hd is a
    // multiple of 4 and the workspace base is aligned): 16-byte copies then
    if (((nh * ncmax) & 1) == 0) {
        for (int e = threadIdx.x; e < nc * hd / 4; e += blockDim.x) lanes_cp16(U + 4 * e, pU + 4 * e);
    } else {
        for (int e = threadIdx.x; e < nc * hd; e += blockDim.x)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(U + e)),
                         "l"(pU + e)
                         : "memory");
    }
    for (int c = threadIdx.x; c < nc; c += blockDim.x) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(Mc + c)),
                     "l"(pm + c)
                     : "memory");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(Sc + c)),
                     "l"(pS + c)
                     : "memory");
    }
    lanes_cp_wait_all();
    __syncthreads();
    // the largest chunk maximum (exact in any order): lane-strided, then across the warp
    float m = -__int_as_float(0x7f800000);
    for (int c = threadIdx.x & 31; c < nc; c += 32) m = fmaxf(m, Mc[c]);
    m = warp_max(m);
    for (int c = threadIdx.x; c < P; c += blockDim.x) wb[c] = (c < nc) ? exp32(__fsub_rn(Mc[c], m)) : 0.0f;
    __syncthreads();
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        PairwiseStream<16> ps;
        for (int c = 0; c < nc; c++) ps.push(__fmul_rn(U[(size_t)c * hd + d], wb[c]));
        o[d] = ps.result();
    }
    __syncthreads();
    for (int c = threadIdx.x; c < P; c += blockDim.x) wb[c] = (c < nc) ? __fmul_rn(Sc[c], wb[c]) : 0.0f;
    const float S = merge_psum(wb, P, red);
    for (int d = threadIdx.x; d < hd; d += blockDim.x) out[((int64_t)i * nh + h) * hd + d] = __fdiv_rn(o[d], S);
}

__global__ void lanes_add_kernel(float *h, const float *y, int64_t n) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
        h[e] = __fadd_rn(h[e], y[e]);
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

int attn_chunks(int max_pos) { return (max_pos + 31) / 32; }

struct LanesWs {
    int32_t *status;
    float *h, *xn, *xs, *q, *k, *v, *att, *y, *g, *u, *attn;
    int8_t *xq;
    void *lm, *tiles;  // tiles: fp16 activation tiles of the tensor-core linears
    size_t lm_bytes, bytes;
};

LanesWs carve_lanes(const t158_model *m, int max_lanes, char *base) {
    LanesWs w{};
    size_t off = 0;
    auto take = [&](size_t b) {
        char *p = base ? base + off : nullptr;
        off += align256(b);
        return p;
    };
    const size_t M = (size_t)max_lanes, d = m->dim, qd = (size_t)m->n_heads * m->head_dim;
    const size_t kvd = (size_t)m->n_kv_heads * m->head_dim, f = m->ffn;
    const size_t big = std::max(std::max(d, qd), f);
    w.status = (int32_t *)take(16);  // must stay first: decode_lanes_t158_status reads offset 0
    w.h = (float *)take(4 * M * d);
    w.xn = (float *)take(4 * M * d);
    w.xq = (int8_t *)take(M * big);
    w.xs = (float *)take(4 * M);
    w.q = (float *)take(4 * M * qd);
    w.k = (float *)take(4 * M * kvd);
    w.v = (float *)take(4 * M * kvd);
    w.att = (float *)take(4 * M * qd);
    w.y = (float *)take(4 * M * d);
    w.g = (float *)take(4 * M * f);
    w.u = (float *)take(4 * M * f);
    w.attn = (float *)take(4 * M * m->n_heads * (size_t)attn_chunks(m->max_pos) * (2 + m->head_dim));
    w.lm_bytes = qlin_lm_head_lanes_workspace_size(m->vocab, m->dim);
    w.lm = take(w.lm_bytes);
    w.tiles = take(max_lanes >= kLanesTensorMin ? t158_tc_workspace_bytes(max_lanes, (int)big) : 0);
    w.bytes = off;
    return w;
}

// The persistent attention kernel for head_dim 64..256 and up to 8 query
// heads per KV head (one CTA per SM over every lane's units); null otherwise.
template <int HD>
const void *attn_kernel_for(int grp) {
    switch (grp <= 1 ? 1 : grp <= 2 ? 2 : grp <= 4 ? 4 : grp <= 8 ? 8 : 0) {
        case 1: return (const void *)lanes_attn_kernel<HD, 1>;
        case 2: return (const void *)lanes_attn_kernel<HD, 2>;
        case 4: return (const void *)lanes_attn_kernel<HD, 4>;
        case 8: return (const void *)lanes_attn_kernel<HD, 8>;
        default: return nullptr;
    }
}
const void *attn_kernel(int hd, int grp) {
    switch (hd) {
        case 64: return attn_kernel_for<64>(grp);
        case 128: return attn_kernel_for<128>(grp);
        case 256: return attn_kernel_for<256>(grp);
        default: return nullptr;
    }
}

qlin_status check_lanes_model(const t158_model *m) {
    QLIN_REQUIRE(m, QLIN_ERR_INVALID_ARG, "decode_lanes_t158: null model");
    QLIN_REQUIRE(m->n_layers >= 1 && m->dim >= 8 && m->dim % 8 == 0 && m->n_heads >= 1 && m->n_kv_heads >= 1 &&
                     m->n_heads % m->n_kv_heads == 0 && m->ffn >= 1 && m->vocab >= 1 && m->max_pos >= 1,
                 QLIN_ERR_INVALID_ARG, "decode_lanes_t158: bad model dimensions");
    QLIN_REQUIRE(m->head_dim >= 16 && m->head_dim <= 256 && (m->head_dim & (m->head_dim - 1)) == 0,
                 QLIN_ERR_UNSUPPORTED, "decode_lanes_t158: head_dim %d not a power of two in 16..256", m->head_dim);
    for (int j = 0; j < T158_NMAT; j++)
        QLIN_REQUIRE(m->w[j] && aligned16(m->w[j]) && m->pitch[j] % 16 == 0, QLIN_ERR_INVALID_ARG,
                     "decode_lanes_t158: weight %d null, misaligned or pitch not a multiple of 16", j);
    QLIN_REQUIRE(m->scales && m->g_attn && m->g_ffn && m->g_final && m->emb && m->rope_cos && m->rope_sin,
                 QLIN_ERR_INVALID_ARG, "decode_lanes_t158: null model tensor");
    QLIN_REQUIRE(aligned16(m->emb), QLIN_ERR_INVALID_ARG, "decode_lanes_t158: emb not 16-byte aligned");
    return QLIN_OK;
}

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" {

qlin_status decode_lanes_t158_workspace_size(const t158_model *m, int max_lanes, size_t *bytes) {
    qlin::clear_error();
    qlin_status st = check_lanes_model(m);
    if (st) return st;
    QLIN_REQUIRE(bytes && max_lanes >= 1 && max_lanes <= 4096, QLIN_ERR_INVALID_ARG,
                 "decode_lanes_t158_workspace_size: max_lanes %d outside 1..4096", max_lanes);
    *bytes = carve_lanes(m, max_lanes, nullptr).bytes;
    return QLIN_OK;
}

qlin_status decode_lanes_t158(const t158_model *m, float *kv_caches, int n_seqs, int n_lanes, const int32_t *tokens,
                              const int32_t *positions, const int32_t *seqs, float *logits, int32_t *next,
                              void *workspace, size_t workspace_bytes, int max_lanes, qlin_stream_t stream) {
    qlin::clear_error();
    qlin_status st = check_lanes_model(m);
    if (st) return st;
    QLIN_REQUIRE(kv_caches && tokens && positions && seqs && next && workspace, QLIN_ERR_INVALID_ARG,
                 "decode_lanes_t158: null pointer");
    QLIN_REQUIRE(n_seqs >= 1 && n_lanes >= 1 && n_lanes <= max_lanes && max_lanes <= 4096, QLIN_ERR_INVALID_ARG,
                 "decode_lanes_t158: n_seqs %d, n_lanes %d, max_lanes %d", n_seqs, n_lanes, max_lanes);
    QLIN_REQUIRE(aligned16(workspace) && aligned16(kv_caches), QLIN_ERR_INVALID_ARG,
                 "decode_lanes_t158: workspace or kv_caches not 16-byte aligned");
    const LanesWs w = carve_lanes(m, max_lanes, (char *)workspace);
    QLIN_REQUIRE(workspace_bytes >= w.bytes, QLIN_ERR_INVALID_ARG, "decode_lanes_t158: workspace %zu < %zu bytes",
                 workspace_bytes, w.bytes);
    cudaStream_t s = (cudaStream_t)stream;
    const int M = n_lanes, L = m->n_layers, d = m->dim, nh = m->n_heads, nkv = m->n_kv_heads, hd = m->head_dim;
    const int qd = nh * hd, kvd = nkv * hd, f = m->ffn;
    const int ncmax = attn_chunks(m->max_pos);
    const uint8_t *W[T158_NMAT];
    for (int j = 0; j < T158_NMAT; j++) W[j] = m->w[j];
    const int rows[T158_NMAT] = {qd, kvd, kvd, d, f, f, d};
    const int cols[T158_NMAT] = {d, d, d, qd, d, d, f};
    // linear j of layer l on the quantised activations in w.xq / w.xs (one
    // lane: the CUDA-core kernels; from kLanesTensorMin lanes lin_group below
    // takes the tensor cores on the tiles the quantisers wrote)
    auto lin = [&](int l, int j, float *out) -> qlin_status {
        return t158_linear_dev_scale(w.xq, w.xs, W[j] + (int64_t)l * rows[j] * m->pitch[j], m->pitch[j],
                                     m->scales + (int64_t)l * T158_NMAT + j, out, M, rows[j], cols[j], s, nullptr,
                                     false);
    };
    // the quantisers write the tensor-core tiles when the linears take that path
    // (and then no int8 codes: nothing reads them), else the codes
    void *const tiles = M >= kLanesTensorMin ? w.tiles : nullptr;
    int8_t *const codes = tiles ? nullptr : w.xq;
    // linears j0 .. j0 + n - 1 of layer l (same input): one tensor-core launch on the tiles, else one each
    auto lin_group = [&](int l, int j0, int n, float *const *out) -> qlin_status {
        if (!tiles) {
            for (int k = 0; k < n; k++)
                if (qlin_status e = lin(l, j0 + k, out[k])) return e;
            return QLIN_OK;
        }
        const uint8_t *wj[3];
        int64_t pj[3];
        const float *sj[3];
        int nj[3];
        for (int k = 0; k < n; k++) {
            const int j = j0 + k;
            wj[k] = W[j] + (int64_t)l * rows[j] * m->pitch[j];
            pj[k] = m->pitch[j];
            sj[k] = m->scales + (int64_t)l * T158_NMAT + j;
            nj[k] = rows[j];
        }
        return t158_linear_tiles_multi(w.xs, n, wj, pj, sj, out, nj, M, cols[j0], tiles, s);
    };
    const int add_blocks = std::max(1, std::min(4 * sm_count(), (int)(((int64_t)M * d + 255) / 256)));
    const size_t attn_smem = (size_t)2 * 32 * hd * sizeof(float);
    const int attn_threads = kAttnGroupThreads * std::min(kAttnMaxGroups, nh / nkv);
    if (attn_smem > 48 * 1024) blocks_per_sm((const void *)lanes_attn_chunk_kernel, attn_smem);  // raises the limit once
    // the merge stages a head's partials in shared memory when they fit in 64 KB
    size_t merge_smem = ((size_t)ncmax * hd + 2 * ncmax + next_pow2(ncmax) + hd) * sizeof(float);
    if (merge_smem > 64 * 1024) merge_smem = 0;
    else if (merge_smem > 48 * 1024) blocks_per_sm((const void *)lanes_attn_merge_smem_kernel, merge_smem);
    // persistent attention: one CTA per SM (or per unit when there are fewer)
    const void *attn_k = attn_kernel(hd, nh / nkv);
    const size_t attn_k_smem = (size_t)kAttnBufs * 2 * 32 * hd * sizeof(float);
    const int64_t attn_units = (int64_t)M * nkv * ncmax;
    const int attn_grid = (int)std::min<int64_t>(sm_count(), attn_units);
    if (attn_k) {
        QLIN_REQUIRE((int)attn_k_smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED, "decode_lanes_t158: attention buffers");
        blocks_per_sm(attn_k, attn_k_smem);  // raises the dynamic shared-memory limit
    }

    lanes_embed_kernel<<<M, 256, 0, s>>>(m->emb, m->vocab, d, tokens, w.h, w.status);
    QLIN_LAUNCHED("lanes_embed_kernel");
    for (int l = 0; l < L; l++) {
        // (the previous layer's FFN output joins the residual stream here)
        if ((st = norm_quant_tiles(w.h, l > 0 ? w.y : nullptr, m->g_attn + (int64_t)l * d, m->eps, codes, w.xs, M, d,
                                   tiles, s)))
            return st;
        {
            float *const qkv[3] = {w.q, w.k, w.v};
            if ((st = lin_group(l, 0, 3, qkv))) return st;
        }
        lanes_rope_kv_kernel<<<M, 256, (size_t)kvd * sizeof(float), s>>>(
            w.q, w.k, w.v, kv_caches, positions, seqs, n_seqs, l, L, m->max_pos, m->rope_cos, m->rope_sin, nh, nkv,
            hd, w.status);
        QLIN_LAUNCHED("lanes_rope_kv_kernel");
        if (attn_k) {
            void *args[] = {(void *)&w.q, (void *)&kv_caches, (void *)&positions, (void *)&seqs, (void *)&n_seqs,
                            (void *)&l, (void *)&L, (void *)&m->max_pos, (void *)&m->n_heads, (void *)&m->n_kv_heads,
                            (void *)&M, (void *)&w.attn, (void *)&ncmax, (void *)&w.status};
            QLIN_CUDA(cudaLaunchKernel(attn_k, dim3(attn_grid), dim3(kAttnThreads), args, attn_k_smem, s));
            QLIN_LAUNCHED("lanes_attn_kernel");
        } else {
            lanes_attn_chunk_kernel<<<dim3(ncmax, nkv, M), attn_threads, attn_smem, s>>>(w.q, kv_caches, positions, seqs, n_seqs,
                                                                                 l, L, m->max_pos, nh, nkv, hd, w.attn,
                                                                                 ncmax);
            QLIN_LAUNCHED("lanes_attn_chunk_kernel");
        }
        if (merge_smem) {
            lanes_attn_merge_smem_kernel<<<dim3(nh, M), 256, merge_smem, s>>>(w.attn, ncmax, positions, seqs, n_seqs,
                                                                            m->max_pos, nh, hd, w.att);
            QLIN_LAUNCHED("lanes_attn_merge_smem_kernel");
        } else {
            lanes_attn_merge_kernel<<<dim3(nh, M), 256, (size_t)next_pow2(ncmax) * sizeof(float), s>>>(
                w.attn, ncmax, positions, seqs, n_seqs, m->max_pos, nh, hd, w.att);
            QLIN_LAUNCHED("lanes_attn_merge_kernel");
        }
        if ((st = quant_i8_tiles(w.att, codes, w.xs, M, qd, tiles, s)) || (st = lin_group(l, 3, 1, &w.y))) return st;
        if ((st = norm_quant_tiles(w.h, w.y, m->g_ffn + (int64_t)l * d, m->eps, codes, w.xs, M, d, tiles, s))) return st;
        {
            float *const gu[2] = {w.g, w.u};
            if ((st = lin_group(l, 4, 2, gu))) return st;
        }
        if ((st = geglu_quant_tiles(w.g, w.u, codes, w.xs, M, f, tiles, s)) || (st = lin_group(l, 6, 1, &w.y))) return st;
    }
    lanes_add_kernel<<<add_blocks, 256, 0, s>>>(w.h, w.y, (int64_t)M * d);  // the last layer's FFN output
    QLIN_LAUNCHED("lanes_add_kernel");
    if ((st = qlin_rmsnorm(w.h, m->g_final, w.xn, M, d, m->eps, stream))) return st;
    // the output layer for all lanes in one pass over the table (tensor cores)
    if ((st = qlin_lm_head_lanes(m->emb, w.xn, m->vocab, d, M, logits, next, w.lm, w.lm_bytes, stream))) return st;
    return QLIN_OK;
}

int decode_lanes_t158_launches(const t158_model *m, int n_lanes) {
    qlin::clear_error();
    if (check_lanes_model(m) || n_lanes < 1) return -1;
    // embed; per layer 4 quantisations (two behind the residual add and RMSNorm, one behind the GeGLU
    // product), 7 linears (3 launches on the tensor cores: q k v, o, gate up, down as 4), rope/append,
    // 2 attention; the last residual add and the final norm; the lanes' output layer (a split and a
    // table pass per 64 lanes)
    const int lin_launches = n_lanes >= kLanesTensorMin ? 4 : 7;
    return 1 + m->n_layers * (7 + lin_launches) + 2 + 2 * ((n_lanes + 63) / 64);
}

qlin_status decode_lanes_t158_status(void *workspace, qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(workspace, QLIN_ERR_INVALID_ARG, "decode_lanes_t158_status: null workspace");
    int32_t stw[4] = {0, 0, 0, 0};
    QLIN_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    QLIN_CUDA(cudaMemcpy(stw, workspace, sizeof stw, cudaMemcpyDeviceToHost));
    QLIN_CUDA(cudaMemset(workspace, 0, sizeof stw));
    QLIN_REQUIRE(!(stw[0] & kLaneStatusBad), QLIN_ERR_INVALID_ARG,
                 "decode_lanes_t158: a lane's token, position or sequence slot was out of range");
    QLIN_REQUIRE(!(stw[0] & kLaneStatusTimeout), QLIN_ERR_TIMEOUT,
                 "decode_lanes_t158: a bounded wait in the attention kernel gave up");
    return QLIN_OK;
}

}  // extern "C"
