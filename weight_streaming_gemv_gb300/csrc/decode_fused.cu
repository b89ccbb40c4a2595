// One decode step of the ternary decoder as a single persistent kernel.
//
// The forward pass of llama2.c "The forward pass -- one token, one position"
// (Steps 0-6), with the block structure of the cpp20gemma README
// ("Architecture & implementation": h += attn(rmsnorm(h)); h += mlp(rmsnorm(h));
// logits = lm_head(rmsnorm(h))), every linear layer ternary on int8-quantised
// inputs ("Gemma 3 1B at 114 tokens per second on a laptop CPU", "Step 2").
//
// Grid: one CTA per SM, launched cooperatively so all CTAs are resident.
// Lane 0 of warp 0 is a TMA producer that streams, in order, this CTA's share
// of every weight matrix of every layer, the cached K/V rows of its attention
// chunks and its rows of the bf16 lm_head table through a byte ring in shared
// memory; it runs ahead of the computation across phase boundaries, so the
// data of a phase is usually on chip before the phase starts.  Warps 1..11
// compute.  Every CTA keeps the whole residual vector h.  Per layer:
//   RMSNorm + quantise (every CTA, from its own h) -> this CTA's Q/K/V rows
//   RoPE, cache append, attention partials per (chunk of 32 positions, head)
//   merge of the chunks for this CTA's share of the attention output
//   quantise the attention output -> this CTA's Wo rows -> h' rows
//   every CTA gathers h' -> RMSNorm + quantise -> gate and up rows -> GeGLU
//   quantise the GeGLU output (its largest |value| gathered from every CTA)
//     -> this CTA's tile of the down projection (a group of input chunks x a
//     group of output rows) -> integer partial sums added into counted words
//   every CTA reads the complete sums -> h'' = h' + y (its own copy of h)
// then the final RMSNorm and the lm_head with a last-CTA argmax.  Every fp32
// operation that feeds a quantiser is the same device code, in the same
// order, as the standalone kernels, so results are bit-identical to them.
#include "decode_fused.cuh"

namespace qlin {

struct FusedSmem {
    // offsets in bytes into dynamic shared memory
    int ringbuf, xr, rope, hvec, xv, lmx, qs, ks, vs, ew, scl, vec, misc, ring, total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline FusedSmem fused_smem(const t158_model &m, int G) {
    FusedSmem s;
    const int d = m.dim, qd = m.n_heads * m.head_dim, kvd = m.n_kv_heads * m.head_dim;
    int maxC = 0;
    for (int j = 0; j < T158_NMAT; j++) maxC = maxC > (int)(m.pitch[j] / 16) ? maxC : (int)(m.pitch[j] / 16);
    int o = 0;
    s.ringbuf = o;
    o += kRingBytes;
    s.xr = o;  // int8 codes in plane order
    o = align_up(o + maxC * 80, 128);
    s.rope = o;  // cos then sin of this position, head_dim/2 each
    o = align_up(o + m.head_dim * 4, 128);
    s.hvec = o;  // this CTA's copy of the residual h
    o = align_up(o + d * 4, 128);
    s.xv = o;  // attention partial U / the final normed x
    o = align_up(o + (d > m.head_dim ? d : m.head_dim) * 4, 128);
    s.lmx = o;
    o = align_up(o + d * 4, 128);
    s.qs = o;
    o = align_up(o + qd * 4, 128);
    s.ks = o;
    o = align_up(o + kvd * 4, 128);
    s.vs = o;
    o = align_up(o + kvd * 4, 128);
    s.ew = o;  // attention weights e_t of a chunk, one copy per consumer warp
    o = align_up(o + kFConsumerWarps * 32 * 4, 128);
    s.scl = o;  // every matrix scale of the model
    o = align_up(o + m.n_layers * T158_NMAT * 4, 128);
    s.vec = o;
    o = align_up(o + (int)sizeof(VecScratch), 128);
    s.misc = o;  // red[32] f32, ired[32] i32, sc[32] f32, flags
    o = align_up(o + 512, 128);
    s.ring = o;
    o = align_up(o + (int)sizeof(ByteRing), 128);
    s.total = o;
    (void)G;
    return s;
}

// The T158 rows of one item against the planes xr, and their epilogue.
enum : int { kEpQKV = 0, kEpWo = 1, kEpGateUp = 2, kEpDown = 3 };

struct PassArgs {
    const uint8_t *slot;    // the item's rows in the ring (gate rows for gate/up)
    const uint8_t *slot_u;  // gate/up: the up rows
    int rows, row_bytes;
    int ep;
    int out_base;  // index in `out` (and hvec) of the item's first row
    float ws, wsu, xs;
    int sumx;      // sum of the codes of the input (of the input slice for kEpDown)
    uint32_t tg;
    uint64_t *out;      // qkvT, hT or aT (tagged words), or the counted words of kEpDown
    const float *hvec;  // kEpWo: the residual
    int skip;           // kEpWo: publish nothing (test hook)
};

// A half warp takes a row (lane j of it chunks j, j + 16, ...) and sums the
// integer dot products over its lanes; gate/up rows go a pair per warp (gate
// in the low half, up in the high half).  A lane's activation codes (its
// chunk's 80 codes) stay in registers for every row when a row has at most
// 16 chunks.  Each warp first collects the sums of all its rows (round j's
// sums in lane j), then those lanes write the rows' results in parallel:
// y = ((acc - sumx) ws) xs as a tagged word (q|k|v), h + y (Wo),
// gelu(y_gate) y_up (GeGLU), or acc - sumx added into the row's counted word
// (the down tile's partial sum).  Returns the largest |GeGLU output| this
// thread wrote (0 otherwise).
__device__ __noinline__ float t158_pass(const PassArgs &P, const uint4 *xr, int lane, int warp, int nwarps) {
    const int C = P.row_bytes / 16;
    const int half = lane >> 4, hl = lane & 15;
    const bool pairs = P.ep == kEpGateUp;
    const int step = pairs ? nwarps : 2 * nwarps;  // rows (pairs) per round over the CTA
    const int first = pairs ? warp : 2 * warp;     // this warp's first row (pair) of a round
    const bool held = C <= 16;                     // one chunk per lane: its codes stay in registers
    uint4 X[5];
#pragma unroll
    for (int i = 0; i < 5; i++) X[i] = (held && hl < C) ? xr[hl * 5 + i] : make_uint4(0u, 0u, 0u, 0u);
    int mine_lo = 0, mine_hi = 0;  // round j's sums land in lane j
    int nr = 0;                    // rounds of this warp (<= 32)
    for (int r0 = first; r0 < P.rows; r0 += step, nr++) {
        const int r = pairs ? r0 : r0 + half;
        int acc = 0;
        if (r < P.rows) {
            const uint8_t *wr = (pairs && half ? P.slot_u : P.slot) + (size_t)r * P.row_bytes;
            if (held) {
                if (hl < C) acc = chunk_dot(lds128(wr + (size_t)hl * 16), X, 0);
            } else {
                for (int c = hl; c < C; c += 16) acc = chunk_dot(lds128(wr + (size_t)c * 16), xr + (size_t)c * 5, acc);
            }
        }
        int lo, hi;
        half_isums(acc, lane, lo, hi);
        if (lane == nr) {
            mine_lo = lo;
            mine_hi = hi;
        }
    }
    float amax = 0.0f;
    if (lane < nr) {
        const int r0 = first + lane * step;
        if (pairs) {
            const float y = __fmul_rn(__fmul_rn((float)(mine_lo - P.sumx), P.ws), P.xs);
            const float u = __fmul_rn(__fmul_rn((float)(mine_hi - P.sumx), P.wsu), P.xs);
            const float a = __fmul_rn(gelu32(y), u);
            amax = fabsf(a);
            st_tagged(P.out + P.out_base + r0, a, P.tg);
        } else {
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int r = r0 + h;
                if (r >= P.rows) continue;
                const int acc = h ? mine_hi : mine_lo;
                const int row = P.out_base + r;
                if (P.ep == kEpDown) {
                    counted_add(P.out + row, acc - P.sumx);
                } else {
                    const float y = __fmul_rn(__fmul_rn((float)(acc - P.sumx), P.ws), P.xs);
                    if (P.ep == kEpQKV)
                        st_tagged(P.out + row, y, P.tg);
                    else if (!P.skip)
                        st_tagged(P.out + row, __fadd_rn(P.hvec[row], y), P.tg);
                }
            }
        }
    }
    return amax;
}

// Scores, weights and value sums of one (chunk, head) item: the arithmetic of
// attention_chunk, the same terms in the same order, laid out for latency.
//   q: smem [hd]; K, V rows t of the chunk at Kc + t*ld, Vc + t*ld (smem);
//   nt valid positions; ew: this CTA's per-warp weight rows [warps][32].
// Scores: lane l holds dims [l S, l S + S) of q (S = hd/32) in registers and
// each warp takes positions warp, warp + 11, warp + 22 together: the lane's
// pairwise subtree over its S products, then the warp's xor shuffles (the
// three positions' interleaved) join the 32 subtrees, adjacent ones first:
// the pairwise tree over hd leaves.  Every warp then takes the chunk's
// maximum, weights and their sum itself; value sums: two dims per thread.
// One group barrier.
template <int HD>
__device__ __forceinline__ void attention_unit(const float *q, const float *Kc, const float *Vc, int ld, int nt,
                                               float *out_m, float *out_S, float *out_U, float *sc, float *ew, Grp g) {
    constexpr int S = HD >= 32 ? HD / 32 : 1;  // dims per lane
    constexpr int TJ = 3;                      // 32 positions over 11 warps
    const int lane = g.lane(), warp = g.warp(), nwarps = g.n >> 5;
    float qr[S];
#pragma unroll
    for (int i = 0; i < S; i++) qr[i] = (HD >= 32 || lane < HD) ? q[lane * S + i] : 0.0f;
    float part[TJ];
#pragma unroll
    for (int j = 0; j < TJ; j++) {
        const int t = warp + nwarps * j;
        const float *k = Kc + (int64_t)(t < nt ? t : 0) * ld;
        float kr[S];
        if constexpr (S == 8) {
            // two 16-byte loads; lanes 4..7 of each shared-memory phase read their
            // upper half first so the 8 lanes of a phase hit distinct banks
            const float4 *k4 = reinterpret_cast<const float4 *>(k + lane * S);
            const int sw = (lane >> 2) & 1;
            const float4 f = k4[sw], s2 = k4[sw ^ 1];
            const float4 lo = sw ? s2 : f, hi = sw ? f : s2;
            kr[0] = lo.x; kr[1] = lo.y; kr[2] = lo.z; kr[3] = lo.w;
            kr[4] = hi.x; kr[5] = hi.y; kr[6] = hi.z; kr[7] = hi.w;
        } else if constexpr (S == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(k + lane * 4);
            kr[0] = v.x; kr[1] = v.y; kr[2] = v.z; kr[3] = v.w;
        } else {
#pragma unroll
            for (int i = 0; i < S; i++) kr[i] = (HD >= 32 || lane < HD) ? k[lane * S + i] : 0.0f;
        }
        float p[S];
#pragma unroll
        for (int i = 0; i < S; i++) p[i] = __fmul_rn(qr[i], kr[i]);
#pragma unroll
        for (int st = 1; st < S; st <<= 1)
#pragma unroll
            for (int i = 0; i < S; i += 2 * st) p[i] = __fadd_rn(p[i], p[i + st]);
        part[j] = (t < nt && (HD >= 32 || lane < HD)) ? p[0] : 0.0f;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float o[TJ];
#pragma unroll
        for (int j = 0; j < TJ; j++) o[j] = __shfl_xor_sync(0xffffffffu, part[j], off);
#pragma unroll
        for (int j = 0; j < TJ; j++) part[j] = __fadd_rn(part[j], o[j]);
    }
    // / sqrt(hd): for hd a power of four the divisor is a power of two and the
    // quotient is the exact product with its reciprocal
    constexpr bool pow4 = HD == 16 || HD == 64 || HD == 256;
    constexpr float rdiv = HD == 16 ? 0.25f : HD == 64 ? 0.125f : 0.0625f;
    if (lane < TJ) {
        const int t = warp + nwarps * lane;
        const float v = lane == 0 ? part[0] : lane == 1 ? part[1] : part[2];
        if (t < 32) sc[t] = (t < nt) ? (pow4 ? __fmul_rn(v, rdiv) : __fdiv_rn(v, __fsqrt_rn((float)HD))) : 0.0f;
    }
    g.sync();
    // every warp: the chunk maximum, the weights e_t = exp(s_t - m) and their pairwise sum
    {
        const bool ok = lane < nt;
        const float s = ok ? sc[lane] : -__int_as_float(0x7f800000);
        const float m = warp_max_any(s);
        const float e = ok ? exp32(__fsub_rn(s, m)) : 0.0f;
        ew[warp * 32 + lane] = e;
        const float Ssum = warp_psum(e);
        if (g.tid == 0) {
            *out_m = m;
            *out_S = Ssum;
        }
        __syncwarp();
    }
    // U: two dims per thread, the pairwise tree over the 32 slots
    const float4 *e4 = reinterpret_cast<const float4 *>(ew + warp * 32);
    for (int i = 2 * g.tid; i < HD; i += 2 * g.n) {
        float e[32];
#pragma unroll
        for (int c = 0; c < 8; c++) {
            const float4 v = e4[c];
            e[4 * c] = v.x;
            e[4 * c + 1] = v.y;
            e[4 * c + 2] = v.z;
            e[4 * c + 3] = v.w;
        }
        float a[32], b[32];
#pragma unroll
        for (int tt = 0; tt < 32; tt++) {
            const float2 v = tt < nt ? *reinterpret_cast<const float2 *>(Vc + (int64_t)tt * ld + i) : make_float2(0.f, 0.f);
            a[tt] = __fmul_rn(e[tt], v.x);
            b[tt] = __fmul_rn(e[tt], v.y);
        }
#pragma unroll
        for (int st = 1; st < 32; st <<= 1)
#pragma unroll
            for (int tt = 0; tt < 32; tt += 2 * st) {
                a[tt] = __fadd_rn(a[tt], a[tt + st]);
                b[tt] = __fadd_rn(b[tt], b[tt + st]);
            }
        out_U[i] = a[0];
        out_U[i + 1] = b[0];
    }
}

__device__ __forceinline__ void attention_unit_any(const float *q, const float *Kc, const float *Vc, int ld, int nt,
                                                   int hd, float *out_m, float *out_S, float *out_U, float *sc,
                                                   float *ew, Grp g) {
    switch (hd) {
        case 16: attention_unit<16>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, ew, g); break;
        case 32: attention_unit<32>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, ew, g); break;
        case 64: attention_unit<64>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, ew, g); break;
        case 128: attention_unit<128>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, ew, g); break;
        default: attention_unit<256>(q, Kc, Vc, ld, nt, out_m, out_S, out_U, sc, ew, g); break;
    }
}

template <int LPT>
__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(const FusedArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    const t158_model &m = A.m;
    const int G = gridDim.x, b = blockIdx.x;
    const FusedSmem L = fused_smem(m, G);
    uint8_t *ringbuf = smem + L.ringbuf;
    ByteRing *ring = reinterpret_cast<ByteRing *>(smem + L.ring);
    float *red = reinterpret_cast<float *>(smem + L.misc);
    int *ired = reinterpret_cast<int *>(smem + L.misc + 128);
    float *sc = reinterpret_cast<float *>(smem + L.misc + 256);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 384);
    int *last_flag = reinterpret_cast<int *>(smem + L.misc + 388);
    unsigned *amax_bits = reinterpret_cast<unsigned *>(smem + L.misc + 396);
    const uint64_t lim = A.wait_ns ? A.wait_ns : kWaitLimitNs;

    if (threadIdx.x == 0) {
        ring->init();
        *abort = 0;
        wait_limit_ns() = lim;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();
        RingCursor cur;
        uint32_t vstart[kRingBars];
        int released = 0;  // items the consumers are known to have released
        bool ok = true;
        auto release_through = [&](int j) {
            while (ok && released <= j) {
                if (*abort || !mbar_wait_for(&ring->empty[released % kRingBars], (released / kRingBars) & 1, lim)) {
                    raise_status(A.status, kStatusTimeout);
                    ok = false;
                    return;
                }
                released++;
            }
        };
        auto push = [&](const Item &it) {
            if (!ok) return;
            const uint32_t alloc = (uint32_t)it.alloc_rows * (uint32_t)it.row_bytes;
            const uint32_t bytes = (uint32_t)it.rows * (uint32_t)it.row_bytes;
            const int i = cur.i;
            if (i >= kRingBars) release_through(i - kRingBars);  // its barrier pair is free again
            // the bytes it will occupy: every older item that starts before its end
            // one lap ago must be released
            uint32_t v0 = cur.v;
            const uint32_t off0 = v0 % kRingBytes;
            if (off0 + alloc > (uint32_t)kRingBytes) v0 += kRingBytes - off0;
            const int64_t limit = (int64_t)v0 + alloc - kRingBytes;
            while (ok && released < i && (int64_t)vstart[released % kRingBars] < limit) release_through(released);
            if (!ok) return;
            uint32_t vs;
            const uint32_t off = cur.place(alloc, vs);
            vstart[i % kRingBars] = vs;
            uint64_t *bar = &ring->full[i % kRingBars];
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes == 0) return;
            if (it.src_stride == it.row_bytes) {
                bulk_g2s(ringbuf + off, it.src, bytes, bar, pol);
            } else {
                for (int r = 0; r < it.rows; r++)
                    bulk_g2s(ringbuf + off + (size_t)r * it.row_bytes, it.src + (int64_t)r * it.src_stride,
                             (uint32_t)it.row_bytes, bar, pol);
            }
        };
        for (int l = 0; l < m.n_layers && ok; l++) layer_items(A, l, b, G, push);
        push(gain_item(m.g_final, m.dim));
        if (!A.final_x) lm_items(A, b, G, push);
        // every copy issued must have landed before the CTA leaves
        for (int u = max(0, cur.i - kRingBars); u < cur.i; u++)
            if (!mbar_wait_for(&ring->full[u % kRingBars], (u / kRingBars) & 1, lim)) raise_status(A.status, kStatusTimeout);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const Grp g{(int)threadIdx.x - 32, 32 * kFConsumerWarps, 1};
    const int d = m.dim, nh = m.n_heads, nkv = m.n_kv_heads, hd = m.head_dim, ff = m.ffn;
    const int qd = nh * hd, kvd = nkv * hd, half = hd / 2;
    int8_t *xr8 = reinterpret_cast<int8_t *>(smem + L.xr);
    const uint4 *xr = reinterpret_cast<const uint4 *>(smem + L.xr);
    float *rc = reinterpret_cast<float *>(smem + L.rope);
    float *hvec = reinterpret_cast<float *>(smem + L.hvec);
    float *xv = reinterpret_cast<float *>(smem + L.xv);
    float4 *lmx = reinterpret_cast<float4 *>(smem + L.lmx);
    float *qs = reinterpret_cast<float *>(smem + L.qs);
    float *ks = reinterpret_cast<float *>(smem + L.ks);
    float *vs = reinterpret_cast<float *>(smem + L.vs);
    float *ew = reinterpret_cast<float *>(smem + L.ew);
    float *scl = reinterpret_cast<float *>(smem + L.scl);
    VecScratch *VS = reinterpret_cast<VecScratch *>(smem + L.vec);

    // The consumers walk the producer's items with their own cursor.  One thread
    // waits for an item; the caller's group barrier then releases the group, so
    // every consumer thread sees the same abort flag.  After an abort nothing
    // waits any more: the remaining items are skipped.
    RingCursor cur;
    auto take = [&](const Item &it, int &idx) -> uint8_t * {  // every warp waits for the item itself
        uint32_t vs0;
        const uint32_t off = cur.place((uint32_t)it.alloc_rows * (uint32_t)it.row_bytes, vs0);
        idx = cur.i - 1;
        if (g.lane() == 0 && !*abort && !mbar_wait_for(&ring->full[idx % kRingBars], (idx / kRingBars) & 1, lim)) {
            raise_status(A.status, kStatusTimeout);
            *abort = 1;
        }
        __syncwarp();
        return ringbuf + off;
    };
    auto give = [&](int idx) {  // this warp is done with the item
        __syncwarp();
        if (g.lane() == 0) mbar_arrive(&ring->empty[idx % kRingBars]);
    };

    int H0, H1;  // residual rows owned by this CTA (Wo outputs)
    share(d, b, G, H0, H1);
    const DownTile dt = down_tile(m, b, G);
    const int KG = down_kgroups(G);
    const int k0 = LPT * g.tid;  // this thread's elements of every register vector
    const uint32_t seq = *reinterpret_cast<volatile const unsigned *>(A.seq) & 0x3fffffu;
    uint64_t *hacc_cur = A.hAcc + (size_t)(seq & 1u) * m.n_layers * d;
    {
        // the other parity's counted words start the next launch at zero
        uint64_t *other = A.hAcc + (size_t)((seq & 1u) ^ 1u) * m.n_layers * d;
        int z0, z1;
        share(m.n_layers * d, b, G, z0, z1);
        for (int i = z0 + g.tid; i < z1; i += g.n) other[i] = 0ull;
    }

    for (int i = g.tid; i < m.n_layers * T158_NMAT; i += g.n) scl[i] = m.scales[i];

    // Step 0: h = emb[token]; every CTA keeps its own copy (hvec) and each thread
    // its elements in registers (hv)
    int tok = *A.token;
    if (tok < 0 || tok >= m.vocab) {
        if (g.tid == 0) raise_status(A.status, kStatusBadToken);
        tok = -1;
    }
    float hv[LPT];
#pragma unroll
    for (int j = 0; j < LPT; j++) {
        const int k = k0 + j;
        hv[j] = (tok >= 0 && k < d) ? __uint_as_float((uint32_t)m.emb[(int64_t)tok * d + k] << 16) : 0.0f;
        if (k < d) hvec[k] = hv[j];
    }
    float *rs = rc + half;
    for (int i = g.tid; i < half; i += g.n) {
        rc[i] = m.rope_cos[(int64_t)A.pos * half + i];
        rs[i] = m.rope_sin[(int64_t)A.pos * half + i];
    }
    g.sync();

    const int nc = A.pos / 32 + 1;
    const int cpos = A.pos / 32;
    int Q0, Q1;  // rows of the concatenation q | k | v owned by this CTA
    qkv_share(qd, kvd, b, G, Q0, Q1);

    int sumx = 0;
    float xs = 0.0f;
    for (int l = 0; l < m.n_layers && !*abort; l++) {
        const float *sc_l = scl + l * T158_NMAT;
        float *kc = A.kv + (int64_t)(2 * l) * m.max_pos * kvd;
        float *vc = A.kv + (int64_t)(2 * l + 1) * m.max_pos * kvd;
        // the T158 rows of one item (two for gate/up): each warp waits for them, does
        // its rows and releases them
        auto rows_pass = [&](int ep, const Item &p, const Item *u, int out_base, uint64_t *out, uint32_t tg, float ws,
                             float wsu, int sx) -> float {
            int i0, i1 = -1;
            PassArgs P;
            P.slot = take(p, i0);
            P.slot_u = u ? take(*u, i1) : nullptr;
            P.rows = p.rows;
            P.row_bytes = p.row_bytes;
            P.ep = ep;
            P.out_base = out_base;
            P.ws = ws;
            P.wsu = wsu;
            P.xs = ep == kEpDown ? 0.0f : xs;
            P.sumx = sx;
            P.tg = tg;
            P.out = out;
            P.hvec = hvec;
            P.skip = ep == kEpWo && A.withhold == l && H0 == 0;  // the test hook withholds row 0's CTA's rows
            const float amax = *abort ? 0.0f : t158_pass(P, xr, g.lane(), g.warp(), kFConsumerWarps);
            give(i0);
            if (u) give(i1);
            return amax;
        };

        // ---- Q K V: RMSNorm + quantise this CTA's copy of h, then its rows of q | k | v
        {
            int ig;
            const float *gam = reinterpret_cast<const float *>(take(gain_item(m.g_attn, d), ig));
            xs = norm_quant_regs<LPT>(hv, gam, d, m.eps, (int)(m.pitch[0] / 16) * 80, xr8, VS, sumx, g);
            give(ig);
            const uint32_t tg = make_tag(seq, l, 1);
            int base = 0;
            const int nrow[3] = {qd, kvd, kvd};
#pragma unroll 1
            for (int jm = 0; jm < 3; jm++) {
                const int a0 = max(Q0, base), a1 = min(Q1, base + nrow[jm]);
                if (a1 > a0) {
                    const float ws = sc_l[jm];
                    const int bb = base;
                    pieces(m.w[jm] + (int64_t)l * nrow[jm] * m.pitch[jm], m.pitch[jm], a0 - base, a1 - base, jm,
                           [&](const Item &p) { rows_pass(kEpQKV, p, nullptr, bb + p.row0, A.qkvT, tg, ws, 0.0f, sumx); },
                           kFMaxRows);
                }
                base += nrow[jm];
            }
        }

        // ---- per (chunk, head) item: RoPE, cache append, attention partials
        {
            g.sync();  // this CTA's q|k|v rows are published
            if (g.tid == 0) {
                hop_arrive(A.lm_ticket + 4);
                if (b < nc * nh) hop_wait(A.lm_ticket + 4, (unsigned)G * (l + 1), abort, A.status);
            }
            g.sync();
            const uint32_t tq = make_tag(seq, l, 1), tp = make_tag(seq, l, 2);
            for (int e = b; e < nc * nh && !*abort; e += G) {
                const int c = e / nh, hh = e % nh;
                const int t0 = 32 * c, npre = min(t0 + 32, A.pos) - t0;
                const int nt = min(32, A.pos + 1 - t0);
                const bool has_pos = c == cpos;
                // the chunk's cached K and V rows: two items, held until the chunk is done
                int ik = -1, iv = -1;
                uint8_t *kslot = nullptr, *vslot = nullptr;
                if (npre > 0) {
                    int n_items = 0;
                    attn_items(A, l, e, [&](const Item &it) {
                        if (n_items++ == 0)
                            kslot = take(it, ik);
                        else
                            vslot = take(it, iv);
                    });
                }
                // q of this head (and k, v of the current position when the chunk holds
                // it), RoPE applied as the words arrive.  Unit u < half: the q pair
                // (u, u + half); then the k pairs of every kv head; then consecutive v pairs.
                {
                    const int nq = half, nk = has_pos ? nkv * half : 0, nvp = has_pos ? kvd / 2 : 0;
                    const int U = nq + nk + nvp;
                    auto word = [&](int u, int which) -> const uint64_t * {
                        if (u < nq) return A.qkvT + hh * hd + u + which * half;
                        u -= nq;
                        if (u < nk) return A.qkvT + qd + (u / half) * hd + (u % half) + which * half;
                        u -= nk;
                        return A.qkvT + qd + kvd + 2 * u + which;
                    };
                    for (int u0 = 0; u0 < U; u0 += 2 * g.n) {
                        const int ua = u0 + g.tid, ub = ua + g.n;
                        const uint32_t mask = (ua < U ? 3u : 0u) | (ub < U ? 12u : 0u);
                        float v4[4];
                        fetch_tagged_at<4>([&](int j) { return word(j < 2 ? ua : ub, j & 1); }, mask, tq, v4, abort,
                                           A.status);
#pragma unroll
                        for (int r = 0; r < 2; r++) {
                            int u = r ? ub : ua;
                            if (u >= U) continue;
                            const float x0 = v4[2 * r], x1 = v4[2 * r + 1];
                            if (u < nq + nk) {
                                float *dst = u < nq ? qs : ks + ((u - nq) / half) * hd;
                                const int i = u < nq ? u : (u - nq) % half;
                                dst[i] = __fsub_rn(__fmul_rn(x0, rc[i]), __fmul_rn(x1, rs[i]));
                                dst[i + half] = __fadd_rn(__fmul_rn(x0, rs[i]), __fmul_rn(x1, rc[i]));
                            } else {
                                u -= nq + nk;
                                vs[2 * u] = x0;
                                vs[2 * u + 1] = x1;
                            }
                        }
                    }
                }
                g.sync();  // q (k, v) staged; the K/V items have landed (thread 0 waited for them)
                const float *Kc = ks, *Vc = vs;
                if (has_pos) {
                    if (hh == 0)  // one CTA appends the rotated k and v at pos
                        for (int i = g.tid; i < kvd; i += g.n) {
                            kc[(int64_t)A.pos * kvd + i] = ks[i];
                            vc[(int64_t)A.pos * kvd + i] = vs[i];
                        }
                    if (npre > 0 && !*abort) {  // the current position goes after the cached rows
                        for (int i = g.tid; i < kvd; i += g.n) {
                            reinterpret_cast<float *>(kslot)[npre * kvd + i] = ks[i];
                            reinterpret_cast<float *>(vslot)[npre * kvd + i] = vs[i];
                        }
                        // generic-proxy writes ordered before the next TMA write of these bytes
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    g.sync();
                }
                if (npre > 0) {
                    Kc = reinterpret_cast<const float *>(kslot);
                    Vc = reinterpret_cast<const float *>(vslot);
                }
                if (!*abort) {
                    const int kvh = hh / (nh / nkv);
                    attention_unit_any(qs, Kc + kvh * hd, Vc + kvh * hd, kvd, nt, hd, &red[16], &red[17], xv, sc, ew, g);
                    g.sync();
                    const int64_t pi = (int64_t)hh * A.ncmax + c;
                    if (g.tid == 0) {
                        st_tagged(A.pmT + pi, red[16], tp);
                        st_tagged(A.pST + pi, red[17], tp);
                    }
                    for (int i = g.tid; i < hd; i += g.n) st_tagged(A.pUT + pi * hd + i, xv[i], tp);
                }
                g.sync();
                if (npre > 0) {
                    give(ik);
                    give(iv);
                }
            }
        }

        // ---- merge, one output element per warp, spread over the CTAs
        {
            if (g.tid == 0) {
                hop_arrive(A.lm_ticket + 5);
                hop_wait(A.lm_ticket + 5, (unsigned)G * (l + 1), abort, A.status);
            }
            g.sync();
            const uint32_t tp = make_tag(seq, l, 2), ta = make_tag(seq, l, 6);
            int o0, o1;
            share(qd, b, G, o0, o1);
            for (int e = o0 + g.warp(); e < o1; e += kFConsumerWarps) {
                const int hh = e / hd, i = e % hd;
                const float o = attention_merge_tagged(A.pmT + (int64_t)hh * A.ncmax, A.pST + (int64_t)hh * A.ncmax,
                                                       A.pUT + (int64_t)hh * A.ncmax * hd, nc, hd, i, g.lane(), tp,
                                                       abort, A.status);
                if (g.lane() == 0) st_tagged(A.attT + e, o, ta);
            }
            g.sync();
            if (g.tid == 0) hop_arrive(A.lm_ticket + 1);
        }

        // ---- Wo: the attention output from every CTA, quantised; this CTA's residual rows
        {
            if (g.tid == 0) hop_wait(A.lm_ticket + 1, (unsigned)G * (l + 1), abort, A.status);
            g.sync();
            float ov[LPT];
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < qd) mask |= 1u << j;
            fetch_tagged_at<LPT>([&](int j) { return A.attT + k0 + j; }, mask, make_tag(seq, l, 6), ov, abort,
                                 A.status);
            xs = quant_regs<LPT>(ov, qd, 0.0f, (int)(m.pitch[3] / 16) * 80, xr8, VS, sumx, g);
            const uint32_t tg = make_tag(seq, l, 3);
            const float ws = sc_l[3];
            wo_items(A, l, b, G, [&](const Item &p) { rows_pass(kEpWo, p, nullptr, p.row0, A.hT, tg, ws, 0.0f, sumx); });
            g.sync();  // every warp has read h before it is overwritten with h'
            if (g.tid == 0) {
                hop_arrive(A.lm_ticket + 2);
                hop_wait(A.lm_ticket + 2, (unsigned)G * (l + 1), abort, A.status);
            }
            g.sync();
        }

        // ---- gate/up: h' from every CTA's rows, RMSNorm + quantise, GeGLU rows
        {
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < d) mask |= 1u << j;
            fetch_tagged_at<LPT>([&](int j) { return A.hT + k0 + j; }, mask, make_tag(seq, l, 3), hv, abort, A.status);
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < d) hvec[k0 + j] = hv[j];  // h' (read by this thread only, before the next barrier)
            if (g.tid == 0) *amax_bits = 0u;  // before the norm's barriers
            int ig;
            const float *gam = reinterpret_cast<const float *>(take(gain_item(m.g_ffn, d), ig));
            xs = norm_quant_regs<LPT>(hv, gam, d, m.eps, (int)(m.pitch[4] / 16) * 80, xr8, VS, sumx, g);
            give(ig);
            const uint32_t tg = make_tag(seq, l, 4);
            float amax = 0.0f;
            gateup_items(A, l, b, G, [&](const Item &p, const Item &u) {
                amax = fmaxf(amax, rows_pass(kEpGateUp, p, &u, p.row0, A.aT, tg, sc_l[4], sc_l[5], sumx));
            });
            amax = warp_max_nonneg(amax);  // every lane that wrote an output holds its |value|
            if (g.lane() == 0) atomicMax(amax_bits, __float_as_uint(amax));  // non-negative floats order as uints
            g.sync();
            if (g.tid == 0) {
                if (!*abort) st_tagged(A.amaxT + b, __uint_as_float(*amax_bits), tg);
                hop_arrive(A.lm_ticket + 6);
                hop_wait(A.lm_ticket + 6, (unsigned)G * (l + 1), abort, A.status);
            }
            g.sync();
        }

        // ---- down: this CTA's input chunks of the GeGLU output and every CTA's
        // largest |value| -> the step and the codes -> its tile's partial sums
        // into the counted words of its output rows
        float xs_d = 0.0f;
        {
            const uint32_t tg = make_tag(seq, l, 4);
            const int ka = 80 * dt.c0, ns = max(0, min(ff, 80 * dt.c1) - ka);
            float av[LPT];
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < ns) mask |= 1u << j;
            fetch_tagged_at<LPT>([&](int j) { return A.aT + ka + k0 + j; }, mask, tg, av, abort, A.status);
            float am[1];
            fetch_tagged_at<1>([&](int) { return A.amaxT + (g.tid < G ? g.tid : 0); }, g.tid < G ? 1u : 0u, tg, am,
                               abort, A.status);
            int sum_slice = 0;
            xs_d = quant_regs<LPT>(av, ns, am[0], (dt.c1 - dt.c0) * 80, xr8, VS, sum_slice, g);
            const Item it = down_item(A, l, b, G);
            uint64_t *hl = hacc_cur + (size_t)l * d;
            if (it.rows > 0) {
                rows_pass(kEpDown, it, nullptr, dt.r0, hl, 0u, 0.0f, 0.0f, sum_slice);
            } else {  // no input chunks: the rows still get this CTA's (empty) contribution
                int idx;
                take(it, idx);
                if (!*abort)
                    for (int r = g.tid; r < dt.r1 - dt.r0; r += g.n) counted_add(hl + dt.r0 + r, 0);
                give(idx);
            }
        }

        // ---- every thread: its elements of the complete down sums -> h'' = h' + y
        // (its registers and this CTA's copy of h)
        {
            g.sync();
            if (g.tid == 0) {
                hop_arrive(A.lm_ticket + 3);
                hop_wait(A.lm_ticket + 3, (unsigned)G * (l + 1), abort, A.status);
            }
            g.sync();
            const uint64_t *hl = hacc_cur + (size_t)l * d;
            const float ws = sc_l[6];
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < d) mask |= 1u << j;
            int a8[LPT];
            fetch_counted_at<LPT>([&](int j) { return hl + k0 + j; }, mask, (uint32_t)KG, a8, abort, A.status);
#pragma unroll
            for (int j = 0; j < LPT; j++)
                if (k0 + j < d) {
                    hv[j] = __fadd_rn(hv[j], __fmul_rn(__fmul_rn((float)a8[j], ws), xs_d));
                    hvec[k0 + j] = hv[j];
                }
            g.sync();
        }
    }

    // ---------------- final norm, lm_head, argmax
    float best_v = -__int_as_float(0x7f800000);
    int best_i = 0x7fffffff;
    {
        int ig;
        const float *gam = reinterpret_cast<const float *>(take(gain_item(m.g_final, d), ig));
        float xn[LPT];
        if (!*abort) rmsnorm_regs<LPT>(hv, gam, d, m.eps, xn, VS, g);
#pragma unroll
        for (int j = 0; j < LPT; j++)
            if (k0 + j < d) xv[k0 + j] = xn[j];
        g.sync();
        give(ig);
    }
    const bool go = !*abort;  // read once, as every stage of the step does
    if (go && A.final_x) {  // the step ends at the final norm: its output goes to another head
        if (b == 0)
            for (int c = g.tid; c < d; c += g.n) A.final_x[c] = xv[c];
    } else if (go) {
        const int C = d / 8;
        for (int c = g.tid; c < C; c += g.n) {
            lmx[c] = make_float4(xv[8 * c], xv[8 * c + 1], xv[8 * c + 2], xv[8 * c + 3]);
            lmx[C + c] = make_float4(xv[8 * c + 4], xv[8 * c + 5], xv[8 * c + 6], xv[8 * c + 7]);
        }
        g.sync();
        const int sub = lane & 15, rsub = lane >> 4, cw = g.warp();
        lm_items(A, b, G, [&](const Item &p) {
            int idx;
            const uint8_t *slot = take(p, idx);
            if (!*abort) {
                for (int r0 = 2 * cw; r0 < p.rows; r0 += 2 * kFConsumerWarps) {
                    const int rit = r0 + rsub;
                    float acc = 0.0f;
                    if (rit < p.rows) {
                        const uint8_t *wrow = slot + (size_t)rit * p.row_bytes;
#pragma unroll 4
                        for (int c = sub; c < C; c += 16) {
                            const uint4 w = lds128(wrow + (size_t)c * 16);
                            const float4 xa = lmx[c], xb = lmx[C + c];
                            acc = fmaf(__uint_as_float(w.x << 16), xa.x, acc);
                            acc = fmaf(__uint_as_float(w.x & 0xffff0000u), xa.y, acc);
                            acc = fmaf(__uint_as_float(w.y << 16), xa.z, acc);
                            acc = fmaf(__uint_as_float(w.y & 0xffff0000u), xa.w, acc);
                            acc = fmaf(__uint_as_float(w.z << 16), xb.x, acc);
                            acc = fmaf(__uint_as_float(w.z & 0xffff0000u), xb.y, acc);
                            acc = fmaf(__uint_as_float(w.w << 16), xb.z, acc);
                            acc = fmaf(__uint_as_float(w.w & 0xffff0000u), xb.w, acc);
                        }
                    }
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                    const int row = p.row0 + rit;
                    if (sub == 0 && rit < p.rows) {
                        if (A.logits) A.logits[row] = acc;
                        if (acc > best_v || (acc == best_v && row < best_i)) {
                            best_v = acc;
                            best_i = row;
                        }
                    }
                }
            }
            give(idx);
        });
    }
    // CTA argmax -> part[b]; the last CTA reduces and resets the shared counters
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best_v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
        if (ov > best_v || (ov == best_v && oi < best_i)) {
            best_v = ov;
            best_i = oi;
        }
    }
    if (lane == 0) {
        red[g.warp()] = best_v;
        ired[g.warp()] = best_i;
    }
    g.sync();
    if (g.tid == 0) {
        float v = red[0];
        int i = ired[0];
        for (int w = 1; w < kFConsumerWarps; w++)
            if (red[w] > v || (red[w] == v && ired[w] < i)) {
                v = red[w];
                i = ired[w];
            }
        A.lm_part[b] = make_float2(v, __int_as_float(i));
        __threadfence();
        *last_flag = (atomicAdd(A.lm_ticket, 1u) == (unsigned)G - 1);
    }
    g.sync();
    if (!*last_flag) return;
    __threadfence();
    if (g.tid < 32) {
        float v = -__int_as_float(0x7f800000);
        int i = 0x7fffffff;
        for (int j = g.tid; j < G; j += 32) {
            const float2 pp = __ldcg(&A.lm_part[j]);
            const int pi = __float_as_int(pp.y);
            if (pp.x > v || (pp.x == v && pi < i)) {
                v = pp.x;
                i = pi;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, off);
            const int oi = __shfl_xor_sync(0xffffffffu, i, off);
            if (ov > v || (ov == v && oi < i)) {
                v = ov;
                i = oi;
            }
        }
        if (g.tid == 0) {
            if (!A.final_x) *A.next = i;
            A.lm_ticket[0] = 0u;
            A.lm_ticket[1] = 0u;  // the hand-off counters start the next launch at zero
            A.lm_ticket[2] = 0u;
            A.lm_ticket[3] = 0u;
            A.lm_ticket[4] = 0u;
            A.lm_ticket[5] = 0u;
            A.lm_ticket[6] = 0u;
            *reinterpret_cast<volatile unsigned *>(A.seq) = (seq + 1u) & 0x3fffffu;  // tags of the next launch
        }
    }
}

size_t fused_smem_bytes(const t158_model *m, int G) { return (size_t)fused_smem(*m, G).total; }

// Elements per consumer thread of the register vectors: 4 when every vector
// (dim, n_heads head_dim, the padded inputs of the T158 rows) fits 4 x 352
// elements, else 16.
int fused_lpt(const t158_model &m, int G) {
    int need = m.dim > m.n_heads * m.head_dim ? m.dim : m.n_heads * m.head_dim;
    for (int j = 0; j < 6; j++) need = need > (int)(m.pitch[j] / 16) * 80 ? need : (int)(m.pitch[j] / 16) * 80;
    const int KG = down_kgroups(G), slice = ((int)(m.pitch[6] / 16) + KG - 1) / KG * 80;  // a down tile's inputs
    need = need > slice ? need : slice;
    return need <= 4 * 32 * kFConsumerWarps ? 4 : need <= 16 * 32 * kFConsumerWarps ? 16 : 0;
}

qlin_status launch_decode_fused(const FusedArgs &args, cudaStream_t st) {
    const int G = sm_count();
    const size_t smem = fused_smem_bytes(&args.m, G);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED,
                 "decode_step_t158: the model needs %zu B of shared memory per CTA", smem);
    const int lpt = fused_lpt(args.m, G);
    QLIN_REQUIRE(lpt > 0 && G <= 32 * kFConsumerWarps, QLIN_ERR_UNSUPPORTED, "decode_step_t158: model too wide");
    const void *kern = lpt == 4 ? (const void *)decode_fused_kernel<4> : (const void *)decode_fused_kernel<16>;
    blocks_per_sm(kern, smem);  // raises the dynamic shared-memory limit
    int per_sm = 0;
    QLIN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFThreads, smem));
    QLIN_REQUIRE(per_sm >= 1, QLIN_ERR_UNSUPPORTED, "decode_step_t158: fused kernel cannot be resident");
    FusedArgs a = args;
    void *params[] = {&a};
    QLIN_CUDA(cudaLaunchCooperativeKernel(kern, dim3(G), dim3(kFThreads), params, smem, st));
    return QLIN_OK;
}

}  // namespace qlin
