// One decode step of the ternary decoder as a single persistent kernel.
//
// The forward pass of llama2.c "The forward pass -- one token, one position"
// (Steps 0-6), with the block structure of the cpp20gemma README
// ("Architecture & implementation": h += attn(rmsnorm(h)); h += mlp(rmsnorm(h));
// logits = lm_head(rmsnorm(h))), every linear layer ternary on int8-quantised
// inputs ("Gemma 3 1B at 114 tokens per second on a laptop CPU", "Step 2").
//
// Grid: one CTA per SM, launched cooperatively so all CTAs are resident.
// Warp 0 (lane 0) is a TMA producer that streams, in order, this CTA's slice
// of every weight matrix of every layer, the cached K/V rows of its attention
// chunks and its rows of the bf16 lm_head table through a ring of shared
// memory slots; it runs ahead of the computation across phase boundaries, so
// the weights of a phase are usually on chip before the phase starts.  Warps
// 1..8 compute.  Per layer there are five phases separated by grid barriers:
//   P1 RMSNorm + quantise (every CTA, redundantly) -> Q/K/V rows
//   P2 RoPE, cache append, attention partials per chunk of 32 positions
//   P3 merge of all chunks (every CTA) -> quantise -> Wo rows -> h += y
//   P4 RMSNorm + quantise -> gate and up rows -> GeGLU
//   P5 quantise GeGLU output -> down rows -> h += y
// then the final RMSNorm and the lm_head with a last-CTA argmax.  Every fp32
// operation that feeds a quantiser is the same device code, in the same
// order, as the standalone kernels, so results are bit-identical to them.
#include "decode_fused.cuh"

namespace qlin {

struct FusedSmem {
    // offsets in bytes into dynamic shared memory
    int slots, xr, seg, rope, racc, hvec, xv, lmx, qs, ks, vs, abuf, scl, misc, ring, total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline FusedSmem fused_smem(const t158_model &m, int G) {
    FusedSmem s;
    const int d = m.dim, qd = m.n_heads * m.head_dim, kvd = m.n_kv_heads * m.head_dim;
    int maxC = 0;
    for (int j = 0; j < T158_NMAT; j++) maxC = maxC > (int)(m.pitch[j] / 16) ? maxC : (int)(m.pitch[j] / 16);
    const int ncmax = (m.max_pos + 31) / 32;
    int o = 0;
    s.slots = o;
    o += kFStages * kFSlot;
    s.xr = o;
    o = align_up(o + maxC * 80, 128);
    s.seg = o;  // 32-element segment sums of a norm (d <= 4096)
    o = align_up(o + 128 * 4, 128);
    s.rope = o;  // cos then sin of this position, head_dim/2 each
    o = align_up(o + m.head_dim * 4, 128);
    s.racc = o;  // integer sums of the rows of one T158 piece (of a gate piece and its up piece)
    o = align_up(o + 2 * kFMaxRows * 4, 128);
    s.hvec = o;
    o = align_up(o + d * 4, 128);
    s.xv = o;
    o = align_up(o + (d > qd ? d : qd) * 4, 128);
    s.lmx = o;
    o = align_up(o + d * 4, 128);
    s.qs = o;
    o = align_up(o + qd * 4, 128);
    s.ks = o;
    o = align_up(o + kvd * 4, 128);
    s.vs = o;
    o = align_up(o + kvd * 4, 128);
    s.abuf = o;
    o = align_up(o + m.ffn * 4, 128);
    s.scl = o;  // every matrix scale of the model
    o = align_up(o + m.n_layers * T158_NMAT * 4, 128);
    s.misc = o;  // red[32] f32, ired[32] i32, sc[32] f32, flags
    o = align_up(o + 512, 128);
    s.ring = o;
    o = align_up(o + (int)sizeof(Ring<kFStages>), 128);
    s.total = o;
    return s;
}

__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(const FusedArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    const t158_model &m = A.m;
    const int G = gridDim.x, b = blockIdx.x;
    const FusedSmem L = fused_smem(m, G);
    uint8_t *slots = smem + L.slots;
    Ring<kFStages> *ring = reinterpret_cast<Ring<kFStages> *>(smem + L.ring);
    float *red = reinterpret_cast<float *>(smem + L.misc);
    int *ired = reinterpret_cast<int *>(smem + L.misc + 128);
    float *sc = reinterpret_cast<float *>(smem + L.misc + 256);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 384);
    int *last_flag = reinterpret_cast<int *>(smem + L.misc + 388);
    int *isum = reinterpret_cast<int *>(smem + L.misc + 392);

    if (threadIdx.x == 0) {
        ring->init(kFConsumerWarps);
        *abort = 0;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();
        int t = 0;
        bool ok = true;
        auto push = [&](const Piece &p) {
            if (!ok) return;
            const int s = t % kFStages;
            if (t >= kFStages && !mbar_wait(&ring->empty[s], ((t / kFStages) - 1) & 1)) {
                raise_status(A.status, kStatusTimeout);
                ok = false;
                return;
            }
            const uint32_t bytes = (uint32_t)p.rows * (uint32_t)p.pitch;
            mbar_arrive_expect_tx(&ring->full[s], bytes);
            bulk_g2s(slots + (size_t)s * kFSlot, p.src, bytes, &ring->full[s], pol);
            t++;
        };
        for (int l = 0; l < m.n_layers && ok; l++) layer_items(A, l, b, G, push);
        if (!A.final_x) lm_items(A, b, G, push);
        for (int u = max(0, t - kFStages); u < t; u++)
            if (!mbar_wait(&ring->full[u % kFStages], (u / kFStages) & 1)) raise_status(A.status, kStatusTimeout);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const Grp g{(int)threadIdx.x - 32, 32 * kFConsumerWarps, 1};
    const int d = m.dim, nh = m.n_heads, nkv = m.n_kv_heads, hd = m.head_dim, ff = m.ffn;
    const int qd = nh * hd, kvd = nkv * hd, half = hd / 2;
    uint4 *xr = reinterpret_cast<uint4 *>(smem + L.xr);
    float *seg = reinterpret_cast<float *>(smem + L.seg);
    float *rc = reinterpret_cast<float *>(smem + L.rope);
    float *hvec = reinterpret_cast<float *>(smem + L.hvec);
    float *xv = reinterpret_cast<float *>(smem + L.xv);
    float4 *lmx = reinterpret_cast<float4 *>(smem + L.lmx);
    float *qs = reinterpret_cast<float *>(smem + L.qs);
    float *ks = reinterpret_cast<float *>(smem + L.ks);
    float *vs = reinterpret_cast<float *>(smem + L.vs);
    int *racc = reinterpret_cast<int *>(smem + L.racc);
    float *abuf = reinterpret_cast<float *>(smem + L.abuf);
    float *scl = reinterpret_cast<float *>(smem + L.scl);

    int t = 0;  // ring item counter, mirrors the producer
    // One thread waits for a slot, then the named barrier releases the group, so
    // every consumer thread sees the same abort flag.  After an abort nothing
    // waits any more: the remaining items are skipped.
    auto wait_full = [&](int item) {
        if (g.tid == 0 && !*abort && !mbar_wait(&ring->full[item % kFStages], (item / kFStages) & 1)) {
            raise_status(A.status, kStatusTimeout);
            *abort = 1;
        }
        g.sync();
    };
    auto take = [&](Piece &) -> const uint8_t * {
        wait_full(t);
        return slots + (size_t)(t % kFStages) * kFSlot;
    };
    auto give = [&]() {
        g.sync();  // every consumer thread is done with the slot
        if (g.lane() == 0 && !*abort) mbar_arrive(&ring->empty[t % kFStages]);
        t++;
    };

    int H0, H1;  // residual rows owned by this CTA (Wo and down outputs)
    share(d, b, G, H0, H1);
    int J0, J1;
    share(ff, b, G, J0, J1);
    const uint32_t seq = *reinterpret_cast<volatile const unsigned *>(A.seq) & 0x3fffffu;

    for (int i = g.tid; i < m.n_layers * T158_NMAT; i += g.n) scl[i] = m.scales[i];
    for (int i = g.tid; i < 2 * kFMaxRows; i += g.n) racc[i] = 0;

    // Step 0: h = emb[token], kept in hvec (owners of residual rows read their rows from it)
    int tok = *A.token;
    if (tok < 0 || tok >= m.vocab) {
        if (g.tid == 0) raise_status(A.status, kStatusBadToken);
        tok = -1;
    }
    for (int i = g.tid; i < d; i += g.n)
        hvec[i] = tok >= 0 ? __uint_as_float((uint32_t)m.emb[(int64_t)tok * d + i] << 16) : 0.0f;
    float *rs = rc + half;
    for (int i = g.tid; i < half; i += g.n) {
        rc[i] = m.rope_cos[(int64_t)A.pos * half + i];
        rs[i] = m.rope_sin[(int64_t)A.pos * half + i];
    }
    g.sync();

    const int nc = A.pos / 32 + 1;
    const int cpos = A.pos / 32;
    const int qkv_rows = qd + 2 * kvd;
    int Q0, Q1;  // rows of the concatenation q | k | v owned by this CTA
    share(qkv_rows, b, G, Q0, Q1);

    // The ops of a layer, in order.  Every kind of work has one code site in
    // the loop body (the loop is not unrolled), so the instructions a layer
    // executes stay few enough to be served from the SM's instruction cache.
    enum : int { kOpQKV = 0, kOpAttn = 1, kOpMerge = 2, kOpWo = 3, kOpGate = 4, kOpUp = 5, kOpDown = 6, kNumOps = 7 };
    int sumx = 0;
    float xs = 0.0f;
    for (int l = 0; l < m.n_layers && !*abort; l++) {
        const float *sc_l = scl + l * T158_NMAT;
        float *kc = A.kv + (int64_t)(2 * l) * m.max_pos * kvd;
        float *vc = A.kv + (int64_t)(2 * l + 1) * m.max_pos * kvd;
#pragma unroll 1
        for (int op = 0; op < kNumOps && !*abort; op++) {
            // ---- input of the op's matrices: RMSNorm + quantise, or quantise
            if (op == kOpQKV || op == kOpGate) {
                const bool qkv = op == kOpQKV;
                // h after layer l-1 (phase 5) for Q K V, h after attention (phase 3) for gate/up
                xs = norm_quant(qkv && l == 0 ? nullptr : A.hT, qkv ? make_tag(seq, l - 1, 5) : make_tag(seq, l, 3),
                                hvec, (qkv ? m.g_attn : m.g_ffn) + (int64_t)l * d, d, m.eps, xv, xr,
                                (int)(m.pitch[qkv ? 0 : 4] / 16), red, seg, isum, &sumx, g, abort, A.status);
            } else if (op == kOpWo || op == kOpDown) {
                const bool wo = op == kOpWo;
                xs = quant_from_tagged(wo ? A.attT : A.aT, wo ? make_tag(seq, l, 6) : make_tag(seq, l, 4),
                                       wo ? qd : ff, wo ? xv : abuf, xr, (int)(m.pitch[wo ? 3 : 6] / 16), red, isum,
                                       &sumx, g, abort, A.status);
            }

            if (op == kOpUp) {
                // up runs together with gate
            } else if (op == kOpAttn) {
                // ---- per (chunk, head) item: RoPE, cache append, attention partials
                const uint32_t tq = make_tag(seq, l, 1), tp = make_tag(seq, l, 2);
                for (int e = b; e < nc * nh; e += G) {
                    const int c = e / nh, hh = e % nh;
                    const int t0 = 32 * c, npre = min(t0 + 32, A.pos) - t0;
                    const int nt = min(32, A.pos + 1 - t0);
                    const bool has_pos = c == cpos;
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
                            fetch_tagged_at<4>([&](int j) { return word(j < 2 ? ua : ub, j & 1); }, mask, tq, v4,
                                               abort, A.status);
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
                    g.sync();
                    if (has_pos && hh == 0) {  // one CTA appends the rotated k and v at pos
                        for (int i = g.tid; i < kvd; i += g.n) {
                            kc[(int64_t)A.pos * kvd + i] = ks[i];
                            vc[(int64_t)A.pos * kvd + i] = vs[i];
                        }
                    }
                    const float *Kc = ks, *Vc = vs;
                    if (npre > 0) {
                        // K rows are item t, V rows item t+1; both are held until the chunk is done
                        if (g.tid == 0 && !*abort &&
                            (!mbar_wait(&ring->full[t % kFStages], (t / kFStages) & 1) ||
                             !mbar_wait(&ring->full[(t + 1) % kFStages], ((t + 1) / kFStages) & 1))) {
                            raise_status(A.status, kStatusTimeout);
                            *abort = 1;
                        }
                        g.sync();
                        uint8_t *kslot = slots + (size_t)(t % kFStages) * kFSlot;
                        uint8_t *vslot = slots + (size_t)((t + 1) % kFStages) * kFSlot;
                        if (nt > npre && !*abort) {  // the current position goes after the cached rows
                            for (int i = g.tid; i < kvd; i += g.n) {
                                reinterpret_cast<float *>(kslot)[npre * kvd + i] = ks[i];
                                reinterpret_cast<float *>(vslot)[npre * kvd + i] = vs[i];
                            }
                            // generic-proxy writes ordered before the next TMA write of the slots
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        }
                        g.sync();
                        Kc = reinterpret_cast<const float *>(kslot);
                        Vc = reinterpret_cast<const float *>(vslot);
                    }
                    if (!*abort) {
                        const int kvh = hh / (nh / nkv);
                        attention_chunk(qs, Kc + kvh * hd, Vc + kvh * hd, kvd, nt, hd, &red[16], &red[17], xv, sc, g);
                        const int64_t pi = (int64_t)hh * A.ncmax + c;
                        if (g.tid == 0) {
                            st_tagged(A.pmT + pi, red[16], tp);
                            st_tagged(A.pST + pi, red[17], tp);
                        }
                        for (int i = g.tid; i < hd; i += g.n) st_tagged(A.pUT + pi * hd + i, xv[i], tp);
                        g.sync();
                    }
                    if (npre > 0) {
                        give();
                        give();
                    }
                }
            } else if (op == kOpMerge) {
                // ---- merge, one output element per warp, spread over the CTAs
                const uint32_t tp = make_tag(seq, l, 2), ta = make_tag(seq, l, 6);
                int o0, o1;
                share(qd, b, G, o0, o1);
                for (int e = o0 + g.warp(); e < o1; e += kFConsumerWarps) {
                    const int hh = e / hd, i = e % hd;
                    const float o = attention_merge_tagged(A.pmT + (int64_t)hh * A.ncmax,
                                                           A.pST + (int64_t)hh * A.ncmax,
                                                           A.pUT + (int64_t)hh * A.ncmax * hd, nc, hd, i, g.lane(), tp,
                                                           abort, A.status);
                    if (g.lane() == 0) st_tagged(A.attT + e, o, ta);
                }
            } else {
                // ---- T158 rows of this CTA and their epilogue.  Q K V is the
                // concatenation q | k | v (three matrices); the others are one matrix.
                int lo, hi;
                if (op == kOpQKV) {
                    lo = Q0;
                    hi = Q1;
                } else if (op == kOpWo || op == kOpDown) {
                    lo = H0;
                    hi = H1;
                } else {
                    lo = J0;
                    hi = J1;
                }
                const uint32_t tg = make_tag(seq, l, op == kOpQKV ? 1 : op == kOpWo ? 3 : op == kOpGate ? 4 : 5);
                const int nmat = op == kOpQKV ? 3 : 1;
#pragma unroll 1
                for (int jm = 0; jm < nmat; jm++) {
                    const int mat = op == kOpQKV ? jm : op == kOpWo ? 3 : op == kOpGate ? 4 : 6;
                    const int base = op == kOpQKV ? (jm == 0 ? 0 : jm == 1 ? qd : qd + kvd) : 0;
                    const int nrows = op == kOpQKV ? (jm == 0 ? qd : kvd) : (op == kOpWo || op == kOpDown ? d : ff);
                    const int a0 = max(lo, base), a1 = min(hi, base + nrows);
                    if (a1 <= a0) continue;
                    const float ws = sc_l[mat], wsu = sc_l[5];
                    const bool gu = op == kOpGate;  // gate piece t, its up piece t + 1
                    pieces(
                        m.w[mat], m.pitch[mat], a0 - base, a1 - base, mat,
                        [&](const Piece &p) {
                            if (gu) {
                                if (g.tid == 0 && !*abort &&
                                    (!mbar_wait(&ring->full[t % kFStages], (t / kFStages) & 1) ||
                                     !mbar_wait(&ring->full[(t + 1) % kFStages], ((t + 1) / kFStages) & 1))) {
                                    raise_status(A.status, kStatusTimeout);
                                    *abort = 1;
                                }
                                g.sync();
                            } else {
                                wait_full(t);
                            }
                            const uint8_t *slot = slots + (size_t)(t % kFStages) * kFSlot;
                            const uint8_t *slot_u = slots + (size_t)((t + 1) % kFStages) * kFSlot;
                            if (!*abort) {
                                // integer row sums to shared memory, then one epilogue
                                // loop (a single copy of the scale / GeGLU / residual code)
                                t158_rows(slot, gu ? 2 * p.rows : p.rows, p.pitch, xr, racc, g, slot_u, p.rows);
                                g.sync();
                                for (int r = g.tid; r < p.rows; r += g.n) {
                                    const int row = base + p.row0 + r;
                                    const int acc = racc[r];
                                    racc[r] = 0;  // zero again for the next piece
                                    const float y = __fmul_rn(__fmul_rn((float)(acc - sumx), ws), xs);
                                    if (op == kOpQKV) {
                                        st_tagged(A.qkvT + row, y, tg);
                                    } else if (gu) {
                                        const int accu = racc[p.rows + r];
                                        racc[p.rows + r] = 0;
                                        const float u = __fmul_rn(__fmul_rn((float)(accu - sumx), wsu), xs);
                                        st_tagged(A.aT + row, __fmul_rn(gelu32(y), u), tg);
                                    } else {  // Wo, down: residual
                                        st_tagged(A.hT + row, __fadd_rn(hvec[row], y), tg);
                                    }
                                }
                            }
                            give();
                            if (gu) give();
                        },
                        kFMaxRows);
                }
            }
        }
    }

    // ---------------- final norm, lm_head, argmax
    float best_v = -__int_as_float(0x7f800000);
    int best_i = 0x7fffffff;
    const bool go = !*abort;  // read once, as every stage of the step does
    if (go && A.final_x) {  // the step ends at the final norm: its output goes to another head
        rmsnorm_from_tagged(A.hT, make_tag(seq, m.n_layers - 1, 5), m.g_final, hvec, xv, d, m.eps, seg, g, abort,
                            A.status);
        if (b == 0)
            for (int c = g.tid; c < d; c += g.n) A.final_x[c] = xv[c];
    } else if (go) {
        rmsnorm_from_tagged(A.hT, make_tag(seq, m.n_layers - 1, 5), m.g_final, hvec, xv, d, m.eps, seg, g, abort,
                            A.status);
        const int C = d / 8;
        for (int c = g.tid; c < C; c += g.n) {
            lmx[c] = make_float4(xv[8 * c], xv[8 * c + 1], xv[8 * c + 2], xv[8 * c + 3]);
            lmx[C + c] = make_float4(xv[8 * c + 4], xv[8 * c + 5], xv[8 * c + 6], xv[8 * c + 7]);
        }
        g.sync();
        const int sub = lane & 15, rsub = lane >> 4, cw = g.warp();
        lm_items(A, b, G, [&](const Piece &p) {
            const uint8_t *slot = take(const_cast<Piece &>(p));
            if (!*abort) {
                for (int r0 = 2 * cw; r0 < p.rows; r0 += 2 * kFConsumerWarps) {
                    const int rit = r0 + rsub;
                    float acc = 0.0f;
                    if (rit < p.rows) {
                        const uint8_t *wrow = slot + (size_t)rit * p.pitch;
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
            give();
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
            *A.lm_ticket = 0u;
            *reinterpret_cast<volatile unsigned *>(A.seq) = (seq + 1u) & 0x3fffffu;  // tags of the next launch
        }
    }
}

size_t fused_smem_bytes(const t158_model *m, int G) { return (size_t)fused_smem(*m, G).total; }

qlin_status launch_decode_fused(const FusedArgs &args, cudaStream_t st) {
    const int G = sm_count();
    const size_t smem = fused_smem_bytes(&args.m, G);
    QLIN_REQUIRE((int)smem <= max_smem_optin(), QLIN_ERR_UNSUPPORTED,
                 "decode_step_t158: the model needs %zu B of shared memory per CTA", smem);
    blocks_per_sm((const void *)decode_fused_kernel, smem);  // raises the dynamic shared-memory limit
    int per_sm = 0;
    QLIN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, kFThreads, smem));
    QLIN_REQUIRE(per_sm >= 1, QLIN_ERR_UNSUPPORTED, "decode_step_t158: fused kernel cannot be resident");
    FusedArgs a = args;
    void *params[] = {&a};
    QLIN_CUDA(cudaLaunchCooperativeKernel((const void *)decode_fused_kernel, dim3(G), dim3(kFThreads), params, smem, st));
    return QLIN_OK;
}

}  // namespace qlin
