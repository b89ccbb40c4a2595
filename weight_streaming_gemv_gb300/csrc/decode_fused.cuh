// Pieces of the fused decode step: the byte ring that streams each CTA's
// weights and cached K/V rows into shared memory (the TMA producer and the
// consumer warps walk the same items in the same order), the words CTAs hand
// to one another (tagged values, counted integer sums), quantise-into-planes,
// and T158 rows from shared memory.
#pragma once

#include "decode_ops.cuh"
#include "stream.cuh"

namespace qlin {

constexpr int kRingBytes = 147456;  // byte ring of variable-size items
constexpr int kRingBars = 32;       // items in flight at most (one full and one empty barrier each)
constexpr int kItemMax = 36864;     // largest item (16 bf16 rows of 1152, 36 rows of 1024 B)
constexpr int kFConsumerWarps = 11;  // + 1 producer warp = 12 warps: 3 per SM sub-partition, up to 168 registers
constexpr int kFThreads = 32 * (kFConsumerWarps + 1);
constexpr int kFMaxRows = 160;  // rows of a T158 item: a warp collects at most 32 rounds of row sums

struct FusedArgs {
    t158_model m;
    float *kv;
    const int32_t *token;
    int pos;
    float *logits;
    int32_t *next;
    float *final_x;  // non-null: stop after the final norm and write it here (no lm_head, next untouched)
    // workspace: vectors passed between CTAs as tagged words (value | tag << 32)
    uint64_t *hT, *qkvT, *attT, *aT, *pmT, *pST, *pUT;
    uint64_t *amaxT;  // [G] each CTA's largest |GeGLU output| (tagged)
    uint64_t *hAcc;   // [2][n_layers][dim] counted integer sums of the down projection (by launch parity)
    int ncmax;
    float2 *lm_part;
    unsigned *lm_ticket;  // [8]: the lm_head ticket, then the counters of the six hand-offs of a layer
    unsigned *seq;  // launch sequence number, advanced by the last CTA of every launch
    int32_t *status;
    uint64_t wait_ns;  // longest wait on another CTA or on a copy before the step gives up
    int withhold;      // test hook: >= 0 makes the CTA owning residual row 0 skip its words of that layer
};

// ---------------------------------------------------------------- tagged words
// A float handed from one CTA to others is stored together with a tag in one
// 8-byte word (relaxed, gpu scope: single-copy atomic), so a reader that sees
// the tag of the current launch, layer and phase also sees the value.  This
// replaces grid-wide barriers: every CTA waits only for the words it reads.
__device__ __forceinline__ uint32_t make_tag(uint32_t seq, int layer, int phase) {
    return (seq << 10) | ((uint32_t)layer << 3) | (uint32_t)phase;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
    const uint64_t w = (uint64_t)__float_as_uint(v) | ((uint64_t)tag << 32);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// The wait limit of the current launch (set once per CTA from FusedArgs).
__device__ __forceinline__ uint64_t &wait_limit_ns() {
    __shared__ uint64_t lim;
    return lim;
}

// One poll round found words still missing: true when the caller should stop
// waiting (its limit ran out, or another CTA already gave up and raised the
// timeout bit in the status word, which this CTA then sees within 64 rounds).
__device__ __forceinline__ bool wait_gives_up(int pass, uint64_t &t0, volatile int *abort, int32_t *status) {
    if (*abort) return true;
    if (pass == 0) t0 = global_ns();
    if ((pass & 63) == 63 && (*reinterpret_cast<volatile int32_t *>(status) & kStatusTimeout)) {
        *abort = 1;
        return true;
    }
    if (global_ns() - t0 > wait_limit_ns()) {
        raise_status(status, kStatusTimeout);
        *abort = 1;
        return true;
    }
    return false;
}

// out[j] = value of the tagged word at ptr(j) for every j whose bit is set in
// `mask`, 0 for the others; waits (bounded) until every one of those words
// carries `tag`.  All loads of a round are in flight together; only words
// still stale are reloaded.  On timeout: status gets kStatusTimeout, *abort
// is set.
template <int N, class Ptr>
__device__ __forceinline__ void fetch_tagged_at(Ptr &&ptr, uint32_t mask, uint32_t tag, float (&out)[N],
                                                volatile int *abort, int32_t *status) {
    uint64_t w[N];
#pragma unroll
    for (int j = 0; j < N; j++) w[j] = 0;
    uint32_t pending = mask;
    uint64_t t0 = 0;
    // one block of loads serves the first pass and every retry (a small loop
    // body keeps the instruction cache free for the rest of the layer)
    for (int pass = 0;; pass++) {
#pragma unroll
        for (int j = 0; j < N; j++)
            if (pending & (1u << j)) w[j] = ld_relaxed_u64(ptr(j));
#pragma unroll
        for (int j = 0; j < N; j++)
            if ((pending & (1u << j)) && (uint32_t)(w[j] >> 32) == tag) pending &= ~(1u << j);
        if (!pending || wait_gives_up(pass, t0, abort, status)) break;
        __nanosleep(32);
    }
#pragma unroll
    for (int j = 0; j < N; j++) out[j] = (mask & (1u << j)) ? __uint_as_float((uint32_t)w[j]) : 0.0f;
}

// ---------------------------------------------------------------- hand-off counters
// An all-to-all hand-off (every CTA publishes words, every CTA reads all of
// them) also counts arrivals: after publishing, each CTA adds one to the
// hand-off's counter (relaxed: the words carry their own tags, so their
// visibility need not be ordered with the count), and a reader polls that one
// word with one thread until every CTA has arrived, then reads the words once
// (re-polling only a word whose tag is still stale).  One polled word per CTA
// instead of every word keeps the poll traffic off the words being written.
__device__ __forceinline__ void hop_arrive(unsigned *c) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
}

__device__ __forceinline__ void hop_wait(const unsigned *c, unsigned want, volatile int *abort, int32_t *status) {
    uint64_t t0 = 0;
    for (int pass = 0;; pass++) {
        unsigned v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        if ((int)(v - want) >= 0 || wait_gives_up(pass, t0, abort, status)) return;
        __nanosleep(20);
    }
}

// ---------------------------------------------------------------- counted integer sums
// An exact int32 sum assembled from several CTAs' partial sums: each
// contributor adds 2^48 + (its partial, as a two's-complement 64-bit value)
// to one 8-byte word with a relaxed atomic.  The low 48 bits then hold the
// running sum (|sum| < 2^47) and the high bits the number of contributions,
// so a reader knows the sum is complete when the count reaches the number of
// contributors; integer addition makes the result independent of their order.
__device__ __forceinline__ void counted_add(uint64_t *p, int partial) {
    const uint64_t v = (1ull << 48) + (uint64_t)(int64_t)partial;
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int64_t counted_sum(uint64_t w) { return ((int64_t)(w << 16)) >> 16; }
__device__ __forceinline__ uint32_t counted_count(uint64_t w) { return (uint32_t)((w - (uint64_t)counted_sum(w)) >> 48); }

// out[j] = the complete sum of word ptr(j) for every j whose bit is set in
// mask (0 for the others), once `want` contributions have arrived (bounded
// wait, as fetch_tagged_at).
template <int N, class Ptr>
__device__ __forceinline__ void fetch_counted_at(Ptr &&ptr, uint32_t mask, uint32_t want, int (&out)[N],
                                                 volatile int *abort, int32_t *status) {
    uint64_t w[N];
#pragma unroll
    for (int j = 0; j < N; j++) w[j] = 0;
    uint32_t pending = mask;
    uint64_t t0 = 0;
    for (int pass = 0;; pass++) {
#pragma unroll
        for (int j = 0; j < N; j++)
            if (pending & (1u << j)) w[j] = ld_relaxed_u64(ptr(j));
#pragma unroll
        for (int j = 0; j < N; j++)
            if ((pending & (1u << j)) && counted_count(w[j]) >= want) pending &= ~(1u << j);
        if (!pending || wait_gives_up(pass, t0, abort, status)) break;
        __nanosleep(32);
    }
#pragma unroll
    for (int j = 0; j < N; j++) out[j] = (mask & (1u << j)) ? (int)counted_sum(w[j]) : 0;
}

// src[first + j * stride] for j < count (count <= N)
template <int N>
__device__ __forceinline__ void fetch_tagged(const uint64_t *src, int first, int stride, int count, uint32_t tag,
                                             float (&out)[N], volatile int *abort, int32_t *status) {
    const uint32_t mask = count >= 32 ? 0xffffffffu : (1u << (count > 0 ? count : 0)) - 1u;
    fetch_tagged_at<N>([&](int j) { return src + first + j * stride; }, mask, tag, out, abort, status);
}

// rows [lo, hi) of n rows owned by CTA b of G
__device__ __forceinline__ void share(int n, int b, int G, int &lo, int &hi) {
    lo = (int)((int64_t)n * b / G);
    hi = (int)((int64_t)n * (b + 1) / G);
}

// rows [lo, hi) of the concatenation q | k | v owned by CTA b of G: the CTAs
// are dealt to the three matrices in proportion to their rows, so that no CTA
// takes rows of two matrices (two items, two passes) and waits the hand-off
// for the others (every matrix gets a CTA; with fewer CTAs, a plain split)
__device__ __forceinline__ void qkv_share(int qd, int kvd, int b, int G, int &lo, int &hi) {
    const int total = qd + 2 * kvd;
    const int gq = (int)(((int64_t)G * qd + total / 2) / total), gk = (int)(((int64_t)G * kvd + total / 2) / total);
    const int gv = G - gq - gk;
    if (gq < 1 || gk < 1 || gv < 1) {
        share(total, b, G, lo, hi);
        return;
    }
    int base = 0;
    if (b < gq) {
        share(qd, b, gq, lo, hi);
    } else if (b < gq + gk) {
        share(kvd, b - gq, gk, lo, hi);
        base = qd;
    } else {
        share(kvd, b - gq - gk, gv, lo, hi);
        base = qd + kvd;
    }
    lo += base;
    hi += base;
}

// ---------------------------------------------------------------- the byte ring
// Every CTA streams its share of the step's data (weight rows, cached K/V
// rows, lm_head rows) through one ring of kRingBytes of shared memory, as a
// sequence of items of any size up to kItemMax.  Item i occupies the next
// bytes of the ring (an item that would cross the end starts at 0 instead)
// and uses barrier pair i % kRingBars: full (one producer arrival plus the
// copied bytes) and empty (one arrival per consumer warp when the warp is done
// with it).  Every consumer warp waits for an item by itself, so warps that
// work on different rows of one item never wait for one another.  Consumers release items in order, so the producer may reuse bytes as
// soon as the oldest items holding them are released: small items no longer
// waste a whole slot, and the producer runs as far ahead as the bytes allow.
struct ByteRing {
    uint64_t full[kRingBars];
    uint64_t empty[kRingBars];

    __device__ __forceinline__ void init() {
        for (int s = 0; s < kRingBars; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kFConsumerWarps);
        }
        fence_mbar_init();
    }
};

// Placement of the items: both sides walk the same sizes, so they agree on
// every item's offset without communicating.
struct RingCursor {
    uint32_t v = 0;  // virtual offset of the next item (bytes streamed so far, with skipped tails)
    int i = 0;       // index of the next item
    __device__ __forceinline__ uint32_t place(uint32_t alloc, uint32_t &vstart) {
        uint32_t off = v % kRingBytes;
        if (off + alloc > (uint32_t)kRingBytes) {
            v += kRingBytes - off;
            off = 0;
        }
        vstart = v;
        v += alloc;
        i++;
        return off;
    }
};

// An item: `rows` rows of row_bytes copied from src (row r at src + r *
// src_stride; one bulk copy when the rows are contiguous), with room for
// alloc_rows rows in the ring.
struct Item {
    const uint8_t *src;
    int64_t src_stride;
    int rows, alloc_rows, row_bytes, row0, mat;
};

__device__ __forceinline__ Item make_item(const uint8_t *src, int rows, int row_bytes, int row0, int mat) {
    Item it;
    it.src = src;
    it.src_stride = row_bytes;
    it.rows = rows;
    it.alloc_rows = rows;
    it.row_bytes = row_bytes;
    it.row0 = row0;
    it.mat = mat;
    return it;
}

// Calls f(item) for every item-sized run of rows [lo, hi) of matrix `mat`.
template <class F>
__device__ __forceinline__ void pieces(const uint8_t *base, int64_t pitch, int lo, int hi, int mat, F &&f,
                                       int max_rows = 1 << 30) {
    int per = (int)(kItemMax / pitch) > 0 ? (int)(kItemMax / pitch) : 1;
    per = per < max_rows ? per : max_rows;
    for (int r = lo; r < hi; r += per) f(make_item(base + (int64_t)r * pitch, min(per, hi - r), (int)pitch, r, mat));
}

// The down projection of a layer is split over the grid in two dimensions:
// KG groups of its input (16-byte chunks of the packed rows: 80 inputs each)
// times NG groups of its output rows, CTA b taking input group b % KG and
// row group b / KG.  Each output row then gets KG partial integer sums.
__host__ __device__ __forceinline__ int down_kgroups(int G) { return G % 8 == 0 ? 8 : G % 4 == 0 ? 4 : G % 2 == 0 ? 2 : 1; }

struct DownTile {
    int c0, c1;  // 16-byte chunks [c0, c1) of a packed row
    int r0, r1;  // output rows
};

__device__ __forceinline__ DownTile down_tile(const t158_model &m, int b, int G) {
    const int KG = down_kgroups(G), NG = G / KG;
    const int kg = b % KG, ng = b / KG;
    const int C = (int)(m.pitch[6] / 16);
    DownTile t;
    t.c0 = C * kg / KG;
    t.c1 = C * (kg + 1) / KG;
    t.r0 = m.dim * ng / NG;
    t.r1 = m.dim * (ng + 1) / NG;
    return t;
}

// The items of layer l for CTA b, in consumption order (layer_items calls
// the five generators below in turn; the consumers call each one at its
// phase).  QKV rows are the concatenation q | k | v; attention item e = chunk
// * n_heads + head (chunk = 32 positions) belongs to CTA e mod G and needs
// the cached rows of its chunk below `pos`, K then V (with room for the
// current position's row when the chunk holds it); Wo rows are the residual
// rows this CTA owns; gate and up share the GeGLU rows; the down projection
// is this CTA's tile (its output rows x its input chunks: one copy per row).
template <class F>
__device__ __forceinline__ void qkv_items(const FusedArgs &A, int l, int b, int G, F &&f) {
    const t158_model &m = A.m;
    const int qd = m.n_heads * m.head_dim, kvd = m.n_kv_heads * m.head_dim;
    const int rows[3] = {qd, kvd, kvd};
    int lo, hi;
    qkv_share(qd, kvd, b, G, lo, hi);
    int base = 0;
#pragma unroll
    for (int j = 0; j < 3; j++) {
        const int a0 = max(lo, base), a1 = min(hi, base + rows[j]);
        if (a1 > a0)
            pieces(m.w[j] + (int64_t)l * rows[j] * m.pitch[j], m.pitch[j], a0 - base, a1 - base, j, f, kFMaxRows);
        base += rows[j];
    }
}

// the K and V items of attention item e (none when the chunk has no cached rows)
template <class F>
__device__ __forceinline__ void attn_items(const FusedArgs &A, int l, int e, F &&f) {
    const t158_model &m = A.m;
    const int kvd = m.n_kv_heads * m.head_dim;
    const int c = e / m.n_heads;
    const int t0 = 32 * c, npre = min(t0 + 32, A.pos) - t0;
    const int nt = min(32, A.pos + 1 - t0);
    if (npre <= 0) return;
    const float *kc = A.kv + (int64_t)(2 * l) * m.max_pos * kvd;
    const float *vc = A.kv + (int64_t)(2 * l + 1) * m.max_pos * kvd;
    Item it = make_item(reinterpret_cast<const uint8_t *>(kc + (int64_t)t0 * kvd), npre, kvd * 4, t0, 7);
    it.alloc_rows = nt;
    f(it);
    it.src = reinterpret_cast<const uint8_t *>(vc + (int64_t)t0 * kvd);
    it.mat = 8;
    f(it);
}

template <class F>
__device__ __forceinline__ void wo_items(const FusedArgs &A, int l, int b, int G, F &&f) {
    const t158_model &m = A.m;
    int lo, hi;
    share(m.dim, b, G, lo, hi);
    pieces(m.w[3] + (int64_t)l * m.dim * m.pitch[3], m.pitch[3], lo, hi, 3, f, kFMaxRows);
}

// gate and up in pairs over the same rows (one pass computes both): f(gate item, up item)
template <class F>
__device__ __forceinline__ void gateup_items(const FusedArgs &A, int l, int b, int G, F &&f) {
    const t158_model &m = A.m;
    int g0, g1;
    share(m.ffn, b, G, g0, g1);
    pieces(m.w[4] + (int64_t)l * m.ffn * m.pitch[4], m.pitch[4], g0, g1, 4, [&](const Item &p) {
        Item u = p;
        u.mat = 5;
        u.src = m.w[5] + (int64_t)l * m.ffn * m.pitch[5] + (int64_t)p.row0 * m.pitch[5];
        f(p, u);
    }, kFMaxRows);
}

// the down tile: rows [r0, r1), bytes [16 c0, 16 c1) of each (always one item, maybe empty)
__device__ __forceinline__ Item down_item(const FusedArgs &A, int l, int b, int G) {
    const t158_model &m = A.m;
    const DownTile dt = down_tile(m, b, G);
    Item it = make_item(m.w[6] + (int64_t)l * m.dim * m.pitch[6] + (int64_t)dt.r0 * m.pitch[6] + 16 * dt.c0,
                        dt.c1 > dt.c0 ? dt.r1 - dt.r0 : 0, 16 * (dt.c1 - dt.c0), dt.r0, 6);
    it.src_stride = m.pitch[6];
    return it;
}

// a vector of norm gains (one row of dim floats)
__device__ __forceinline__ Item gain_item(const float *gam, int dim) {
    return make_item(reinterpret_cast<const uint8_t *>(gam), 1, dim * 4, 0, 10);
}

template <class F>
__device__ __forceinline__ void layer_items(const FusedArgs &A, int l, int b, int G, F &&f) {
    f(gain_item(A.m.g_attn + (int64_t)l * A.m.dim, A.m.dim));
    qkv_items(A, l, b, G, f);
    const int nc = A.pos / 32 + 1;
    for (int e = b; e < nc * A.m.n_heads; e += G) attn_items(A, l, e, f);
    wo_items(A, l, b, G, f);
    f(gain_item(A.m.g_ffn + (int64_t)l * A.m.dim, A.m.dim));
    gateup_items(A, l, b, G, [&](const Item &p, const Item &u) {
        f(p);
        f(u);
    });
    f(down_item(A, l, b, G));
}

// lm_head tiles of CTA b
template <class F>
__device__ __forceinline__ void lm_items(const FusedArgs &A, int b, int G, F &&f) {
    const int dim = A.m.dim;
    int lo, hi;
    share(A.m.vocab, b, G, lo, hi);
    // two rows per consumer warp per tile: every warp does one pass
    pieces(reinterpret_cast<const uint8_t *>(A.m.emb), (int64_t)dim * 2, lo, hi, 9, f, 2 * kFConsumerWarps);
}

// ---------------------------------------------------------------- vectors held in registers
// Every vector of the step that feeds a quantiser (h, h', the attention
// output, a slice of the GeGLU output) is held LPT elements per consumer
// thread: thread t owns elements [LPT t, LPT t + LPT).  LPT is 4 for vectors
// of up to 4 x 352 = 1408 elements and 16 above.

// The plane byte of element k of a quantised vector: word c*20 + 4i + w holds,
// in byte b, the code of element 5(16c + 4w + b) + i (c = k / 80).
__device__ __forceinline__ int plane_byte(int k) {
    const int c = k / 80, q = k - 80 * c;
    const int j = q / 5, i = q - 5 * j;
    return (c * 20 + 4 * i + (j >> 2)) * 4 + (j & 3);
}

// Codes of this thread's elements (k = k0 + j < K; zero for K <= k < Kpad)
// for step `scale` written into the planes; returns the sum of the codes.
template <int LPT>
__device__ __forceinline__ int codes_to_planes(const float (&v)[LPT], int k0, int K, int Kpad, float scale,
                                               int8_t *planes) {
    const float rinv = __fdiv_rn(1.0f, scale);
    int s = 0;
#pragma unroll
    for (int j = 0; j < LPT; j++) {
        const int k = k0 + j;
        if (k < Kpad) {
            const int q = k < K ? quant_code_r(v[j], scale, rinv) : 0;
            planes[plane_byte(k)] = (int8_t)q;
            s += q;
        }
    }
    return s;
}

__device__ __forceinline__ int warp_isum(int v) { return __reduce_add_sync(0xffffffffu, v); }

// Largest of a warp's non-negative floats (their bit patterns order as unsigned integers).
__device__ __forceinline__ float warp_max_nonneg(float v) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Largest of a warp's floats (any sign, no NaN): the bits mapped to a signed key
// that orders as the floats do.
__device__ __forceinline__ float warp_max_any(float v) {
    const int b = __float_as_int(v);
    const int k = __reduce_max_sync(0xffffffffu, b ^ ((b >> 31) & 0x7fffffff));
    return __int_as_float(k ^ ((k >> 31) & 0x7fffffff));
}

// Scratch of the register-vector helpers (shared memory, per CTA).
struct VecScratch {
    float wsum[32];  // warp subtree sums of a norm
    float wmax[32];  // warp maxima
    int wisum[32];   // warp code sums
};

// Sum of squares of the vector (d elements) as the pairwise tree over
// next_pow2(d) zero-padded leaves: each thread's LPT leaves in place, then the
// warp's 32 lanes by xor shuffles (adjacent subtrees first), then every thread
// adds the warp subtrees (32 LPT leaves each) in a balanced tree.  One group
// barrier.
template <int LPT>
__device__ __forceinline__ float sumsq_tree(const float (&v)[LPT], int d, VecScratch *S, Grp g) {
    float a[LPT];
#pragma unroll
    for (int j = 0; j < LPT; j++) a[j] = __fmul_rn(v[j], v[j]);
#pragma unroll
    for (int st = 1; st < LPT; st <<= 1)
#pragma unroll
        for (int j = 0; j < LPT; j += 2 * st) a[j] = __fadd_rn(a[j], a[j + st]);
    const float w = warp_psum(a[0]);
    if (g.lane() == 0) S->wsum[g.warp()] = w;
    g.sync();
    const int P = next_pow2(d), W = 32 * LPT, nw = g.n >> 5;
    const int nsub = P > W ? P / W : 1;  // <= 16 for the supported sizes
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; i++) t[i] = (i < nsub && i < nw) ? S->wsum[i] : 0.0f;
#pragma unroll
    for (int st = 1; st < 16; st <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2 * st)
            if (i + st < nsub) t[i] = __fadd_rn(t[i], t[i + st]);
    return t[0];
}

// Absmax quantisation of this thread's elements (values v, K elements, the
// vector's largest |value| at least amax_in) into the planes (bytes up to
// Kpad).  Returns the step; sumx gets the sum of the codes.  Two group
// barriers.
template <int LPT>
__device__ __forceinline__ float quant_regs(const float (&v)[LPT], int K, float amax_in, int Kpad, int8_t *planes,
                                            VecScratch *S, int &sumx, Grp g) {
    const int k0 = LPT * g.tid;
    float amax = amax_in;
#pragma unroll
    for (int j = 0; j < LPT; j++)
        if (k0 + j < K) amax = fmaxf(amax, fabsf(v[j]));
    amax = warp_max_nonneg(amax);
    if (g.lane() == 0) S->wmax[g.warp()] = amax;
    g.sync();
    const int nw = g.n >> 5;
    float m = S->wmax[0];
    for (int w = 1; w < nw; w++) m = fmaxf(m, S->wmax[w]);
    const float scale = quant_scale(m);
    const int s = warp_isum(codes_to_planes<LPT>(v, k0, K, Kpad, scale, planes));
    if (g.lane() == 0) S->wisum[g.warp()] = s;
    g.sync();
    int t = 0;
    for (int w = 0; w < nw; w++) t += S->wisum[w];
    sumx = t;
    return scale;
}

// RMSNorm of this thread's elements of x (d elements, gains gam in shared
// memory), as rmsnorm_row: ss = pairwise sum of x^2, ss = ss/d + eps,
// r = 1/sqrtf(ss), o = g*(r*x).  One group barrier.
template <int LPT>
__device__ __forceinline__ void rmsnorm_regs(const float (&x)[LPT], const float *gam, int d, float eps, float (&o)[LPT],
                                             VecScratch *S, Grp g) {
    float ss = sumsq_tree<LPT>(x, d, S, g);
    ss = __fdiv_rn(ss, (float)d);
    ss = __fadd_rn(ss, eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ss));
    const int k0 = LPT * g.tid;
#pragma unroll
    for (int j = 0; j < LPT; j++) o[j] = (k0 + j < d) ? __fmul_rn(gam[k0 + j], __fmul_rn(r, x[j])) : 0.0f;
}

// RMSNorm, then absmax quantisation into the planes: the step; sumx the sum
// of the codes.  Three group barriers.
template <int LPT>
__device__ __forceinline__ float norm_quant_regs(const float (&x)[LPT], const float *gam, int d, float eps, int Kpad,
                                                 int8_t *planes, VecScratch *S, int &sumx, Grp g) {
    float o[LPT];
    rmsnorm_regs<LPT>(x, gam, d, eps, o, S, g);
    return quant_regs<LPT>(o, d, 0.0f, Kpad, planes, S, sumx, g);
}

// attention_merge_one on tagged partials (pm/pS [chunk], pU [chunk][hd] of
// one head), waiting for each word's tag: one output element per warp.
__device__ __forceinline__ float attention_merge_tagged(const uint64_t *pm, const uint64_t *pS, const uint64_t *pU,
                                                        int nc, int hd, int i, int lane, uint32_t tag,
                                                        volatile int *abort, int32_t *status) {
    const int P = next_pow2(nc);
    const int Lf = P > 32 ? P / 32 : 1;  // leaves per lane: 1, 2 or 4 (nc <= 128)
    const int c0 = lane * Lf;
    const int cnt = c0 < nc ? min(Lf, nc - c0) : 0;
    float all[12];
    const uint32_t m4 = (1u << cnt) - 1u;
    fetch_tagged_at<12>(
        [&](int j) {
            const int c = c0 + (j & 3);
            return j < 4 ? pm + c : j < 8 ? pS + c : pU + (int64_t)c * hd + i;
        },
        m4 | (m4 << 4) | (m4 << 8), tag, all, abort, status);
    float mv[4], sv[4], uv[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        mv[j] = all[j];
        sv[j] = all[4 + j];
        uv[j] = all[8 + j];
    }
    float m = -__int_as_float(0x7f800000);
#pragma unroll
    for (int j = 0; j < 4; j++)
        if (j < cnt) m = fmaxf(m, mv[j]);
    m = warp_max(m);
    float ws[4], wu[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const bool ok = j < cnt;
        const float w = ok ? exp32(__fsub_rn(mv[j], m)) : 0.0f;
        ws[j] = ok ? __fmul_rn(sv[j], w) : 0.0f;
        wu[j] = ok ? __fmul_rn(uv[j], w) : 0.0f;
    }
    float s_l = ws[0], u_l = wu[0];
    if (Lf == 2) {
        s_l = __fadd_rn(ws[0], ws[1]);
        u_l = __fadd_rn(wu[0], wu[1]);
    } else if (Lf == 4) {
        s_l = __fadd_rn(__fadd_rn(ws[0], ws[1]), __fadd_rn(ws[2], ws[3]));
        u_l = __fadd_rn(__fadd_rn(wu[0], wu[1]), __fadd_rn(wu[2], wu[3]));
    }
    const float S = warp_psum(s_l);
    const float U = warp_psum(u_l);
    return __fdiv_rn(U, S);
}

// ---------------------------------------------------------------- T158 rows from a slot
// acc + the dot product of one 16-byte chunk of packed trits (digits 0..2)
// with its 80 activation codes in plane order X[0..5).
__device__ __forceinline__ int chunk_dot(const uint4 wv, const uint4 *X, int acc) {
    uint32_t D[4][5];
    t158_planes(wv.x, D[0]);
    t158_planes(wv.y, D[1]);
    t158_planes(wv.z, D[2]);
    t158_planes(wv.w, D[3]);
    // four independent accumulator chains (integer sums: exact in any order)
    int a0 = acc, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int i = 0; i < 5; i++) {
        const uint4 xv = X[i];
        a0 = dp4a(D[0][i], xv.x, a0);
        a1 = dp4a(D[1][i], xv.y, a1);
        a2 = dp4a(D[2][i], xv.z, a2);
        a3 = dp4a(D[3][i], xv.w, a3);
    }
    return (a0 + a1) + (a2 + a3);
}

// Sums over the two 16-lane halves of a warp (integer: exact in any order);
// every lane of the warp must call it.  lo: the low half's sum, hi: the high half's.
__device__ __forceinline__ void half_isums(int v, int lane, int &lo, int &hi) {
    lo = __reduce_add_sync(0xffffffffu, lane < 16 ? v : 0);
    hi = __reduce_add_sync(0xffffffffu, lane < 16 ? 0 : v);
}

}  // namespace qlin
