// Compressed attention on the tensor cores: O = softmax(Q . Kbar^T / sqrt(d)) . Vbar
// ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// the n x k score matrix replaces n x n and the queries are not compressed;
// section Transformer and Self-Attention: softmax along the key axis; padded
// query rows produce zero output, section Model, padding paragraph).
//
// Persistent CTAs walk a contiguous range of live 128-row query tiles (tiles that
// hold at least one valid row, unit-major), cut so that every CTA gets the same
// total cost; tile j of the range uses TMEM buffer j % 2 (two 256-column buffers).
//
// Each tile's key columns are cut into two halves (a: columns [0, c_b),
// b: [c_b, k)).  Roles (512 threads):
//   warps 0-7   softmax: warp w takes TMEM lane quarter w % 4 and key half
//               w / 4 of every tile and normalises its half by the half's own
//               maximum (no exchange with the other half); each writes its P
//               half (fp16, packed two per column) over the scores it has read
//               and its half's maximum and row sum to shared memory;
//   warps 8-11  epilogue, every live tile in order: O = O_a + g O_b out of TMEM
//               (g brings half b to half a's maximum; this frees the buffer),
//               scaled by 2^e / row sum, rounded, staged with the 128-byte
//               swizzle and stored by TMA in 16 KB pieces;
//   warp 12     producer: Q per tile by TMA into a ring, and per unit the
//               projection step's pre-swizzled Kbar hi/lo images by bulk copy,
//               as soon as the previous unit's score products have finished;
//               its other 31 lanes write the CTA's share of fully padded tiles
//               as zeros;
//   warp 13     one thread issues the score products of each tile once its
//               buffer is free;
//   warps 14-15 one thread each issues P.V of one key half once the tile's P
//               is ready, into its own accumulator O_a / O_b; warp 14 also
//               loads the unit's Vbar image(s) after the previous unit's P.V.
// A single thread issues at most about one MMA per 70-80 cycles whatever its
// shape, so P.V (16 MMAs of N = 64 per tile) is spread over two threads.
// In a buffer (256 columns), with c_b = 128 when k_pad > 128:
//   S   = Q . Kbar_hi^T + Q . Kbar_lo^T   fp32, columns [0, k_pad)
//   P_a over S columns [0, c_b / 2), P_b over [c_b, c_b + (k_pad - c_b) / 2)
//   O_a = P_a . Vbar_a at column 64 (128 when k_pad <= 128), O_b at column 192
// Units whose |Vbar| is larger take two products for P . Vbar (P_hi . Vbar_lo
// added) or, larger still, three (P_lo . Vbar_hi too).  With k_pad > 128 P_lo sits in
// the other buffer at the same columns as P, so such a tile holds both buffers and runs
// alone.  With k_pad <= 128 (a separate instantiation, kLoHere: its code would otherwise
// change the register allocation of the common path of the k_pad > 128 one) a half has
// at most two chunks, both read before anything is written, and P_lo follows the half's
// P over its own scores, so such a tile keeps one buffer and the double buffering.
// The softmax is exact and two-pass (row max, then exp2 with the 1/sqrt(d)
// scale folded in, row sum); scores never leave the SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

namespace linformer {
namespace tc {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kEpilogueWarp = 8, kProducerWarp = 12, kQkWarp = 13, kPvWarp = 14;
// Registers per thread by warpgroup (launched with 128 each): the two softmax
// warpgroups take 136, the epilogue keeps 128, the copy and MMA-issue warpgroup
// gives up 16.  2 x 136 + 128 + 112 = 4 x 128.
constexpr uint32_t kSoftmaxRegs = 136, kIssueRegs = 112;
static_assert(2 * kSoftmaxRegs + 128 + kIssueRegs == 4 * 128, "register split");
constexpr uint32_t kBufCols = 256, kTmemCols = 512;
constexpr uint32_t kImg = 32768;    // largest image: 256 rows x 128 bytes
constexpr uint32_t kQBytes = 16384;
constexpr int kQSlots = 3;
constexpr uint32_t kPiece = 16384;  // one staged store: 128 rows x 128 bytes
// Slots of the per-row maxima and sums: with k_pad <= 128 a tile's scores leave its
// buffer's O columns alone, so the next score products into the buffer wait only for
// the previous tile's P.V, and its softmax may end before that tile's epilogue has read
// the row sums: they rotate over four slots by tile; with k_pad > 128 one per buffer.
constexpr int kRowSlots = 4;
constexpr uint32_t kEpilogueBarrier = 1;

__device__ __forceinline__ int valid_length(const int32_t *pad, int batch, int n) {
    if (!pad) return n;
    const int L = pad[batch];
    return L < 0 ? 0 : (L > n ? n : L);
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Split of a tile's key columns between the two softmax halves.
struct KeySplit {
    int cb;      // first column of half b
    int n0, n1;  // 32-column chunks per half (the last chunk may be ragged)
    int s0, s1;  // 16-key MMA steps per half
    int oa, ob;  // TMEM columns of O_a, O_b within a buffer
};
__device__ __forceinline__ KeySplit key_split(int k, int kpad) {
    const int nch = (k + 31) >> 5;
    KeySplit s;
    if (kpad > 128) {
        s.n0 = 4;
        s.cb = 128;
        s.oa = 64;  // the second half of half a's S columns, consumed by then
    } else {
        s.n0 = (nch + 1) >> 1;
        s.cb = 32 * s.n0;
        s.oa = 128;
    }
    s.n1 = nch - s.n0;
    s.ob = 192;
    s.s0 = (s.cb < kpad ? s.cb : kpad) >> 4;
    s.s1 = s.n1 > 0 ? (kpad - s.cb) >> 4 : 0;
    return s;
}

// Query tiles of a unit that hold at least one valid row, and the relative cost
// of one such tile (by the number of P.Vbar products: measured about 1 : 1.1 : 1.9 in
// launches of one count, but a three-product tile with k_pad > 128, which holds both
// buffers, costs about 2.5 among tiles of other counts (the ragged per-head workload:
// 397.8 -> 374.5 us per forward with 25 instead of 19); 1.3 with k_pad <= 128, where such
// a tile keeps the double buffering).  Only mixed launches use the weights.
__device__ __forceinline__ void unit_cost(const AttnParams &p, int u, int &live, int &weight) {
    const int L = valid_length(p.pad, u / p.h, p.n);
    live = (L + kTileM - 1) / kTileM;
    const int terms = p.forced_terms ? p.forced_terms : info_terms(__ldg(p.info + u));
    weight = terms == 1 ? 10 : (terms == 2 ? 11 : (p.kpad <= 128 ? 13 : 25));
}

// A CTA's share of the work.  Live tiles (unit-major, then tile) are cut into
// gridDim.x ranges of equal total weight: tile (u, t) starts at weight S = (the
// weights of all live tiles before it) and belongs to CTA floor(S G / W).  Fully
// padded tiles are cut into equal counts; their rows are written as zero.
struct TileRanges {
    int u0, t0, u1, t1;  // live tiles from (u0, t0) up to, not including, (u1, t1)
    int du, dt;          // first padded tile
    long long dn;        // number of padded tiles
};

// ceil(c X / G) for 0 <= c <= G (G > 0 at most a few thousand), from q = X / G and
// r = X % G: c X / G = c q + c r / G with c r < G^2.
__device__ __forceinline__ long long part_start(int c, int G, long long q, long long r) {
    return (long long)c * q + (long long)(((unsigned)c * (unsigned)r + (unsigned)G - 1u) / (unsigned)G);
}

// The whole CTA, when lengths or costs differ between units: thread i sums units
// [i U / T, (i+1) U / T) (T threads, at most one unit each for U <= T), a block
// scan gives each thread's base, and the threads holding a range boundary locate
// it within their units.  `scan` is shared scratch of 2 x (warps) 64-bit words.
__device__ __noinline__ void split_tiles_scan(const AttnParams &p, TileRanges *r, long long *scan) {
    constexpr int T = kThreads, NW = kThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int U = p.units, G = gridDim.x, c = blockIdx.x, tpu = p.tiles_per_unit;
    const int ua = (int)(((long long)U * tid) / T), ub = (int)(((long long)U * (tid + 1)) / T);
    int live0 = 0, wt0 = 0;  // the thread's first unit, kept for the boundary search
    if (ua < ub) unit_cost(p, ua, live0, wt0);
    long long ws = (long long)live0 * wt0, ds = ua < ub ? tpu - live0 : 0;
    for (int u = ua + 1; u < ub; ++u) {
        int live, wt;
        unit_cost(p, u, live, wt);
        ws += (long long)live * wt;
        ds += tpu - live;
    }
    long long wi = ws, di = ds;  // inclusive scans within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long x = __shfl_up_sync(0xffffffffu, wi, o), y = __shfl_up_sync(0xffffffffu, di, o);
        if (lane >= o) {
            wi += x;
            di += y;
        }
    }
    if (lane == 31) {
        scan[warp] = wi;
        scan[NW + warp] = di;
    }
    if (tid == 0) {  // defaults: a boundary at the very end
        r->u0 = r->u1 = r->du = U;
        r->t0 = r->t1 = r->dt = 0;
    }
    __syncthreads();
    long long W = 0, D = 0, wb = wi - ws, db = di - ds;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const long long x = scan[i], y = scan[NW + i];
        if (i < warp) {
            wb += x;
            db += y;
        }
        W += x;
        D += y;
    }
    const long long wq = W / G, wr = W - wq * G, dq = D / G, dr = D - dq * G;
    const long long DB = part_start(c, G, dq, dr);  // the first padded tile of this CTA
    if (tid == 0) r->dn = part_start(c + 1, G, dq, dr) - DB;
#pragma unroll 1
    for (int e = 0; e < 2; ++e) {  // the first live tile of this CTA and of the next
        const long long B = part_start(c + e, G, wq, wr);
        if (ws > 0 && wb <= B && B < wb + ws) {
            long long acc = wb;
            for (int u = ua; u < ub; ++u) {
                int live = live0, wt = wt0;
                if (u != ua) unit_cost(p, u, live, wt);
                const long long uw = (long long)live * wt;
                if (B < acc + uw) {
                    const int t = (int)((B - acc + wt - 1) / wt);
                    if (e == 0) {
                        r->u0 = u;
                        r->t0 = t;
                    } else {
                        r->u1 = u;
                        r->t1 = t;
                    }
                    break;
                }
                acc += uw;
            }
        }
    }
    if (ds > 0 && db <= DB && DB < db + ds) {
        long long acc = db;
        for (int u = ua; u < ub; ++u) {
            int live = live0, wt = wt0;
            if (u != ua) unit_cost(p, u, live, wt);
            if (DB < acc + (tpu - live)) {
                r->du = u;
                r->dt = live + (int)(DB - acc);
                break;
            }
            acc += tpu - live;
        }
    }
}

// This CTA's ranges.  Every tile live and of one cost (no lengths, one product
// count): equal tile counts, no scan (the same decision in every thread of every
// CTA).  Otherwise the weighted scan, kept out of line.
__device__ __forceinline__ void split_tiles(const AttnParams &p, TileRanges *r, long long *scan) {
    const int U = p.units, G = gridDim.x, c = blockIdx.x, tpu = p.tiles_per_unit;
    // One product count throughout: forced, or the same in every unit's info word
    // (the whole CTA checks; every thread takes part in the vote).
    bool uniform = p.forced_terms != 0;
    if (p.pad == nullptr && !uniform) {
        const int t0 = info_terms(__ldg(p.info));
        int same = 1;
        for (int u = threadIdx.x; u < U; u += blockDim.x) same &= info_terms(__ldg(p.info + u)) == t0;
        uniform = __syncthreads_and(same) != 0;
    }
    if (p.pad == nullptr && uniform) {
        if (threadIdx.x == 0) {
            const long long X = (long long)U * tpu;
            long long b0, b1;
            if (X * (G + 1) < (1LL << 32)) {  // 32-bit arithmetic suffices
                b0 = ((unsigned)c * (unsigned)X + (unsigned)G - 1u) / (unsigned)G;
                b1 = ((unsigned)(c + 1) * (unsigned)X + (unsigned)G - 1u) / (unsigned)G;
                r->u0 = (int)((unsigned)b0 / (unsigned)tpu);
                r->u1 = (int)((unsigned)b1 / (unsigned)tpu);
            } else {
                const long long q = X / G, rr = X - q * G;
                b0 = part_start(c, G, q, rr);
                b1 = part_start(c + 1, G, q, rr);
                r->u0 = (int)(b0 / tpu);
                r->u1 = (int)(b1 / tpu);
            }
            r->t0 = (int)(b0 - (long long)r->u0 * tpu);
            r->t1 = (int)(b1 - (long long)r->u1 * tpu);
            r->du = U;
            r->dt = 0;
            r->dn = 0;
        }
    } else {
        split_tiles_scan(p, r, scan);
    }
}

// Walks a CTA's live tiles with the unit, tile, valid length and product count
// kept up to date incrementally (units without live tiles are passed over).
struct TileWalk {
    int u, t, L, live, terms, u1, t1;
    __device__ __forceinline__ TileWalk(const AttnParams &p, const TileRanges &r)
        : u(r.u0), t(r.t0), L(0), live(0), terms(1), u1(r.u1), t1(r.t1) {
        if (u < p.units) load_unit(p);
        settle(p);
    }
    __device__ __forceinline__ void load_unit(const AttnParams &p) {
        L = valid_length(p.pad, u / p.h, p.n);
        live = (L + kTileM - 1) / kTileM;
        terms = p.forced_terms ? p.forced_terms : info_terms(__ldg(p.info + u));
    }
    __device__ __forceinline__ void settle(const AttnParams &p) {
        while (t >= live && u < u1) {
            ++u;
            t = 0;
            if (u < p.units) load_unit(p);
            else live = 0;
        }
    }
    __device__ __forceinline__ bool more() const { return u < u1 || (u == u1 && t < t1); }
    __device__ __forceinline__ void next(const AttnParams &p) {
        ++t;
        settle(p);
    }
};

// Walks a CTA's fully padded tiles: tiles [live, tiles_per_unit) of each unit.
struct PadWalk {
    int u, t, end;
    long long left;
    __device__ __forceinline__ PadWalk(const AttnParams &p, const TileRanges &r)
        : u(r.du), t(r.dt), end(p.tiles_per_unit), left(r.dn) {
        settle(p);
    }
    __device__ __forceinline__ void settle(const AttnParams &p) {
        while (left > 0 && t >= end && u + 1 < p.units) {
            ++u;
            t = (valid_length(p.pad, u / p.h, p.n) + kTileM - 1) / kTileM;
        }
        if (t >= end) left = 0;  // nothing further (only if the count ran past the end)
    }
    __device__ __forceinline__ bool more() const { return left > 0; }
    __device__ __forceinline__ void next(const AttnParams &p) {
        ++t;
        --left;
        settle(p);
    }
};

// Padded tile (u, t) written as zero with plain 16-byte stores, shared by `count`
// threads (this one is number `idx`); the tile's rows are contiguous in O.
__device__ __forceinline__ void zero_tile(const AttnParams &p, int u, int t, int idx, int count) {
    const int rows = min(kTileM, p.n - t * kTileM);
    const int chunks = rows * (p.out_fp32 ? 16 : 8);  // 16-byte chunks: 8 or 16 per row
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) +
                                           ((size_t)u * p.n + (size_t)t * kTileM) *
                                               (size_t)(p.out_fp32 ? 256 : 128));
    for (int i = idx; i < chunks; i += count) dst[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Running row max over one 32-column chunk (MASKED: columns >= k are ignored).
template <bool MASKED>
__device__ __forceinline__ void max_chunk(const uint32_t (&v)[32], int c0, int k, float &m0,
                                          float &m1, float &m2, float &m3) {
    if (MASKED) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            if (c0 + i < k) m0 = fmaxf(m0, __uint_as_float(v[i]));
            if (c0 + i + 1 < k) m1 = fmaxf(m1, __uint_as_float(v[i + 1]));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            m0 = max3(m0, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            m1 = max3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            m2 = max3(m2, __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
            m3 = max3(m3, __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
        }
    }
}

// Second-pass work on one 32-column chunk at column c0: p = 2^(s * scale - mb)
// (MASKED: columns >= k give zero), written as packed fp16 to the 16 columns
// at pcol (already read).  The row sum adds p in fp32.
template <bool MASKED>
__device__ __forceinline__ void exp_chunk(const uint32_t (&v)[32], uint32_t pcol, int c0, int k,
                                          float scale, float mb, float &l0, float &l1) {
    uint32_t ph[16];
    const float2 sc = make_float2(scale, scale), nb = make_float2(-mb, -mb);
    float2 acc = make_float2(l0, l1);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float2 x =
            ffma2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc, nb);
        float p0 = ex2_approx(x.x);
        float p1 = ex2_approx(x.y);
        if (MASKED) {
            if (c0 + 2 * e >= k) p0 = 0.f;
            if (c0 + 2 * e + 1 >= k) p1 = 0.f;
        }
        ph[e] = pack_f16(p0, p1);
        acc = fadd2(acc, make_float2(p0, p1));
    }
    l0 = acc.x;
    l1 = acc.y;
    tmem_st16_async(pcol, ph);
}

// The same for three products: P_hi at pcol and P_lo = fp16(p - P_hi) at lcol
// (the other buffer), the row sum of p in fp32.
template <bool MASKED>
__device__ __forceinline__ void exp_chunk3(const uint32_t (&v)[32], uint32_t pcol, uint32_t lcol,
                                           int c0, int k, float scale, float mb, float &l0,
                                           float &l1) {
    const float nb = -mb;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // two halves of 16 columns keep the registers in budget
        uint32_t ph[8], pl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = 16 * h + 2 * e;
            float p0 = ex2_approx(fmaf(__uint_as_float(v[i]), scale, nb));
            float p1 = ex2_approx(fmaf(__uint_as_float(v[i + 1]), scale, nb));
            if (MASKED) {
                if (c0 + i >= k) p0 = 0.f;
                if (c0 + i + 1 >= k) p1 = 0.f;
            }
            ph[e] = pack_f16(p0, p1);
            const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&ph[e]));
            pl[e] = pack_f16(p0 - hf.x, p1 - hf.y);
            l0 += p0;
            l1 += p1;
        }
        tmem_st8_async(pcol + 8 * h, ph);
        tmem_st8_async(lcol + 8 * h, pl);
    }
}

// O_a + g O_b over 32 columns: the two key halves, each normalised by its own
// maximum, brought to the first half's (g = 2^(m_b - m_a)).
__device__ __forceinline__ void combine_halves(uint32_t *o, const uint32_t (&ob)[32], float g) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
        o[i] = __float_as_uint(fmaf(__uint_as_float(ob[i]), g, __uint_as_float(o[i])));
}

// This thread's half of one tile row: chunks [0, nch) starting at column c0 of
// `buf` (all columns >= k are masked), normalised by the half's own maximum, so
// that the two halves of a row never wait for each other; the epilogue brings
// them to the row maximum.  Returns the half's row sum and (in mb) its maximum
// in scaled log2 units.  TMEM loads run one chunk ahead of the arithmetic.
template <bool kLoHere>
__device__ __forceinline__ float softmax_half(uint32_t buf, uint32_t other, int c0, int nch,
                                              int k, float scale, bool three, float &mb) {
    uint32_t va[32], vb[32];
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
    if (nch > 0) tmem_ld32_async(buf + c0, va);
#pragma unroll 1
    for (int c = 0; c < nch; c += 2) {
        const int ca = c0 + 32 * c, cb = ca + 32;
        tmem_wait_ld(va);
        if (c + 1 < nch) tmem_ld32_async(buf + cb, vb);
        if (ca + 32 <= k) max_chunk<false>(va, ca, k, m0, m1, m2, m3);
        else max_chunk<true>(va, ca, k, m0, m1, m2, m3);
        if (c + 1 < nch) {
            tmem_wait_ld(vb);
            if (c + 2 < nch) tmem_ld32_async(buf + cb + 32, va);
            if (cb + 32 <= k) max_chunk<false>(vb, cb, k, m0, m1, m2, m3);
            else max_chunk<true>(vb, cb, k, m0, m1, m2, m3);
        }
    }
    mb = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * scale;
    float l0 = 0.f, l1 = 0.f;
    if (three) {
        // rare; one chunk in registers at a time.  P_lo goes to the other buffer, or with
        // kLoHere (k_pad <= 128: at most two chunks) after this half's P, over scores that
        // must be read first: the second chunk is loaded with the first and moved over.
        if (kLoHere && nch > 1) tmem_ld32_async(buf + c0 + 32, vb);
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            const int ca = c0 + 32 * c;
            if (kLoHere && c == 1) {
#pragma unroll
                for (int i = 0; i < 32; ++i) va[i] = vb[i];
            } else {
                tmem_ld32_async(buf + ca, va);
            }
            tmem_wait_ld(va);
            if (kLoHere && nch > 1 && c == 0) tie32(vb);
            const uint32_t lcol = kLoHere ? buf + c0 + 16 * (nch + c) : other + c0 + 16 * c;
            if (ca + 32 <= k)
                exp_chunk3<false>(va, buf + c0 + 16 * c, lcol, ca, k, scale, mb, l0, l1);
            else
                exp_chunk3<true>(va, buf + c0 + 16 * c, lcol, ca, k, scale, mb, l0, l1);
        }
    } else {
        if (nch > 0) tmem_ld32_async(buf + c0, va);
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
            const int ca = c0 + 32 * c, cb = ca + 32;
            tmem_wait_ld(va);
            if (c + 1 < nch) tmem_ld32_async(buf + cb, vb);
            if (ca + 32 <= k) exp_chunk<false>(va, buf + c0 + 16 * c, ca, k, scale, mb, l0, l1);
            else exp_chunk<true>(va, buf + c0 + 16 * c, ca, k, scale, mb, l0, l1);
            if (c + 1 < nch) {
                tmem_wait_ld(vb);
                if (c + 2 < nch) tmem_ld32_async(buf + cb + 32, va);
                if (cb + 32 <= k)
                    exp_chunk<false>(vb, buf + c0 + 16 * (c + 1), cb, k, scale, mb, l0, l1);
                else
                    exp_chunk<true>(vb, buf + c0 + 16 * (c + 1), cb, k, scale, mb, l0, l1);
            }
        }
    }
    tmem_wait_st();
    return l0 + l1;
}

template <bool kLoHere>
__global__ void __launch_bounds__(kThreads, 1)
    tc_attend_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tO,
                     const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sKh = smem, *sKl = smem + kImg, *sVh = smem + 2 * kImg, *sVl = smem + 3 * kImg;
    uint8_t *sQ = smem + 4 * kImg;          // kQSlots x 16 KB
    uint8_t *sO = sQ + kQSlots * kQBytes;   // two 16 KB staging pieces
    float *rmax = reinterpret_cast<float *>(sO + 2 * kPiece);  // [slot][half][row]
    float *rsum = rmax + kRowSlots * 2 * kTileM;               // [slot][half][row]
    uint64_t *bars = reinterpret_cast<uint64_t *>(rsum + kRowSlots * 2 * kTileM);
    uint64_t *k_full = bars + 0, *k_empty = bars + 1, *v_full = bars + 2, *v_empty = bars + 3;
    uint64_t *q_full = bars + 4, *q_empty = bars + 4 + kQSlots;
    uint64_t *s_full = bars + 4 + 2 * kQSlots;
    uint64_t *p_full = s_full + 2;  // [buffer][key half]
    uint64_t *o_full = s_full + 6, *tmem_free = s_full + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(s_full + 10);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    TileRanges *ranges = reinterpret_cast<TileRanges *>(s_full + 11);
    // One per MMA-issuing thread (scores, P.V half a, P.V half b): a final commit that
    // lets the thread wait for its own products before the CTA frees TMEM, also when
    // a wait elsewhere gave up.
    uint64_t *drain = s_full + 15;
    // k_pad <= 128: one per row slot, completed by the eight softmax warps once the tile's
    // row maxima and sums are written (the epilogue's signal; p_full may by then have run
    // a phase ahead, its next tile in the buffer no longer waiting for the epilogue).
    uint64_t *rows_ready = drain + 3;
    static_assert(4 + 2 * kQSlots + 15 + 3 + kRowSlots <= 32, "barrier area");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t img_bytes = (uint32_t)p.kpad * kRowBytes;
    const KeySplit ks = key_split(p.k, p.kpad);

    if (tid == 0) {
        mbar_init(k_full, 1);
        mbar_init(k_empty, 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 2);  // both P.V threads
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(s_full + s, 1);
            mbar_init(p_full + 2 * s, 4);      // one arrival per softmax warp of key half 0
            mbar_init(p_full + 2 * s + 1, 4);  // ... and of key half 1
            mbar_init(o_full + s, 2);     // both P.V threads
            mbar_init(tmem_free + s, 4);  // one arrival per epilogue warp
        }
        for (int i = 0; i < 3; ++i) mbar_init(drain + i, 1);
        for (int i = 0; i < kRowSlots; ++i) mbar_init(rows_ready + i, 8);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tQ);
        prefetch_tmap(&tO);
    }
    if (warp == kProducerWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // L2 prefetches of the first query tiles of this CTA's range as the closed-form
    // partition gives it (a hint: a prefetch reads nothing into the CTA and cannot be
    // stale; useless only if the weighted partition applies).  Only in the k_pad <= 128
    // instantiation: RoBERTa shape 50.1 -> 48.2 us per forward; the other one is slower
    // with it (headline 143.0 -> 144.1 us), with the same registers and spills.
    if (kLoHere && tid == 0 && p.pad == nullptr) {
        const long long X = (long long)p.units * p.tiles_per_unit;
        const long long q = X / gridDim.x, r = X - q * gridDim.x;
        long long b = part_start(blockIdx.x, gridDim.x, q, r);
        const long long e = part_start(blockIdx.x + 1, gridDim.x, q, r);
        for (int i = 0; i < kQSlots && b < e; ++i, ++b)
            tma_prefetch_3d(&tQ, 0, (int)(b % p.tiles_per_unit) * kTileM, (int)(b / p.tiles_per_unit));
    }
    // Everything above overlaps the projection's last CTAs; its images and info
    // words are read only after this.
    wait_prerequisites();
    // The next forward's projection may be scheduled on SMs as this grid's CTAs leave
    // (it waits for the whole grid before it touches the workspace).
    if (tid == 0) launch_dependents();
    split_tiles(p, ranges, reinterpret_cast<long long *>(rsum));  // rsum is free until the tiles
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const TileRanges rg = *ranges;

    if (warp >= kProducerWarp) {
        setmaxnreg_dec<kIssueRegs>();
        if (warp == kProducerWarp) {
            if (lane == 0) {  // ---------------- producer: Kbar images and Q tiles
                int cur = -1, nk = 0, qit = 0;
                for (TileWalk wk(p, rg); wk.more(); wk.next(p)) {
                    const int u = wk.u, t = wk.t;
                    // The Q tile first (from HBM, the longer wait), then, on a change of
                    // unit, the unit's Kbar images (from L2), once its predecessor's score
                    // products are done.
                    const int s = qit % kQSlots;
                    if (qit >= kQSlots &&
                        !mbar_wait(q_empty + s, ((qit / kQSlots) - 1) & 1, p.status, 22, abort_flag))
                        break;
                    mbar_arrive_expect_tx(q_full + s, kQBytes);
                    tma_load_3d(sQ + s * kQBytes, &tQ, q_full + s, 0, t * kTileM, u);
                    ++qit;
                    if (u != cur) {
                        if (nk > 0 && !mbar_wait(k_empty, (nk - 1) & 1, p.status, 21, abort_flag))
                            break;
                        const uint8_t *src = p.images + (size_t)u * 4 * img_bytes;
                        mbar_arrive_expect_tx(k_full, 2 * img_bytes);
                        bulk_load(sKh, src, img_bytes, k_full);
                        bulk_load(sKl, src + img_bytes, img_bytes, k_full);
                        ++nk;
                        cur = u;
                    }
                }
                // Let every copy this thread started land before the CTA may exit
                // (also after an abort: a copy must not outlive the CTA).
                if (nk > 0) mbar_wait_drain(k_full, (nk - 1) & 1);
                for (int i = qit > kQSlots ? qit - kQSlots : 0; i < qit; ++i)
                    mbar_wait_drain(q_full + (i % kQSlots), (i / kQSlots) & 1);
            } else {  // ---------------- the other 31 lanes: this CTA's fully padded tiles
                for (PadWalk pw(p, rg); pw.more(); pw.next(p)) zero_tile(p, pw.u, pw.t, lane - 1, 31);
            }
            __syncwarp();
        } else if (warp == kQkWarp) {
            if (lane == 0) {  // ---------------- score products S = Q . Kbar^T, tile by tile
                const uint32_t idesc_qk = idesc_f16(128, p.kpad, 1, 0, 0);
                const uint64_t dkh = sdesc(smem_u32(sKh), 16, 1024, kSwizzle128B);
                const uint64_t dkl = sdesc(smem_u32(sKl), 16, 1024, kSwizzle128B);
                uint32_t uses0 = 0, uses1 = 0;  // tiles that have held each buffer
                int j = 0, cur = -1, nk = 0;
                for (TileWalk wk(p, rg); wk.more(); wk.next(p)) {
                    const int u = wk.u, w = j & 1, slot = j % kQSlots, terms = wk.terms;
                    if (u != cur) {
                        // All score products of the previous unit are issued: its Kbar may
                        // be replaced once they finish.
                        if (cur >= 0) mma_commit(k_empty);
                        if (!mbar_wait(k_full, nk & 1, p.status, 23, abort_flag)) break;
                        ++nk;
                        cur = u;
                    }
                    const uint32_t uw = w ? uses1 : uses0, uo = w ? uses0 : uses1;
                    // The buffer's previous tile must be done with its columns: with k_pad <= 128
                    // the scores cover P (consumed once its P.V is done) but not O (read by
                    // the epilogue, which the next P.V into O waits for instead).
                    if (uw > 0 && !mbar_wait(kLoHere ? o_full + w : tmem_free + w, (uw - 1) & 1, p.status,
                                             24, abort_flag))
                        break;
                    if (terms == 3 && !kLoHere && uo > 0 &&
                        !mbar_wait(tmem_free + (w ^ 1), (uo - 1) & 1, p.status, 24, abort_flag))
                        break;
                    if (!mbar_wait(q_full + slot, (j / kQSlots) & 1, p.status, 25, abort_flag)) break;
                    tc_fence_after();
                    const uint64_t dq = sdesc(smem_u32(sQ + slot * kQBytes), 16, 1024, kSwizzle128B);
                    const uint32_t d = tmem + kBufCols * w;
    #pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ss(d, dq + 2 * s, dkh + 2 * s, idesc_qk, s > 0 ? 1u : 0u);
    #pragma unroll
                    for (int s = 0; s < 4; ++s) mma_ss(d, dq + 2 * s, dkl + 2 * s, idesc_qk, 1u);
                    mma_commit(s_full + w);
                    mma_commit(q_empty + slot);
                    if (w) ++uses1;
                    else ++uses0;
                    if (terms == 3 && !kLoHere) {
                        if (w) ++uses0;
                        else ++uses1;
                    }
                    ++j;
                }
                mma_commit(drain);
                mbar_wait_drain(drain, 0);
            }
            __syncwarp();
        } else if (warp >= kPvWarp) {
            if (lane == 0) {  // ---------------- O_half = P_half . Vbar_half, tile by tile
                const int h = warp - kPvWarp;  // key half
                const uint32_t idesc_pv = idesc_f16(128, 64, 0, 0, 1);
                const int c0 = h ? ks.cb : 0, steps = h ? ks.s1 : ks.s0;
                const uint32_t ocol = h ? ks.ob : ks.oa;
                // Vbar rows of this half: the image row of key c sits at byte 128 c.
                const uint64_t dvh =
                    sdesc(smem_u32(sVh), 16, 1024, kSwizzle128B) + (uint64_t)(c0 * kRowBytes >> 4);
                const uint64_t dvl =
                    sdesc(smem_u32(sVl), 16, 1024, kSwizzle128B) + (uint64_t)(c0 * kRowBytes >> 4);
                uint32_t par0 = 0, par1 = 0;
                int j = 0, cur = -1, nv = 0;
                bool fresh = false;  // Vbar of the current unit requested, not yet waited for
                for (TileWalk wk(p, rg); wk.more(); wk.next(p)) {
                    const int u = wk.u, w = j & 1, terms = wk.terms;
                    if (u != cur) {
                        // The previous unit's products must finish before its Vbar is
                        // replaced; the load is half a's job, both wait for it.
                        if (cur >= 0) mma_commit(v_empty);
                        if (h == 0) {
                            if (cur >= 0 && !mbar_wait(v_empty, (nv - 1) & 1, p.status, 21, abort_flag))
                                break;
                            const uint8_t *src = p.images + (size_t)u * 4 * img_bytes;
                            mbar_arrive_expect_tx(v_full, img_bytes * (terms >= 2 ? 2u : 1u));
                            bulk_load(sVh, src + 2 * img_bytes, img_bytes, v_full);
                            if (terms >= 2) bulk_load(sVl, src + 3 * img_bytes, img_bytes, v_full);
                        }
                        ++nv;
                        cur = u;
                        fresh = true;
                    }
                    if (!mbar_wait(p_full + 2 * w + h, w ? par1 : par0, p.status, 26, abort_flag)) break;
                    if (w) par1 ^= 1u;
                    else par0 ^= 1u;
                    if (fresh) {
                        if (!mbar_wait(v_full, (nv - 1) & 1, p.status, 23, abort_flag)) break;
                        fresh = false;
                    }
                    // k_pad <= 128: O of the buffer's previous tile read by the epilogue
                    if (kLoHere && j >= 2 &&
                        !mbar_wait(tmem_free + w, ((j >> 1) - 1) & 1, p.status, 24, abort_flag))
                        break;
                    tc_fence_after();
                    const uint32_t a = tmem + kBufCols * w + c0;          // P_half: 8 columns per step
                    // P_lo (three products): after the half's P, or in the other buffer
                    const uint32_t alo = kLoHere ? tmem + kBufCols * w + c0 + 16 * (h ? ks.n1 : ks.n0)
                                                 : tmem + kBufCols * (w ^ 1) + c0;
                    const uint32_t dO = tmem + kBufCols * w + ocol;
                    // At most 8 steps of 16 keys per half; the issue rate of one thread, not
                    // the loop, bounds these (rolled loops: smaller code, measured faster).
    #pragma unroll 1
                    for (int s = 0; s < steps; ++s)
                        mma_ts(dO, a + 8 * s, dvh + (uint64_t)(s * 128), idesc_pv, s > 0 ? 1u : 0u);
                    if (terms >= 2) {  // P_hi . Vbar_lo
    #pragma unroll 1
                        for (int s = 0; s < steps; ++s)
                            mma_ts(dO, a + 8 * s, dvl + (uint64_t)(s * 128), idesc_pv, 1u);
                    }
                    if (terms == 3) {  // P_lo . Vbar_hi
    #pragma unroll 1
                        for (int s = 0; s < steps; ++s)
                            mma_ts(dO, alo + 8 * s, dvh + (uint64_t)(s * 128), idesc_pv, 1u);
                    }
                    mma_commit(o_full + w);
                    ++j;
                }
                mma_commit(drain + 1 + h);
                mbar_wait_drain(drain + 1 + h, 0);
                if (h == 0 && nv > 0) mbar_wait_drain(v_full, (nv - 1) & 1);  // no copy outlives the CTA
            }
            __syncwarp();
        }
    } else if (warp >= kEpilogueWarp) {  // ---------------- epilogue, every live tile in order
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int tw = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const bool has_b = ks.n1 > 0;
        int j = 0, sb = 0;
        uint32_t par0 = 0, par1 = 0;
        int cur_u = -1, info = 0;
        for (TileWalk wk(p, rg); wk.more(); wk.next(p)) {
            const int u = wk.u, t = wk.t, L = wk.L;
            if (u != cur_u) {
                cur_u = u;
                info = __ldg(p.info + u);
            }
            float l = 1.f;
            bool ok = true;
            uint32_t oa[64];  // O of this row: both key halves, to the first half's maximum
            {
                const int w = j & 1;
                const int rs = kLoHere ? (j & (kRowSlots - 1)) : w;  // row maxima and sums
                const uint32_t rpar = (uint32_t)(j / kRowSlots) & 1u;
                ++j;
                const uint32_t par = w ? par1 : par0;
                ok = kLoHere ? warp_wait(rows_ready + rs, rpar, p.status, 27, abort_flag)
                             : warp_wait(p_full + 2 * w, par, p.status, 27, abort_flag) &&
                                   warp_wait(p_full + 2 * w + 1, par, p.status, 27, abort_flag);
                // Row = (O_a + g O_b) / (l_a + g l_b), g = 2^(m_b - m_a).  g is capped
                // at 2^100: beyond that O_a's share is below fp32 resolution anyway,
                // and O_b g stays finite (|O_b| < 2^21).
                float g = 0.f;
                if (ok) {
                    l = rsum[(rs * 2) * kTileM + tw];
                    if (has_b) {
                        g = ex2_approx(fminf(rmax[(rs * 2 + 1) * kTileM + tw] - rmax[(rs * 2) * kTileM + tw],
                                             100.f));
                        l = fmaf(rsum[(rs * 2 + 1) * kTileM + tw], g, l);
                    }
                    ok = warp_wait(o_full + w, par, p.status, 28, abort_flag);
                }
                if (w) par1 ^= 1u;
                else par0 ^= 1u;
                if (ok) {
                    // Take all of O out of TMEM first and free the buffer at once:
                    // the next score product into it waits for this, nothing else.
                    tc_fence_after();
                    const uint32_t ob_col = tmem + lane_off + kBufCols * w;
                    tmem_ld64_async(ob_col + ks.oa, oa);
                    if (has_b) {
                        uint32_t ob[32];
                        tmem_ld32_async(ob_col + ks.ob, ob);
                        tmem_wait_ld64(oa);
                        tmem_wait_ld(ob);
                        combine_halves(oa, ob, g);
                        tmem_ld32_async(ob_col + ks.ob + 32, ob);
                        tmem_wait_ld(ob);
                        combine_halves(oa + 32, ob, g);
                    } else {
                        tmem_wait_ld64(oa);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(tmem_free + w);
                        if (wk.terms == 3 && !kLoHere) mbar_arrive(tmem_free + (w ^ 1));
                    }
                }
            }
            // Claim the staging buffer(s): one 16 KB piece per tile for bf16, two
            // for fp32; the stores that last used them must have read them.  The
            // four warps leave together if any of their waits failed.
            if (tw == 0) {
                if (p.out_fp32) bulk_wait_read0();
                else bulk_wait_read1();
            }
            if (!named_barrier_and(kEpilogueBarrier, 128, ok)) break;
            // Padded query rows are written as zero (selected, not scaled: their
            // scores may hold anything, NaN included).
            const bool valid = t * kTileM + tw < L;
            const uint32_t keep = valid ? 0xffffffffu : 0u;
            // 2^e (e = the unit's Vbar scale exponent, 0..100) times 1 / row sum.
            const float inv = __int_as_float((info_exp(info) + 127) << 23) * __frcp_rn(l);
#pragma unroll
            for (int i = 0; i < 64; ++i) oa[i] = keep & __float_as_uint(__uint_as_float(oa[i]) * inv);
            if (!p.out_fp32) {  // bf16 row: 8 chunks of 16 bytes
                uint8_t *rowp = sO + sb * kPiece + tw * kRowBytes;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack_bf16(__uint_as_float(oa[8 * c + 2 * e]),
                                          __uint_as_float(oa[8 * c + 2 * e + 1]));
                    *reinterpret_cast<uint4 *>(rowp + ((c ^ (tw & 7)) << 4)) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            } else {  // fp32 row: pieces 0 (columns 0-31) and 1 (32-63)
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    uint8_t *rp = sO + pc * kPiece + tw * kRowBytes;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int b0 = 32 * pc + 4 * c;
                        *reinterpret_cast<uint4 *>(rp + ((c ^ (tw & 7)) << 4)) =
                            make_uint4(oa[b0], oa[b0 + 1], oa[b0 + 2], oa[b0 + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(kEpilogueBarrier, 128);
            if (tw == 0) {
                tma_store_3d(&tO, sO + sb * kPiece, 0, t * kTileM, u);
                if (p.out_fp32) tma_store_3d(&tO, sO + kPiece, 32, t * kTileM, u);
                bulk_commit();
            }
            if (!p.out_fp32) sb ^= 1;
        }
        if (tw == 0) bulk_wait0();
    } else {  // ---------------- softmax, half a row per thread
        setmaxnreg_inc<kSoftmaxRegs>();
        const int h = warp >> 2;  // key half
        const int tw = tid & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int c0 = h ? ks.cb : 0, nch = h ? ks.n1 : ks.n0;
        int j = 0;
        uint32_t par0 = 0, par1 = 0;
        for (TileWalk wk(p, rg); wk.more(); wk.next(p)) {
            const int w = j & 1;
            bool ok = warp_wait(s_full + w, w ? par1 : par0, p.status, 26, abort_flag);
            if (w) par1 ^= 1u;
            else par0 ^= 1u;
            tc_fence_after();
            if (!ok) break;
            float mb;
            const float l = softmax_half<kLoHere>(tmem + lane_off + kBufCols * w,
                                         tmem + lane_off + kBufCols * (w ^ 1), c0, nch, p.k,
                                         p.scale_log2, wk.terms == 3, mb);
            const int rs = kLoHere ? (j & (kRowSlots - 1)) : w;
            rsum[(rs * 2 + h) * kTileM + tw] = l;
            rmax[(rs * 2 + h) * kTileM + tw] = mb;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(p_full + 2 * w + h);
                if (kLoHere) mbar_arrive(rows_ready + rs);
            }
            ++j;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t attend_smem_bytes(int) {
    return 1024 + 4 * kImg + kQSlots * kQBytes + 2 * kPiece + 2 * kRowSlots * 2 * kTileM * sizeof(float) +
           256;
}

int launch_attend(const CUtensorMap &tQ, const CUtensorMap &tO, const AttnParams &p, int grid,
                  cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(tc_attend_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attend_smem_bytes(1)) != cudaSuccess ||
            cudaFuncSetAttribute(tc_attend_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attend_smem_bytes(1)) != cudaSuccess)
            return LINFORMER_ERR_LAUNCH;
        configured_dev = dev;
    }
    KernelScope scope(LINFORMER_KERNEL_ATTEND_TC, s);
    // Programmatic serialisation: the kernel may start while the projection's last
    // CTAs finish (it waits for them before reading their output).
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attend_smem_bytes(p.out_fp32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // k_pad <= 128: the instantiation that keeps three-product tiles in one buffer.
    const cudaError_t e = p.kpad <= 128 ? cudaLaunchKernelEx(&cfg, tc_attend_kernel<true>, tQ, tO, p)
                                        : cudaLaunchKernelEx(&cfg, tc_attend_kernel<false>, tQ, tO, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LINFORMER_ERR_LAUNCH;
    }
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace tc
}  // namespace linformer
