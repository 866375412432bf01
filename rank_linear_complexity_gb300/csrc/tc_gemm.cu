// Batched fp32 matrix products on the tensor cores (declared in simt_gemm.cuh):
// C_z = alpha A_z B_z + beta C_z over units z, with the operand conventions of
// batched_gemm (each operand a row-major matrix of its unit, of its head, or shared,
// read as stored or transposed, with rows or columns at or past the unit's sequence
// length read as zero), and two further forms the backward of the Linformer attention
// needs ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// the forward's definition; the gradients are its chain rule):
//   - a pair item: S = alpha A B and dP = alpha2 A2 B2 of one row tile in two
//     accumulators, the epilogue writing P = the row softmax of S (C) and
//     dS = P (dP - rowsum(P dP)) (C2), the tile holding whole rows;
//   - a sum over units: output matrix g = sum over the units u of its group of A_u B_u
//     (+ A2_u B2_u), the gradient of a projection matrix shared by those units.
//
// fp32 precision from bf16 tensor-core products: every operand element a is split
// as a_hi = bf16(a), a_lo = bf16(a - a_hi) (|a - a_hi - a_lo| <= 2^-18 |a|), and
// C = A_hi B_hi + A_hi B_lo + A_lo B_hi in fp32 (the dropped A_lo B_lo term is at most
// 2^-18 of each product term).
//
// Persistent and warp-specialized: one CTA per SM walks the work items (a 128 x BN
// output tile of one unit, or of one split of its K range, or of one chunk of a group
// of units) in a fixed order, and three roles run through that order concurrently:
//   - eight producer warps read the fp32 tiles of A (128 x 64) and B (64 x BN) of each
//     64-deep step from global memory, coalesced along each operand's contiguous axis,
//     split them and write hi and lo into a ring of shared-memory stages in the
//     128-byte-swizzled layout the MMA reads (K-major when the operand's K axis is
//     contiguous in memory, MN-major when its M or N axis is); a step's loads stay in
//     flight while its producers wait for a free stage;
//   - one thread issues the twelve MMAs of a step (four 16-deep slices, three products
//     each) into one of two TMEM accumulators of BN fp32 columns, the tiles alternating;
//   - four epilogue warps (TMEM lane quarters 0..3) drain the other accumulator, each
//     lane its row, through staging rows in shared memory, so that every fp32 store
//     instruction of C (or of a split's partial) writes four whole 128-byte row pieces.
// So the loads of later steps, the products and the stores of earlier tiles overlap.
// Every wait is bounded (the status word gets 31..34 and the roles stop).
#include <cuda_bf16.h>

#include <algorithm>

#include "simt_gemm.cuh"
#include "sm100_ptx.cuh"

namespace linformer {
namespace simt {
namespace {

using namespace ptx;

constexpr int kTM = 128;                 // output rows per tile
constexpr int kTK = 64;                  // K per step (one 128-byte row of bf16)
constexpr int kProducerWarps = 8;
constexpr int kProducers = kProducerWarps * 32;
constexpr int kEpilogueWarp0 = kProducerWarps;  // warps 8..11: lane quarters 0..3
constexpr int kMmaWarp = kProducerWarps + 4;     // warp 12
constexpr int kThreads = (kMmaWarp + 1) * 32;    // 416
constexpr int kStagePitch = 36;                  // floats per lane's staging row (144 B)
static_assert(kEpilogueWarp0 % 4 == 0, "epilogue warp w reads TMEM lanes 32 (w % 4) ..");

// Stages of the ring (192 KB of operand tiles for every BN) and the shared memory in all.
template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 64 ? 4 : (BN == 128 ? 3 : 2);
    static constexpr uint32_t kA = kTM * kTK * 2, kB = BN * kTK * 2;  // one hi (or lo) tile
    static constexpr uint32_t kStage = 2 * kA + 2 * kB;
    static constexpr uint32_t kRing = kStages * kStage;
    static constexpr uint32_t kTranspose = 4 * 32 * kStagePitch * 4;  // staging rows
    static constexpr uint32_t kTmemCols = 2 * BN;  // 128, 256 or 512: a power of two
    static constexpr size_t kSmem = 1024 + kRing + kTranspose + 256;
};

__device__ __forceinline__ int tc_unit_length(const int32_t *pad, int unit, int h, int n) {
    if (!pad) return n;
    const int L = pad[unit / h];
    return L < 0 ? 0 : (L > n ? n : L);
}

// Byte offset of the 8-byte group of 4 elements starting at (x, k) of an X x 64 tile:
// K-major (row x of 128 bytes holds k = 0..63; k a multiple of 4) or MN-major (row k
// of each 64-wide x block holds x .. x + 63, blocks 8 KB apart; x a multiple of 4).
// 16-byte chunk c of row r sits at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t kmajor_off(int x, int k) {
    return (uint32_t)(x * 128 + ((((k * 2) >> 4) ^ (x & 7)) << 4) + ((k * 2) & 15));
}
__device__ __forceinline__ uint32_t mnmajor_off(int x, int k) {
    const int xi = x & 63;
    return (uint32_t)((x >> 6) * (kTK * 128) + k * 128 + ((((xi * 2) >> 4) ^ (k & 7)) << 4) +
                      ((xi * 2) & 15));
}

// hi and lo bf16 parts of four values, as two 8-byte words.
__device__ __forceinline__ void split4(float4 f, uint2 &hi, uint2 &lo) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(f.x, f.y), h1 = __floats2bfloat162_rn(f.z, f.w);
    const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);  // exact
    const __nv_bfloat162 l0 = __floats2bfloat162_rn(f.x - f0.x, f.y - f0.y);
    const __nv_bfloat162 l1 = __floats2bfloat162_rn(f.z - f1.x, f.w - f1.y);
    hi = make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
    lo = make_uint2(*reinterpret_cast<const uint32_t *>(&l0), *reinterpret_cast<const uint32_t *>(&l1));
}

// A producer thread's share of one BX x 64 operand tile: groups of four consecutive
// elements along the stored matrix's contiguous axis.  Along x (xfast): BX / 4 threads
// cover one k row, group g of thread t is at x = 4 (t % (BX / 4)), k = t / (BX / 4) +
// g (1024 / BX).  Along k: 16 threads cover one x row, x = t / 16 + 16 g, k = 4 (t % 16).
template <int BX>
struct Frag {
    static constexpr int kGroups = BX * kTK / 4 / kProducers;
    static constexpr int kRowThreads = BX / 4;                 // xfast: threads per k row
    static constexpr int kKRowsPerGroup = kProducers / kRowThreads;
    float4 v[kGroups];
};

// Issues the loads of tile (x0 .., k0 ..) of matrix m.  Elements out of range (x >= X,
// k >= K) or masked (x or k at or past the unit's length L, per the operand's masks)
// are zero.  A tile wholly inside and unmasked (the usual case) is read with one 16-byte
// load per group from a per-thread base address; otherwise each group is checked, and
// a wholly valid one is still one 16-byte load when the operand allows it.
template <int BX>
__device__ __forceinline__ void frag_load(Frag<BX> &f, const Operand &o, const float *m, int x0,
                                          int k0, int X, int K, int L, int tid) {
    using F = Frag<BX>;
    const bool inside = o.vec && x0 + BX <= X && k0 + kTK <= K && (!o.mask_x || x0 + BX <= L) &&
                        (!o.mask_k || k0 + kTK <= L);
    if (inside) {
        const float *p;
        long long step;
        if (o.xfast) {
            p = m + (long long)(k0 + tid / F::kRowThreads) * o.ld + x0 + (tid % F::kRowThreads) * 4;
            step = (long long)F::kKRowsPerGroup * o.ld;
        } else {
            p = m + (long long)(x0 + tid / 16) * o.ld + k0 + (tid % 16) * 4;
            step = 16LL * o.ld;
        }
#pragma unroll
        for (int g = 0; g < F::kGroups; ++g) f.v[g] = __ldg(reinterpret_cast<const float4 *>(p + g * step));
        return;
    }
#pragma unroll
    for (int g = 0; g < F::kGroups; ++g) {
        const int x = o.xfast ? x0 + (tid % F::kRowThreads) * 4 : x0 + tid / 16 + 16 * g;
        const int k = o.xfast ? k0 + tid / F::kRowThreads + g * F::kKRowsPerGroup : k0 + (tid % 16) * 4;
        const long long base = o.xfast ? (long long)k * o.ld + x : (long long)x * o.ld + k;
        bool in[4];
        bool all = true;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int xe = o.xfast ? x + e : x, ke = o.xfast ? k : k + e;
            in[e] = xe < X && ke < K && !(o.mask_x && xe >= L) && !(o.mask_k && ke >= L);
            all = all && in[e];
        }
        if (all && o.vec) {
            f.v[g] = __ldg(reinterpret_cast<const float4 *>(m + base));
        } else {
            f.v[g].x = in[0] ? __ldg(m + base) : 0.f;
            f.v[g].y = in[1] ? __ldg(m + base + 1) : 0.f;
            f.v[g].z = in[2] ? __ldg(m + base + 2) : 0.f;
            f.v[g].w = in[3] ? __ldg(m + base + 3) : 0.f;
        }
    }
}

// The hi and lo parts of a thread's groups.
template <int BX>
struct Split {
    uint2 h[Frag<BX>::kGroups], l[Frag<BX>::kGroups];
};
template <int BX>
__device__ __forceinline__ void split_frag(const Frag<BX> &f, Split<BX> &sp) {
#pragma unroll
    for (int g = 0; g < Frag<BX>::kGroups; ++g) split4(f.v[g], sp.h[g], sp.l[g]);
}
// Writes the split groups into their hi and lo tiles.  The swizzle phase of a group's
// row (row % 8) is the same for all of a thread's groups except along x with BX = 256,
// where it alternates.
template <int BX>
__device__ __forceinline__ void store_split(const Split<BX> &sp, int xfast, uint8_t *hi, uint8_t *lo,
                                            int tid) {
    using F = Frag<BX>;
    if (xfast) {
        const int xr = (tid % F::kRowThreads) * 4, kr0 = tid / F::kRowThreads;
#pragma unroll
        for (int g = 0; g < F::kGroups; ++g) {
            const uint32_t off = mnmajor_off(xr, kr0 + g * F::kKRowsPerGroup);
            *reinterpret_cast<uint2 *>(hi + off) = sp.h[g];
            *reinterpret_cast<uint2 *>(lo + off) = sp.l[g];
        }
    } else {
        const uint32_t off0 = kmajor_off(tid / 16, (tid % 16) * 4);
#pragma unroll
        for (int g = 0; g < F::kGroups; ++g) {
            const uint32_t off = off0 + (uint32_t)g * 16u * 128u;  // 16 rows on, same phase
            *reinterpret_cast<uint2 *>(hi + off) = sp.h[g];
            *reinterpret_cast<uint2 *>(lo + off) = sp.l[g];
        }
    }
}

// Shared-memory descriptor of a tile and its advance per 16-deep K slice.  K-major:
// 8-row groups 1 KB apart, +32 bytes a slice (inside the swizzle atom).  MN-major:
// 64-wide x blocks 8 KB apart, 8-row (k) groups 1 KB apart, +2 KB a slice.
__device__ __forceinline__ uint64_t tile_desc(const uint8_t *t, int mn) {
    return sdesc(smem_u32(t), mn ? kTK * 128 : 16, 1024, kSwizzle128B);
}
__device__ __forceinline__ uint64_t slice_step(int mn) { return mn ? 128u : 2u; }

// The work items of one launch, in the order every role walks them: item w is tile
// row mt = w % tiles_m of tile column nt = (w / tiles_m) % tiles_n, of split (or unit
// chunk) sp and output matrix z (a unit, or a group of units in a sum).
struct Sched {
    int tiles_m, tiles_n, splits, zcount;
    long long items;
    int ksteps;              // 64-deep steps of one unit's whole K
    int usum;                // 1: z is a group; its terms i < per_group are units g * ga + i * gb
    int per_group, ga, gb, uc, terms;  // chunks of uc units; terms 2 with A2 B2
    int pair;                // 1: two products per tile (A B, then A2 B2), one accumulator each
};

struct Item {
    int z, row0, col0, split, nk;
    int kbeg, kend, first;   // K range (plain) or first unit term of the chunk (sum)
};

template <int BN>
__device__ __forceinline__ Item item_at(const GemmArgs &g, const Sched &sc, long long w) {
    Item it;
    const int mt = (int)(w % sc.tiles_m);
    w /= sc.tiles_m;
    const int nt = (int)(w % sc.tiles_n);
    w /= sc.tiles_n;
    it.split = (int)(w % sc.splits);
    it.z = (int)(w / sc.splits);
    it.row0 = mt * kTM;
    it.col0 = nt * BN;
    if (sc.usum) {
        it.first = it.split * sc.uc;
        const int cnt = min(sc.per_group - it.first, sc.uc);
        it.nk = cnt > 0 ? cnt * sc.terms * sc.ksteps : 0;
        it.kbeg = 0;
        it.kend = g.K;
    } else if (sc.pair) {
        it.first = 0;
        it.kbeg = 0;
        it.kend = g.K;
        it.nk = 2 * sc.ksteps;
    } else {
        it.first = 0;
        it.kbeg = it.split * g.kchunk;
        it.kend = min(g.K, it.kbeg + g.kchunk);
        it.nk = it.kend > it.kbeg ? (it.kend - it.kbeg + kTK - 1) / kTK : 0;
    }
    return it;
}

// Step s of item `it`: the operands, the unit they are read for, and the K window.
struct StepSrc {
    Operand a, b;
    int unit, k0, kend;
};
__device__ __forceinline__ StepSrc step_src(const GemmArgs &g, const Sched &sc, const Item &it,
                                            int s) {
    StepSrc r;
    if (sc.usum) {
        const int per_unit = sc.terms * sc.ksteps;
        const int i = it.first + s / per_unit, rem = s % per_unit;
        const int term = rem / sc.ksteps;
        r.unit = it.z * sc.ga + i * sc.gb;
        r.k0 = (rem % sc.ksteps) * kTK;
        r.kend = g.K;
        r.a = term ? g.A2 : g.A;
        r.b = term ? g.B2 : g.B;
    } else if (sc.pair) {
        const int term = s / sc.ksteps;
        r.unit = it.z;
        r.k0 = (s % sc.ksteps) * kTK;
        r.kend = g.K;
        r.a = term ? g.A2 : g.A;
        r.b = term ? g.B2 : g.B;
    } else {
        r.unit = it.z;
        r.k0 = it.kbeg + s * kTK;
        r.kend = it.kend;
        r.a = g.A;
        r.b = g.B;
    }
    return r;
}

// The producers' position in the walk: item w (its decoded form) and step s in it.
template <int BN>
struct Cursor {
    long long w;
    int s;
    Item it;
    __device__ __forceinline__ bool valid(const Sched &sc) const { return w < sc.items; }
    // Moves to the next step, skipping items without steps.
    __device__ __forceinline__ void skip_empty(const GemmArgs &g, const Sched &sc) {
        while (w < sc.items && s >= it.nk) {
            w += gridDim.x;
            s = 0;
            if (w < sc.items) it = item_at<BN>(g, sc, w);
        }
    }
    __device__ __forceinline__ void start(const GemmArgs &g, const Sched &sc) {
        w = blockIdx.x;
        s = 0;
        if (w < sc.items) it = item_at<BN>(g, sc, w);
        skip_empty(g, sc);
    }
    __device__ __forceinline__ void next(const GemmArgs &g, const Sched &sc) {
        ++s;
        skip_empty(g, sc);
    }
};

template <int BN>
__device__ __forceinline__ void load_step(Frag<kTM> &fa, Frag<BN> &fb, const GemmArgs &g,
                                          const Sched &sc, const Cursor<BN> &c, int tid) {
    const StepSrc src = step_src(g, sc, c.it, c.s);
    const int L = tc_unit_length(g.pad, src.unit, g.h, g.n);
    frag_load<kTM>(fa, src.a, src.a.mat(src.unit, g.h), c.it.row0, src.k0, g.M, src.kend, L, tid);
    const float *mb = src.b.mat(src.unit, g.h);
    int Lb = L;
    if (src.b.xblk) {
        // the thread's columns lie in one block (x is fixed across its groups): its unit's
        // matrix and length; mb is offset so that mb + k ld + x addresses column x
        const int x = min(c.it.col0 + (tid % Frag<BN>::kRowThreads) * 4, g.N - 1);
        const int blk = x / src.b.xblk;
        mb += blk * src.b.blk_stride - (long long)blk * src.b.xblk;
        Lb = tc_unit_length(g.pad, c.it.z * g.blk_ua + blk * g.blk_ub, g.h, g.n);
    }
    frag_load<BN>(fb, src.b, mb, c.it.col0, src.k0, g.N, src.kend, Lb, tid);
}
// Waits until ring stage step % stages is free, writes the step's split tiles into it
// and marks it full.  False when a wait ran out (or another role gave up).
// The loads stay in flight during the wait; the split follows it.
template <int BN>
__device__ __forceinline__ bool put_step(const Frag<kTM> &fa, const Frag<BN> &fb, int a_mn,
                                         int b_mn, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                         uint32_t &step, int *status, volatile int *abort_flag,
                                         int tid) {
    using C = Cfg<BN>;
    const int s = (int)(step % C::kStages);
    if (step >= (uint32_t)C::kStages &&
        !warp_wait(empty + s, ((step / C::kStages) - 1) & 1, status, 32, abort_flag))
        return false;
    Split<kTM> sa;
    Split<BN> sb;
    split_frag<kTM>(fa, sa);
    split_frag<BN>(fb, sb);
    uint8_t *st = ring + s * C::kStage;
    store_split<kTM>(sa, a_mn, st, st + C::kA, tid);
    store_split<BN>(sb, b_mn, st + 2 * C::kA, st + 2 * C::kA + C::kB, tid);
    fence_proxy_async_smem();
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(full + s);  // one arrival per producer warp
    ++step;
    return true;
}

constexpr float kLog2e = 1.4426950408889634f;

// The warp's output of one 32-column chunk of rows r0 .. r0 + 31 (lane l holds row
// r0 + l in val): each lane writes its row into the warp's staging rows (kStagePitch
// floats apart: a quarter-warp's 16-byte stores or loads fall in distinct banks), then
// each store instruction writes four whole 128-byte row pieces, eight lanes a row.
// chunk points at row 0 of the chunk's first column (row stride ld); rows >= M and
// columns >= ncols are not written; `vec`: 16-byte stores (16-byte-aligned rows).
__device__ __forceinline__ void emit_rows32(const float (&val)[32], float *chunk, long long ld,
                                            int r0, int ncols, int M, float *stg, int lane,
                                            bool vec) {
    float4 *mine = reinterpret_cast<float4 *>(stg + lane * kStagePitch);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        mine[j] = make_float4(val[4 * j], val[4 * j + 1], val[4 * j + 2], val[4 * j + 3]);
    __syncwarp();
    const int cc = (lane & 7) * 4;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int rr = 4 * t + (lane >> 3), gr = r0 + rr;
        const float4 x = reinterpret_cast<const float4 *>(stg + rr * kStagePitch)[lane & 7];
        if (gr < M && cc < ncols) {
            float *dst = chunk + (long long)gr * ld + cc;
            if (vec && cc + 4 <= ncols) {
                *reinterpret_cast<float4 *>(dst) = x;
            } else {
                dst[0] = x.x;
                if (cc + 1 < ncols) dst[1] = x.y;
                if (cc + 2 < ncols) dst[2] = x.z;
                if (cc + 3 < ncols) dst[3] = x.w;
            }
        }
    }
    __syncwarp();
}

// Epilogue of one tile by warp q: lane l owns row r0 + l (r0 = row0 + 32 q, TMEM lane
// 32 q + l) and reads the accumulator of TMEM columns taddr .., 32 at a time; stg is
// the warp's 32 staging rows.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmArgs &g, const Sched &sc, const Item &it,
                                              uint32_t taddr, float *stg, int q, int lane) {
    const int r0 = it.row0 + q * 32, row = r0 + lane;
    const bool acc = it.nk > 0;  // no product: the accumulator reads as zero
    const bool row_ok = row < g.M;
    auto fetch = [&](int c, uint32_t (&v)[32]) {
        if (acc) {
            tmem_ld32(taddr + (uint32_t)c, v);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
    };
    if (g.epi == kEpiPlain) {
        const int L = sc.usum ? g.n : tc_unit_length(g.pad, it.z, g.h, g.n);
        const bool part = g.splits > 1;
        const bool blocks = !part && g.cblk > 0;
        float *out = part ? g.part + ((long long)it.split * sc.zcount + it.z) * g.M * g.N
                          : g.C + (long long)it.z * g.sC;
        const int ld = part ? g.N : g.ldc;
        const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0 && (ld & 3) == 0 &&
                         (!blocks || (g.cblk_stride & 3) == 0);
        const bool beta = !part && g.beta != 0.f;
        for (int c = 0; c < BN && it.col0 + c < g.N; c += 32) {
            uint32_t v[32];
            fetch(c, v);
            const int gc = it.col0 + c;
            // the chunk's place in C, its first column within its block and its length
            float *chunk = out + gc;
            int cb = gc, Lc = L;
            if (blocks) {
                const int blk = gc / g.cblk;
                cb = gc - blk * g.cblk;
                chunk = out + blk * g.cblk_stride + cb;
                Lc = tc_unit_length(g.pad, it.z * g.blk_ua + blk * g.blk_ub, g.h, g.n);
            }
            float val[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) val[i] = g.alpha * __uint_as_float(v[i]);
            if (beta && row_ok) {
                const float *cr = chunk + (long long)row * ld;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (gc + i < g.N) val[i] = fmaf(g.beta, cr[i], val[i]);
            }
            if (!part) {
                const bool zero_row = g.mask_rows && row >= Lc;
                if (zero_row || g.mask_cols) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (zero_row || (g.mask_cols && cb + i >= Lc)) val[i] = 0.f;
                }
            }
            emit_rows32(val, chunk, ld, r0, min(32, g.N - gc), g.M, stg, lane, vec);
        }
        return;
    }
    // kEpiSoftmaxPair, whole rows (col0 = 0, N <= BN): S in this accumulator, dP =
    // alpha2 * the next one; p = 2^(a2 s - m) / l with a2 = alpha log2(e), one FFMA and
    // one ex2 a value.  Pass 1: the row maximum of S (alpha > 0, so m = a2 max s).
    // Pass 2: e = 2^(a2 s - m), l = sum e and D' = sum e dP together (the two
    // accumulators' chunks read under one wait).  Pass 3: e again, P = e / l and
    // dS = P (dP - D'/l) written together.
    const int L = tc_unit_length(g.pad, it.z, g.h, g.n);
    const bool live = row < L;
    const int N = g.N;
    float *out = g.C + (long long)it.z * g.sC;
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0 && (g.ldc & 3) == 0;
    const float a2 = g.alpha * kLog2e;
    {
        const uint32_t tdp = taddr + (uint32_t)BN;
        auto fetch_dp = [&](int c, uint32_t (&v)[32]) {
            if (acc) {
                tmem_ld32(tdp + (uint32_t)c, v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
        };
        auto fetch2 = [&](int c, uint32_t (&vs)[32], uint32_t (&vd)[32]) {
            if (acc) {
                tmem_ld32_async(taddr + (uint32_t)c, vs);
                tmem_ld32_async(tdp + (uint32_t)c, vd);
                tmem_wait_ld(vs);
                tie32(vd);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) vs[i] = vd[i] = 0u;
            }
        };
        // columns at or past N: the accumulator holds zeros there (B's rows are zero), so
        // only the maximum and the exponentials need the bound; a whole chunk (the usual
        // case) has none.  Rows at or past the length are written as exact zeros.
        float mx0 = -INFINITY, mx1 = -INFINITY;
        for (int c = 0; c < N; c += 32) {
            uint32_t v[32];
            fetch(c, v);
            const int nv = N - c;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                if (nv >= 32 || i < nv) mx0 = fmaxf(mx0, __uint_as_float(v[i]));
                if (nv >= 32 || i + 1 < nv) mx1 = fmaxf(mx1, __uint_as_float(v[i + 1]));
            }
        }
        const float m = a2 * fmaxf(mx0, mx1);
        float l0 = 0.f, l1 = 0.f, D0 = 0.f, D1 = 0.f;
        for (int c = 0; c < N; c += 32) {
            uint32_t vs[32], vd[32];
            fetch2(c, vs, vd);
            float e[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) e[i] = ex2_approx(fmaf(a2, __uint_as_float(vs[i]), -m));
            if (N - c < 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i >= N - c) e[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                l0 += e[i];
                l1 += e[i + 1];
                D0 = fmaf(e[i], __uint_as_float(vd[i]), D0);
                D1 = fmaf(e[i + 1], __uint_as_float(vd[i + 1]), D1);
            }
        }
        const float inv = 1.f / (l0 + l1);
        const float D = g.alpha2 * inv * (D0 + D1);
        float *out2 = g.C2 + (long long)it.z * g.sC;
        for (int c = 0; c < N; c += 32) {
            float val[32];
            {
                uint32_t vs[32];
                fetch(c, vs);  // warp-wide: outside any branch on the lane's row
                if (live) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        val[i] = ex2_approx(fmaf(a2, __uint_as_float(vs[i]), -m)) * inv;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) val[i] = 0.f;
                }
            }
            emit_rows32(val, out + c, g.ldc, r0, min(32, N - c), g.M, stg, lane, vec);
            uint32_t vd[32];
            fetch_dp(c, vd);
            if (live) {
#pragma unroll
                for (int i = 0; i < 32; ++i) val[i] *= fmaf(g.alpha2, __uint_as_float(vd[i]), -D);
            }
            emit_rows32(val, out2 + c, g.ldc, r0, min(32, N - c), g.M, stg, lane, vec);
        }
        return;
    }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const GemmArgs g, const Sched sc) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *transpose = reinterpret_cast<float *>(ring + C::kRing);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + C::kRing + C::kTranspose);
    uint64_t *empty = full + C::kStages;
    uint64_t *acc_full = empty + C::kStages;  // [2]
    uint64_t *acc_empty = acc_full + 2;       // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full + s, kProducerWarps);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int a_mn = g.A.xfast, b_mn = g.B.xfast;

    if (warp < kProducerWarps) {
        // ---- producers: global fp32 -> split bf16 hi / lo -> ring stage
        uint32_t step = 0;
        Cursor<BN> cur;
        cur.start(g, sc);
        while (cur.valid(sc)) {
            Frag<kTM> fa;
            Frag<BN> fb;
            load_step<BN>(fa, fb, g, sc, cur, tid);
            if (!put_step<BN>(fa, fb, a_mn, b_mn, ring, full, empty, step, g.status, abort_flag, tid))
                break;
            cur.next(g, sc);
        }
    } else if (warp < kMmaWarp) {
        // ---- epilogue: TMEM accumulator -> C (or the split's partial)
        const int q = warp & 3;
        float *stg = transpose + q * 32 * kStagePitch;
        // two accumulators alternate between tiles, or (pair) serve one tile together
        const int bufs = sc.pair ? 1 : 2;
        int tcount = 0;
        for (long long w = blockIdx.x; w < sc.items; w += gridDim.x, ++tcount) {
            const Item it = item_at<BN>(g, sc, w);
            const int b = tcount % bufs, use = tcount / bufs;
            if (!warp_wait(acc_full + b, use & 1, g.status, 33, abort_flag)) break;
            tc_fence_after();
            if (*abort_flag) break;
            epilogue_tile<BN>(g, sc, it, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN), stg,
                              q, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + b);  // one arrival per epilogue warp
        }
    } else if (lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = idesc_f16(kTM, BN, 1, a_mn, b_mn);
        const uint64_t sa = slice_step(a_mn), sb = slice_step(b_mn);
        uint32_t step = 0;
        const int bufs = sc.pair ? 1 : 2;
        int tcount = 0;
        bool ok = true;
        for (long long w = blockIdx.x; ok && w < sc.items; w += gridDim.x, ++tcount) {
            const Item it = item_at<BN>(g, sc, w);
            const int b = tcount % bufs, use = tcount / bufs;
            if (use >= 1) ok = mbar_wait(acc_empty + b, (use - 1) & 1, g.status, 34, abort_flag);
            if (!ok) break;
            tc_fence_after();
            for (int s = 0; s < it.nk; ++s, ++step) {
                // pair: the first product's steps into accumulator 0, the second's into 1
                const int term = sc.pair ? s / sc.ksteps : 0, ks = sc.pair ? s % sc.ksteps : s;
                const uint32_t d = tmem + (uint32_t)((sc.pair ? term : b) * BN);
                const int st = (int)(step % C::kStages);
                ok = mbar_wait(full + st, (step / C::kStages) & 1, g.status, 31, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint8_t *base = ring + st * C::kStage;
                const uint64_t ah = tile_desc(base, a_mn), al = tile_desc(base + C::kA, a_mn);
                const uint64_t bh = tile_desc(base + 2 * C::kA, b_mn),
                               bl = tile_desc(base + 2 * C::kA + C::kB, b_mn);
#pragma unroll
                for (int k = 0; k < kTK / 16; ++k) {
                    mma_ss(d, ah + k * sa, bh + k * sb, idesc, (ks > 0 || k > 0) ? 1u : 0u);
                    mma_ss(d, ah + k * sa, bl + k * sb, idesc, 1u);
                    mma_ss(d, al + k * sa, bh + k * sb, idesc, 1u);
                }
                mma_commit(empty + st);
            }
            if (!ok) break;
            if (it.nk > 0) mma_commit(acc_full + b);
            else mbar_arrive(acc_full + b);
        }
        // every product issued has finished before TMEM is released
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int BN>
int launch_tc_gemm(const GemmArgs &g, const Sched &sc, int sms, cudaStream_t s, int kernel_id) {
    using C = Cfg<BN>;
    static_assert(C::kSmem <= 227 * 1024, "shared memory of one CTA");
    if (sc.items <= 0) return LINFORMER_OK;
    const long long grid = std::min<long long>(sc.items, sms);
    if (cudaFuncSetAttribute(tc_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmem) != cudaSuccess)
        return LINFORMER_ERR_LAUNCH;
    {
        KernelScope scope(kernel_id, s);
        tc_gemm_kernel<BN><<<(unsigned)grid, kThreads, C::kSmem, s>>>(g, sc);
    }
    if (cudaPeekAtLastError() != cudaSuccess) return LINFORMER_ERR_LAUNCH;
    if (g.splits > 1) return launch_splitk_reduce(g, sc.zcount, s, kernel_id);
    return LINFORMER_OK;
}

// ------------------------------------------------------------------ the pair kernel
// kEpiSoftmaxPair specialised for d <= 64 with 16-byte-aligned K-major operands (the
// backward's Q, dO, Kbar and Vbar): a CTA walks a contiguous range of row tiles, so
// consecutive tiles share their unit and its Kbar and Vbar (B operands, N x 64 each)
// stay in shared memory, split once per unit; the producers only read each tile's Q and
// dO.  That frees four producer warps for the epilogue, which the pair item is bound by:
// eight epilogue warps, two per TMEM lane quarter, each taking 128 of the 256 columns of
// its 32 rows and exchanging the row maximum, sum and sum e dP with its partner through
// shared memory.  S and dP fill the 512 TMEM columns, so a tile's products wait for the
// previous tile's epilogue to have read them.
constexpr int kPairProducerWarps = 4;
constexpr int kPairEpiWarp0 = 4;  // warps 4..11: lane quarter w % 4, column half (w - 4) / 4
constexpr int kPairMmaWarp = 12;
constexpr int kPairThreads = (kPairMmaWarp + 1) * 32;  // 416
constexpr uint32_t kPairImg = 256 * 128;               // a 256-row K-major bf16 tile (32 KB)
constexpr uint32_t kPairTile = kTM * 128;              // a 128-row tile (16 KB)
constexpr uint32_t kPairStg = 32 * 32 * 4;             // a warp's staging rows (swizzled)
constexpr size_t kPairSmem = 1024 + 4 * kPairImg + 4 * kPairTile + 8 * kPairStg + 256;
static_assert(kPairSmem <= 227 * 1024, "shared memory of one CTA");
static_assert(kPairEpiWarp0 % 4 == 0, "epilogue warp w reads TMEM lanes 32 (w % 4) ..");

// Rows x0 .. x0 + 8 nb of a row-major fp32 matrix m (row stride ld; rows >= X, and rows
// >= L when masked, read as zero; the K <= 64 valid columns, K % 4 == 0), split into hi
// and lo K-major tiles (128-byte rows, swizzled) by the 128 producer threads: thread t
// takes columns 4 (t % 16) .. of rows t / 16 + 8 j, eight rows' loads in flight at once.
__device__ __forceinline__ void pair_load_rows(const float *m, long long ld, int x0, int nb, int X,
                                               int K, int L, bool mask, uint8_t *hi, uint8_t *lo,
                                               int tid) {
    const int kc = (tid % 16) * 4;
    const bool kin = kc < K;
#pragma unroll 1
    for (int b0 = 0; b0 < nb; b0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = tid / 16 + 8 * (b0 + j), x = x0 + row;
            const bool in = kin && x < X && !(mask && x >= L);
            v[j] = in ? __ldg(reinterpret_cast<const float4 *>(m + (long long)x * ld + kc))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = tid / 16 + 8 * (b0 + j);
            uint2 h, l;
            split4(v[j], h, l);
            const uint32_t off = kmajor_off(row, kc);
            *reinterpret_cast<uint2 *>(hi + off) = h;
            *reinterpret_cast<uint2 *>(lo + off) = l;
        }
    }
}

// The warp's output of one 32-column chunk of rows r0 .. r0 + 31 (lane l holds row r0 + l):
// each lane writes its row into the warp's staging rows (128 bytes a row, 16-byte piece
// j of row r at position j ^ (r % 8): a quarter-warp's accesses fall in distinct banks),
// then each store instruction writes four whole 128-byte row pieces.  Rows >= M and
// columns >= ncols are not written.
__device__ __forceinline__ void pair_emit(const float (&val)[32], float *chunk, long long ld,
                                          int r0, int ncols, int M, float4 *stg, int lane) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        stg[lane * 8 + (j ^ (lane & 7))] =
            make_float4(val[4 * j], val[4 * j + 1], val[4 * j + 2], val[4 * j + 3]);
    __syncwarp();
    const int cc = (lane & 7) * 4;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int rr = 4 * t + (lane >> 3), gr = r0 + rr;
        const float4 x = stg[rr * 8 + ((lane & 7) ^ (rr & 7))];
        if (gr < M && cc < ncols) {
            float *dst = chunk + (long long)gr * ld + cc;
            if (cc + 4 <= ncols) {
                *reinterpret_cast<float4 *>(dst) = x;
            } else {
                dst[0] = x.x;
                if (cc + 1 < ncols) dst[1] = x.y;
                if (cc + 2 < ncols) dst[2] = x.z;
            }
        }
    }
    __syncwarp();
}

// Named barrier of epilogue warps 4 + q and 8 + q (literal ids 1..4), and the same
// barrier returning whether v held in every thread of both warps (the pair leaves its
// loop together, so that neither waits at the barrier for one that has left).
__device__ __forceinline__ void pair_sync(int q) {
    switch (q) {
        case 0: named_barrier_sync(1, 64); break;
        case 1: named_barrier_sync(2, 64); break;
        case 2: named_barrier_sync(3, 64); break;
        default: named_barrier_sync(4, 64); break;
    }
}
__device__ __forceinline__ bool pair_and(int q, bool v) {
    switch (q) {
        case 0: return named_barrier_and(1, 64, v);
        case 1: return named_barrier_and(2, 64, v);
        case 2: return named_barrier_and(3, 64, v);
        default: return named_barrier_and(4, 64, v);
    }
}

__global__ void __launch_bounds__(kPairThreads, 1) tc_pair_kernel(const GemmArgs g, int tiles_m,
                                                                   long long tiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *img = base;                                   // Kbar hi, lo, Vbar hi, lo
    uint8_t *ring = base + 4 * kPairImg;                   // Q hi, lo, dO hi, lo
    float4 *stg_all = reinterpret_cast<float4 *>(ring + 4 * kPairTile);
    uint64_t *a_full = reinterpret_cast<uint64_t *>(ring + 4 * kPairTile + 8 * kPairStg);  // [2]
    uint64_t *a_empty = a_full + 2;    // [2]
    uint64_t *b_full = a_empty + 2, *b_empty = b_full + 1;
    uint64_t *acc_full = b_empty + 1, *acc_empty = acc_full + 1, *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's row tiles [t0, t1): unit t / tiles_m, tile t % tiles_m
    const long long t0 = tiles * blockIdx.x / gridDim.x, t1 = tiles * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(a_full + i, kPairProducerWarps);
            mbar_init(a_empty + i, 1);
        }
        mbar_init(b_full, kPairProducerWarps);
        mbar_init(b_empty, 1);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kPairMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kPairProducerWarps) {
        // ---- producers: each unit's Kbar and Vbar once, each tile's Q and dO
        int ub = 0, cur_z = -1;
        bool ok = true;
        for (long long t = t0; ok && t < t1; ++t) {
            const int i = (int)(t - t0), z = (int)(t / tiles_m), mt = (int)(t % tiles_m);
            if (z != cur_z) {
                if (ub >= 1 && !warp_wait(b_empty, (ub - 1) & 1, g.status, 36, abort_flag)) break;
                pair_load_rows(g.B.mat(z, g.h), g.B.ld, 0, 32, g.N, g.K, 0, false, img, img + kPairImg, tid);
                pair_load_rows(g.B2.mat(z, g.h), g.B2.ld, 0, 32, g.N, g.K, 0, false, img + 2 * kPairImg,
                               img + 3 * kPairImg, tid);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_full);
                ++ub;
                cur_z = z;
            }
            const int L = tc_unit_length(g.pad, z, g.h, g.n);
#pragma unroll 1
            for (int term = 0; term < 2; ++term) {
                if (i >= 1 && !warp_wait(a_empty + term, (i - 1) & 1, g.status, 32, abort_flag)) {
                    ok = false;
                    break;
                }
                const Operand o = term ? g.A2 : g.A;
                uint8_t *st = ring + term * 2 * kPairTile;
                pair_load_rows(o.mat(z, g.h), o.ld, mt * kTM, 16, g.M, g.K, L, o.mask_x != 0, st,
                               st + kPairTile, tid);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full + term);
            }
        }
    } else if (warp < kPairMmaWarp) {
        // ---- epilogue: warp (q, hc) owns rows 32 q .. of the tile and columns 128 hc ..
        const int q = warp & 3, hc = (warp - kPairEpiWarp0) >> 2;
        float4 *stg = stg_all + (warp - kPairEpiWarp0) * (kPairStg / 16);
        const float *xchg = reinterpret_cast<const float *>(stg_all + ((warp - kPairEpiWarp0) ^ 4) * (kPairStg / 16));
        float *mine = reinterpret_cast<float *>(stg);
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const int cbeg = 128 * hc, nloc = max(0, min(128, g.N - cbeg));
        const float a2 = g.alpha * kLog2e;
        for (long long t = t0; t < t1; ++t) {
            const int i = (int)(t - t0), z = (int)(t / tiles_m), mt = (int)(t % tiles_m);
            bool ok = warp_wait(acc_full, i & 1, g.status, 33, abort_flag);
            tc_fence_after();
            if (!pair_and(q, ok && *abort_flag == 0)) break;
            const int r0 = mt * kTM + q * 32, row = r0 + lane;
            const bool live = row < tc_unit_length(g.pad, z, g.h, g.n);
            const uint32_t ts = tmem + lanes + (uint32_t)cbeg, td = ts + 256u;
            // pass 1: the row maximum of S over both column halves
            float mx0 = -INFINITY, mx1 = -INFINITY;
            for (int c = 0; c < nloc; c += 32) {
                uint32_t v[32];
                tmem_ld32(ts + (uint32_t)c, v);
                const int nv = nloc - c;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    if (nv >= 32 || e < nv) mx0 = fmaxf(mx0, __uint_as_float(v[e]));
                    if (nv >= 32 || e + 1 < nv) mx1 = fmaxf(mx1, __uint_as_float(v[e + 1]));
                }
            }
            mine[lane] = fmaxf(mx0, mx1);
            pair_sync(q);
            const float m = a2 * fmaxf(mine[lane], xchg[lane]);
            // pass 2: e = 2^(a2 s - m), its sum and sum e dP, both halves
            float l0 = 0.f, l1 = 0.f, D0 = 0.f, D1 = 0.f;
            for (int c = 0; c < nloc; c += 32) {
                uint32_t vs[32], vd[32];
                tmem_ld32_async(ts + (uint32_t)c, vs);
                tmem_ld32_async(td + (uint32_t)c, vd);
                tmem_wait_ld(vs);
                tie32(vd);
                float e[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) e[j] = ex2_approx(fmaf(a2, __uint_as_float(vs[j]), -m));
                if (nloc - c < 32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j >= nloc - c) e[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    l0 += e[j];
                    l1 += e[j + 1];
                    D0 = fmaf(e[j], __uint_as_float(vd[j]), D0);
                    D1 = fmaf(e[j + 1], __uint_as_float(vd[j + 1]), D1);
                }
            }
            mine[32 + lane] = l0 + l1;
            mine[64 + lane] = D0 + D1;
            pair_sync(q);
            const float inv = 1.f / (mine[32 + lane] + xchg[32 + lane]);
            const float D = g.alpha2 * inv * (mine[64 + lane] + xchg[64 + lane]);
            pair_sync(q);  // the partner has read these before the staging rows are reused
            // pass 3: P and dS of the warp's columns (rows at or past the length: zeros)
            float *outP = g.C + (long long)z * g.sC + cbeg, *outS = g.C2 + (long long)z * g.sC + cbeg;
            for (int c = 0; c < nloc; c += 32) {
                float val[32];
                {
                    uint32_t vs[32];
                    tmem_ld32(ts + (uint32_t)c, vs);
                    if (live) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            val[j] = ex2_approx(fmaf(a2, __uint_as_float(vs[j]), -m)) * inv;
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) val[j] = 0.f;
                    }
                }
                pair_emit(val, outP + c, g.ldc, r0, min(32, nloc - c), g.M, stg, lane);
                uint32_t vd[32];
                tmem_ld32(td + (uint32_t)c, vd);
                if (live) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) val[j] *= fmaf(g.alpha2, __uint_as_float(vd[j]), -D);
                }
                pair_emit(val, outS + c, g.ldc, r0, min(32, nloc - c), g.M, stg, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);  // one arrival per epilogue warp
        }
    } else if (lane == 0) {
        // ---- MMA issuer: S = alpha Q Kbar^T into columns 0.., dP = dO Vbar^T into 256..
        const int nmma = (g.N + 31) / 32 * 32;
        const uint32_t idesc = idesc_f16(kTM, nmma, 1, 0, 0);
        int ub = 0, cur_z = -1;
        bool ok = true;
        for (long long t = t0; ok && t < t1; ++t) {
            const int i = (int)(t - t0), z = (int)(t / tiles_m);
            if (z != cur_z) {
                if (ub >= 1) mma_commit(b_empty);  // the previous unit's products release Kbar, Vbar
                ok = mbar_wait(b_full, ub & 1, g.status, 35, abort_flag);
                if (!ok) break;
                ++ub;
                cur_z = z;
            }
            if (i >= 1) ok = mbar_wait(acc_empty, (i - 1) & 1, g.status, 34, abort_flag);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int term = 0; term < 2; ++term) {
                ok = mbar_wait(a_full + term, i & 1, g.status, 31, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint8_t *st = ring + term * 2 * kPairTile, *bt = img + term * 2 * kPairImg;
                const uint64_t ah = tile_desc(st, 0), al = tile_desc(st + kPairTile, 0);
                const uint64_t bh = tile_desc(bt, 0), bl = tile_desc(bt + kPairImg, 0);
                const uint32_t d = tmem + (uint32_t)(term * 256);
#pragma unroll
                for (int k = 0; k < kTK / 16; ++k) {
                    mma_ss(d, ah + 2 * k, bh + 2 * k, idesc, k > 0 ? 1u : 0u);
                    mma_ss(d, ah + 2 * k, bl + 2 * k, idesc, 1u);
                    mma_ss(d, al + 2 * k, bh + 2 * k, idesc, 1u);
                }
                mma_commit(a_empty + term);
            }
            if (!ok) break;
            mma_commit(acc_full);
        }
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPairMmaWarp) tmem_dealloc(tmem, 512);
}

// Whether the pair kernel serves this kEpiSoftmaxPair product: d <= 64 (one 64-deep
// step), K-major operands whose rows are 16-byte groups, outputs whose rows are too.
bool pair_kernel_fits(const GemmArgs &g) {
    auto kmajor_vec = [](const Operand &o) { return !o.xfast && o.vec && !o.mask_k; };
    return g.K <= kTK && g.K % 4 == 0 && g.N % 4 == 0 && g.N <= 256 && kmajor_vec(g.A) &&
           kmajor_vec(g.B) && kmajor_vec(g.A2) && kmajor_vec(g.B2) && !g.B.mask_x &&
           !g.B2.mask_x && (reinterpret_cast<uintptr_t>(g.C) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(g.C2) & 15) == 0 && g.ldc % 4 == 0 && g.sC % 4 == 0;
}

int launch_pair(const GemmArgs &g, int units, int sms, cudaStream_t s, int kernel_id) {
    const int tiles_m = (g.M + kTM - 1) / kTM;
    const long long tiles = (long long)tiles_m * units;
    if (tiles <= 0) return LINFORMER_OK;
    const long long grid = std::min<long long>(tiles, sms);
    if (cudaFuncSetAttribute(tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPairSmem) != cudaSuccess)
        return LINFORMER_ERR_LAUNCH;
    {
        KernelScope scope(kernel_id, s);
        tc_pair_kernel<<<(unsigned)grid, kPairThreads, kPairSmem, s>>>(g, tiles_m, tiles);
    }
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace

int tc_batched_gemm(GemmArgs g, int units, cudaStream_t s, float *part, size_t part_floats,
                    int sms, int kernel_id) {
    if (g.M <= 0 || g.N <= 0 || units <= 0) return LINFORMER_OK;
    if (sms <= 0) sms = sm_count();
    set_operand_vec(g.A, g.A.xfast ? g.M : g.K);
    set_operand_vec(g.B, g.B.xfast ? g.N : g.K);
    const bool usum = g.usum_groups > 0, two = usum && g.A2.p != nullptr;
    if (two) {
        if (g.A2.xfast != g.A.xfast || g.B2.xfast != g.B.xfast) return LINFORMER_ERR_SIZE;
        set_operand_vec(g.A2, g.A2.xfast ? g.M : g.K);
        set_operand_vec(g.B2, g.B2.xfast ? g.N : g.K);
    }
    if (g.B.xblk || g.cblk || g.A.xblk) {
        // column blocks: B x-contiguous in blocks of a multiple of 32 columns, C blocked
        // alike, the length masks only on B's sequence axis and C's rows
        if (g.A.xblk || !g.B.xfast || g.B.xblk <= 0 || g.B.xblk % 32 || g.cblk != g.B.xblk ||
            g.B.mask_x || g.A.mask_x || g.A.mask_k || g.mask_cols || usum || g.epi != kEpiPlain)
            return LINFORMER_ERR_SIZE;
        if (g.B.blk_stride & 3) g.B.vec = 0;
    }
    const int BN = g.N <= 64 ? 64 : (g.N <= 128 ? 128 : 256);
    const bool pair = g.epi == kEpiSoftmaxPair;
    if (g.epi != kEpiPlain && (g.epi != kEpiSoftmaxPair || g.N > BN || usum))
        return LINFORMER_ERR_SIZE;
    if (pair) {
        if (!g.A2.p || !g.B2.p || !g.C2 || g.A2.xfast != g.A.xfast || g.B2.xfast != g.B.xfast ||
            !(g.alpha > 0.f))
            return LINFORMER_ERR_SIZE;
        set_operand_vec(g.A2, g.A2.xfast ? g.M : g.K);
        set_operand_vec(g.B2, g.B2.xfast ? g.N : g.K);
        if (pair_kernel_fits(g)) {
            g.status = device_status_ptr();
            return launch_pair(g, units, sms, s, kernel_id);
        }
    }
    Sched sc{};
    sc.tiles_m = (g.M + kTM - 1) / kTM;
    sc.tiles_n = (g.N + BN - 1) / BN;
    sc.ksteps = (g.K + kTK - 1) / kTK;
    sc.usum = usum ? 1 : 0;
    sc.zcount = usum ? g.usum_groups : units;
    sc.terms = two ? 2 : 1;
    sc.pair = pair ? 1 : 0;
    sc.per_group = g.usum_per_group;
    sc.ga = g.usum_ga;
    sc.gb = g.usum_gb;
    g.splits = 1;
    g.kchunk = sc.ksteps * kTK;
    g.part = part;
    g.status = device_status_ptr();
    const long long tiles = (long long)sc.tiles_m * sc.tiles_n * sc.zcount;
    const long long out_floats = (long long)sc.zcount * g.M * g.N;
    // Splits (or unit chunks) for about four work items per SM, as far as the partials
    // fit in `part`; a split is at least four steps deep.
    long long want = 1;
    if (g.epi == kEpiPlain && part && tiles < 4LL * sms) {
        want = (4LL * sms + tiles - 1) / tiles;
        want = std::min<long long>(want, (long long)(part_floats / (size_t)out_floats));
        if (usum)
            want = std::min<long long>(want, sc.per_group);
        else
            want = std::min<long long>(want, std::max(1, sc.ksteps / 4));
        want = std::max<long long>(want, 1);
    }
    if (usum) {
        sc.uc = (int)((sc.per_group + want - 1) / want);
        g.splits = sc.uc > 0 ? (sc.per_group + sc.uc - 1) / sc.uc : 1;
    } else if (want > 1) {
        const int steps = (int)((sc.ksteps + want - 1) / want);
        g.kchunk = steps * kTK;
        g.splits = (sc.ksteps + steps - 1) / steps;
    }
    sc.splits = g.splits;
    sc.items = tiles * sc.splits;
    if (BN == 64) return launch_tc_gemm<64>(g, sc, sms, s, kernel_id);
    if (BN == 128) return launch_tc_gemm<128>(g, sc, sms, s, kernel_id);
    return launch_tc_gemm<256>(g, sc, sms, s, kernel_id);
}

}  // namespace simt
}  // namespace linformer
