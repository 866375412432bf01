// Projection step on the tensor cores: Kbar = Ehat . K and Vbar = Fhat . V
// ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// E, F are k x n, row j of E merges the n positions into compressed position j;
// padded rows t >= L count as zero, section Model, padding paragraph).
//
// One CTA owns one (unit, sequence chunk) pair, or two unsplit units of the same
// sharing group (E = F, no lengths).  Per 64-row stage three warps TMA-load the E
// (and F) tile, k_pad x 64, K-major, in one box, and each unit's K and V tiles,
// 64 x 64 each, whose d axis is contiguous (MN-major operand).  One thread issues
// tcgen05.mma into TMEM: with E = F a single product of N = 128 per unit covers K
// and V (the E tile is read once for all of them); with E != F two N = 64 products.
// Accumulators: M-half mh (rows 128 mh ..) at TMEM columns [128 u mh, ..) for u
// units, per unit 64 Kbar columns then 64 Vbar columns.  The epilogue turns them into
// the images the attention step reads, with four warps, or with eight (Kbar and Vbar
// in parallel) when the launch runs one CTA per SM.
//
// Chunks of the same unit are summed in a fixed order, so the result does not depend
// on scheduling: in groups of chunks (chunk order) by the last CTA of each group to
// arrive, then the groups' sums (group order) by the last group to arrive (one level
// below 9 chunks).  Those CTAs pull the other sums in as 32 KB slices by bulk copy; the
// last one converts to the split images the attention step reads and picks the number
// of P.Vbar products from max|Vbar|.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

namespace linformer {
namespace tc {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kSlice = 64 * 128;  // floats in one 64-column half of a 128-row block

__device__ __forceinline__ int valid_length(const int32_t *pad, int batch, int n) {
    if (!pad) return n;
    const int L = pad[batch];
    return L < 0 ? 0 : (L > n ? n : L);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 16-byte chunk q (0..7) of row j inside a 128-byte-swizzled image.
__device__ __forceinline__ uint4 *image_chunk(uint8_t *img, int j, int q) {
    return reinterpret_cast<uint4 *>(img + (size_t)j * kRowBytes + ((q ^ (j & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// kOut: also write Kbar and Vbar in fp32 (the projection entry point).  The forward
// pass launches the variant without that code, whose epilogue is much smaller: its
// first execution on every SM at once is a wave of instruction fetches.
template <bool kOut>
__global__ void __launch_bounds__(2 * kThreads, 1)
    tc_project_kernel(const __grid_constant__ CUtensorMap tE, const __grid_constant__ CUtensorMap tF,
                      const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
                      const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (group g, chunk c, slot); members of a group share E (and F).  Slots
    // below p.pairs take members 2 slot and 2 slot + 1 (one E tile per stage for
    // both; only unsplit units, E = F, no lengths), the others one member each.
    const int bid = blockIdx.x;
    const int per_group = p.members - p.pairs;
    const int slot = bid % per_group;
    const int gc = bid / per_group;
    const int c = gc % p.C;
    const int g = gc / p.C;
    const int nunits = slot < p.pairs ? 2 : 1;
    const int m = slot < p.pairs ? 2 * slot : slot + p.pairs;
    const int u = p.per_head ? m * p.h + g : m;
    // the second unit of a pair (the next member of the same group)
    const int u_b = p.per_head ? (m + 1) * p.h + g : m + 1;
    const int gproj = p.per_head ? g : 0;

    // Launched as a programmatic dependent of the previous kernel in the stream (the
    // previous forward's attention, say, which reads this workspace): nothing is read
    // or written before that grid has completed.  Only L2 prefetches of this CTA's
    // first stages of K, V and E go out before the wait, as if every row were valid
    // (the lengths may not be read yet): a prefetch reads nothing into the CTA, and L2
    // is where every write lands, so what the main loop later reads cannot be stale.
    // Then this forward's attention kernel may take SMs as this grid's CTAs leave; it
    // waits for the whole grid before it reads anything written here.
    if (tid == 0) {
        // the ring, the main loop's own prefetch distance and, without lengths, four more
        // (measured at the headline: 0, 6, 10, 16, 24 stages gave 148.0, 145.2, 144.2,
        // 145.0, 147.6 us; with lengths the rows may be padding, and the ragged per-head
        // workload took 373.6 us with the first two terms and 379.0 with four more)
        const int early = (nunits == 2 ? p.stages2 : p.stages) + p.prefetch + (p.pad ? 0 : 4);
        const int nmax = (min(p.CH, p.n - c * p.CH) + kBK - 1) / kBK;
        for (int j = 0; j < early && j < nmax; ++j) {
            const int x = c * p.CH + j * kBK;
            tma_prefetch_3d(&tK, 0, x, u);
            tma_prefetch_3d(&tV, 0, x, u);
            if (nunits == 2) {
                tma_prefetch_3d(&tK, 0, x, u_b);
                tma_prefetch_3d(&tV, 0, x, u_b);
            }
            tma_prefetch_3d(&tE, x, 0, gproj);
            if (p.distinct) tma_prefetch_3d(&tF, x, 0, gproj);
        }
    }
    wait_prerequisites();
    if (tid == 0) launch_dependents();
    const int L = valid_length(p.pad, u / p.h, p.n);
    const int Cu = L > 0 ? (L + p.CH - 1) / p.CH : 1;
    if (c >= Cu) return;  // chunk entirely in the padding: nothing to add
    const int row0 = c * p.CH;
    const int rows = max(0, min(p.CH, L - row0));
    const int nkb = (rows + kBK - 1) / kBK;

    // Stage: the E (and F) tile, then K and V tiles of 8 KB per unit, in the order
    // K_0 V_0 K_1 V_1 (one operand of 64-column atoms 8 KB apart).
    const uint32_t a_bytes = (uint32_t)p.mhalves * 16384u;
    const uint32_t stage_bytes = a_bytes * (1 + p.distinct) + 16384u * (uint32_t)nunits;
    const int S = nunits == 2 ? p.stages2 : p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *fin = acc_full + 1;  // three slice buffers of the split reduction
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    float *red = reinterpret_cast<float *>(tmem_slot + 4);
    // TMEM: M-half mh at columns [128 nunits mh, ..): per unit 64 Kbar then 64 Vbar columns.
    const uint32_t ncols = (uint32_t)(p.mhalves * nunits) * 128u;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 3);  // the E/F, K and V loaders
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        for (int i = 0; i < 3; ++i) mbar_init(fin + i, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tE);
        prefetch_tmap(&tF);
        prefetch_tmap(&tK);
        prefetch_tmap(&tV);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 2 || warp == 3) {
        // ---------------- TMA loads, one kind per warp: copies issued by one thread
        // are handled one after another, so the E (and F) tile (one k_pad-row box)
        // comes from warp 0, the K tile from warp 2 and the V tile from warp 3, each
        // arming its own bytes on the stage barrier.
        if (lane == 0) {
            // Tiles of stage j fetched into L2 only, p.prefetch stages beyond the ring.
            auto prefetch = [&](int j) {
                if (j >= nkb) return;
                const int x = row0 + j * kBK;
                if (warp == 0) {
                    if (!p.prefetch_proj) return;
                    tma_prefetch_3d(&tE, x, 0, gproj);
                    if (p.distinct) tma_prefetch_3d(&tF, x, 0, gproj);
                } else {
                    tma_prefetch_3d(warp == 2 ? &tK : &tV, 0, x, u);
                    if (nunits == 2) tma_prefetch_3d(warp == 2 ? &tK : &tV, 0, x, u_b);
                }
            };
            for (int j = S; j < S + p.prefetch; ++j) prefetch(j);
            int issued = 0;
            for (int it = 0; it < nkb; ++it) {
                const int s = it % S;
                if (it >= S && !mbar_wait(empty + s, ((it / S) - 1) & 1, p.status, 11, abort_flag))
                    break;
                uint8_t *st = smem + (size_t)s * stage_bytes;
                uint8_t *bk = st + a_bytes * (1 + p.distinct);
                const int x = row0 + it * kBK;
                if (warp == 0) {
                    mbar_arrive_expect_tx(full + s, a_bytes * (1 + p.distinct));
                    tma_load_3d(st, &tE, full + s, x, 0, gproj);
                    if (p.distinct) tma_load_3d(st + a_bytes, &tF, full + s, x, 0, gproj);
                } else {  // warp 2: K tiles at +0 (+16 KB), warp 3: V tiles at +8 KB (+24 KB)
                    const CUtensorMap *map = warp == 2 ? &tK : &tV;
                    uint8_t *dst = bk + (warp == 2 ? 0 : 8192);
                    mbar_arrive_expect_tx(full + s, 8192u * (uint32_t)nunits);
                    tma_load_3d(dst, map, full + s, 0, x, u);
                    if (nunits == 2) tma_load_3d(dst + 16384, map, full + s, 0, x, u_b);
                }
                issued = it + 1;
                if (p.prefetch > 0) prefetch(it + S + p.prefetch);
            }
            // Let every copy this thread started land before the CTA may exit
            // (also after an abort: a copy must not outlive the CTA).
            for (int it = issued > S ? issued - S : 0; it < issued; ++it)
                mbar_wait_drain(full + (it % S), (it / S) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread waits, zeroes rows past the length
        // (only in the last stage of a chunk) and issues; no warp-wide step per stage.
        const uint32_t idesc128 = idesc_f16(128, 128, 1, 0, 1);
        const uint32_t idesc256 = idesc_f16(128, 256, 1, 0, 1);
        const uint32_t idesc64 = idesc_f16(128, 64, 1, 0, 1);
        if (lane == 0) {
            bool ok = true;
            int issued = 0;  // stages whose products were issued
            for (int it = 0; it < nkb; ++it) {
                const int s = it % S;
                if (!mbar_wait(full + s, (it / S) & 1, p.status, 13, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t *st = smem + (size_t)s * stage_bytes;
                uint8_t *bk = st + a_bytes * (1 + p.distinct);
                uint8_t *bv = bk + 8192;
                const int valid = rows - it * kBK;
                if (valid < kBK) {  // rows past the valid length count as zero
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    for (int r = valid; r < kBK; ++r)
                        for (int q = 0; q < 8 * 2 * nunits; ++q)  // K and V tiles of every unit
                            reinterpret_cast<uint4 *>(bk + (q >> 3) * 8192 + r * kRowBytes)[q & 7] = z;
                    fence_proxy_async_smem();
                }
                // Descriptors built once per stage and stepped by adding to the address
                // field (16-byte units): +2 per 16 K-elements of A (32 B), +1024 per
                // 128-row half of A (16 KB), +128 per 16 rows of B (2 KB).
                const uint64_t da = sdesc(smem_u32(st), 16, 1024, kSwizzle128B);
                const bool two = p.mhalves == 2;
                const uint32_t d0 = tmem, d1 = tmem + 128 * nunits;
                if (!p.distinct) {
                    // N = 128 per unit: the unit's K tile, then its V tile (64 columns each).
                    const uint64_t db = sdesc(smem_u32(bk), 8192, 1024, kSwizzle128B);
                    const uint32_t idesc = nunits == 2 ? idesc256 : idesc128;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (it > 0 || ks > 0) ? 1u : 0u;
                        mma_ss(d0, da + 2 * ks, db + 128 * ks, idesc, acc);
                        if (two) mma_ss(d1, da + 1024 + 2 * ks, db + 128 * ks, idesc, acc);
                    }
                } else {
                    const uint64_t df = sdesc(smem_u32(st + a_bytes), 16, 1024, kSwizzle128B);
                    const uint64_t dbk = sdesc(smem_u32(bk), 16, 1024, kSwizzle128B);
                    const uint64_t dbv = sdesc(smem_u32(bv), 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (it > 0 || ks > 0) ? 1u : 0u;
                        mma_ss(d0, da + 2 * ks, dbk + 128 * ks, idesc64, acc);
                        mma_ss(d0 + 64, df + 2 * ks, dbv + 128 * ks, idesc64, acc);
                        if (two) {
                            mma_ss(d1, da + 1024 + 2 * ks, dbk + 128 * ks, idesc64, acc);
                            mma_ss(d1 + 64, df + 1024 + 2 * ks, dbv + 128 * ks, idesc64, acc);
                        }
                    }
                }
                mma_commit(empty + s);
                issued = it + 1;
            }
            // The accumulators are final (or, after an abort, every product issued has
            // finished) when acc_full completes: the epilogue and the TMEM release wait
            // for it.
            if (issued > 0)
                mma_commit(acc_full);
            else
                mbar_arrive(acc_full);
            (void)ok;
        }
        __syncwarp();
    }

    // ---------------- epilogue: thread = TMEM lane = projected row
    mbar_wait(acc_full, 0, p.status, 14, abort_flag);
    tc_fence_after();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    const int jl = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);

    if (blockDim.x == 2 * kThreads) {
        // Eight warps (launched only for unsplit units, E = F): warps 0-3 write the
        // Kbar images while warps 4-7 find max|Vbar| and write the Vbar images.  The
        // accumulators are final in TMEM; rows past k are zero there (so are E's).
        // Each group puts one M-half of its two images (hi and lo, 16 KB each) into
        // shared memory in the images' own layout, and one of its threads copies them
        // out with two bulk stores: whole lines, where a warp's 16-byte stores would
        // touch 32 lines each.  The ring is idle now; each group double-buffers its
        // steps in its own 64 KB of it.
        const bool vgroup = warp >= 4;
        const int gt = tid & 127;              // thread within the group
        // the group's named barrier (literal ids, so that the compiler sees which ones)
        auto gsync = [&]() {
            if (vgroup) named_barrier_sync(3, 128);
            else named_barrier_sync(2, 128);
        };
        int step = 0;                          // M-halves staged by this group so far
        auto claim = [&]() -> uint8_t * {      // staging buffer of this step, once free
            if (gt == 0 && step >= 2) bulk_wait_read1();
            gsync();
            return smem + (vgroup ? 65536 : 0) + 32768 * (step & 1);
        };
        auto flush = [&](uint8_t *stg, uint8_t *img_hi, uint8_t *img_lo, int mh, int rows) {
            fence_proxy_async_smem();
            gsync();
            if (gt == 0) {
                bulk_store(img_hi + (size_t)mh * 16384, stg, (uint32_t)rows * kRowBytes);
                if (img_lo)
                    bulk_store(img_lo + (size_t)mh * 16384, stg + 16384, (uint32_t)rows * kRowBytes);
                bulk_commit();
            }
            ++step;
        };
#pragma unroll 1
        for (int us = 0; us < nunits && !aborted; ++us) {
            const int uu = us ? u_b : u;
            const uint32_t ucol = (uint32_t)us * 128u;
            uint8_t *img = p.images + (size_t)uu * 4 * image_bytes(p.kpad);
            if (!vgroup) {
#pragma unroll 1
                for (int mh = 0; mh < p.mhalves; ++mh) {
                    const int rows = min(128, p.kpad - 128 * mh);
                    uint8_t *stg = claim();
                    // Rolled, 8 columns a step: this code runs once per unit, on every SM
                    // at once and from a cold instruction cache, so its length costs more
                    // than the eight short TMEM round trips.
#pragma unroll 1
                    for (int q = 0; q < 8; ++q) {
                        uint32_t v[8];
                        tmem_ld8(lane_base + mh * 128 * nunits + ucol + 8 * q, v);
                        if (jl < rows) {
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x0 = __uint_as_float(v[2 * e]);
                                const float x1 = __uint_as_float(v[2 * e + 1]);
                                const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                                const float2 hf = __bfloat1622float2(h);  // exact
                                hi[e] = *reinterpret_cast<const uint32_t *>(&h);
                                lo[e] = pack_bf16(x0 - hf.x, x1 - hf.y);
                            }
                            *image_chunk(stg, jl, q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            *image_chunk(stg + 16384, jl, q) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                    flush(stg, img, img + image_bytes(p.kpad), mh, rows);
                }
            } else {
                float vmax = 0.f;
#pragma unroll 1
                for (int mh = 0; mh < p.mhalves; ++mh) {
                    uint32_t v[64];
                    tmem_ld64(lane_base + mh * 128 * nunits + ucol + 64, v);
#pragma unroll
                    for (int i = 0; i < 64; ++i) vmax = fmaxf(vmax, fabsf(__uint_as_float(v[i])));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
                if (lane == 0) red[warp & 3] = vmax;
                named_barrier_sync(1, 128);
                vmax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
                int e = 0;
                while (e < 100 && vmax * exp2f(-(float)e) >= 16384.f) ++e;
                const float vscale = exp2f(-(float)e);
                const int terms = p.forced_terms
                                      ? p.forced_terms
                                      : (vmax < kOneTermMaxV ? 1 : (vmax < kTwoTermMaxV ? 2 : 3));
#pragma unroll 1
                for (int mh = 0; mh < p.mhalves; ++mh) {
                    const int rows = min(128, p.kpad - 128 * mh);
                    uint8_t *stg = claim();
#pragma unroll 1
                    for (int q = 0; q < 8; ++q) {  // rolled, as for Kbar
                        uint32_t v[8];
                        tmem_ld8(lane_base + mh * 128 * nunits + ucol + 64 + 8 * q, v);
                        if (jl < rows) {
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                const float x0 = __uint_as_float(v[2 * e2]) * vscale;
                                const float x1 = __uint_as_float(v[2 * e2 + 1]) * vscale;
                                const __half2 h = __floats2half2_rn(x0, x1);
                                const float2 hf = __half22float2(h);  // exact
                                hi[e2] = *reinterpret_cast<const uint32_t *>(&h);
                                lo[e2] = pack_f16(x0 - hf.x, x1 - hf.y);
                            }
                            *image_chunk(stg, jl, q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            if (terms >= 2)
                                *image_chunk(stg + 16384, jl, q) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                    // Vbar lo is read only by units with two or more P.Vbar products.
                    flush(stg, img + 2 * image_bytes(p.kpad),
                          terms >= 2 ? img + 3 * image_bytes(p.kpad) : nullptr, mh, rows);
                }
                if (jl == 0) p.info[uu] = pack_info(terms, e);
                named_barrier_sync(1, 128);  // red[] is reused by the next unit
            }
        }
        if (gt == 0) bulk_wait0();  // the images are written before the CTA exits
    } else {
    // ---- Split units: the chunk sums are added in a fixed order, in two levels.  Chunk c
    // belongs to group c / G (G = split_group(Cu), chunks in the unit's order); the last CTA
    // of a group to arrive adds the group's chunks in chunk order and leaves the sum in its
    // TMEM; with more than one group it also stores that sum in the slot of the group's
    // first chunk, and the last group to arrive adds the groups' sums in group order.
    // Whichever CTAs arrive last, every sum is formed in the same order, so the result does
    // not depend on scheduling; the longest chain of slices one CTA reads is about
    // 2 sqrt(Cu) chunks instead of Cu - 1.
    // A chunk's sums in the partial buffer: [half of k_pad][column][row] (a warp stores 128
    // contiguous bytes); the other chunks' sums come in as 32 KB slices (one 64-column half
    // of one 128-row block) by bulk copy into three shared buffers (the ring is idle).
    auto store_partial = [&](int slot) {
        float *dst = p.partial + ((size_t)u * p.C + slot) * p.mhalves * 2 * kSlice;
#pragma unroll 1
        for (int mh = 0; mh < p.mhalves; ++mh) {
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tmem_ld32(lane_base + mh * 128 + cc * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    dst[(size_t)mh * 2 * kSlice + (cc * 32 + i) * 128 + jl] = __uint_as_float(v[i]);
            }
        }
    };
    constexpr int kSliceBufs = 3;
    float *sbuf = reinterpret_cast<float *>(smem);
    int sl_issued = 0, sl_used = 0;  // slices started (thread 0's count) and consumed, per CTA
    // Adds, for each M-half and column half, the sums of chunks src(0 .. npos - 1) in that
    // order, position `own` being this CTA's TMEM; the result goes back to TMEM.
    auto reduce = [&](int npos, int own, int first, int stride) -> bool {
        const int per = npos - 1;
        const int nslices = p.mhalves * 2 * per;
        auto slice_src = [&](int idx) {
            const int mh = idx / (2 * per), rem = idx % (2 * per);
            const int half = rem / per, k2 = rem % per;
            const int pos = k2 < own ? k2 : k2 + 1;
            return p.partial + (((size_t)u * p.C + first + pos * stride) * p.mhalves + mh) * 2 * kSlice +
                   half * kSlice;
        };
        const int base = sl_used;  // slice index of this call's first slice
        if (tid == 0) {
            fence_proxy_async_global();
            for (int i = 0; i < kSliceBufs && i < nslices; ++i, ++sl_issued) {
                const int b = sl_issued % kSliceBufs;
                mbar_arrive_expect_tx(fin + b, kSlice * 4);
                bulk_load(sbuf + b * kSlice, slice_src(i), kSlice * 4, fin + b);
            }
        }
        bool ok = true;
#pragma unroll 1
        for (int mh = 0; mh < p.mhalves; ++mh) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const uint32_t tcol = lane_base + mh * 128 + half * 64;
                float acc[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[i] = 0.f;
#pragma unroll 1
                for (int pos = 0; pos < npos; ++pos) {
                    if (pos == own) {
                        uint32_t v[64];
                        tmem_ld64(tcol, v);
#pragma unroll
                        for (int i = 0; i < 64; ++i) acc[i] += __uint_as_float(v[i]);
                        continue;
                    }
                    const int b = sl_used % kSliceBufs;
                    if (!mbar_wait(fin + b, (sl_used / kSliceBufs) & 1, p.status, 15, abort_flag)) ok = false;
                    const float *sb = sbuf + b * kSlice;
#pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] += sb[i * 128 + jl];
                    __syncthreads();
                    const int next = sl_used - base + kSliceBufs;  // this call's slice to start next
                    if (tid == 0 && ok && next < nslices) {
                        mbar_arrive_expect_tx(fin + b, kSlice * 4);
                        bulk_load(sbuf + b * kSlice, slice_src(next), kSlice * 4, fin + b);
                        ++sl_issued;
                    }
                    ++sl_used;
                }
                uint32_t w0[32], w1[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    w0[i] = __float_as_uint(acc[i]);
                    w1[i] = __float_as_uint(acc[32 + i]);
                }
                tmem_st32(tcol, w0);
                tmem_st32(tcol + 32, w1);
            }
        }
        if (tid == 0)  // copies that were started but not consumed (only after an abort)
            for (int i = sl_used; i < sl_issued; ++i)
                mbar_wait_drain(fin + (i % kSliceBufs), (i / kSliceBufs) & 1);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        return ok;
    };
    bool finish = Cu == 1;  // this CTA writes the unit's images
    int *ucnt = p.counters + (size_t)u * kCountersPerUnit;
    if (!aborted && Cu > 1) {
        const int G = split_group(Cu), ng = (Cu + G - 1) / G, gi = c / G;
        const int g0 = gi * G, gn = min(Cu, g0 + G) - g0;
        store_partial(c);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            *last_flag = (atomicAdd(ucnt + 1 + gi, 1) == gn - 1) ? 1 : 0;
            __threadfence();  // the other chunks' stores are seen before their sums are read
        }
        __syncthreads();
        bool last = *last_flag != 0;
        if (last && gn > 1) last = reduce(gn, c - g0, g0, 1);
        if (last && ng == 1) {
            finish = true;
        } else if (last) {
            store_partial(g0);
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                *last_flag = (atomicAdd(ucnt, 1) == ng - 1) ? 1 : 0;
                __threadfence();
            }
            __syncthreads();
            if (*last_flag) finish = reduce(ng, gi, 0, G);
        }
    }

    // Images leave through shared memory: all 128 threads put one M-half of two images
    // (hi and lo, 16 KB each) into one of two 32 KB buffers of the idle ring (the sums are
    // complete by now), in the images' own layout, and thread 0 copies them out with two
    // bulk stores (whole lines rather than 16-byte pieces of 32 rows per store
    // instruction); a buffer is reused once the stores of two steps back have read it.
    int staged = 0;  // bulk groups thread 0 has committed
    auto stage_claim = [&]() -> uint8_t * {
        if (tid == 0 && staged > 1) bulk_wait_read1();
        __syncthreads();
        return smem + 32768 * (staged & 1);
    };
    auto stage_flush = [&](uint8_t *stg, uint8_t *img_hi, uint8_t *img_lo, int mh) {
        const int rows = min(128, p.kpad - 128 * mh);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_store(img_hi + (size_t)mh * 16384, stg, (uint32_t)rows * kRowBytes);
            if (img_lo)
                bulk_store(img_lo + (size_t)mh * 16384, stg + 16384, (uint32_t)rows * kRowBytes);
            bulk_commit();
        }
        ++staged;
    };
    // Images, info word and product count of each unit of the CTA (a pair of units
    // only ever comes unsplit), from the sums in TMEM (rows past k are zero there).
#pragma unroll 1
    for (int us = 0; us < nunits; ++us) {
        if (aborted || !finish || *abort_flag) break;
        const int uu = us ? u_b : u;
        const uint32_t ucol = (uint32_t)us * 128u;  // the unit's columns within an M-half
        uint8_t *img = p.images + (size_t)uu * 4 * image_bytes(p.kpad);
        // Kbar: bf16 hi + bf16 lo images
#pragma unroll 1
        for (int mh = 0; mh < p.mhalves; ++mh) {
            const int j = mh * 128 + jl;
            uint8_t *stg = stage_claim();
            // Rolled, 8 columns a step: this code runs once per unit, on every SM at once
            // and from a cold instruction cache, so its length costs more than the eight
            // short TMEM round trips.
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                uint32_t v[8];
                tmem_ld8(lane_base + mh * 128 * nunits + ucol + 8 * q, v);
                if (j < p.kpad) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x0 = j < p.k ? __uint_as_float(v[2 * e]) : 0.f;
                        const float x1 = j < p.k ? __uint_as_float(v[2 * e + 1]) : 0.f;
                        const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                        const float2 hf = __bfloat1622float2(h);  // exact
                        const float r0 = x0 - hf.x, r1 = x1 - hf.y;
                        hi[e] = *reinterpret_cast<const uint32_t *>(&h);
                        lo[e] = pack_bf16(r0, r1);
                        if (kOut && p.kbar_out && j < p.k) {
                            float *o = p.kbar_out + ((size_t)uu * p.k + j) * kD + q * 8 + 2 * e;
                            o[0] = hf.x + __bfloat162float(__float2bfloat16_rn(r0));
                            o[1] = hf.y + __bfloat162float(__float2bfloat16_rn(r1));
                        }
                    }
                    *image_chunk(stg, jl, q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *image_chunk(stg + 16384, jl, q) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            stage_flush(stg, img, img + image_bytes(p.kpad), mh);
        }
        // Unit-wide max|Vbar| -> scale exponent and number of P.Vbar products.
        float vmax = 0.f;
#pragma unroll 1
        for (int mh = 0; mh < p.mhalves; ++mh) {
            uint32_t v[64];
            tmem_ld64(lane_base + mh * 128 * nunits + ucol + 64, v);
            if (mh * 128 + jl < p.k) {
#pragma unroll
                for (int i = 0; i < 64; ++i) vmax = fmaxf(vmax, fabsf(__uint_as_float(v[i])));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        if (lane == 0) red[warp] = vmax;
        __syncthreads();
        vmax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        int e = 0;
        while (e < 100 && vmax * exp2f(-(float)e) >= 16384.f) ++e;
        const float vscale = exp2f(-(float)e);
        const int terms = p.forced_terms ? p.forced_terms
                                         : (vmax < kOneTermMaxV ? 1 : (vmax < kTwoTermMaxV ? 2 : 3));
#pragma unroll 1
        for (int mh = 0; mh < p.mhalves; ++mh) {
            const int j = mh * 128 + jl;
            uint8_t *stg = stage_claim();
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {  // rolled, as for Kbar
                uint32_t v[8];
                tmem_ld8(lane_base + mh * 128 * nunits + ucol + 64 + 8 * q, v);
                if (j < p.kpad) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const float x0 = j < p.k ? __uint_as_float(v[2 * e2]) * vscale : 0.f;
                        const float x1 = j < p.k ? __uint_as_float(v[2 * e2 + 1]) * vscale : 0.f;
                        const __half2 h = __floats2half2_rn(x0, x1);
                        const float2 hf = __half22float2(h);  // exact
                        const float r0 = x0 - hf.x, r1 = x1 - hf.y;
                        hi[e2] = *reinterpret_cast<const uint32_t *>(&h);
                        lo[e2] = pack_f16(r0, r1);
                        if (kOut && p.vbar_out && j < p.k) {
                            float *o = p.vbar_out + ((size_t)uu * p.k + j) * kD + q * 8 + 2 * e2;
                            o[0] = (hf.x + __half2float(__float2half_rn(r0))) / vscale;
                            o[1] = (hf.y + __half2float(__float2half_rn(r1))) / vscale;
                        }
                    }
                    *image_chunk(stg, jl, q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    if (terms >= 2)
                        *image_chunk(stg + 16384, jl, q) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            // Vbar lo is read only by units with two or more P.Vbar products.
            stage_flush(stg, img + 2 * image_bytes(p.kpad),
                        terms >= 2 ? img + 3 * image_bytes(p.kpad) : nullptr, mh);
        }
        if (tid == 0) {
            p.info[uu] = pack_info(terms, e);
            for (int i = 0; i < kCountersPerUnit; ++i) p.counters[(size_t)uu * kCountersPerUnit + i] = 0;
        }
        __syncthreads();  // red[] is reused by the next unit
    }
    if (tid == 0 && staged > 0) bulk_wait0();  // the images are written before the CTA exits
    }  // four-warp epilogue
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace

size_t project_smem_bytes(int mhalves, int distinct, int stages) {
    const size_t stage = (size_t)mhalves * 16384 * (1 + distinct) + 16384;
    return 1024 + stage * stages + 256;
}

int launch_project(const CUtensorMap &tE, const CUtensorMap &tF, const CUtensorMap &tK,
                   const CUtensorMap &tV, const ProjParams &p, int grid, int threads, size_t smem,
                   cudaStream_t s) {
    if (threads != kThreads && threads != 2 * kThreads) return LINFORMER_ERR_LAUNCH;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(tc_project_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess ||
            cudaFuncSetAttribute(tc_project_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
            return LINFORMER_ERR_LAUNCH;
        configured_dev = dev;
    }
    KernelScope scope(LINFORMER_KERNEL_PROJECT_TC, s);
    // Programmatic serialisation: the grid may be scheduled while the previous kernel in
    // the stream finishes (the kernel waits for it before touching memory).
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = (p.kbar_out || p.vbar_out)
                              ? cudaLaunchKernelEx(&cfg, tc_project_kernel<true>, tE, tF, tK, tV, p)
                              : cudaLaunchKernelEx(&cfg, tc_project_kernel<false>, tE, tF, tK, tV, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LINFORMER_ERR_LAUNCH;
    }
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace tc
}  // namespace linformer
