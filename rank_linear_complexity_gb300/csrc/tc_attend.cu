// Compressed attention on the tensor cores: O = softmax(Q . Kbar^T / sqrt(d)) . Vbar
// ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// the n x k score matrix replaces n x n and the queries are not compressed;
// section Transformer and Self-Attention: softmax along the key axis; padded
// query rows produce zero output, section Model, padding paragraph).
//
// Persistent CTAs walk a contiguous range of 128-row query tiles (unit-major).
// Roles (320 threads):
//   warps 0-3  softmax/epilogue group 0, warps 4-7 group 1: tiles of the range
//              alternate between the groups (ping-pong), one query row per
//              thread (TMEM lane = row);
//   warp 8     producer: Q per tile by TMA into a ring, and the projection
//              step's pre-swizzled images (Kbar hi/lo bf16, Vbar hi[/lo] fp16)
//              once per unit by bulk copy;
//   warp 9     MMA issuer (one thread), one tile of look-ahead so that the
//              scores of the next tile are computed while a group is busy with
//              the softmax of the current one.
// TMEM (512 columns) holds two 256-column buffers, one per group.  In a buffer:
//   S  = Q . Kbar_hi^T + Q . Kbar_lo^T   fp32, columns [0, k_pad)
//   P  (fp16, packed two per column)     over the consumed S columns [0, k_pad/2)
//   O  = P . Vbar_hi                     fp32, columns [128, 192)
// Units whose |Vbar| is large take three products for P . Vbar (P_lo . Vbar_hi
// and P_hi . Vbar_lo added); such a tile also uses the other group's buffer
// (P_lo at its column 0, O at its column 128) and runs without look-ahead.
// The softmax is exact and two-pass (row max, then exp2 with the 1/sqrt(d)
// scale folded in, row sum).  The epilogue scales by 2^e / sum, rounds, stages
// a 128-byte-swizzled tile and TMA-stores it; scores never leave the SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

namespace linformer {
namespace tc {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kBufCols = 256, kColO = 128, kTmemCols = 512;
constexpr uint32_t kImg = 32768;  // largest image: 256 rows x 128 bytes
constexpr uint32_t kQBytes = 16384;
constexpr int kMaxQSlots = 4;     // Q ring depth with bf16 output (2 with fp32 output)

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

// One lane polls the barrier; the warp then continues together.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *status, int code,
                                          volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status, code, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // orders the poller's acquire before the other lanes' reads
    return ok != 0;
}

// One 32-column chunk of the second softmax pass: p = 2^(s * scale - mb) for the
// valid columns (MASKED: columns >= k are set to zero), written back as packed
// fp16 over S columns [cc/2, cc/2 + 16) (all already read).  One product keeps
// the row sum of the rounded values; three products keep P_lo = fp16(p - P_hi)
// in the other buffer and sum p itself.
template <int TERMS, bool MASKED>
__device__ __forceinline__ void softmax_chunk(uint32_t buf, uint32_t other, int cc, int k,
                                              float scale, float mb, float &l0, float &l1) {
    uint32_t v[32];
    tmem_ld32(buf + cc, v);
    uint32_t ph[16], pl[16];
    const float2 sc = make_float2(scale, scale), nb = make_float2(-mb, -mb);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float2 x = ffma2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc, nb);
        float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
        if (MASKED) {
            if (cc + 2 * e >= k) p0 = 0.f;
            if (cc + 2 * e + 1 >= k) p1 = 0.f;
        }
        const __half2 h = __floats2half2_rn(p0, p1);
        ph[e] = *reinterpret_cast<const uint32_t *>(&h);
        if (TERMS == 1) {
            l0 = add_f32_f16(l0, __low2half(h));
            l1 = add_f32_f16(l1, __high2half(h));
        } else {
            const float2 hf = __half22float2(h);
            pl[e] = pack_f16(p0 - hf.x, p1 - hf.y);
            l0 += p0;
            l1 += p1;
        }
    }
    tmem_st16(buf + (cc >> 1), ph);
    if (TERMS == 3) tmem_st16(other + (cc >> 1), pl);
}

// Exact two-pass row softmax of one tile row (this thread's TMEM lane); returns
// the row sum.  P replaces S in `buf` (and P_lo goes to `other` for 3 products).
template <int TERMS>
__device__ __forceinline__ float softmax_row(uint32_t buf, uint32_t other, int k, float scale) {
    const int kfull = k & ~63;  // columns in whole 64-column chunks
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 1
    for (int cc = 0; cc < kfull; cc += 64) {
        uint32_t v[64];
        tmem_ld64(buf + cc, v);
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
            m0 = max3(m0, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            m1 = max3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
    }
    if (kfull < k) {
        uint32_t v[64];
        tmem_ld64(buf + kfull, v);
#pragma unroll
        for (int i = 0; i < 64; ++i)
            if (kfull + i < k) m0 = fmaxf(m0, __uint_as_float(v[i]));
    }
    const float mb = fmaxf(m0, m1) * scale;
    float l0 = 0.f, l1 = 0.f;
    const int k32 = k & ~31;  // columns in whole 32-column chunks
#pragma unroll 1
    for (int cc = 0; cc < k32; cc += 32)
        softmax_chunk<TERMS, false>(buf, other, cc, k, scale, mb, l0, l1);
    if (k32 < k) softmax_chunk<TERMS, true>(buf, other, k32, k, scale, mb, l0, l1);
    return l0 + l1;
}

struct Tile {
    int u, t, w, terms;
};

__global__ void __launch_bounds__(kThreads, 1)
    tc_attend_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tO,
                     const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stage_o = p.out_fp32 ? 32768u : 16384u;
    const int QS = p.out_fp32 ? 2 : kMaxQSlots;  // Q ring slots
    uint8_t *sKh = smem, *sKl = smem + kImg, *sVh = smem + 2 * kImg, *sVl = smem + 3 * kImg;
    uint8_t *sQ = smem + 4 * kImg;    // QS x 16 KB
    uint8_t *sO = sQ + QS * kQBytes;  // one staging tile per group
    uint64_t *bars = reinterpret_cast<uint64_t *>(sO + 2 * stage_o);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1;
    uint64_t *q_full = bars + 2, *q_empty = bars + 2 + kMaxQSlots;
    uint64_t *s_full = bars + 2 + 2 * kMaxQSlots, *p_full = s_full + 2, *o_full = s_full + 4;
    uint64_t *tmem_free = s_full + 6;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(s_full + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long total = (long long)p.units * p.tiles_per_unit;
    const long long t_begin = total * blockIdx.x / gridDim.x;
    const long long t_end = total * (blockIdx.x + 1) / gridDim.x;
    const uint32_t img_bytes = (uint32_t)p.kpad * kRowBytes;

    if (tid == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < kMaxQSlots; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(s_full + s, 1);
            mbar_init(p_full + s, 4);  // one arrival per warp of the group
            mbar_init(o_full + s, 1);
            mbar_init(tmem_free + s, 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tQ);
        prefetch_tmap(&tO);
    }
    if (warp == kProducerWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto terms_of = [&](int u) {
        return p.forced_terms ? p.forced_terms : info_terms(__ldg(p.info + u));
    };

    if (warp == kProducerWarp) {
        if (lane == 0) {  // ---------------- producer: Q per tile, images per unit
            int cur = -1, nload = 0, qit = 0;
            for (long long T = t_begin; T < t_end; ++T) {
                const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
                const int L = valid_length(p.pad, u / p.h, p.n);
                if (t * kTileM >= L) continue;
                // Q first: its slot does not depend on the images of the unit.
                const int s = qit % QS;
                if (qit >= QS && !mbar_wait(q_empty + s, ((qit / QS) - 1) & 1, p.status, 22, abort_flag))
                    break;
                mbar_arrive_expect_tx(q_full + s, kQBytes);
                tma_load_3d(sQ + s * kQBytes, &tQ, q_full + s, 0, t * kTileM, u);
                ++qit;
                if (u != cur) {
                    if (nload > 0 && !mbar_wait(kv_empty, (nload - 1) & 1, p.status, 21, abort_flag))
                        break;
                    const int terms = terms_of(u);
                    const uint8_t *src = p.images + (size_t)u * 4 * img_bytes;
                    mbar_arrive_expect_tx(kv_full, img_bytes * (terms == 3 ? 4u : 3u));
                    bulk_load(sKh, src, img_bytes, kv_full);
                    bulk_load(sKl, src + img_bytes, img_bytes, kv_full);
                    bulk_load(sVh, src + 2 * img_bytes, img_bytes, kv_full);
                    if (terms == 3) bulk_load(sVl, src + 3 * img_bytes, img_bytes, kv_full);
                    cur = u;
                    ++nload;
                }
            }
            // Let every copy this thread started land before the CTA may exit
            // (also after an abort: a copy must not outlive the CTA).
            if (nload > 0) mbar_wait_drain(kv_full, (nload - 1) & 1);
            for (int i = qit > QS ? qit - QS : 0; i < qit; ++i)
                mbar_wait_drain(q_full + (i % QS), (i / QS) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {  // ---------------- MMA issuer
            const uint32_t idesc_qk = idesc_f16(128, p.kpad, 1, 0, 0);
            const uint32_t idesc_pv = idesc_f16(128, 64, 0, 0, 1);
            const uint32_t kh = smem_u32(sKh), kl = smem_u32(sKl);
            const uint32_t vh = smem_u32(sVh), vl = smem_u32(sVl);
            const int nks = p.kpad / 16;
            // Per group: P.V products issued so far, and the product count of its
            // latest tile (kept in registers, not local-memory arrays).
            int cnt0 = 0, cnt1 = 0, last0 = 1, last1 = 1;
            int cur_unit = -1, nload = 0, qit = 0;
            long long T = t_begin;
            auto next_tile = [&](Tile &X) -> bool {
                while (T < t_end) {
                    const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
                    const int w = (int)((T - t_begin) & 1);
                    ++T;
                    if (t * kTileM < valid_length(p.pad, u / p.h, p.n)) {
                        X = Tile{u, t, w, terms_of(u)};
                        return true;
                    }
                }
                return false;
            };
            auto issue_qk = [&](const Tile &X) -> bool {
                if (X.u != cur_unit) {
                    if (nload > 0) mma_commit(kv_empty);  // old images free once issued MMAs finish
                    if (!mbar_wait(kv_full, nload & 1, p.status, 23, abort_flag)) return false;
                    cur_unit = X.u;
                    ++nload;
                }
                const int s = qit % QS, w = X.w, o = 1 - w;
                if (!mbar_wait(q_full + s, (qit / QS) & 1, p.status, 24, abort_flag)) return false;
                const int cw = w ? cnt1 : cnt0, co = w ? cnt0 : cnt1, lo = w ? last0 : last1;
                if (cw > 0 && !mbar_wait(tmem_free + w, (cw - 1) & 1, p.status, 25, abort_flag))
                    return false;
                if ((X.terms == 3 || lo == 3) && co > 0 &&
                    !mbar_wait(tmem_free + o, (co - 1) & 1, p.status, 25, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t q0 = smem_u32(sQ + s * kQBytes);
                const uint32_t d = tmem + kBufCols * w;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(d, sdesc(q0 + ks * 32, 16, 1024, kSwizzle128B),
                           sdesc(kh + ks * 32, 16, 1024, kSwizzle128B), idesc_qk, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(d, sdesc(q0 + ks * 32, 16, 1024, kSwizzle128B),
                           sdesc(kl + ks * 32, 16, 1024, kSwizzle128B), idesc_qk, 1u);
                mma_commit(s_full + w);
                mma_commit(q_empty + s);
                ++qit;
                return true;
            };
            auto issue_pv = [&](const Tile &X) -> bool {
                const int w = X.w, o = 1 - w;
                if (!mbar_wait(p_full + w, (w ? cnt1 : cnt0) & 1, p.status, 26, abort_flag)) return false;
                tc_fence_after();
                const uint32_t a = tmem + kBufCols * w;
                const uint32_t dO = X.terms == 3 ? tmem + kBufCols * o + kColO : a + kColO;
                for (int ks = 0; ks < nks; ++ks)
                    mma_ts(dO, a + ks * 8, sdesc(vh + ks * 2048, 16, 1024, kSwizzle128B), idesc_pv,
                           ks > 0 ? 1u : 0u);
                if (X.terms == 3) {
                    const uint32_t alo = tmem + kBufCols * o;
                    for (int ks = 0; ks < nks; ++ks)
                        mma_ts(dO, alo + ks * 8, sdesc(vh + ks * 2048, 16, 1024, kSwizzle128B),
                               idesc_pv, 1u);
                    for (int ks = 0; ks < nks; ++ks)
                        mma_ts(dO, a + ks * 8, sdesc(vl + ks * 2048, 16, 1024, kSwizzle128B),
                               idesc_pv, 1u);
                }
                mma_commit(o_full + w);
                if (w) {
                    ++cnt1;
                    last1 = X.terms;
                } else {
                    ++cnt0;
                    last0 = X.terms;
                }
                return true;
            };
            Tile cur{}, nxt{};
            bool have = next_tile(cur);
            bool ok = !have || issue_qk(cur);
            while (have && ok) {
                const bool have_n = next_tile(nxt);
                // Look ahead (scores of the next tile before P.V of this one) only
                // within a unit and when both tiles use just their own buffer.
                const bool look = have_n && nxt.u == cur.u && cur.terms == 1 && nxt.terms == 1;
                if (look) ok = issue_qk(nxt);
                if (ok) ok = issue_pv(cur);
                if (ok && have_n && !look) ok = issue_qk(nxt);
                cur = nxt;
                have = have_n;
            }
        }
        __syncwarp();
    } else {  // ---------------- groups 0/1: softmax + epilogue, one query row per thread
        const int w = warp >> 2;                 // group
        const int tw = tid & 127;                // row within the tile
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t buf = tmem + lane_off + kBufCols * w;
        const uint32_t other = tmem + lane_off + kBufCols * (1 - w);
        uint8_t *stage = sO + w * stage_o;
        const uint32_t bar_id = 1 + w;
        int done = 0;
        int cur_u = -1, L = 0, info = 0, terms = 1;
        for (long long T = t_begin + w; T < t_end; T += 2) {
            const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
            if (u != cur_u) {  // per-unit values, read once per unit
                cur_u = u;
                L = valid_length(p.pad, u / p.h, p.n);
                info = __ldg(p.info + u);
                terms = p.forced_terms ? p.forced_terms : info_terms(info);
            }
            const int row = t * kTileM + tw;
            // The tile row as output words: fp32 bits, or packed bf16 pairs in ov[0..31].
            uint32_t ov[64];
            if (t * kTileM < L) {
                if (!warp_wait(s_full + w, done & 1, p.status, 27, abort_flag)) break;
                tc_fence_after();
                const float l = terms == 3 ? softmax_row<3>(buf, other, p.k, p.scale_log2)
                                           : softmax_row<1>(buf, other, p.k, p.scale_log2);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + w);
                if (!warp_wait(o_full + w, done & 1, p.status, 28, abort_flag)) break;
                tc_fence_after();
                tmem_ld64((terms == 3 ? other : buf) + kColO, ov);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tmem_free + w);
                ++done;
                // Padded query rows are written as zero (selected, not scaled: their
                // scores may hold anything, NaN included).
                const bool valid = row < L;
                const float inv = exp2f((float)info_exp(info)) / l;
                if (!p.out_fp32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        ov[i] = valid ? pack_bf16(__uint_as_float(ov[2 * i]) * inv,
                                                  __uint_as_float(ov[2 * i + 1]) * inv)
                                      : 0u;
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        ov[i] = valid ? __float_as_uint(__uint_as_float(ov[i]) * inv) : 0u;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) ov[i] = 0u;
            }
            // Stage the tile (128-byte swizzle) once the previous store has read it.
            if (tw == 0) bulk_wait_read0();
            named_barrier_sync(bar_id, 128);
            if (!p.out_fp32) {
                uint8_t *rowp = stage + tw * kRowBytes;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4 *>(rowp + ((q ^ (tw & 7)) << 4)) =
                        make_uint4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint8_t *rowp = stage + half * 16384 + tw * kRowBytes;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int b0 = half * 32 + q * 4;
                        *reinterpret_cast<uint4 *>(rowp + ((q ^ (tw & 7)) << 4)) =
                            make_uint4(ov[b0], ov[b0 + 1], ov[b0 + 2], ov[b0 + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(bar_id, 128);
            if (tw == 0) {
                tma_store_3d(&tO, stage, 0, t * kTileM, u);
                if (p.out_fp32) tma_store_3d(&tO, stage + 16384, 32, t * kTileM, u);
                bulk_commit();
            }
        }
        if (tw == 0) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t attend_smem_bytes(int out_fp32) {
    return 1024 + 4 * kImg + (out_fp32 ? 2 : kMaxQSlots) * kQBytes +
           2 * (out_fp32 ? 32768 : 16384) + 256;
}

int launch_attend(const CUtensorMap &tQ, const CUtensorMap &tO, const AttnParams &p, int grid,
                  cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(tc_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attend_smem_bytes(1)) != cudaSuccess)
            return LINFORMER_ERR_LAUNCH;
        configured_dev = dev;
    }
    KernelScope scope(LINFORMER_KERNEL_ATTEND_TC, s);
    tc_attend_kernel<<<grid, kThreads, attend_smem_bytes(p.out_fp32), s>>>(tQ, tO, p);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace tc
}  // namespace linformer
