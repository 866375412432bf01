// Compressed attention on the tensor cores: O = softmax(Q . Kbar^T / sqrt(d)) . Vbar
// ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// the n x k score matrix replaces n x n and the queries are not compressed;
// section Transformer and Self-Attention: softmax along the key axis; padded
// query rows produce zero output, section Model, padding paragraph).
//
// Persistent CTAs walk a contiguous range of 128-row query tiles (unit-major).
// Per unit the producer bulk-copies the projection step's pre-swizzled images
// (Kbar hi/lo in bf16, Vbar hi[/lo] in fp16) into shared memory once; per tile
// it TMA-loads Q.  One thread issues the MMAs:
//   S (TMEM cols [0, k_pad), fp32) = Q . Kbar_hi^T + Q . Kbar_lo^T
//   O (TMEM cols [384, 448), fp32) = P_hi . Vbar_hi [+ P_lo . Vbar_hi + P_hi . Vbar_lo]
// with P read straight from TMEM.  Four warps own one query row per thread
// (TMEM lane = row): exact two-pass softmax over the k columns (max, then
// exp2 with the scale folded in and the row sum), P_hi written as packed fp16
// over the already-consumed S columns, P_lo at TMEM cols [256, 384).  The
// epilogue scales by 2^e / sum, rounds, stages a 128-byte-swizzled tile and
// TMA-stores it; the n x k scores never leave the SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

namespace linformer {
namespace tc {
namespace {

using namespace ptx;

constexpr int kThreads = 192;  // warps 0-3 softmax/epilogue, 4 TMA producer, 5 MMA issuer
constexpr uint32_t kColP_lo = 256, kColO = 384, kTmemCols = 512;
constexpr uint32_t kImg = 32768;  // largest image: 256 rows x 128 bytes

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

__global__ void __launch_bounds__(kThreads, 1)
    tc_attend_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tO,
                     const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sKh = smem, *sKl = smem + kImg, *sVh = smem + 2 * kImg, *sVl = smem + 3 * kImg;
    uint8_t *sQ = smem + 4 * kImg;                  // 2 x 16 KB
    uint8_t *sO = sQ + 2 * 16384;                   // 16 KB (bf16) or 32 KB (fp32)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sO + 32768);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1, *q_full = bars + 2, *q_empty = bars + 4;
    uint64_t *s_full = bars + 6, *p_full = bars + 7, *o_full = bars + 8, *tmem_free = bars + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 10);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long total = (long long)p.units * p.tiles_per_unit;
    const long long t_begin = total * blockIdx.x / gridDim.x;
    const long long t_end = total * (blockIdx.x + 1) / gridDim.x;
    const uint32_t img_bytes = (uint32_t)p.kpad * kRowBytes;

    if (tid == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 128);
        mbar_init(o_full, 1);
        mbar_init(tmem_free, 128);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tQ);
        prefetch_tmap(&tO);
    }
    if (warp == 4) {
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

    if (warp == 4) {
        if (lane == 0) {  // ---------------- producer: images per unit, Q per tile
            int cur = -1, nload = 0, qit = 0;
            for (long long T = t_begin; T < t_end; ++T) {
                const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
                const int L = valid_length(p.pad, u / p.h, p.n);
                if (t * kTileM >= L) continue;
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
                const int s = qit & 1;
                if (qit >= 2 && !mbar_wait(q_empty + s, ((qit >> 1) - 1) & 1, p.status, 22, abort_flag))
                    break;
                mbar_arrive_expect_tx(q_full + s, 16384);
                tma_load_3d(sQ + s * 16384, &tQ, q_full + s, 0, t * kTileM, u);
                ++qit;
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {  // ---------------- MMA issuer
            const uint32_t idesc_qk = idesc_f16(128, p.kpad, 1, 0, 0);
            const uint32_t idesc_pv = idesc_f16(128, 64, 0, 0, 1);
            const uint32_t kh = smem_u32(sKh), kl = smem_u32(sKl);
            const uint32_t vh = smem_u32(sVh), vl = smem_u32(sVl);
            const int nks = p.kpad / 16;
            int cur = -1, nload = 0, qit = 0, done = 0, terms = 1;
            for (long long T = t_begin; T < t_end; ++T) {
                const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
                const int L = valid_length(p.pad, u / p.h, p.n);
                if (t * kTileM >= L) continue;
                if (u != cur) {
                    if (nload > 0) mma_commit(kv_empty);  // old images free once issued MMAs finish
                    if (!mbar_wait(kv_full, nload & 1, p.status, 23, abort_flag)) break;
                    cur = u;
                    ++nload;
                    terms = terms_of(u);
                }
                const int s = qit & 1;
                if (!mbar_wait(q_full + s, (qit >> 1) & 1, p.status, 24, abort_flag)) break;
                if (done > 0 && !mbar_wait(tmem_free, (done - 1) & 1, p.status, 25, abort_flag)) break;
                tc_fence_after();
                const uint32_t q0 = smem_u32(sQ + s * 16384);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem, sdesc(q0 + ks * 32, 16, 1024, kSwizzle128B),
                           sdesc(kh + ks * 32, 16, 1024, kSwizzle128B), idesc_qk, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem, sdesc(q0 + ks * 32, 16, 1024, kSwizzle128B),
                           sdesc(kl + ks * 32, 16, 1024, kSwizzle128B), idesc_qk, 1u);
                mma_commit(s_full);
                mma_commit(q_empty + s);
                ++qit;
                if (!mbar_wait(p_full, done & 1, p.status, 26, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < nks; ++ks)
                    mma_ts(tmem + kColO, tmem + ks * 8, sdesc(vh + ks * 2048, 16, 1024, kSwizzle128B),
                           idesc_pv, ks > 0 ? 1u : 0u);
                if (terms == 3) {
                    for (int ks = 0; ks < nks; ++ks)
                        mma_ts(tmem + kColO, tmem + kColP_lo + ks * 8,
                               sdesc(vh + ks * 2048, 16, 1024, kSwizzle128B), idesc_pv, 1u);
                    for (int ks = 0; ks < nks; ++ks)
                        mma_ts(tmem + kColO, tmem + ks * 8,
                               sdesc(vl + ks * 2048, 16, 1024, kSwizzle128B), idesc_pv, 1u);
                }
                mma_commit(o_full);
                ++done;
            }
        }
        __syncwarp();
    } else {  // ---------------- warps 0-3: softmax + epilogue, one query row per thread
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
        int done = 0;
        for (long long T = t_begin; T < t_end; ++T) {
            const int u = (int)(T / p.tiles_per_unit), t = (int)(T % p.tiles_per_unit);
            const int L = valid_length(p.pad, u / p.h, p.n);
            const int row = t * kTileM + tid;
            float o[64];
            if (t * kTileM < L) {
                const int info = __ldg(p.info + u);
                const int terms = p.forced_terms ? p.forced_terms : info_terms(info);
                if (!mbar_wait(s_full, done & 1, p.status, 27, abort_flag)) break;
                tc_fence_after();
                float mx = -INFINITY;
                for (int cc = 0; cc < p.kpad; cc += 32) {
                    uint32_t v[32];
                    tmem_ld32(taddr + cc, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cc + i < p.k) mx = fmaxf(mx, __uint_as_float(v[i]));
                }
                const float mb = mx * p.scale_log2;
                float l = 0.f;
                for (int cc = 0; cc < p.kpad; cc += 32) {
                    uint32_t v[32];
                    tmem_ld32(taddr + cc, v);
                    uint32_t ph[16], pl[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j0 = cc + 2 * e;
                        const float p0 = j0 < p.k ? ex2_approx(fmaf(__uint_as_float(v[2 * e]), p.scale_log2, -mb)) : 0.f;
                        const float p1 = j0 + 1 < p.k ? ex2_approx(fmaf(__uint_as_float(v[2 * e + 1]), p.scale_log2, -mb)) : 0.f;
                        const __half h0 = __float2half_rn(p0), h1 = __float2half_rn(p1);
                        ph[e] = pack_f16(__half2float(h0), __half2float(h1));
                        if (terms == 3) {
                            pl[e] = pack_f16(p0 - __half2float(h0), p1 - __half2float(h1));
                            l += p0 + p1;
                        } else {
                            l += __half2float(h0) + __half2float(h1);
                        }
                    }
                    // P_hi goes over S columns [cc/2, cc/2 + 16), all already read.
                    tmem_st16(taddr + (cc >> 1), ph);
                    if (terms == 3) tmem_st16(taddr + kColP_lo + (cc >> 1), pl);
                }
                tc_fence_before();
                mbar_arrive(p_full);
                if (!mbar_wait(o_full, done & 1, p.status, 28, abort_flag)) break;
                tc_fence_after();
                uint32_t v0[32], v1[32];
                tmem_ld32(taddr + kColO, v0);
                tmem_ld32(taddr + kColO + 32, v1);
                tc_fence_before();
                mbar_arrive(tmem_free);
                ++done;
                const float inv = (row < L) ? exp2f((float)info_exp(info)) / l : 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    o[i] = __uint_as_float(v0[i]) * inv;
                    o[32 + i] = __uint_as_float(v1[i]) * inv;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) o[i] = 0.f;
            }
            // Stage the tile (128-byte swizzle) once the previous store has read it.
            if (tid == 0) bulk_wait_read0();
            named_barrier_sync(1, 128);
            if (!p.out_fp32) {
                uint8_t *rowp = sO + tid * kRowBytes;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint4 w = make_uint4(pack_bf16(o[q * 8 + 0], o[q * 8 + 1]),
                                         pack_bf16(o[q * 8 + 2], o[q * 8 + 3]),
                                         pack_bf16(o[q * 8 + 4], o[q * 8 + 5]),
                                         pack_bf16(o[q * 8 + 6], o[q * 8 + 7]));
                    *reinterpret_cast<uint4 *>(rowp + ((q ^ (tid & 7)) << 4)) = w;
                }
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint8_t *rowp = sO + half * 16384 + tid * kRowBytes;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float *src = o + half * 32 + q * 4;
                        uint4 w = make_uint4(__float_as_uint(src[0]), __float_as_uint(src[1]),
                                             __float_as_uint(src[2]), __float_as_uint(src[3]));
                        *reinterpret_cast<uint4 *>(rowp + ((q ^ (tid & 7)) << 4)) = w;
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(1, 128);
            if (tid == 0) {
                if (!p.out_fp32) {
                    tma_store_3d(&tO, sO, 0, t * kTileM, u);
                } else {
                    tma_store_3d(&tO, sO, 0, t * kTileM, u);
                    tma_store_3d(&tO, sO + 16384, 32, t * kTileM, u);
                }
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t attend_smem_bytes(int) { return 1024 + 4 * kImg + 2 * 16384 + 32768 + 256; }

int launch_attend(const CUtensorMap &tQ, const CUtensorMap &tO, const AttnParams &p, int grid,
                  cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = attend_smem_bytes(p.out_fp32);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(tc_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return LINFORMER_ERR_LAUNCH;
        configured_dev = dev;
    }
    KernelScope scope(LINFORMER_KERNEL_ATTEND_TC, s);
    tc_attend_kernel<<<grid, kThreads, smem, s>>>(tQ, tO, p);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace tc
}  // namespace linformer
