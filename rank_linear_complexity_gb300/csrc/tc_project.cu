// Projection step on the tensor cores: Kbar = Ehat . K and Vbar = Fhat . V
// ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
// E, F are k x n, row j of E merges the n positions into compressed position j;
// padded rows t >= L count as zero, section Model, padding paragraph).
//
// One CTA owns one (unit, sequence chunk) pair.  Per 64-row stage it TMA-loads
// the E (and F) tile, k_pad x 64, K-major, and the unit's K and V tiles,
// 64 x 64 each, whose d axis is contiguous (MN-major operand).  One thread
// issues tcgen05.mma into TMEM: with E = F a single N = 128 product covers K
// and V (the E tile is read once for both); with E != F two N = 64 products.
// Accumulators: M-half mh (rows 128 mh ..) at TMEM columns [128 mh, 128 mh + 128),
// columns 0-63 Kbar, 64-127 Vbar.
//
// Chunks of the same unit are summed in a fixed order (chunk 0, 1, ...) by
// whichever CTA of the unit arrives last, so the result does not depend on
// scheduling.  That CTA converts to the split images the attention step reads
// and picks the number of P.Vbar products from max|Vbar|.
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
constexpr int kVsStride = 65;  // fp32 scratch row stride (conflict-free per-row access)

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

__global__ void __launch_bounds__(kThreads, 1)
    tc_project_kernel(const __grid_constant__ CUtensorMap tE, const __grid_constant__ CUtensorMap tF,
                      const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
                      const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // CTA -> (group g, chunk c, member m); members of a group share E (and F).
    const int bid = blockIdx.x;
    const int m = bid % p.members;
    const int gc = bid / p.members;
    const int c = gc % p.C;
    const int g = gc / p.C;
    const int u = p.per_head ? m * p.h + g : m;
    const int L = valid_length(p.pad, u / p.h, p.n);
    const int Cu = L > 0 ? (L + p.CH - 1) / p.CH : 1;
    if (c >= Cu) return;  // chunk entirely in the padding: nothing to add
    const int row0 = c * p.CH;
    const int rows = max(0, min(p.CH, L - row0));
    const int nkb = (rows + kBK - 1) / kBK;
    const int gproj = p.per_head ? g : 0;

    const uint32_t a_bytes = (uint32_t)p.mhalves * 16384u;
    const uint32_t stage_bytes = a_bytes * (1 + p.distinct) + 16384u;
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    float *red = reinterpret_cast<float *>(tmem_slot + 4);
    const uint32_t ncols = (uint32_t)p.mhalves * 128u;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
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

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            for (int it = 0; it < nkb; ++it) {
                const int s = it % S;
                if (it >= S && !mbar_wait(empty + s, ((it / S) - 1) & 1, p.status, 11, abort_flag))
                    break;
                uint8_t *st = smem + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(full + s, stage_bytes);
                const int x = row0 + it * kBK;
                for (int mh = 0; mh < p.mhalves; ++mh)
                    tma_load_3d(st + mh * 16384, &tE, full + s, x, mh * 128, gproj);
                if (p.distinct)
                    for (int mh = 0; mh < p.mhalves; ++mh)
                        tma_load_3d(st + a_bytes + mh * 16384, &tF, full + s, x, mh * 128, gproj);
                uint8_t *bk = st + a_bytes * (1 + p.distinct);
                tma_load_3d(bk, &tK, full + s, 0, x, u);
                tma_load_3d(bk + 8192, &tV, full + s, 0, x, u);
            }
            // Let every copy this thread started land before the CTA may exit.
            const int first = nkb > S ? nkb - S : 0;
            for (int it = first; it < nkb; ++it)
                mbar_wait(full + (it % S), (it / S) & 1, p.status, 12, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            const uint32_t idesc128 = idesc_f16(128, 128, 1, 0, 1);
            const uint32_t idesc64 = idesc_f16(128, 64, 1, 0, 1);
            bool ok = true;
            for (int it = 0; it < nkb && ok; ++it) {
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
                    for (int r = valid; r < kBK; ++r) {
                        uint4 *rk = reinterpret_cast<uint4 *>(bk + r * kRowBytes);
                        uint4 *rv = reinterpret_cast<uint4 *>(bv + r * kRowBytes);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            rk[q] = z;
                            rv[q] = z;
                        }
                    }
                    fence_proxy_async_smem();
                }
                const uint32_t a0 = smem_u32(st), f0 = smem_u32(st + a_bytes);
                const uint32_t k0 = smem_u32(bk), v0 = smem_u32(bv);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = (it > 0 || ks > 0) ? 1u : 0u;
                    for (int mh = 0; mh < p.mhalves; ++mh) {
                        const uint64_t a = sdesc(a0 + mh * 16384 + ks * 32, 16, 1024, kSwizzle128B);
                        if (!p.distinct) {
                            // N = 128: columns 0-63 from the K tile, 64-127 from the V tile.
                            const uint64_t b = sdesc(k0 + ks * 2048, v0 - k0, 1024, kSwizzle128B);
                            mma_ss(tmem + mh * 128, a, b, idesc128, acc);
                        } else {
                            const uint64_t b = sdesc(k0 + ks * 2048, 16, 1024, kSwizzle128B);
                            mma_ss(tmem + mh * 128, a, b, idesc64, acc);
                            const uint64_t af =
                                sdesc(f0 + mh * 16384 + ks * 32, 16, 1024, kSwizzle128B);
                            const uint64_t bvd = sdesc(v0 + ks * 2048, 16, 1024, kSwizzle128B);
                            mma_ss(tmem + mh * 128 + 64, af, bvd, idesc64, acc);
                        }
                    }
                }
                mma_commit(empty + s);
            }
            if (ok && nkb > 0)
                mma_commit(acc_full);
            else
                mbar_arrive(acc_full);
        }
        __syncwarp();
    }

    // ---------------- epilogue: all four warps, thread = TMEM lane = projected row
    mbar_wait(acc_full, 0, p.status, 14, abort_flag);
    tc_fence_after();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    const int jl = warp * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const size_t part_unit = (size_t)p.kpad * 128;  // floats per (unit, chunk) partial

    if (!aborted && Cu > 1) {
        // Partial layout [unit][chunk][column][row]: a warp stores 32 consecutive floats.
        float *mine = p.partial + ((size_t)u * p.C + c) * part_unit;
        for (int mh = 0; mh < p.mhalves; ++mh) {
            const int j = mh * 128 + jl;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                if (nkb) {
                    tmem_ld32(lane_base + mh * 128 + cc * 32, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
                if (j < p.kpad) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        mine[(size_t)(cc * 32 + i) * p.kpad + j] = __uint_as_float(v[i]);
                }
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) *last_flag = (atomicAdd(p.counters + u, 1) == Cu - 1) ? 1 : 0;
        __syncthreads();
    }

    if (!aborted && (Cu == 1 || *last_flag)) {
        __threadfence();
        float *vs = reinterpret_cast<float *>(smem);  // [kpad][65] fp32 Vbar sums (stages are idle)
        uint8_t *img = p.images + (size_t)u * 4 * image_bytes(p.kpad);
        float vmax = 0.f;
        for (int mh = 0; mh < p.mhalves; ++mh) {
            const int j = mh * 128 + jl;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                float acc[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                for (int c2 = 0; c2 < Cu; ++c2) {  // fixed order: chunk 0, 1, ...
                    if (c2 == c) {
                        if (nkb) {
                            uint32_t v[32];
                            tmem_ld32(lane_base + mh * 128 + cc * 32, v);
#pragma unroll
                            for (int i = 0; i < 32; ++i) acc[i] += __uint_as_float(v[i]);
                        }
                    } else if (j < p.kpad) {
                        const float *src = p.partial + ((size_t)u * p.C + c2) * part_unit;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            acc[i] += __ldcg(src + (size_t)(cc * 32 + i) * p.kpad + j);
                    }
                }
                if (j >= p.kpad) continue;
                if (j >= p.k) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                }
                if (cc < 2) {  // Kbar: bf16 hi + bf16 lo
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = acc[q4 * 8 + 2 * e], x1 = acc[q4 * 8 + 2 * e + 1];
                            const __nv_bfloat16 h0 = __float2bfloat16_rn(x0);
                            const __nv_bfloat16 h1 = __float2bfloat16_rn(x1);
                            hi[e] = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                            lo[e] = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                            if (p.kbar_out && j < p.k) {
                                const __nv_bfloat162 l2 = *reinterpret_cast<__nv_bfloat162 *>(&lo[e]);
                                float *o = p.kbar_out + ((size_t)u * p.k + j) * kD + cc * 32 + q4 * 8 + 2 * e;
                                o[0] = __bfloat162float(h0) + __bfloat162float(l2.x);
                                o[1] = __bfloat162float(h1) + __bfloat162float(l2.y);
                            }
                        }
                        const int q = cc * 4 + q4;
                        *image_chunk(img, j, q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *image_chunk(img + image_bytes(p.kpad), j, q) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                } else {  // Vbar: keep fp32 until the unit's magnitude is known
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        vs[j * kVsStride + (cc - 2) * 32 + i] = acc[i];
                        vmax = fmaxf(vmax, fabsf(acc[i]));
                    }
                }
            }
        }
        // Unit-wide max|Vbar| -> scale exponent and number of P.Vbar products.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        if (lane == 0) red[warp] = vmax;
        __syncthreads();
        vmax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        int e = 0;
        while (e < 100 && vmax * exp2f(-(float)e) >= 16384.f) ++e;
        const float vscale = exp2f(-(float)e);
        const int terms = p.forced_terms ? p.forced_terms : (vmax < kOneTermMaxV ? 1 : 3);
        for (int mh = 0; mh < p.mhalves; ++mh) {
            const int j = mh * 128 + jl;
            if (j >= p.kpad) continue;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float x0 = vs[j * kVsStride + q * 8 + 2 * e2] * vscale;
                    const float x1 = vs[j * kVsStride + q * 8 + 2 * e2 + 1] * vscale;
                    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
                    hi[e2] = pack_f16(__half2float(h0), __half2float(h1));
                    lo[e2] = pack_f16(x0 - __half2float(h0), x1 - __half2float(h1));
                    if (p.vbar_out && j < p.k) {
                        const __half2 l2 = *reinterpret_cast<__half2 *>(&lo[e2]);
                        float *o = p.vbar_out + ((size_t)u * p.k + j) * kD + q * 8 + 2 * e2;
                        o[0] = (__half2float(h0) + __half2float(l2.x)) / vscale;
                        o[1] = (__half2float(h1) + __half2float(l2.y)) / vscale;
                    }
                }
                *image_chunk(img + 2 * image_bytes(p.kpad), j, q) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *image_chunk(img + 3 * image_bytes(p.kpad), j, q) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        if (tid == 0) {
            p.info[u] = pack_info(terms, e);
            p.counters[u] = 0;
        }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace

size_t project_smem_bytes(int mhalves, int distinct, int stages) {
    const size_t stage = (size_t)mhalves * 16384 * (1 + distinct) + 16384;
    return 1024 + stage * stages + 256;
}

int launch_project(const CUtensorMap &tE, const CUtensorMap &tF, const CUtensorMap &tK,
                   const CUtensorMap &tV, const ProjParams &p, int grid, size_t smem,
                   cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(tc_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024) != cudaSuccess)
            return LINFORMER_ERR_LAUNCH;
        configured_dev = dev;
    }
    KernelScope scope(LINFORMER_KERNEL_PROJECT_TC, s);
    tc_project_kernel<<<grid, kThreads, smem, s>>>(tE, tF, tK, tV, p);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace tc
}  // namespace linformer
