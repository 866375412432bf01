// Batched fp32 SIMT matrix products and the row softmax (declared in simt_gemm.cuh).
#include <algorithm>

#include "simt_gemm.cuh"

namespace linformer {
namespace simt {
namespace {

constexpr int kBK = 16;        // depth of one product step
constexpr int kThreads = 256;  // 16 x 16 threads, each owning (BM/16) x (BN/16) outputs

__device__ __forceinline__ int unit_length(const int32_t *pad, int unit, int h, int n) {
    if (!pad) return n;
    const int L = pad[unit / h];
    return L < 0 ? 0 : (L > n ? n : L);
}

constexpr int kStages = 3;  // shared-memory slabs in flight

__device__ __forceinline__ void cp_async16(float *dst, const float *src, int src_bytes) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *src, int src_bytes) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Asynchronous copy of one BX x kBK operand tile (x0.., k0..) into s[kk][x] (row stride
// BX + 4).  Elements out of range or masked are zero-filled by the copy itself (a
// source size of 0, or fewer than 16 bytes at the edge of a masked range); their
// source address is then the matrix base, which is never read.  Groups of four along
// a contiguous x go as 16-byte copies (vec); everything else as 4-byte copies in
// which consecutive threads read consecutive addresses (in the transposing kk-fast
// case, 16 threads read one 64-byte row segment).
template <int BX>
__device__ __forceinline__ void copy_tile(const Operand &o, const float *m, int x0, int k0, int X,
                                          int K, int L, float *s) {
    if (o.xfast && o.vec) {
#pragma unroll
        for (int g = 0; g < BX / 64; ++g) {
            const int idx = threadIdx.x + g * kThreads;
            const int xr = (idx % (BX / 4)) * 4, kk = idx / (BX / 4);
            const int x = x0 + xr, ka = k0 + kk;
            int bytes = 0;
            if (x < X && ka < K && !(o.mask_k && ka >= L)) {
                const int lim = o.mask_x ? min(4, L - x) : 4;
                bytes = lim > 0 ? lim * 4 : 0;
            }
            cp_async16(s + kk * (BX + 4) + xr, bytes ? m + (long long)ka * o.ld + x : m, bytes);
        }
    } else {
#pragma unroll
        for (int e = 0; e < BX / 16; ++e) {
            const int idx = threadIdx.x + e * kThreads;
            const int xr = o.xfast ? idx % BX : idx / kBK;
            const int kk = o.xfast ? idx / BX : idx % kBK;
            const int x = x0 + xr, ka = k0 + kk;
            const bool in = x < X && ka < K && !(o.mask_x && x >= L) && !(o.mask_k && ka >= L);
            const long long off = o.xfast ? (long long)ka * o.ld + x : (long long)x * o.ld + ka;
            cp_async4(s + kk * (BX + 4) + xr, in ? m + off : m, in ? 4 : 0);
        }
    }
}

// One BM x BN output tile of unit blockIdx.z per CTA.  Thread (tx, ty) owns rows
// ty*4 + {0..3} (+ 64, + 128 ... for BM > 64) and columns tx*4 + {0..3} (+ 64 ...), so
// its shared-memory reads are 16-byte loads that a warp serves in two passes.  Slabs
// of kBK arrive by asynchronous copies kStages - 1 steps ahead of their use; one
// barrier per step both publishes the arrived slab and frees the one about to be
// overwritten.  Dynamic shared memory: kStages * kBK * (BM + BN + 8) floats.
template <int BM, int BN>
__global__ void __launch_bounds__(kThreads, 2) batched_gemm_kernel(const GemmArgs g) {
    constexpr int TM = BM / 16, TN = BN / 16;
    constexpr int SA = kBK * (BM + 4), SB = kBK * (BN + 4);
    extern __shared__ __align__(16) float smem[];
    float *sA = smem, *sB = smem + kStages * SA;
    const int z = blockIdx.z, tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int tiles_n = gridDim.x / g.splits, split = blockIdx.x / tiles_n;
    const int row0 = blockIdx.y * BM, col0 = (blockIdx.x % tiles_n) * BN;
    const int kbeg = split * g.kchunk, kend = min(g.K, kbeg + g.kchunk);
    const int nslabs = kend > kbeg ? (kend - kbeg + kBK - 1) / kBK : 0;
    const float *A = g.A.mat(z, g.h), *B = g.B.mat(z, g.h);
    const int L = unit_length(g.pad, z, g.h, g.n);
    float acc[TM][TN] = {};
    auto issue = [&](int slab) {
        if (slab < nslabs) {
            const int k0 = kbeg + slab * kBK, st = slab % kStages;
            copy_tile<BM>(g.A, A, row0, k0, g.M, kend, L, sA + st * SA);
            copy_tile<BN>(g.B, B, col0, k0, g.N, kend, L, sB + st * SB);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) issue(st);
    for (int it = 0; it < nslabs; ++it) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        issue(it + kStages - 1);
        const float *a_s = sA + (it % kStages) * SA, *b_s = sB + (it % kStages) * SB;
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int q = 0; q < TM / 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(a_s + kk * (BM + 4) + q * 64 + ty * 4);
                a[q * 4] = t.x;
                a[q * 4 + 1] = t.y;
                a[q * 4 + 2] = t.z;
                a[q * 4 + 3] = t.w;
            }
#pragma unroll
            for (int q = 0; q < TN / 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(b_s + kk * (BN + 4) + q * 64 + tx * 4);
                b[q * 4] = t.x;
                b[q * 4 + 1] = t.y;
                b[q * 4 + 2] = t.z;
                b[q * 4 + 3] = t.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();
    if (g.splits > 1) {
        float *Pt = g.part + ((long long)split * gridDim.z + z) * g.M * g.N;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = row0 + (i / 4) * 64 + ty * 4 + (i % 4);
            if (r >= g.M) continue;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int c = col0 + (j / 4) * 64 + tx * 4 + (j % 4);
                if (c < g.N) Pt[(long long)r * g.N + c] = g.alpha * acc[i][j];
            }
        }
        return;
    }
    float *C = g.C + (long long)z * g.sC;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int r = row0 + (i / 4) * 64 + ty * 4 + (i % 4);
        if (r >= g.M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int c = col0 + (j / 4) * 64 + tx * 4 + (j % 4);
            if (c >= g.N) continue;
            float v = g.alpha * acc[i][j];
            if (g.beta != 0.f) v = fmaf(g.beta, C[(long long)r * g.ldc + c], v);
            if ((g.mask_rows && r >= L) || (g.mask_cols && c >= L)) v = 0.f;
            C[(long long)r * g.ldc + c] = v;
        }
    }
}

// C = sum over splits of part[split] (+ beta C), with the output masks, in split order.
__global__ void splitk_reduce_kernel(const GemmArgs g, long long units) {
    const long long mn = (long long)g.M * g.N;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= units * mn) return;
    const int z = (int)(i / mn);
    const long long e = i % mn;
    const int r = (int)(e / g.N), c = (int)(e % g.N);
    // column blocks (tensor-core product): block c / cblk of unit z blk_ua + block blk_ub
    const int blk = g.cblk > 0 ? c / g.cblk : 0, cc = g.cblk > 0 ? c % g.cblk : c;
    const int unit = g.cblk > 0 ? z * g.blk_ua + blk * g.blk_ub : z;
    const int L = unit_length(g.pad, unit, g.h, g.n);
    float v = 0.f;
    for (int sp = 0; sp < g.splits; ++sp) v += g.part[((long long)sp * units + z) * mn + e];
    float *C = g.C + (long long)z * g.sC + blk * g.cblk_stride + (long long)r * g.ldc + cc;
    if (g.beta != 0.f) v = fmaf(g.beta, *C, v);
    if ((g.mask_rows && r >= L) || (g.mask_cols && cc >= L)) v = 0.f;
    *C = v;
}

// Rows of S (units x rows_per_unit x cols, in place): softmax for rows i < L (over the
// columns j < L when mask_cols), zero for i >= L.  One warp per row; the first pass
// keeps a running maximum and a rescaled running sum, the second writes p.
__global__ void softmax_rows_kernel(float *S, const int32_t *pad, int h, int rows_per_unit,
                                    int cols, long long rows, int mask_cols) {
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const int z = (int)(row / rows_per_unit), i = (int)(row % rows_per_unit);
    int L = pad ? pad[z / h] : rows_per_unit;
    L = L < 0 ? 0 : (L > rows_per_unit ? rows_per_unit : L);
    float *s = S + row * cols;
    if (i >= L) {
        for (int j = lane; j < cols; j += 32) s[j] = 0.f;
        return;
    }
    const int live = mask_cols ? (L < cols ? L : cols) : cols;
    float m = -INFINITY, l = 0.f;
    for (int j = lane; j < live; j += 32) {
        const float v = s[j];
        if (v > m) {
            l = l * expf(m - v) + 1.f;
            m = v;
        } else {
            l += expf(v - m);
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const float lo = __shfl_xor_sync(0xffffffffu, l, o);
        const float mn = fmaxf(m, mo);
        l = (m == -INFINITY ? 0.f : l * expf(m - mn)) + (mo == -INFINITY ? 0.f : lo * expf(mo - mn));
        m = mn;
    }
    const float inv = 1.f / l;
    for (int j = lane; j < cols; j += 32) s[j] = j < live ? expf(s[j] - m) * inv : 0.f;
}

// Whether an operand's 4-element groups along its contiguous axis can be 16-byte
// loads: aligned base, strides and ld, and a contiguous extent that is a multiple of 4.
void set_vec(Operand &o, int contiguous_extent) {
    o.vec = (reinterpret_cast<uintptr_t>(o.p) & 15u) == 0 && o.ld % 4 == 0 &&
            (o.index == kShared || o.stride % 4 == 0) && contiguous_extent % 4 == 0;
}

template <int BM, int BN>
int launch_gemm(const GemmArgs &g, int units, cudaStream_t s, int kernel_id) {
    const long long gx = (long long)((g.N + BN - 1) / BN) * g.splits;
    dim3 grid((unsigned)gx, (unsigned)((g.M + BM - 1) / BM), (unsigned)units);
    if (gx > 0x7fffffffLL || grid.y > 65535u || grid.z > 65535u) return LINFORMER_ERR_SIZE;
    constexpr size_t smem = sizeof(float) * kStages * kBK * (BM + BN + 8);
    if (cudaFuncSetAttribute(batched_gemm_kernel<BM, BN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LINFORMER_ERR_LAUNCH;
    {
        KernelScope scope(kernel_id, s);
        batched_gemm_kernel<BM, BN><<<grid, kThreads, smem, s>>>(g);
    }
    if (g.splits > 1) {
        const long long total = (long long)units * g.M * g.N;
        KernelScope scope(kernel_id, s);
        splitk_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(g, units);
    }
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace

int launch_splitk_reduce(const GemmArgs &g, int units, cudaStream_t s, int kernel_id) {
    const long long total = (long long)units * g.M * g.N;
    KernelScope scope(kernel_id, s);
    splitk_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(g, units);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

void set_operand_vec(Operand &o, int contiguous_extent) { set_vec(o, contiguous_extent); }

int batched_gemm(GemmArgs g, int units, cudaStream_t s, float *part, int max_splits, int sms,
                 int kernel_id) {
    set_vec(g.A, g.A.xfast ? g.M : g.K);
    set_vec(g.B, g.B.xfast ? g.N : g.K);
    const int BM = g.M <= 64 ? 64 : 128, BN = (g.M <= 64 || g.N <= 64) ? 64 : 128;
    g.splits = 1;
    g.kchunk = (g.K + kBK - 1) / kBK * kBK;
    g.part = part;
    if (part && max_splits > 1) {
        const long long ctas = (long long)((g.N + BN - 1) / BN) * ((g.M + BM - 1) / BM) * units;
        long long want = (8LL * sms + ctas - 1) / ctas;
        want = std::min<long long>(want, std::min<long long>(max_splits, std::max(1, g.K / 256)));
        if (want > 1) {
            const int chunk = (g.K + (int)want - 1) / (int)want;
            g.kchunk = (chunk + kBK - 1) / kBK * kBK;
            g.splits = (g.K + g.kchunk - 1) / g.kchunk;
        }
    }
    if (BM == 64) return launch_gemm<64, 64>(g, units, s, kernel_id);
    if (BN == 64) return launch_gemm<128, 64>(g, units, s, kernel_id);
    return launch_gemm<128, 128>(g, units, s, kernel_id);
}


int softmax_rows(float *S, const int32_t *pad, int h, int rows_per_unit, int cols,
                 long long units, int mask_cols, cudaStream_t s, int kernel_id) {
    const long long rows = units * rows_per_unit;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return LINFORMER_ERR_SIZE;
    KernelScope scope(kernel_id, s);
    softmax_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(S, pad, h, rows_per_unit, cols, rows,
                                                       mask_cols);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

int project_f32(const Problem &p, float *Kbar, float *Vbar, float *part, int kernel_id,
                bool tensor) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k;
    const long long kd = (long long)k * d, nd = (long long)n * d, kn = (long long)k * n;
    const bool per_head = p.proj_per_head();
    const int pidx = per_head ? kPerHead : kShared;
    const int sms = sm_count();
    const float *K = static_cast<const float *>(p.K), *V = static_cast<const float *>(p.V);
    const float *E = static_cast<const float *>(p.E), *F = static_cast<const float *>(p.f_or_e());
    GemmArgs g{opA(E, kn, n, 0, pidx), opB(K, nd, d, 0, kPerUnit, 1), Kbar, kd, d, k, d, n, 1.f,
               0.f, p.pad, p.h, n, 0, 0, 1, 0, nullptr};
    int zcount = units;
    if (tensor && d % 32 == 0) {
        // the units sharing E side by side along N: E's tiles feed several units at once
        const int groups = per_head ? p.h : 1, ub = per_head ? p.h : 1;
        zcount = groups;
        g.N = (units / groups) * d;
        g.B.xblk = d;
        g.B.blk_stride = ub * nd;
        g.cblk = d;
        g.cblk_stride = ub * kd;
        g.blk_ua = per_head ? 1 : 0;
        g.blk_ub = ub;
    }
    auto product = [&](const GemmArgs &a) {
        return tensor ? tc_batched_gemm(a, zcount, p.stream, part,
                                        (size_t)kMaxSplits * units * kd, sms, kernel_id)
                      : batched_gemm(a, units, p.stream, part, kMaxSplits, sms, kernel_id);
    };
    int st = product(g);
    if (st) return st;
    g.A = opA(F, kn, n, 0, pidx);
    const Operand b = g.B;
    g.B = opB(V, nd, d, 0, kPerUnit, 1);
    g.B.xblk = b.xblk;
    g.B.blk_stride = b.blk_stride;
    g.C = Vbar;
    return product(g);
}

int attend_f32(const Problem &p, const float *Kbar, const float *Vbar, float *P,
               int kernel_id) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k;
    const long long kd = (long long)k * d, nd = (long long)n * d, nk = (long long)n * k;
    GemmArgs g{opA(static_cast<const float *>(p.Q), nd, d, 0, kPerUnit),
               opB(Kbar, kd, d, 1, kPerUnit), P, nk, k, n, k, d, 1.f / sqrtf((float)d), 0.f,
               p.pad, p.h, n, 0, 0, 1, 0, nullptr};
    int st = batched_gemm(g, units, p.stream, nullptr, 1, 0, kernel_id);
    if (!st) st = softmax_rows(P, p.pad, p.h, n, k, units, 0, p.stream, kernel_id);
    if (st) return st;
    g = GemmArgs{opA(P, nk, k, 0, kPerUnit), opB(Vbar, kd, d, 0, kPerUnit),
                 static_cast<float *>(p.O), nd, d, n, d, k, 1.f, 0.f, p.pad, p.h, n, 1, 0,
                 1, 0, nullptr};
    return batched_gemm(g, units, p.stream, nullptr, 1, 0, kernel_id);
}

int sm_count() {
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

}  // namespace simt
}  // namespace linformer
