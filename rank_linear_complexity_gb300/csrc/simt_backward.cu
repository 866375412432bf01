// Backward of the Linformer attention forward in fp32 (SIMT): the gradients of O with
// respect to Q, K, V, E and F given dO.  The forward is the definition in "Linformer
// (Self-Attention with Linear Complexity) 요약 설명", section Model (Kbar = E.K,
// Vbar = F.V, E and F of shape k x n; rows t >= L of K and V count as zero and query
// rows i >= L give O = 0, padding paragraph), with the scaled dot product; the pages
// train models with it (section Experiments), and its gradients are the chain rule
// through that definition:
//   P = softmax(Q Kbar^T / sqrt(d)) (rows >= L zero)       O = P Vbar
//   dVbar = P^T dO                 dP = dO Vbar^T            dS = P * (dP - rowsum(P * dP))
//   dQ = dS Kbar / sqrt(d)         dKbar = dS^T Q / sqrt(d)
//   dK = E^T dKbar, dV = F^T dVbar (rows >= L zero)
//   dE = sum over the units sharing E of dKbar K^T (+ dVbar V^T when F is E), dF alike,
//   with the columns t >= L of each unit's term zero.
// Every product, Kbar and Vbar included, runs on one batched SIMT matrix-product
// kernel (split over the sequence for the four k x d results that sum over it); small
// kernels do the split sums, the softmax rows, the softmax backward rows and the sums
// over sharing groups.
#include <algorithm>

#include "internal.cuh"

namespace linformer {
namespace {

constexpr int kBK = 16;        // depth of one product step
constexpr int kThreads = 256;  // 16 x 16 threads, each owning (BM/16) x (BN/16) outputs

__device__ __forceinline__ int unit_length(const int32_t *pad, int unit, int h, int n) {
    if (!pad) return n;
    const int L = pad[unit / h];
    return L < 0 ? 0 : (L > n ? n : L);
}

// Which matrix of a batched operand unit z reads: its own, its head's, or one shared.
enum OperandIndex { kPerUnit = 0, kPerHead = 1, kShared = 2 };

// One operand of the batched product, seen as X x K (X = M for A, N for B): element
// (x, kk) is stored at m[kk * ld + x] when xfast (x contiguous) else m[x * ld + kk].
struct Operand {
    const float *p;
    long long stride;  // elements between consecutive matrices
    int ld;            // row stride of the stored matrix
    int xfast;         // 1: the x index is the contiguous one in memory
    int index;         // OperandIndex
    int mask_x, mask_k;  // 1: x (resp. kk) >= the unit's length reads as zero (the
                         // sequence axis of Q, K, V, dO: padded rows may hold anything)
    int vec;           // 1: 4-element groups along the contiguous axis are 16-byte loads
    __device__ __forceinline__ const float *mat(int z, int h) const {
        const int m = index == kPerUnit ? z : (index == kPerHead ? z % h : 0);
        return p + (long long)m * stride;
    }
};

struct GemmArgs {
    Operand A, B;  // C (M x N) = alpha A (M x K) B (K x N) + beta C
    float *C;
    long long sC;
    int ldc, M, N, K;
    float alpha, beta;
    const int32_t *pad;
    int h, n;
    int mask_rows, mask_cols;  // output rows / columns at or past the unit's length: zero
    // Split of the K range over `splits` CTAs of kchunk (a multiple of kBK) each; with
    // splits > 1 each CTA writes alpha times its partial product to part[split][z]
    // (M x N, dense) and splitk_reduce_kernel forms C.
    int splits, kchunk;
    float *part;
};

// Register staging of one BX x kBK operand tile: BX / 16 elements per thread, taken as
// groups of four along the contiguous axis (a group is wholly in or out of range
// when vec is set: the contiguous extent is then a multiple of four).
template <int BX>
struct Stage {
    static constexpr int kGroups = BX / 64;  // groups of four per thread
    float v[kGroups][4];

    __device__ __forceinline__ void load(const Operand &o, const float *m, int x0, int k0, int X,
                                         int K, int L) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            const int idx = threadIdx.x + g * kThreads;
            int x, kk;
            if (o.xfast) {
                x = x0 + (idx % (BX / 4)) * 4;
                kk = k0 + idx / (BX / 4);
            } else {
                x = x0 + idx / (kBK / 4);
                kk = k0 + (idx % (kBK / 4)) * 4;
            }
            if (o.vec) {
                const bool in = x < X && kk < K;
                float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in) {
                    const long long off = o.xfast ? (long long)kk * o.ld + x : (long long)x * o.ld + kk;
                    q = __ldg(reinterpret_cast<const float4 *>(m + off));
                }
                v[g][0] = q.x;
                v[g][1] = q.y;
                v[g][2] = q.z;
                v[g][3] = q.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int xe = o.xfast ? x + e : x, ke = o.xfast ? kk : kk + e;
                    v[g][e] = (xe < X && ke < K)
                                  ? __ldg(m + (o.xfast ? (long long)ke * o.ld + xe
                                                       : (long long)xe * o.ld + ke))
                                  : 0.f;
                }
            }
            if (o.mask_x | o.mask_k) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int xe = o.xfast ? x + e : x, ke = o.xfast ? kk : kk + e;
                    if ((o.mask_x && xe >= L) || (o.mask_k && ke >= L)) v[g][e] = 0.f;
                }
            }
        }
    }

    // into s[kk][x] (row stride BX + 4)
    __device__ __forceinline__ void store(const Operand &o, float *s) const {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            const int idx = threadIdx.x + g * kThreads;
            if (o.xfast) {
                const int x = (idx % (BX / 4)) * 4, kk = idx / (BX / 4);
                *reinterpret_cast<float4 *>(s + kk * (BX + 4) + x) =
                    make_float4(v[g][0], v[g][1], v[g][2], v[g][3]);
            } else {
                const int x = idx / (kBK / 4), kk = (idx % (kBK / 4)) * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) s[(kk + e) * (BX + 4) + x] = v[g][e];
            }
        }
    }
};

// One BM x BN output tile of unit blockIdx.z per CTA.  Thread (tx, ty) owns rows
// ty*4 + {0..3} (+ 64, + 128 ... for BM > 64) and columns tx*4 + {0..3} (+ 64 ...), so
// its shared-memory reads are 16-byte loads that a warp serves in two passes.  The
// next tile's global loads are in registers while the current one is multiplied.
template <int BM, int BN>
__global__ void __launch_bounds__(kThreads, 2) batched_gemm_kernel(const GemmArgs g) {
    constexpr int TM = BM / 16, TN = BN / 16;
    __shared__ __align__(16) float sA[2][kBK * (BM + 4)];
    __shared__ __align__(16) float sB[2][kBK * (BN + 4)];
    const int z = blockIdx.z, tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int tiles_n = gridDim.x / g.splits, split = blockIdx.x / tiles_n;
    const int row0 = blockIdx.y * BM, col0 = (blockIdx.x % tiles_n) * BN;
    const int kbeg = split * g.kchunk, kend = min(g.K, kbeg + g.kchunk);
    const float *A = g.A.mat(z, g.h), *B = g.B.mat(z, g.h);
    const int L = unit_length(g.pad, z, g.h, g.n);
    Stage<BM> ra;
    Stage<BN> rb;
    float acc[TM][TN] = {};
    ra.load(g.A, A, row0, kbeg, g.M, kend, L);
    rb.load(g.B, B, col0, kbeg, g.N, kend, L);
    ra.store(g.A, sA[0]);
    rb.store(g.B, sB[0]);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += kBK) {
        const bool more = k0 + kBK < kend;
        if (more) {
            ra.load(g.A, A, row0, k0 + kBK, g.M, kend, L);
            rb.load(g.B, B, col0, k0 + kBK, g.N, kend, L);
        }
        const float *a_s = sA[buf], *b_s = sB[buf];
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
        if (more) {
            buf ^= 1;
            ra.store(g.A, sA[buf]);
            rb.store(g.B, sB[buf]);
        }
        __syncthreads();
    }
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
    const int L = unit_length(g.pad, z, g.h, g.n);
    float v = 0.f;
    for (int sp = 0; sp < g.splits; ++sp) v += g.part[((long long)sp * units + z) * mn + e];
    float *C = g.C + (long long)z * g.sC + (long long)r * g.ldc + c;
    if (g.beta != 0.f) v = fmaf(g.beta, *C, v);
    if ((g.mask_rows && r >= L) || (g.mask_cols && c >= L)) v = 0.f;
    *C = v;
}

// Rows of S (units x n x k, in place): softmax for rows i < L, zero for i >= L.
// One warp per row.
__global__ void softmax_rows_kernel(float *S, const int32_t *pad, int h, int n, int k,
                                    long long rows) {
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const int z = (int)(row / n), i = (int)(row % n);
    float *s = S + row * k;
    if (i >= unit_length(pad, z, h, n)) {
        for (int j = lane; j < k; j += 32) s[j] = 0.f;
        return;
    }
    float m = -INFINITY;
    for (int j = lane; j < k; j += 32) m = fmaxf(m, s[j]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int j = lane; j < k; j += 32) {
        const float e = expf(s[j] - m);
        s[j] = e;
        l += e;
    }
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const float inv = 1.f / l;
    for (int j = lane; j < k; j += 32) s[j] *= inv;
}

// dS = P * (dP - sum_j P dP) row by row, in place over dP.  One warp per row.
__global__ void softmax_bwd_rows_kernel(const float *P, float *dP, int k, long long rows) {
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const float *p = P + row * k;
    float *g = dP + row * k;
    float dsum = 0.f;
    for (int j = lane; j < k; j += 32) dsum = fmaf(p[j], g[j], dsum);
    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    for (int j = lane; j < k; j += 32) g[j] = p[j] * (g[j] - dsum);
}

// out[m] = sum over the units sharing matrix m of per_unit[unit] (k x n each), in unit
// order; per_head: matrix m = head, units b*h + m; else one matrix for all units.
__global__ void group_sum_kernel(const float *per_unit, float *out, int b, int h, int per_head,
                                 long long elems) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int groups = per_head ? h : 1;
    if (i >= elems * groups) return;
    const int m = (int)(i / elems);
    const long long e = i % elems;
    float acc = 0.f;
    if (per_head) {
        for (int bi = 0; bi < b; ++bi) acc += per_unit[((long long)bi * h + m) * elems + e];
    } else {
        for (long long z = 0; z < (long long)b * h; ++z) acc += per_unit[z * elems + e];
    }
    out[i] = acc;
}

// Whether an operand's 4-element groups along its contiguous axis can be 16-byte
// loads: aligned base, strides and ld, and a contiguous extent that is a multiple of 4.
void set_vec(Operand &o, int contiguous_extent) {
    o.vec = (reinterpret_cast<uintptr_t>(o.p) & 15u) == 0 && o.ld % 4 == 0 &&
            (o.index == kShared || o.stride % 4 == 0) && contiguous_extent % 4 == 0;
}

template <int BM, int BN>
int launch_gemm(const GemmArgs &g, int units, cudaStream_t s) {
    const long long gx = (long long)((g.N + BN - 1) / BN) * g.splits;
    dim3 grid((unsigned)gx, (unsigned)((g.M + BM - 1) / BM), (unsigned)units);
    if (gx > 0x7fffffffLL || grid.y > 65535u || grid.z > 65535u) return LINFORMER_ERR_SIZE;
    {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        batched_gemm_kernel<BM, BN><<<grid, kThreads, 0, s>>>(g);
    }
    if (g.splits > 1) {
        const long long total = (long long)units * g.M * g.N;
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        splitk_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(g, units);
    }
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

// splits = 1 unless part is given: then enough K splits (each at least 256 deep) for
// about eight CTAs per SM, at most max_splits.
int gemm(GemmArgs g, int units, cudaStream_t s, float *part = nullptr, int max_splits = 1,
         int sms = 0) {
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
    if (BM == 64) return launch_gemm<64, 64>(g, units, s);
    if (BN == 64) return launch_gemm<128, 64>(g, units, s);
    return launch_gemm<128, 128>(g, units, s);
}

// Operand A (M x K) or B (K x N) of a product from a stored row-major matrix: `trans`
// says the stored matrix is the operand's transpose; nmask 1 zeroes operand rows >= L,
// 2 operand columns >= L.
Operand opA(const float *p, long long stride, int ld, int trans, int index, int nmask = 0) {
    return Operand{p, stride, ld, trans, index, nmask == 1, nmask == 2, 0};
}
Operand opB(const float *p, long long stride, int ld, int trans, int index, int nmask = 0) {
    return Operand{p, stride, ld, !trans, index, nmask == 2, nmask == 1, 0};
}

}  // namespace

int simt_backward(const Problem &p, const float *dO, float *dQ, float *dK, float *dV, float *dE,
                  float *dF) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k, h = p.h;
    const bool per_head = p.proj_per_head(), distinct = p.distinct_f();
    const long long kd = (long long)k * d, nk = (long long)n * k, nd = (long long)n * d,
                    kn = (long long)k * n;
    // split-K partials of the four k x d products that sum over the sequence
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    sms = sms > 0 ? sms : 148;
    constexpr int kMaxSplits = 8;
    const size_t bytes = sizeof(float) * ((size_t)units * (4 * kd + 2 * nk + kn * (distinct ? 2 : 1)) +
                                          (size_t)kMaxSplits * units * kd);
    void *ws = nullptr;
    if (workspace_alloc(&ws, bytes, p.stream) != LINFORMER_OK) return LINFORMER_ERR_ALLOC;
    float *Kb = static_cast<float *>(ws), *Vb = Kb + units * kd;
    float *P = Vb + units * kd, *dS = P + units * nk;
    float *dKb = dS + units * nk, *dVb = dKb + units * kd;
    float *gE = dVb + units * kd, *gF = distinct ? gE + units * kn : gE;
    float *part = gF + units * kn;
    const float *Q = static_cast<const float *>(p.Q), *K = static_cast<const float *>(p.K),
                *V = static_cast<const float *>(p.V), *E = static_cast<const float *>(p.E),
                *F = static_cast<const float *>(p.f_or_e());
    const int pidx = per_head ? kPerHead : kShared;
    const float scale = 1.f / sqrtf((float)d);
    cudaStream_t s = p.stream;
    auto args = [&](Operand A, Operand B, float *C, long long sC, int ldc, int M, int N, int K_,
                    float alpha, float beta, int mrows, int mcols) {
        return GemmArgs{A, B, C, sC, ldc, M, N, K_, alpha, beta, p.pad, h, n, mrows, mcols,
                        1, 0, nullptr};
    };
    // Kbar = E K, Vbar = F V over rows t < L
    int st = gemm(args(opA(E, kn, n, 0, pidx), opB(K, nd, d, 0, kPerUnit, 1), Kb, kd, d, k, d, n,
                       1.f, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    if (!st) st = gemm(args(opA(F, kn, n, 0, pidx), opB(V, nd, d, 0, kPerUnit, 1), Vb, kd, d, k, d,
                            n, 1.f, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    // S = Q Kbar^T / sqrt(d), then P (rows >= L zero)
    if (!st) st = gemm(args(opA(Q, nd, d, 0, kPerUnit), opB(Kb, kd, d, 1, kPerUnit), P, nk, k, n, k,
                            d, scale, 0.f, 0, 0), units, s);
    const long long rows = (long long)units * n;
    const unsigned rblocks = (unsigned)((rows + 7) / 8);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        softmax_rows_kernel<<<rblocks, 256, 0, s>>>(P, p.pad, h, n, k, rows);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    // dP = dO Vbar^T, then dS in place
    if (!st) st = gemm(args(opA(dO, nd, d, 0, kPerUnit, 1), opB(Vb, kd, d, 1, kPerUnit), dS, nk, k,
                            n, k, d, 1.f, 0.f, 0, 0), units, s);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        softmax_bwd_rows_kernel<<<rblocks, 256, 0, s>>>(P, dS, k, rows);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    // dVbar = P^T dO; dQ = dS Kbar / sqrt(d); dKbar = dS^T Q / sqrt(d)
    if (!st) st = gemm(args(opA(P, nk, k, 1, kPerUnit), opB(dO, nd, d, 0, kPerUnit, 1), dVb, kd, d,
                            k, d, n, 1.f, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    if (!st) st = gemm(args(opA(dS, nk, k, 0, kPerUnit), opB(Kb, kd, d, 0, kPerUnit), dQ, nd, d, n,
                            d, k, scale, 0.f, 1, 0), units, s);
    if (!st) st = gemm(args(opA(dS, nk, k, 1, kPerUnit), opB(Q, nd, d, 0, kPerUnit, 1), dKb, kd, d,
                            k, d, n, scale, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    // dK = E^T dKbar, dV = F^T dVbar (rows >= L zero)
    if (!st) st = gemm(args(opA(E, kn, n, 1, pidx), opB(dKb, kd, d, 0, kPerUnit), dK, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    if (!st) st = gemm(args(opA(F, kn, n, 1, pidx), opB(dVb, kd, d, 0, kPerUnit), dV, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    // per-unit E (and F) terms, columns t >= L zero, then the sums over sharing groups
    if (!st) st = gemm(args(opA(dKb, kd, d, 0, kPerUnit), opB(K, nd, d, 1, kPerUnit, 2), gE, kn, n,
                            k, n, d, 1.f, 0.f, 0, 1), units, s);
    if (!st) st = gemm(args(opA(dVb, kd, d, 0, kPerUnit), opB(V, nd, d, 1, kPerUnit, 2), gF, kn, n,
                            k, n, d, 1.f, distinct ? 0.f : 1.f, 0, 1), units, s);
    const long long groups = per_head ? h : 1;
    const unsigned gblocks = (unsigned)((groups * kn + 255) / 256);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        group_sum_kernel<<<gblocks, 256, 0, s>>>(gE, dE, p.b, h, per_head ? 1 : 0, kn);
        if (distinct) group_sum_kernel<<<gblocks, 256, 0, s>>>(gF, dF, p.b, h, per_head ? 1 : 0, kn);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    workspace_free(ws, s);
    return st;
}

}  // namespace linformer
