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
// Kbar and Vbar are recomputed by the forward's projection kernel.  The products run
// on one batched SIMT matrix-product kernel; three small kernels do the softmax rows,
// the softmax backward rows and the sums over sharing groups.
#include "internal.cuh"

namespace linformer {
namespace {

constexpr int kBM = 64, kBN = 64, kBKt = 16;  // product tile: 64 x 64 outputs, 16-deep

__device__ __forceinline__ int unit_length(const int32_t *pad, int unit, int h, int n) {
    if (!pad) return n;
    const int L = pad[unit / h];
    return L < 0 ? 0 : (L > n ? n : L);
}

// Which matrix of a batched operand unit z reads: its own, its head's, or one shared.
enum OperandIndex { kPerUnit = 0, kPerHead = 1, kShared = 2 };

struct Operand {
    const float *p;
    long long stride;  // elements between consecutive matrices
    int ld;            // row stride of the stored matrix
    int trans;         // 1: the stored matrix is the transpose of the operand
    int index;         // OperandIndex
    int nmask;         // 1: operand rows >= L read as zero, 2: operand columns >= L (the
                       // sequence axis of Q, K, V, dO: padded rows may hold anything)
    __device__ __forceinline__ const float *mat(int z, int h) const {
        const int m = index == kPerUnit ? z : (index == kPerHead ? z % h : 0);
        return p + (long long)m * stride;
    }
    // element (r, c) of the operand
    __device__ __forceinline__ float at(const float *m, int r, int c) const {
        return trans ? m[(long long)c * ld + r] : m[(long long)r * ld + c];
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
};

// One 64 x 64 output tile of unit blockIdx.z per CTA, 256 threads, 4 x 4 outputs each.
__global__ void __launch_bounds__(256) batched_gemm_kernel(const GemmArgs g) {
    __shared__ float sA[kBKt][kBM + 1];
    __shared__ float sB[kBKt][kBN + 1];
    const int z = blockIdx.z, tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int row0 = blockIdx.y * kBM, col0 = blockIdx.x * kBN;
    const float *A = g.A.mat(z, g.h), *B = g.B.mat(z, g.h);
    const int L = unit_length(g.pad, z, g.h, g.n);
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += kBKt) {
        for (int i = threadIdx.x; i < kBKt * kBM; i += 256) {
            const int kk = i / kBM, r = i % kBM;
            const int gr = row0 + r, gk = k0 + kk;
            const bool in = gr < g.M && gk < g.K && !(g.A.nmask == 1 && gr >= L) &&
                            !(g.A.nmask == 2 && gk >= L);
            sA[kk][r] = in ? g.A.at(A, gr, gk) : 0.f;
        }
        for (int i = threadIdx.x; i < kBKt * kBN; i += 256) {
            const int kk = i / kBN, c = i % kBN;
            const int gc = col0 + c, gk = k0 + kk;
            const bool in = gc < g.N && gk < g.K && !(g.B.nmask == 1 && gk >= L) &&
                            !(g.B.nmask == 2 && gc >= L);
            sB[kk][c] = in ? g.B.at(B, gk, gc) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBKt; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sA[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = sB[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *C = g.C + (long long)z * g.sC;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + ty * 4 + i;
        if (r >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = col0 + tx * 4 + j;
            if (c >= g.N) continue;
            float v = g.alpha * acc[i][j];
            if (g.beta != 0.f) v = fmaf(g.beta, C[(long long)r * g.ldc + c], v);
            if ((g.mask_rows && r >= L) || (g.mask_cols && c >= L)) v = 0.f;
            C[(long long)r * g.ldc + c] = v;
        }
    }
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

int gemm(const GemmArgs &g, int units, cudaStream_t s) {
    dim3 grid((unsigned)((g.N + kBN - 1) / kBN), (unsigned)((g.M + kBM - 1) / kBM), (unsigned)units);
    if (grid.y > 65535u || grid.z > 65535u) return LINFORMER_ERR_SIZE;
    KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
    batched_gemm_kernel<<<grid, 256, 0, s>>>(g);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

Operand op(const float *p, long long stride, int ld, int trans, int index, int nmask = 0) {
    return Operand{p, stride, ld, trans, index, nmask};
}

}  // namespace

int simt_backward(const Problem &p, const float *dO, float *dQ, float *dK, float *dV, float *dE,
                  float *dF) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k, h = p.h;
    const bool per_head = p.proj_per_head(), distinct = p.distinct_f();
    const long long kd = (long long)k * d, nk = (long long)n * k, nd = (long long)n * d,
                    kn = (long long)k * n;
    const size_t bytes = sizeof(float) * ((size_t)units * (4 * kd + 2 * nk + kn * (distinct ? 2 : 1)));
    void *ws = nullptr;
    if (workspace_alloc(&ws, bytes, p.stream) != LINFORMER_OK) return LINFORMER_ERR_ALLOC;
    float *Kb = static_cast<float *>(ws), *Vb = Kb + units * kd;
    float *P = Vb + units * kd, *dS = P + units * nk;
    float *dKb = dS + units * nk, *dVb = dKb + units * kd;
    float *gE = dVb + units * kd, *gF = distinct ? gE + units * kn : gE;
    const float *Q = static_cast<const float *>(p.Q), *K = static_cast<const float *>(p.K),
                *V = static_cast<const float *>(p.V), *E = static_cast<const float *>(p.E),
                *F = static_cast<const float *>(p.f_or_e());
    const int pidx = per_head ? kPerHead : kShared;
    const float scale = 1.f / sqrtf((float)d);
    cudaStream_t s = p.stream;
    auto args = [&](Operand A, Operand B, float *C, long long sC, int ldc, int M, int N, int K_,
                    float alpha, float beta, int mrows, int mcols) {
        return GemmArgs{A, B, C, sC, ldc, M, N, K_, alpha, beta, p.pad, h, n, mrows, mcols};
    };
    int st = simt_project(p, Kb, Vb);
    // S = Q Kbar^T / sqrt(d), then P (rows >= L zero)
    if (!st) st = gemm(args(op(Q, nd, d, 0, kPerUnit), op(Kb, kd, d, 1, kPerUnit), P, nk, k, n, k,
                            d, scale, 0.f, 0, 0), units, s);
    const long long rows = (long long)units * n;
    const unsigned rblocks = (unsigned)((rows + 7) / 8);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        softmax_rows_kernel<<<rblocks, 256, 0, s>>>(P, p.pad, h, n, k, rows);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    // dP = dO Vbar^T, then dS in place
    if (!st) st = gemm(args(op(dO, nd, d, 0, kPerUnit, 1), op(Vb, kd, d, 1, kPerUnit), dS, nk, k,
                            n, k, d, 1.f, 0.f, 0, 0), units, s);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        softmax_bwd_rows_kernel<<<rblocks, 256, 0, s>>>(P, dS, k, rows);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    // dVbar = P^T dO; dQ = dS Kbar / sqrt(d); dKbar = dS^T Q / sqrt(d)
    if (!st) st = gemm(args(op(P, nk, k, 1, kPerUnit), op(dO, nd, d, 0, kPerUnit, 1), dVb, kd, d,
                            k, d, n, 1.f, 0.f, 0, 0), units, s);
    if (!st) st = gemm(args(op(dS, nk, k, 0, kPerUnit), op(Kb, kd, d, 0, kPerUnit), dQ, nd, d, n,
                            d, k, scale, 0.f, 1, 0), units, s);
    if (!st) st = gemm(args(op(dS, nk, k, 1, kPerUnit), op(Q, nd, d, 0, kPerUnit, 1), dKb, kd, d,
                            k, d, n, scale, 0.f, 0, 0), units, s);
    // dK = E^T dKbar, dV = F^T dVbar (rows >= L zero)
    if (!st) st = gemm(args(op(E, kn, n, 1, pidx), op(dKb, kd, d, 0, kPerUnit), dK, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    if (!st) st = gemm(args(op(F, kn, n, 1, pidx), op(dVb, kd, d, 0, kPerUnit), dV, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    // per-unit E (and F) terms, columns t >= L zero, then the sums over sharing groups
    if (!st) st = gemm(args(op(dKb, kd, d, 0, kPerUnit), op(K, nd, d, 1, kPerUnit, 2), gE, kn, n,
                            k, n, d, 1.f, 0.f, 0, 1), units, s);
    if (!st) st = gemm(args(op(dVb, kd, d, 0, kPerUnit), op(V, nd, d, 1, kPerUnit, 2), gF, kn, n,
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
