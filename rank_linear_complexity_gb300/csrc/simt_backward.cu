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
// Every product, Kbar and Vbar included, runs on the batched SIMT matrix product of
// simt_gemm.cu (split over the sequence for the four k x d results that sum over it);
// two kernels here do the softmax backward rows and the sums over sharing groups.
#include "simt_gemm.cuh"

namespace linformer {
namespace {

using namespace simt;

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

}  // namespace

int simt_backward(const Problem &p, const float *dO, float *dQ, float *dK, float *dV, float *dE,
                  float *dF) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k, h = p.h;
    const bool per_head = p.proj_per_head(), distinct = p.distinct_f();
    const long long kd = (long long)k * d, nk = (long long)n * k, nd = (long long)n * d,
                    kn = (long long)k * n;
    // split-K partials of the four k x d products that sum over the sequence
    const int sms = sm_count();
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
    int st = project_f32(p, Kb, Vb, part, LINFORMER_KERNEL_BACKWARD);
    // S = Q Kbar^T / sqrt(d), then P (rows >= L zero)
    if (!st) st = batched_gemm(args(opA(Q, nd, d, 0, kPerUnit), opB(Kb, kd, d, 1, kPerUnit), P, nk, k, n, k,
                            d, scale, 0.f, 0, 0), units, s);
    const long long rows = (long long)units * n;
    const unsigned rblocks = (unsigned)((rows + 7) / 8);
    if (!st) st = softmax_rows(P, p.pad, h, n, k, units, 0, s);
    // dP = dO Vbar^T, then dS in place
    if (!st) st = batched_gemm(args(opA(dO, nd, d, 0, kPerUnit, 1), opB(Vb, kd, d, 1, kPerUnit), dS, nk, k,
                            n, k, d, 1.f, 0.f, 0, 0), units, s);
    if (!st) {
        KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
        softmax_bwd_rows_kernel<<<rblocks, 256, 0, s>>>(P, dS, k, rows);
        if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
    }
    // dVbar = P^T dO; dQ = dS Kbar / sqrt(d); dKbar = dS^T Q / sqrt(d)
    if (!st) st = batched_gemm(args(opA(P, nk, k, 1, kPerUnit), opB(dO, nd, d, 0, kPerUnit, 1), dVb, kd, d,
                            k, d, n, 1.f, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    if (!st) st = batched_gemm(args(opA(dS, nk, k, 0, kPerUnit), opB(Kb, kd, d, 0, kPerUnit), dQ, nd, d, n,
                            d, k, scale, 0.f, 1, 0), units, s);
    if (!st) st = batched_gemm(args(opA(dS, nk, k, 1, kPerUnit), opB(Q, nd, d, 0, kPerUnit, 1), dKb, kd, d,
                            k, d, n, scale, 0.f, 0, 0), units, s, part, kMaxSplits, sms);
    // dK = E^T dKbar, dV = F^T dVbar (rows >= L zero)
    if (!st) st = batched_gemm(args(opA(E, kn, n, 1, pidx), opB(dKb, kd, d, 0, kPerUnit), dK, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    if (!st) st = batched_gemm(args(opA(F, kn, n, 1, pidx), opB(dVb, kd, d, 0, kPerUnit), dV, nd, d, n, d, k,
                            1.f, 0.f, 1, 0), units, s);
    // per-unit E (and F) terms, columns t >= L zero, then the sums over sharing groups
    if (!st) st = batched_gemm(args(opA(dKb, kd, d, 0, kPerUnit), opB(K, nd, d, 1, kPerUnit, 2), gE, kn, n,
                            k, n, d, 1.f, 0.f, 0, 1), units, s);
    if (!st) st = batched_gemm(args(opA(dVb, kd, d, 0, kPerUnit), opB(V, nd, d, 1, kPerUnit, 2), gF, kn, n,
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
