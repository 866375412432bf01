// Backward of the Linformer attention forward in fp32: the gradients of O with respect
// to Q, K, V, E and F given dO.  The forward is the definition in "Linformer
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
// Every product, Kbar and Vbar included, runs on the batched tensor-core product of
// tc_gemm.cu (fp32 operands split into bf16 hi + lo, three products, fp32 accumulation):
// split over the sequence for the four k x d results that sum over it; with k <= 256
// S and dP of a row tile as one work item whose epilogue writes P and dS (else the row
// softmax of simt_gemm.cu and the row kernel here); Kbar, Vbar, dK and dV with the
// units sharing E or F side by side; dE and dF as sums over units inside the product,
// in chunks of units whose partials are then added.
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

}  // namespace

int simt_backward(const Problem &p, const float *dO, float *dQ, float *dK, float *dV, float *dE,
                  float *dF) {
    const int units = (int)p.units(), n = p.n, d = p.d, k = p.k, h = p.h;
    const bool per_head = p.proj_per_head(), distinct = p.distinct_f();
    const long long kd = (long long)k * d, nk = (long long)n * k, nd = (long long)n * d,
                    kn = (long long)k * n;
    const int sms = sm_count();
    // Kbar, Vbar, dKbar, dVbar, P, dS, and the split-K partials of the k x d products
    const size_t part_floats = (size_t)kMaxSplits * units * kd;
    const size_t bytes = sizeof(float) * ((size_t)units * (4 * kd + 2 * nk) + part_floats);
    void *ws = nullptr;
    if (workspace_alloc(&ws, bytes, p.stream) != LINFORMER_OK) return LINFORMER_ERR_ALLOC;
    float *Kb = static_cast<float *>(ws), *Vb = Kb + units * kd;
    float *dKb = Vb + units * kd, *dVb = dKb + units * kd;
    float *P = dVb + units * kd, *dS = P + units * nk;
    float *part = dS + units * nk;
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
    // Row forms fused into the products' epilogues while a tile holds whole rows
    const bool fused = k <= 256;
    // Kbar = E K, Vbar = F V over rows t < L
    int st = project_f32(p, Kb, Vb, part, LINFORMER_KERNEL_BACKWARD, true);
    // P = softmax(Q Kbar^T / sqrt(d)) (rows >= L zero); dP = dO Vbar^T and
    // dS = P * (dP - rowsum(P * dP)): with k <= 256 both products of a row tile in one
    // work item, P and dS formed together in its epilogue
    GemmArgs gs = args(opA(Q, nd, d, 0, kPerUnit), opB(Kb, kd, d, 1, kPerUnit), P, nk, k, n, k, d,
                       scale, 0.f, 0, 0);
    const Operand dOa = opA(dO, nd, d, 0, kPerUnit, 1), Vbb = opB(Vb, kd, d, 1, kPerUnit);
    if (fused) {
        gs.epi = kEpiSoftmaxPair;
        gs.A2 = dOa;
        gs.B2 = Vbb;
        gs.C2 = dS;
        gs.alpha2 = 1.f;
        if (!st) st = tc_batched_gemm(gs, units, s, nullptr, 0, sms);
    } else {
        if (!st) st = tc_batched_gemm(gs, units, s, nullptr, 0, sms);
        if (!st) st = softmax_rows(P, p.pad, h, n, k, units, 0, s);
        if (!st) st = tc_batched_gemm(args(dOa, Vbb, dS, nk, k, n, k, d, 1.f, 0.f, 0, 0), units, s,
                                      nullptr, 0, sms);
        if (!st) {
            const long long rows = (long long)units * n;
            KernelScope scope(LINFORMER_KERNEL_BACKWARD, s);
            softmax_bwd_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(P, dS, k, rows);
            if (cudaPeekAtLastError() != cudaSuccess) st = LINFORMER_ERR_LAUNCH;
        }
    }
    // dVbar = P^T dO; dQ = dS Kbar / sqrt(d); dKbar = dS^T Q / sqrt(d)
    if (!st) st = tc_batched_gemm(args(opA(P, nk, k, 1, kPerUnit), opB(dO, nd, d, 0, kPerUnit, 1), dVb,
                                       kd, d, k, d, n, 1.f, 0.f, 0, 0),
                                  units, s, part, part_floats, sms);
    if (!st) st = tc_batched_gemm(args(opA(dS, nk, k, 0, kPerUnit), opB(Kb, kd, d, 0, kPerUnit), dQ, nd,
                                       d, n, d, k, scale, 0.f, 1, 0),
                                  units, s, nullptr, 0, sms);
    if (!st) st = tc_batched_gemm(args(opA(dS, nk, k, 1, kPerUnit), opB(Q, nd, d, 0, kPerUnit, 1), dKb,
                                       kd, d, k, d, n, scale, 0.f, 0, 0),
                                  units, s, part, part_floats, sms);
    // dK = E^T dKbar, dV = F^T dVbar (rows >= L zero); with d a multiple of 32 the units
    // sharing E (F) side by side along N
    auto project_back = [&](const float *X, const float *dXb, float *dX) {
        GemmArgs g = args(opA(X, kn, n, 1, pidx), opB(dXb, kd, d, 0, kPerUnit), dX, nd, d, n, d, k,
                          1.f, 0.f, 1, 0);
        int zcount = units;
        if (d % 32 == 0) {
            const int groups = per_head ? h : 1, ub = per_head ? h : 1;
            zcount = groups;
            g.N = (units / groups) * d;
            g.B.xblk = d;
            g.B.blk_stride = ub * kd;
            g.cblk = d;
            g.cblk_stride = ub * nd;
            g.blk_ua = per_head ? 1 : 0;
            g.blk_ub = ub;
        }
        return tc_batched_gemm(g, zcount, s, nullptr, 0, sms);
    };
    if (!st) st = project_back(E, dKb, dK);
    if (!st) st = project_back(F, dVb, dV);
    // dE (and dF) = the sum over the units sharing the matrix of dKbar K^T (dVbar V^T),
    // columns t >= L of each unit's term zero; P and dS, no longer needed, hold the
    // partial sums.
    const int groups = per_head ? h : 1, per_group = per_head ? p.b : units;
    auto grad = [&](float *out, const float *dX, const float *X, const float *dX2,
                    const float *X2) {
        GemmArgs g = args(opA(dX, kd, d, 0, kPerUnit), opB(X, nd, d, 1, kPerUnit, 2), out, kn, n, k,
                          n, d, 1.f, 0.f, 0, 0);
        g.usum_groups = groups;
        g.usum_per_group = per_group;
        g.usum_ga = per_head ? 1 : 0;
        g.usum_gb = per_head ? h : 1;
        if (dX2) {
            g.A2 = opA(dX2, kd, d, 0, kPerUnit);
            g.B2 = opB(X2, nd, d, 1, kPerUnit, 2);
        }
        return tc_batched_gemm(g, units, s, P, (size_t)2 * units * nk, sms);
    };
    if (!st) st = distinct ? grad(dE, dKb, K, nullptr, nullptr) : grad(dE, dKb, K, dVb, V);
    if (!st && distinct) st = grad(dF, dVb, V, nullptr, nullptr);
    workspace_free(ws, s);
    return st;
}

}  // namespace linformer
