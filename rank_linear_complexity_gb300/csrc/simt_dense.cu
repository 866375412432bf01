// Dense softmax attention in fp32, the full-attention counterpart the Linformer pages
// time their method against ("Linformer 요약 설명", section Inference-time Efficiency
// Results: the standard Transformer on the same GPU, compared by time and by the
// largest batch that fits): O = softmax(Q K^T / sqrt(d)) V with the n x n score matrix
// of every unit held in device memory, as the standard implementation holds it.
// Padding follows the usual key mask: keys t >= L take no part in any row's softmax
// and query rows i >= L give O = 0.  The two products run on the batched SIMT
// matrix-product kernel and the softmax on its row kernel (simt_gemm.cu).
#include "simt_gemm.cuh"

namespace linformer {

using namespace simt;

int simt_dense_attention(const Problem &p) {
    const int units = (int)p.units(), n = p.n, d = p.d, h = p.h;
    const long long nn = (long long)n * n, nd = (long long)n * d;
    void *ws = nullptr;
    if (workspace_alloc(&ws, sizeof(float) * (size_t)units * nn, p.stream) != LINFORMER_OK)
        return LINFORMER_ERR_ALLOC;
    float *S = static_cast<float *>(ws);
    const float *Q = static_cast<const float *>(p.Q), *K = static_cast<const float *>(p.K),
                *V = static_cast<const float *>(p.V);
    float *O = static_cast<float *>(p.O);
    const int id = LINFORMER_KERNEL_DENSE;
    // S = Q K^T / sqrt(d)
    GemmArgs g{opA(Q, nd, d, 0, kPerUnit), opB(K, nd, d, 1, kPerUnit), S, nn, n, n, n, d,
               1.f / sqrtf((float)d), 0.f, p.pad, h, n, 0, 0, 1, 0, nullptr};
    int st = batched_gemm(g, units, p.stream, nullptr, 1, 0, id);
    // P = softmax over the keys t < L, rows i >= L zero
    if (!st) st = softmax_rows(S, p.pad, h, n, n, units, 1, p.stream, id);
    // O = P V (V rows t >= L read as zero; P is zero there already), rows i >= L zero
    if (!st) {
        g = GemmArgs{opA(S, nn, n, 0, kPerUnit), opB(V, nd, d, 0, kPerUnit, 1), O, nd, d, n, d, n,
                     1.f, 0.f, p.pad, h, n, 1, 0, 1, 0, nullptr};
        st = batched_gemm(g, units, p.stream, nullptr, 1, 0, id);
    }
    workspace_free(ws, p.stream);
    return st;
}

}  // namespace linformer
