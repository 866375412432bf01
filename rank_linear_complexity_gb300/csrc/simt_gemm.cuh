// Batched fp32 SIMT matrix products and row softmax shared by the backward and the
// dense attention: C_z = alpha A_z B_z + beta C_z over units z, each operand read from a
// row-major matrix of its own unit, of its head, or shared, with optional zeroing of
// the rows or columns at or past the unit's sequence length.
#pragma once

#include "internal.cuh"

namespace linformer {
namespace simt {

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
    const int32_t *pad;  // unit z has length pad[z / h] clamped to [0, n] (n if NULL)
    int h, n;
    int mask_rows, mask_cols;  // output rows / columns at or past the unit's length: zero
    // Split of the K range over `splits` CTAs of kchunk (a multiple of 16) each; with
    // splits > 1 each CTA writes alpha times its partial product to part[split][z]
    // (M x N, dense) and a second kernel forms C.  Set by batched_gemm.
    int splits, kchunk;
    float *part;
};

// Operand A (M x K) or B (K x N) of a product from a stored row-major matrix: `trans`
// says the stored matrix is the operand's transpose; nmask 1 zeroes operand rows >= L,
// 2 operand columns >= L.
inline Operand opA(const float *p, long long stride, int ld, int trans, int index,
                   int nmask = 0) {
    return Operand{p, stride, ld, trans, index, nmask == 1, nmask == 2, 0};
}
inline Operand opB(const float *p, long long stride, int ld, int trans, int index,
                   int nmask = 0) {
    return Operand{p, stride, ld, !trans, index, nmask == 2, nmask == 1, 0};
}

// The product over `units` units (blockIdx.z).  With `part` (room for max_splits *
// units * M * N floats) and max_splits > 1, K is split over enough CTAs for about
// eight per SM (each split at least 256 deep) and the partials are added in split
// order.  Returns LINFORMER_OK, LINFORMER_ERR_SIZE (more than 65535 units or row
// tiles) or LINFORMER_ERR_LAUNCH.
int batched_gemm(GemmArgs g, int units, cudaStream_t s, float *part = nullptr,
                 int max_splits = 1, int sms = 0, int kernel_id = LINFORMER_KERNEL_BACKWARD);

// Row softmax in place over S (units x rows_per_unit rows of `cols` values): rows
// i >= L are written as zero; with mask_cols, columns j >= L take no part (p = 0).
int softmax_rows(float *S, const int32_t *pad, int h, int rows_per_unit, int cols,
                 long long units, int mask_cols, cudaStream_t s,
                 int kernel_id = LINFORMER_KERNEL_BACKWARD);

// Maximum number of K splits of the k x d projections (partials: kMaxSplits * units *
// k * d floats per projection, one at a time).
constexpr int kMaxSplits = 8;

// Kbar = Ehat K and Vbar = Fhat V over the rows t < L for fp32 inputs, as two split
// products; `part` holds kMaxSplits * units * k * d floats.
int project_f32(const Problem &p, float *Kbar, float *Vbar, float *part, int kernel_id);

// O = softmax(Q Kbar^T / sqrt(d)) Vbar for fp32 Q and O, query rows i >= L zero, as
// two products around the row softmax; `P` holds units * n * k floats.
int attend_f32(const Problem &p, const float *Kbar, const float *Vbar, float *P,
               int kernel_id);

// Multiprocessor count of the current device.
int sm_count();

}  // namespace simt
}  // namespace linformer
