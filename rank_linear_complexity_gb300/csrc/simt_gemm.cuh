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
    // Tensor-core product only, x contiguous: x splits into blocks of xblk (a multiple of
    // 32; 0: none), block j of matrix z at mat(z) + j blk_stride, so that one product
    // covers the units that share the other operand side by side along N.
    int xblk = 0;
    long long blk_stride = 0;
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
    int *status;  // device status word for bounded waits that run out (tensor-core kernel)
    // Tensor-core product only (tc_batched_gemm):
    int epi = 0;  // an EpilogueKind
    // usum_groups > 0: a sum over units.  Output matrix g < usum_groups (C + g sC) is the
    // sum over i < usum_per_group of A_u B_u (+ A2_u B2_u when A2.p is set), unit
    // u = g usum_ga + i usum_gb, each term with its own unit's length masks; the
    // output masks must be off.
    int usum_groups = 0, usum_per_group = 0, usum_ga = 0, usum_gb = 0;
    Operand A2{}, B2{};
    // cblk > 0 (with B.xblk == cblk): C's columns in blocks of cblk, block j of output
    // matrix z at C + z sC + j cblk_stride; block j of matrix z belongs to unit
    // z blk_ua + j blk_ub (its length masks B's sequence axis and C's rows).
    int cblk = 0;
    long long cblk_stride = 0;
    int blk_ua = 0, blk_ub = 0;
    // kEpiSoftmaxPair: the second output (laid out as C) and the second product's scale
    float *C2 = nullptr;
    float alpha2 = 1.f;
};

// What the tensor-core product writes: alpha A B (+ beta C, output masks), or, from
// two products of each row tile (kEpiSoftmaxPair), C = P = the row softmax of
// alpha A B (rows at or past the unit's length zero) and C2 = P * (dP - rowsum(P * dP))
// with dP = alpha2 A2 B2.  The pair needs N <= 256 (a tile holds whole rows),
// alpha > 0 and no sum over units.
enum EpilogueKind { kEpiPlain = 0, kEpiSoftmaxPair = 1 };

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

// The same product on the tensor cores (tc_gemm.cu): fp32 operands are split into bf16
// hi + lo parts on the way into shared memory and C = A_hi B_hi + A_hi B_lo + A_lo B_hi
// accumulates in fp32 (the dropped A_lo B_lo and the split's residual are about 2^-18
// of each term), with the epilogue forms and sums over units of GemmArgs.  With `part`
// (part_floats floats) a plain product may split K (a sum over units, its units) for
// about four work items per SM; partials are added in split order.  Returns
// LINFORMER_OK, LINFORMER_ERR_SIZE (a pair with N > 256 or a sum, mismatched second
// operands, blocks that break the rules of Operand.xblk) or LINFORMER_ERR_LAUNCH.
int tc_batched_gemm(GemmArgs g, int units, cudaStream_t s, float *part = nullptr,
                    size_t part_floats = 0, int sms = 0,
                    int kernel_id = LINFORMER_KERNEL_BACKWARD);

// C = the sum over splits of g.part (+ beta C), with the output masks (split order).
int launch_splitk_reduce(const GemmArgs &g, int units, cudaStream_t s, int kernel_id);
// Sets o.vec: whether 4-element groups along o's contiguous axis may be 16-byte loads.
void set_operand_vec(Operand &o, int contiguous_extent);

// Row softmax in place over S (units x rows_per_unit rows of `cols` values): rows
// i >= L are written as zero; with mask_cols, columns j >= L take no part (p = 0).
int softmax_rows(float *S, const int32_t *pad, int h, int rows_per_unit, int cols,
                 long long units, int mask_cols, cudaStream_t s,
                 int kernel_id = LINFORMER_KERNEL_BACKWARD);

// Maximum number of K splits of the k x d projections (partials: kMaxSplits * units *
// k * d floats per projection, one at a time).
constexpr int kMaxSplits = 8;

// Kbar = Ehat K and Vbar = Fhat V over the rows t < L for fp32 inputs, as two split
// products (on the tensor cores with `tensor`); `part` holds kMaxSplits * units * k * d
// floats.
int project_f32(const Problem &p, float *Kbar, float *Vbar, float *part, int kernel_id,
                bool tensor = false);

// O = softmax(Q Kbar^T / sqrt(d)) Vbar for fp32 Q and O, query rows i >= L zero, as
// two products around the row softmax; `P` holds units * n * k floats.
int attend_f32(const Problem &p, const float *Kbar, const float *Vbar, float *P,
               int kernel_id);

// Multiprocessor count of the current device.
int sm_count();

}  // namespace simt
}  // namespace linformer
