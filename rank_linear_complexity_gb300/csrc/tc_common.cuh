// Parameters and workspace layout shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace linformer {
namespace tc {

constexpr int kD = 64;           // head dimension of the tensor-core path
constexpr int kRowBytes = 128;   // one 64-element bf16/fp16 row
constexpr int kMaxK = 256;       // projected length limit (one S tile in TMEM)
constexpr int kTileM = 128;      // query rows per attention tile
constexpr int kBK = 64;          // sequence rows per projection pipeline stage

// Per unit the projection writes four k_pad x 64 images, each row 128 bytes,
// already in the 128-byte-swizzled shared-memory layout the attention kernel's
// MMAs read (16-byte chunk q of row j sits at chunk position q ^ (j % 8)):
//   0: Kbar hi (bf16)   1: Kbar lo (bf16)   2: Vbar hi (fp16)   3: Vbar lo (fp16)
// Vbar is stored scaled by 2^-e (e >= 0 keeps it inside the fp16 range).
__host__ __device__ inline size_t image_bytes(int kpad) { return (size_t)kpad * kRowBytes; }

// info word per unit: bits 0-7 = number of P.Vbar products (1 or 3), bits 8-15 = e.
__host__ __device__ inline int pack_info(int terms, int e) { return terms | (e << 8); }
__host__ __device__ inline int info_terms(int info) { return info & 0xff; }
__host__ __device__ inline int info_exp(int info) { return (info >> 8) & 0xff; }

// Vbar magnitude below which one fp16 product suffices for P.Vbar: the fp16
// rounding of Vbar costs at most 2^-7 absolute below 32, and the fp16 rounding
// of P acts as a logit perturbation of at most 2^-11, worth at most about
// 2^-11 * max|Vbar| <= 0.0117 at 24 -- together under the 2e-2 absolute bar.
constexpr float kOneTermMaxV = 24.0f;

struct ProjParams {
    const int32_t *pad;
    float *partial;      // [units][C][kpad][128] fp32 (used when C > 1)
    uint8_t *images;     // [units][4][kpad * 128 bytes]
    int *counters;       // [units], zero on entry, left zero on exit
    int *info;           // [units]
    float *kbar_out;     // optional fp32 [units][k][64]
    float *vbar_out;     // optional fp32 [units][k][64]
    int *status;
    int h, n, k, kpad, mhalves, C, CH, stages, distinct, per_head, members, forced_terms;
};

struct AttnParams {
    const int32_t *pad;
    const uint8_t *images;
    const int *info;
    int *status;
    int h, n, k, kpad, units, tiles_per_unit, forced_terms, out_fp32;
    float scale_log2;    // log2(e) / sqrt(d)
};

int launch_project(const CUtensorMap &tE, const CUtensorMap &tF, const CUtensorMap &tK,
                   const CUtensorMap &tV, const ProjParams &p, int grid, size_t smem,
                   cudaStream_t s);
size_t project_smem_bytes(int mhalves, int distinct, int stages);

int launch_attend(const CUtensorMap &tQ, const CUtensorMap &tO, const AttnParams &p, int grid,
                  cudaStream_t s);
size_t attend_smem_bytes(int out_fp32);

}  // namespace tc
}  // namespace linformer
