// Parameters and workspace layout shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.cuh"

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
// Vbar is stored scaled by 2^-e (e >= 0 keeps it inside the fp16 range).  Image 3 is
// written only for units that take two or more P.Vbar products (the only readers).
__host__ __device__ inline size_t image_bytes(int kpad) { return (size_t)kpad * kRowBytes; }

// info word per unit: bits 0-7 = number of P.Vbar products (1, 2 or 3), bits 8-15 = e.
__host__ __device__ inline int pack_info(int terms, int e) { return terms | (e << 8); }
__host__ __device__ inline int info_terms(int info) { return info & 0xff; }
__host__ __device__ inline int info_exp(int info) { return (info >> 8) & 0xff; }

// Vbar magnitudes that decide the number of fp16 products in P.Vbar.  O is a
// convex combination of Vbar rows, so a relative rounding of 2^-11 in either P
// (fp16) or Vbar (fp16) moves O by at most 2^-11 max|Vbar|.
//   1 product, P_hi Vbar_hi: both roundings, 2^-10 max|Vbar| < 0.0235 below 24
//     (the P part is a logit shift that mostly cancels in the normalisation).
//   2 products, + P_hi Vbar_lo: Vbar exact to 2^-22, P's rounding only,
//     2^-11 max|Vbar| < 0.0196 below 40.
//   3 products, + P_lo Vbar_hi: both to about 2^-21 relative, any magnitude.
// against an absolute bar of 2e-2 (plus 2^-8 |O| for the output rounding).
constexpr float kOneTermMaxV = 24.0f;
constexpr float kTwoTermMaxV = 40.0f;

// Split-n partial sums: per (unit, chunk, 128-row half of k_pad) one contiguous
// 64 KB block [128 columns][128 rows] fp32 (columns 0-63 Kbar, 64-127 Vbar), so
// that each 64-column half is one 32 KB slice for a single bulk copy.
__host__ __device__ inline size_t partial_bytes(int64_t units, int C, int mhalves) {
    return C > 1 ? (size_t)units * C * mhalves * 128 * 128 * sizeof(float) : 0;
}

// Chunks per unit for the projection.  Splitting a unit costs its CTAs a partial
// sum written and read back, so a unit is split only as far as needed to fill one
// wave of CTA slots (slots = SMs x CTAs resident per SM).  With ragged lengths,
// unknown on the host, chunks are also kept to about 6144 rows or fewer so that
// the longest valid lengths do not leave a long tail.  Chunk counts whose partial
// sums exceed part_budget are not taken.
inline int choose_chunks(int n, int64_t units, int slots, bool ragged, int mhalves,
                         size_t part_budget = ~size_t(0)) {
    const int max_c = n / 256 > 1 ? (n / 256 < 64 ? n / 256 : 64) : 1;
    int64_t c = units > 0 ? slots / units : 1;
    if (ragged) {
        const int64_t r = (n + 6143) / 6144;
        if (r > c) c = r;
    }
    if (c < 1) c = 1;
    if (c > max_c) c = max_c;
    while (c > 1) {
        const int ch = (int)(((n + c - 1) / c + kBK - 1) / kBK * kBK);
        const int c2 = (n + ch - 1) / ch;
        if (partial_bytes(units, c2, mhalves) <= part_budget) return c2;
        --c;
    }
    return 1;
}

// Shared-memory ring depth of the projection: stages of 64 sequence rows (the E
// and F tiles plus 8 KB each of K and V), as many as fit in about 100 KB so that
// two CTAs share an SM, between 2 and 6.
inline int project_stages(int mhalves, int distinct) {
    const size_t stage = (size_t)mhalves * 16384 * (1 + distinct) + 16384;
    const size_t s = (100 * 1024) / stage;
    return s < 2 ? 2 : (s > 6 ? 6 : (int)s);
}

// CTAs of the projection resident per SM for a given dynamic shared-memory size.
inline int project_ctas_per_sm(size_t smem) { return smem <= 113 * 1024 ? 2 : 1; }

// L2 prefetch of the projection's tiles, issued by each loader two stages beyond
// the shared-memory ring: K and V when a chunk runs long enough for it to pay
// (16 stages or more); E and F only when they are too large to stay in L2 across
// the units that share them (a prefetch of a tile already in L2 only delays the
// loader's next copy).
constexpr int kProjectPrefetch = 2;
inline int project_prefetch(int chunk_rows) { return chunk_rows >= 16 * kBK ? kProjectPrefetch : 0; }
inline int project_prefetch_proj(size_t proj_bytes) { return proj_bytes > (size_t(32) << 20) ? 1 : 0; }

// Bytes of one projection stage: the E (and F) tile plus 16 KB of K and V per unit.
inline size_t project_stage_bytes(int mhalves, int distinct, int nunits) {
    return (size_t)mhalves * 16384 * (1 + distinct) + (size_t)16384 * nunits;
}

// The projection's launch.  Chunks per unit as choose_chunks says; then, when units
// are not split, E = F and lengths are absent, and one wave of CTA slots cannot give
// every unit its own CTA, `pairs` CTAs per sharing group take two of its members:
// one E tile per stage serves both (one N = 256 product), which takes a third less
// traffic per unit.  With k_pad > 128 a pair fills the 512 TMEM columns, so every CTA
// of that launch runs alone on its SM with a deeper ring.
struct ProjPlan {
    int C, CH;            // chunks per unit, rows per chunk
    int stages, stages2;  // ring depth of one-unit and two-unit CTAs
    int pairs;            // two-member CTAs per sharing group
    int threads;          // 128, or 256 (an eight-warp epilogue) for the one-CTA-per-SM pairs
    size_t smem;          // dynamic shared memory per CTA
    int64_t grid;
};
inline ProjPlan plan_projection(int n, int64_t members, int64_t groups, int mhalves, int distinct,
                                bool ragged, int sms, size_t part_budget = ~size_t(0)) {
    ProjPlan pl{};
    const int64_t units = members * groups;
    pl.stages = project_stages(mhalves, distinct);
    pl.smem = 1024 + project_stage_bytes(mhalves, distinct, 1) * pl.stages + 256;
    pl.C = choose_chunks(n, units, sms * project_ctas_per_sm(pl.smem), ragged, mhalves,
                         part_budget);
    pl.CH = ((n + pl.C - 1) / pl.C + kBK - 1) / kBK * kBK;
    if (pl.C == 1 && !distinct && !ragged && members >= 2) {
        const bool wide = mhalves == 2;
        const size_t budget = wide ? 200 * 1024 : 100 * 1024;
        const size_t st1 = project_stage_bytes(mhalves, 0, 1), st2 = project_stage_bytes(mhalves, 0, 2);
        const int64_t slots = (int64_t)sms * (wide ? 1 : 2);
        int64_t P = members - slots / groups;
        if (P > members / 2) P = members / 2;
        if (P > 0 && budget / st2 >= 2) {
            pl.pairs = (int)P;
            pl.stages = (int)(budget / st1 < 6 ? budget / st1 : 6);
            pl.stages2 = (int)(budget / st2 < 6 ? budget / st2 : 6);
            const size_t ring = st1 * pl.stages > st2 * pl.stages2 ? st1 * pl.stages : st2 * pl.stages2;
            pl.smem = 1024 + ring + 256;
        }
    }
    pl.threads = pl.pairs > 0 && mhalves == 2 ? 256 : 128;
    pl.grid = groups * pl.C * (members - pl.pairs);
    return pl;
}

// After the main loop the projection reuses its ring: the split reduction's three 32 KB
// slice buffers at [0, 96 KB), then, in four-warp launches, two 32 KB image staging
// buffers at [0, 64 KB); eight-warp launches stage in [0, 128 KB) (two groups, two
// buffers each).  Every plan above gives at least 96 KB, and 192 KB to eight-warp launches.
constexpr size_t kProjectMinRing = 96 * 1024;
constexpr size_t kProjectMinRingWide = 128 * 1024;

// Arrival counters of a unit whose sequence is split into C chunks: one for the unit,
// one per group of chunks (the two-level reduction of tc_project.cu).  Groups hold
// split_group(C) chunks: all C below 9 (one level: the second level's extra store and
// arrival cost more than it saves there), else ceil(sqrt(C)); C <= 64 gives at most 8.
constexpr int kCountersPerUnit = 9;
__host__ __device__ inline int split_group(int C) {
    if (C < 9) return C;
    int g = 1;
    while (g * g < C) ++g;
    return g;
}

struct ProjParams {
    const int32_t *pad;
    float *partial;      // see partial_bytes (used when C > 1)
    uint8_t *images;     // [units][4][kpad * 128 bytes]
    int *counters;       // [units][kCountersPerUnit], zero on entry, left zero on exit
    int *info;           // [units]
    float *kbar_out;     // optional fp32 [units][k][64]
    float *vbar_out;     // optional fp32 [units][k][64]
    int *status;
    int h, n, k, kpad, mhalves, C, CH, stages, distinct, per_head, members, forced_terms;
    int pairs;           // per group and chunk: CTAs that take two members (see ProjPlan)
    int stages2;         // ring depth of those CTAs
    int prefetch;        // stages fetched into L2 ahead of the ring (0: none)
    int prefetch_proj;   // whether the E (and F) tiles are prefetched as well
};

struct AttnParams {
    const int32_t *pad;
    void *out;           // O, [units][n][64] bf16 or fp32: fully padded tiles are zeroed through it
    const uint8_t *images;
    const int *info;
    int *status;
    int h, n, k, kpad, units, tiles_per_unit, forced_terms, out_fp32;
    float scale_log2;    // log2(e) / sqrt(d)
};

// The host's plan of one tensor-core forward: the projection's launch and the
// workspace layout (images, split partials, per-unit counters, per-unit info words,
// each piece rounded up to 256 bytes).
struct ForwardPlan {
    ProjPlan proj;
    int64_t units, members, groups;
    int kpad, mhalves, distinct, per_head, sms;
    size_t img, part, cnt;
    size_t bytes() const { return img + part + 2 * cnt; }
};

// Plans a forward of the validated problem p (tc_supported shapes) on the current
// device.  part_budget: ~0 for a workspace sized to the plan; otherwise the size of a
// fixed workspace, which must hold the images, counters and info words (else
// LINFORMER_ERR_SIZE), the split partials taking what is left.
int plan_forward(const Problem &p, size_t part_budget, ForwardPlan *f);
// Launches the projection (writes Kbar/Vbar in fp32 and stops there when Kbar_out is
// given) and the attention on p.stream, with the workspace ws of f.bytes() bytes.
int run_forward(const Problem &p, const ForwardPlan &f, char *ws, float *Kbar_out,
                float *Vbar_out);

// threads: 128, or 256 for unsplit units without the fp32 Kbar/Vbar outputs.
int launch_project(const CUtensorMap &tE, const CUtensorMap &tF, const CUtensorMap &tK,
                   const CUtensorMap &tV, const ProjParams &p, int grid, int threads, size_t smem,
                   cudaStream_t s);

int launch_attend(const CUtensorMap &tQ, const CUtensorMap &tO, const AttnParams &p, int grid,
                  cudaStream_t s);
size_t attend_smem_bytes(int out_fp32);

}  // namespace tc
}  // namespace linformer
