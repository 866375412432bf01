// Host side of the tensor-core path: TMA descriptors, split-n chunking, the
// stream-ordered workspace and the two launches (projection, then attention).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace linformer {

bool tc_supported(int n, int d, int k, int dtype) {
    return dtype != LINFORMER_F32 && d == tc::kD && k >= 1 && k <= tc::kMaxK && n % 8 == 0 &&
           n <= (1 << 30);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

constexpr int kMaxDev = 64;
int g_sms[kMaxDev] = {};

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDev) return 148;
    if (!g_sms[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = v > 0 ? v : 148;
    }
    return g_sms[dev];
}

// 3-D tiled map, 128-byte swizzle, out-of-range elements read as zero.
bool encode3d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem,
              uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * elem, d0 * d1 * elem};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace tc {

int plan_forward(const Problem &p, size_t part_budget, ForwardPlan *fp) {
    if (!encoder()) return LINFORMER_ERR_LAUNCH;
    ForwardPlan f{};
    f.units = p.units();
    f.kpad = (p.k + 15) / 16 * 16;
    f.mhalves = (f.kpad + 127) / 128;
    f.distinct = p.distinct_f() ? 1 : 0;
    f.per_head = p.proj_per_head() ? 1 : 0;
    f.sms = sm_count();
    f.members = f.per_head ? p.b : f.units;
    f.groups = f.units / f.members;
    f.img = up256(f.units * 4 * image_bytes(f.kpad));
    // per unit the split reduction's arrival counters
    f.cnt = up256(f.units * kCountersPerUnit * sizeof(int));
    if (part_budget != ~size_t(0)) {  // a fixed workspace: images, counters and info first
        if (f.img + 2 * f.cnt > part_budget) return LINFORMER_ERR_SIZE;
        part_budget -= f.img + 2 * f.cnt;
    }
    f.proj = plan_projection(p.n, f.members, f.groups, f.mhalves, f.distinct, p.pad != nullptr,
                             f.sms, part_budget);
    if (f.proj.smem < 1024 + kProjectMinRing + 256 ||
        (f.proj.threads == 256 && f.proj.smem < 1024 + kProjectMinRingWide + 256))
        return LINFORMER_ERR_UNSUPPORTED;
    if (f.proj.grid > 0x7fffffffLL) return LINFORMER_ERR_SIZE;
    f.part = up256(partial_bytes(f.units, f.proj.C, f.mhalves));
    *fp = f;
    return LINFORMER_OK;
}

int run_forward(const Problem &p, const ForwardPlan &f, char *ws, float *Kbar_out,
                float *Vbar_out) {
    const int64_t units = f.units;
    uint8_t *images = reinterpret_cast<uint8_t *>(ws);
    float *partial = f.proj.C > 1 ? reinterpret_cast<float *>(ws + f.img) : nullptr;
    int *counters = reinterpret_cast<int *>(ws + f.img + f.part);
    int *info = reinterpret_cast<int *>(ws + f.img + f.part + f.cnt);
    // The split reduction's counters start at zero (also when the workspace is reused
    // from an earlier call); unsplit units use none, and then nothing comes between
    // the previous kernel in the stream and the projection, which may start early.
    if (f.proj.C > 1 && cudaMemsetAsync(counters, 0, f.cnt, p.stream) != cudaSuccess)
        return LINFORMER_ERR_LAUNCH;

    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t groups = (uint64_t)f.groups;
    CUtensorMap tE, tF, tK, tV;
    if (!(encode3d(&tE, p.E, bf, 2, p.n, p.k, groups, 64, 128 * f.mhalves) &&
          encode3d(&tF, p.f_or_e(), bf, 2, p.n, p.k, groups, 64, 128 * f.mhalves) &&
          encode3d(&tK, p.K, bf, 2, kD, p.n, units, 64, kBK) &&
          encode3d(&tV, p.V, bf, 2, kD, p.n, units, 64, kBK)))
        return LINFORMER_ERR_LAUNCH;

    int *status = device_status_ptr();
    ProjParams pp{};
    pp.pad = p.pad;
    pp.partial = partial;
    pp.images = images;
    pp.counters = counters;
    pp.info = info;
    pp.kbar_out = Kbar_out;
    pp.vbar_out = Vbar_out;
    pp.status = status;
    pp.h = p.h;
    pp.n = p.n;
    pp.k = p.k;
    pp.kpad = f.kpad;
    pp.mhalves = f.mhalves;
    pp.C = f.proj.C;
    pp.CH = f.proj.CH;
    pp.stages = f.proj.stages;
    pp.stages2 = f.proj.stages2;
    pp.pairs = f.proj.pairs;
    pp.prefetch = project_prefetch(f.proj.CH);
    pp.prefetch_proj =
        project_prefetch_proj((size_t)groups * p.k * p.n * 2 * (1 + f.distinct));
    pp.distinct = f.distinct;
    pp.per_head = f.per_head;
    pp.members = (int)f.members;
    pp.forced_terms = pv_terms_setting();
    int st = launch_project(tE, tF, tK, tV, pp, (int)f.proj.grid,
                            Kbar_out ? 128 : f.proj.threads, f.proj.smem, p.stream);
    if (st != LINFORMER_OK || Kbar_out) return st;

    CUtensorMap tQ, tO;
    const bool f32out = p.dtype == LINFORMER_BF16_F32OUT;
    if (!(encode3d(&tQ, p.Q, bf, 2, kD, p.n, units, 64, kTileM) &&
          (f32out ? encode3d(&tO, p.O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kD, p.n, units, 32,
                             kTileM)
                  : encode3d(&tO, p.O, bf, 2, kD, p.n, units, 64, kTileM))))
        return LINFORMER_ERR_LAUNCH;
    AttnParams ap{};
    ap.pad = p.pad;
    ap.out = p.O;
    ap.images = images;
    ap.info = info;
    ap.status = status;
    ap.h = p.h;
    ap.n = p.n;
    ap.k = p.k;
    ap.kpad = f.kpad;
    ap.units = (int)units;
    ap.tiles_per_unit = (p.n + kTileM - 1) / kTileM;
    ap.forced_terms = pp.forced_terms;
    ap.out_fp32 = f32out ? 1 : 0;
    ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.d));
    const int64_t tiles = units * ap.tiles_per_unit;
    const int grid = (int)std::min<int64_t>(f.sms, tiles);
    return launch_attend(tQ, tO, ap, grid, p.stream);
}

}  // namespace tc

int tc_forward(const Problem &p, float *Kbar_out, float *Vbar_out) {
    tc::ForwardPlan f;
    int st = tc::plan_forward(p, ~size_t(0), &f);
    if (st != LINFORMER_OK) return st;
    char *ws = nullptr;
    if (workspace_alloc(reinterpret_cast<void **>(&ws), f.bytes(), p.stream) != LINFORMER_OK)
        return LINFORMER_ERR_ALLOC;
    st = tc::run_forward(p, f, ws, Kbar_out, Vbar_out);
    workspace_free(ws, p.stream);
    return st;
}

}  // namespace linformer
