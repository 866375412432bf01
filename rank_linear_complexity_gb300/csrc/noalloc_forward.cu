// linformer_attn_fwd_noalloc: the tensor-core forward for callers that may not
// allocate device memory.
//
// Some callers cannot call cudaMalloc or cudaMallocAsync at the moment they run
// the attention: a serving process that reserved its whole memory budget at
// start-up and forbids allocation afterwards, a plugin inside a host framework
// that owns every device allocation, code running from an allocator's or an
// out-of-memory handler's own callback, or a device/driver setup without
// stream-ordered memory pools.  This entry point does the same work as
// linformer_attn_fwd on the same kinds of buffers, but takes its workspace from
// one fixed array that lives in device memory for as long as the library is
// loaded (every GPU that loads the library holds it until the process exits).
//
// Rules of use:
//   * Capacity: kScratchBytes (32 MiB).  A problem whose workspace does not fit
//     even without splitting the sequence is rejected with LINFORMER_ERR_SIZE
//     before anything is launched.
//   * The first call on a device looks up the array's device address on that
//     device (cudaGetSymbolAddress); make that first call before any stream
//     capture begins.
//   * All calls share the one array and find it as the previous call left it;
//     the per-unit counters are cleared at the start of each call.  Two calls
//     whose work overlaps on the GPU (different streams, or different host
//     threads) race on the array: serialise them.
//   * Only the tensor-core configurations are served (bf16 inputs, d = 64,
//     k <= 256, n % 8 == 0); others return LINFORMER_ERR_UNSUPPORTED.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace linformer {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

// The workspace.  In host code this name is only a handle for
// cudaGetSymbolAddress: never pass it to a kernel directly.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
uint8_t *g_scratch_addr[kMaxDev] = {};
int g_sm_count[kMaxDev] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;

// Device address of the array on the current device (looked up once per device).
uint8_t *scratch_on_current_device(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return nullptr;
        }
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = v > 0 ? v : 148;
        g_scratch_addr[dev] = static_cast<uint8_t *>(ptr);
    }
    if (!g_enc) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *sms = g_sm_count[dev];
    return g_scratch_addr[dev];
}

bool map3d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem, uint64_t d0,
           uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * elem, d0 * d1 * elem};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace linformer

using namespace linformer;

extern "C" int linformer_attn_fwd_noalloc(const void *Q, const void *K, const void *V,
                                          const void *E, const void *F,
                                          const int32_t *pad_lengths, void *O, int b, int h,
                                          int n, int d, int k, int share_mode, int dtype,
                                          void *stream) {
    using namespace tc;
    if (!Q || !K || !V || !E || !O) return LINFORMER_ERR_NULL;
    if (b < 1 || h < 1 || n < 1 || d < 1 || k < 1) return LINFORMER_ERR_SIZE;
    if (share_mode < LINFORMER_SHARE_PER_HEAD || share_mode > LINFORMER_SHARE_LAYERWISE ||
        dtype < LINFORMER_F32 || dtype > LINFORMER_BF16_F32OUT)
        return LINFORMER_ERR_ENUM;
    const bool distinct_f = share_mode == LINFORMER_SHARE_PER_HEAD ||
                            share_mode == LINFORMER_SHARE_HEADWISE;
    if (distinct_f && !F) return LINFORMER_ERR_F_MODE;
    if (!distinct_f && F && F != E) return LINFORMER_ERR_F_MODE;
    auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(Q) || misaligned(K) || misaligned(V) || misaligned(E) || misaligned(O) ||
        (F && misaligned(F)) || (reinterpret_cast<uintptr_t>(pad_lengths) & 3u))
        return LINFORMER_ERR_ALIGN;
    if (!tc_supported(n, d, k, dtype)) return LINFORMER_ERR_UNSUPPORTED;
    const int64_t units = (int64_t)b * h;
    if (units > (1LL << 31) - 1) return LINFORMER_ERR_SIZE;

    // Workspace plan: images + counters + info always; split partials only if they fit.
    const int kpad = (k + 15) / 16 * 16;
    const int mhalves = (kpad + 127) / 128;
    const int distinct = distinct_f ? 1 : 0;
    const int per_head = (share_mode == LINFORMER_SHARE_PER_HEAD ||
                          share_mode == LINFORMER_SHARE_KV) ? 1 : 0;
    const size_t img = round256((size_t)units * 4 * image_bytes(kpad));
    const size_t cnt = round256((size_t)(units + 1) * sizeof(int));  // + product-count summary
    if (img + 2 * cnt > kScratchBytes) return LINFORMER_ERR_SIZE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int sms = 0;
    uint8_t *scratch = scratch_on_current_device(&sms);
    if (!scratch) return LINFORMER_ERR_LAUNCH;

    // The allocating path's plan, among chunk counts whose fp32 partials still fit
    // next to the images.
    const int64_t members = per_head ? b : units;
    const ProjPlan plan = plan_projection(n, members, units / members, mhalves, distinct,
                                          pad_lengths != nullptr, sms, kScratchBytes - img - 2 * cnt);
    const int C = plan.C, CH = plan.CH;
    if (plan.smem < 1024 + kProjectMinRing + 256) return LINFORMER_ERR_UNSUPPORTED;
    const size_t part = round256(partial_bytes(units, C, mhalves));
    uint8_t *images = scratch;
    float *partial = C > 1 ? reinterpret_cast<float *>(scratch + img) : nullptr;
    int *counters = reinterpret_cast<int *>(scratch + img + part);
    int *info = reinterpret_cast<int *>(scratch + img + part + cnt);
    if (cudaMemsetAsync(counters, 0, cnt, s) != cudaSuccess) return LINFORMER_ERR_LAUNCH;

    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t groups = per_head ? (uint64_t)h : 1;
    const void *Fm = distinct ? F : E;
    CUtensorMap tE, tF, tK, tV, tQ, tO;
    const bool f32out = dtype == LINFORMER_BF16_F32OUT;
    if (!(map3d(&tE, E, bf, 2, n, k, groups, 64, 128 * mhalves) && map3d(&tF, Fm, bf, 2, n, k, groups, 64, 128 * mhalves) &&
          map3d(&tK, K, bf, 2, kD, n, units, 64, kBK) && map3d(&tV, V, bf, 2, kD, n, units, 64, kBK) &&
          map3d(&tQ, Q, bf, 2, kD, n, units, 64, kTileM) &&
          (f32out ? map3d(&tO, O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kD, n, units, 32, kTileM)
                  : map3d(&tO, O, bf, 2, kD, n, units, 64, kTileM))))
        return LINFORMER_ERR_LAUNCH;

    ProjParams pp{};
    pp.pad = pad_lengths;
    pp.partial = partial;
    pp.images = images;
    pp.counters = counters;
    pp.terms_seen = counters + units;
    pp.info = info;
    pp.status = device_status_ptr();
    pp.h = h;
    pp.n = n;
    pp.k = k;
    pp.kpad = kpad;
    pp.mhalves = mhalves;
    pp.C = C;
    pp.CH = CH;
    pp.stages = plan.stages;
    pp.stages2 = plan.stages2;
    pp.pairs = plan.pairs;
    pp.prefetch = project_prefetch(CH);
    pp.prefetch_proj = project_prefetch_proj((size_t)groups * k * n * 2 * (1 + distinct));
    pp.distinct = distinct;
    pp.per_head = per_head;
    pp.members = (int)members;
    pp.forced_terms = pv_terms_setting();
    if (plan.grid > 0x7fffffffLL) return LINFORMER_ERR_SIZE;
    int st = launch_project(tE, tF, tK, tV, pp, (int)plan.grid, plan.threads, plan.smem, s);
    if (st != LINFORMER_OK) return st;

    AttnParams ap{};
    ap.pad = pad_lengths;
    ap.out = O;
    ap.images = images;
    ap.info = info;
    ap.terms_seen = counters + units;
    ap.status = pp.status;
    ap.h = h;
    ap.n = n;
    ap.k = k;
    ap.kpad = kpad;
    ap.units = (int)units;
    ap.tiles_per_unit = (n + kTileM - 1) / kTileM;
    ap.forced_terms = pp.forced_terms;
    ap.out_fp32 = f32out ? 1 : 0;
    ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    const int agrid = (int)std::min<int64_t>(sms, units * ap.tiles_per_unit);
    return launch_attend(tQ, tO, ap, agrid, s);
}
