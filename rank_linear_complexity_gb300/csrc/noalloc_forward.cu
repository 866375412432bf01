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
// Argument rules, the launch plan and the launches themselves are those of
// linformer_attn_fwd (validate_forward, tc::plan_forward, tc::run_forward); only the
// workspace differs.
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

// Device address of the array on the current device (looked up once per device,
// with that device current).
uint8_t *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = static_cast<uint8_t *>(ptr);
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace linformer

using namespace linformer;

extern "C" int linformer_attn_fwd_noalloc(const void *Q, const void *K, const void *V,
                                          const void *E, const void *F,
                                          const int32_t *pad_lengths, void *O, int b, int h,
                                          int n, int d, int k, int share_mode, int dtype,
                                          void *stream) {
    int st = validate_forward(Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    if (!tc_supported(n, d, k, dtype)) return LINFORMER_ERR_UNSUPPORTED;
    const Problem p{Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode, dtype,
                    reinterpret_cast<cudaStream_t>(stream)};
    // The allocating path's plan, among chunk counts whose fp32 partials still fit next
    // to the images, counters and info words (LINFORMER_ERR_SIZE if those do not).
    tc::ForwardPlan plan;
    if ((st = tc::plan_forward(p, kScratchBytes, &plan))) return st;
    if (plan.bytes() > kScratchBytes) return LINFORMER_ERR_SIZE;
    uint8_t *scratch = scratch_on_current_device();
    if (!scratch) return LINFORMER_ERR_LAUNCH;
    return tc::run_forward(p, plan, reinterpret_cast<char *>(scratch), nullptr, nullptr);
}
