// Stream-ordered workspaces: a library-owned memory pool per device whose freed
// memory stays mapped between calls (the device's default pool unmaps freed memory
// at every synchronisation, and the next allocation maps it again).
//
// Two switches, read at every allocation, exist for tests of the host-side error
// paths and of out-of-range writes (no GPU fault is involved in either):
//   LINFORMER_FAIL_ALLOC=1       every workspace allocation fails: the entry point
//                                returns LINFORMER_ERR_ALLOC before it launches
//                                anything;
//   LINFORMER_WORKSPACE_GUARD=1  every workspace is followed by kGuardBytes of a
//                                fixed pattern (allocated with it); when the
//                                workspace is freed a small kernel compares them, and
//                                if any byte changed it records kGuardCode in the
//                                device status word (read with
//                                linformer_debug_read_device_status).
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "internal.cuh"

namespace linformer {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kGuardBytes = 4096;
constexpr unsigned char kGuardByte = 0xA5;
constexpr int kGuardCode = 60;

cudaMemPool_t g_pools[kMaxDevices] = {};
std::mutex g_pool_mu;

std::mutex g_guard_mu;
std::unordered_map<void *, size_t> g_guarded;  // workspace -> its size (guard follows it)

bool switch_on(const char *name) {
    const char *v = std::getenv(name);
    return v && *v && std::strcmp(v, "0") != 0;
}

// One thread per 16 guard bytes, compared byte by byte (the guard may start at any
// byte offset).
__global__ void __launch_bounds__(256) guard_check_kernel(const unsigned char *guard, int *status) {
    const unsigned char *g = guard + 16 * threadIdx.x;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 16; ++i) ok &= g[i] == kGuardByte;
    if (!ok && status) atomicExch(status, kGuardCode);
}
static_assert(kGuardBytes == 16 * 256, "one 256-thread block checks the guard");

}  // namespace

cudaMemPool_t library_pool(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = ~uint64_t(0);
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pools[dev] = pool;
    }
    return g_pools[dev];
}

int workspace_alloc(void **ptr, size_t bytes, cudaStream_t s) {
    *ptr = nullptr;
    if (switch_on("LINFORMER_FAIL_ALLOC")) return LINFORMER_ERR_ALLOC;
    const bool guard = switch_on("LINFORMER_WORKSPACE_GUARD");
    const size_t total = bytes + (guard ? kGuardBytes : 0);
    int dev = 0;
    cudaMemPool_t pool = nullptr;
    if (cudaGetDevice(&dev) == cudaSuccess) pool = library_pool(dev);
    const cudaError_t e =
        pool ? cudaMallocFromPoolAsync(ptr, total, pool, s) : cudaMallocAsync(ptr, total, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return LINFORMER_ERR_ALLOC;
    }
    if (guard) {
        if (cudaMemsetAsync(static_cast<char *>(*ptr) + bytes, kGuardByte, kGuardBytes, s) !=
            cudaSuccess) {
            cudaGetLastError();
            cudaFreeAsync(*ptr, s);
            *ptr = nullptr;
            return LINFORMER_ERR_ALLOC;
        }
        std::lock_guard<std::mutex> lock(g_guard_mu);
        g_guarded[*ptr] = bytes;
    }
    return LINFORMER_OK;
}

void workspace_free(void *ptr, cudaStream_t s) {
    if (!ptr) return;
    size_t bytes = 0;
    bool guarded = false;
    {
        std::lock_guard<std::mutex> lock(g_guard_mu);
        auto it = g_guarded.find(ptr);
        if (it != g_guarded.end()) {
            bytes = it->second;
            guarded = true;
            g_guarded.erase(it);
        }
    }
    if (guarded) {
        guard_check_kernel<<<1, 256, 0, s>>>(static_cast<const unsigned char *>(ptr) + bytes,
                                              device_status_ptr());
        cudaGetLastError();
    }
    cudaFreeAsync(ptr, s);  // back to its pool
}

}  // namespace linformer
