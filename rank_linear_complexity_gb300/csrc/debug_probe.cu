// linformer_debug_wait_probe: one warp waits, through the same bounded wait the
// kernels use, on an mbarrier that nothing ever arrives on.  The wait gives up after
// its limit (2 s), records code 90 in the device status word and the kernel returns:
// the device-side failure path, exercised without a fault, a trap or a hang.
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace linformer {
namespace {

constexpr int kProbeCode = 90;

__global__ void __launch_bounds__(32) wait_probe_kernel(int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncwarp();
    // phase 0 never completes: no thread arrives and no copy is pending on `bar`
    ptx::warp_wait(&bar, 0, status, kProbeCode, &abort_flag);
}

}  // namespace
}  // namespace linformer

extern "C" int linformer_debug_wait_probe(void *stream) {
    int *status = linformer::device_status_ptr();
    if (!status) return LINFORMER_ERR_LAUNCH;
    linformer::wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}
