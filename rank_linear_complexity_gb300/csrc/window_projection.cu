// Compression by pooling or convolution along the sequence ("Linformer(Self-Attention
// with Linear Complexity) 요약 설명", section "Additional Efficiency Techniques": the
// learned linear projection may be replaced by pooling or a convolution).  With a window
// of s = n / k positions moved by s, both are linear maps k x n in which row j reads
// positions [j s, (j + 1) s) only, so they run through the same projection kernels as a
// learned E.  This file writes that map.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace linformer {
namespace {

// P[j][t] = w(t - j s) if t lies in row j's window, else 0; w = 1 / s without weights.
template <typename T>
__global__ void window_projection_kernel(T *P, const float *weights, int n, int k, int s) {
    const long long total = (long long)n * k;
    const float mean = 1.0f / (float)s;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i / n), t = (int)(i - (long long)j * n);
        const int off = t - j * s;
        float v = 0.f;
        if (off >= 0 && off < s) v = weights ? weights[off] : mean;
        if constexpr (sizeof(T) == 2)
            P[i] = __float2bfloat16_rn(v);
        else
            P[i] = v;
    }
}

}  // namespace
}  // namespace linformer

using namespace linformer;

extern "C" int linformer_window_projection(void *P, const float *weights, int n, int k, int dtype,
                                           void *stream) {
    if (!P) return LINFORMER_ERR_NULL;
    if (n < 1 || k < 1 || n % k != 0) return LINFORMER_ERR_SIZE;
    if (dtype != LINFORMER_F32 && dtype != LINFORMER_BF16 && dtype != LINFORMER_BF16_F32OUT)
        return LINFORMER_ERR_ENUM;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long total = (long long)n * k;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    KernelScope scope(LINFORMER_KERNEL_WINDOW, s);
    if (dtype == LINFORMER_F32)
        window_projection_kernel<float><<<grid, 256, 0, s>>>(static_cast<float *>(P), weights, n, k,
                                                             n / k);
    else
        window_projection_kernel<__nv_bfloat16>
            <<<grid, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(P), weights, n, k, n / k);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}
