// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "linformer_attn.h"

namespace linformer {

// One call's arguments, already validated.
struct Problem {
    const void *Q, *K, *V, *E, *F;
    const int32_t *pad;
    void *O;
    int b, h, n, d, k, share_mode, dtype;
    cudaStream_t stream;

    int64_t units() const { return (int64_t)b * h; }
    // E (and F) carry a leading head index in these modes.
    bool proj_per_head() const {
        return share_mode == LINFORMER_SHARE_PER_HEAD || share_mode == LINFORMER_SHARE_KV;
    }
    // F is its own tensor (not E) in these modes.
    bool distinct_f() const {
        return share_mode == LINFORMER_SHARE_PER_HEAD || share_mode == LINFORMER_SHARE_HEADWISE;
    }
    const void *f_or_e() const { return distinct_f() ? F : E; }
    size_t in_elem() const { return dtype == LINFORMER_F32 ? 4 : 2; }
    size_t out_elem() const { return dtype == LINFORMER_BF16 ? 2 : 4; }
};

// Brackets one kernel launch: counts it and, while profiling is on, records CUDA
// events around it on its stream.
class KernelScope {
  public:
    KernelScope(int kernel_id, cudaStream_t s);
    ~KernelScope();

  private:
    int id_;
    cudaStream_t s_;
    cudaEvent_t a_ = nullptr, b_ = nullptr;
};

// Argument rules shared by the entry points (linformer_api.cu).
bool aligned16(const void *p);
int validate_common(int b, int h, int n, int d, int k, int share_mode, int dtype);
int validate_f(int share_mode, const void *E, const void *F);
// Null pointers, sizes, enums, the F rule and alignment of a forward call on device
// buffers: LINFORMER_OK or the status the entry point returns.
int validate_forward(const void *Q, const void *K, const void *V, const void *E, const void *F,
                     const int32_t *pad_lengths, const void *O, int b, int h, int n, int d, int k,
                     int share_mode, int dtype);

// Device status word of the current device (set by bounded waits that ran out).
int *device_status_ptr();

// Stream-ordered workspace on the current device from a library-owned memory pool
// whose freed memory stays mapped between calls (the device's default pool unmaps
// freed memory at every synchronisation, and the next allocation maps it again).
// Returns LINFORMER_OK or LINFORMER_ERR_ALLOC; free with workspace_free on a stream.
// (workspace.cu: also the LINFORMER_FAIL_ALLOC and LINFORMER_WORKSPACE_GUARD switches.)
int workspace_alloc(void **ptr, size_t bytes, cudaStream_t s);
void workspace_free(void *ptr, cudaStream_t s);
// The library's pool on device `dev` (created on first use), or nullptr.
cudaMemPool_t library_pool(int dev);

// Process-wide P.Vbar product-count setting (0 = automatic, 1, 2 or 3).
int pv_terms_setting();

// Fused SIMT kernels for bf16 inputs off the tensor-core shapes (simt_kernels.cu);
// fp32 inputs return LINFORMER_ERR_UNSUPPORTED (they run on simt_gemm.cu).
int simt_project(const Problem &p, float *Kbar, float *Vbar);
int simt_attend(const Problem &p, const float *Kbar, const float *Vbar);

// fp32 dense softmax attention (simt_dense.cu).
int simt_dense_attention(const Problem &p);

// fp32 backward (simt_backward.cu).
int simt_backward(const Problem &p, const float *dO, float *dQ, float *dK, float *dV, float *dE,
                  float *dF);

// Tensor-core kernels (tc_project.cu, tc_attend.cu).
bool tc_supported(int n, int d, int k, int dtype);
int tc_forward(const Problem &p, float *Kbar_out, float *Vbar_out);

}  // namespace linformer
