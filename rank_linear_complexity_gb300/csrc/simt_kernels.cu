// Fused FFMA kernels for the Linformer attention forward on bf16 inputs whose shape
// is outside the tensor-core path (d != 64, k > 256, n not a multiple of 8).  fp32
// inputs run on the matrix-product kernels of simt_gemm.cu instead.  All arithmetic
// is fp32; the projection accumulates over the sequence in order, the softmax is the
// exact two-pass form.
//
// Steps ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model):
//   simt_project_kernel: Kbar = Ehat . K and Vbar = Fhat . V over rows t < L.
//   simt_attend_kernel:  O = softmax(Q . Kbar^T / sqrt(d)) . Vbar, rows i < L;
//                        rows i >= L are written as zero.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace linformer {
namespace {

__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ int valid_length(const int32_t *pad, int batch, int n) {
    if (!pad) return n;
    int L = pad[batch];
    return L < 0 ? 0 : (L > n ? n : L);
}

constexpr int PJ = 32;      // projected rows per block
constexpr int PT = 32;      // sequence rows per step
constexpr int MAXD = 128;

// grid: (units, ceil(k / PJ), 2); z = 0 projects K with E, z = 1 projects V with F.
template <typename TIn>
__global__ void __launch_bounds__(256) simt_project_kernel(
    const TIn *__restrict__ K, const TIn *__restrict__ V, const TIn *__restrict__ E,
    const TIn *__restrict__ F, const int32_t *__restrict__ pad, float *__restrict__ Kbar,
    float *__restrict__ Vbar, int h, int n, int d, int k, int proj_per_head) {
    __shared__ float Es[PJ][PT + 1];
    __shared__ float Xs[PT][MAXD];
    const int64_t u = blockIdx.x;
    const int batch = (int)(u / h), head = (int)(u % h);
    const int j0 = blockIdx.y * PJ;
    const bool is_v = blockIdx.z == 1;
    const TIn *X = (is_v ? V : K) + u * (int64_t)n * d;
    const TIn *P = (is_v ? F : E) + (proj_per_head ? (int64_t)head * k * n : 0);
    float *out = (is_v ? Vbar : Kbar) + u * (int64_t)k * d;
    const int L = valid_length(pad, batch, n);

    const int tid = threadIdx.x;
    const int jl = tid >> 3;  // 0..31
    const int cg = tid & 7;   // column group: columns cg, cg + 8, ...
    float acc[MAXD / 8];
#pragma unroll
    for (int i = 0; i < MAXD / 8; ++i) acc[i] = 0.f;

    for (int t0 = 0; t0 < L; t0 += PT) {
        for (int e = tid; e < PJ * PT; e += blockDim.x) {
            int jj = e / PT, tt = e % PT;
            int j = j0 + jj, t = t0 + tt;
            Es[jj][tt] = (j < k && t < L) ? to_f32(P[(int64_t)j * n + t]) : 0.f;
        }
        for (int e = tid; e < PT * d; e += blockDim.x) {
            int tt = e / d, c = e % d;
            int t = t0 + tt;
            Xs[tt][c] = (t < L) ? to_f32(X[(int64_t)t * d + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int tt = 0; tt < PT; ++tt) {
            const float e = Es[jl][tt];
#pragma unroll
            for (int i = 0; i < MAXD / 8; ++i) {
                const int c = cg + 8 * i;
                if (c < d) acc[i] = fmaf(e, Xs[tt][c], acc[i]);
            }
        }
        __syncthreads();
    }
    const int j = j0 + jl;
    if (j < k) {
#pragma unroll
        for (int i = 0; i < MAXD / 8; ++i) {
            const int c = cg + 8 * i;
            if (c < d) out[(int64_t)j * d + c] = acc[i];
        }
    }
}

constexpr int AW = 8;        // warps per block
constexpr int AROWS = 64;    // query rows per block

// grid: units * ceil(n / AROWS) blocks (flattened); one warp per query row at a time.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(AW * 32) simt_attend_kernel(
    const TIn *__restrict__ Q, const float *__restrict__ Kbar, const float *__restrict__ Vbar,
    const int32_t *__restrict__ pad, TOut *__restrict__ O, int h, int n, int d, int k,
    int64_t tiles_per_unit) {
    extern __shared__ float smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *qs = smem + warp * (MAXD + k);
    float *ss = qs + MAXD;
    const int64_t u = blockIdx.x / tiles_per_unit;
    const int64_t tile = blockIdx.x % tiles_per_unit;
    const int L = valid_length(pad, (int)(u / h), n);
    const float *Kb = Kbar + u * (int64_t)k * d;
    const float *Vb = Vbar + u * (int64_t)k * d;
    const float scale = 1.0f / sqrtf((float)d);

    for (int r = warp; r < AROWS; r += AW) {
        const int64_t i = tile * AROWS + r;
        if (i >= n) break;
        TOut *orow = O + (u * n + i) * (int64_t)d;
        if (i >= L) {
            for (int c = lane; c < d; c += 32) store_out(orow + c, 0.f);
            continue;
        }
        const TIn *qrow = Q + (u * n + i) * (int64_t)d;
        for (int c = lane; c < d; c += 32) qs[c] = to_f32(qrow[c]);
        __syncwarp();
        float m = -INFINITY;
        for (int j = lane; j < k; j += 32) {
            const float *kr = Kb + (int64_t)j * d;
            float dot = 0.f;
            for (int c = 0; c < d; ++c) dot = fmaf(qs[c], kr[c], dot);
            const float s = dot * scale;
            ss[j] = s;
            m = fmaxf(m, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
        for (int j = lane; j < k; j += 32) {
            const float p = expf(ss[j] - m);
            ss[j] = p;
            sum += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.0f / sum;
        __syncwarp();
        for (int c = lane; c < d; c += 32) {
            float acc = 0.f;
            for (int j = 0; j < k; ++j) acc = fmaf(ss[j], Vb[(int64_t)j * d + c], acc);
            store_out(orow + c, acc * inv);
        }
        __syncwarp();
    }
}

}  // namespace

int simt_project(const Problem &p, float *Kbar, float *Vbar) {
    dim3 grid((unsigned)p.units(), (unsigned)((p.k + PJ - 1) / PJ), 2);
    if (p.dtype == LINFORMER_F32) return LINFORMER_ERR_UNSUPPORTED;  // simt_gemm.cu's
    KernelScope scope(LINFORMER_KERNEL_PROJECT_SIMT, p.stream);
    simt_project_kernel<__nv_bfloat16><<<grid, 256, 0, p.stream>>>(
        (const __nv_bfloat16 *)p.K, (const __nv_bfloat16 *)p.V, (const __nv_bfloat16 *)p.E,
        (const __nv_bfloat16 *)p.f_or_e(), p.pad, Kbar, Vbar, p.h, p.n, p.d, p.k,
        p.proj_per_head() ? 1 : 0);
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

int simt_attend(const Problem &p, const float *Kbar, const float *Vbar) {
    if (p.dtype == LINFORMER_F32) return LINFORMER_ERR_UNSUPPORTED;  // simt_gemm.cu's
    const int64_t tiles = (p.n + AROWS - 1) / AROWS;
    const int64_t blocks = p.units() * tiles;
    if (blocks > 0x7fffffffLL) return LINFORMER_ERR_SIZE;
    const size_t smem = (size_t)AW * (MAXD + p.k) * sizeof(float);
    KernelScope scope(LINFORMER_KERNEL_ATTEND_SIMT, p.stream);
    cudaError_t err = cudaSuccess;
#define LAUNCH_ATTEND(TI, TO)                                                              \
    do {                                                                                   \
        auto kern = simt_attend_kernel<TI, TO>;                                            \
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                   (int)smem);                                             \
        if (err == cudaSuccess)                                                            \
            kern<<<(unsigned)blocks, AW * 32, smem, p.stream>>>(                           \
                (const TI *)p.Q, Kbar, Vbar, p.pad, (TO *)p.O, p.h, p.n, p.d, p.k, tiles); \
    } while (0)
    if (p.dtype == LINFORMER_BF16)
        LAUNCH_ATTEND(__nv_bfloat16, __nv_bfloat16);
    else
        LAUNCH_ATTEND(__nv_bfloat16, float);
#undef LAUNCH_ATTEND
    if (err != cudaSuccess) return LINFORMER_ERR_LAUNCH;
    return cudaPeekAtLastError() == cudaSuccess ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
}

}  // namespace linformer
