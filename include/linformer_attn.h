/*
 * linformer_attn.h -- C ABI of the GB300 (sm_103a) Linformer attention forward.
 *
 * The operation ("Linformer(Self-Attention with Linear Complexity) 요약 설명",
 * section Model; "Linformer: Self-Attention with Linear Complexity - 中文验证版",
 * section 方法适配): for every batch index beta < b and head eta < h (a "unit"),
 *
 *     Kbar = Ehat . K[beta][eta]        (k x n) . (n x d) -> k x d
 *     Vbar = Fhat . V[beta][eta]        (k x n) . (n x d) -> k x d
 *     O[beta][eta] = softmax(Q[beta][eta] . Kbar^T / sqrt(d)) . Vbar   -> n x d
 *
 * E and F project the sequence axis (length n) down to k positions; the queries
 * are not compressed, so O has one row per input position and the n x k score
 * matrix never leaves the chip.  The scale 1/sqrt(d) is the scaled dot product
 * of the PaperWeekly efficient-Transformer survey, section 2.1.
 *
 * Sharing modes (中文验证版, section 方法适配; 요약 설명, section Additional
 * Efficiency Techniques):
 *   LINFORMER_SHARE_PER_HEAD  E, F: [h][k][n], each head its own pair
 *   LINFORMER_SHARE_KV        E:    [h][k][n], F = E (F must be NULL or == E)
 *   LINFORMER_SHARE_HEADWISE  E, F: [k][n], one pair for all heads
 *   LINFORMER_SHARE_LAYERWISE E:    [k][n], one projection for all heads and for
 *                                   keys and values (F must be NULL or == E)
 * In every mode E and F are shared across the batch (they are parameters).
 *
 * Padding (요약 설명, section Model, padding paragraph): pad_lengths[beta] is the
 * valid length L of batch entry beta (clamped to [0, n] on the device).  Rows
 * t >= L of K and V count as zero before the projection, whatever they hold,
 * and query rows i >= L get O = 0.  NULL means L = n for every entry.
 *
 * Layouts: every tensor is dense and row-major.  Q, K, V, O: [b][h][n][d].
 * E, F: as listed above ([k][n] rows of length n).
 *
 * Number types (dtype):
 *   LINFORMER_F32          Q, K, V, E, F, O in fp32; all arithmetic in fp32.
 *   LINFORMER_BF16         Q, K, V, E, F, O in bf16; fp32 accumulation.
 *   LINFORMER_BF16_F32OUT  inputs in bf16, O in fp32.
 *
 * Ownership: the caller owns every buffer.  All pointers of linformer_attn_fwd
 * and linformer_project_fwd are device pointers of the current CUDA device, 16-byte
 * aligned.  The library writes only O (or Kbar/Vbar) and a stream-ordered
 * workspace that it allocates and frees on `stream` (cudaMallocFromPoolAsync /
 * cudaFreeAsync) from a memory pool of its own per device, created on first use,
 * which keeps freed memory mapped for the next call until the process exits (as much
 * as the largest call in flight needed).  Calls are asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream): inputs must stay unchanged until the stream has
 * passed the call.  Calls on different streams may run concurrently.  The forward's
 * first kernel is launched with programmatic stream serialisation and waits for the
 * kernel before it (griddepcontrol.wait) before it reads or writes memory; its last
 * kernel lets the next kernel in the stream launch early, so a caller's kernel that
 * is itself launched with programmatic stream serialisation after a call must wait
 * for its prerequisite grid (cudaGridDependencySynchronize) before it reads O, as
 * CUDA requires of any such kernel.  Kernels launched without that attribute are
 * ordered as usual.
 *
 * Errors: every function returns LINFORMER_OK (0) or a negative status; no call
 * traps or aborts.  Argument errors are detected on the host before anything is
 * launched.  Device-side failures (a bounded wait that ran out) set a device
 * status word that linformer_debug_read_device_status() reads and clears.
 */
#ifndef LINFORMER_ATTN_H
#define LINFORMER_ATTN_H

#include <stdint.h>

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define LINFORMER_API __attribute__((visibility("default")))
#else
#define LINFORMER_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LINFORMER_F32 = 0,
    LINFORMER_BF16 = 1,
    LINFORMER_BF16_F32OUT = 2
} linformer_dtype;

typedef enum {
    LINFORMER_SHARE_PER_HEAD = 0,
    LINFORMER_SHARE_KV = 1,
    LINFORMER_SHARE_HEADWISE = 2,
    LINFORMER_SHARE_LAYERWISE = 3
} linformer_share_mode;

typedef enum {
    LINFORMER_OK = 0,
    LINFORMER_ERR_NULL = -1,        /* a required pointer is NULL */
    LINFORMER_ERR_SIZE = -2,        /* b, h, n, d or k < 1, or a size overflows */
    LINFORMER_ERR_UNSUPPORTED = -3, /* d > 128 or k > 1024 */
    LINFORMER_ERR_ENUM = -4,        /* bad share_mode or dtype */
    LINFORMER_ERR_ALIGN = -5,       /* a pointer is not 16-byte aligned */
    LINFORMER_ERR_F_MODE = -6,      /* F given (and != E) in KV / LAYERWISE mode, or
                                       missing in PER_HEAD / HEADWISE mode */
    LINFORMER_ERR_ALLOC = -7,       /* workspace allocation failed */
    LINFORMER_ERR_LAUNCH = -8,      /* a CUDA call or kernel launch failed */
    LINFORMER_ERR_DEVICE = -9       /* a device-side bounded wait ran out */
} linformer_status;

/* Which kernels a call uses. */
typedef enum {
    LINFORMER_PATH_SIMT = 0,        /* fp32 FFMA kernels: any supported shape */
    LINFORMER_PATH_TENSOR = 1       /* tcgen05/TMA kernels: bf16 inputs, d = 64,
                                       k <= 256, n a multiple of 8 */
} linformer_path_kind;

/* Kernel identifiers for the profiling counters. */
typedef enum {
    LINFORMER_KERNEL_PROJECT_TC = 0,
    LINFORMER_KERNEL_ATTEND_TC = 1,
    LINFORMER_KERNEL_PROJECT_SIMT = 2,
    LINFORMER_KERNEL_ATTEND_SIMT = 3,
    LINFORMER_KERNEL_WINDOW = 4,    /* linformer_window_projection */
    LINFORMER_KERNEL_BACKWARD = 5,  /* the kernels of linformer_attn_bwd */
    LINFORMER_KERNEL_DENSE = 6,     /* the kernels of linformer_dense_attn_fwd */
    LINFORMER_KERNEL_COUNT = 7
} linformer_kernel_id;

/*
 * The whole Linformer attention forward (all steps above) for b*h units.
 * Q, K, V: [b][h][n][d] (dtype in); E, F: see the sharing modes; pad_lengths:
 * device int32[b] or NULL; O: [b][h][n][d] (dtype out).  Supported: d <= 128,
 * k <= 1024 (the tensor-core path takes bf16 inputs with d = 64, k <= 256 and
 * n % 8 == 0; other shapes run on the fp32 SIMT kernels).
 */
LINFORMER_API int linformer_attn_fwd(const void *Q, const void *K, const void *V,
                       const void *E, const void *F,
                       const int32_t *pad_lengths, void *O,
                       int b, int h, int n, int d, int k,
                       int share_mode, int dtype, void *stream);

/*
 * The projection step alone: Kbar = Ehat . K and Vbar = Fhat . V over the valid
 * rows (요약 설명, section Model), written as fp32 [b][h][k][d] into the
 * caller's device buffers Kbar and Vbar.  Same argument rules as above.  On the
 * tensor-core path Kbar and Vbar are the exact sums of the on-chip split
 * representation the attention step consumes.
 */
LINFORMER_API int linformer_project_fwd(const void *K, const void *V, const void *E, const void *F,
                          const int32_t *pad_lengths, float *Kbar, float *Vbar,
                          int b, int h, int n, int d, int k,
                          int share_mode, int dtype, void *stream);

/*
 * Same operation as linformer_attn_fwd, for callers whose data is in HOST memory
 * (page-locked memory gives the fastest copies).  Q, K, V, E, F, pad_lengths and
 * O are host pointers.  The call allocates device buffers on `stream`, copies
 * the inputs in, runs the forward, copies O back and synchronises `stream`
 * before returning, so O is complete on return.
 */
LINFORMER_API int linformer_attn_fwd_host(const void *Q, const void *K, const void *V,
                            const void *E, const void *F,
                            const int32_t *pad_lengths, void *O,
                            int b, int h, int n, int d, int k,
                            int share_mode, int dtype, void *stream);

/*
 * linformer_attn_fwd_noalloc: the same operation, arguments and device buffers as
 * linformer_attn_fwd, for callers that must not allocate device memory while they
 * run it -- for example a server that reserved its whole memory budget at start-up,
 * a plugin whose host framework owns every device allocation, code called from an
 * allocator or out-of-memory handler, or a setup without stream-ordered memory
 * pools.  It allocates nothing: its workspace is one fixed 32 MiB array in device
 * memory that every GPU loading this library holds until the process exits.
 *   - Problems whose workspace does not fit in 32 MiB even without splitting the
 *     sequence (about b*h*k_pad*512 bytes, k_pad = k rounded up to 16) return
 *     LINFORMER_ERR_SIZE before anything is launched.
 *   - Only tensor-core configurations (bf16 inputs, d = 64, k <= 256, n % 8 == 0)
 *     are served; others return LINFORMER_ERR_UNSUPPORTED.
 *   - The first call on a device looks up the array's address on that device;
 *     make it before any stream capture starts.
 *   - Every call reuses the same array and clears its per-unit counters itself;
 *     calls that overlap on the GPU (other streams, other host threads) race on
 *     the array and must be serialised by the caller.
 * The pages describe no counterpart: this is a deployment variant, not part of the
 * method.
 */
LINFORMER_API int linformer_attn_fwd_noalloc(const void *Q, const void *K, const void *V,
                                             const void *E, const void *F,
                                             const int32_t *pad_lengths, void *O,
                                             int b, int h, int n, int d, int k,
                                             int share_mode, int dtype, void *stream);

/*
 * The backward of linformer_attn_fwd: given dO = dLoss/dO, writes dQ, dK, dV
 * ([b][h][n][d]) and dE (shaped like E) and, in PER_HEAD and HEADWISE modes, dF
 * (shaped like F; in KV and LAYERWISE modes F is E and dE holds both terms, dF must be
 * NULL).  The chain rule through the forward's definition (요약 설명, section Model):
 * rows t >= L of K and V and query rows i >= L take no part (their gradients are
 * zero), and the gradient of a shared E or F sums the terms of every unit that shares
 * it.  fp32 only (LINFORMER_F32; other dtypes return LINFORMER_ERR_UNSUPPORTED),
 * d <= 128, k <= 1024, b*h <= 65535 (else LINFORMER_ERR_SIZE).  All pointers are
 * device pointers, 16-byte aligned; the caller owns every buffer; a stream-ordered
 * workspace of b*h*(2 n k + 12 k d) floats (8 k d of the 12 hold split partial sums;
 * the 2 n k, once P and dS are used, the partial sums of dE and dF) comes from the
 * library's pool and is returned to it in stream order.
 */
LINFORMER_API int linformer_attn_bwd(const void *Q, const void *K, const void *V,
                                     const void *E, const void *F, const int32_t *pad_lengths,
                                     const void *dO, void *dQ, void *dK, void *dV, void *dE,
                                     void *dF, int b, int h, int n, int d, int k,
                                     int share_mode, int dtype, void *stream);

/*
 * Dense softmax attention, the full-attention baseline that the pages' inference table
 * ("Linformer 요약 설명", section Inference-time Efficiency Results) compares the
 * method with: O = softmax(Q K^T / sqrt(d)) V per unit, Q, K, V, O [b][h][n][d] fp32.
 * With pad_lengths, keys t >= L take no part in the softmax and query rows i >= L are
 * written as zero.  The n x n scores of every unit live in a stream-ordered workspace
 * of b*h*n*n floats from the library's pool (the memory the standard form needs).
 * fp32 only (else LINFORMER_ERR_UNSUPPORTED); d <= 128; b*h <= 65535 and n <= 8388480
 * (else LINFORMER_ERR_SIZE); pointers device, 16-byte aligned; the caller owns them.
 */
LINFORMER_API int linformer_dense_attn_fwd(const void *Q, const void *K, const void *V,
                                           const int32_t *pad_lengths, void *O, int b, int h,
                                           int n, int d, int dtype, void *stream);

/*
 * Largest number of bytes the library's workspace pool on the current device has had
 * in use at once since the pool was created or last reset; reset != 0 then sets the
 * mark back to the bytes in use now.  Returns -1 if the pool cannot be queried.
 */
LINFORMER_API int64_t linformer_pool_peak_bytes(int reset);

/*
 * Pooling or convolution instead of a learned projection (요약 설명, section
 * "Additional Efficiency Techniques").  With s = n / k (n % k == 0), writes into the
 * caller's device buffer P, [k][n] in the input dtype (bf16 for LINFORMER_BF16 and
 * LINFORMER_BF16_F32OUT, fp32 for LINFORMER_F32), the map whose row j averages or
 * convolves the window of positions [j s, (j + 1) s):
 *   weights == NULL: mean pooling, P[j][j s + t] = 1 / s (rounded to the dtype);
 *   weights: device float[s], a convolution with kernel size = stride = s,
 *            P[j][j s + t] = weights[t];
 * every other entry 0.  Pass P as E (and F) of linformer_attn_fwd with a shared mode
 * (LAYERWISE, HEADWISE), or fill one [k][n] slice per head for the per-head modes.
 * Asynchronous on `stream`; P is owned by the caller.  Errors: LINFORMER_ERR_NULL,
 * LINFORMER_ERR_SIZE (n % k != 0 or a size < 1), LINFORMER_ERR_ENUM, LINFORMER_ERR_LAUNCH.
 */
LINFORMER_API int linformer_window_projection(void *P, const float *weights, int n, int k,
                                              int dtype, void *stream);

/* Which path (linformer_path_kind) a call with these arguments takes, or a
 * negative status if the arguments are invalid.  Host only; launches nothing. */
LINFORMER_API int linformer_select_path(int b, int h, int n, int d, int k, int share_mode, int dtype);

/* Human-readable text for a status code (static storage). */
LINFORMER_API const char *linformer_status_string(int status);

/* Synchronises `stream`, returns LINFORMER_ERR_DEVICE if a kernel of this library
 * recorded a device-side failure on the current device since the last read (and
 * clears it), else LINFORMER_OK.  For tests and debugging. */
LINFORMER_API int linformer_debug_read_device_status(void *stream);

/* Test of the device-side failure path: launches one warp on `stream` that waits,
 * through the same bounded wait as the kernels, on a barrier nothing completes.  After
 * the wait limit (2 s) the warp records a failure in the device status word and exits;
 * no fault, trap or hang.  Returns LINFORMER_OK once launched;
 * linformer_debug_read_device_status() then reports LINFORMER_ERR_DEVICE, and the
 * library keeps working on the same context.  For tests and debugging. */
LINFORMER_API int linformer_debug_wait_probe(void *stream);

/* Number of products in the P.Vbar step of the tensor-core path: 0 = chosen per
 * unit on the device from max|Vbar| (default: 1 below 24, 2 below 40, else 3),
 * 1 = one product (fp16 P, fp16 Vbar), 2 = P times the hi/lo split of Vbar,
 * 3 = three products (hi/lo splits of P and Vbar).  Process-wide setting for
 * tests and tuning; returns the previous value, or LINFORMER_ERR_ENUM. */
LINFORMER_API int linformer_set_pv_terms(int terms);

/* Number of kernels this library has launched in this process (all devices). */
LINFORMER_API int64_t linformer_launch_count(void);

/* Profiling: while enabled, every kernel launch is bracketed by CUDA events on
 * its own stream.  linformer_profile_collect() synchronises those events, adds
 * each kernel's total milliseconds and launch count into ms[id] and launches[id]
 * (arrays of LINFORMER_KERNEL_COUNT entries), and clears the record. */
LINFORMER_API int linformer_profile_enable(int enable);
LINFORMER_API int linformer_profile_collect(double *ms, int64_t *launches);

/* Name of a linformer_kernel_id (static storage), or NULL. */
LINFORMER_API const char *linformer_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* LINFORMER_ATTN_H */
