// Host side of the C ABI declared in include/linformer_attn.h: argument
// validation, path selection, launch bookkeeping, profiling events and the device
// status word (the workspace pool is in workspace.cu).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"
#include "simt_gemm.cuh"

namespace linformer {

// Set to a non-zero code by a kernel whose bounded wait ran out.
__device__ int g_device_status;

namespace {

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_profiling{0};
std::atomic<int> g_pv_terms{0};

struct ProfileRecord {
    int id;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::vector<ProfileRecord> g_prof;

constexpr int kMaxDevices = 64;
int *g_status_addr[kMaxDevices] = {};
std::mutex g_status_mu;

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

int select_path(int n, int d, int k, int dtype) {
    return tc_supported(n, d, k, dtype) ? LINFORMER_PATH_TENSOR : LINFORMER_PATH_SIMT;
}

// The forward on device pointers (arguments already validated).  Kbar_out and
// Vbar_out, when non-null, receive the fp32 projections and O is not computed.
int run_forward(const Problem &p, float *Kbar_out, float *Vbar_out) {
    if (select_path(p.n, p.d, p.k, p.dtype) == LINFORMER_PATH_TENSOR)
        return tc_forward(p, Kbar_out, Vbar_out);
    float *Kb = Kbar_out, *Vb = Vbar_out;
    void *ws = nullptr;
    const size_t bytes = (size_t)p.units() * p.k * p.d * sizeof(float);
    // fp32 inputs: the SIMT matrix-product kernel (split projections, then scores,
    // row softmax and P Vbar; the partials and P share the space after Kbar and Vbar);
    // bf16 inputs: the fused SIMT projection and attention kernels
    const bool f32 = p.dtype == LINFORMER_F32;
    const size_t scores = Kbar_out ? 0 : (size_t)p.units() * p.n * p.k * sizeof(float);
    const size_t part = f32 ? std::max((size_t)simt::kMaxSplits * bytes, scores) : 0;
    const size_t need = (Kb ? 0 : 2 * bytes) + part;
    if (need && workspace_alloc(&ws, need, p.stream) != LINFORMER_OK) return LINFORMER_ERR_ALLOC;
    char *wp = static_cast<char *>(ws);
    if (!Kb) {
        Kb = reinterpret_cast<float *>(wp);
        Vb = reinterpret_cast<float *>(wp + bytes);
        wp += 2 * bytes;
    }
    int st = f32 ? simt::project_f32(p, Kb, Vb, reinterpret_cast<float *>(wp),
                                     LINFORMER_KERNEL_PROJECT_SIMT)
                 : simt_project(p, Kb, Vb);
    if (st == LINFORMER_OK && !Kbar_out)
        st = f32 ? simt::attend_f32(p, Kb, Vb, reinterpret_cast<float *>(wp),
                                    LINFORMER_KERNEL_ATTEND_SIMT)
                 : simt_attend(p, Kb, Vb);
    if (ws) workspace_free(ws, p.stream);
    return st;
}

}  // namespace

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_common(int b, int h, int n, int d, int k, int share_mode, int dtype) {
    if (b < 1 || h < 1 || n < 1 || d < 1 || k < 1) return LINFORMER_ERR_SIZE;
    if (share_mode < LINFORMER_SHARE_PER_HEAD || share_mode > LINFORMER_SHARE_LAYERWISE)
        return LINFORMER_ERR_ENUM;
    if (dtype < LINFORMER_F32 || dtype > LINFORMER_BF16_F32OUT) return LINFORMER_ERR_ENUM;
    if (d > 128 || k > 1024) return LINFORMER_ERR_UNSUPPORTED;
    const int64_t units = (int64_t)b * h;
    if (units > (1LL << 31) - 1) return LINFORMER_ERR_SIZE;
    if (units * (int64_t)n > (1LL << 40) || units * (int64_t)n * d > (1LL << 46))
        return LINFORMER_ERR_SIZE;
    return LINFORMER_OK;
}

int validate_f(int share_mode, const void *E, const void *F) {
    const bool distinct = share_mode == LINFORMER_SHARE_PER_HEAD ||
                          share_mode == LINFORMER_SHARE_HEADWISE;
    if (distinct && !F) return LINFORMER_ERR_F_MODE;
    if (!distinct && F && F != E) return LINFORMER_ERR_F_MODE;
    return LINFORMER_OK;
}

// Every argument rule of the forward entry points (device buffers).
int validate_forward(const void *Q, const void *K, const void *V, const void *E, const void *F,
                     const int32_t *pad_lengths, const void *O, int b, int h, int n, int d, int k,
                     int share_mode, int dtype) {
    if (!Q || !K || !V || !E || !O) return LINFORMER_ERR_NULL;
    int st = validate_common(b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    if ((st = validate_f(share_mode, E, F))) return st;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(E) || !aligned16(O) ||
        (F && !aligned16(F)) || (reinterpret_cast<uintptr_t>(pad_lengths) & 3u))
        return LINFORMER_ERR_ALIGN;
    return LINFORMER_OK;
}

// Batch chunks of the host entry point's copy/compute pipeline.
constexpr int kHostChunks = 8;

// Two non-blocking streams per device for the host entry point's copies.
cudaStream_t g_side[kMaxDevices][2] = {};
std::mutex g_side_mu;

cudaStream_t side_stream(int i) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_side_mu);
    if (!g_side[dev][i] &&
        cudaStreamCreateWithFlags(&g_side[dev][i], cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        g_side[dev][i] = nullptr;
    }
    return g_side[dev][i];
}

KernelScope::KernelScope(int kernel_id, cudaStream_t s) : id_(kernel_id), s_(s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_profiling.load(std::memory_order_relaxed)) {
        if (cudaEventCreate(&a_) == cudaSuccess && cudaEventCreate(&b_) == cudaSuccess) {
            cudaEventRecord(a_, s_);
        } else {
            a_ = b_ = nullptr;
        }
    }
}

KernelScope::~KernelScope() {
    if (!a_) return;
    cudaEventRecord(b_, s_);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof.push_back({id_, a_, b_});
}

int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<int *>(ptr);
    }
    return g_status_addr[dev];
}

int pv_terms_setting() { return g_pv_terms.load(std::memory_order_relaxed); }

}  // namespace linformer

using namespace linformer;

extern "C" int linformer_attn_fwd(const void *Q, const void *K, const void *V, const void *E,
                                  const void *F, const int32_t *pad_lengths, void *O, int b,
                                  int h, int n, int d, int k, int share_mode, int dtype,
                                  void *stream) {
    const int st = validate_forward(Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode,
                                    dtype);
    if (st) return st;
    Problem p{Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode, dtype,
              as_stream(stream)};
    return run_forward(p, nullptr, nullptr);
}

extern "C" int linformer_project_fwd(const void *K, const void *V, const void *E,
                                     const void *F, const int32_t *pad_lengths, float *Kbar,
                                     float *Vbar, int b, int h, int n, int d, int k,
                                     int share_mode, int dtype, void *stream) {
    if (!K || !V || !E || !Kbar || !Vbar) return LINFORMER_ERR_NULL;
    int st = validate_common(b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    if ((st = validate_f(share_mode, E, F))) return st;
    if (!aligned16(K) || !aligned16(V) || !aligned16(E) || !aligned16(Kbar) ||
        !aligned16(Vbar) || (F && !aligned16(F)) ||
        (reinterpret_cast<uintptr_t>(pad_lengths) & 3u))
        return LINFORMER_ERR_ALIGN;
    Problem p{nullptr, K, V, E, F, pad_lengths, nullptr, b, h, n, d, k, share_mode, dtype,
              as_stream(stream)};
    return run_forward(p, Kbar, Vbar);
}

extern "C" int linformer_attn_bwd(const void *Q, const void *K, const void *V, const void *E,
                                  const void *F, const int32_t *pad_lengths, const void *dO,
                                  void *dQ, void *dK, void *dV, void *dE, void *dF, int b, int h,
                                  int n, int d, int k, int share_mode, int dtype, void *stream) {
    if (!Q || !K || !V || !E || !dO || !dQ || !dK || !dV || !dE) return LINFORMER_ERR_NULL;
    int st = validate_common(b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    if ((st = validate_f(share_mode, E, F))) return st;
    if (dtype != LINFORMER_F32) return LINFORMER_ERR_UNSUPPORTED;
    const bool distinct = share_mode == LINFORMER_SHARE_PER_HEAD ||
                          share_mode == LINFORMER_SHARE_HEADWISE;
    if (distinct != (dF != nullptr)) return distinct ? LINFORMER_ERR_NULL : LINFORMER_ERR_F_MODE;
    const void *ptrs[] = {Q, K, V, E, F, dO, dQ, dK, dV, dE, dF};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return LINFORMER_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(pad_lengths) & 3u) return LINFORMER_ERR_ALIGN;
    if ((int64_t)b * h > 65535) return LINFORMER_ERR_SIZE;
    Problem p{Q, K, V, E, F, pad_lengths, nullptr, b, h, n, d, k, share_mode, dtype,
              as_stream(stream)};
    return simt_backward(p, static_cast<const float *>(dO), static_cast<float *>(dQ),
                         static_cast<float *>(dK), static_cast<float *>(dV),
                         static_cast<float *>(dE), static_cast<float *>(dF));
}

extern "C" int linformer_dense_attn_fwd(const void *Q, const void *K, const void *V,
                                        const int32_t *pad_lengths, void *O, int b, int h, int n,
                                        int d, int dtype, void *stream) {
    if (!Q || !K || !V || !O) return LINFORMER_ERR_NULL;
    int st = validate_common(b, h, n, d, 1, LINFORMER_SHARE_PER_HEAD, dtype);
    if (st) return st;
    if (dtype != LINFORMER_F32) return LINFORMER_ERR_UNSUPPORTED;
    const void *ptrs[] = {Q, K, V, O};
    for (const void *q : ptrs)
        if (!aligned16(q)) return LINFORMER_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(pad_lengths) & 3u) return LINFORMER_ERR_ALIGN;
    if ((int64_t)b * h > 65535 || n > 65535 * 128) return LINFORMER_ERR_SIZE;
    Problem p{Q, K, V, nullptr, nullptr, pad_lengths, O, b, h, n, d, 1, LINFORMER_SHARE_PER_HEAD,
              dtype, as_stream(stream)};
    return simt_dense_attention(p);
}

extern "C" int64_t linformer_pool_peak_bytes(int reset) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    cudaMemPool_t pool = library_pool(dev);
    if (!pool) return -1;
    uint64_t high = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &high) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (reset) {
        uint64_t zero = 0;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero);
    }
    return (int64_t)high;
}

extern "C" int linformer_attn_fwd_host(const void *Q, const void *K, const void *V,
                                       const void *E, const void *F,
                                       const int32_t *pad_lengths, void *O, int b, int h,
                                       int n, int d, int k, int share_mode, int dtype,
                                       void *stream) {
    if (!Q || !K || !V || !E || !O) return LINFORMER_ERR_NULL;
    int st = validate_common(b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    if ((st = validate_f(share_mode, E, F))) return st;
    const bool distinct = share_mode == LINFORMER_SHARE_PER_HEAD ||
                          share_mode == LINFORMER_SHARE_HEADWISE;
    const bool per_head = share_mode == LINFORMER_SHARE_PER_HEAD ||
                          share_mode == LINFORMER_SHARE_KV;
    const size_t in_e = dtype == LINFORMER_F32 ? 4 : 2;
    const size_t out_e = dtype == LINFORMER_BF16 ? 2 : 4;
    const size_t qkv = (size_t)b * h * n * d * in_e;
    const size_t proj = (size_t)(per_head ? h : 1) * k * n * in_e;
    const size_t obytes = (size_t)b * h * n * d * out_e;
    const size_t pbytes = pad_lengths ? (size_t)b * sizeof(int32_t) : 0;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t total = 3 * up(qkv) + up(proj) * (distinct ? 2 : 1) + up(obytes) + up(pbytes);
    cudaStream_t s = as_stream(stream);
    char *base = nullptr;
    if (workspace_alloc(reinterpret_cast<void **>(&base), total, s) != LINFORMER_OK)
        return LINFORMER_ERR_ALLOC;
    char *dQ = base, *dK = dQ + up(qkv), *dV = dK + up(qkv), *dE = dV + up(qkv);
    char *dF = distinct ? dE + up(proj) : nullptr;
    char *dO = (distinct ? dF : dE) + up(proj);
    char *dP = pad_lengths ? dO + up(obytes) : nullptr;
    // A pipeline over batch chunks: inputs come in on one side stream, each chunk's
    // forward runs on `s` once its inputs are in, and its O goes out on the other
    // side stream while later chunks compute (the two copy directions overlap).
    // Events made for this call carry every dependency.
    const size_t qrow = qkv / b, orow = obytes / b;  // bytes of one batch entry
    // Chunk boundaries keep the kernels' 16-byte alignment only if a batch entry does.
    const int chunks = (qrow % 256 || orow % 256) ? 1 : (b < kHostChunks ? b : kHostChunks);
    cudaStream_t in = side_stream(0), out = side_stream(1);
    cudaEvent_t ev[2 * kHostChunks + 2] = {};
    const int nev = 2 * chunks + 2;
    bool ok = in && out;
    for (int i = 0; i < nev && ok; ++i)
        ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventRecord(ev[0], s) == cudaSuccess &&  // after the allocation
         cudaStreamWaitEvent(in, ev[0], 0) == cudaSuccess &&
         cudaMemcpyAsync(dE, E, proj, cudaMemcpyHostToDevice, in) == cudaSuccess &&
         (!dF || cudaMemcpyAsync(dF, F, proj, cudaMemcpyHostToDevice, in) == cudaSuccess) &&
         (!dP || cudaMemcpyAsync(dP, pad_lengths, pbytes, cudaMemcpyHostToDevice, in) ==
                     cudaSuccess);
    st = ok ? LINFORMER_OK : LINFORMER_ERR_LAUNCH;
    for (int c = 0; c < chunks && st == LINFORMER_OK; ++c) {
        const int b0 = (int)((int64_t)b * c / chunks), b1 = (int)((int64_t)b * (c + 1) / chunks);
        const size_t off = qrow * b0, len = qrow * (b1 - b0);
        cudaEvent_t inputs = ev[1 + 2 * c], done = ev[2 + 2 * c];
        ok = cudaMemcpyAsync(dQ + off, static_cast<const char *>(Q) + off, len,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaMemcpyAsync(dK + off, static_cast<const char *>(K) + off, len,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaMemcpyAsync(dV + off, static_cast<const char *>(V) + off, len,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaEventRecord(inputs, in) == cudaSuccess &&
             cudaStreamWaitEvent(s, inputs, 0) == cudaSuccess;
        if (!ok) {
            st = LINFORMER_ERR_LAUNCH;
            break;
        }
        Problem p{dQ + off, dK + off, dV + off, dE, dF,
                  dP ? reinterpret_cast<const int32_t *>(dP) + b0 : nullptr, dO + orow * b0,
                  b1 - b0, h, n, d, k, share_mode, dtype, s};
        st = run_forward(p, nullptr, nullptr);
        if (st == LINFORMER_OK &&
            !(cudaEventRecord(done, s) == cudaSuccess &&
              cudaStreamWaitEvent(out, done, 0) == cudaSuccess &&
              cudaMemcpyAsync(static_cast<char *>(O) + orow * b0, dO + orow * b0,
                              orow * (b1 - b0), cudaMemcpyDeviceToHost, out) == cudaSuccess))
            st = LINFORMER_ERR_LAUNCH;
    }
    // `s` goes on (and frees the workspace) only after both side streams are done.
    const bool joined = in && out && ev[nev - 1] &&
                        cudaEventRecord(ev[nev - 1], out) == cudaSuccess &&
                        cudaStreamWaitEvent(s, ev[nev - 1], 0) == cudaSuccess;
    cudaEvent_t in_done = nullptr;
    const bool joined_in = in && cudaEventCreateWithFlags(&in_done, cudaEventDisableTiming) ==
                                     cudaSuccess &&
                           cudaEventRecord(in_done, in) == cudaSuccess &&
                           cudaStreamWaitEvent(s, in_done, 0) == cudaSuccess;
    if (in_done) cudaEventDestroy(in_done);
    for (int i = 0; i < nev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);  // released once the stream work is done
    if (!joined || !joined_in) {  // queued copies must end before the free below
        cudaGetLastError();
        if (in) cudaStreamSynchronize(in);
        if (out) cudaStreamSynchronize(out);
        if (st == LINFORMER_OK) st = LINFORMER_ERR_LAUNCH;
    }
    workspace_free(base, s);
    if (cudaStreamSynchronize(s) != cudaSuccess && st == LINFORMER_OK) st = LINFORMER_ERR_LAUNCH;
    return st;
}

extern "C" int linformer_select_path(int b, int h, int n, int d, int k, int share_mode,
                                     int dtype) {
    int st = validate_common(b, h, n, d, k, share_mode, dtype);
    if (st) return st;
    return select_path(n, d, k, dtype);
}

extern "C" const char *linformer_status_string(int status) {
    switch (status) {
        case LINFORMER_OK: return "ok";
        case LINFORMER_ERR_NULL: return "a required pointer is NULL";
        case LINFORMER_ERR_SIZE: return "bad size (b, h, n, d, k must be >= 1 and fit)";
        case LINFORMER_ERR_UNSUPPORTED: return "unsupported shape (d <= 128, k <= 1024)";
        case LINFORMER_ERR_ENUM: return "bad share_mode or dtype";
        case LINFORMER_ERR_ALIGN: return "pointer not 16-byte aligned";
        case LINFORMER_ERR_F_MODE: return "F inconsistent with the sharing mode";
        case LINFORMER_ERR_ALLOC: return "workspace allocation failed";
        case LINFORMER_ERR_LAUNCH: return "CUDA call or kernel launch failed";
        case LINFORMER_ERR_DEVICE: return "device-side bounded wait ran out";
        default: return "unknown status";
    }
}

extern "C" int linformer_debug_read_device_status(void *stream) {
    cudaStream_t s = as_stream(stream);
    int *addr = device_status_ptr();
    if (!addr) return LINFORMER_ERR_LAUNCH;
    int value = 0;
    if (cudaMemcpyAsync(&value, addr, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(addr, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return LINFORMER_ERR_LAUNCH;
    return value ? LINFORMER_ERR_DEVICE : LINFORMER_OK;
}

extern "C" int linformer_set_pv_terms(int terms) {
    if (terms < 0 || terms > 3) return LINFORMER_ERR_ENUM;
    return g_pv_terms.exchange(terms);
}

extern "C" int64_t linformer_launch_count(void) { return g_launches.load(); }

extern "C" int linformer_profile_enable(int enable) {
    return g_profiling.exchange(enable ? 1 : 0);
}

extern "C" int linformer_profile_collect(double *ms, int64_t *launches) {
    std::vector<ProfileRecord> recs;
    {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        recs.swap(g_prof);
    }
    int st = LINFORMER_OK;
    for (auto &r : recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            st = LINFORMER_ERR_LAUNCH;
        if (r.id >= 0 && r.id < LINFORMER_KERNEL_COUNT) {
            if (ms) ms[r.id] += t;
            if (launches) launches[r.id] += 1;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    return st;
}

extern "C" const char *linformer_kernel_name(int id) {
    static const char *names[LINFORMER_KERNEL_COUNT] = {
        "tc_project_kernel", "tc_attend_kernel", "simt_project_kernel", "simt_attend_kernel",
        "window_projection_kernel", "backward_kernels", "dense_attention_kernels"};
    return (id >= 0 && id < LINFORMER_KERNEL_COUNT) ? names[id] : nullptr;
}
