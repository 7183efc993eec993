// attn_api.cu -- the C ABI: argument validation, per-device state, dispatch.
//
// Validation follows the pages' convention of checking shapes, contiguity
// and device placement before any launch (page "TritonForge", the
// shape_validator / device-placement layers of its fallback router; page
// "14. Triton and kernel fusion", the ValueError checks of its wrappers) --
// but an invalid call returns an error code instead of routing elsewhere:
// there is no fallback path.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per barrier wait

constexpr int kHostMaxChunks = 8;  // attn_fwd_host: chunks of batch*head per call

struct DeviceState {
    bool ready = false;
    attn_status init_status = ATTN_OK;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;  // 256 bytes of device memory, first word used
    // attn_fwd_host: copy streams and events, made on its first call; `host_mu`
    // serialises the calls that enqueue work on them.
    bool host_ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev[2 + 2 * kHostMaxChunks] = {};
    std::mutex host_mu;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Set up (once) and return the state of the current device.
attn_status device_state(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &s = g_dev[dev];
    *out = &s;
    if (s.ready) return s.init_status;
    // Only a settled answer is cached (success, or a device of the wrong
    // architecture); a failed runtime call, for example one made while a
    // stream is being captured, is retried on the next call.
    int sm_count = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    s.sm_count = sm_count;
    s.cc_major = major;
    s.cc_minor = minor;
    if (major != 10 || minor != 3) {
        s.ready = true;
        s.init_status = ATTN_ERR_ARCH;
        return s.init_status;
    }
    uint32_t *word = nullptr;
    if (check_launch(cudaMalloc(reinterpret_cast<void **>(&word), 256), ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    if (check_launch(cudaMemset(word, 0, 256), ATTN_ERR_CUDA) != ATTN_OK) {
        (void)cudaFree(word);
        return ATTN_ERR_CUDA;
    }
    s.status = word;
    s.init_status = ATTN_OK;
    s.ready = true;
    return ATTN_OK;
}

// A device pointer usable by kernels on the current device.
attn_status check_device_ptr(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // clear the sticky-free error this can leave
        return ATTN_ERR_NOT_DEVICE;
    }
    if (a.type == cudaMemoryTypeManaged) return ATTN_OK;
    if (a.type != cudaMemoryTypeDevice) return ATTN_ERR_NOT_DEVICE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || a.device != dev) return ATTN_ERR_NOT_DEVICE;
    return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Overflow-free a*b*c*d < 2^62 for positive factors.
bool product_fits(int64_t a, int64_t b, int64_t c, int64_t d) {
    const int64_t lim = (int64_t)1 << 62;
    int64_t p = a;
    for (int64_t f : {b, c, d}) {
        if (p > lim / f) return false;
        p *= f;
    }
    return p < lim;
}

LaunchCtx make_ctx(const DeviceState &s, void *stream, uint64_t timeout_ns) {
    return LaunchCtx{static_cast<cudaStream_t>(stream), s.status, timeout_ns, s.sm_count};
}

thread_local cudaError_t t_last_error = cudaSuccess;

}  // namespace

attn_status check_launch(cudaError_t e, attn_status on_error) {
    if (e == cudaSuccess) return ATTN_OK;
    t_last_error = e;
    return on_error;
}

}  // namespace attn

using namespace attn;

namespace attn {

// Shape, dtype and head-dim rules of attn_fwd, shared by every forward entry
// point (no pointer checks).
attn_status check_fwd_shape(int64_t B, int64_t H, int64_t N, int64_t d, int dtype) {
    if (B < 1 || H < 1 || N < 1 || N > INT32_MAX || !product_fits(B, H, N, d > 0 ? d : 1))
        return ATTN_ERR_SHAPE;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
    if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
    const int64_t BH = B * H;
    if (dtype == ATTN_BF16 &&
        (N > kMaxNBf16 || BH > INT32_MAX || BH * ((N + 255) / 256) > INT32_MAX))
        return ATTN_ERR_SHAPE;
    if (dtype == ATTN_F32 && (BH > 65535 || (N + 31) / 32 > INT32_MAX)) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

// The attn_status a non-zero device status word stands for: an out-of-range
// access found by the bounds-checking debug build comes first (it usually
// also leaves a wait to time out), then a timeout.
attn_status status_from_word(uint32_t word) {
    if (word & STATUS_BOUNDS) return ATTN_ERR_DEVICE_BOUNDS;
    if (word & STATUS_TIMEOUT) return ATTN_ERR_DEVICE_TIMEOUT;
    return ATTN_OK;
}

// The softmax multiplier: any finite value.  Beyond about 2.3e38 its base-2
// form (scale * log2 e), which the kernels use, would overflow, so those are
// rejected with NaN and the infinities.
attn_status check_scale(float scale) {
    return std::fabs(scale) <= 2.0e38f ? ATTN_OK : ATTN_ERR_SCALE;
}

}  // namespace attn

extern "C" attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                                int causal, int dtype, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_NULL;
    attn_status st = check_fwd_shape(B, H, N, d, dtype);
    if (st != ATTN_OK || (st = check_scale(scale)) != ATTN_OK) return st;
    const int64_t BH = B * H;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    if ((st = device_state(&s)) != ATTN_OK) return st;
    for (const void *p : {q, k, v, static_cast<const void *>(o)})
        if ((st = check_device_ptr(p)) != ATTN_OK) return st;
    if (lse && (st = check_device_ptr(lse)) != ATTN_OK) return st;
    const LaunchCtx ctx = make_ctx(*s, stream, kDefaultTimeoutNs);
    if (dtype == ATTN_BF16)
        return launch_attn_fwd_bf16(q, k, v, o, lse, BH, N, (int)d, scale, causal != 0, ctx);
    return launch_attn_fwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                               static_cast<const float *>(v), static_cast<float *>(o), lse, BH, N,
                               (int)d, scale, causal != 0, ctx);
}

namespace {

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace layout of attn_fwd_host: Q, K, V, O, LSE, each 256-byte aligned.
struct HostLayout {
    size_t tensor, lse, total;
};
HostLayout host_layout(int64_t B, int64_t H, int64_t N, int64_t d, int dtype) {
    const size_t elt = dtype == ATTN_F32 ? 4 : 2;
    const size_t tensor = round256((size_t)(B * H * N * d) * elt);
    const size_t lse = round256((size_t)(B * H * N) * 4);
    return {tensor, lse, 4 * tensor + lse};
}

attn_status host_setup(DeviceState &s) {
    if (s.host_ready) return ATTN_OK;
    if (cudaStreamCreateWithFlags(&s.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&s.s_out, cudaStreamNonBlocking) != cudaSuccess)
        return ATTN_ERR_CUDA;
    for (cudaEvent_t &e : s.ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return ATTN_ERR_CUDA;
    s.host_ready = true;
    return ATTN_OK;
}

}  // namespace

extern "C" size_t attn_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d,
                                                int dtype) {
    if (check_fwd_shape(B, H, N, d, dtype) != ATTN_OK) return 0;
    return host_layout(B, H, N, d, dtype).total;
}

extern "C" attn_status attn_fwd_host(const void *q, const void *k, const void *v, void *o,
                                     float *lse, int64_t B, int64_t H, int64_t N, int64_t d,
                                     float scale, int causal, int dtype, void *workspace,
                                     size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !o || !workspace) return ATTN_ERR_NULL;
    attn_status st = check_fwd_shape(B, H, N, d, dtype);
    if (st != ATTN_OK || (st = check_scale(scale)) != ATTN_OK) return st;
    const HostLayout lay = host_layout(B, H, N, d, dtype);
    if (workspace_bytes < lay.total) return ATTN_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    if ((st = device_state(&s)) != ATTN_OK) return st;
    if ((st = check_device_ptr(workspace)) != ATTN_OK) return st;
    std::lock_guard<std::mutex> lk(s->host_mu);
    if ((st = host_setup(*s)) != ATTN_OK) return st;

    const int64_t BH = B * H;
    const size_t elt = dtype == ATTN_F32 ? 4 : 2;
    const size_t head = (size_t)N * (size_t)d * elt, head_lse = (size_t)N * 4;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *dq = ws, *dk = ws + lay.tensor, *dv = ws + 2 * lay.tensor, *dout = ws + 3 * lay.tensor;
    float *dlse = reinterpret_cast<float *>(ws + 4 * lay.tensor);
    // Chunks of consecutive (batch, head) pairs, about 16 MB of copies or more
    // each, at most kHostMaxChunks: the copy in of chunk c+1, the forward of
    // chunk c and the copy out of chunk c-1 overlap.
    const size_t bytes = (size_t)BH * (4 * head + head_lse);
    int64_t nc = (int64_t)(bytes / (16u << 20));
    if (nc > kHostMaxChunks) nc = kHostMaxChunks;
    if (nc > BH) nc = BH;
    if (nc < 1) nc = 1;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaEvent_t e_start = s->ev[0], e_done = s->ev[1];
    const LaunchCtx ctx = make_ctx(*s, stream, kDefaultTimeoutNs);
    // Work already on `stream` (earlier users of the workspace or the host
    // buffers) comes first.
    if ((st = check_launch(cudaEventRecord(e_start, cs), ATTN_ERR_CUDA)) != ATTN_OK ||
        (st = check_launch(cudaStreamWaitEvent(s->s_in, e_start, 0), ATTN_ERR_CUDA)) !=
            ATTN_OK ||
        (st = check_launch(cudaStreamWaitEvent(s->s_out, e_start, 0), ATTN_ERR_CUDA)) != ATTN_OK)
        return st;
    for (int64_t c = 0; c < nc; ++c) {
        const int64_t h0 = BH * c / nc, h1 = BH * (c + 1) / nc, nh = h1 - h0;
        const size_t off = (size_t)h0 * head, len = (size_t)nh * head;
        cudaEvent_t e_in = s->ev[2 + 2 * c], e_comp = s->ev[3 + 2 * c];
        // One copy per tensor and chunk.
        for (int t = 0; t < 3; ++t) {
            const uint8_t *src = static_cast<const uint8_t *>(t == 0 ? q : (t == 1 ? k : v));
            uint8_t *dst = t == 0 ? dq : (t == 1 ? dk : dv);
            if ((st = check_launch(cudaMemcpyAsync(dst + off, src + off, len, cudaMemcpyDefault,
                                                   s->s_in),
                                   ATTN_ERR_CUDA)) != ATTN_OK)
                return st;
        }
        if ((st = check_launch(cudaEventRecord(e_in, s->s_in), ATTN_ERR_CUDA)) != ATTN_OK ||
            (st = check_launch(cudaStreamWaitEvent(cs, e_in, 0), ATTN_ERR_CUDA)) != ATTN_OK)
            return st;
        float *lse_c = lse ? dlse + h0 * N : nullptr;
        st = dtype == ATTN_BF16
                 ? launch_attn_fwd_bf16(dq + off, dk + off, dv + off, dout + off, lse_c, nh, N,
                                        (int)d, scale, causal != 0, ctx)
                 : launch_attn_fwd_f32(reinterpret_cast<const float *>(dq + off),
                                       reinterpret_cast<const float *>(dk + off),
                                       reinterpret_cast<const float *>(dv + off),
                                       reinterpret_cast<float *>(dout + off), lse_c, nh, N,
                                       (int)d, scale, causal != 0, ctx);
        if (st != ATTN_OK) return st;
        if ((st = check_launch(cudaEventRecord(e_comp, cs), ATTN_ERR_CUDA)) != ATTN_OK ||
            (st = check_launch(cudaStreamWaitEvent(s->s_out, e_comp, 0), ATTN_ERR_CUDA)) !=
                ATTN_OK ||
            (st = check_launch(cudaMemcpyAsync(static_cast<uint8_t *>(o) + off, dout + off, len,
                                               cudaMemcpyDefault, s->s_out),
                               ATTN_ERR_CUDA)) != ATTN_OK)
            return st;
        if (lse &&
            (st = check_launch(cudaMemcpyAsync(lse + h0 * N, lse_c, (size_t)nh * head_lse,
                                               cudaMemcpyDefault, s->s_out),
                               ATTN_ERR_CUDA)) != ATTN_OK)
            return st;
    }
    // Everything, the last copy out included, is ordered before later work on `stream`.
    if ((st = check_launch(cudaEventRecord(e_done, s->s_out), ATTN_ERR_CUDA)) != ATTN_OK)
        return st;
    return check_launch(cudaStreamWaitEvent(cs, e_done, 0), ATTN_ERR_CUDA);
}

extern "C" attn_status attn_row_softmax(const float *x, float *y, float *lse, int64_t rows,
                                        int64_t width, void *stream) {
    if (!x || !y) return ATTN_ERR_NULL;
    if (rows < 1 || width < 1 || !product_fits(rows, width, 1, 1)) return ATTN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
    if ((st = check_device_ptr(x)) != ATTN_OK || (st = check_device_ptr(y)) != ATTN_OK) return st;
    if (lse && (st = check_device_ptr(lse)) != ATTN_OK) return st;
    return launch_row_softmax(x, y, lse, rows, width, make_ctx(*s, stream, kDefaultTimeoutNs));
}

extern "C" attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, float *delta, void *dq,
                                void *dk, void *dv, int64_t B, int64_t H, int64_t N, int64_t d,
                                float scale, int causal, int dtype, void *stream) {
    if (!q || !k || !v || !o || !dout || !lse || !delta || !dq || !dk || !dv)
        return ATTN_ERR_NULL;
    if (B < 1 || H < 1 || N < 1 || N > INT32_MAX || !product_fits(B, H, N, d > 0 ? d : 1))
        return ATTN_ERR_SHAPE;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
    if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
    if (B * H > 65535) return ATTN_ERR_SHAPE;
    if (check_scale(scale) != ATTN_OK) return ATTN_ERR_SCALE;
    for (const void *p : {q, k, v, o, dout, static_cast<const void *>(lse),
                          static_cast<const void *>(delta), static_cast<const void *>(dq),
                          static_cast<const void *>(dk), static_cast<const void *>(dv)})
        if (!aligned16(p)) return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
    for (const void *p : {q, k, v, o, dout, static_cast<const void *>(lse),
                          static_cast<const void *>(delta), static_cast<const void *>(dq),
                          static_cast<const void *>(dk), static_cast<const void *>(dv)})
        if ((st = check_device_ptr(p)) != ATTN_OK) return st;
    return launch_attn_bwd(q, k, v, o, dout, lse, delta, dq, dk, dv, B * H, N, (int)d, scale,
                           causal != 0, dtype, make_ctx(*s, stream, kDefaultTimeoutNs));
}

extern "C" attn_status attn_add_rmsnorm(const void *x, const void *residual, const void *weight,
                                        void *out, void *res_out, int64_t rows, int64_t width,
                                        float eps, int dtype, void *stream) {
    if (!x || !weight || !out || (residual && !res_out)) return ATTN_ERR_NULL;
    if (rows < 1 || width < 1 || width > INT32_MAX || !product_fits(rows, width, 1, 1))
        return ATTN_ERR_SHAPE;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(out) ||
        !aligned16(res_out))
        return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
    for (const void *p : {x, weight, static_cast<const void *>(out)})
        if ((st = check_device_ptr(p)) != ATTN_OK) return st;
    if (residual && ((st = check_device_ptr(residual)) != ATTN_OK ||
                     (st = check_device_ptr(res_out)) != ATTN_OK))
        return st;
    return launch_add_rmsnorm(x, residual, weight, out, residual ? res_out : nullptr, rows, width,
                              eps, dtype, make_ctx(*s, stream, kDefaultTimeoutNs));
}

extern "C" attn_status attn_device_status(void *stream) {
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return ATTN_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, s->status, sizeof(word), cudaMemcpyDeviceToHost, cs) !=
            cudaSuccess ||
        cudaMemsetAsync(s->status, 0, sizeof(word), cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return status_from_word(word);
}

extern "C" attn_status attn_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
    if (timeout_ns < 1000ull) timeout_ns = 1000ull;
    if (timeout_ns > 5000000000ull) timeout_ns = 5000000000ull;
    if ((st = launch_wait_selftest(make_ctx(*s, stream, timeout_ns))) != ATTN_OK) return st;
    return attn_device_status(stream);
}

extern "C" const char *attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "null pointer argument";
        case ATTN_ERR_SHAPE: return "invalid or unsupported shape";
        case ATTN_ERR_DTYPE: return "unknown dtype";
        case ATTN_ERR_HEADDIM: return "head dimension must be 64 or 128";
        case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ATTN_ERR_ARCH: return "device is not sm_103 (compute capability 10.3)";
        case ATTN_ERR_LAUNCH: return "kernel launch failed";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (device timeout)";
        case ATTN_ERR_NOT_DEVICE: return "pointer is not device memory of the current device";
        case ATTN_ERR_CUDA: return "CUDA runtime call failed";
        case ATTN_ERR_SCALE: return "scale is not finite (or |scale| > 2e38)";
        case ATTN_ERR_DEVICE_BOUNDS:
            return "a kernel found an index out of range (bounds-checking build)";
        default: return "unknown status";
    }
}

extern "C" const char *attn_last_cuda_error(void) {
    return cudaGetErrorString(t_last_error);
}

extern "C" int attn_version(void) { return 10200; }
