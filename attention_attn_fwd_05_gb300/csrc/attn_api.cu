// attn_api.cu -- the C ABI: argument validation, per-device state, dispatch.
//
// Validation follows the pages' convention of checking shapes, contiguity
// and device placement before any launch (page "TritonForge", the
// shape_validator / device-placement layers of its fallback router; page
// "14. Triton and kernel fusion", the ValueError checks of its wrappers) --
// but an invalid call returns an error code instead of routing elsewhere:
// there is no fallback path.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per barrier wait

struct DeviceState {
    bool ready = false;
    attn_status init_status = ATTN_OK;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;  // 256 bytes of device memory, first word used
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Set up (once) and return the state of the current device.
attn_status device_state(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        s.ready = true;
        s.init_status = ATTN_ERR_CUDA;
        if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) ==
                cudaSuccess &&
            cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev) ==
                cudaSuccess &&
            cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) ==
                cudaSuccess) {
            if (s.cc_major != 10 || s.cc_minor != 3) {
                s.init_status = ATTN_ERR_ARCH;
            } else if (cudaMalloc(reinterpret_cast<void **>(&s.status), 256) == cudaSuccess &&
                       cudaMemset(s.status, 0, 256) == cudaSuccess) {
                s.init_status = ATTN_OK;
            }
        }
    }
    *out = &s;
    return s.init_status;
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

extern "C" attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                                int causal, int dtype, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_NULL;
    if (B < 1 || H < 1 || N < 1 || N > INT32_MAX || !product_fits(B, H, N, d > 0 ? d : 1))
        return ATTN_ERR_SHAPE;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
    if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
    const int64_t BH = B * H;
    if (dtype == ATTN_BF16 && (N > kMaxNBf16 || BH > INT32_MAX || BH * ((N + 255) / 256) > INT32_MAX))
        return ATTN_ERR_SHAPE;
    if (dtype == ATTN_F32 && (BH > 65535 || (N + 31) / 32 > INT32_MAX)) return ATTN_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_ALIGN;
    DeviceState *s = nullptr;
    attn_status st = device_state(&s);
    if (st != ATTN_OK) return st;
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
    return word ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
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
        default: return "unknown status";
    }
}

extern "C" const char *attn_last_cuda_error(void) {
    return cudaGetErrorString(t_last_error);
}

extern "C" int attn_version(void) { return 10000; }
