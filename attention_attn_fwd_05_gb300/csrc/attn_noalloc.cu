// attn_noalloc.cu -- attn_fwd_noalloc: attn_fwd for callers that must not
// allocate device memory.
//
// attn_fwd keeps one small piece of scratch memory per device: the status
// word in which the bf16 kernel records a bounded-wait timeout.  It obtains
// that word with cudaMalloc on its first call on a device.  Some callers
// cannot allow that: code that runs with a fixed memory budget handed out by
// its own allocator (an inference server that owns every byte of the GPU),
// code called from inside a region where device allocation is forbidden or
// would synchronise the device, or a host library that must not touch the
// CUDA allocator at all.  This entry point runs the same kernels but keeps its
// scratch in a file-scope __device__ array that the CUDA module carries, so no
// call ever allocates.
#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

// Scratch of this entry point.  Word 0 is the bounded-wait status word of the
// bf16 kernel; the rest is reserved.  The kernels need kScratchNeeded bytes
// whatever B, H, N and d are, so no problem size can exceed kScratchBytes.
constexpr size_t kScratchBytes = 256;
constexpr size_t kScratchNeeded = sizeof(uint32_t);
static_assert(kScratchNeeded <= kScratchBytes, "scratch array too small");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchBytes / sizeof(uint32_t)];

constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per barrier wait, as attn_fwd

struct NoAllocDevice {
    bool ready = false;
    attn_status status = ATTN_OK;
    int sm_count = 0;
    uint32_t *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_na_mu;
NoAllocDevice g_na[kMaxDevices];

// Once per device, with that device current: check the architecture and look
// up the device address of the scratch array.  In host code the array's name
// is only a host-side stand-in, so the kernels get this looked-up address.
attn_status noalloc_setup(NoAllocDevice **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_na_mu);
    NoAllocDevice &s = g_na[dev];
    *out = &s;
    if (s.ready) return s.status;
    // Only a settled answer is cached (success, or a device of the wrong
    // architecture); a failed runtime call, for example one made while a
    // stream is being captured, is retried on the next call.
    int sm_count = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) {
        s.ready = true;
        s.status = ATTN_ERR_ARCH;
        return s.status;
    }
    uint32_t *addr = nullptr;
    if (check_launch(cudaGetSymbolAddress(reinterpret_cast<void **>(&addr), g_noalloc_scratch),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    s.sm_count = sm_count;
    s.scratch = addr;
    s.status = ATTN_OK;
    s.ready = true;
    return ATTN_OK;
}

bool is_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status device_pointer(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return ATTN_ERR_NOT_DEVICE;
    }
    if (a.type == cudaMemoryTypeManaged) return ATTN_OK;
    if (a.type != cudaMemoryTypeDevice) return ATTN_ERR_NOT_DEVICE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || a.device != dev) return ATTN_ERR_NOT_DEVICE;
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                                        float *lse, int64_t B, int64_t H, int64_t N, int64_t d,
                                        float scale, int causal, int dtype, void *stream) {
    // The same argument rules as attn_fwd.
    if (!q || !k || !v || !o) return ATTN_ERR_NULL;
    attn_status st = check_fwd_shape(B, H, N, d, dtype);
    if (st != ATTN_OK || (st = check_scale(scale)) != ATTN_OK) return st;
    const int64_t BH = B * H;
    if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o) ||
        !is_aligned16(lse))
        return ATTN_ERR_ALIGN;
    NoAllocDevice *s = nullptr;
    if ((st = noalloc_setup(&s)) != ATTN_OK) return st;
    for (const void *p : {q, k, v, static_cast<const void *>(o)})
        if ((st = device_pointer(p)) != ATTN_OK) return st;
    if (lse && (st = device_pointer(lse)) != ATTN_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // The status word must start each call at zero: a timeout left by an
    // earlier call would otherwise make this call's waits give up at once.
    if (check_launch(cudaMemsetAsync(s->scratch, 0, kScratchNeeded, cs), ATTN_ERR_CUDA) !=
        ATTN_OK)
        return ATTN_ERR_CUDA;
    const LaunchCtx ctx{cs, s->scratch, kTimeoutNs, s->sm_count};
    if (dtype == ATTN_BF16)
        return launch_attn_fwd_bf16(q, k, v, o, lse, BH, N, (int)d, scale, causal != 0, ctx);
    return launch_attn_fwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                               static_cast<const float *>(v), static_cast<float *>(o), lse, BH, N,
                               (int)d, scale, causal != 0, ctx);
}

extern "C" attn_status attn_fwd_noalloc_status(void *stream) {
    NoAllocDevice *s = nullptr;
    attn_status st = noalloc_setup(&s);
    if (st != ATTN_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // Read the word into host stack memory and clear it, in stream order after
    // the calls to be checked; nothing here allocates.
    uint32_t word = 0;
    if (check_launch(cudaStreamSynchronize(cs), ATTN_ERR_CUDA) != ATTN_OK ||
        check_launch(cudaMemcpyAsync(&word, s->scratch, sizeof(word), cudaMemcpyDeviceToHost, cs),
                     ATTN_ERR_CUDA) != ATTN_OK ||
        check_launch(cudaMemsetAsync(s->scratch, 0, sizeof(word), cs), ATTN_ERR_CUDA) != ATTN_OK ||
        check_launch(cudaStreamSynchronize(cs), ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    return status_from_word(word);
}
