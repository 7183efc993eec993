// attn_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn_fwd.h"

namespace attn {

// Everything a kernel launch needs besides the tensors themselves.
struct LaunchCtx {
    cudaStream_t stream;
    uint32_t *status;     // device status word (bounded-wait timeouts)
    uint64_t timeout_ns;  // limit for one barrier wait inside a kernel
    int sm_count;
};

// bf16 path: tcgen05 tensor-core kernel (attn_fwd_tc.cu).
attn_status launch_attn_fwd_bf16(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int64_t BH, int64_t N, int d, float scale, bool causal,
                                 const LaunchCtx &ctx);

// fp32 path: exact CUDA-core kernel (attn_fwd_f32.cu).
attn_status launch_attn_fwd_f32(const float *q, const float *k, const float *v, float *o,
                                float *lse, int64_t BH, int64_t N, int d, float scale,
                                bool causal, const LaunchCtx &ctx);

// Row softmax (row_softmax.cu).
attn_status launch_row_softmax(const float *x, float *y, float *lse, int64_t rows, int64_t width,
                               const LaunchCtx &ctx);

// [BH, N, d] bf16 tensor map with 64-column x 128-row boxes and 128-byte
// swizzle (attn_fwd_tc.cu); false if the driver entry point or the encode fails.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t BH, int64_t N, int d);

// D = rowsum(dO * O) for the backward (attn_bwd.cu).
attn_status launch_bwd_delta(const void *o, const void *dout, float *delta, int64_t rows, int d,
                             int dtype, const LaunchCtx &ctx);

// bf16 attention backward on tensor cores (attn_bwd_tc.cu); delta must hold D.
attn_status launch_attn_bwd_bf16_tc(const void *q, const void *k, const void *v, const void *dout,
                                    const float *lse, const float *delta, void *dq, void *dk,
                                    void *dv, int64_t BH, int64_t N, int d, float scale,
                                    bool causal, const LaunchCtx &ctx);

// Attention backward (attn_bwd.cu).
attn_status launch_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, float *delta, void *dq, void *dk,
                            void *dv, int64_t BH, int64_t N, int d, float scale, bool causal,
                            int dtype, const LaunchCtx &ctx);

// Residual add + RMSNorm (add_rmsnorm.cu).
attn_status launch_add_rmsnorm(const void *x, const void *residual, const void *weight, void *out,
                               void *res_out, int64_t rows, int64_t width, float eps, int dtype,
                               const LaunchCtx &ctx);

// Bounded-wait self test (attn_fwd_tc.cu).
attn_status launch_wait_selftest(const LaunchCtx &ctx);

// Record `e` (if it is an error) as this thread's last CUDA error and return
// `on_error`, else ATTN_OK.  Used right after every launch.
attn_status check_launch(cudaError_t e, attn_status on_error);

// Largest N the bf16 path accepts.  The kernels' grids are 1-D (the items
// are counted by the B*H*ceil(N/256) < 2^31 rule of check_fwd_shape) and
// their row and key indices are 32-bit, so no index limit binds below 2^31;
// the cap is a tested-range limit (GPU parity reaches N = 131072 on sampled
// rows; a host test checks the rejection just above the cap).
constexpr int64_t kMaxNBf16 = 65535LL * 128;

// Shape, dtype and head-dim rules of attn_fwd (ATTN_OK or the error code),
// shared by attn_fwd, attn_fwd_noalloc and attn_fwd_host.
attn_status check_fwd_shape(int64_t B, int64_t H, int64_t N, int64_t d, int dtype);

// The attn_status a device status word stands for (ATTN_OK when it is 0).
attn_status status_from_word(uint32_t word);

// ATTN_OK for a usable softmax multiplier (finite, |scale| <= 2e38), else
// ATTN_ERR_SCALE.  Shared by every entry point that takes a scale.
attn_status check_scale(float scale);

}  // namespace attn
