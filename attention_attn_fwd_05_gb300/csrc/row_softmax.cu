// row_softmax.cu -- row softmax with a running maximum and sum.
//
// y[r, :] = exp(x[r, :] - max) / sum(exp(x[r, :] - max)), lse[r] = max + ln sum
// (page "14. Triton and kernel fusion", section "Fusion": subtract the row
// max, exponentiate, divide by the sum, reading the row once; and its
// exercise on rows longer than one block, done here with the online
// normalisation identity of page "Hardware Acceleration & Custom Kernels",
// section 2: m_new = max(m_old, x), d_new = d_old e^(m_old - m_new) + e^(x - m_new)).
//
// One CTA per row (grid-stride over rows).  Pass 1 walks the row once, each
// thread keeping its own (m, d) pair over 4-element groups; the pairs are
// merged across the CTA with the same identity.  Pass 2 writes the output,
// reading the row from shared memory when it was cached there in pass 1
// (rows up to kCacheFloats), otherwise from global memory again (L2-resident
// for moderate rows).  Any width is accepted; there is no 65536 cap.  -inf
// entries (masked positions) get probability 0; y may alias x.
#include <cmath>

#include "attn_internal.h"

namespace attn {
namespace rsm {

constexpr int NUM_THREADS = 512;
constexpr int kCacheFloats = 11 * 1024;  // 44 KB: static shared memory stays under 48 KB

struct MD {
    float m, d;
};

__device__ __forceinline__ MD merge(MD a, MD b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return {M, 0.f};
    return {M, a.d * expf(a.m - M) + b.d * expf(b.m - M)};
}

__global__ void __launch_bounds__(NUM_THREADS)
    row_softmax_kernel(const float *x, float *y, float *__restrict__ lse,
                       int64_t rows, int64_t width, int vec4) {
    __shared__ __align__(16) float cache[kCacheFloats];
    __shared__ MD warp_md[NUM_THREADS / 32];
    __shared__ MD row_md;
    const bool cached = width <= kCacheFloats;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *xr = x + r * width;
        float *yr = y + r * width;
        MD md{-INFINITY, 0.f};
        if (vec4) {
            const int64_t n4 = width / 4;
            for (int64_t i = threadIdx.x; i < n4; i += NUM_THREADS) {
                const float4 v = reinterpret_cast<const float4 *>(xr)[i];
                if (cached) reinterpret_cast<float4 *>(cache)[i] = v;
                const float gm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                const float M = fmaxf(md.m, gm);
                if (M == -INFINITY) continue;  // only masked (-inf) entries so far
                md.d = md.d * expf(md.m - M) + expf(v.x - M) + expf(v.y - M) + expf(v.z - M) +
                       expf(v.w - M);
                md.m = M;
            }
        } else {
            for (int64_t i = threadIdx.x; i < width; i += NUM_THREADS) {
                const float v = xr[i];
                if (cached) cache[i] = v;
                const float M = fmaxf(md.m, v);
                if (M == -INFINITY) continue;
                md.d = md.d * expf(md.m - M) + expf(v - M);
                md.m = M;
            }
        }
        // Threads that saw no element carry (-inf, 0); merge() handles them.
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            MD o{__shfl_xor_sync(0xffffffffu, md.m, off), __shfl_xor_sync(0xffffffffu, md.d, off)};
            md = merge(md, o);
        }
        if ((threadIdx.x & 31) == 0) warp_md[threadIdx.x >> 5] = md;
        __syncthreads();
        if (threadIdx.x < 32) {
            MD w = threadIdx.x < NUM_THREADS / 32 ? warp_md[threadIdx.x] : MD{-INFINITY, 0.f};
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                MD o{__shfl_xor_sync(0xffffffffu, w.m, off), __shfl_xor_sync(0xffffffffu, w.d, off)};
                w = merge(w, o);
            }
            if (threadIdx.x == 0) {
                row_md = w;
                if (lse != nullptr) lse[r] = w.m + logf(w.d);
            }
        }
        __syncthreads();
        const float M = row_md.m, inv_d = 1.f / row_md.d;
        if (vec4) {
            const int64_t n4 = width / 4;
            for (int64_t i = threadIdx.x; i < n4; i += NUM_THREADS) {
                const float4 v = cached ? reinterpret_cast<const float4 *>(cache)[i]
                                        : reinterpret_cast<const float4 *>(xr)[i];
                float4 o;
                o.x = expf(v.x - M) * inv_d;
                o.y = expf(v.y - M) * inv_d;
                o.z = expf(v.z - M) * inv_d;
                o.w = expf(v.w - M) * inv_d;
                reinterpret_cast<float4 *>(yr)[i] = o;
            }
        } else {
            for (int64_t i = threadIdx.x; i < width; i += NUM_THREADS) {
                const float v = cached ? cache[i] : xr[i];
                yr[i] = expf(v - M) * inv_d;
            }
        }
        __syncthreads();  // cache and row_md are reused by the next row
    }
}

}  // namespace rsm

attn_status launch_row_softmax(const float *x, float *y, float *lse, int64_t rows, int64_t width,
                               const LaunchCtx &ctx) {
    const bool vec4 = (width % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    const int64_t max_grid = (int64_t)ctx.sm_count * 4;
    const unsigned grid = (unsigned)(rows < max_grid ? rows : max_grid);
    rsm::row_softmax_kernel<<<grid, rsm::NUM_THREADS, 0, ctx.stream>>>(x, y, lse, rows, width,
                                                                       vec4 ? 1 : 0);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace attn
