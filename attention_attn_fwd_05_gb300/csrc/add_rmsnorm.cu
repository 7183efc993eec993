// add_rmsnorm.cu -- fused residual add + RMSNorm.
//
//   h   = x + residual                          (h = x without a residual)
//   out = h / sqrt(mean_c h_c^2 + eps) * weight
//   res_out = h                                 (with a residual)
//
// (page "14. Triton and kernel fusion", section "Fused residual add +
// RMSNorm": two reads and two writes in one pass instead of five; the
// normalisation formula of page "TritonForge").  Arithmetic is fp32 whatever
// the storage type; bf16 outputs are rounded once, on store.
//
// One CTA of 256 threads per row (grid-stride over rows).  Rows up to 8192
// elements whose width is a multiple of 8 keep h in registers between the
// two halves of the computation, so each input element is read once and each
// output written once: the kernel is bound by HBM bandwidth.  Other rows take
// a two-pass path that reads x (and residual) twice.
#include <cstdint>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace rms {

constexpr int NT = 256;
constexpr int VEC = 8;                    // elements per vector access
constexpr int MAXV = 4;                   // register-resident vectors per thread
constexpr int MAX_FAST = NT * VEC * MAXV;  // 8192

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8-element vector loads/stores as fp32.
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const uint16_t *p, float (&v)[8]) {
    const uint4 a = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(uint16_t *p, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}
__device__ __forceinline__ float load1(const float *p) { return *p; }
__device__ __forceinline__ float load1(const uint16_t *p) { return bf16_to_f32(*p); }
__device__ __forceinline__ void store1(float *p, float v) { *p = v; }
__device__ __forceinline__ void store1(uint16_t *p, float v) {
    *p = (uint16_t)(pack2(v, 0.f) & 0xffffu);
}

// Sum over the CTA; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = threadIdx.x < NT / 32 ? red[threadIdx.x] : 0.f;
    if (threadIdx.x < 32) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (threadIdx.x == 0) red[NT / 32] = t;
    }
    __syncthreads();
    const float s = red[NT / 32];
    __syncthreads();  // red is reused by the next row
    return s;
}

template <typename T>
__global__ void __launch_bounds__(NT)
    add_rmsnorm_kernel(const T *__restrict__ x, const T *__restrict__ res, const T *__restrict__ w,
                       T *__restrict__ out, T *__restrict__ res_out, int64_t rows, int width,
                       float eps, int fast) {
    __shared__ float red[NT / 32 + 1];
    const bool has_res = res != nullptr;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const T *xr = x + r * width;
        const T *rr = has_res ? res + r * width : nullptr;
        T *orow = out + r * width;
        T *hrow = has_res ? res_out + r * width : nullptr;
        if (fast) {
            const int nvec = width / VEC;
            float h[MAXV][VEC];
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
                const int vi = threadIdx.x + k * NT;
                if (vi < nvec) {
                    load8(xr + vi * VEC, h[k]);
                    if (has_res) {
                        float b[VEC];
                        load8(rr + vi * VEC, b);
#pragma unroll
                        for (int i = 0; i < VEC; ++i) h[k][i] += b[i];
                        store8(hrow + vi * VEC, h[k]);
                    }
#pragma unroll
                    for (int i = 0; i < VEC; ++i) ss = fmaf(h[k][i], h[k][i], ss);
                }
            }
            const float inv = 1.f / sqrtf(block_sum(ss, red) / (float)width + eps);
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
                const int vi = threadIdx.x + k * NT;
                if (vi < nvec) {
                    float g[VEC];
                    load8(w + vi * VEC, g);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) h[k][i] = h[k][i] * inv * g[i];
                    store8(orow + vi * VEC, h[k]);
                }
            }
        } else {
            float ss = 0.f;
            for (int c = threadIdx.x; c < width; c += NT) {
                float h = load1(xr + c);
                if (has_res) {
                    h += load1(rr + c);
                    store1(hrow + c, h);
                }
                ss = fmaf(h, h, ss);
            }
            const float inv = 1.f / sqrtf(block_sum(ss, red) / (float)width + eps);
            for (int c = threadIdx.x; c < width; c += NT) {
                float h = load1(xr + c);
                if (has_res) h += load1(rr + c);
                store1(orow + c, h * inv * load1(w + c));
            }
        }
    }
}

// ------------------------------------------------------------------ streamed ---
// The register-resident path with its input rows streamed: each CTA copies
// the x (and residual) rows of its next row into the other of two
// shared-memory stages with bulk async copies while it works on the current
// one, so reads stay in flight through the row's reduction and stores.

constexpr uint32_t ST_HDR = 256;  // two barriers, abort flag, reduction scratch

template <typename T>
__device__ __forceinline__ void load8s(const uint8_t *p, float (&v)[8]) {
    load8(reinterpret_cast<const T *>(p), v);
}

template <typename T, int KMAX>
__global__ void __launch_bounds__(NT)
    add_rmsnorm_stream_kernel(const T *__restrict__ x, const T *__restrict__ res,
                              const T *__restrict__ w, T *__restrict__ out,
                              T *__restrict__ res_out, int64_t rows, int width, float eps,
                              uint32_t *status, uint64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);  // barrier of stage s at sbase + 8s
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + 64);
    float *red = reinterpret_cast<float *>(sm + 96);  // [NT / 32 + 1]
    const bool has_res = res != nullptr;
    const uint32_t row_bytes = (uint32_t)width * (uint32_t)sizeof(T);
    const uint32_t stride = (row_bytes + 127u) & ~127u;
    const uint32_t stage_bytes = (has_res ? 2u : 1u) * stride;
    const int nvec = width / VEC;
    const WaitCtl ctl{abort_flag, status, timeout_ns};
    const int64_t G = gridDim.x;
    int n_issued = 0;  // rows of this CTA whose copies thread 0 started
    auto issue = [&]() {
        const int64_t row = (int64_t)blockIdx.x + (int64_t)n_issued * G;
        if (row >= rows) return;
        const uint32_t s = (uint32_t)(n_issued & 1), bar = sbase + 8u * s;
        const uint32_t dst = sbase + ST_HDR + s * stage_bytes;
        mbar_arrive_expect_tx(bar, (has_res ? 2u : 1u) * row_bytes);
        bulk_copy_g2s(dst, x + row * (int64_t)width, row_bytes, bar);
        if (has_res) bulk_copy_g2s(dst + stride, res + row * (int64_t)width, row_bytes, bar);
        ++n_issued;
    };
    if (threadIdx.x == 0) {
        mbar_init(sbase, 1);
        mbar_init(sbase + 8, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        issue();
        issue();
    }
    __syncthreads();

    int i = 0;
    for (int64_t r = blockIdx.x; r < rows; ++i, r += G) {
        const uint32_t s = (uint32_t)(i & 1);
        if (!__syncthreads_and(
                bounded_wait_warp(sbase + 8u * s, (uint32_t)(i >> 1) & 1u, ctl) ? 1 : 0))
            break;
        const uint8_t *sx = sm + ST_HDR + s * stage_bytes;
        float h[KMAX][VEC];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int vi = threadIdx.x + k * NT;
            if (vi < nvec) {
                load8s<T>(sx + (uint32_t)vi * VEC * sizeof(T), h[k]);
                if (has_res) {
                    float b[VEC];
                    load8s<T>(sx + stride + (uint32_t)vi * VEC * sizeof(T), b);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) h[k][e] += b[e];
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) ss = fmaf(h[k][e], h[k][e], ss);
            }
        }
        // block_sum's barriers also mean every thread is done with stage s.
        const float inv = 1.f / sqrtf(block_sum(ss, red) / (float)width + eps);
        if (threadIdx.x == 0) issue();  // row i + 2 into stage s
        T *orow = out + r * (int64_t)width;
        T *hrow = has_res ? res_out + r * (int64_t)width : nullptr;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int vi = threadIdx.x + k * NT;
            if (vi < nvec) {
                if (has_res) store8(hrow + vi * VEC, h[k]);
                float g[VEC];
                load8(w + vi * VEC, g);
#pragma unroll
                for (int e = 0; e < VEC; ++e) h[k][e] = h[k][e] * inv * g[e];
                store8(orow + vi * VEC, h[k]);
            }
        }
    }
    // After a timeout, let copies still in flight land before the CTA exits.
    if (threadIdx.x == 0 && *abort_flag != 0u) {
        for (int c = i; c < n_issued; ++c) {
            const uint32_t bar = sbase + 8u * (uint32_t)(c & 1);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, (uint32_t)(c >> 1) & 1u))
                if (globaltimer_ns() - t0 > timeout_ns) break;
        }
    }
}

template <typename T>
static attn_status launch_stream(const T *x, const T *residual, const T *weight, T *out,
                                 T *res_out, int64_t rows, int width, float eps,
                                 const LaunchCtx &ctx) {
    const uint32_t stride = ((uint32_t)width * (uint32_t)sizeof(T) + 127u) & ~127u;
    const int smem = (int)(ST_HDR + 2u * (residual ? 2u : 1u) * stride);
    auto kern = add_rmsnorm_stream_kernel<T, MAXV>;
    if (check_launch(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    int per_sm = 0;
    if (check_launch(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    const int64_t max_grid = (int64_t)ctx.sm_count * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(rows < max_grid ? rows : max_grid);
    kern<<<grid, NT, smem, ctx.stream>>>(x, residual, weight, out, res_out, rows, width, eps,
                                         ctx.status, ctx.timeout_ns);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace rms

attn_status launch_add_rmsnorm(const void *x, const void *residual, const void *weight, void *out,
                               void *res_out, int64_t rows, int64_t width, float eps, int dtype,
                               const LaunchCtx &ctx) {
    const int fast = (width % rms::VEC == 0 && width <= rms::MAX_FAST) ? 1 : 0;
    if (fast && dtype != ATTN_F32)
        return rms::launch_stream<uint16_t>(
            static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(residual),
            static_cast<const uint16_t *>(weight), static_cast<uint16_t *>(out),
            static_cast<uint16_t *>(res_out), rows, (int)width, eps, ctx);
    const int64_t max_grid = (int64_t)ctx.sm_count * 8;
    const unsigned grid = (unsigned)(rows < max_grid ? rows : max_grid);
    if (dtype == ATTN_F32) {
        rms::add_rmsnorm_kernel<float><<<grid, rms::NT, 0, ctx.stream>>>(
            static_cast<const float *>(x), static_cast<const float *>(residual),
            static_cast<const float *>(weight), static_cast<float *>(out),
            static_cast<float *>(res_out), rows, (int)width, eps, fast);
    } else {
        rms::add_rmsnorm_kernel<uint16_t><<<grid, rms::NT, 0, ctx.stream>>>(
            static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(residual),
            static_cast<const uint16_t *>(weight), static_cast<uint16_t *>(out),
            static_cast<uint16_t *>(res_out), rows, (int)width, eps, fast);
    }
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace attn
