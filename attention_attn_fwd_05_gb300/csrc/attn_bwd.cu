// attn_bwd.cu -- attention backward on CUDA cores, fp32 arithmetic (the fp32
// path; bf16 goes to the tensor-core kernels of attn_bwd_tc.cu after the D
// kernel here).
//
// The exact gradient of O = softmax(scale Q K^T) V, using the forward's saved
// O and LSE (the pages give no attention backward; this is the plain
// derivative of the forward formula of page "Hardware Acceleration & Custom
// Kernels", section 2):
//     P_ij  = exp(scale q_i.k_j - LSE_i)         (0 for masked keys)
//     D_i   = dO_i . O_i
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
//     dV_j  = sum_i P_ij dO_i
//
// Three launches, no atomics: (1) D for every row; (2) per group of keys,
// walk the queries that see them and accumulate dK, dV in registers; (3) per
// group of queries, walk their keys and accumulate dQ.  Work layout as in the
// exact-fp32 forward: TPR threads share a row, each owning D/TPR dimensions
// in 16-byte chunks interleaved across the TPR threads; tiles of the other
// operand are staged in shared memory (fp32) and read as broadcasts.
#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace bwd {

constexpr int NT = 128;
constexpr int BT = 32;  // rows of the other operand per shared-memory tile

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const uint16_t *p) {
    return __uint_as_float((uint32_t)*p << 16);
}
__device__ __forceinline__ void st(float *p, float v) { *p = v; }
__device__ __forceinline__ void st(uint16_t *p, float v) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(v));
    *p = (uint16_t)(r & 0xffffu);
}

// D_i = dO_i . O_i, one warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(256)
    bwd_delta_kernel(const T *__restrict__ o, const T *__restrict__ dout,
                     float *__restrict__ delta, int64_t rows) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    float acc = 0.f;
#pragma unroll
    for (int c = lane; c < D; c += 32) acc = fmaf(ld(dout + r * D + c), ld(o + r * D + c), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[r] = acc;
}

// Stage rows [r0, r0 + BT) of a [N, D] slice into shared memory as fp32
// (zeros beyond N).
template <typename T, int D>
__device__ __forceinline__ void stage(float *dst, const T *src, int r0, int N) {
    for (int e = threadIdx.x; e < BT * D; e += NT) {
        const int r = r0 + e / D;
        dst[e] = r < N ? ld(src + (size_t)r * D + (e % D)) : 0.f;
    }
}

// dK and dV for ROWS = NT / TPR keys per CTA.
template <typename T, int D, int TPR>
__global__ void __launch_bounds__(NT)
    bwd_dkdv_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                    const T *__restrict__ dO, const float *__restrict__ LSE,
                    const float *__restrict__ DEL, T *__restrict__ dK, T *__restrict__ dV, int N,
                    float scale, int causal) {
    constexpr int ROWS = NT / TPR;
    constexpr int NCH = D / 4 / TPR;
    __shared__ __align__(16) float qs[BT * D];
    __shared__ __align__(16) float gs[BT * D];
    __shared__ float ls[BT], ds_[BT];
    const int bh = blockIdx.y;
    const int j0 = blockIdx.x * ROWS;
    const int lr = threadIdx.x / TPR, part = threadIdx.x % TPR;
    const int j = j0 + lr;
    const bool valid = j < N;
    const size_t base = (size_t)bh * N * D;
    float kr[NCH * 4], vr[NCH * 4], dk[NCH * 4], dv[NCH * 4];
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * (ci * TPR + part) + e;
            kr[4 * ci + e] = valid ? ld(K + base + (size_t)j * D + c) : 0.f;
            vr[4 * ci + e] = valid ? ld(V + base + (size_t)j * D + c) : 0.f;
            dk[4 * ci + e] = dv[4 * ci + e] = 0.f;
        }
    // Queries that can see a key of this group: all, or i >= j0 with the mask.
    for (int i0 = causal ? (j0 / BT) * BT : 0; i0 < N; i0 += BT) {
        __syncthreads();
        stage<T, D>(qs, Q + base, i0, N);
        stage<T, D>(gs, dO + base, i0, N);
        if (threadIdx.x < BT) {
            const int i = i0 + threadIdx.x;
            ls[threadIdx.x] = i < N ? LSE[(size_t)bh * N + i] : 0.f;
            ds_[threadIdx.x] = i < N ? DEL[(size_t)bh * N + i] : 0.f;
        }
        __syncthreads();
        const int nq = min(BT, N - i0);
        for (int ii = 0; ii < nq; ++ii) {
            const int i = i0 + ii;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 qv = *reinterpret_cast<const float4 *>(qs + ii * D + 4 * (ci * TPR + part));
                const float4 gv = *reinterpret_cast<const float4 *>(gs + ii * D + 4 * (ci * TPR + part));
                s = fmaf(qv.x, kr[4 * ci + 0], fmaf(qv.y, kr[4 * ci + 1], fmaf(qv.z, kr[4 * ci + 2], fmaf(qv.w, kr[4 * ci + 3], s))));
                dp = fmaf(gv.x, vr[4 * ci + 0], fmaf(gv.y, vr[4 * ci + 1], fmaf(gv.z, vr[4 * ci + 2], fmaf(gv.w, vr[4 * ci + 3], dp))));
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) {
                s += __shfl_xor_sync(0xffffffffu, s, off);
                dp += __shfl_xor_sync(0xffffffffu, dp, off);
            }
            const bool vis = valid && (!causal || j <= i);
            const float p = vis ? expf(scale * s - ls[ii]) : 0.f;
            const float gsc = scale * p * (dp - ds_[ii]);
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 qv = *reinterpret_cast<const float4 *>(qs + ii * D + 4 * (ci * TPR + part));
                const float4 gv = *reinterpret_cast<const float4 *>(gs + ii * D + 4 * (ci * TPR + part));
                dv[4 * ci + 0] = fmaf(p, gv.x, dv[4 * ci + 0]);
                dv[4 * ci + 1] = fmaf(p, gv.y, dv[4 * ci + 1]);
                dv[4 * ci + 2] = fmaf(p, gv.z, dv[4 * ci + 2]);
                dv[4 * ci + 3] = fmaf(p, gv.w, dv[4 * ci + 3]);
                dk[4 * ci + 0] = fmaf(gsc, qv.x, dk[4 * ci + 0]);
                dk[4 * ci + 1] = fmaf(gsc, qv.y, dk[4 * ci + 1]);
                dk[4 * ci + 2] = fmaf(gsc, qv.z, dk[4 * ci + 2]);
                dk[4 * ci + 3] = fmaf(gsc, qv.w, dk[4 * ci + 3]);
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 4 * (ci * TPR + part) + e;
                st(dK + base + (size_t)j * D + c, dk[4 * ci + e]);
                st(dV + base + (size_t)j * D + c, dv[4 * ci + e]);
            }
    }
}

// dQ for ROWS = NT / TPR queries per CTA.
template <typename T, int D, int TPR>
__global__ void __launch_bounds__(NT)
    bwd_dq_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                  const T *__restrict__ dO, const float *__restrict__ LSE,
                  const float *__restrict__ DEL, T *__restrict__ dQ, int N, float scale,
                  int causal) {
    constexpr int ROWS = NT / TPR;
    constexpr int NCH = D / 4 / TPR;
    __shared__ __align__(16) float ks[BT * D];
    __shared__ __align__(16) float vs[BT * D];
    const int bh = blockIdx.y;
    const int i0 = blockIdx.x * ROWS;
    const int lr = threadIdx.x / TPR, part = threadIdx.x % TPR;
    const int i = i0 + lr;
    const bool valid = i < N;
    const size_t base = (size_t)bh * N * D;
    float qr[NCH * 4], gr[NCH * 4], dq[NCH * 4];
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * (ci * TPR + part) + e;
            qr[4 * ci + e] = valid ? ld(Q + base + (size_t)i * D + c) : 0.f;
            gr[4 * ci + e] = valid ? ld(dO + base + (size_t)i * D + c) : 0.f;
            dq[4 * ci + e] = 0.f;
        }
    const float lse = valid ? LSE[(size_t)bh * N + i] : 0.f;
    const float del = valid ? DEL[(size_t)bh * N + i] : 0.f;
    const int kend = causal ? min(N, i0 + ROWS) : N;
    for (int j0 = 0; j0 < kend; j0 += BT) {
        __syncthreads();
        stage<T, D>(ks, K + base, j0, N);
        stage<T, D>(vs, V + base, j0, N);
        __syncthreads();
        const int nk = min(BT, kend - j0);
        for (int jj = 0; jj < nk; ++jj) {
            const int j = j0 + jj;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 kv = *reinterpret_cast<const float4 *>(ks + jj * D + 4 * (ci * TPR + part));
                const float4 vv = *reinterpret_cast<const float4 *>(vs + jj * D + 4 * (ci * TPR + part));
                s = fmaf(qr[4 * ci + 0], kv.x, fmaf(qr[4 * ci + 1], kv.y, fmaf(qr[4 * ci + 2], kv.z, fmaf(qr[4 * ci + 3], kv.w, s))));
                dp = fmaf(gr[4 * ci + 0], vv.x, fmaf(gr[4 * ci + 1], vv.y, fmaf(gr[4 * ci + 2], vv.z, fmaf(gr[4 * ci + 3], vv.w, dp))));
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) {
                s += __shfl_xor_sync(0xffffffffu, s, off);
                dp += __shfl_xor_sync(0xffffffffu, dp, off);
            }
            const bool vis = valid && (!causal || j <= i);
            const float p = vis ? expf(scale * s - lse) : 0.f;
            const float gsc = scale * p * (dp - del);
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 kv = *reinterpret_cast<const float4 *>(ks + jj * D + 4 * (ci * TPR + part));
                dq[4 * ci + 0] = fmaf(gsc, kv.x, dq[4 * ci + 0]);
                dq[4 * ci + 1] = fmaf(gsc, kv.y, dq[4 * ci + 1]);
                dq[4 * ci + 2] = fmaf(gsc, kv.z, dq[4 * ci + 2]);
                dq[4 * ci + 3] = fmaf(gsc, kv.w, dq[4 * ci + 3]);
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                st(dQ + base + (size_t)i * D + 4 * (ci * TPR + part) + e, dq[4 * ci + e]);
    }
}

template <typename T, int D>
static attn_status launch_t(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, float *delta, void *dq, void *dk,
                            void *dv, int64_t BH, int64_t N, float scale, bool causal,
                            const LaunchCtx &ctx) {
    constexpr int TPR = D / 16;  // 16 dimensions per thread
    constexpr int ROWS = NT / TPR;
    const T *Q = static_cast<const T *>(q), *K = static_cast<const T *>(k);
    const T *V = static_cast<const T *>(v), *O = static_cast<const T *>(o);
    const T *G = static_cast<const T *>(dout);
    const int64_t rows = BH * N;
    bwd_delta_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, ctx.stream>>>(O, G, delta, rows);
    attn_status st = check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
    if (st != ATTN_OK) return st;
    dim3 grid((unsigned)((N + ROWS - 1) / ROWS), (unsigned)BH);
    bwd_dkdv_kernel<T, D, TPR><<<grid, NT, 0, ctx.stream>>>(
        Q, K, V, G, lse, delta, static_cast<T *>(dk), static_cast<T *>(dv), (int)N, scale,
        causal ? 1 : 0);
    if ((st = check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH)) != ATTN_OK) return st;
    bwd_dq_kernel<T, D, TPR><<<grid, NT, 0, ctx.stream>>>(Q, K, V, G, lse, delta,
                                                          static_cast<T *>(dq), (int)N, scale,
                                                          causal ? 1 : 0);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace bwd

attn_status launch_bwd_delta(const void *o, const void *dout, float *delta, int64_t rows, int d,
                             int dtype, const LaunchCtx &ctx) {
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (dtype == ATTN_F32) {
        const float *O = static_cast<const float *>(o), *G = static_cast<const float *>(dout);
        if (d == 64)
            bwd::bwd_delta_kernel<float, 64><<<grid, 256, 0, ctx.stream>>>(O, G, delta, rows);
        else
            bwd::bwd_delta_kernel<float, 128><<<grid, 256, 0, ctx.stream>>>(O, G, delta, rows);
    } else {
        const uint16_t *O = static_cast<const uint16_t *>(o);
        const uint16_t *G = static_cast<const uint16_t *>(dout);
        if (d == 64)
            bwd::bwd_delta_kernel<uint16_t, 64><<<grid, 256, 0, ctx.stream>>>(O, G, delta, rows);
        else
            bwd::bwd_delta_kernel<uint16_t, 128><<<grid, 256, 0, ctx.stream>>>(O, G, delta, rows);
    }
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

attn_status launch_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, float *delta, void *dq, void *dk,
                            void *dv, int64_t BH, int64_t N, int d, float scale, bool causal,
                            int dtype, const LaunchCtx &ctx) {
    if (dtype == ATTN_F32) {
        if (d == 64)
            return bwd::launch_t<float, 64>(q, k, v, o, dout, lse, delta, dq, dk, dv, BH, N, scale,
                                            causal, ctx);
        return bwd::launch_t<float, 128>(q, k, v, o, dout, lse, delta, dq, dk, dv, BH, N, scale,
                                         causal, ctx);
    }
    // bf16: D on CUDA cores, then the two tensor-core kernels (attn_bwd_tc.cu).
    const attn_status st = launch_bwd_delta(o, dout, delta, BH * N, d, dtype, ctx);
    if (st != ATTN_OK) return st;
    return launch_attn_bwd_bf16_tc(q, k, v, dout, lse, delta, dq, dk, dv, BH, N, d, scale, causal,
                                   ctx);
}

}  // namespace attn
