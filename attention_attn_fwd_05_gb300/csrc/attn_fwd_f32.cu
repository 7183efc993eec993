// attn_fwd_f32.cu -- exact-fp32 attention forward on CUDA cores (no TF32).
//
// Same computation as the bf16 tensor-core kernel (page "Hardware
// Acceleration & Custom Kernels", section 2: softmax(Q K^T * scale) V with
// the online normalisation applied per key tile), in plain fp32 FMA with
// accurate expf/logf, for fp32 inputs and outputs.
//
// A CTA of 128 threads owns BR = 32 query rows and walks key tiles of BC = 64
// keys.  The threads form an 8 x 16 grid (ty, tx):
//   S = Q K^T    thread (ty, tx) computes rows 4ty..4ty+3 x keys 4tx..4tx+3
//                from Q^T and K^T staged in shared memory (per dimension c:
//                two 16-byte loads, 16 FMAs; each logit is one sequential
//                fp32 dot product over c = 0..d-1);
//   softmax      row max and row sum combine the 16 threads of a row with
//                shuffles (the 16 threads of a row are one half-warp), so
//                every exponential is computed exactly once;
//   O += P V     P^T goes to shared memory; the same thread owns rows
//                4ty..4ty+3 x columns {4tx + 64k} of O, so the row rescale
//                factor is already in its registers.
#include <cmath>

#include "attn_internal.h"

namespace attn {
namespace f32 {

constexpr int NUM_THREADS = 128;
constexpr int BR = 32;  // query rows per CTA
constexpr int BC = 64;  // keys per tile

template <int D>
struct Smem {
    float qt[D][BR];   // Q^T
    float kt[D][BC];   // K^T
    float v[BC][D];    // V
    float pt[BC][BR];  // P^T
};

template <int D>
__global__ void __launch_bounds__(NUM_THREADS)
    attn_fwd_f32_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                        const float *__restrict__ V, float *__restrict__ O,
                        float *__restrict__ LSE, int N, float scale, int causal) {
    constexpr int OC = D / 64;  // float4 column groups of O per thread
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);
    const int bh = blockIdx.y;
    const int row0 = blockIdx.x * BR;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const size_t base = (size_t)bh * (size_t)N * D;

    // Q^T, zero rows past N.
    for (int idx = threadIdx.x; idx < BR * (D / 4); idx += NUM_THREADS) {
        const int r = idx % BR, c4 = idx / BR;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < N) x = *reinterpret_cast<const float4 *>(Q + base + (size_t)(row0 + r) * D + 4 * c4);
        sm.qt[4 * c4 + 0][r] = x.x;
        sm.qt[4 * c4 + 1][r] = x.y;
        sm.qt[4 * c4 + 2][r] = x.z;
        sm.qt[4 * c4 + 3][r] = x.w;
    }

    float m[4], l[4], o[4][OC * 4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < OC * 4; ++c) o[i][c] = 0.f;
    }
    const int kv_end = causal ? min(N, row0 + BR) : N;
    for (int k0 = 0; k0 < kv_end; k0 += BC) {
        __syncthreads();  // previous tile's readers are done
        for (int idx = threadIdx.x; idx < BC * (D / 4); idx += NUM_THREADS) {
            const int kr = idx % BC, c4 = idx / BC;
            float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
            if (k0 + kr < N) {
                const size_t off = base + (size_t)(k0 + kr) * D + 4 * c4;
                kx = *reinterpret_cast<const float4 *>(K + off);
                vx = *reinterpret_cast<const float4 *>(V + off);
            }
            sm.kt[4 * c4 + 0][kr] = kx.x;
            sm.kt[4 * c4 + 1][kr] = kx.y;
            sm.kt[4 * c4 + 2][kr] = kx.z;
            sm.kt[4 * c4 + 3][kr] = kx.w;
            *reinterpret_cast<float4 *>(&sm.v[kr][4 * c4]) = vx;
        }
        __syncthreads();

        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) s[i][jj] = 0.f;
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
            const float4 qv = *reinterpret_cast<const float4 *>(&sm.qt[c][4 * ty]);
            const float4 kv = *reinterpret_cast<const float4 *>(&sm.kt[c][4 * tx]);
            const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
            const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) s[i][jj] = fmaf(qa[i], ka[jj], s[i][jj]);
        }

        float alpha[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = row0 + 4 * ty + i;
            const int limit = causal ? min(N, row + 1) : N;
            float mx = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int key = k0 + 4 * tx + jj;
                s[i][jj] = key < limit ? s[i][jj] * scale : -INFINITY;
                mx = fmaxf(mx, s[i][jj]);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);  // finite: key 0 is visible to every row
            alpha[i] = expf(m[i] - m_new);
            float rs = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                s[i][jj] = expf(s[i][jj] - m_new);
                rs += s[i][jj];
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
            l[i] = l[i] * alpha[i] + rs;
            m[i] = m_new;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<float4 *>(&sm.pt[4 * tx + jj][4 * ty]) =
                make_float4(s[0][jj], s[1][jj], s[2][jj], s[3][jj]);
        __syncthreads();

#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < OC * 4; ++c) o[i][c] *= alpha[i];
        const int nk = min(BC, kv_end - k0);
        for (int kk = 0; kk < nk; ++kk) {
            const float4 pv = *reinterpret_cast<const float4 *>(&sm.pt[kk][4 * ty]);
            const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int g = 0; g < OC; ++g) {
                const float4 vv = *reinterpret_cast<const float4 *>(&sm.v[kk][64 * g + 4 * tx]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[i][4 * g + 0] = fmaf(pa[i], vv.x, o[i][4 * g + 0]);
                    o[i][4 * g + 1] = fmaf(pa[i], vv.y, o[i][4 * g + 1]);
                    o[i][4 * g + 2] = fmaf(pa[i], vv.z, o[i][4 * g + 2]);
                    o[i][4 * g + 3] = fmaf(pa[i], vv.w, o[i][4 * g + 3]);
                }
            }
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = row0 + 4 * ty + i;
        if (row >= N) continue;
        const float inv_l = 1.f / l[i];
#pragma unroll
        for (int g = 0; g < OC; ++g)
            *reinterpret_cast<float4 *>(O + base + (size_t)row * D + 64 * g + 4 * tx) =
                make_float4(o[i][4 * g + 0] * inv_l, o[i][4 * g + 1] * inv_l,
                            o[i][4 * g + 2] * inv_l, o[i][4 * g + 3] * inv_l);
        if (LSE != nullptr && tx == 0) LSE[(size_t)bh * N + row] = m[i] + logf(l[i]);
    }
}

template <int D>
static attn_status launch(const float *q, const float *k, const float *v, float *o, float *lse,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    const int smem = (int)sizeof(Smem<D>);
    if (check_launch(cudaFuncSetAttribute(attn_fwd_f32_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    dim3 grid((unsigned)((N + BR - 1) / BR), (unsigned)BH);
    attn_fwd_f32_kernel<D><<<grid, NUM_THREADS, smem, ctx.stream>>>(q, k, v, o, lse, (int)N,
                                                                     scale, causal ? 1 : 0);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace f32

attn_status launch_attn_fwd_f32(const float *q, const float *k, const float *v, float *o,
                                float *lse, int64_t BH, int64_t N, int d, float scale,
                                bool causal, const LaunchCtx &ctx) {
    if (d == 64) return f32::launch<64>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    if (d == 128) return f32::launch<128>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    return ATTN_ERR_HEADDIM;
}

}  // namespace attn
