// attn_fwd_f32.cu -- exact-fp32 attention forward on CUDA cores (no TF32).
//
// Same computation as the bf16 tensor-core kernel (page "Hardware
// Acceleration & Custom Kernels", section 2: softmax(Q K^T * scale) V with
// the online normalisation applied per key tile), in plain fp32 FMA with
// accurate expf/logf, for fp32 inputs and outputs.
//
// Layout of the work: TPR threads share one query row, each owning D/TPR of
// its head dimensions (in 16-byte chunks interleaved across the TPR threads so
// that shared-memory reads of a key row are conflict-free broadcasts).  A CTA
// of 128 threads covers 128/TPR rows; K and V tiles of BC keys are staged in
// shared memory with a two-buffer cp.async pipeline.  Per key tile each thread
// forms partial dot products for its dimensions, the TPR partials are summed
// with shuffles, then the running maximum / sum / output update follows the
// online recurrence.
#include <cmath>

#include "attn_internal.h"

namespace attn {
namespace f32 {

constexpr int NUM_THREADS = 128;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;  // zero-fill rows past N
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_1() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_0() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Keys per shared-memory tile: 32 KB of K and V double buffers either way.
template <int D>
constexpr int kBC = (D == 128) ? 16 : 32;

template <int D, int TPR>
__global__ void __launch_bounds__(NUM_THREADS)
    attn_fwd_f32_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                        const float *__restrict__ V, float *__restrict__ O,
                        float *__restrict__ LSE, int N, float scale, int causal) {
    constexpr int BC = kBC<D>;
    constexpr int ROWS = NUM_THREADS / TPR;  // query rows per CTA
    constexpr int NCH = D / 4 / TPR;         // float4 chunks per thread
    constexpr int TILE_F4 = BC * D / 4;      // float4s per K (or V) tile
    __shared__ __align__(16) float Ks[2][BC * D];
    __shared__ __align__(16) float Vs[2][BC * D];

    const int bh = blockIdx.y;
    const int row0 = blockIdx.x * ROWS;
    const int lr = threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    const int row = row0 + lr;
    const bool valid = row < N;
    const size_t base = (size_t)bh * (size_t)N * D;
    const float *Kh = K + base;
    const float *Vh = V + base;

    // Chunk ci of this thread covers dims [4*(ci*TPR + part), +4).
    float q[NCH * 4], o[NCH * 4];
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid)
            x = *reinterpret_cast<const float4 *>(Q + base + (size_t)row * D +
                                                  4 * (ci * TPR + part));
        q[4 * ci + 0] = x.x;
        q[4 * ci + 1] = x.y;
        q[4 * ci + 2] = x.z;
        q[4 * ci + 3] = x.w;
        o[4 * ci + 0] = o[4 * ci + 1] = o[4 * ci + 2] = o[4 * ci + 3] = 0.f;
    }

    // Keys this CTA needs: all N, or up to its last row with the causal mask.
    const int kv_end = causal ? min(N, row0 + ROWS) : N;
    const int ntiles = (kv_end + BC - 1) / BC;
    const int limit = causal ? min(N, row + 1) : N;  // keys [0, limit) visible to this row

    auto load_tile = [&](int tile, int buf) {
        const int k0 = tile * BC;
        for (int i = threadIdx.x; i < TILE_F4; i += NUM_THREADS) {
            const int kr = i / (D / 4), c4 = i % (D / 4);
            const bool ok = k0 + kr < N;
            const size_t off = (size_t)(ok ? k0 + kr : 0) * D + 4 * c4;
            cp_async16(&Ks[buf][kr * D + 4 * c4], Kh + off, ok);
            cp_async16(&Vs[buf][kr * D + 4 * c4], Vh + off, ok);
        }
        cp_async_commit();
    };

    float m = -INFINITY, l = 0.f;
    if (ntiles > 0) load_tile(0, 0);
    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < ntiles) {
            load_tile(tile + 1, buf ^ 1);
            cp_async_wait_1();
        } else {
            cp_async_wait_0();
        }
        __syncthreads();

        const float *Kt = Ks[buf];
        const float *Vt = Vs[buf];
        float s[BC];
#pragma unroll
        for (int j = 0; j < BC; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 kv =
                    *reinterpret_cast<const float4 *>(Kt + j * D + 4 * (ci * TPR + part));
                acc = fmaf(q[4 * ci + 0], kv.x, acc);
                acc = fmaf(q[4 * ci + 1], kv.y, acc);
                acc = fmaf(q[4 * ci + 2], kv.z, acc);
                acc = fmaf(q[4 * ci + 3], kv.w, acc);
            }
            s[j] = acc;
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int j = 0; j < BC; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j], off);
        }
        const int k0 = tile * BC;
        float mx = m;
#pragma unroll
        for (int j = 0; j < BC; ++j) {
            s[j] = (k0 + j < limit) ? s[j] * scale : -INFINITY;
            mx = fmaxf(mx, s[j]);
        }
        // Every row sees key 0 in the first tile, so mx is finite from here on.
        const float alpha = expf(m - mx);
        l *= alpha;
#pragma unroll
        for (int i = 0; i < NCH * 4; ++i) o[i] *= alpha;
#pragma unroll
        for (int j = 0; j < BC; ++j) {
            const float p = expf(s[j] - mx);
            l += p;
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
                const float4 vv =
                    *reinterpret_cast<const float4 *>(Vt + j * D + 4 * (ci * TPR + part));
                o[4 * ci + 0] = fmaf(p, vv.x, o[4 * ci + 0]);
                o[4 * ci + 1] = fmaf(p, vv.y, o[4 * ci + 1]);
                o[4 * ci + 2] = fmaf(p, vv.z, o[4 * ci + 2]);
                o[4 * ci + 3] = fmaf(p, vv.w, o[4 * ci + 3]);
            }
        }
        m = mx;
        __syncthreads();  // this buffer is refilled two tiles later
    }

    if (valid) {
        const float inv_l = 1.f / l;
#pragma unroll
        for (int ci = 0; ci < NCH; ++ci) {
            float4 y;
            y.x = o[4 * ci + 0] * inv_l;
            y.y = o[4 * ci + 1] * inv_l;
            y.z = o[4 * ci + 2] * inv_l;
            y.w = o[4 * ci + 3] * inv_l;
            *reinterpret_cast<float4 *>(O + base + (size_t)row * D + 4 * (ci * TPR + part)) = y;
        }
        if (LSE != nullptr && part == 0) LSE[(size_t)bh * N + row] = m + logf(l);
    }
}

template <int D, int TPR>
static attn_status launch(const float *q, const float *k, const float *v, float *o, float *lse,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    constexpr int ROWS = NUM_THREADS / TPR;
    dim3 grid((unsigned)((N + ROWS - 1) / ROWS), (unsigned)BH);
    attn_fwd_f32_kernel<D, TPR><<<grid, NUM_THREADS, 0, ctx.stream>>>(q, k, v, o, lse, (int)N,
                                                                       scale, causal ? 1 : 0);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace f32

attn_status launch_attn_fwd_f32(const float *q, const float *k, const float *v, float *o,
                                float *lse, int64_t BH, int64_t N, int d, float scale,
                                bool causal, const LaunchCtx &ctx) {
    if (d == 64) return f32::launch<64, 4>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    if (d == 128) return f32::launch<128, 4>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    return ATTN_ERR_HEADDIM;
}

}  // namespace attn
