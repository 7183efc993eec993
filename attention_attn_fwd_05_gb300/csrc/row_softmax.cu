// row_softmax.cu -- row softmax with a running maximum and sum.
//
// y[r, :] = exp(x[r, :] - max) / sum(exp(x[r, :] - max)), lse[r] = max + ln sum
// (page "14. Triton and kernel fusion", section "Fusion": subtract the row
// max, exponentiate, divide by the sum, reading the row once; and its
// exercise on rows longer than one block, done here with the online
// normalisation identity of page "Hardware Acceleration & Custom Kernels",
// section 2: m_new = max(m_old, x), d_new = d_old e^(m_old - m_new) + e^(x - m_new)).
//
// Two kernels, one CTA per row (grid-stride over rows), each thread keeping a
// running (m, d) pair that the CTA merges with the same identity:
//
// row_softmax_stream_kernel -- rows of up to kStreamMaxWidth floats with
//   16-byte aligned rows.  Each CTA streams its rows into two shared-memory
//   buffers with bulk async copies (one instruction per row), so the copy of
//   the next row runs while one is worked on.  Two buffers, not more: more
//   shared memory per CTA costs more in CTAs per SM than deeper prefetch
//   gains (measured 15-20 % slower at widths 1024-2048 with 8 buffers).  A thread holds its elements in registers:
//   pass 1 takes its maximum m_t and e = exp(x - m_t), the CTA merges the
//   (m_t, sum e) pairs into (M, D), and pass 2 writes y = e * exp(m_t - M) / D,
//   one exponential per element in all.
// row_softmax_cluster_kernel -- aligned rows longer than kStreamMaxWidth
//   when there are too few of them to fill the GPU one CTA per row: a
//   thread-block cluster of CTAs per row, merged through distributed shared
//   memory (see there).
// row_softmax_kernel -- any other row: pass 1 walks the row updating (m, d)
//   per 4-element group; pass 2 writes the output, reading the row from shared
//   memory when it was cached there in pass 1 (rows up to kCacheFloats),
//   otherwise from global memory again (L2-resident for moderate rows).
//
// Any width is accepted; there is no 65536 cap.  -inf entries (masked
// positions) get probability 0, and a row of -inf only gets all zeros and
// LSE = -inf; y may alias x.
#include <cmath>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

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
            // Four float4 groups per step, loaded before any is used, so each
            // thread keeps four loads in flight; the running pair is rescaled
            // once per step.
            constexpr int U = 4;
            for (int64_t i0 = threadIdx.x; i0 < n4; i0 += U * NUM_THREADS) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = i0 + (int64_t)u * NUM_THREADS;
                    v[u] = i < n4 ? reinterpret_cast<const float4 *>(xr)[i]
                                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
                float gm = -INFINITY;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = i0 + (int64_t)u * NUM_THREADS;
                    if (cached && i < n4) reinterpret_cast<float4 *>(cache)[i] = v[u];
                    gm = fmaxf(gm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
                }
                const float M = fmaxf(md.m, gm);
                if (M == -INFINITY) continue;  // only masked (-inf) entries so far
                float add = 0.f;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    add += (expf(v[u].x - M) + expf(v[u].y - M)) +
                           (expf(v[u].z - M) + expf(v[u].w - M));
                md.d = md.d * expf(md.m - M) + add;
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
        // A row of -inf only has M = -inf and d = 0: every probability is 0.
        const bool dead = row_md.m == -INFINITY;
        const float M = dead ? 0.f : row_md.m, inv_d = dead ? 0.f : 1.f / row_md.d;
        if (vec4) {
            const int64_t n4 = width / 4;
            constexpr int U = 4;
            for (int64_t i0 = threadIdx.x; i0 < n4; i0 += U * NUM_THREADS) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = i0 + (int64_t)u * NUM_THREADS;
                    if (i < n4)
                        v[u] = cached ? reinterpret_cast<const float4 *>(cache)[i]
                                      : reinterpret_cast<const float4 *>(xr)[i];
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = i0 + (int64_t)u * NUM_THREADS;
                    if (i < n4)
                        reinterpret_cast<float4 *>(yr)[i] =
                            make_float4(expf(v[u].x - M) * inv_d, expf(v[u].y - M) * inv_d,
                                        expf(v[u].z - M) * inv_d, expf(v[u].w - M) * inv_d);
                }
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

// ------------------------------------------------------------------ streamed ---

// (max, sum) of the pairs (m, d) held by the 32 lanes of a warp: M = max m,
// D = sum d e^(m - M); lanes with m = -inf hold d = 0 and add nothing.
// Every lane gets the result.
__device__ __forceinline__ MD merge_group(float m, float d) {
    float M = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float D = m == -INFINITY ? 0.f : d * expf(m - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) D += __shfl_xor_sync(0xffffffffu, D, off);
    return {M, D};
}

// Streamed rows: NT threads per CTA, at most KMAX float4 groups per thread
// (width <= 4 * NT * KMAX), NS row buffers in shared memory.
constexpr int NS = 2;
constexpr uint32_t ST_HDR = 256;  // NS barriers, abort flag, reduction scratch
constexpr int64_t kStreamMaxWidth = 12288;

__device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    return true;
}

template <int NT, int KMAX>
__global__ void __launch_bounds__(NT)
    row_softmax_stream_kernel(const float *x, float *y, float *__restrict__ lse, int64_t rows,
                              int width, uint32_t *status, uint64_t timeout_ns) {
    static_assert(NT % 32 == 0 && NT / 32 <= 16, "reduction scratch holds 16 warps");
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);  // barrier of buffer b at sbase + 8b
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + 64);
    MD *warp_md = reinterpret_cast<MD *>(sm + 96);  // [NT / 32]
    MD *row_md = reinterpret_cast<MD *>(sm + 96 + 16 * sizeof(MD));
    const uint32_t row_bytes = (uint32_t)width * 4u;
    const uint32_t buf_stride = (row_bytes + 127u) & ~127u;
    const int n4 = width / 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const WaitCtl ctl{abort_flag, status, timeout_ns};
    const int64_t G = gridDim.x;
    // Row i of this CTA (row blockIdx.x + i*G) goes to buffer i % NS as that
    // buffer's (i / NS)-th copy.  n_issued: rows whose copy thread 0 started.
    int n_issued = 0;
    auto issue = [&]() {
        const int64_t row = (int64_t)blockIdx.x + (int64_t)n_issued * G;
        if (row >= rows) return;
        const uint32_t b = (uint32_t)(n_issued % NS);
        mbar_arrive_expect_tx(sbase + 8u * b, row_bytes);
        bulk_copy_g2s(sbase + ST_HDR + b * buf_stride, x + row * (int64_t)width, row_bytes,
                      sbase + 8u * b);
        ++n_issued;
    };
    if (threadIdx.x == 0) {
        for (int b = 0; b < NS; ++b) mbar_init(sbase + 8u * (uint32_t)b, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        for (int b = 0; b < NS; ++b) issue();
    }
    __syncthreads();

    int i = 0;
    for (int64_t r = blockIdx.x; r < rows; ++i, r += G) {
        const uint32_t b = (uint32_t)(i % NS);
        // Row i landed in buffer b; the answer is the same in every thread.
        if (!__syncthreads_and(
                bounded_wait_warp(sbase + 8u * b, (uint32_t)(i / NS) & 1u, ctl) ? 1 : 0))
            break;
        const float4 *buf = reinterpret_cast<const float4 *>(sm + ST_HDR + b * buf_stride);
        // Pass 1: this thread's groups, their maximum, e = exp(x - m_t).
        float4 e[KMAX];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int idx = threadIdx.x + k * NT;
            if (idx < n4) {
                e[k] = buf[idx];
                m = fmaxf(m, fmaxf(fmaxf(e[k].x, e[k].y), fmaxf(e[k].z, e[k].w)));
            }
        }
        float d = 0.f;
        const float mt = m == -INFINITY ? 0.f : m;  // all -inf: every e is 0
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int idx = threadIdx.x + k * NT;
            if (idx < n4) {
                e[k].x = expf(e[k].x - mt);
                e[k].y = expf(e[k].y - mt);
                e[k].z = expf(e[k].z - mt);
                e[k].w = expf(e[k].w - mt);
                d += (e[k].x + e[k].y) + (e[k].z + e[k].w);
            }
        }
        // Merge the (m_t, d_t) pairs: the maximum first, then every sum
        // rescaled to it once, then the sums (the same identity, one
        // exponential per thread and level instead of one per shuffle).
        const MD wmd = merge_group(m, d);
        if (lane == 0) warp_md[warp] = wmd;
        __syncthreads();
        if (warp == 0) {
            const MD w = lane < NT / 32 ? warp_md[lane] : MD{-INFINITY, 0.f};
            const MD tot = merge_group(w.m, w.d);
            if (lane == 0) {
                *row_md = tot;
                if (lse != nullptr) lse[r] = tot.m + logf(tot.d);
            }
        }
        __syncthreads();  // row_md is ready and every thread is done with buffer b
        if (threadIdx.x == 0) issue();  // row i + NS into buffer b
        // Pass 2: y = e * exp(m_t - M) / D.
        const MD tot = *row_md;
        const float c = m == -INFINITY ? 0.f : expf(m - tot.m) / tot.d;
        float4 *yr = reinterpret_cast<float4 *>(y + r * (int64_t)width);
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int idx = threadIdx.x + k * NT;
            if (idx < n4)
                yr[idx] = make_float4(e[k].x * c, e[k].y * c, e[k].z * c, e[k].w * c);
        }
    }
    // After a timeout, let copies still in flight land before the CTA exits
    // (on the normal path every issued copy has been waited for).
    if (threadIdx.x == 0 && *abort_flag != 0u)
        for (int c = i; c < n_issued; ++c)
            drain(sbase + 8u * (uint32_t)(c % NS), (uint32_t)(c / NS) & 1u, timeout_ns);
}

template <int NT, int KMAX>
attn_status launch_stream(const float *x, float *y, float *lse, int64_t rows, int64_t width,
                          const LaunchCtx &ctx) {
    const uint32_t buf = ((uint32_t)width * 4u + 127u) & ~127u;
    const int smem = (int)(ST_HDR + (uint32_t)NS * buf);
    auto kern = row_softmax_stream_kernel<NT, KMAX>;
    if (check_launch(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    int per_sm = 0;
    if (check_launch(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    const int64_t max_grid = (int64_t)ctx.sm_count * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(rows < max_grid ? rows : max_grid);
    kern<<<grid, NT, smem, ctx.stream>>>(x, y, lse, rows, (int)width, ctx.status,
                                         ctx.timeout_ns);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

// ------------------------------------------------------------- clusters ---
// Aligned rows longer than kStreamMaxWidth when there are too few of them for
// one CTA per row to fill the GPU: a cluster of CL CTAs (2..8) per row, CTA
// `rank` taking the slice [rank, rank + 1) * width / CL.  Each CTA reduces its
// slice to one (m, d) pair, stores it into slot `rank` of every cluster CTA's
// shared memory and arrives on their barriers; once a CTA's barrier has all CL
// arrivals it merges the pairs (in rank order, the same in every CTA) and
// writes y for its slice.  Rows alternate between two barriers and two sets of
// slots, so a CTA one row ahead never overwrites slots still being read.  Every
// wait is bounded, and a cluster barrier before exit keeps each CTA's shared
// memory alive until no other CTA of the cluster can still store into it.

constexpr int CL_THREADS = 512;
constexpr int CL_MAX = 8;

struct ClusterSmem {
    uint64_t xbar[2];            // per row parity: CL arrivals, one per cluster CTA
    MD pairs[2][CL_MAX];         // per row parity: (m, d) of every cluster CTA
    MD warp_md[CL_THREADS / 32];
    MD cta_md;
    uint32_t abort;
};

__global__ void __launch_bounds__(CL_THREADS)
    row_softmax_cluster_kernel(const float *x, float *y, float *__restrict__ lse, int64_t rows,
                               int width, int CL, uint32_t *status, uint64_t timeout_ns) {
    __shared__ ClusterSmem sm;
    const uint32_t rank = cluster_ctarank();
    const int64_t cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&sm.xbar[0]), (uint32_t)CL);
        mbar_init(smem_u32(&sm.xbar[1]), (uint32_t)CL);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Every CTA's barriers are initialised before any CTA arrives on them.
    cluster_sync_all();
    const int64_t n4 = width / 4;
    const int64_t c0 = n4 * rank / CL, c1 = n4 * (rank + 1) / CL;
    constexpr int U = 4;
    int it = 0;
    for (int64_t r = cid; r < rows; r += ncl, ++it) {
        const int par = it & 1;
        const float4 *xr = reinterpret_cast<const float4 *>(x + r * (int64_t)width);
        // Pass 1 over this CTA's slice: a running (m, d), four groups per step.
        MD md{-INFINITY, 0.f};
        for (int64_t i0 = c0 + threadIdx.x; i0 < c1; i0 += U * CL_THREADS) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * CL_THREADS;
                v[u] = i < c1 ? xr[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            float gm = -INFINITY;
#pragma unroll
            for (int u = 0; u < U; ++u)
                gm = fmaxf(gm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
            const float M = fmaxf(md.m, gm);
            if (M == -INFINITY) continue;
            float add = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u)
                add += (expf(v[u].x - M) + expf(v[u].y - M)) + (expf(v[u].z - M) + expf(v[u].w - M));
            md.d = md.d * expf(md.m - M) + add;
            md.m = M;
        }
        const MD wmd = merge_group(md.m, md.d);
        if (lane == 0) sm.warp_md[warp] = wmd;
        __syncthreads();
        if (warp == 0) {
            const MD w = lane < CL_THREADS / 32 ? sm.warp_md[lane] : MD{-INFINITY, 0.f};
            const MD tot = merge_group(w.m, w.d);
            if (lane == 0) {
                // This CTA's pair into slot `rank` of every cluster CTA, then
                // one arrival on each of their barriers for this row.
                const uint32_t slot = smem_u32(&sm.pairs[par][rank]);
                const uint32_t xb = smem_u32(&sm.xbar[par]);
                for (int dst = 0; dst < CL; ++dst) {
                    st_cluster_f32x2(map_shared_to_rank(slot, (uint32_t)dst), tot.m, tot.d);
                    arrive_remote(map_shared_to_rank(xb, (uint32_t)dst));
                }
            }
        }
        bool ok = true;
        if (lane == 0)
            ok = wait_cluster_bounded(smem_u32(&sm.xbar[par]), (uint32_t)(it >> 1) & 1u, status,
                                      timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!__syncthreads_and(ok ? 1 : 0)) break;
        // Every slice's pair, merged in rank order.
        float M = -INFINITY;
        for (int c = 0; c < CL; ++c) M = fmaxf(M, sm.pairs[par][c].m);
        float D = 0.f;
        if (M != -INFINITY)
            for (int c = 0; c < CL; ++c)
                if (sm.pairs[par][c].m != -INFINITY)
                    D += sm.pairs[par][c].d * expf(sm.pairs[par][c].m - M);
        if (rank == 0 && threadIdx.x == 0 && lse != nullptr) lse[r] = M + logf(D);
        // A row of -inf only has M = -inf and D = 0: every probability is 0.
        const bool dead = M == -INFINITY;
        const float Ms = dead ? 0.f : M, inv_d = dead ? 0.f : 1.f / D;
        float4 *yr = reinterpret_cast<float4 *>(y + r * (int64_t)width);
        for (int64_t i0 = c0 + threadIdx.x; i0 < c1; i0 += U * CL_THREADS) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * CL_THREADS;
                if (i < c1) v[u] = xr[i];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * CL_THREADS;
                if (i < c1)
                    yr[i] = make_float4(expf(v[u].x - Ms) * inv_d, expf(v[u].y - Ms) * inv_d,
                                        expf(v[u].z - Ms) * inv_d, expf(v[u].w - Ms) * inv_d);
            }
        }
        __syncthreads();  // warp_md is reused by the next row
    }
    // No CTA leaves while another CTA of the cluster may still store into its
    // shared memory.
    cluster_sync_all();
}

}  // namespace rsm

attn_status launch_row_softmax(const float *x, float *y, float *lse, int64_t rows, int64_t width,
                               const LaunchCtx &ctx) {
    const bool vec4 = (width % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    // Aligned rows up to 12288 floats stream through shared memory, with the
    // CTA size picked so each thread holds at most 4-6 float4 groups.
    if (vec4 && width <= 2048) return rsm::launch_stream<128, 4>(x, y, lse, rows, width, ctx);
    if (vec4 && width <= 4096) return rsm::launch_stream<256, 4>(x, y, lse, rows, width, ctx);
    if (vec4 && width <= rsm::kStreamMaxWidth)
        return rsm::launch_stream<512, 6>(x, y, lse, rows, width, ctx);
    // Longer aligned rows, too few of them for one CTA per row to fill the
    // GPU (two per SM): a cluster of CL CTAs per row, every slice at least
    // 8192 floats.
    const int64_t slots = 2 * (int64_t)ctx.sm_count;
    if (vec4 && rows < slots && width <= INT32_MAX) {
        int64_t cl = (slots + rows - 1) / rows;
        if (cl > rsm::CL_MAX) cl = rsm::CL_MAX;
        while (cl > 1 && width / cl < 8192) --cl;
        if (cl > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(rows * cl));
            cfg.blockDim = dim3(rsm::CL_THREADS);
            cfg.stream = ctx.stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)cl;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return check_launch(cudaLaunchKernelEx(&cfg, rsm::row_softmax_cluster_kernel, x, y,
                                                   lse, rows, (int)width, (int)cl, ctx.status,
                                                   ctx.timeout_ns),
                                ATTN_ERR_LAUNCH);
        }
    }
    const int64_t max_grid = (int64_t)ctx.sm_count * 4;
    const unsigned grid = (unsigned)(rows < max_grid ? rows : max_grid);
    rsm::row_softmax_kernel<<<grid, rsm::NUM_THREADS, 0, ctx.stream>>>(x, y, lse, rows, width,
                                                                       vec4 ? 1 : 0);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace attn
