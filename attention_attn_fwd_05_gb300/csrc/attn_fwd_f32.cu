// attn_fwd_f32.cu -- exact-fp32 attention forward on CUDA cores (no TF32).
//
// Same computation as the bf16 tensor-core kernel (page "Hardware
// Acceleration & Custom Kernels", section 2: softmax(Q K^T * scale) V with
// the online normalisation applied per key tile), in plain fp32 FMA with
// accurate expf/logf, for fp32 inputs and outputs.
//
// A CTA owns BR = 32 query rows.  It has G groups of 128 threads (G = 1 or 2,
// chosen per launch); group g walks the key tiles g, g + G, g + 2G, ... of
// BC = 64 keys with its own online state, and the G partial states (m, l, O)
// are merged at the end with the same rescale rule.  Each group streams its K
// and V tiles through two shared-memory buffers with cp.async, so the copy of
// tile t+G overlaps the arithmetic on tile t.  A group's threads form an
// 8 x 16 grid (ty, tx):
//   S = Q K^T    thread (ty, tx) computes rows 4ty..4ty+3 x keys tx + 16jj
//                (jj = 0..3) from Q and K rows in shared memory (row-major,
//                rows padded by 16 bytes so the 16 key rows a half-warp reads
//                fall in distinct banks); per 4 dimensions: 8 16-byte loads,
//                64 FMAs; each logit is one sequential fp32 dot product over
//                c = 0..d-1;
//   softmax      row max and row sum combine the 16 threads of a row with
//                shuffles (the 16 threads of a row are one half-warp), so
//                every exponential is computed exactly once;
//   O += P V     P^T goes to shared memory; the same thread owns rows
//                4ty..4ty+3 x columns {4tx + 64k} of O, so the row rescale
//                factor is already in its registers.
#include <cmath>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace f32 {

constexpr int GROUP_THREADS = 128;
constexpr int BR = 32;  // query rows per CTA
constexpr int BC = 64;  // keys per tile

template <int D>
struct GroupSmem {
    float k[2][BC][D + 4];  // K rows, two buffers
    float v[2][BC][D];      // V rows, two buffers
    float pt[BC][BR + 4];   // P^T
};
template <int D, int G>
struct Smem {
    float q[BR][D + 4];  // Q rows, shared by the groups
    GroupSmem<D> grp[G];
};

// Running state of one thread: 4 rows x (4 * D/64) columns of O.
template <int D>
struct RowState {
    float m[4], l[4], o[4][D / 16];
};

// 16-byte global -> shared copy; rows past N are zero-filled (no bytes read).
__device__ __forceinline__ void cp_async16(float *dst, const float *src, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// The explicit minimum of one CTA per SM matters: without it ptxas capped the
// d = 64, one-group kernel at 80 registers and spilled 60 bytes inside the key
// loop (5 % slower on B=1 H=8 N=1024); with it every instantiation stays at
// 128-168 registers without spills.
template <int D, int G>
__global__ void __launch_bounds__(GROUP_THREADS * G, 1)
    attn_fwd_f32_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                        const float *__restrict__ V, float *__restrict__ O,
                        float *__restrict__ LSE, int N, float scale, int causal, int BH,
                        uint32_t *status) {
    constexpr int OC = D / 64;  // float4 column groups of O per thread
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem<D, G> &sm = *reinterpret_cast<Smem<D, G> *>(smem_raw);
    const int g = threadIdx.x / GROUP_THREADS;  // key-split group
    GroupSmem<D> &gs = sm.grp[g];
    const int tid = threadIdx.x % GROUP_THREADS;
    const int bh = blockIdx.y;
    const int row0 = blockIdx.x * BR;
    const int tx = tid & 15, ty = tid >> 4;
    const size_t base = (size_t)bh * (size_t)N * D;
    // Each group has its own named barrier (id 1 + g) for its tile loop: the
    // groups walk different numbers of key tiles.  Immediate ids keep the
    // CTA's barrier count at G + 1.
    auto group_sync = [&]() {
        if (g == 0)
            asm volatile("bar.sync 1, %0;" ::"n"(GROUP_THREADS) : "memory");
        else
            asm volatile("bar.sync 2, %0;" ::"n"(GROUP_THREADS) : "memory");
    };
    // Copy key tile k0 (K and V rows, zero past N) into buffer b.
    auto load_tile = [&](int k0, int b) {
        for (int idx = tid; idx < BC * (D / 4); idx += GROUP_THREADS) {
            const int kr = idx / (D / 4), c4 = idx % (D / 4);
            const bool ok = k0 + kr < N &&
                            ATTN_IN_BOUNDS(bh < BH && k0 + kr >= 0 && 4 * c4 + 4 <= D, status);
            const size_t off = ok ? base + (size_t)(k0 + kr) * D + 4 * c4 : 0;
            cp_async16(&gs.k[b][kr][4 * c4], K + off, ok);
            cp_async16(&gs.v[b][kr][4 * c4], V + off, ok);
        }
    };

    const int kv_end = causal ? min(N, row0 + BR) : N;
    // Group g takes key tiles g, g + G, g + 2G, ...: each group runs the
    // online recurrence over its own subset of keys, and the partial states
    // are merged at the end (the same max/rescale rule applied once more).
    int k0 = g * BC;
    if (k0 < kv_end) load_tile(k0, 0);
    cp_async_commit();

    // Q rows, zero past N (plain loads; they overlap the first tile's copy).
    for (int idx = threadIdx.x; idx < BR * (D / 4); idx += GROUP_THREADS * G) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < N && ATTN_IN_BOUNDS(bh < BH && 4 * c4 + 4 <= D, status))
            x = *reinterpret_cast<const float4 *>(Q + base + (size_t)(row0 + r) * D + 4 * c4);
        *reinterpret_cast<float4 *>(&sm.q[r][4 * c4]) = x;
    }
    __syncthreads();

    RowState<D> st;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        st.m[i] = -INFINITY;
        st.l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < OC * 4; ++c) st.o[i][c] = 0.f;
    }
    for (int t = 0; k0 < kv_end; ++t, k0 += G * BC) {
        const int b = t & 1;
        // Everyone is done with buffer b^1 (the previous tile): refill it with
        // the next tile while this one is used.
        group_sync();
        if (k0 + G * BC < kv_end) load_tile(k0 + G * BC, b ^ 1);
        cp_async_commit();
        cp_async_wait_1();  // this thread's copies of tile t have landed
        group_sync();       // ... and everyone else's

        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) s[i][jj] = 0.f;
        // Fully unrolled at d = 64 (+3-5 % measured); at d = 128 that ran 14-16 %
        // slower, so it keeps four dimensions' worth per iteration.
#pragma unroll(D == 64 ? 16 : 4)
        for (int c = 0; c < D; c += 4) {
            float4 qv[4], kv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const float4 *>(&sm.q[4 * ty + i][c]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                kv[jj] = *reinterpret_cast<const float4 *>(&gs.k[b][tx + 16 * jj][c]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float a = s[i][jj];
                    a = fmaf(qv[i].x, kv[jj].x, a);
                    a = fmaf(qv[i].y, kv[jj].y, a);
                    a = fmaf(qv[i].z, kv[jj].z, a);
                    s[i][jj] = fmaf(qv[i].w, kv[jj].w, a);
                }
        }

        float alpha[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = row0 + 4 * ty + i;
            const int limit = causal ? min(N, row + 1) : N;
            float mx = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int key = k0 + tx + 16 * jj;
                s[i][jj] = key < limit ? s[i][jj] * scale : -INFINITY;
                mx = fmaxf(mx, s[i][jj]);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            // A tile can be fully masked for a row (a group's later tiles with
            // the causal mask); the max then stays where it was.
            const float m_new = fmaxf(st.m[i], mx);
            const float m_ref = m_new == -INFINITY ? 0.f : m_new;
            alpha[i] = expf(st.m[i] - m_ref);
            float rs = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                s[i][jj] = expf(s[i][jj] - m_ref);
                rs += s[i][jj];
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
            st.l[i] = st.l[i] * alpha[i] + rs;
            st.m[i] = m_new;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<float4 *>(&gs.pt[tx + 16 * jj][4 * ty]) =
                make_float4(s[0][jj], s[1][jj], s[2][jj], s[3][jj]);
        group_sync();

#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < OC * 4; ++c) st.o[i][c] *= alpha[i];
        const int nk = min(BC, kv_end - k0);
#pragma unroll(D == 64 ? 8 : 4)
        for (int kk = 0; kk < nk; ++kk) {
            const float4 pv = *reinterpret_cast<const float4 *>(&gs.pt[kk][4 * ty]);
            const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int gg = 0; gg < OC; ++gg) {
                const float4 vv = *reinterpret_cast<const float4 *>(&gs.v[b][kk][64 * gg + 4 * tx]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    st.o[i][4 * gg + 0] = fmaf(pa[i], vv.x, st.o[i][4 * gg + 0]);
                    st.o[i][4 * gg + 1] = fmaf(pa[i], vv.y, st.o[i][4 * gg + 1]);
                    st.o[i][4 * gg + 2] = fmaf(pa[i], vv.z, st.o[i][4 * gg + 2]);
                    st.o[i][4 * gg + 3] = fmaf(pa[i], vv.w, st.o[i][4 * gg + 3]);
                }
            }
        }
    }

    if constexpr (G > 1) {
        // Merge: group 1 parks its state in its own K area (free once the
        // CTA-wide barrier below has passed), laid out [field][thread] so each
        // access is coalesced; group 0 folds it into its own with the same
        // rescale rule.
        constexpr int NF = 8 + 4 * (D / 16);
        static_assert(NF * GROUP_THREADS * sizeof(float) <= sizeof(float) * 2 * BC * (D + 4),
                      "merge area too small");
        __syncthreads();
        if (g == 1) {
            float *park = &gs.k[0][0][0];
            const float *f = reinterpret_cast<const float *>(&st);
#pragma unroll
            for (int i = 0; i < NF; ++i) park[i * GROUP_THREADS + tid] = f[i];
        }
        __syncthreads();
        if (g == 0) {
            const float *park = &sm.grp[1].k[0][0][0];
            RowState<D> o;
            float *f = reinterpret_cast<float *>(&o);
#pragma unroll
            for (int i = 0; i < NF; ++i) f[i] = park[i * GROUP_THREADS + tid];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m_new = fmaxf(st.m[i], o.m[i]);  // finite: group 0 saw key 0
                const float a = expf(st.m[i] - m_new), bb = expf(o.m[i] - m_new);
                st.l[i] = st.l[i] * a + o.l[i] * bb;
#pragma unroll
                for (int c = 0; c < OC * 4; ++c) st.o[i][c] = st.o[i][c] * a + o.o[i][c] * bb;
                st.m[i] = m_new;
            }
        }
    }

    if (g == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = row0 + 4 * ty + i;
            if (row >= N || !ATTN_IN_BOUNDS(bh < BH && row >= 0, status)) continue;
            const float inv_l = 1.f / st.l[i];
#pragma unroll
            for (int gg = 0; gg < OC; ++gg)
                *reinterpret_cast<float4 *>(O + base + (size_t)row * D + 64 * gg + 4 * tx) =
                    make_float4(st.o[i][4 * gg + 0] * inv_l, st.o[i][4 * gg + 1] * inv_l,
                                st.o[i][4 * gg + 2] * inv_l, st.o[i][4 * gg + 3] * inv_l);
            if (LSE != nullptr && tx == 0) LSE[(size_t)bh * N + row] = st.m[i] + logf(st.l[i]);
        }
    }
}

template <int D, int G>
static attn_status launch_g(const float *q, const float *k, const float *v, float *o, float *lse,
                            int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    const int smem = (int)sizeof(Smem<D, G>);
    if (check_launch(cudaFuncSetAttribute(attn_fwd_f32_kernel<D, G>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    dim3 grid((unsigned)((N + BR - 1) / BR), (unsigned)BH);
    attn_fwd_f32_kernel<D, G><<<grid, GROUP_THREADS * G, smem, ctx.stream>>>(
        q, k, v, o, lse, (int)N, scale, causal ? 1 : 0, (int)BH, ctx.status);
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

// Number of key-split groups per CTA.  A small grid leaves most of each SM
// idle while one 4-warp CTA walks its key tiles in series; two groups walk
// interleaved halves at once.  G is the one that minimises (waves of CTAs) /
// G, where the CTAs one SM holds follow from the shared memory each needs;
// ties go to the smaller G, and G never exceeds the number of key tiles.
template <int D>
static int pick_groups(int64_t BH, int64_t N, int sm_count) {
    const int64_t ctas = BH * ((N + BR - 1) / BR);
    const int64_t key_tiles = (N + BC - 1) / BC;
    constexpr int64_t kSmemPerSm = 228 * 1024;
    int best = 1;
    double best_cost = 1e30;
    for (int G = 1; G <= 2; ++G) {
        if (G > 1 && (G > key_tiles || sizeof(Smem<D, 2>) > 227 * 1024)) break;
        const int64_t bytes = (int64_t)(G == 1 ? sizeof(Smem<D, 1>) : sizeof(Smem<D, 2>)) + 1024;
        int64_t per_sm = kSmemPerSm / bytes;
        const int64_t by_threads = 2048 / (GROUP_THREADS * G);
        if (per_sm > by_threads) per_sm = by_threads;
        if (per_sm < 1) break;
        const int64_t slots = per_sm * (int64_t)sm_count;
        const double cost = (double)((ctas + slots - 1) / slots) / G;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = G;
        }
    }
    return best;
}

template <int D>
static attn_status launch(const float *q, const float *k, const float *v, float *o, float *lse,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    if constexpr (sizeof(Smem<D, 2>) <= 227 * 1024) {
        if (pick_groups<D>(BH, N, ctx.sm_count) == 2)
            return launch_g<D, 2>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    }
    return launch_g<D, 1>(q, k, v, o, lse, BH, N, scale, causal, ctx);
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
