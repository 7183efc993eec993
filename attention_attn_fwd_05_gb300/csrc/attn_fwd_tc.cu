// attn_fwd_tc.cu -- bf16 exact attention forward on sm_103a tensor cores.
//
// Computes O = softmax(scale * Q K^T) V and LSE per row (page "Hardware
// Acceleration & Custom Kernels", section 2: the attention formula, SRAM
// tiling into B_r x d and B_c x d blocks, and the online normalisation
// m_new = max(m_old, x), d_new = d_old e^(m_old - m_new) + e^(x - m_new)
// applied per key tile, rescaling the running output sums as tiles arrive).
//
// One CTA owns one 128-row query tile of one (batch, head) and walks the key
// tiles j = 0 .. T-1 (up to the diagonal with the causal mask).  Roles:
//
//   warp 4      TMA producer: Q once, then K_j and V_j into an NSTAGE-deep
//               shared-memory ring (128-byte swizzle, 64-column boxes).
//   warp 5      TMEM allocator and MMA issuer (one thread):
//                 S_j  = Q K_j^T  -> TMEM buffer j%2 (128 lanes x 128 fp32 cols)
//                 O   += P_j V_j  -> TMEM (128 lanes x d fp32 cols)
//               S_{j+1} is issued before waiting for P_j, so the tensor core
//               computes the next logits while the softmax warps work.
//   warps 0-3   softmax and epilogue, one query row per thread (TMEM lane =
//               row): read S_j, scale to log2 units, mask, running max m and
//               sum l, P_j = 2^(s - m) as bf16 into shared memory, rescale the
//               O row in TMEM by 2^(m_old - m_new) when the max moved; at the
//               end O / l -> bf16 -> shared -> TMA store, LSE = (m + log2 l) ln 2.
//
// The N x N logits live only in TMEM and registers; device memory sees Q, K,
// V read and O, LSE written.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace tc {

constexpr int BM = 128;           // query rows per tile (one per TMEM lane)
constexpr int BN = 128;           // keys per tile
constexpr int NUM_THREADS = 192;  // 4 softmax warps + producer warp + MMA warp
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S0 = 0, TMEM_S1 = 128, TMEM_O = 256;
constexpr float LN2 = 0.69314718055994530942f;

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
    static constexpr int NSTAGE = (D == 128) ? 2 : 4;
    static constexpr int DBLK = D / 64;  // 128-byte column blocks per row
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    static constexpr uint32_t P_BYTES = BM * BN * 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NSTAGE * KV_BYTES;
    static constexpr uint32_t OFF_P = OFF_V + NSTAGE * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + base alignment slack
    // Barrier slots (8 bytes each) inside the BAR area.
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + NSTAGE;
    static constexpr int B_KVEMPTY = B_VFULL + NSTAGE;
    static constexpr int B_SFULL = B_KVEMPTY + NSTAGE;  // 2
    static constexpr int B_SFREE = B_SFULL + 2;         // 2
    static constexpr int B_PFULL = B_SFREE + 2;
    static constexpr int B_ODONE = B_PFULL + 1;
    static constexpr int B_DRAIN = B_ODONE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
    static_assert(8 * NUM_BARS + 8 <= BAR_BYTES, "barrier area too small");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
};

// Wait that only honours the time limit (not the abort flag): used to drain
// copies and MMAs still in flight before the CTA exits.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO, float *__restrict__ lse,
                            int N, int num_q_tiles, float scale_log2, int causal,
                            uint32_t *status, uint64_t timeout_ns) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q;
    const uint32_t sK0 = sbase + C::OFF_K;
    const uint32_t sV0 = sbase + C::OFF_V;
    const uint32_t sP = sbase + C::OFF_P;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    // Heaviest causal tiles first: grid.y walks query tiles from the end.
    const int q_tile = causal ? (num_q_tiles - 1 - (int)blockIdx.y) : (int)blockIdx.y;
    const int row0 = q_tile * BM;
    const int nkv = (N + BN - 1) / BN;
    const int T = causal ? min(q_tile + 1, nkv) : nkv;  // key tiles this CTA visits

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_Q), 1);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_SFREE + b), BM);
        }
        mbar_init(bar(C::B_PFULL), BM);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_Q), C::Q_BYTES);
            for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(sQ + c * (BM * 128), &tmQ, c * 64, row0, bh, bar(C::B_Q));
            int j = 0;
            for (; j < T; ++j) {
                const int s = j % C::NSTAGE;
                if (j >= C::NSTAGE &&
                    !bounded_wait(bar(C::B_KVEMPTY + s), ((j / C::NSTAGE) - 1) & 1, ctl))
                    break;
                const uint32_t sK = sK0 + s * C::KV_BYTES, sV = sV0 + s * C::KV_BYTES;
                mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::KV_BYTES);
                for (int c = 0; c < C::DBLK; ++c)
                    tma_load_3d(sK + c * (BN * 128), &tmK, c * 64, j * BN, bh,
                                bar(C::B_KFULL + s));
                mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::KV_BYTES);
                for (int c = 0; c < C::DBLK; ++c)
                    tma_load_3d(sV + c * (BN * 128), &tmV, c * 64, j * BN, bh,
                                bar(C::B_VFULL + s));
            }
            // Let the copies issued last on each stage land before exiting
            // (already complete on the normal path).
            drain_wait(bar(C::B_Q), 0, timeout_ns);
            for (int jj = (j > C::NSTAGE ? j - C::NSTAGE : 0); jj < j; ++jj) {
                const int s = jj % C::NSTAGE;
                drain_wait(bar(C::B_KFULL + s), (jj / C::NSTAGE) & 1, timeout_ns);
                drain_wait(bar(C::B_VFULL + s), (jj / C::NSTAGE) & 1, timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------- MMA ---
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, false, true);
            auto issue_s = [&](int jt) {
                const int s = jt % C::NSTAGE;
                const uint32_t sK = sK0 + s * C::KV_BYTES;
                const uint32_t dS = tmem + ((jt & 1) ? TMEM_S1 : TMEM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    const uint64_t a = sdesc_sw128(sQ + koff, 16, 1024);
                    const uint64_t b = sdesc_sw128(sK + (kk >> 2) * (BN * 128) + (kk & 3) * 32,
                                                   16, 1024);
                    mma_bf16_ss(dS, a, b, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::B_SFULL + (jt & 1)));
            };
            bool ok = bounded_wait(bar(C::B_Q), 0, ctl) &&
                      bounded_wait(bar(C::B_KFULL + 0), 0, ctl);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; ok && j < T; ++j) {
                if (j + 1 < T) {
                    const int jn = j + 1;
                    ok = bounded_wait(bar(C::B_KFULL + jn % C::NSTAGE), (jn / C::NSTAGE) & 1, ctl);
                    if (ok && jn >= 2)
                        ok = bounded_wait(bar(C::B_SFREE + (jn & 1)), ((jn >> 1) - 1) & 1, ctl);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(jn);
                }
                const int s = j % C::NSTAGE;
                ok = bounded_wait(bar(C::B_PFULL), j & 1, ctl) &&
                     bounded_wait(bar(C::B_VFULL + s), (j / C::NSTAGE) & 1, ctl);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sV = sV0 + s * C::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t a =
                        sdesc_sw128(sP + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
                    // V tile is MN-major (d contiguous): 16 keys = 2 swizzle atoms of
                    // 8 rows x 128 B; the two 64-column halves sit BN*128 bytes apart.
                    const uint64_t b = sdesc_sw128(sV + kk * (16 * 128), BN * 128, 1024);
                    mma_bf16_ss(tmem + TMEM_O, a, b, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::B_ODONE));
                mma_commit(bar(C::B_KVEMPTY + s));
            }
            // Every MMA issued above must finish before TMEM is released.
            mma_commit(bar(C::B_DRAIN));
            drain_wait(bar(C::B_DRAIN), 0, timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax + epilogue ---
        const int t = threadIdx.x;  // row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t tO = tmem + lane_base + TMEM_O;
        const int row = row0 + t;
        const int limit = causal ? min(N, row + 1) : N;  // keys [0, limit) are visible
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_SFULL + b), (j >> 1) & 1, ctl));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_base + (b ? TMEM_S1 : TMEM_S0);
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld_32x32b_x32(tS + 0, r0);
            tmem_ld_32x32b_x32(tS + 32, r1);
            tmem_ld_32x32b_x32(tS + 64, r2);
            tmem_ld_32x32b_x32(tS + 96, r3);
            tmem_wait_ld_x32(r0);
            tmem_wait_ld_x32(r1);
            tmem_wait_ld_x32(r2);
            tmem_wait_ld_x32(r3);
            tc_fence_before();
            mbar_arrive(bar(C::B_SFREE + b));

            float s[BN];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(r0[c]) * scale_log2;
                s[32 + c] = __uint_as_float(r1[c]) * scale_log2;
                s[64 + c] = __uint_as_float(r2[c]) * scale_log2;
                s[96 + c] = __uint_as_float(r3[c]) * scale_log2;
            }
            const int key0 = j * BN;
            if (key0 + BN > limit) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (key0 + c >= limit) s[c] = -INFINITY;
            }
            float mx = m_run;
#pragma unroll
            for (int c = 0; c < BN; ++c) mx = fmaxf(mx, s[c]);
            const float m_use = (mx == -INFINITY) ? 0.f : mx;
            const float alpha = ex2_approx(m_run - m_use);
            float rs = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                const float p0 = ex2_approx(s[c] - m_use);
                const float p1 = ex2_approx(s[c + 1] - m_use);
                rs += p0 + p1;
                pk[c / 2] = pack_bf16x2(p0, p1);
            }

            if (j > 0) {
                // P_{j-1} V_{j-1} must be done: it reads the P buffer and
                // accumulates into the O row rescaled below.
                ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_ODONE), (j - 1) & 1, ctl));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(tO + c, o);
                        tmem_wait_ld_x32(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st_32x32b_x32(tO + c, o);
                    }
                    tmem_wait_st();
                }
            }
            // P row t -> shared memory, K-major with the 128-byte swizzle the
            // MMA descriptor expects (16-byte chunk c of row t at chunk c ^ (t & 7)).
#pragma unroll
            for (int c16 = 0; c16 < BN / 8; ++c16) {
                const uint32_t addr = sP + (c16 >> 3) * (BM * 128) + t * 128 +
                                      ((((uint32_t)c16 & 7u) ^ ((uint32_t)t & 7u)) << 4);
                st_shared_v4(addr, pk[c16 * 4 + 0], pk[c16 * 4 + 1], pk[c16 * 4 + 2],
                             pk[c16 * 4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL));
            l_run = l_run * alpha + rs;
            m_run = mx;
        }
        if (ok) ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_ODONE), (T - 1) & 1, ctl));
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l_run;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tO + c, o);
                tmem_wait_ld_x32(o);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int dcol = c + i * 8;
                    const uint32_t chunk = (uint32_t)(dcol & 63) >> 3;
                    const uint32_t addr = sP + (dcol >> 6) * (BM * 128) + t * 128 +
                                          ((chunk ^ ((uint32_t)t & 7u)) << 4);
                    st_shared_v4(addr,
                                 pack_bf16x2(__uint_as_float(o[i * 8 + 0]) * inv_l,
                                             __uint_as_float(o[i * 8 + 1]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[i * 8 + 2]) * inv_l,
                                             __uint_as_float(o[i * 8 + 3]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[i * 8 + 4]) * inv_l,
                                             __uint_as_float(o[i * 8 + 5]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[i * 8 + 6]) * inv_l,
                                             __uint_as_float(o[i * 8 + 7]) * inv_l));
                }
            }
            if (lse != nullptr && row < N)
                lse[(size_t)bh * (size_t)N + (size_t)row] = (m_run + log2f(l_run)) * LN2;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, BM);
        if (t == 0 && *abort_flag == 0u) {
            // The tensor map clips rows >= N, so a ragged last tile is safe.
            for (int c = 0; c < C::DBLK; ++c)
                tma_store_3d(&tmO, sP + c * (BM * 128), c * 64, row0, bh);
            tma_store_commit();
            tma_store_wait_read();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// A kernel whose only job is to wait, through bounded_wait, on a barrier that
// nothing signals: exercises the timeout path without hanging the GPU.
__global__ void wait_selftest_kernel(uint32_t *status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t b;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&b), 1);
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, status, timeout_ns};
    if (threadIdx.x == 0) (void)bounded_wait(smem_u32(&b), 0, ctl);
    __syncthreads();
}

// ------------------------------------------------------------- host side ---

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [BH, N, d] bf16 tensor as a 3-D map with 64-column x 128-row boxes, 128-byte
// swizzle; rows beyond N read as zero and are clipped on store.
static bool make_tmap(CUtensorMap *m, const void *ptr, int64_t BH, int64_t N, int d) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
static attn_status launch(const void *q, const void *k, const void *v, void *o, float *lse,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap(&tq, q, BH, N, D) || !make_tmap(&tk, k, BH, N, D) ||
        !make_tmap(&tv, v, BH, N, D) || !make_tmap(&to, o, BH, N, D))
        return ATTN_ERR_CUDA;
    if (cudaFuncSetAttribute(attn_fwd_bf16_tc_kernel<D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int num_q_tiles = (int)((N + BM - 1) / BM);
    const float scale_log2 = scale * 1.44269504088896340736f;
    dim3 grid((unsigned)BH, (unsigned)num_q_tiles);
    attn_fwd_bf16_tc_kernel<D><<<grid, NUM_THREADS, C::SMEM_BYTES, ctx.stream>>>(
        tq, tk, tv, to, lse, (int)N, num_q_tiles, scale_log2, causal ? 1 : 0, ctx.status,
        ctx.timeout_ns);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace tc

attn_status launch_attn_fwd_bf16(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int64_t BH, int64_t N, int d, float scale, bool causal,
                                 const LaunchCtx &ctx) {
    if (d == 64) return tc::launch<64>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    if (d == 128) return tc::launch<128>(q, k, v, o, lse, BH, N, scale, causal, ctx);
    return ATTN_ERR_HEADDIM;
}

attn_status launch_wait_selftest(const LaunchCtx &ctx) {
    tc::wait_selftest_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, ctx.timeout_ns);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace attn
