// attn_bwd_tc.cu -- bf16 attention backward on sm_103a tensor cores.
//
// The gradient of O = softmax(scale Q K^T) V from the forward's saved LSE (the
// pages give no attention backward; this is the plain derivative of the
// forward formula of page "Hardware Acceleration & Custom Kernels", section
// 2, the same one the CUDA-core backward computes):
//     P_ij  = exp(scale q_i.k_j - LSE_i)        (0 for masked keys)
//     D_i   = dO_i . O_i
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO.
//
// Two kernels, no atomics, both built like the forward kernel (TMA producer
// warp, one MMA-issuing thread, four warps that own one TMEM lane = one row
// each):
//
//   bwd_dkdv_tc_kernel   one CTA per 128-key block (keys on the TMEM lanes).
//       K and V stay in shared memory; Q and dO blocks stream through a ring
//       of block pairs (two stages at d = 128, three at d = 64).  Per query
//       block:
//         S^T = K Q^T,  dP^T = V dO^T                  (SS MMAs -> TMEM)
//         P^T = exp2(S^T scale log2e - LSE log2e),  dS^T = P^T (dP^T - D)
//                                                     (CUDA cores, bf16 -> TMEM)
//         dV += P^T dO,  dK += dS^T Q                  (TS MMAs, A from TMEM)
//       issued as dV(t), S^T(t+1), dK(t), dP^T(t+1), so the row warps' work
//       on block t overlaps dP^T(t), dV(t) and S^T(t+1).
//   bwd_dq_tc_kernel     one CTA per 128-query block (queries on the lanes).
//       Q and dO stay; K and V blocks stream through rings of their own (three
//       K slots, two V slots at d = 128, three at d = 64).  Per key block:
//         S = Q K^T,  dP = dO V^T;  dS = P (dP - D);  dQ += dS K,
//       with S of the next block issued as soon as the row warps have read S.
//
// The dQ kernel is launched as a programmatic dependent of the dK/dV kernel:
// it reads nothing the first one writes, so its CTAs start on SMs the first
// one's last wave leaves free, and it completes only after it.
//
// S and dP are recomputed in the second kernel (7 GEMMs where a single pass
// with atomic dQ updates would do 5) so that every output row has exactly one
// writer.  P and dS are rounded to bf16 for the MMAs; every sum accumulates
// in fp32 in TMEM.  TMEM (512 columns): S/P, dP/dS, then dV and dK (or dQ).
#include <cuda.h>

#include <cmath>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace bwdtc {

constexpr int BM = 128;            // rows of the block a CTA owns
constexpr int BN = 128;            // rows of a streamed block
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr int NUM_THREADS = 192;   // 4 row warps + TMA warp + MMA warp
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E = 1.44269504088896340736f;

// TMEM columns of both kernels, and the dK/dV kernel's shared memory (the dQ
// kernel's is DqCfg below).
template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
    // Ring depth: two streamed block pairs at d = 128 (shared memory is full),
    // three at d = 64.
    static constexpr int NS = (D == 64) ? 3 : 2;
    static constexpr int DBLK = D / 64;                  // 128-byte column blocks per row
    static constexpr uint32_t TILE = BM * D * 2;          // one 128-row bf16 tile
    static constexpr uint32_t OFF_RES = 0;                // two resident tiles
    static constexpr uint32_t OFF_RING = 2 * TILE;        // NS x two streamed tiles
    static constexpr uint32_t OFF_VEC = OFF_RING + NS * 2 * TILE;  // [2 buf][2][BN] floats
    static constexpr uint32_t OFF_BAR = OFF_VEC + 2 * 2 * BN * 4;
    static constexpr uint32_t BAR_BYTES = 128;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + base alignment slack
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_ACC0 = 256, TM_ACC1 = 256 + D;
    static constexpr int B_RES = 0;                  // resident tiles landed
    static constexpr int B_FULL = 1;                 // [NS] streamed pair landed
    static constexpr int B_EMPTY = B_FULL + NS;  // [NS] streamed pair consumed
    static constexpr int B_SFULL = B_EMPTY + NS; // S in TMEM
    static constexpr int B_DPRDY = B_SFULL + 1;      // dP in TMEM
    static constexpr int B_PFULL = B_DPRDY + 1;      // P in TMEM (dK/dV kernel; one arrival per row)
    static constexpr int B_DSRDY = B_PFULL + 1;      // dS in TMEM (one arrival per row)
    static constexpr int B_DONE = B_DSRDY + 1;       // every MMA finished
    static constexpr int NUM_BARS = B_DONE + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
    static_assert(8 * NUM_BARS + 8 <= BAR_BYTES, "barrier area too small");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    static_assert(TM_ACC1 + D <= TMEM_COLS, "TMEM budget exceeded");
};

// The dQ kernel's shared memory: Q and dO resident, and K and V streamed
// through rings of their own, KS slots for K (S of the next key block is
// issued as soon as the row warps have read S, so its K is wanted early) and
// VS for V.  A V slot comes back with the K slot of the same key block: dQ +=
// dS K, whose completion frees that K slot, is issued after dP has read V.
template <int D>
struct DqCfg {
    using C = Cfg<D>;
    static constexpr int KS = 3;
    static constexpr int VS = (D == 64) ? 3 : 2;
    static constexpr int DBLK = C::DBLK;
    static constexpr uint32_t TILE = C::TILE;
    static constexpr uint32_t TM_S = C::TM_S, TM_DP = C::TM_DP, TM_ACC0 = C::TM_ACC0;
    static constexpr uint32_t OFF_RES = 0;                     // Q, dO
    static constexpr uint32_t OFF_K = 2 * TILE;                // KS K slots
    static constexpr uint32_t OFF_V = OFF_K + KS * TILE;       // VS V slots
    static constexpr uint32_t OFF_BAR = OFF_V + VS * TILE;
    static constexpr int B_RES = 0;
    static constexpr int B_FULLK = 1;                 // [KS] K slot landed
    static constexpr int B_EMPTYK = B_FULLK + KS;     // [KS] K slot (and the V of that block) consumed
    static constexpr int B_FULLV = B_EMPTYK + KS;     // [VS] V slot landed
    static constexpr int B_SFULL = B_FULLV + VS;
    static constexpr int B_DPRDY = B_SFULL + 1;
    static constexpr int B_PFULL = B_DPRDY + 1;
    static constexpr int B_DSRDY = B_PFULL + 1;
    static constexpr int B_DONE = B_DSRDY + 1;
    static constexpr int NUM_BARS = B_DONE + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
    static constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + base alignment slack
    static_assert(VS <= KS, "a V slot is freed through the K ring");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// Row r of a 128-row tile staged in the tensor maps' 128-byte swizzle: 16-byte
// chunk c (8 bf16) of 64-column block b.
__device__ __forceinline__ uint32_t swz_addr(uint32_t tile, int r, int col) {
    const uint32_t chunk = (uint32_t)(col & 63) >> 3;
    return tile + (uint32_t)(col >> 6) * (BM * 128) + (uint32_t)r * 128 +
           ((chunk ^ ((uint32_t)r & 7u)) << 4);
}

// Write a row of D fp32 accumulator columns (times `mul`) as bf16 into a
// staged tile.
template <int D>
__device__ __forceinline__ void stage_row(uint32_t tacc, uint32_t tile, int r, float mul) {
#pragma unroll
    for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tacc + c, o);
        tmem_wait_ld_x32(o);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_shared_v4(swz_addr(tile, r, c + 8 * i),
                         pack_bf16x2(__uint_as_float(o[8 * i + 0]) * mul,
                                     __uint_as_float(o[8 * i + 1]) * mul),
                         pack_bf16x2(__uint_as_float(o[8 * i + 2]) * mul,
                                     __uint_as_float(o[8 * i + 3]) * mul),
                         pack_bf16x2(__uint_as_float(o[8 * i + 4]) * mul,
                                     __uint_as_float(o[8 * i + 5]) * mul),
                         pack_bf16x2(__uint_as_float(o[8 * i + 6]) * mul,
                                     __uint_as_float(o[8 * i + 7]) * mul));
    }
}

// dS = P (dP - D) for one row of 128 columns: P (fp32) is in p[]; dP is read
// from TMEM 32 columns at a time and dS (bf16 pairs) written back over the
// first 64 dP columns.  Chunk ch writes columns [16 ch, 16 ch + 16), all of
// which belong to dP chunks already read.  `ndl(c)` gives the packed pair
// (-D_c, -D_{c+1}); the arithmetic is packed (f32x2).
template <typename NegDeltaFn>
__device__ __forceinline__ void ds_row(uint32_t tdp, const float (&p)[128], NegDeltaFn ndl) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        uint32_t g[32];
        tmem_ld_32x32b_x32(tdp + 32 * ch, g);
        tmem_wait_ld_x32(g);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = 32 * ch + 2 * i;
            const uint64_t diff =
                fadd2(pack_f32x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1])), ndl(c));
            float d0, d1;
            unpack_f32x2(fmul2(pack_f32x2(p[c], p[c + 1]), diff), d0, d1);
            pk[i] = pack_bf16x2(d0, d1);
        }
        tmem_st_32x32b_x16(tdp + 16 * ch, pk);
    }
}

// P for one row of 128 columns: p[c] = 2^(s_c * sl + nb(c)), with nb(c) the
// packed pair of biases for columns c, c+1; columns c < first_col are zero.
// The mask is applied only where a block needs it.
template <typename BiasFn>
__device__ __forceinline__ void p_row(const uint32_t (&r)[4][32], float sl, BiasFn nb, int first_col,
                                      int last_col, bool masked, float (&p)[128]) {
    const uint64_t sl2 = pack_f32x2(sl, sl);
    if (!masked) {
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
            float a0, a1;
            unpack_f32x2(ffma2(pack_f32x2(__uint_as_float(r[c >> 5][c & 31]),
                                          __uint_as_float(r[c >> 5][(c & 31) + 1])),
                               sl2, nb(c)),
                         a0, a1);
            p[c] = ex2_approx(a0);
            p[c + 1] = ex2_approx(a1);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
            float a0, a1;
            unpack_f32x2(ffma2(pack_f32x2(__uint_as_float(r[c >> 5][c & 31]),
                                          __uint_as_float(r[c >> 5][(c & 31) + 1])),
                               sl2, nb(c)),
                         a0, a1);
            p[c] = (c >= first_col && c < last_col) ? ex2_approx(a0) : 0.f;
            p[c + 1] = (c + 1 >= first_col && c + 1 < last_col) ? ex2_approx(a1) : 0.f;
        }
    }
}

// --------------------------------------------------------- dK and dV ---

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmG,
                       const __grid_constant__ CUtensorMap tmDK,
                       const __grid_constant__ CUtensorMap tmDV, const float *__restrict__ lse,
                       const float *__restrict__ delta, int N, float scale, int causal,
                       uint32_t *status, uint64_t timeout_ns) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::OFF_RES, sV = sK + C::TILE;
    auto sQ = [&](int s) -> uint32_t { return sbase + C::OFF_RING + (uint32_t)s * 2 * C::TILE; };
    auto sG = [&](int s) -> uint32_t { return sQ(s) + C::TILE; };
    float *vec = reinterpret_cast<float *>(smem + C::OFF_VEC);  // [buf][0: -LSE log2e, 1: D][BN]
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int kb = blockIdx.y;  // key block (small kb = most query blocks with the causal mask)
    const int nq = (N + BN - 1) / BN;
    const int q0 = causal ? kb : 0;  // query blocks q0 .. nq-1 see this key block
    const int T = nq - q0;
    // The dQ launch that follows reads nothing this kernel writes: let it
    // start on SMs this launch has finished with.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_RES), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPRDY), 1);
        mbar_init(bar(C::B_PFULL), BM);
        mbar_init(bar(C::B_DSRDY), BM);
        mbar_init(bar(C::B_DONE), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (warp == WARP_TMA) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_RES), 2 * C::TILE);
            for (int c = 0; c < C::DBLK; ++c) {
                tma_load_3d(sK + c * (BM * 128), &tmK, c * 64, kb * BM, bh, bar(C::B_RES));
                tma_load_3d(sV + c * (BM * 128), &tmV, c * 64, kb * BM, bh, bar(C::B_RES));
            }
            int t = 0;
            for (; t < T; ++t) {
                const int s = t % C::NS;
                if (t >= C::NS &&
                    !bounded_wait(bar(C::B_EMPTY + s), ((t / C::NS) - 1) & 1, ctl))
                    break;
                const int qr = (q0 + t) * BN;
                mbar_arrive_expect_tx(bar(C::B_FULL + s), 2 * C::TILE);
                for (int c = 0; c < C::DBLK; ++c) {
                    tma_load_3d(sQ(s) + c * (BN * 128), &tmQ, c * 64, qr, bh, bar(C::B_FULL + s));
                    tma_load_3d(sG(s) + c * (BN * 128), &tmG, c * 64, qr, bh, bar(C::B_FULL + s));
                }
            }
            drain_wait(bar(C::B_RES), 0, timeout_ns);
            for (int i = (t > C::NS ? t - C::NS : 0); i < t; ++i)
                drain_wait(bar(C::B_FULL + i % C::NS), (i / C::NS) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, false, true);
            const uint64_t kdesc = sdesc_sw128(sK, 16, 1024), vdesc = sdesc_sw128(sV, 16, 1024);
            // S^T = K Q^T and dP^T = V dO^T of query block t (both operands
            // K-major), each on its own barrier so the row warps start on P^T
            // while dP^T is still being computed.
            auto issue_s = [&](int t) {
                const uint64_t b = sdesc_sw128(sQ(t % C::NS), 16, 1024);
                if constexpr (D == 128)
                    gemm_ss_k8(tmem + C::TM_S, kdesc, b, idesc_s, 0u);
                else
                    gemm_ss_k4(tmem + C::TM_S, kdesc, b, idesc_s, 0u);
                mma_commit(bar(C::B_SFULL));
            };
            auto issue_dp = [&](int t) {
                const uint64_t b = sdesc_sw128(sG(t % C::NS), 16, 1024);
                if constexpr (D == 128)
                    gemm_ss_k8(tmem + C::TM_DP, vdesc, b, idesc_s, 0u);
                else
                    gemm_ss_k4(tmem + C::TM_DP, vdesc, b, idesc_s, 0u);
                mma_commit(bar(C::B_DPRDY));
            };
            bool ok = bounded_wait(bar(C::B_RES), 0, ctl) && bounded_wait(bar(C::B_FULL), 0, ctl);
            if (ok) {
                issue_s(0);
                issue_dp(0);
            }
            // Per block t: dV += P^T dO, then S^T of block t+1 (it overwrites
            // P^T, after dV in issue order), then dK += dS^T Q, then dP^T of
            // block t+1 (it overwrites dS^T, after dK).  The row warps' work
            // on block t overlaps dP^T(t), dV(t) and S^T(t+1).  A (bf16 pairs)
            // comes from TMEM; B is the streamed tile read MN-major (d
            // contiguous; the two 64-column halves BN*128 bytes apart).
            for (int t = 0; ok && t < T; ++t) {
                const int s = t % C::NS;
                if (!(ok = spin_wait(bar(C::B_PFULL), t & 1, ctl))) break;
                tc_fence_after();
                gemm_ts_k8(tmem + C::TM_ACC0, tmem + C::TM_S, sdesc_sw128(sG(s), BN * 128, 1024),
                           idesc_o, t > 0 ? 1u : 0u);
                if (t + 1 < T) {
                    if (!(ok = bounded_wait(bar(C::B_FULL + (t + 1) % C::NS),
                                            ((t + 1) / C::NS) & 1, ctl)))
                        break;
                    issue_s(t + 1);
                }
                if (!(ok = spin_wait(bar(C::B_DSRDY), t & 1, ctl))) break;
                tc_fence_after();
                gemm_ts_k8(tmem + C::TM_ACC1, tmem + C::TM_DP, sdesc_sw128(sQ(s), BN * 128, 1024),
                           idesc_o, t > 0 ? 1u : 0u);
                mma_commit(bar(C::B_EMPTY + s));
                if (t + 1 < T) issue_dp(t + 1);
            }
            mma_commit(bar(C::B_DONE));
            drain_wait(bar(C::B_DONE), 0, timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------- rows: one key per thread ---
        const int t = threadIdx.x;  // 0..127 == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::TM_S, tDP = tmem + lane_base + C::TM_DP;
        const float sl = scale * LOG2E;
        const float *lse_bh = lse + (size_t)bh * (size_t)N;
        const float *dl_bh = delta + (size_t)bh * (size_t)N;
        bool ok = true;
        // All four warps run every step (a failed wait only makes the rest
        // return at once), so the named barrier below always sees them all.
        // This thread's query column of the next block is read from global
        // memory one step ahead, so its latency hides behind a block's work.
        auto col_vals = [&](int st_, float &nb_, float &dv_) {
            const int qi = (q0 + st_) * BN + t;
            nb_ = qi < N ? -lse_bh[qi] * LOG2E : -INFINITY;  // rows past N: P = 0
            dv_ = qi < N ? -dl_bh[qi] : 0.f;                 // -D, for the packed dP - D
        };
        float nb_next = 0.f, dv_next = 0.f;
        if (T > 0) col_vals(0, nb_next, dv_next);
        for (int st = 0; st < T; ++st) {
            const int qb = q0 + st;
            float *nb = vec + (st & 1) * 2 * BN;  // -LSE log2e per query column
            float *dv = nb + BN;                 // -D per query column
            nb[t] = nb_next;
            dv[t] = dv_next;
            if (st + 1 < T) col_vals(st + 1, nb_next, dv_next);
            named_bar_sync(1, BM);
            ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_SFULL), st & 1, ctl)) && ok;
            tc_fence_after();
            uint32_t r[4][32];
            tmem_ld_32x32b_x32(tS + 0, r[0]);
            tmem_ld_32x32b_x32(tS + 32, r[1]);
            tmem_ld_32x32b_x32(tS + 64, r[2]);
            tmem_ld_32x32b_x32(tS + 96, r[3]);
            tmem_wait_ld_x32(r[0]);
            tmem_wait_ld_x32(r[1]);
            tmem_wait_ld_x32(r[2]);
            tmem_wait_ld_x32(r[3]);
            // On the diagonal block, query column c sees this key only if c >= t
            // (query rows past N already have a -inf bias).
            const bool diag = causal && qb == kb;
            float p[128];
            p_row(r, sl, [&](int c) { return *reinterpret_cast<const uint64_t *>(nb + c); },
                  diag ? t : 0, 128, diag, p);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(p[64 * h + 2 * i], p[64 * h + 2 * i + 1]);
                tmem_st_32x32b_x32(tS + 32 * h, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL));  // dV += P^T dO may start
            ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_DPRDY), st & 1, ctl)) && ok;
            tc_fence_after();
            ds_row(tDP, p, [&](int c) { return *reinterpret_cast<const uint64_t *>(dv + c); });
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_DSRDY));
        }
        ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_DONE), 0, ctl)) && ok;
        // K and V are no longer read (every MMA is done): stage dV and dK there.
        if (ok) {
            tc_fence_after();
            stage_row<D>(tmem + lane_base + C::TM_ACC0, sV, t, 1.f);
            stage_row<D>(tmem + lane_base + C::TM_ACC1, sK, t, scale);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, BM);
        if (t == 0 && ok && *abort_flag == 0u) {
            // The tensor maps clip rows >= N.
            for (int c = 0; c < C::DBLK; ++c) {
                tma_store_3d(&tmDV, sV + c * (BM * 128), c * 64, kb * BM, bh);
                tma_store_3d(&tmDK, sK + c * (BM * 128), c * 64, kb * BM, bh);
            }
            tma_store_commit();
            tma_store_wait_read();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- dQ ---

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmDQ, const float *__restrict__ lse,
                     const float *__restrict__ delta, int N, float scale, int causal,
                     uint32_t *status, uint64_t timeout_ns) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_RES, sG = sQ + C::TILE;
    auto sK = [&](int s) -> uint32_t { return sbase + C::OFF_K + (uint32_t)s * C::TILE; };
    auto sV = [&](int s) -> uint32_t { return sbase + C::OFF_V + (uint32_t)s * C::TILE; };
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int nq = (N + BM - 1) / BM;
    // Heaviest query blocks first with the causal mask.
    const int qb = causal ? (nq - 1 - (int)blockIdx.y) : (int)blockIdx.y;
    const int nk = (N + BN - 1) / BN;
    const int T = causal ? qb + 1 : nk;  // key blocks 0 .. T-1

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_RES), 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar(C::B_FULLK + s), 1);
            mbar_init(bar(C::B_EMPTYK + s), 1);
        }
        for (int s = 0; s < C::VS; ++s) mbar_init(bar(C::B_FULLV + s), 1);
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPRDY), 1);
        mbar_init(bar(C::B_PFULL), BM);
        mbar_init(bar(C::B_DSRDY), BM);
        mbar_init(bar(C::B_DONE), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (warp == WARP_TMA) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_RES), 2 * C::TILE);
            for (int c = 0; c < C::DBLK; ++c) {
                tma_load_3d(sQ + c * (BM * 128), &tmQ, c * 64, qb * BM, bh, bar(C::B_RES));
                tma_load_3d(sG + c * (BM * 128), &tmG, c * 64, qb * BM, bh, bar(C::B_RES));
            }
            int tk = 0, tv = 0;  // K and V loads issued
            for (int t = 0; t < T; ++t) {
                const int sk = t % C::KS, sv = t % C::VS;
                if (t >= C::KS &&
                    !bounded_wait(bar(C::B_EMPTYK + sk), ((t / C::KS) - 1) & 1, ctl))
                    break;
                mbar_arrive_expect_tx(bar(C::B_FULLK + sk), C::TILE);
                for (int c = 0; c < C::DBLK; ++c)
                    tma_load_3d(sK(sk) + c * (BN * 128), &tmK, c * 64, t * BN, bh,
                                bar(C::B_FULLK + sk));
                tk = t + 1;
                // The V slot held V(t - VS), read by dP(t - VS), which was
                // issued before dQ(t - VS): that K slot's release frees it.
                if (t >= C::VS && !bounded_wait(bar(C::B_EMPTYK + (t - C::VS) % C::KS),
                                                ((t - C::VS) / C::KS) & 1, ctl))
                    break;
                mbar_arrive_expect_tx(bar(C::B_FULLV + sv), C::TILE);
                for (int c = 0; c < C::DBLK; ++c)
                    tma_load_3d(sV(sv) + c * (BN * 128), &tmV, c * 64, t * BN, bh,
                                bar(C::B_FULLV + sv));
                tv = t + 1;
            }
            drain_wait(bar(C::B_RES), 0, timeout_ns);
            for (int i = (tk > C::KS ? tk - C::KS : 0); i < tk; ++i)
                drain_wait(bar(C::B_FULLK + i % C::KS), (i / C::KS) & 1, timeout_ns);
            for (int i = (tv > C::VS ? tv - C::VS : 0); i < tv; ++i)
                drain_wait(bar(C::B_FULLV + i % C::VS), (i / C::VS) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, false, true);
            const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024), gdesc = sdesc_sw128(sG, 16, 1024);
            // S = Q K^T and dP = dO V^T of key block t, each on its own barrier.
            auto issue_s = [&](int t) {
                const uint64_t b = sdesc_sw128(sK(t % C::KS), 16, 1024);
                if constexpr (D == 128)
                    gemm_ss_k8(tmem + C::TM_S, qdesc, b, idesc_s, 0u);
                else
                    gemm_ss_k4(tmem + C::TM_S, qdesc, b, idesc_s, 0u);
                mma_commit(bar(C::B_SFULL));
            };
            auto issue_dp = [&](int t) {
                const uint64_t b = sdesc_sw128(sV(t % C::VS), 16, 1024);
                if constexpr (D == 128)
                    gemm_ss_k8(tmem + C::TM_DP, gdesc, b, idesc_s, 0u);
                else
                    gemm_ss_k4(tmem + C::TM_DP, gdesc, b, idesc_s, 0u);
                mma_commit(bar(C::B_DPRDY));
            };
            auto full_k = [&](int t) {
                return bounded_wait(bar(C::B_FULLK + t % C::KS), (t / C::KS) & 1, ctl);
            };
            auto full_v = [&](int t) {
                return bounded_wait(bar(C::B_FULLV + t % C::VS), (t / C::VS) & 1, ctl);
            };
            bool ok = bounded_wait(bar(C::B_RES), 0, ctl) && full_k(0);
            if (ok) issue_s(0);
            if (ok && (ok = full_v(0))) issue_dp(0);
            // Per block t: S of block t+1 as soon as the row warps have read S
            // and K of block t+1 has landed (if it has not landed yet, after
            // dQ), dQ += dS K (A = dS from TMEM, B = the K tile read MN-major),
            // then dP of block t+1 (it overwrites dS, after dQ in issue order).
            for (int t = 0; ok && t < T; ++t) {
                const int sk = t % C::KS;
                bool s_next = false;
                if (t + 1 < T) {
                    if (!(ok = spin_wait(bar(C::B_PFULL), t & 1, ctl))) break;  // S(t) read
                    tc_fence_after();
                    if (mbar_test_wait(bar(C::B_FULLK + (t + 1) % C::KS), ((t + 1) / C::KS) & 1)) {
                        issue_s(t + 1);
                        s_next = true;
                    }
                }
                if (!(ok = spin_wait(bar(C::B_DSRDY), t & 1, ctl))) break;
                tc_fence_after();
                gemm_ts_k8(tmem + C::TM_ACC0, tmem + C::TM_DP, sdesc_sw128(sK(sk), BN * 128, 1024),
                           idesc_o, t > 0 ? 1u : 0u);
                mma_commit(bar(C::B_EMPTYK + sk));
                if (t + 1 < T) {
                    if (!s_next) {
                        if (!(ok = full_k(t + 1))) break;
                        issue_s(t + 1);
                    }
                    if (!(ok = full_v(t + 1))) break;
                    issue_dp(t + 1);
                }
            }
            mma_commit(bar(C::B_DONE));
            drain_wait(bar(C::B_DONE), 0, timeout_ns);
        }
        __syncwarp();
    } else {
        // ----------------------------------- rows: one query per thread ---
        const int t = threadIdx.x;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::TM_S, tDP = tmem + lane_base + C::TM_DP;
        const int row = qb * BM + t;
        const float sl = scale * LOG2E;
        const float nb = row < N ? -lse[(size_t)bh * N + row] * LOG2E : -INFINITY;
        const float dl = row < N ? delta[(size_t)bh * N + row] : 0.f;
        const uint64_t nb2 = pack_f32x2(nb, nb), ndl2 = pack_f32x2(-dl, -dl);
        const int limit = causal ? min(N, row + 1) : N;  // keys [0, limit) are visible
        bool ok = true;
        for (int st = 0; st < T; ++st) {
            ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_SFULL), st & 1, ctl)) && ok;
            tc_fence_after();
            uint32_t r[4][32];
            tmem_ld_32x32b_x32(tS + 0, r[0]);
            tmem_ld_32x32b_x32(tS + 32, r[1]);
            tmem_ld_32x32b_x32(tS + 64, r[2]);
            tmem_ld_32x32b_x32(tS + 96, r[3]);
            tmem_wait_ld_x32(r[0]);
            tmem_wait_ld_x32(r[1]);
            tmem_wait_ld_x32(r[2]);
            tmem_wait_ld_x32(r[3]);
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL));  // S read: the next S may overwrite it
            // Key columns [0, limit - key0) are visible; only the diagonal block
            // (causal) and the block holding key N-1 need the mask.
            const int key0 = st * BN;
            const bool masked = key0 + BN > (causal ? min(N, qb * BM + 1) : N);
            float p[128];
            p_row(r, sl, [&](int) { return nb2; }, 0, limit - key0, masked, p);
            ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_DPRDY), st & 1, ctl)) && ok;
            tc_fence_after();
            ds_row(tDP, p, [&](int) { return ndl2; });
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_DSRDY));
        }
        ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_DONE), 0, ctl)) && ok;
        // Q is no longer read: stage dQ there.
        if (ok) {
            tc_fence_after();
            stage_row<D>(tmem + lane_base + C::TM_ACC0, sQ, t, scale);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, BM);
        if (t == 0 && ok && *abort_flag == 0u) {
            for (int c = 0; c < C::DBLK; ++c)
                tma_store_3d(&tmDQ, sQ + c * (BM * 128), c * 64, qb * BM, bh);
            tma_store_commit();
            tma_store_wait_read();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // This launch may start before the dK/dV kernel of the same call has
    // finished; it completes only after it.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int D>
static attn_status launch(const void *q, const void *k, const void *v, const void *dout,
                          const float *lse, const float *delta, void *dq, void *dk, void *dv,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv, tg, tdq, tdk, tdv;
    if (!make_tmap_bf16(&tq, q, BH, N, D) || !make_tmap_bf16(&tk, k, BH, N, D) ||
        !make_tmap_bf16(&tv, v, BH, N, D) || !make_tmap_bf16(&tg, dout, BH, N, D) ||
        !make_tmap_bf16(&tdq, dq, BH, N, D) || !make_tmap_bf16(&tdk, dk, BH, N, D) ||
        !make_tmap_bf16(&tdv, dv, BH, N, D))
        return ATTN_ERR_CUDA;
    if (check_launch(cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)C::SMEM_BYTES),
                     ATTN_ERR_CUDA) != ATTN_OK ||
        check_launch(cudaFuncSetAttribute(bwd_dq_tc_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)DqCfg<D>::SMEM_BYTES),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    const dim3 grid((unsigned)BH, (unsigned)((N + BM - 1) / BM));
    bwd_dkdv_tc_kernel<D><<<grid, NUM_THREADS, C::SMEM_BYTES, ctx.stream>>>(
        tq, tk, tv, tg, tdk, tdv, lse, delta, (int)N, scale, causal ? 1 : 0, ctx.status,
        ctx.timeout_ns);
    attn_status st = check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
    if (st != ATTN_OK) return st;
    // dQ as a programmatic dependent of dK/dV: both only read what earlier
    // launches (D included) wrote, so dQ's CTAs may start early.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = DqCfg<D>::SMEM_BYTES;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_launch(cudaLaunchKernelEx(&cfg, bwd_dq_tc_kernel<D>, tq, tk, tv, tg, tdq, lse,
                                           delta, (int)N, scale, causal ? 1 : 0, ctx.status,
                                           ctx.timeout_ns),
                        ATTN_ERR_LAUNCH);
}

}  // namespace bwdtc

attn_status launch_attn_bwd_bf16_tc(const void *q, const void *k, const void *v, const void *dout,
                                    const float *lse, const float *delta, void *dq, void *dk,
                                    void *dv, int64_t BH, int64_t N, int d, float scale,
                                    bool causal, const LaunchCtx &ctx) {
    if (d == 64)
        return bwdtc::launch<64>(q, k, v, dout, lse, delta, dq, dk, dv, BH, N, scale, causal, ctx);
    if (d == 128)
        return bwdtc::launch<128>(q, k, v, dout, lse, delta, dq, dk, dv, BH, N, scale, causal, ctx);
    return ATTN_ERR_HEADDIM;
}

}  // namespace attn
