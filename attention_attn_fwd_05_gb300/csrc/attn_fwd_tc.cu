// attn_fwd_tc.cu -- bf16 exact attention forward on sm_103a tensor cores.
//
// Computes O = softmax(scale * Q K^T) V and LSE per row (page "Hardware
// Acceleration & Custom Kernels", section 2: the attention formula, SRAM
// tiling into B_r x d and B_c x d blocks, and the online normalisation
// m_new = max(m_old, x), d_new = d_old e^(m_old - m_new) + e^(x - m_new)
// applied per key tile, rescaling the running output sums as tiles arrive).
//
// One CTA owns two 128-row query tiles (A: rows r0..r0+127, B: r0+128..r0+255)
// of one (batch, head) and walks the key tiles j = 0 .. T-1 (up to the
// diagonal with the causal mask).  Both tiles share every K and V tile.
//
//   warp 8      TMA producer: initialises the barriers and issues Q_A, K_0,
//               Q_B, V_0 (each query tile on its own barrier, so S_A(0) waits
//               only for Q_A and K_0) before the CTA-wide barrier, which lets
//               those copies overlap the TMEM allocation; it also warms L2
//               with the query block of the CTA that will start next.  Then
//               K_1, V_1, K_2, ... into a ring of NSLOT shared-memory slots
//               (128-byte swizzle, 64-column boxes).  Slots come back when the
//               softmax sees S complete (see softmax_warpgroup).
//   d = 128:
//   warp 9      TMEM allocator and MMA issuer (one thread).  Per key tile j it
//               issues, in this order,
//                 S_A(j) = Q_A K_j^T,  O_B += P_B(j-1) V_{j-1},
//                 S_B(j) = Q_B K_j^T,  O_A += P_A(j) V_j,
//               so the tensor core works on one tile's products while the
//               other tile's softmax runs.  S and O accumulate in TMEM (fp32).
//               P (bf16) is written by the softmax threads into TMEM over the
//               S columns it came from and is read from there by the P V MMA
//               (A operand in TMEM): P never touches shared memory.  The next
//               S of a tile is issued after that tile's P V in the MMA stream,
//               and tcgen05 MMAs from one thread execute in issue order, so it
//               overwrites P only after P V has read it.  The S_X(j) commit
//               also covers O_X += P_X(j-1) V_{j-1}, so O is complete when S
//               is.
//   d = 64:
//   warps 9, 10 one MMA issuer per tile; each tile's P has TMEM columns of its
//               own, and its next S is issued as soon as its softmax has read
//               the current one (see the issuer).
//   warps 0-3   softmax + epilogue of tile A, one query row per thread (TMEM
//   warps 4-7   lane = row); same for tile B.  Per key tile: read S, mask,
//               row max (tree), p = 2^(s*scale*log2e - m) packed to bf16 into
//               TMEM, row sum.  The O row is rescaled only when the row max grew
//               by more than 2^8 since the reference it was last scaled to (the
//               reference only has to bound the exponentials; O and l always
//               share it, so the result is unchanged).  At the end O / l ->
//               bf16 -> shared (the Q buffer of the tile, no longer read) -> TMA
//               store, and LSE = (m + log2 l) ln 2.
//
// The launch is a list of items, one per (batch*head, 256-row query block),
// on a 1-D grid.  Heads go in groups whose K and V fit in half of L2, one group
// after the other; inside a group batch*head is fastest and the heaviest
// causal blocks come first, so the hardware's in-order dispatch acts as a
// longest-first schedule and the CTAs running together re-read K and V from
// L2 (at N = 16384, d = 128: 0.81 GB of DRAM traffic per launch instead of
// 2.27 GB with all heads in one group, for 0.54 GB of inputs and outputs).  Items that
// would leave a last wave at most half full (without the causal mask), or all
// items of a grid that fills at most half the SMs, go to a second launch of
// attn_fwd_bf16_tc_split_kernel: two CTAs per item, each on one 128-row half,
// with tile A on the even and tile B on the odd key tiles (see there).  That
// launch is a programmatic dependent of the first, so its CTAs start on the
// SMs the main kernel's last wave leaves free.
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
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 320;  // 2 softmax warpgroups + TMA warp + MMA warp
// At d = 64 each query tile has its own MMA-issuing warp (tile A: WARP_MMA,
// tile B: WARP_MMA_B).  One thread issues at most one tcgen05.mma per about 64
// cycles on GB300, the time a 128 x 128 x 16 MMA takes; a 128 x 64 x 16 product
// (P V at d = 64) takes half that, so a single issuer left the tensor pipe
// idle half of the P V time.  Two issuers reach its rate.
constexpr int WARP_MMA_B = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr float LN2 = 0.69314718055994530942f;
// Rescale O only when the running max grew by more than this (log2 units):
// exponentials are then bounded by 2^8, far inside fp32 and bf16 range.
constexpr float RESCALE_THRESHOLD = 8.0f;

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
    static constexpr int NSLOT = (D == 128) ? 5 : 8;
    static constexpr int DBLK = D / 64;  // 128-byte column blocks per row
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t SLOT_BYTES = BN * D * 2;  // one K or V tile
    static constexpr uint32_t OFF_Q = 0;                       // Q_A, Q_B (O staging later)
    static constexpr uint32_t OFF_KV = OFF_Q + 2 * Q_BYTES;    // ring
    static constexpr uint32_t OFF_BAR = OFF_KV + NSLOT * SLOT_BYTES;
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + base alignment slack
    // TMEM columns: S_A, S_B (128 fp32 columns each), then at d = 128 O_A,
    // O_B (128 each) with each P written as bf16 pairs over the first 64
    // columns of its S.  At d = 64 each tile also has a P area of its own
    // (64 columns) and O_A, O_B take 64 each: with S and P apart, the next S
    // of a tile can be computed as soon as its softmax has read the current
    // one, and each tile gets its own MMA issuer (PER_TILE).
    static constexpr bool PER_TILE = (D == 64);
    static constexpr uint32_t TM_S0 = 0, TM_S1 = 128;
    static constexpr uint32_t TM_P0 = PER_TILE ? 256 : TM_S0, TM_P1 = PER_TILE ? 320 : TM_S1;
    static constexpr uint32_t TM_O0 = PER_TILE ? 384 : 256, TM_O1 = TM_O0 + D;
    static constexpr int THREADS = PER_TILE ? NUM_THREADS + 32 : NUM_THREADS;
    // Barrier slots (8 bytes each).
    static constexpr int B_Q = 0;     // [2] Q_A, Q_B landed
    static constexpr int B_FULL = 2;                   // [NSLOT + 1] (the split kernel's ring
    static constexpr int B_EMPTY = B_FULL + NSLOT + 1;  //  has one more slot)
    static constexpr int B_SFULL = B_EMPTY + NSLOT + 1;  // [2]
    static constexpr int B_PFULL = B_SFULL + 2;      // [2]
    static constexpr int B_ODONE = B_PFULL + 2;      // [2]
    static constexpr int B_DRAIN = B_ODONE + 2;
    // PER_TILE: the softmax has read S_x (the issuer may overwrite it);
    // O_x += P_x V complete (the softmax may overwrite P_x and rescale O_x);
    // tile B's issuer drains on its own barrier.
    static constexpr int B_SFREE = B_DRAIN + 1;   // [2]
    static constexpr int B_PVDONE = B_SFREE + 2;  // [2]
    static constexpr int B_DRAIN_B = B_PVDONE + 2;
    static constexpr int NUM_BARS = B_DRAIN_B + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
    static_assert(8 * NUM_BARS + 8 <= BAR_BYTES, "barrier area too small");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    static_assert(TM_O1 + D <= TMEM_COLS, "TMEM budget exceeded");
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

// Key tiles each query tile of a CTA visits: T_A <= T_B.
__device__ __forceinline__ void tile_counts(int N, int cta_tile, int causal, int &TA, int &TB) {
    const int nkv = (N + BN - 1) / BN;
    if (causal) {
        TA = min(2 * cta_tile + 1, nkv);
        TB = min(2 * cta_tile + 2, nkv);
    } else {
        TA = TB = nkv;
    }
}

// What one softmax step leaves for its caller: the O rescale factor, the row
// sum of the tile's exponentials and the reference maximum they used.  The
// caller signals P first and folds these into its running state after, off
// the path to the MMA issuer.
struct TileStep {
    float alpha, rs, m_use;
};

// One key tile of the online softmax for the calling thread's row, shared by
// every forward kernel.  S (128 fp32 columns at tS, already complete in TMEM)
// is read, keys >= limit are masked, and against the row's reference maximum
// m_ref (log2 units) the tile's exponentials p = 2^(s * scale_log2 - m_use)
// are written to tP as bf16 pairs (P in TMEM, 64 columns; tP == tS writes
// them over the first 64 S columns).  The reference moves only when the
// tile's maximum exceeds it by more than RESCALE_THRESHOLD; the O row at tO
// is then rescaled by alpha (allowed only when `rescale_o`).  Returns after
// the P stores have completed (tcgen05.wait::st) and the tcgen05 fence, so
// the caller can arrive on the P barrier.
// PER_TILE (P apart from S): once S is read, each warp arrives on sfree_bar
// (S may then be overwritten), and before P is written (when rescale_o, i.e.
// not on the first tile) the caller's previous P V product, which reads P and
// writes O, is waited for: phase pv_parity of pv_bar.
template <int D, bool PER_TILE = false>
__device__ __forceinline__ TileStep softmax_tile(uint32_t tS, uint32_t tP, uint32_t tO, int key0,
                                                 int limit, uint64_t scale2, float scale_log2,
                                                 float m_ref, bool rescale_o,
                                                 uint32_t sfree_bar = 0, uint32_t pv_bar = 0,
                                                 uint32_t pv_parity = 0,
                                                 const WaitCtl *ctl = nullptr) {
    uint32_t r[4][32];
    tmem_ld_32x32b_x32(tS + 0, r[0]);
    tmem_ld_32x32b_x32(tS + 32, r[1]);
    tmem_ld_32x32b_x32(tS + 64, r[2]);
    tmem_ld_32x32b_x32(tS + 96, r[3]);
    tmem_wait_ld_x32(r[0]);
    tmem_wait_ld_x32(r[1]);
    tmem_wait_ld_x32(r[2]);
    tmem_wait_ld_x32(r[3]);
    if constexpr (PER_TILE) {
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(sfree_bar);
    }

    if (key0 + BN > limit) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
            if (key0 + c >= limit) r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
    }
    // Row max of the raw logits (scale_log2 > 0 commutes with max; the
    // launcher folds a negative scale into the S MMA): 8 independent
    // 3-input chains, then a short combine.
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(r[i >> 1][(i & 1) * 16]);
#pragma unroll
    for (int c = 1; c < 16; c += 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int base = (i & 1) * 16;
            mx8[i] = fmax3(mx8[i], __uint_as_float(r[i >> 1][base + c]),
                           __uint_as_float(r[i >> 1][base + (c + 1 < 16 ? c + 1 : c)]));
        }
    }
    const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                           fmaxf(mx8[6], mx8[7]));
    const float m_new = mx * scale_log2;
    const bool upd = m_new > m_ref + RESCALE_THRESHOLD;
    float m_use = upd ? m_new : m_ref;
    if (m_use == -INFINITY) m_use = 0.f;  // row fully masked so far (never for valid rows)
    const float alpha = upd ? ex2_approx(m_ref - m_use) : 1.f;  // 0 on the first tile

    // p = 2^(s * scale_log2 - m_use): one packed FMA per pair, one MUFU
    // exp2 per element; four packed partial sums.  The packed bf16 pairs
    // are written back over the first 64 S columns (P in TMEM).
    const uint64_t neg_m = pack_f32x2(-m_use, -m_use);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
    uint32_t pk[2][32];
#pragma unroll
    for (int c = 0; c < BN; c += 2) {
        const uint64_t sv = pack_f32x2(__uint_as_float(r[c >> 5][c & 31]),
                                       __uint_as_float(r[c >> 5][(c & 31) + 1]));
        float a0, a1;
        unpack_f32x2(ffma2(sv, scale2, neg_m), a0, a1);
        const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
        acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], pack_f32x2(p0, p1));
        pk[c >> 6][(c >> 1) & 31] = pack_bf16x2(p0, p1);
    }
    if constexpr (PER_TILE) {
        if (rescale_o) {
            (void)bounded_wait(pv_bar, pv_parity, *ctl);
            tc_fence_after();
        }
    }
    tmem_st_32x32b_x32(tP + 0, pk[0]);
    tmem_st_32x32b_x32(tP + 32, pk[1]);
    float s0, s1, s2, s3, s4, s5, s6, s7;
    unpack_f32x2(acc[0], s0, s1);
    unpack_f32x2(acc[1], s2, s3);
    unpack_f32x2(acc[2], s4, s5);
    unpack_f32x2(acc[3], s6, s7);
    const float rs = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));

    if (rescale_o && __any_sync(0xffffffffu, upd)) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + c, o);
            tmem_wait_ld_x32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_32x32b_x32(tO + c, o);
        }
    }
    tmem_wait_st();
    tc_fence_before();
    return TileStep{alpha, rs, m_use};
}

template <int D>
__device__ __forceinline__ void softmax_warpgroup(
    int x, int t, int warp, uint32_t tmem, uint32_t sbase, int T, int row0, int N, int BH,
    int causal, float scale_log2, float *__restrict__ lse, int bh, const CUtensorMap *tmO,
    const WaitCtl &ctl, volatile uint32_t *abort_flag) {
    using C = Cfg<D>;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::TM_S1 : C::TM_S0);
    const uint32_t tP = tmem + lane_base + (x ? C::TM_P1 : C::TM_P0);
    const uint32_t tO = tmem + lane_base + (x ? C::TM_O1 : C::TM_O0);
    const uint32_t sStage = sbase + C::OFF_Q + x * C::Q_BYTES;  // Q_x, reused for O
    const int tile_row0 = row0 + x * BM;
    const int row = tile_row0 + t;
    const int limit = causal ? min(N, row + 1) : N;  // keys [0, limit) are visible
    const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
        ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_SFULL + x), j & 1, ctl));
        if (!ok) break;
        if constexpr (C::PER_TILE) {
            if (t == 0) {
                // S_x(j) is complete, and with it every MMA this tile's issuer
                // sent before it: S_x(j) read K_j, and O_x += P_x(j-2) V_{j-2}
                // came earlier.  Both tiles read every slot, so each slot
                // takes two releases.
                mbar_arrive(bar(C::B_EMPTY + (2 * j) % C::NSLOT));
                if (j >= 2) mbar_arrive(bar(C::B_EMPTY + (2 * j - 3) % C::NSLOT));
            }
            tc_fence_after();
            const TileStep st = softmax_tile<D, true>(
                tS, tP, tO, j * BN, limit, scale2, scale_log2, m_ref, j > 0, bar(C::B_SFREE + x),
                bar(C::B_PVDONE + x), (uint32_t)(j - 1) & 1u, &ctl);
            mbar_arrive(bar(C::B_PFULL + x));
            l_run = l_run * st.alpha + st.rs;
            m_ref = st.m_use;
            continue;
        }
        if (x == 1 && t == 0) {
            // S_B(j) is complete, and with it every MMA issued before it: S_A(j)
            // (the last reader of K_j) and O_B += P_B(j-1) V_{j-1} (the last
            // reader of V_{j-1}).  Hand both slots back to the producer here,
            // which keeps two commits per key tile off the MMA issuer.
            mbar_arrive(bar(C::B_EMPTY + (2 * j) % C::NSLOT));
            if (j >= 1) mbar_arrive(bar(C::B_EMPTY + (2 * j - 1) % C::NSLOT));
        }
        tc_fence_after();
        const TileStep st =
            softmax_tile<D>(tS, tS, tO, j * BN, limit, scale2, scale_log2, m_ref, j > 0);
        mbar_arrive(bar(C::B_PFULL + x));
        l_run = l_run * st.alpha + st.rs;
        m_ref = st.m_use;
    }
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_ODONE + x), 0, ctl));
    if (ok) {
        // Q_x is no longer read: its last S MMA completed before this tile's
        // last S was observed.  Stage O there in the O tensor map's swizzle.
        tc_fence_after();
        const float inv_l = 1.f / l_run;
#pragma unroll
        for (int c = 0; c < D; c += 64) {
            uint32_t o[2][32];
            tmem_ld_32x32b_x32(tO + c, o[0]);
            tmem_ld_32x32b_x32(tO + c + 32, o[1]);
            tmem_wait_ld_x32(o[0]);
            tmem_wait_ld_x32(o[1]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int dcol = c + i * 8;
                const uint32_t chunk = (uint32_t)(dcol & 63) >> 3;
                const uint32_t addr = sStage + (dcol >> 6) * (BM * 128) + t * 128 +
                                      ((chunk ^ ((uint32_t)t & 7u)) << 4);
                const uint32_t *v = &o[i >> 2][(i & 3) * 8];
                st_shared_v4(addr,
                             pack_bf16x2(__uint_as_float(v[0]) * inv_l,
                                         __uint_as_float(v[1]) * inv_l),
                             pack_bf16x2(__uint_as_float(v[2]) * inv_l,
                                         __uint_as_float(v[3]) * inv_l),
                             pack_bf16x2(__uint_as_float(v[4]) * inv_l,
                                         __uint_as_float(v[5]) * inv_l),
                             pack_bf16x2(__uint_as_float(v[6]) * inv_l,
                                         __uint_as_float(v[7]) * inv_l));
            }
        }
        if (lse != nullptr && row < N &&
            ATTN_IN_BOUNDS(bh >= 0 && bh < BH && row >= 0, ctl.status))
            lse[(size_t)bh * (size_t)N + (size_t)row] = (m_ref + log2f(l_run)) * LN2;
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + x, BM);
    if (t == 0 && *abort_flag == 0u && tile_row0 < N &&
        ATTN_IN_BOUNDS(bh >= 0 && bh < BH && tile_row0 >= 0, ctl.status)) {
        // The tensor map clips rows >= N, so a ragged last tile is safe.
        for (int c = 0; c < C::DBLK; ++c)
            tma_store_3d(tmO, sStage + c * (BM * 128), c * 64, tile_row0, bh);
        tma_store_commit();
        tma_store_wait_read();
    }
}

template <int D>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    attn_fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO, float *__restrict__ lse,
                            int N, int BH, int num_cta_tiles, float scale_log2, int causal,
                            uint32_t idesc_s, uint32_t *status, uint64_t timeout_ns, int num_sms,
                            int GH) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q;
    const uint32_t sKV = sbase + C::OFF_KV;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Items in launch order: batch*head fastest, heaviest causal tiles first.
    // Items in launch order: heads in groups of GH, one group after the other;
    // inside a group batch*head fastest, heaviest causal tiles first.
    auto decode = [&](int it, int &bh_, int &tile_) {
        const int per_group = GH * num_cta_tiles;
        const int g = it / per_group, rem = it - g * per_group;
        const int gh = min(GH, BH - g * GH);
        const int y = rem / gh;
        bh_ = g * GH + (rem - y * gh);
        tile_ = causal ? (num_cta_tiles - 1 - y) : y;
    };
    int bh, cta_tile;
    decode((int)blockIdx.x, bh, cta_tile);
    // The split-CTA launch that may follow reads nothing this kernel writes:
    // let it start on SMs this launch has finished with.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row0 = cta_tile * (2 * BM);
    int TA, TB;
    tile_counts(N, cta_tile, causal, TA, TB);

    const uint32_t sQ_ = sQ;
    auto load_q = [&](int x) {
        mbar_arrive_expect_tx(bar(C::B_Q + x), C::Q_BYTES);
        // Tile A starts inside the sequence; tile B may lie past its end (the
        // tensor map then fills zeros).
        if (ATTN_IN_BOUNDS(bh >= 0 && bh < BH && row0 >= 0 && row0 < N, status))
            for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(sQ_ + x * C::Q_BYTES + c * (BM * 128), &tmQ, c * 64, row0 + x * BM,
                            bh, bar(C::B_Q + x));
    };
    auto load_kv = [&](int n) {  // load n of the sequence K_0, V_0, K_1, ... into slot n % NSLOT
        const int s = n % C::NSLOT;
        mbar_arrive_expect_tx(bar(C::B_FULL + s), C::SLOT_BYTES);
        if (ATTN_IN_BOUNDS(bh >= 0 && bh < BH && n >= 0 && (n >> 1) * BN < N, status))
            for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(sKV + s * C::SLOT_BYTES + c * (BN * 128), (n & 1) ? &tmV : &tmK,
                            c * 64, (n >> 1) * BN, bh, bar(C::B_FULL + s));
    };
    if (warp == WARP_TMA && lane == 0) {
        // The producer sets up the barriers itself and starts the first copies
        // before the CTA-wide barrier, so they overlap the TMEM allocation:
        // Q_A and K_0 first (all S_A(0) needs), then Q_B and V_0.
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_Q + x), 1);
            mbar_init(bar(C::B_SFULL + x), 1);
            mbar_init(bar(C::B_PFULL + x), BM);
            mbar_init(bar(C::B_ODONE + x), 1);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), C::PER_TILE ? 2 : 1);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        if constexpr (C::PER_TILE) {
            for (int x = 0; x < 2; ++x) {
                mbar_init(bar(C::B_SFREE + x), 4);  // one arrival per softmax warp
                mbar_init(bar(C::B_PVDONE + x), 1);
            }
            mbar_init(bar(C::B_DRAIN_B), 1);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        load_q(0);
        load_kv(0);
        load_q(1);
        load_kv(1);
        // Warm L2 with the query block of the CTA that will most likely start
        // next on a free SM (blocks are dispatched in launch order, so that is
        // the one num_sms further on).
        const int next = (int)blockIdx.x + num_sms;
        if (next < (int)gridDim.x) {
            int nbh, ntile;
            decode(next, nbh, ntile);
            for (int x = 0; x < 2; ++x) {
                const int r = ntile * (2 * BM) + x * BM;
                if (r < N && ATTN_IN_BOUNDS(nbh >= 0 && nbh < BH, status))
                    for (int c = 0; c < C::DBLK; ++c) tma_prefetch_l2_3d(&tmQ, c * 64, r, nbh);
            }
        }
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
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            // Loads 0 and 1 (K_0, V_0) were issued before the CTA-wide barrier.
            int n = 2;
            for (; n < 2 * TB; ++n) {
                const int s = n % C::NSLOT;
                if (n >= C::NSLOT &&
                    !bounded_wait(bar(C::B_EMPTY + s), ((n / C::NSLOT) - 1) & 1, ctl))
                    break;
                load_kv(n);
            }
            // Let the copies issued last land before exiting (already complete
            // on the normal path).
            drain_wait(bar(C::B_Q + 0), 0, timeout_ns);
            drain_wait(bar(C::B_Q + 1), 0, timeout_ns);
            for (int i = (n > C::NSLOT ? n - C::NSLOT : 0); i < n; ++i)
                drain_wait(bar(C::B_FULL + i % C::NSLOT), (i / C::NSLOT) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == WARP_MMA || (C::PER_TILE && warp == WARP_MMA_B)) {
        // ----------------------------------------------------------- MMA ---
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, false, true);
            // Slot and phase of load n (K_j is load 2j, V_j is load 2j+1).
            auto slot_addr = [&](int n) -> uint32_t { return sKV + (n % C::NSLOT) * C::SLOT_BYTES; };
            auto wait_full = [&](int n) -> bool {
                return bounded_wait(bar(C::B_FULL + n % C::NSLOT), (n / C::NSLOT) & 1, ctl);
            };
            // Descriptor bases; each GEMM adds fixed per-step offsets inside
            // one asm block, so the issue loop does no descriptor arithmetic.
            const uint64_t qdesc[2] = {sdesc_sw128(sQ, 16, 1024),
                                       sdesc_sw128(sQ + C::Q_BYTES, 16, 1024)};
            auto issue_s = [&](int x, uint32_t sK) {
                const uint32_t dS = tmem + (x ? C::TM_S1 : C::TM_S0);
                if constexpr (D == 128)
                    gemm_ss_k8(dS, qdesc[x], sdesc_sw128(sK, 16, 1024), idesc_s, 0u);
                else
                    gemm_ss_k4(dS, qdesc[x], sdesc_sw128(sK, 16, 1024), idesc_s, 0u);
                mma_commit(bar(C::B_SFULL + x));
            };
            auto issue_pv = [&](int x, uint32_t sV, bool first) {
                // P: 16 keys of bf16 pairs = 8 TMEM columns per step.  V is
                // MN-major (d contiguous): 16 keys = 2 swizzle atoms of 8 rows
                // x 128 B; the two 64-column halves sit BN*128 B apart.
                gemm_ts_k8(tmem + (x ? C::TM_O1 : C::TM_O0), tmem + (x ? C::TM_S1 : C::TM_S0),
                           sdesc_sw128(sV, BN * 128, 1024), idesc_o, first ? 0u : 1u);
            };
            if constexpr (C::PER_TILE) {
                // One issuer per tile, each with its own S, P and O, so the two
                // never wait for each other.  Tile x's next S is issued as soon
                // as its softmax has read the current one:
                //   S_x(0), then per key tile j
                //   [S read] S_x(j+1), [P_x(j) written] O_x += P_x(j) V_j.
                const int x = warp - WARP_MMA;
                const int T = x ? TB : TA;
                const uint32_t tS = tmem + (x ? C::TM_S1 : C::TM_S0);
                const uint32_t tP = tmem + (x ? C::TM_P1 : C::TM_P0);
                const uint32_t tO = tmem + (x ? C::TM_O1 : C::TM_O0);
                auto issue_s1 = [&](int j) {
                    gemm_ss_k4(tS, qdesc[x], sdesc_sw128(slot_addr(2 * j), 16, 1024), idesc_s, 0u);
                    mma_commit(bar(C::B_SFULL + x));
                };
                bool ok = bounded_wait(bar(C::B_Q + x), 0, ctl) && wait_full(0);
                if (ok) issue_s1(0);
                for (int j = 0; ok && j < T; ++j) {
                    if (j + 1 < T) {
                        if (!(ok = bounded_wait(bar(C::B_SFREE + x), j & 1, ctl) &&
                                   wait_full(2 * j + 2)))
                            break;
                        tc_fence_after();
                        issue_s1(j + 1);
                    }
                    if (!(ok = bounded_wait(bar(C::B_PFULL + x), j & 1, ctl) &&
                               wait_full(2 * j + 1)))
                        break;
                    tc_fence_after();
                    gemm_ts_k8(tO, tP, sdesc_sw128(slot_addr(2 * j + 1), BN * 128, 1024), idesc_o,
                               j == 0 ? 0u : 1u);
                    mma_commit(bar(C::B_PVDONE + x));
                    if (j == T - 1) mma_commit(bar(C::B_ODONE + x));
                }
                // Every MMA this thread issued must finish before TMEM is released.
                const uint32_t drain = bar(x ? C::B_DRAIN_B : C::B_DRAIN);
                mma_commit(drain);
                drain_wait(drain, 0, timeout_ns);
            } else {
                // Two S buffers (d = 128), one issuer for both tiles.  Tile A's
                // P V product waits first for its V tile (long landed, off the
                // critical path) and then, spinning, for the softmax's P, so the
                // issuer goes from "P is ready" straight to the MMAs (+0.5-3 %
                // measured); tile B's product with the same V tile one GEMM
                // later only waits for its P.
                // Key tile 0, then the steady state with no run-time choices
                // (key tiles 1 .. T_A - 1: whole groups of NSLOT tiles with
                // constant ring positions, then the remainder), then tile B's
                // extra key tile (causal, T_B = T_A + 1) and its last product.
                bool ok = bounded_wait(bar(C::B_Q + 0), 0, ctl) && wait_full(0);
                if (ok) {
                    issue_s(0, slot_addr(0));
                    ok = bounded_wait(bar(C::B_Q + 1), 0, ctl);
                }
                if (ok) {
                    issue_s(1, slot_addr(0));
                    ok = wait_full(1) && spin_wait(bar(C::B_PFULL + 0), 0, ctl);
                }
                if (ok) {
                    tc_fence_after();
                    issue_pv(0, slot_addr(1), true);
                }
                // Steady state in groups of NSLOT key tiles: tile 1 + NSLOT g + i
                // loads K into slot (2 + 2 i) % NSLOT and V into the next one,
                // with phases that depend on i alone (2 NSLOT loads per group
                // are an even number of ring turns), so inside a group every
                // slot address and barrier phase is a constant.
                constexpr int NS = C::NSLOT;
                const int groups = (TA - 1) / NS;
                for (int g = 0; ok && g < groups; ++g) {
#pragma unroll
                    for (int i = 0; i < NS; ++i) {
                        const int j = 1 + NS * g + i;
                        const int sk = (2 + 2 * i) % NS, pk = ((2 + 2 * i) / NS) & 1;
                        const int sv = (3 + 2 * i) % NS, pv = ((3 + 2 * i) / NS) & 1;
                        const int sp = (1 + 2 * i) % NS;  // V_{j-1}
                        if (!(ok = bounded_wait(bar(C::B_FULL + sk), (uint32_t)pk, ctl))) break;
                        issue_s(0, sKV + (uint32_t)sk * C::SLOT_BYTES);
                        if (!(ok = spin_wait(bar(C::B_PFULL + 1), (j - 1) & 1, ctl))) break;
                        tc_fence_after();
                        issue_pv(1, sKV + (uint32_t)sp * C::SLOT_BYTES, j == 1);
                        issue_s(1, sKV + (uint32_t)sk * C::SLOT_BYTES);
                        if (!(ok = bounded_wait(bar(C::B_FULL + sv), (uint32_t)pv, ctl) &&
                                   spin_wait(bar(C::B_PFULL + 0), j & 1, ctl)))
                            break;
                        tc_fence_after();
                        issue_pv(0, sKV + (uint32_t)sv * C::SLOT_BYTES, false);
                    }
                }
                for (int j = 1 + NS * groups; ok && j < TA; ++j) {
                    const int nK = 2 * j;
                    if (!(ok = wait_full(nK))) break;
                    issue_s(0, slot_addr(nK));
                    // O_B += P_B(j-1) V_{j-1}; V_{j-1} was seen complete before
                    // O_A += P_A(j-1) V_{j-1}.
                    if (!(ok = spin_wait(bar(C::B_PFULL + 1), (j - 1) & 1, ctl))) break;
                    tc_fence_after();
                    issue_pv(1, slot_addr(nK - 1), j == 1);
                    issue_s(1, slot_addr(nK));
                    if (!(ok = wait_full(nK + 1) && spin_wait(bar(C::B_PFULL + 0), j & 1, ctl)))
                        break;
                    tc_fence_after();
                    issue_pv(0, slot_addr(nK + 1), false);
                }
                if (ok) mma_commit(bar(C::B_ODONE + 0));
                if (ok && TB > TA) {
                    // Tile B's key tile T_A (causal): O_B += P_B(T_A - 1) V, S_B(T_A).
                    const int nK = 2 * TA;
                    ok = wait_full(nK) && spin_wait(bar(C::B_PFULL + 1), (TA - 1) & 1, ctl);
                    if (ok) {
                        tc_fence_after();
                        issue_pv(1, slot_addr(nK - 1), TA == 1);
                        issue_s(1, slot_addr(nK));
                    }
                }
                if (ok) {
                    // V_{T_B-1} was seen before O_A's last product unless T_A < T_B.
                    const int j = TB - 1, nV = 2 * j + 1;
                    ok = (j < TA || wait_full(nV)) && spin_wait(bar(C::B_PFULL + 1), j & 1, ctl);
                    if (ok) {
                        tc_fence_after();
                        issue_pv(1, slot_addr(nV), j == 0);
                        mma_commit(bar(C::B_ODONE + 1));
                    }
                }
                // Every MMA issued above must finish before TMEM is released.
                mma_commit(bar(C::B_DRAIN));
                drain_wait(bar(C::B_DRAIN), 0, timeout_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax + epilogue ---
        const int x = warp >> 2;          // 0: tile A, 1: tile B
        const int t = threadIdx.x & 127;  // row within the tile == TMEM lane
        softmax_warpgroup<D>(x, t, warp, tmem, sbase, x ? TB : TA, row0, N, BH, causal,
                             scale_log2, lse, bh, &tmO, ctl, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------ split CTAs ---
//
// For the items of a last, partly filled wave (without the causal mask), or
// for every item of a grid that fills at most half the SMs, two CTAs share an
// item, one per 128-row half.  In such a CTA both query tiles hold the same
// rows (Q is loaded once, into Q_A): tile A walks the even key tiles and tile
// B the odd ones.  At d = 128 one issuer runs S_A(j), O_B += P_B(j-1) V,
// S_B(j), O_A += P_A(j) V, so the tensor core works on one tile while the
// other's softmax runs; at d = 64 each tile has its own issuer, S apart from
// P, as in the main kernel.  At the end the two partial
// results (m, l, O) of each row are merged with the online rule.  Every step
// streams two K and two V tiles, so the ring gets one more slot: the unused
// Q_B buffer.

// Ring entries of step j: tile x takes key tile 2j + x, whose K is entry
// 2(2j + x) and V the next one.
__device__ __forceinline__ int split_entry_k(int x, int j) { return 4 * j + 2 * x; }

template <int D>
__device__ __forceinline__ uint32_t split_slot_addr(uint32_t sbase, int n) {
    using C = Cfg<D>;
    const int s = n % (C::NSLOT + 1);
    return s < C::NSLOT ? sbase + C::OFF_KV + (uint32_t)s * C::SLOT_BYTES
                        : sbase + C::OFF_Q + C::Q_BYTES;
}

template <int D>
__device__ __forceinline__ void split_softmax(int x, int t, int warp, uint32_t tmem, uint32_t sbase,
                                              float *xch, int T, int TB, int row0, int N,
                                              int BH, int causal, float scale_log2,
                                              float *__restrict__ lse, int bh,
                                              const CUtensorMap *tmO, const WaitCtl &ctl,
                                              volatile uint32_t *abort_flag) {
    using C = Cfg<D>;
    constexpr int NS = C::NSLOT + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::TM_S1 : C::TM_S0);
    const uint32_t tP = tmem + lane_base + (x ? C::TM_P1 : C::TM_P0);
    const uint32_t tO = tmem + lane_base + (x ? C::TM_O1 : C::TM_O0);
    const int row = row0 + t;
    const int limit = causal ? min(N, row + 1) : N;
    const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
        ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_SFULL + x), j & 1, ctl));
        if (!ok) break;
        const int e = split_entry_k(x, j);
        if constexpr (C::PER_TILE) {
            // One issuer per tile: S_x(j) complete frees its own K tile; the V
            // tile read in the previous step is free once the softmax has seen
            // O_x += P_x(j-1) V complete (inside softmax_tile, before P is
            // overwritten).
            if (t == 0) mbar_arrive(bar(C::B_EMPTY + e % NS));
            tc_fence_after();
            const TileStep st = softmax_tile<D, true>(
                tS, tP, tO, (2 * j + x) * BN, limit, scale2, scale_log2, m_ref, j > 0,
                bar(C::B_SFREE + x), bar(C::B_PVDONE + x), (uint32_t)(j - 1) & 1u, &ctl);
            if (t == 0 && j >= 1) mbar_arrive(bar(C::B_EMPTY + (e - 3) % NS));
            mbar_arrive(bar(C::B_PFULL + x));
            l_run = l_run * st.alpha + st.rs;
            m_ref = st.m_use;
            continue;
        }
        if (t == 0) {
            // S_x(j) is complete, and with it every MMA issued before it: its
            // own K tile is free, and so is the V tile this tile read in the
            // previous step (O_x += P_x(j-1) V was issued before S_x(j)).
            mbar_arrive(bar(C::B_EMPTY + e % NS));
            if (j >= 1) mbar_arrive(bar(C::B_EMPTY + (e - 3) % NS));
        }
        tc_fence_after();
        const TileStep st =
            softmax_tile<D>(tS, tS, tO, (2 * j + x) * BN, limit, scale2, scale_log2, m_ref, j > 0);
        mbar_arrive(bar(C::B_PFULL + x));
        l_run = l_run * st.alpha + st.rs;
        m_ref = st.m_use;
    }
    // Merge.  The exchange area is a ring slot (Q_B), which the other tile's
    // last O += P V may still be reading: both tiles wait until every MMA of
    // the CTA is done (tile B has none when the rows see only one key tile).
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_ODONE + 0), 0, ctl));
    if (ok && TB > 0) ok = __all_sync(0xffffffffu, bounded_wait(bar(C::B_ODONE + 1), 0, ctl));
    xch[(2 * x) * BM + t] = T > 0 ? m_ref : -INFINITY;
    xch[(2 * x + 1) * BM + t] = l_run;
    named_bar_sync(3, 2 * BM);
    const float mA = xch[t], lA = xch[BM + t], mB = xch[2 * BM + t], lB = xch[3 * BM + t];
    const float m = fmaxf(mA, mB);
    const float a = ex2_approx(mA - m);
    const float b = TB > 0 ? ex2_approx(mB - m) : 0.f;
    const float l = a * lA + b * lB;
    if (ok) {
        tc_fence_after();
        const float ia = a / l, ib = b / l;
        const uint32_t sOut = sbase + C::OFF_Q;  // Q_A: no MMA reads it any more
        const uint32_t tOA = tmem + lane_base + C::TM_O0, tOB = tmem + lane_base + C::TM_O1;
        // Tile A's threads merge columns [0, D/2), tile B's [D/2, D).
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            const int c = x * (D / 2) + c0;
            uint32_t oa[32], ob[32];
            tmem_ld_32x32b_x32(tOA + c, oa);
            tmem_wait_ld_x32(oa);
            if (TB > 0) {
                tmem_ld_32x32b_x32(tOB + c, ob);
                tmem_wait_ld_x32(ob);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) ob[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int dcol = c + i * 8;
                const uint32_t chunk = (uint32_t)(dcol & 63) >> 3;
                const uint32_t addr = sOut + (dcol >> 6) * (BM * 128) + t * 128 +
                                      ((chunk ^ ((uint32_t)t & 7u)) << 4);
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = __uint_as_float(oa[i * 8 + e]) * ia + __uint_as_float(ob[i * 8 + e]) * ib;
                st_shared_v4(addr, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                             pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            }
        }
        if (x == 0 && lse != nullptr && row < N &&
            ATTN_IN_BOUNDS(bh >= 0 && bh < BH && row >= 0, ctl.status))
            lse[(size_t)bh * (size_t)N + (size_t)row] = (m + log2f(l)) * LN2;
    }
    fence_proxy_async_smem();
    named_bar_sync(3, 2 * BM);
    if (x == 0 && t == 0 && ok && *abort_flag == 0u &&
        ATTN_IN_BOUNDS(bh >= 0 && bh < BH && row0 >= 0 && row0 < N, ctl.status)) {
        for (int c = 0; c < C::DBLK; ++c)
            tma_store_3d(tmO, sbase + C::OFF_Q + c * (BM * 128), c * 64, row0, bh);
        tma_store_commit();
        tma_store_wait_read();
    }
}

template <int D>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    attn_fwd_bf16_tc_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                                  const __grid_constant__ CUtensorMap tmK,
                                  const __grid_constant__ CUtensorMap tmV,
                                  const __grid_constant__ CUtensorMap tmO,
                                  float *__restrict__ lse, int N, int BH, int num_cta_tiles,
                                  int first_item, float scale_log2, int causal, uint32_t idesc_s,
                                  uint32_t *status, uint64_t timeout_ns) {
    using C = Cfg<D>;
    constexpr int NS = C::NSLOT + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_ABORT);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA 2i + h takes the 128-row half h of item first_item + i.
    const int item = first_item + (int)(blockIdx.x >> 1);
    const int bh = item % BH;
    const int rank = item / BH;
    const int cta_tile = causal ? (num_cta_tiles - 1 - rank) : rank;
    const int row0 = cta_tile * (2 * BM) + (int)(blockIdx.x & 1) * BM;
    if (row0 >= N) return;  // rows past N: nothing to do (uniform, before any setup)
    const int nkv = (N + BN - 1) / BN;
    const int KT = causal ? min(row0 / BM + 1, nkv) : nkv;  // key tiles these rows see
    const int TA = (KT + 1) >> 1, TB = KT >> 1;              // even / odd key tiles

    auto load_kv = [&](int n) {  // entry n: K (even n) or V (odd n) of key tile n / 2
        const int s = n % NS;
        mbar_arrive_expect_tx(bar(C::B_FULL + s), C::SLOT_BYTES);
        const uint32_t dst = split_slot_addr<D>(sbase, n);
        if (ATTN_IN_BOUNDS(bh >= 0 && bh < BH && n >= 0 && (n >> 1) * BN < N, status))
            for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(dst + c * (BN * 128), (n & 1) ? &tmV : &tmK, c * 64, (n >> 1) * BN,
                            bh, bar(C::B_FULL + s));
    };
    if (warp == WARP_TMA && lane == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_Q + x), 1);
            mbar_init(bar(C::B_SFULL + x), 1);
            mbar_init(bar(C::B_PFULL + x), BM);
            mbar_init(bar(C::B_ODONE + x), 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        if constexpr (C::PER_TILE) {
            for (int x = 0; x < 2; ++x) {
                mbar_init(bar(C::B_SFREE + x), 4);  // one arrival per softmax warp
                mbar_init(bar(C::B_PVDONE + x), 1);
            }
            mbar_init(bar(C::B_DRAIN_B), 1);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        mbar_arrive_expect_tx(bar(C::B_Q), C::Q_BYTES);
        if (ATTN_IN_BOUNDS(rank >= 0 && rank < num_cta_tiles && bh >= 0 && bh < BH, status))
            for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(sQ + c * (BM * 128), &tmQ, c * 64, row0, bh, bar(C::B_Q));
        load_kv(0);
        load_kv(1);
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
            const int n_loads = 2 * KT;
            int n = 2;
            for (; n < n_loads; ++n) {
                const int s = n % NS;
                if (n >= NS && !bounded_wait(bar(C::B_EMPTY + s), ((n / NS) - 1) & 1, ctl)) break;
                load_kv(n);
            }
            drain_wait(bar(C::B_Q), 0, timeout_ns);
            for (int i = (n > NS ? n - NS : 0); i < n; ++i)
                drain_wait(bar(C::B_FULL + i % NS), (i / NS) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == WARP_MMA || (C::PER_TILE && warp == WARP_MMA_B)) {
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, false, true);
            auto wait_full = [&](int n) -> bool {
                return bounded_wait(bar(C::B_FULL + n % NS), (n / NS) & 1, ctl);
            };
            const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);  // both tiles read Q_A
            if constexpr (C::PER_TILE) {
                // d = 64: one issuer per tile, as in the main kernel (the two
                // tiles read different key tiles, so they share nothing but Q).
                const int x = warp - WARP_MMA;
                const int T = x ? TB : TA;
                const uint32_t tS = tmem + (x ? C::TM_S1 : C::TM_S0);
                const uint32_t tP = tmem + (x ? C::TM_P1 : C::TM_P0);
                const uint32_t tO = tmem + (x ? C::TM_O1 : C::TM_O0);
                auto issue_s1 = [&](int j) {
                    const uint64_t kd =
                        sdesc_sw128(split_slot_addr<D>(sbase, split_entry_k(x, j)), 16, 1024);
                    gemm_ss_k4(tS, qdesc, kd, idesc_s, 0u);
                    mma_commit(bar(C::B_SFULL + x));
                };
                bool ok = T > 0 && bounded_wait(bar(C::B_Q), 0, ctl) &&
                          wait_full(split_entry_k(x, 0));
                if (ok) issue_s1(0);
                for (int j = 0; ok && j < T; ++j) {
                    if (j + 1 < T) {
                        if (!(ok = bounded_wait(bar(C::B_SFREE + x), j & 1, ctl) &&
                                   wait_full(split_entry_k(x, j + 1))))
                            break;
                        tc_fence_after();
                        issue_s1(j + 1);
                    }
                    const int nV = split_entry_k(x, j) + 1;
                    if (!(ok = bounded_wait(bar(C::B_PFULL + x), j & 1, ctl) && wait_full(nV)))
                        break;
                    tc_fence_after();
                    gemm_ts_k8(tO, tP, sdesc_sw128(split_slot_addr<D>(sbase, nV), BN * 128, 1024),
                               idesc_o, j == 0 ? 0u : 1u);
                    mma_commit(bar(C::B_PVDONE + x));
                    if (j == T - 1) mma_commit(bar(C::B_ODONE + x));
                }
                const uint32_t drain = bar(x ? C::B_DRAIN_B : C::B_DRAIN);
                mma_commit(drain);
                drain_wait(drain, 0, timeout_ns);
            } else {
                // d = 128: one issuer for both tiles.
                auto issue_s = [&](int x, int n) {
                    const uint32_t dS = tmem + (x ? C::TM_S1 : C::TM_S0);
                    const uint64_t kd = sdesc_sw128(split_slot_addr<D>(sbase, n), 16, 1024);
                    if constexpr (D == 128)
                        gemm_ss_k8(dS, qdesc, kd, idesc_s, 0u);
                    else
                        gemm_ss_k4(dS, qdesc, kd, idesc_s, 0u);
                    mma_commit(bar(C::B_SFULL + x));
                };
                auto issue_pv = [&](int x, int n, bool first) {
                    gemm_ts_k8(tmem + (x ? C::TM_O1 : C::TM_O0), tmem + (x ? C::TM_S1 : C::TM_S0),
                               sdesc_sw128(split_slot_addr<D>(sbase, n), BN * 128, 1024), idesc_o,
                               first ? 0u : 1u);
                };
                bool ok = bounded_wait(bar(C::B_Q), 0, ctl);
                for (int j = 0; ok && j < TA; ++j) {  // TA >= TB
                    const int nKA = split_entry_k(0, j), nKB = split_entry_k(1, j);
                    if (!(ok = wait_full(nKA))) break;
                    issue_s(0, nKA);
                    if (j >= 1) {
                        // O_B += P_B(j-1) V (key tile 2j - 1).
                        const int nV = split_entry_k(1, j - 1) + 1;
                        if (!(ok = bounded_wait(bar(C::B_PFULL + 1), (j - 1) & 1, ctl) &&
                                   wait_full(nV)))
                            break;
                        tc_fence_after();
                        issue_pv(1, nV, j == 1);
                        if (j - 1 == TB - 1) mma_commit(bar(C::B_ODONE + 1));
                    }
                    if (j < TB) {
                        if (!(ok = wait_full(nKB))) break;
                        issue_s(1, nKB);
                    }
                    const int nV = nKA + 1;
                    if (!(ok = bounded_wait(bar(C::B_PFULL + 0), j & 1, ctl) && wait_full(nV))) break;
                    tc_fence_after();
                    issue_pv(0, nV, j == 0);
                    if (j == TA - 1) mma_commit(bar(C::B_ODONE + 0));
                }
                if (ok && TB >= 1 && TA == TB) {
                    const int j = TB - 1, nV = split_entry_k(1, j) + 1;
                    ok = bounded_wait(bar(C::B_PFULL + 1), j & 1, ctl) && wait_full(nV);
                    if (ok) {
                        tc_fence_after();
                        issue_pv(1, nV, j == 0);
                        mma_commit(bar(C::B_ODONE + 1));
                    }
                }
                mma_commit(bar(C::B_DRAIN));
                drain_wait(bar(C::B_DRAIN), 0, timeout_ns);
            }
        }
        __syncwarp();
    } else {
        const int x = warp >> 2;
        const int t = threadIdx.x & 127;
        // The merge exchanges (m, l) through the start of Q_B, which no MMA
        // reads by then.
        split_softmax<D>(x, t, warp, tmem, sbase,
                         reinterpret_cast<float *>(smem + C::OFF_Q + C::Q_BYTES), x ? TB : TA, TB,
                         row0, N, BH, causal, scale_log2, lse, bh, &tmO, ctl, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // This launch may start before the main kernel of the same call has
    // finished; it completes only after it, so later work on the stream sees
    // every output row.  (Returns at once without a preceding main kernel.)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
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

}  // namespace tc

// [BH, N, d] bf16 tensor as a 3-D map with 64-column x 128-row boxes, 128-byte
// swizzle; rows beyond N read as zero and are clipped on store.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t BH, int64_t N, int d) {
    using tc::EncodeTiledFn;
    EncodeTiledFn enc = tc::get_encode_fn();
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

namespace tc {

template <int D>
static attn_status launch(const void *q, const void *k, const void *v, void *o, float *lse,
                          int64_t BH, int64_t N, float scale, bool causal, const LaunchCtx &ctx) {
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_bf16(&tq, q, BH, N, D) || !make_tmap_bf16(&tk, k, BH, N, D) ||
        !make_tmap_bf16(&tv, v, BH, N, D) || !make_tmap_bf16(&to, o, BH, N, D))
        return ATTN_ERR_CUDA;
    if (check_launch(cudaFuncSetAttribute(attn_fwd_bf16_tc_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)C::SMEM_BYTES),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    if (check_launch(cudaFuncSetAttribute(attn_fwd_bf16_tc_split_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)C::SMEM_BYTES),
                     ATTN_ERR_CUDA) != ATTN_OK)
        return ATTN_ERR_CUDA;
    const int num_cta_tiles = (int)((N + 2 * BM - 1) / (2 * BM));
    const int64_t n_items = BH * num_cta_tiles;
    // Items taken by two split CTAs (one per 128-row half): all of them when
    // they fill at most half the SMs; without the causal mask, also the items
    // that would otherwise run in a last wave filling at most half the SMs.
    // Those go to a second launch, after whole waves of the main kernel.
    // (With the mask the last items are the lightest: no split.)
    const int64_t sms = ctx.sm_count > 0 ? ctx.sm_count : 1;
    int64_t n_split = 0;
    if (2 * n_items <= sms) {
        n_split = n_items;
    } else if (!causal) {
        const int64_t rem = n_items % sms;
        if (rem > 0 && 2 * rem <= sms) n_split = rem;
    }
    const int64_t n_main = n_items - n_split;
    // Heads per group: the K and V of one group fit in half of L2, so the
    // CTAs that run together re-read K and V from L2 rather than HBM.  With
    // split CTAs (which take the last items in batch*head-fastest order) the
    // order stays ungrouped.
    const int64_t kv_head = 4 * N * (int64_t)D;
    int64_t gh64 = (64ll << 20) / (kv_head > 0 ? kv_head : 1);
    if (gh64 < 1) gh64 = 1;
    if (gh64 > BH || n_split > 0) gh64 = BH;
    const int gh = (int)gh64;
    // The softmax takes each row's maximum of the raw logits and multiplies it
    // by scale_log2, which is the maximum of the scaled logits only for a
    // positive multiplier.  A negative scale is therefore folded into the
    // product: the S MMA negates its A operand (instruction-descriptor bit 13),
    // giving exactly -(Q K^T) (a sign flip of bf16 operands rounds like the
    // original), and the kernel runs with |scale|.  A zero scale runs as the
    // smallest normal float: masked logits (-inf) then still scale to -inf
    // instead of -inf * 0 = NaN, and every visible scaled logit is below
    // 2^-100 in magnitude, so each weight rounds to exp2(0) = 1 as with 0.
    const bool negate_qk = scale < 0.f;
    const float abs_scale = fmaxf(fabsf(scale), 1.17549435e-38f);
    const uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false) | (negate_qk ? (1u << 13) : 0u);
    const float scale_log2 = abs_scale * 1.44269504088896340736f;
    if (n_main > 0) {
        attn_fwd_bf16_tc_kernel<D><<<(unsigned)n_main, C::THREADS, C::SMEM_BYTES, ctx.stream>>>(
            tq, tk, tv, to, lse, (int)N, (int)BH, num_cta_tiles, scale_log2, causal ? 1 : 0,
            idesc_s, ctx.status, ctx.timeout_ns, ctx.sm_count, gh);
        const attn_status st = check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
        if (st != ATTN_OK) return st;
    }
    if (n_split > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(2 * n_split));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = ctx.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = n_main > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return check_launch(cudaLaunchKernelEx(&cfg, attn_fwd_bf16_tc_split_kernel<D>, tq, tk, tv,
                                               to, lse, (int)N, (int)BH, num_cta_tiles,
                                               (int)n_main, scale_log2, causal ? 1 : 0,
                                               idesc_s, ctx.status, ctx.timeout_ns),
                            ATTN_ERR_LAUNCH);
    }
    return ATTN_OK;
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
    return check_launch(cudaGetLastError(), ATTN_ERR_LAUNCH);
}

}  // namespace attn
