// Grouped MXFP8 GEMM on a CTA pair (tcgen05 cta_group::2), sm_103a.
//
// Same contract as the 1-SM kernel in gemm.cu ([TE-JAX] "Optimization 1:
// Grouped GEMM": one launch for every expert, each over its own rows, MXFP8
// block scaling), with the tile split over two SMs of a cluster:
//
//   pair tile = 256 rows x 256 columns; CTA r of the pair holds A rows
//   [128 r, 128 r + 128) of the tile and B rows [128 r, 128 r + 128) (half of
//   N) in its own shared memory, and the scales of its A rows and of all 256
//   B rows.  The leader CTA (rank 0) issues tcgen05.mma.cta_group::2 with
//   M = 256, N = 256: each SM's tensor core multiplies its own A rows by the
//   whole B, reading the peer's B half over the cluster.  Per SM and k-step
//   this moves 32 KB through the TMA and 32 KB of operand reads instead of
//   48 + 48 KB for a 128 x 256 tile on one SM, which is what bounds the 1-SM
//   mainloop.
//
// Synchronisation (all waits bounded, as in gemm.cu):
//   full[s]   in the leader: both CTAs' TMA loads (cta_group::2 form, which
//             lets a load complete on the peer CTA's barrier) count their
//             bytes on it, so the leader's MMA starts once both halves are in
//             shared memory.  Scale atoms come through small TMA tensor maps
//             (rows of 256 bytes) for the same reason.
//   empty[s]  tcgen05.commit multicast from the leader to both CTAs.
//   tfull     tcgen05.commit multicast: the accumulator halves are ready.
//   tempty    in the leader, count 2 x 8 epilogue warps (the follower's
//             warps arrive remotely).
// A group's rows are 128-aligned, so a 256-row pair tile may have only its
// first half inside the group; the second CTA then multiplies duplicate rows
// and discards them (its stores are skipped).

#include "gemm_common.cuh"

namespace moe {
namespace gg {
namespace sm2 {

// Pair-tile configurations: N = 256 (one accumulator per CTA), N = 128 or
// N = 224 (two accumulators per CTA, so the epilogue of one tile overlaps
// the mainloop of the next).  Each CTA loads BN/2 rows of B.  Two 256-column
// accumulators would fill all 512 TMEM columns and leave none for the block
// scales; two of 224 columns leave 64, room for five stages of scales (A: 4
// columns, B: 8).  N = 224 serves the weight gradients (MOE_GEMM_WGRAD),
// whose short contractions (one group's rows) otherwise leave the tensor
// pipe idle while the single accumulator is drained; its B scales come in
// the tile-224 layout (two atoms per 224 rows, include/moe.h), since 224-row
// tiles do not start on the 128-row atoms of the plain layout.
// NVF4: NVFP4 operands (packed E2M1, UE4M3 scales per 16, kind::mxf4nvf4):
// four scale atoms per 128 rows and k-step instead of one, plain epilogues
// only (no TMA-store staging).
template <int BN_, bool NVF4 = false>
struct C2 {
    static constexpr int BN = BN_;
    static constexpr int BH = BN_ / 2;                  // B rows per CTA
    static constexpr int NACC = BN_ == 256 ? 1 : 2;
    static constexpr int STAGES = BN_ == 128 ? 8 : (BN_ == 224 || NVF4 || kEpiBoxCols == 64 ? 5 : 6);
    static constexpr int A_STAGE = BM * BK;             // this CTA's 128 A rows
    static constexpr int B_STAGE = BH * BK;             // this CTA's half of B
    static constexpr int SFA_BYTES = NVF4 ? 2048 : 512;
    static constexpr int SFB_BYTES = ((BN_ + 127) / 128) * SFA_BYTES;   // scales of all BN B rows
    static constexpr uint32_t STAGE_TX = A_STAGE + B_STAGE + SFA_BYTES + SFB_BYTES;
    static constexpr uint32_t SF0 = NACC * BN_;         // TMEM: accumulators, then scales
    static constexpr uint32_t SF_COLS = NVF4 ? 16 + 16 * (BN_ / 128) : (BN_ == 224 ? 12 : TMEM_SF_STRIDE);
    // TMA-store staging of the epilogue: one box per epilogue warp (N = 256),
    // two that alternate and one box of zeros for the tiles of empty groups
    // (N = 224, whose smaller stages leave the room)
    static constexpr int EPI_BYTES =
        (BN_ >= 224 && !NVF4) ? EPI_WARPS * kEpiBoxBytes * (BN_ == 224 ? 2 : 1) + (BN_ == 224 ? kEpiBoxBytes : 0) : 0;
    static constexpr int OFF_ZERO_IN_EPI = EPI_WARPS * kEpiBoxBytes * (BN_ == 224 ? 2 : 1);
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE;       // 1024-byte aligned
    static constexpr int OFF_SFA = OFF_EPI + EPI_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;  // full[S], empty[S], tfull[A], tempty[A], drain
    static constexpr int NBAR = 2 * STAGES + 2 * NACC + 1;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
    static constexpr int OFF_GOFS = OFF_MISC + 16;
    static constexpr int OFF_PT = OFF_GOFS + (MAX_G + 1) * 4;
    static constexpr int SMEM_BYTES = OFF_PT + (MAX_G + 1) * 4 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(SF0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(OFF_EPI % 1024 == 0, "swizzled staging alignment");
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of `addr` (a shared::cta address) in CTA `rank`
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Bounded wait whose arrivals may come from the peer CTA.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const Params& p,
                                                  volatile int* abort_flag) {
    uint64_t start = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (start == 0) {
                start = now;
            } else if (now - start > p.timeout_ns || it >= kMaxSpin) {
                set_err(p.err, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// TMA loads into this CTA's shared memory whose completion is counted on a
// barrier that may live in the peer CTA (cta_group::2 form).
__device__ __forceinline__ void tma2_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma2_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                             uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_cp_sf2(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tc_mma2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// arrive on the barrier at the same shared offset in both CTAs of the pair
// once every tcgen05 op issued so far by this thread has completed
__device__ __forceinline__ void tc_commit_both(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(bar),
                 "h"(mask)
                 : "memory");
}
__device__ __forceinline__ void tc_commit_local2(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma2_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// M = 256, N = BN, E2M1 A and B, UE4M3 scales (scale_vec::4X, ids 0)
template <int BN>
__device__ __forceinline__ uint32_t make_idesc2_nvf4() {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}
// M = 256 (two CTAs x 128 rows), N = BN
template <int BN>
__device__ __forceinline__ uint32_t make_idesc2(uint32_t sf_id) {
    return (sf_id << 4) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) | ((uint32_t)(256 >> 4) << 24) | (sf_id << 29);
}

struct Tile2 {
    int g;
    int64_t a_row;      // first A row this CTA loads
    int b_row_pair;     // first of the BN B rows of the pair tile
    int64_t kbeg;
    int nk;
    int64_t out_row;    // first output row of this CTA
    bool valid;         // this CTA's rows belong to the tile's group
    int nt;
};

template <int BN>
__device__ __forceinline__ void get_tile2(const Params& p, const int* s_gofs, const int* s_pt, int64_t total_pm,
                                          int64_t t, uint32_t rank, Tile2& ti) {
    int64_t pm;
    int nt;
    if (p.mode != MOE_GEMM_WGRAD) {
        band_decode(t, total_pm, p.n_tiles, p.band, pm, nt);
        const int g = find_group(s_pt, p.G, pm);
        const int64_t base = (int64_t)s_gofs[g] + 256 * (pm - s_pt[g]);
        const int64_t mine = base + 128 * rank;
        ti.g = g;
        ti.valid = mine < (int64_t)s_gofs[g + 1];
        ti.a_row = ti.valid ? mine : base;
        ti.out_row = mine;
        ti.kbeg = 0;
        ti.nk = (int)(p.K / BK);
    } else {
        // WGRAD: the tiles of group g (or of the gi-th group that passes
        // the row filter, listed in s_pt) are [gi * tpg, (gi + 1) * tpg)
        const int64_t mp = p.M / 256;
        const int64_t tpg = mp * p.n_tiles;
        const int gi = (int)(t / tpg);
        const int g = p.wg_filter ? s_pt[gi] : gi;
        band_decode(t - (int64_t)gi * tpg, mp, p.n_tiles, p.band, pm, nt);
        ti.g = g;
        ti.valid = true;
        ti.a_row = pm * 256 + 128 * rank;
        ti.out_row = (int64_t)g * p.M + ti.a_row;
        ti.kbeg = s_gofs[g] / BK;
        ti.nk = (s_gofs[g + 1] - s_gofs[g]) / BK;
    }
    ti.b_row_pair = nt * BN;
    ti.nt = nt;
}

template <int BN, int EPI, bool NVF4 = false>
__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_gemm_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                       const __grid_constant__ CUtensorMap tmD, const Params p) {
    using C = C2<BN, NVF4>;
    static_assert(!NVF4 || (BN == 256 && (EPI == MOE_EPI_NONE || EPI == MOE_EPI_NONE_F32)), "NVFP4 pair instances");
    static_assert(BN != 224 || (EPI == MOE_EPI_NONE && !NVF4), "224-wide pair tiles: weight gradients, bf16 out");
    constexpr int STAGES = C::STAGES, NACC = C::NACC, BH = C::BH;
    constexpr int OFF_A = C::OFF_A, OFF_B = C::OFF_B, OFF_SFA = C::OFF_SFA, OFF_SFB = C::OFF_SFB;
    constexpr int OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC, OFF_GOFS = C::OFF_GOFS, OFF_PT = C::OFF_PT;
    constexpr int A_STAGE = C::A_STAGE, B_STAGE = C::B_STAGE, SFA_BYTES = C::SFA_BYTES, SFB_BYTES = C::SFB_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + NACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * NACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
    int* s_gofs = reinterpret_cast<int*>(smem + OFF_GOFS);
    int* s_pt = reinterpret_cast<int*>(smem + OFF_PT);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort_flag = 0;
        *bad_flag = 0;
    }
    for (int i = threadIdx.x; i <= p.G; i += THREADS) s_gofs[i] = p.gofs[i];
    const uint32_t zbox = smem_u32(smem + C::OFF_EPI + C::OFF_ZERO_IN_EPI);   // the box of zeros
    if constexpr (BN == 224) {
        if (threadIdx.x < kEpiBoxBytes / 16) st_shared_v4(zbox + 16u * threadIdx.x, 0u, 0u, 0u, 0u);
        fence_proxy_async_shared();      // visible to the TMA stores that read it
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // offsets: start at 0, monotone, 128-aligned, inside the buffer
        bool ok = s_gofs[0] == 0;
        for (int g = 0; g < p.G && ok; ++g) ok = s_gofs[g + 1] >= s_gofs[g] && (s_gofs[g + 1] % BM) == 0;
        const int64_t limit = p.mode == MOE_GEMM_WGRAD ? p.K : p.M;
        ok = ok && (int64_t)s_gofs[p.G] <= limit;
        if (!ok) {
            *bad_flag = 1;
            if (blockIdx.x == 0) set_err(p.err, MOE_ERR_BAD_OFFSETS);
        }
        if (p.mode != MOE_GEMM_WGRAD) {
            // pair tiles per group: ceil(rows / 256)
            int acc = 0;
            for (int g = 0; g < p.G; ++g) {
                s_pt[g] = acc;
                acc += ok ? (s_gofs[g + 1] - s_gofs[g] + 255) / 256 : 0;
            }
            s_pt[p.G] = acc;
        } else if (p.wg_filter) {
            // the groups whose row count passes the filter, in order; their
            // number at s_pt[G]
            int n = 0;
            for (int g = 0; g < p.G && ok; ++g) {
                const int r = s_gofs[g + 1] - s_gofs[g];
                const bool in = p.wg_hi == 0 ? r >= p.wg_lo
                                             : (p.wg_lo < p.wg_hi ? (r >= p.wg_lo && r < p.wg_hi)
                                                                  : (r < p.wg_hi || r >= p.wg_lo));
                if (in) s_pt[n++] = g;
            }
            s_pt[p.G] = n;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the peer's barriers are initialised and TMEM is allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const bool bad = *bad_flag != 0;
    const int64_t total_pm = p.mode == MOE_GEMM_WGRAD ? 0 : (int64_t)s_pt[p.G];
    const int64_t wg_groups = p.mode == MOE_GEMM_WGRAD ? (p.wg_filter ? (int64_t)s_pt[p.G] : (int64_t)p.G) : 0;
    const int64_t total = bad ? 0
                              : (p.mode == MOE_GEMM_WGRAD ? wg_groups * (p.M / 256) * p.n_tiles
                                                          : total_pm * p.n_tiles);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer ----
        uint32_t leader_full[STAGES];
        for (int s = 0; s < STAGES; ++s) leader_full[s] = mapa(full_bar(s), 0);
        int pend[STAGES];
        for (int s = 0; s < STAGES; ++s) pend[s] = -1;
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        for (int64_t t = pair; t < total && !aborted; t += npairs) {
            Tile2 ti;
            get_tile2<BN>(p, s_gofs, s_pt, total_pm, t, rank, ti);
            const int gB = p.mode == MOE_GEMM_WGRAD ? 0 : ti.g;
            for (int ks = 0; ks < ti.nk; ++ks) {
                // freed by the leader's MMA completion (commit multicast)
                if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, p, abort_flag)) {
                    aborted = true;
                    break;
                }
                const int64_t kg = ti.kbeg + ks;
                const int kx = (int)(kg * BK);
                // both CTAs' bytes complete on the leader's full barrier
                const uint32_t fb = leader_full[stage];
                if (leader) mbar_expect_tx(full_bar(stage), 2 * C::STAGE_TX);
                tma2_load_2d(smem_u32(smem + OFF_A + stage * A_STAGE), &tmA, kx, (int)ti.a_row, fb);
                tma2_load_3d(smem_u32(smem + OFF_B + stage * B_STAGE), &tmB, kx, ti.b_row_pair + BH * (int)rank, gB,
                             fb);
                // scale atoms as rows of 256 bytes: atom i = rows 2i, 2i+1; the
                // two B atoms of the pair tile are adjacent in every layout
                // (NVFP4: a k-step's four atoms of a 128-row tile are 2 KB in
                // a row, the pair tile's two row tiles 4 KB)
                const int64_t sfa_row = (kg * p.a_sf_kstride + (ti.a_row / 128) * SFA_BYTES) / 256;
                // (tile-224 layout: the tile's two atoms at nt * 1024 of the k-step)
                const int64_t sfb_tile = BN == 224 ? (int64_t)ti.nt * 1024 : (int64_t)(ti.b_row_pair / 128) * SFA_BYTES;
                const int64_t sfb_row = ((int64_t)gB * p.b_sf_gstride + kg * p.b_sf_kstride + sfb_tile) / 256;
                tma2_load_2d(smem_u32(smem + OFF_SFA + stage * SFA_BYTES), &tmSFA, 0, (int)sfa_row, fb);
                tma2_load_2d(smem_u32(smem + OFF_SFB + stage * SFB_BYTES), &tmSFB, 0, (int)sfb_row, fb);
                pend[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (aborted && leader) {
            // the leader's full barriers count both CTAs' bytes; the follower
            // leaves only after the closing cluster barrier, i.e. after this
            Params q = p;
            q.timeout_ns = 200000000ull;
            volatile int no_abort = 0;
            for (int s = 0; s < STAGES; ++s)
                if (pend[s] >= 0) mbar_wait_cluster(full_bar(s), (uint32_t)pend[s], q, &no_abort);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------------------------------- MMA issuer (leader) ----
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool aborted = false, issued = false;
        for (int64_t t = pair; t < total && !aborted; t += npairs) {
            Tile2 ti;
            get_tile2<BN>(p, s_gofs, s_pt, total_pm, t, rank, ti);
            if (ti.nk == 0) continue;
            if (!mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, p, abort_flag)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int ks = 0; ks < ti.nk; ++ks) {
                if (!mbar_wait_cluster(full_bar(stage), phase, p, abort_flag)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t t_sfa = tmem_base + C::SF0 + C::SF_COLS * stage;
                const uint32_t t_sfb = t_sfa + (NVF4 ? 16 : 4);
                const uint32_t s_sfa = smem_u32(smem + OFF_SFA + stage * SFA_BYTES);
                const uint32_t s_sfb = smem_u32(smem + OFF_SFB + stage * SFB_BYTES);
                const uint64_t adesc = desc_sw128(smem_u32(smem + OFF_A + stage * A_STAGE));
                const uint64_t bdesc = desc_sw128(smem_u32(smem + OFF_B + stage * B_STAGE));
                if constexpr (NVF4) {
                    // atom j (64 K-elements): A -> t_sfa + 4j, B rows
                    // [128h, 128h + 128) -> t_sfb + 8j + 4h; MMA j reads them
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tc_cp_sf2(t_sfa + 4 * j, desc_sf(s_sfa + 512 * j));
#pragma unroll
                        for (int h = 0; h < BN / 128; ++h)
                            tc_cp_sf2(t_sfb + 8 * j + 4 * h, desc_sf(s_sfb + 2048 * h + 512 * j));
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma2_nvf4(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                                     make_idesc2_nvf4<BN>(), t_sfa + 4 * kk, t_sfb + 8 * kk, (ks | kk) != 0 ? 1u : 0u);
                } else {
                    tc_cp_sf2(t_sfa, desc_sf(s_sfa));
#pragma unroll
                    for (int h = 0; h < (BN + 127) / 128; ++h) tc_cp_sf2(t_sfb + 4 * h, desc_sf(s_sfb + 512 * h));
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)
                        tc_mma2(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                                make_idesc2<BN>((uint32_t)kk), t_sfa, t_sfb, (ks | kk) != 0 ? 1u : 0u);
                }
                issued = true;
                tc_commit_both(empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            tc_commit_both(tfull_bar(acc));
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (issued) {
            tc_commit_local2(drain_bar);
            Params q = p;
            q.timeout_ns = 200000000ull;
            volatile int no_abort = 0;
            mbar_wait(drain_bar, 0, q, &no_abort);
        }
    } else if (warp >= 4) {
        // ----------------------------------------------------- epilogue ----
        const int ew = warp - 4;
        const int quarter = ew & 3, half = ew >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t nbox = 0;       // TMA-store boxes this warp has issued (224-wide tiles)
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        for (int64_t t = pair; t < total; t += npairs) {
            Tile2 ti;
            get_tile2<BN>(p, s_gofs, s_pt, total_pm, t, rank, ti);
            const int64_t row = ti.out_row + quarter * 32 + lane;
            if (ti.nk == 0) {      // an empty group's weight gradient: zeros
                if constexpr (BN == 224)
                    epilogue_zero_tma<224>(&tmD, zbox, row - lane, ti.nt, half, lane, p.N);
                else if (!NVF4 && BN == 256 && p.tma_store)
                    epilogue_zero_tma256(&tmD, smem_u32(smem + C::OFF_EPI + kEpiBoxBytes * ew), row - lane, ti.nt,
                                         half, lane);
                else
                    epilogue_zero<BN>(p, row, ti.nt, half);
                continue;
            }
            ApreChunk apre;
            if (EPI == MOE_EPI_SWIGLU_BWD && ti.valid) {
                if (t + npairs < total) {
                    Tile2 tn;
                    get_tile2<BN>(p, s_gofs, s_pt, total_pm, t + npairs, rank, tn);
                    if (tn.valid) swiglu_bwd_prefetch_l2<BN>(p, tn.out_row + quarter * 32 + lane, tn.nt, half);
                }
                swiglu_bwd_prefetch<BN>(p, row, ti.nt, half, 0, apre);
            }
            if (!mbar_wait_cluster(tfull_bar(acc), acc_phase, p, abort_flag)) break;
            tc_fence_after();
            const uint32_t tacc = lane_base + (uint32_t)(acc * BN);
            const uint32_t tempty = mapa(tempty_bar(acc), 0);
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty);
            };
            if (!ti.valid) {
                release();
            } else if constexpr (EPI == MOE_EPI_SWIGLU_BWD) {
                epilogue_swiglu_bwd<BN>(p, tacc, row, ti.nt, half, release, apre);
            } else if constexpr (BN == 224) {
                epilogue_tile_tma224(&tmD, smem_u32(smem + C::OFF_EPI + 2 * kEpiBoxBytes * ew), tacc, row - lane,
                                     ti.nt, half, lane, p.N, nbox, release);
            } else if (!NVF4 && BN == 256 && EPI == MOE_EPI_NONE && p.tma_store) {
                epilogue_tile_tma(&tmD, smem_u32(smem + C::OFF_EPI + kEpiBoxBytes * ew), tacc, row - lane, ti.nt, half, lane,
                                  release);
            } else if constexpr (BN == 256) {
                epilogue_tile_staged<EPI, NVF4>(p, tacc, row, ti.nt, half, release);
            } else {
                epilogue_tile<BN, EPI>(p, tacc, row, ti.nt, half);
                release();
            }
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // the TMA stores issued from this warp's staging buffer are complete
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();      // both CTAs are done with TMEM and with each other's barriers
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
}

}  // namespace sm2
}  // namespace gg

static int g_max_clusters[3] = {0, 0, 0};   // [N = 128, N = 256, N = 224]

template <int BN>
static cudaLaunchConfig_t launch_cfg(int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(gg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gg::sm2::C2<BN>::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int BN, int EPI>
static cudaError_t set_attr_one() {
    return cudaFuncSetAttribute(gg::sm2::k_grouped_gemm_2sm<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gg::sm2::C2<BN>::SMEM_BYTES);
}

template <int BN>
static cudaError_t set_attr_2sm(int* max_clusters) {
    const cudaError_t es[] = {set_attr_one<BN, MOE_EPI_NONE>(), set_attr_one<BN, MOE_EPI_SWIGLU>(),
                              set_attr_one<BN, MOE_EPI_SWIGLU_BWD>(), set_attr_one<BN, MOE_EPI_NONE_F32>()};
    for (cudaError_t e : es)
        if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg<BN>(1024, nullptr, attr);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, gg::sm2::k_grouped_gemm_2sm<BN, MOE_EPI_NONE>, &cfg);
    if (e != cudaSuccess) return e;
    *max_clusters = n;
    return cudaSuccess;
}

cudaError_t gemm_set_attributes_2sm() {
    cudaError_t e = set_attr_2sm<128>(&g_max_clusters[0]);
    if (e != cudaSuccess) return e;
    e = set_attr_2sm<256>(&g_max_clusters[1]);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gg::sm2::k_grouped_gemm_2sm<224, MOE_EPI_NONE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gg::sm2::C2<224>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = launch_cfg<224>(1024, nullptr, attr);
        e = cudaOccupancyMaxActiveClusters(&g_max_clusters[2], gg::sm2::k_grouped_gemm_2sm<224, MOE_EPI_NONE>, &cfg);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t es[] = {
        cudaFuncSetAttribute(gg::sm2::k_grouped_gemm_2sm<256, MOE_EPI_NONE, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, gg::sm2::C2<256, true>::SMEM_BYTES),
        cudaFuncSetAttribute(gg::sm2::k_grouped_gemm_2sm<256, MOE_EPI_NONE_F32, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, gg::sm2::C2<256, true>::SMEM_BYTES)};
    for (cudaError_t x : es)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

// NVFP4 pair kernel (N = 256, MOE_EPI_NONE or MOE_EPI_NONE_F32); `clusters`
// must not exceed gemm_max_clusters_2sm(256) (its shared memory is smaller,
// so as many pairs are co-resident).
cudaError_t gemm_launch_2sm_nvf4(int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const CUtensorMap& tmSFA, const CUtensorMap& tmSFB, const gg::Params& p,
                                 int clusters, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg<256>(clusters, stream, attr);
    cfg.dynamicSmemBytes = gg::sm2::C2<256, true>::SMEM_BYTES;
    if (epilogue == MOE_EPI_NONE_F32)
        return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<256, MOE_EPI_NONE_F32, true>, tmA, tmB, tmSFA,
                                  tmSFB, tmA, p);
    return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<256, MOE_EPI_NONE, true>, tmA, tmB, tmSFA, tmSFB, tmA,
                              p);
}

int gemm_max_clusters_2sm(int bn) { return g_max_clusters[bn == 256 ? 1 : (bn == 224 ? 2 : 0)]; }

template <int BN>
static cudaError_t launch_2sm(int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                              const CUtensorMap& tmSFB, const CUtensorMap& tmD, const gg::Params& p, int clusters,
                              cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg<BN>(clusters, stream, attr);
    switch (epilogue) {
        case MOE_EPI_SWIGLU:
            return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<BN, MOE_EPI_SWIGLU>, tmA, tmB, tmSFA, tmSFB,
                                      tmD, p);
        case MOE_EPI_SWIGLU_BWD:
            return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<BN, MOE_EPI_SWIGLU_BWD>, tmA, tmB, tmSFA,
                                      tmSFB, tmD, p);
        case MOE_EPI_NONE_F32:
            return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<BN, MOE_EPI_NONE_F32>, tmA, tmB, tmSFA, tmSFB,
                                      tmD, p);
        default:
            return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<BN, MOE_EPI_NONE>, tmA, tmB, tmSFA, tmSFB,
                                      tmD, p);
    }
}

cudaError_t gemm_launch_2sm(int bn, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmSFA, const CUtensorMap& tmSFB, const CUtensorMap& tmD,
                            const gg::Params& p, int clusters, cudaStream_t stream) {
    if (bn == 256) return launch_2sm<256>(epilogue, tmA, tmB, tmSFA, tmSFB, tmD, p, clusters, stream);
    if (bn == 224) {
        if (epilogue != MOE_EPI_NONE) return cudaErrorInvalidValue;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = launch_cfg<224>(clusters, stream, attr);
        return cudaLaunchKernelEx(&cfg, gg::sm2::k_grouped_gemm_2sm<224, MOE_EPI_NONE>, tmA, tmB, tmSFA, tmSFB, tmD, p);
    }
    return launch_2sm<128>(epilogue, tmA, tmB, tmSFA, tmSFB, tmD, p, clusters, stream);
}

}  // namespace moe
