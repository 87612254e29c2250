// MXFP8 grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// [TE-JAX] "Optimization 1: Grouped GEMM": every expert's GEMM runs in one
// kernel call, each over its actual rows, and only regions with valid tokens
// are computed; on Blackwell the expert GEMMs take MXFP8 operands with block
// scales (same section).
// [TE-JAX] Figure 3: the grouped MLP is two grouped GEMMs (up/gate, down);
// the SwiGLU between them is fused into the up/gate epilogue here.
//
// Design (one persistent CTA per SM, 384 threads, warp-specialised):
//   warp 0 lane 0   TMA producer: per k-step one 128x128 A box, two 128x128
//                   B boxes (N = 256) and the three 512-byte scale atoms, all
//                   completing on one mbarrier (expect_tx).
//   warp 1          allocates 512 TMEM columns; lane 0 issues
//                   tcgen05.cp (scales smem -> TMEM) and 4 x
//                   tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) per
//                   k-step into a 128x256 fp32 accumulator in TMEM.
//   warps 4..11     epilogue, two warps per TMEM lane quarter (one per
//                   128-column half): tcgen05.ld of their 32 lanes, bf16
//                   conversion, fused SwiGLU / SwiGLU-backward, stores.
// The tile list is derived on the device from the group offsets (multiples
// of 128), so a tile never straddles two groups and the host never sees the
// counts.  Every mbarrier wait is bounded: on timeout the CTA records
// MOE_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM
// and returns.

#include <algorithm>

#include "gemm_common.cuh"

namespace moe {
namespace gg {

// Tile configurations.  BN = 128 keeps two accumulators in TMEM so the
// epilogue of one tile overlaps the mainloop of the next; BN = 256 halves
// the A re-reads but has a single accumulator.
// Operand formats of the 1-SM kernel.
enum { FMT_MXF8 = 0, FMT_BF16 = 1, FMT_NVF4 = 2 };

template <int BN_, int FMT = FMT_MXF8>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int NACC = BN_ == 128 ? 2 : 1;
    static constexpr int STAGES = BN_ == 128 ? 6 : 4;
    static constexpr int A_STAGE = BM * BK;
    static constexpr int B_STAGE = BN_ * BK;
    // scale bytes per 128 rows and k-step: MXFP8 one 512-byte atom (4
    // blocks of 32), NVFP4 four atoms (16 blocks of 16 E2M1 values: a
    // 128-byte k-step holds 256 of them)
    static constexpr int SFA_STG = FMT == FMT_NVF4 ? 4 * SFA_STAGE : SFA_STAGE;
    static constexpr int SFB_STAGE = (BN_ / 128) * SFA_STG;
    static constexpr uint32_t STAGE_TX = A_STAGE + B_STAGE + SFA_STG + SFB_STAGE;
    // TMEM: accumulators at [0, NACC*BN); stage s scales at SF0 + SF_COLS s
    // (MXFP8: A 4 columns, B BN/32; NVFP4: A 16, B BN/8), so a stage's scale
    // columns are rewritten only after the MMAs that read them completed.
    static constexpr uint32_t SF_COLS = FMT == FMT_NVF4 ? 16 + 16 * (BN_ / 128) : TMEM_SF_STRIDE;
    static constexpr uint32_t SF0 = NACC * BN_;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STG;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
    static constexpr int NBAR = 2 * STAGES + 2 * NACC + 1;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
    static constexpr int OFF_GOFS = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = OFF_GOFS + (MAX_G + 1) * 4 + 1024;   // + alignment slack
    static_assert(SF0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Tile {
    int g;            // group of the B operand (FWD/DGRAD) / output group (WGRAD)
    int64_t a_row;    // first row of the A box
    int b_row;        // first row of the B boxes (BN consecutive rows)
    int64_t kbeg;     // first k-step (units of 128 along K)
    int nk;           // number of k-steps
    int64_t out_row;  // first output row
    int nt;           // tile index along N
    int kq;           // NVFP4 WGRAD: 64-row MMAs in the last k-step (4, or 2 for a group ending half-way)
};

// FWD / DGRAD tile t -> (m-tile, n-tile), in raster bands of p.band
// m-tiles (consecutive tiles walk the n-tiles of a band, which share each B
// tile).  With p.group_bands the tiles are taken group by group (group g
// owns m-tiles gofs[g]/128 .. gofs[g+1]/128 and their n_tiles tiles each, so
// the group of tile t is the group of row (t / n_tiles) * 128) and the bands
// restart at each group's first m-tile: a band never mixes two experts'
// weight blocks, and a band as wide as the group streams that group's
// weights from DRAM once.
__device__ __forceinline__ void fwd_tile_mn(const Params& p, const int* s_gofs, int64_t total_mt, int64_t t,
                                            int64_t& mt, int& nt) {
    if (!p.group_bands) {
        band_decode(t, total_mt, p.n_tiles, p.band, mt, nt);
        return;
    }
    const int g = find_group(s_gofs, p.G, (t / p.n_tiles) * BM);
    const int64_t m0 = s_gofs[g] / BM, mg = (s_gofs[g + 1] - s_gofs[g]) / BM;
    int64_t ml;
    band_decode(t - m0 * p.n_tiles, mg, p.n_tiles, p.band, ml, nt);
    mt = m0 + ml;
}

// NVF4: NVFP4 WGRAD counts its contraction in rows (k-steps of 256 rows,
// 128 packed bytes), so kbeg is the group's first row and a group whose
// row count is an odd multiple of 128 ends with a half k-step.
template <int BN, bool NVF4 = false>
__device__ __forceinline__ void get_tile(const Params& p, const int* s_gofs, int64_t total_mt, int64_t t, Tile& ti) {
    ti.kq = 4;
    int64_t mt;
    int nt;
    if (p.mode != MOE_GEMM_WGRAD) {
        fwd_tile_mn(p, s_gofs, total_mt, t, mt, nt);
        const int64_t row = mt * BM;
        ti.g = find_group(s_gofs, p.G, row);
        ti.a_row = row;
        ti.out_row = row;
        ti.kbeg = 0;
        ti.nk = (int)((p.K + (p.k_ceil ? BK - 1 : 0)) / BK);
    } else {
        const int64_t tpg = (int64_t)p.m_tiles * p.n_tiles;
        const int g = (int)(t / tpg);
        band_decode(t - (int64_t)g * tpg, p.m_tiles, p.n_tiles, p.band, mt, nt);
        ti.g = g;
        ti.a_row = mt * BM;
        if constexpr (NVF4) {
            const int rows = s_gofs[g + 1] - s_gofs[g];
            ti.kbeg = s_gofs[g];
            ti.nk = (rows + 255) / 256;
            ti.kq = (rows & 255) != 0 ? 2 : 4;
        } else {
            ti.kbeg = s_gofs[g] / BK;
            ti.nk = (s_gofs[g + 1] - s_gofs[g]) / BK;
        }
        ti.out_row = (int64_t)g * p.M + mt * BM;
    }
    ti.b_row = nt * BN;
    ti.nt = nt;
}

// --------------------------------------------------------------- kernel ----

// EPI: the epilogue (moe_epilogue_t), fixed at compile time so each
// instance keeps only its own epilogue's registers.  FMT: FMT_MXF8 (E4M3
// with E8M0 scales per 32, kind::mxf8f6f4); FMT_BF16 (plain bf16 operands,
// kind::f16, no scale factors; 64 elements per 128-byte k-step), for the
// router's dense GEMMs; FMT_NVF4 (packed E2M1 with UE4M3 scales per 16 and
// per-tensor fp32 scales, kind::mxf4nvf4; 256 elements per 128-byte
// k-step, plain epilogues only).
template <int BN, int EPI, int FMT = FMT_MXF8>
__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
    using C = Cfg<BN, FMT>;
    constexpr bool BF16 = FMT == FMT_BF16, NVF4 = FMT == FMT_NVF4;
    static_assert(!NVF4 || (BN == 256 && (EPI == MOE_EPI_NONE || EPI == MOE_EPI_NONE_F32)), "NVFP4 instances");
    constexpr int STAGES = C::STAGES, NACC = C::NACC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + NACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * NACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    int* s_gofs = reinterpret_cast<int*>(smem + C::OFF_GOFS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort_flag = 0;
        *bad_flag = 0;
    }
    if (p.gofs != nullptr) {
        for (int i = threadIdx.x; i <= p.G; i += THREADS) s_gofs[i] = p.gofs[i];
    } else if (threadIdx.x == 0) {      // dense: one group of all M rows
        s_gofs[0] = 0;
        s_gofs[1] = (int)p.M;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    __syncthreads();
    // offsets must start at 0, be monotone, 128-aligned and fit the buffer
    if (threadIdx.x == 0) {
        bool ok = s_gofs[0] == 0;
        for (int g = 0; g < p.G && ok; ++g) ok = s_gofs[g + 1] >= s_gofs[g] && (s_gofs[g + 1] % BM) == 0;
        const int64_t limit = p.mode == MOE_GEMM_WGRAD ? p.K : p.M;
        ok = ok && (int64_t)s_gofs[p.G] <= limit;
        if (!ok) {
            *bad_flag = 1;
            if (blockIdx.x == 0) set_err(p.err, MOE_ERR_BAD_OFFSETS);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const bool bad = *bad_flag != 0;

    const int64_t total_mt = p.mode == MOE_GEMM_WGRAD ? 0 : (int64_t)s_gofs[p.G] / BM;
    const int64_t total = bad ? 0
                              : (p.mode == MOE_GEMM_WGRAD ? (int64_t)p.G * p.m_tiles * p.n_tiles
                                                          : total_mt * p.n_tiles);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer ----
        uint8_t* sA = smem + C::OFF_A;
        uint8_t* sB = smem + C::OFF_B;
        uint8_t* sSFA = smem + C::OFF_SFA;
        uint8_t* sSFB = smem + C::OFF_SFB;
        int pend[STAGES];
        for (int s = 0; s < STAGES; ++s) pend[s] = -1;
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        for (int64_t t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
            Tile ti;
            get_tile<BN, NVF4>(p, s_gofs, total_mt, t, ti);
            const int gB = p.mode == MOE_GEMM_WGRAD ? 0 : ti.g;
            for (int ks = 0; ks < ti.nk; ++ks) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, p, abort_flag)) {
                    aborted = true;
                    break;
                }
                const int64_t kg = ti.kbeg + ks;
                const uint32_t fb = full_bar(stage);
                if constexpr (NVF4) {
                    // k-step = 128 packed bytes = 256 elements = four 64-element
                    // scale atoms; WGRAD steps start at the group's rows (a
                    // multiple of 128 rows, so possibly mid-chunk) and the
                    // last one may hold only two atoms
                    const bool wg = p.mode == MOE_GEMM_WGRAD;
                    const int nq = (wg && ks == ti.nk - 1) ? ti.kq : 4;
                    const int kx = wg ? (int)((ti.kbeg + 256 * (int64_t)ks) / 2) : (int)(kg * BK);
                    const int64_t a0 = wg ? (ti.kbeg + 256 * (int64_t)ks) / 64 : 4 * kg;
                    mbar_expect_tx(fb, (uint32_t)(C::A_STAGE + C::B_STAGE + nq * 512 * (1 + BN / 128)));
                    tma_load_2d(smem_u32(sA + stage * C::A_STAGE), &tmA, kx, (int)ti.a_row, fb);
                    const bool whole = nq == 4 && (a0 & 3) == 0;
                    const uint8_t* sfa = p.a_sf + (ti.a_row / 128) * 2048;
                    if (whole) {
                        bulk_load(smem_u32(sSFA + stage * C::SFA_STG), sfa + (a0 >> 2) * p.a_sf_kstride, 2048, fb);
                    } else {
                        for (int j = 0; j < nq; ++j) {
                            const int64_t a = a0 + j;
                            bulk_load(smem_u32(sSFA + stage * C::SFA_STG + 512 * j),
                                      sfa + (a >> 2) * p.a_sf_kstride + (a & 3) * 512, 512, fb);
                        }
                    }
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) {
                        const int brow = ti.b_row + 128 * h;
                        tma_load_3d(smem_u32(sB + stage * C::B_STAGE + h * 16384), &tmB, kx, brow, gB, fb);
                        const uint8_t* sfb = p.b_sf + (int64_t)gB * p.b_sf_gstride + (int64_t)(brow / 128) * 2048;
                        const uint32_t dst = smem_u32(sSFB + stage * C::SFB_STAGE + h * C::SFA_STG);
                        if (whole) {
                            bulk_load(dst, sfb + (a0 >> 2) * p.b_sf_kstride, 2048, fb);
                        } else {
                            for (int j = 0; j < nq; ++j) {
                                const int64_t a = a0 + j;
                                bulk_load(dst + 512 * j, sfb + (a >> 2) * p.b_sf_kstride + (a & 3) * 512, 512, fb);
                            }
                        }
                    }
                } else {
                    const int kx = (int)(kg * BK);
                    mbar_expect_tx(fb, BF16 ? (uint32_t)(C::A_STAGE + C::B_STAGE) : C::STAGE_TX);
                    tma_load_2d(smem_u32(sA + stage * C::A_STAGE), &tmA, kx, (int)ti.a_row, fb);
                    const uint8_t* sfa = p.a_sf + kg * p.a_sf_kstride + (ti.a_row / 128) * C::SFA_STG;
                    const uint8_t* sfb = p.b_sf + (int64_t)gB * p.b_sf_gstride + kg * p.b_sf_kstride;
                    if constexpr (!BF16) bulk_load(smem_u32(sSFA + stage * C::SFA_STG), sfa, C::SFA_STG, fb);
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) {
                        const int brow = ti.b_row + 128 * h;
                        tma_load_3d(smem_u32(sB + stage * C::B_STAGE + h * 16384), &tmB, kx, brow, gB, fb);
                        if constexpr (!BF16)
                            bulk_load(smem_u32(sSFB + stage * C::SFB_STAGE + h * C::SFA_STG),
                                      sfb + (int64_t)(brow / 128) * C::SFA_STG, C::SFA_STG, fb);
                    }
                }
                pend[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (aborted) {
            // let every copy still in flight land before the CTA exits
            Params q = p;
            q.timeout_ns = 200000000ull;
            volatile int no_abort = 0;
            for (int s = 0; s < STAGES; ++s)
                if (pend[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend[s], q, &no_abort);
        }
    } else if (warp == 1 && lane == 0) {
        // --------------------------------------------------- MMA issuer ----
        const uint8_t* sA = smem + C::OFF_A;
        const uint8_t* sB = smem + C::OFF_B;
        const uint8_t* sSFA = smem + C::OFF_SFA;
        const uint8_t* sSFB = smem + C::OFF_SFB;
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool aborted = false;
        bool issued = false;
        for (int64_t t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
            Tile ti;
            get_tile<BN, NVF4>(p, s_gofs, total_mt, t, ti);
            if (ti.nk == 0) continue;
            if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, p, abort_flag)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int ks = 0; ks < ti.nk; ++ks) {
                if (!mbar_wait(full_bar(stage), phase, p, abort_flag)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t t_sfa = tmem_base + C::SF0 + C::SF_COLS * stage;
                const uint32_t t_sfb = t_sfa + (NVF4 ? 16 : 4);
                // NVFP4: 64-element MMAs in this k-step (WGRAD's last step
                // of a group ending half-way has 2)
                const int nq = (NVF4 && p.mode == MOE_GEMM_WGRAD && ks == ti.nk - 1) ? ti.kq : 4;
                if constexpr (NVF4) {
                    // atom j (64 K-elements) of A -> columns t_sfa + 4j; atom
                    // j of B rows [128h, 128h + 128) -> t_sfb + 8j + 4h, so
                    // the MMA over K-elements [64j, 64j + 64) reads A's 4
                    // columns at t_sfa + 4j and B's 8 at t_sfb + 8j
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j < nq) {
                            tc_cp_sf(t_sfa + 4 * j, desc_sf(smem_u32(sSFA + stage * C::SFA_STG + 512 * j)));
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h)
                                tc_cp_sf(t_sfb + 8 * j + 4 * h,
                                         desc_sf(smem_u32(sSFB + stage * C::SFB_STAGE + h * C::SFA_STG + 512 * j)));
                        }
                    }
                } else if constexpr (!BF16) {
                    tc_cp_sf(t_sfa, desc_sf(smem_u32(sSFA + stage * C::SFA_STG)));
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        tc_cp_sf(t_sfb + 4 * h, desc_sf(smem_u32(sSFB + stage * C::SFB_STAGE + 512 * h)));
                }
                const uint64_t adesc = desc_sw128(smem_u32(sA + stage * C::A_STAGE));
                const uint64_t bdesc = desc_sw128(smem_u32(sB + stage * C::B_STAGE));
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk) {
                    // advance 32 bytes along K inside the 128-byte swizzled row
                    // (32 fp8 elements with block scales, 16 bf16, or 64
                    // packed E2M1 elements)
                    if constexpr (BF16)
                        tc_mma_bf16(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                                    make_idesc_bf16<BN>(), (ks | kk) != 0 ? 1u : 0u);
                    else if constexpr (NVF4) {
                        if (kk < nq)
                            tc_mma_nvf4(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                                        make_idesc_nvf4<BN>(), t_sfa + 4 * kk, t_sfb + 8 * kk,
                                        (ks | kk) != 0 ? 1u : 0u);
                    }
                    else
                        tc_mma(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                               make_idesc<BN>((uint32_t)kk), t_sfa, t_sfb, (ks | kk) != 0 ? 1u : 0u);
                }
                issued = true;
                tc_commit(empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            tc_commit(tfull_bar(acc));
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (issued) {
            // every MMA issued by this thread completes before TMEM is freed
            tc_commit(drain_bar);
            Params q = p;
            q.timeout_ns = 200000000ull;
            volatile int no_abort = 0;
            mbar_wait(drain_bar, 0, q, &no_abort);
        }
    } else if (warp >= 4) {
        // ----------------------------------------------------- epilogue ----
        // warp (4 + e): TMEM lane quarter e % 4, column half e / 4
        const int ew = warp - 4;
        const int quarter = ew & 3, half = ew >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
            Tile ti;
            get_tile<BN, NVF4>(p, s_gofs, total_mt, t, ti);
            const int64_t row = ti.out_row + quarter * 32 + lane;
            if (ti.nk == 0) {   // WGRAD of an empty group
                epilogue_zero<BN>(p, row, ti.nt, half);
                continue;
            }
            ApreChunk apre;
            if constexpr (EPI == MOE_EPI_SWIGLU_BWD) {
                if (t + gridDim.x < total) {      // FWD/DGRAD only: rows = m-tile * 128
                    int64_t mt;
                    int nt;
                    fwd_tile_mn(p, s_gofs, total_mt, t + gridDim.x, mt, nt);
                    swiglu_bwd_prefetch_l2<BN>(p, mt * BM + quarter * 32 + lane, nt, half);
                }
                swiglu_bwd_prefetch<BN>(p, row, ti.nt, half, 0, apre);
            }
            if (!mbar_wait(tfull_bar(acc), acc_phase, p, abort_flag)) break;
            tc_fence_after();
            const uint32_t tacc = lane_base + (uint32_t)(acc * BN);
            const uint32_t tempty = tempty_bar(acc);
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
            };
            if constexpr (EPI == MOE_EPI_SWIGLU_BWD) {
                epilogue_swiglu_bwd<BN>(p, tacc, row, ti.nt, half, release, apre);
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
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
}

}  // namespace gg

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t gemm_init_driver() {
    if (g_encode) return cudaSuccess;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorUnknown;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

template <int BN, int EPI>
static cudaError_t set_attr_1sm() {
    return cudaFuncSetAttribute(gg::k_grouped_gemm<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gg::Cfg<BN>::SMEM_BYTES);
}

cudaError_t gemm_set_attributes() {
    const cudaError_t es[] = {set_attr_1sm<128, MOE_EPI_NONE>(),     set_attr_1sm<128, MOE_EPI_SWIGLU>(),
                              set_attr_1sm<128, MOE_EPI_SWIGLU_BWD>(), set_attr_1sm<128, MOE_EPI_NONE_F32>(),
                              set_attr_1sm<256, MOE_EPI_NONE>(),     set_attr_1sm<256, MOE_EPI_SWIGLU>(),
                              set_attr_1sm<256, MOE_EPI_SWIGLU_BWD>(), set_attr_1sm<256, MOE_EPI_NONE_F32>(),
                              cudaFuncSetAttribute(gg::k_grouped_gemm<256, MOE_EPI_NONE_F32, gg::FMT_BF16>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   gg::Cfg<256, gg::FMT_BF16>::SMEM_BYTES),
                              cudaFuncSetAttribute(gg::k_grouped_gemm<256, MOE_EPI_NONE, gg::FMT_NVF4>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   gg::Cfg<256, gg::FMT_NVF4>::SMEM_BYTES),
                              cudaFuncSetAttribute(gg::k_grouped_gemm<256, MOE_EPI_NONE_F32, gg::FMT_NVF4>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   gg::Cfg<256, gg::FMT_NVF4>::SMEM_BYTES)};
    for (cudaError_t e : es)
        if (e != cudaSuccess) return e;
    return gemm_set_attributes_2sm();
}

template <int BN>
static void launch_1sm(int epilogue, int grid, const CUtensorMap& tmA, const CUtensorMap& tmB, const gg::Params& p,
                       cudaStream_t s) {
    using namespace gg;
    switch (epilogue) {
        case MOE_EPI_SWIGLU:
            k_grouped_gemm<BN, MOE_EPI_SWIGLU><<<grid, THREADS, Cfg<BN>::SMEM_BYTES, s>>>(tmA, tmB, p);
            break;
        case MOE_EPI_SWIGLU_BWD:
            k_grouped_gemm<BN, MOE_EPI_SWIGLU_BWD><<<grid, THREADS, Cfg<BN>::SMEM_BYTES, s>>>(tmA, tmB, p);
            break;
        case MOE_EPI_NONE_F32:
            k_grouped_gemm<BN, MOE_EPI_NONE_F32><<<grid, THREADS, Cfg<BN>::SMEM_BYTES, s>>>(tmA, tmB, p);
            break;
        default:
            k_grouped_gemm<BN, MOE_EPI_NONE><<<grid, THREADS, Cfg<BN>::SMEM_BYTES, s>>>(tmA, tmB, p);
    }
}

// Kernel choice.  WGRAD runs on the CTA-pair kernel (gemm2sm.cu, 256 x 256
// pair tiles, TMA-store epilogue): its short contraction (one group's rows)
// makes the 1-SM kernel wait on operand loads, and the pair halves each SM's
// operand traffic.  FWD and DGRAD run on the 1-SM kernel with 128 x 256
// tiles, except plain-epilogue ones with K <= 2048 over many rows: a
// group's last 128-row tile leaves half of a 256-row pair tile idle, which
// cost more than the pair kernel saved on the longer contractions, with the
// fused epilogues, on small problems and with small groups (measured on
// the DeepSeek-V3 layer and the grouped GEMM sweep).  A caller can force one
// kernel per call through moe_gemm_opts_t (the measured alternatives stay
// selectable and parity-tested); WGRAD with M % 256 != 0 always uses the
// 1-SM kernel.
struct GemmChoice {
    int sel;              // 0 = 1-SM kernel; 256 / 128 = CTA pair with 256- / 128-wide tiles
    int bn_1sm;           // 1-SM tile width: 256, or 128 (two TMEM accumulators)
    int band;             // m-tiles per raster band, 0 = the kernel's default
    bool register_stores; // pair kernel, plain epilogue: register-staged stores instead of TMA stores
    int wg_lo, wg_hi;     // WGRAD group filter by row count (0, 0 = every group)
};

static bool gemm_opts_valid(const moe_gemm_opts_t* o) {
    return o == nullptr || (o->kernel >= MOE_GEMM_KERNEL_AUTO && o->kernel <= MOE_GEMM_KERNEL_PAIR_N128 &&
                            o->band >= 0 && o->band <= 64 && (o->register_stores == 0 || o->register_stores == 1) &&
                            o->wgrad_rows_lo >= 0 && o->wgrad_rows_hi >= 0);
}

// sel = -1 leaves the choice to the default rule of the call.
static GemmChoice gemm_choice(const moe_gemm_opts_t* o) {
    GemmChoice c{-1, 256, 0, false, 0, 0};
    if (o == nullptr) return c;
    c.wg_lo = o->wgrad_rows_lo;
    c.wg_hi = o->wgrad_rows_hi;
    switch (o->kernel) {
        case MOE_GEMM_KERNEL_1SM: c.sel = 0; break;
        case MOE_GEMM_KERNEL_1SM_N128: c.sel = 0; c.bn_1sm = 128; break;
        case MOE_GEMM_KERNEL_PAIR: c.sel = 256; break;
        case MOE_GEMM_KERNEL_PAIR_N128: c.sel = 128; break;
        default: break;
    }
    c.band = o->band;
    c.register_stores = o->register_stores != 0;
    return c;
}

// Scale atoms (512 bytes each) seen as a 2-D uint8 tensor of 256-byte rows:
// `atoms` atoms, boxes of `box_rows` rows (2 = one atom, 4 = two atoms).
static bool make_sf_map(CUtensorMap* m, const void* base, int64_t atoms, int box_rows) {
    cuuint64_t gdim[2] = {256, (cuuint64_t)(2 * atoms)}, gstr[1] = {256};
    cuuint32_t box[2] = {256, (cuuint32_t)box_rows}, estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstr, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 output [rows, N] for TMA stores: 32-row x kEpiBoxCols-column boxes
// (rows of 128 bytes with the 128-byte swizzle, or 64 with the 64-byte one).
static bool make_d_map(CUtensorMap* m, void* base, int64_t rows, int N) {
    cuuint64_t gdim[2] = {(cuuint64_t)N, (cuuint64_t)rows}, gstr[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {(cuuint32_t)gg::kEpiBoxCols, 32}, estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstr, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          gg::kEpiBoxCols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// rank-2/3 uint8 tensor map, 128x128 boxes, 128-byte swizzle
static bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     int box_rows = 128) {
    cuuint64_t gdim[3], gstr[2];
    cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1}, estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
    for (int i = 0; i < rank - 1; ++i) gstr[i] = strides_bytes[i];
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), gdim, gstr,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

// MXFP8 outputs of h for the SwiGLU epilogue (all NULL: not produced)
struct HQuantOut {
    uint8_t* codes_row;
    uint8_t* scales_row;
    uint8_t* codes_col;
    uint8_t* scales_col;
};

static moe_status_t gemm_run(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                             int b_layout, const int32_t* gofs, int G, int64_t M, int N, int64_t K, int epilogue,
                             const void* epi_aux, void* d, void* d2, const HQuantOut& hq,
                             const moe_gemm_opts_t* opts, int32_t* err, void* stream) {
    using namespace gg;
    MOE_REQUIRE(gemm_opts_valid(opts), MOE_ERR_INVALID_ARG);
    const GemmChoice choice = gemm_choice(opts);
    MOE_REQUIRE(mode == MOE_GEMM_FWD || mode == MOE_GEMM_DGRAD || mode == MOE_GEMM_WGRAD, MOE_ERR_INVALID_ARG);
    const bool wg_filter = choice.wg_lo > 0 || choice.wg_hi > 0;
    MOE_REQUIRE(!wg_filter || mode == MOE_GEMM_WGRAD, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(a && a_sf && b && b_sf && gofs && d, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(G >= 1 && G <= MAX_G && M > 0 && N > 0 && K > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(M % 128 == 0 && K % BK == 0 && N % 128 == 0, MOE_ERR_UNSUPPORTED);
    const int BN = (choice.bn_1sm == 256 && N % 256 == 0) ? 256 : 128;
    MOE_REQUIRE(K <= 0x7FFFFF80LL && M <= 0x7FFFFF80LL, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(a) && moe_aligned16(b) && moe_aligned16(a_sf) && moe_aligned16(b_sf) &&
                    moe_aligned16(d) && (d2 == nullptr || moe_aligned16(d2)) &&
                    (epi_aux == nullptr || moe_aligned16(epi_aux)),
                MOE_ERR_ALIGNMENT);
    const bool t224 = mode == MOE_GEMM_WGRAD && b_layout == MOE_B_SF_TILE224;
    if (mode == MOE_GEMM_WGRAD) {
        MOE_REQUIRE(epilogue == MOE_EPI_NONE, MOE_ERR_INVALID_ARG);
        MOE_REQUIRE(b_layout == MOE_B_GNK || b_layout == MOE_B_NGK || t224, MOE_ERR_INVALID_ARG);
    } else {
        MOE_REQUIRE(b_layout == MOE_B_GNK || b_layout == MOE_B_NGK, MOE_ERR_INVALID_ARG);
        MOE_REQUIRE(epilogue == MOE_EPI_NONE || epilogue == MOE_EPI_SWIGLU || epilogue == MOE_EPI_SWIGLU_BWD ||
                        epilogue == MOE_EPI_NONE_F32,
                    MOE_ERR_INVALID_ARG);
        if (epilogue == MOE_EPI_SWIGLU) MOE_REQUIRE(d2 != nullptr || hq.codes_row != nullptr, MOE_ERR_INVALID_ARG);
        if (epilogue == MOE_EPI_SWIGLU_BWD) MOE_REQUIRE(epi_aux != nullptr, MOE_ERR_INVALID_ARG);
    }
    MOE_REQUIRE(device_initialized() && g_encode != nullptr, MOE_ERR_NOT_INITIALIZED);
    if (t224) MOE_REQUIRE(M % 256 == 0 && gemm_max_clusters_2sm(224) > 0, MOE_ERR_UNSUPPORTED);

    CUtensorMap tmA, tmB;
    Params p{};
    p.mode = mode;
    p.epi = epilogue;
    p.G = G;
    p.N = N;
    p.M = M;
    p.K = K;
    p.gofs = gofs;
    p.a_sf = a_sf;
    p.b_sf = b_sf;
    p.d = (__nv_bfloat16*)d;
    p.d2 = (__nv_bfloat16*)d2;
    p.n_out = N;
    p.ldd = N;
    p.k_ceil = 0;
    p.hq_r = hq.codes_row;
    p.hs_r = hq.scales_row;
    p.hq_c = hq.codes_col;
    p.hs_c = hq.scales_col;
    p.aux = (const __nv_bfloat16*)epi_aux;
    p.err = err;
    p.timeout_ns = 2000000000ull;   // 2 s per wait
    // m-tiles per raster band: 3 for long contractions, 4 for K <= 2048
    // (measured on the DeepSeek-V3 layer against 2, 4, 8, 16 and 32).  The
    // fp32-output dgrad takes group-aligned bands: its DRAM reads fall from
    // 6.3 to 5.6 GB a launch at the DeepSeek-V3 shape, its time is the same.
    // The other GEMMs keep bands across group boundaries: group-aligned
    // bands made the plain dgrad 3 % slower, and the SwiGLU up/gate GEMM
    // 1-3 % slower even with bands of a whole group, which cut its reads
    // from 12.6 to 9.4 GB (it is not bound by DRAM).
    p.group_bands = mode != MOE_GEMM_WGRAD && epilogue == MOE_EPI_NONE_F32;
    p.band = choice.band > 0 ? choice.band : (K <= 2048 ? 4 : 3);
    p.n_tiles = N / BN;
    int64_t upper_tiles;
    if (mode == MOE_GEMM_WGRAD) {
        // A [M, K], B [N, K], both columnwise codes; scales: atom layout of
        // the [M, K] / [N, K] matrices
        const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K};
        const uint64_t db[3] = {(uint64_t)K, (uint64_t)N, 1}, sb[2] = {(uint64_t)K, (uint64_t)K * N};
        MOE_REQUIRE(make_map(&tmA, a, 2, da, sa) && make_map(&tmB, b, 3, db, sb), MOE_ERR_CUDA);
        p.m_tiles = (int)(M / BM);
        p.a_sf_kstride = (M / 128) * 512;
        p.b_sf_kstride = (int64_t)(N / 128) * 512;
        p.b_sf_gstride = 0;
        upper_tiles = (int64_t)G * p.m_tiles * p.n_tiles;
    } else {
        const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K};
        uint64_t db[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G}, sb[2];
        if (b_layout == MOE_B_GNK) {
            sb[0] = (uint64_t)K;
            sb[1] = (uint64_t)N * K;
            p.b_sf_kstride = (int64_t)G * N / 128 * 512;
            p.b_sf_gstride = (int64_t)(N / 128) * 512;
        } else {
            sb[0] = (uint64_t)G * K;
            sb[1] = (uint64_t)K;
            p.b_sf_kstride = (int64_t)(N / 128) * 512;
            p.b_sf_gstride = (K / 128) * (int64_t)(N / 128) * 512;
        }
        MOE_REQUIRE(make_map(&tmA, a, 2, da, sa) && make_map(&tmB, b, 3, db, sb), MOE_ERR_CUDA);
        p.m_tiles = 0;
        p.a_sf_kstride = (M / 128) * 512;
        upper_tiles = (M / BM) * p.n_tiles;
    }
    const int sms = device_sm_count();
    MOE_REQUIRE(sms > 0, MOE_ERR_NOT_INITIALIZED);
    const int grid = (int)(upper_tiles < sms ? (upper_tiles > 0 ? upper_tiles : 1) : sms);
    int sel = choice.sel;
    // the CTA-pair kernel for the weight gradients, and for plain-epilogue
    // FWD/DGRAD with short contractions (K <= 2048) over many rows (at
    // least 65,536, and 512 per group on average): there its lower fixed
    // cost per tile outweighs a group's half-idle odd last pair tile
    const bool pair_fwd = epilogue == MOE_EPI_NONE && K <= 2048 && N % 256 == 0 && M >= 65536 && M >= 512LL * G;
    if (sel < 0) sel = (mode == MOE_GEMM_WGRAD || pair_fwd) ? 256 : 0;
    if (t224) sel = 224;      // the scale layout of b fixes the tile
    const int bn2 = sel == 224 ? 224 : (sel == 256 && N % 256 == 0 ? 256 : 128);
    const bool two_sm = sel != 0 && gemm_max_clusters_2sm(bn2) > 0 && (mode != MOE_GEMM_WGRAD || M % 256 == 0);
    MOE_REQUIRE(!wg_filter || two_sm, MOE_ERR_UNSUPPORTED);   // only the pair kernel filters groups
    if (two_sm) {
        p.wg_filter = wg_filter ? 1 : 0;
        p.wg_lo = choice.wg_lo;
        p.wg_hi = choice.wg_hi;
        p.n_tiles = (N + bn2 - 1) / bn2;
        p.band = choice.band > 0 ? choice.band : 2;     // measured: 2 beat 4, 8 and 16
        const int64_t upper_pairs = mode == MOE_GEMM_WGRAD ? (int64_t)G * (M / 256) * p.n_tiles
                                                           : (M / BM) * (int64_t)p.n_tiles;
        if (t224) p.b_sf_kstride = (int64_t)p.n_tiles * 1024;     // tile-224 layout of b's scales
        const int clusters = (int)std::min<int64_t>(std::max<int64_t>(upper_pairs, 1), gemm_max_clusters_2sm(bn2));
        // B boxes of bn2/2 rows (each CTA of the pair loads half of the tile's B rows)
        CUtensorMap tmB2;
        if (mode == MOE_GEMM_WGRAD) {
            const uint64_t db[3] = {(uint64_t)K, (uint64_t)N, 1}, sb[2] = {(uint64_t)K, (uint64_t)K * N};
            MOE_REQUIRE(make_map(&tmB2, b, 3, db, sb, bn2 / 2), MOE_ERR_CUDA);
        } else {
            const uint64_t db[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G};
            uint64_t sb[2];
            if (b_layout == MOE_B_GNK) {
                sb[0] = (uint64_t)K;
                sb[1] = (uint64_t)N * K;
            } else {
                sb[0] = (uint64_t)G * K;
                sb[1] = (uint64_t)K;
            }
            MOE_REQUIRE(make_map(&tmB2, b, 3, db, sb, bn2 / 2), MOE_ERR_CUDA);
        }
        // atoms in the scale arrays (bounds of the scale tensor maps)
        const int64_t atoms_a = (K / 128) * (M / 128);
        int64_t atoms_b;
        if (t224) atoms_b = (K / 128) * (int64_t)p.n_tiles * 2;
        else if (mode == MOE_GEMM_WGRAD) atoms_b = (K / 128) * (N / 128);
        else atoms_b = (int64_t)G * (K / 128) * (N / 128);
        CUtensorMap tmSFA, tmSFB;
        MOE_REQUIRE(make_sf_map(&tmSFA, a_sf, atoms_a, 2) &&
                        make_sf_map(&tmSFB, b_sf, atoms_b, 2 * ((bn2 + 127) / 128)),
                    MOE_ERR_CUDA);
        // D through the TMA: bf16 [rows, N] in 32-row x 64-column boxes
        CUtensorMap tmD = tmA;
        p.tma_store = (bn2 == 256 && epilogue == MOE_EPI_NONE && !choice.register_stores) || bn2 == 224;
        if (p.tma_store) {
            const int64_t drows = mode == MOE_GEMM_WGRAD ? (int64_t)G * M : M;
            MOE_REQUIRE(make_d_map(&tmD, d, drows, N), MOE_ERR_CUDA);
        }
        if (gemm_launch_2sm(bn2, epilogue, tmA, tmB2, tmSFA, tmSFB, tmD, p, clusters, (cudaStream_t)stream) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    } else if (BN == 256)
        launch_1sm<256>(epilogue, grid, tmA, tmB, p, (cudaStream_t)stream);
    else
        launch_1sm<128>(epilogue, grid, tmA, tmB, p, (cudaStream_t)stream);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t grouped_gemm_mxfp8_ex(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                              const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G,
                                              int64_t M, int N, int64_t K, int epilogue, const void* epi_aux, void* d,
                                              void* d2, const moe_gemm_opts_t* opts, int32_t* err, void* stream) {
    if (epilogue == MOE_EPI_SWIGLU && d2 == nullptr) return MOE_ERR_INVALID_ARG;
    const HQuantOut none = {nullptr, nullptr, nullptr, nullptr};
    return gemm_run(mode, a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, epilogue, epi_aux, d, d2, none, opts, err,
                    stream);
}

extern "C" moe_status_t grouped_gemm_mxfp8(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                           const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G, int64_t M,
                                           int N, int64_t K, int epilogue, const void* epi_aux, void* d, void* d2,
                                           int32_t* err, void* stream) {
    return grouped_gemm_mxfp8_ex(mode, a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, epilogue, epi_aux, d, d2,
                                 nullptr, err, stream);
}

extern "C" moe_status_t grouped_gemm_mxfp8_swiglu_quant_ex(const uint8_t* a, const uint8_t* a_sf,
                                                           const uint8_t* b, const uint8_t* b_sf, int b_layout,
                                                           const int32_t* gofs, int G, int64_t M, int N, int64_t K,
                                                           void* a_pre, void* h, uint8_t* h_codes_row,
                                                           uint8_t* h_scales_row, uint8_t* h_codes_col,
                                                           uint8_t* h_scales_col, const moe_gemm_opts_t* opts,
                                                           int32_t* err, void* stream) {
    MOE_REQUIRE(h_codes_row && h_scales_row && h_codes_col && h_scales_col, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(N > 0 && N % 256 == 0, MOE_ERR_UNSUPPORTED);      // f = N/2 a multiple of 128
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(h_codes_row) & 31) == 0, MOE_ERR_ALIGNMENT);
    const HQuantOut hq = {h_codes_row, h_scales_row, h_codes_col, h_scales_col};
    return gemm_run(MOE_GEMM_FWD, a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, MOE_EPI_SWIGLU, nullptr, a_pre, h, hq,
                    opts, err, stream);
}

extern "C" moe_status_t grouped_gemm_mxfp8_swiglu_quant(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                                        const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G,
                                                        int64_t M, int N, int64_t K, void* a_pre, void* h,
                                                        uint8_t* h_codes_row, uint8_t* h_scales_row,
                                                        uint8_t* h_codes_col, uint8_t* h_scales_col, int32_t* err,
                                                        void* stream) {
    return grouped_gemm_mxfp8_swiglu_quant_ex(a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, a_pre, h, h_codes_row,
                                              h_scales_row, h_codes_col, h_scales_col, nullptr, err, stream);
}

extern "C" moe_status_t gemm_bf16_nt(const void* a, const void* b, int64_t M, int N, int64_t K, float* d,
                                     int32_t* err, void* stream) {
    using namespace gg;
    MOE_REQUIRE(a && b && d && M > 0 && N > 0 && K > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(M % 128 == 0 && M <= 0x7FFFFF80LL && N % 8 == 0 && K % 8 == 0 && K <= (1LL << 30),
                MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(a) && moe_aligned16(b) && (reinterpret_cast<uintptr_t>(d) & 31) == 0,
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized() && g_encode != nullptr, MOE_ERR_NOT_INITIALIZED);
    // bf16 rows seen as bytes: K-steps of 128 bytes = 64 elements; columns of
    // B past N (and bytes past 2K) are zero-filled by the TMA
    const int64_t Kb = 2 * K;
    const int Npad = (N + 255) / 256 * 256;
    CUtensorMap tmA, tmB;
    const uint64_t da[2] = {(uint64_t)Kb, (uint64_t)M}, sa[1] = {(uint64_t)Kb};
    const uint64_t db[3] = {(uint64_t)Kb, (uint64_t)N, 1}, sb[2] = {(uint64_t)Kb, (uint64_t)Kb * N};
    MOE_REQUIRE(make_map(&tmA, a, 2, da, sa) && make_map(&tmB, b, 3, db, sb), MOE_ERR_CUDA);
    Params p{};
    p.mode = MOE_GEMM_FWD;
    p.epi = MOE_EPI_NONE_F32;
    p.G = 1;
    p.N = Npad;
    p.M = M;
    p.K = Kb;
    p.gofs = nullptr;
    p.d = (__nv_bfloat16*)d;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    p.band = 8;
    p.n_tiles = Npad / 256;
    p.n_out = N;
    p.ldd = N;
    p.k_ceil = 1;
    const int sms = device_sm_count();
    MOE_REQUIRE(sms > 0, MOE_ERR_NOT_INITIALIZED);
    const int64_t tiles = (M / BM) * p.n_tiles;
    const int grid = (int)std::min<int64_t>(tiles, sms);
    k_grouped_gemm<256, MOE_EPI_NONE_F32, FMT_BF16>
        <<<grid, THREADS, Cfg<256, FMT_BF16>::SMEM_BYTES, (cudaStream_t)stream>>>(tmA, tmB, p);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t grouped_gemm_nvfp4_ex(int mode, const uint8_t* a, const uint8_t* a_sf,
                                              const float* a_scale, const uint8_t* b, const uint8_t* b_sf,
                                              const float* b_scale, const int32_t* gofs, int G, int64_t M, int N,
                                              int64_t K, int epilogue, void* d, const moe_gemm_opts_t* opts,
                                              int32_t* err, void* stream) {
    using namespace gg;
    MOE_REQUIRE(gemm_opts_valid(opts), MOE_ERR_INVALID_ARG);
    const GemmChoice choice = gemm_choice(opts);
    MOE_REQUIRE(choice.wg_lo == 0 && choice.wg_hi == 0, MOE_ERR_UNSUPPORTED);   // group filter: MXFP8 pair kernel only
    MOE_REQUIRE(mode == MOE_GEMM_FWD || mode == MOE_GEMM_DGRAD || mode == MOE_GEMM_WGRAD, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(epilogue == MOE_EPI_NONE || (epilogue == MOE_EPI_NONE_F32 && mode != MOE_GEMM_WGRAD),
                MOE_ERR_INVALID_ARG);      // WGRAD writes bf16 (an empty group's tile is zero-filled as bf16)
    MOE_REQUIRE(a && a_sf && a_scale && b && b_sf && b_scale && gofs && d, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(G >= 1 && G <= MAX_G && M > 0 && N > 0 && K > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(M % 128 == 0 && N % 256 == 0 && K % 256 == 0 && M <= 0x7FFFFF80LL && K <= (1LL << 30),
                MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(a) && moe_aligned16(b) && moe_aligned16(a_sf) && moe_aligned16(b_sf) &&
                    (reinterpret_cast<uintptr_t>(d) & 31) == 0 && (reinterpret_cast<uintptr_t>(a_scale) & 3) == 0 &&
                    (reinterpret_cast<uintptr_t>(b_scale) & 3) == 0,
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized() && g_encode != nullptr, MOE_ERR_NOT_INITIALIZED);
    const bool wg = mode == MOE_GEMM_WGRAD;
    // packed E2M1 rows seen as bytes: K/2 bytes per row, 128-byte k-steps.
    // FWD/DGRAD: A [M, K], B [G][N][K]; WGRAD: A [M, K] and B [N, K] are the
    // transposed (columnwise) codes of the two row-permuted operands, K the
    // rows, D [G][M][N] (each group's contraction runs over its own rows)
    const int64_t Kb = K / 2;
    CUtensorMap tmA, tmB;
    const uint64_t da[2] = {(uint64_t)Kb, (uint64_t)M}, sa[1] = {(uint64_t)Kb};
    const uint64_t db[3] = {(uint64_t)Kb, (uint64_t)N, wg ? 1ull : (uint64_t)G},
                   sb[2] = {(uint64_t)Kb, (uint64_t)N * Kb};
    MOE_REQUIRE(make_map(&tmA, a, 2, da, sa) && make_map(&tmB, b, 3, db, sb), MOE_ERR_CUDA);
    Params p{};
    p.mode = mode;
    p.epi = epilogue;
    p.G = G;
    p.N = N;
    p.M = M;
    p.K = wg ? K : Kb;      // WGRAD: rows (the offsets' bound); FWD/DGRAD: bytes (k-steps of 128)
    p.gofs = gofs;
    p.a_sf = a_sf;
    p.b_sf = b_sf;
    // NVFP4 scale atoms: [k-step][row tile][4 x 512]; FWD/DGRAD: B's rows are
    // the G*N rows of the [G][N] weight operand
    p.a_sf_kstride = (M / 128) * 2048;
    p.b_sf_kstride = (wg ? 1 : (int64_t)G) * (N / 128) * 2048;
    p.b_sf_gstride = wg ? 0 : (int64_t)(N / 128) * 2048;
    p.alpha_a = a_scale;
    p.alpha_b = b_scale;
    p.d = (__nv_bfloat16*)d;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    p.band = choice.band > 0 ? choice.band : 8;
    p.n_tiles = N / 256;
    p.m_tiles = (int)(M / BM);
    p.n_out = N;
    p.ldd = N;
    const int sms = device_sm_count();
    MOE_REQUIRE(sms > 0, MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    // FWD / DGRAD run on the 1-SM kernel; MOE_GEMM_KERNEL_PAIR (or _PAIR_N128)
    // selects the CTA-pair kernel's NVFP4 instance (256 x 256 pair tiles,
    // half of B per SM), kept for measurement: at the DeepSeek-V3 shapes it
    // was slower (a group's odd last 128-row tile idles half a pair tile) and
    // on dense shapes it only matched the 1-SM kernel
    if (!wg && choice.sel > 0 && gemm_max_clusters_2sm(256) > 0) {
        CUtensorMap tmB2, tmSFA, tmSFB;
        MOE_REQUIRE(make_map(&tmB2, b, 3, db, sb, 128), MOE_ERR_CUDA);
        MOE_REQUIRE(make_sf_map(&tmSFA, a_sf, M * K / 16 / 512, 8) &&
                        make_sf_map(&tmSFB, b_sf, (int64_t)G * N * K / 16 / 512, 16),
                    MOE_ERR_CUDA);
        p.band = choice.band > 0 ? choice.band : 4;
        const int64_t upper_pairs = (M / BM) * (int64_t)p.n_tiles;
        const int clusters = (int)std::min<int64_t>(std::max<int64_t>(upper_pairs, 1), gemm_max_clusters_2sm(256));
        if (gemm_launch_2sm_nvf4(epilogue, tmA, tmB2, tmSFA, tmSFB, p, clusters, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        MOE_CHECK_LAUNCH();
        return MOE_OK;
    }
    const int64_t tiles = wg ? (int64_t)G * p.m_tiles * p.n_tiles : (M / BM) * p.n_tiles;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, sms));
    if (epilogue == MOE_EPI_NONE_F32)
        k_grouped_gemm<256, MOE_EPI_NONE_F32, FMT_NVF4><<<grid, THREADS, Cfg<256, FMT_NVF4>::SMEM_BYTES, s>>>(tmA, tmB, p);
    else
        k_grouped_gemm<256, MOE_EPI_NONE, FMT_NVF4><<<grid, THREADS, Cfg<256, FMT_NVF4>::SMEM_BYTES, s>>>(tmA, tmB, p);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t grouped_gemm_nvfp4(int mode, const uint8_t* a, const uint8_t* a_sf, const float* a_scale,
                                           const uint8_t* b, const uint8_t* b_sf, const float* b_scale,
                                           const int32_t* gofs, int G, int64_t M, int N, int64_t K, int epilogue,
                                           void* d, int32_t* err, void* stream) {
    return grouped_gemm_nvfp4_ex(mode, a, a_sf, a_scale, b, b_sf, b_scale, gofs, G, M, N, K, epilogue, d, nullptr,
                                 err, stream);
}

namespace moe {
namespace gg {
// One thread waits, with the GEMM kernels' bounded wait, on an mbarrier
// that nothing arrives at: the wait must give up after timeout_ns, record
// MOE_ERR_DEVICE_TIMEOUT and return, leaving the context usable.
__global__ void k_wait_selftest(uint64_t timeout_ns, int32_t* err, int32_t* completed) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Params p{};
        p.err = err;
        p.timeout_ns = timeout_ns;
        *completed = mbar_wait(smem_u32(&bar), 0u, p, &abort_flag) ? 1 : 0;
    }
}
}  // namespace gg
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(uint64_t timeout_ns, int32_t* err, int32_t* completed,
                                                  void* stream) {
    MOE_REQUIRE(err && completed && timeout_ns > 0 && timeout_ns <= 10000000000ull, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    gg::k_wait_selftest<<<1, 32, 0, (cudaStream_t)stream>>>(timeout_ns, err, completed);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

