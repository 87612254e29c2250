// MXFP8 grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// [TE-JAX] "Optimization 1: Grouped GEMM": every expert's GEMM runs in one
// kernel call, each over its actual rows, and only regions with valid tokens
// are computed; "On Blackwell ... MXFP8 block scaling for expert matmuls".
// [TE-JAX] Figure 3: the grouped MLP is two grouped GEMMs (up/gate, down);
// the SwiGLU between them is fused into the up/gate epilogue here.
//
// Design (one persistent CTA per SM, 256 threads, warp-specialised):
//   warp 0 lane 0   TMA producer: per k-step one 128x128 A box, two 128x128
//                   B boxes (N = 256) and the three 512-byte scale atoms, all
//                   completing on one mbarrier (expect_tx).
//   warp 1          allocates 512 TMEM columns; lane 0 issues
//                   tcgen05.cp (scales smem -> TMEM) and 4 x
//                   tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) per
//                   k-step into a 128x256 fp32 accumulator in TMEM.
//   warps 4..7      epilogue: tcgen05.ld of their 32 TMEM lanes, bf16
//                   conversion, fused SwiGLU / SwiGLU-backward, stores.
// The tile list is derived on the device from the group offsets (multiples
// of 128), so a tile never straddles two groups and the host never sees the
// counts.  Every mbarrier wait is bounded: on timeout the CTA records
// MOE_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <stdlib.h>

#include "common.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128, BK = 128;             // BK in fp8 elements (= bytes)
constexpr int SFA_STAGE = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SF_STRIDE = 16;       // TMEM columns of scales per pipeline stage
constexpr int BAND = 8;                       // m-tiles per raster band
constexpr int MAX_G = 1024;
constexpr int EPI_WARPS = 8;                  // two warps per TMEM lane quarter
constexpr int THREADS = 128 + 32 * EPI_WARPS;

// Tile configurations.  BN = 128 keeps two accumulators in TMEM so the
// epilogue of one tile overlaps the mainloop of the next; BN = 256 halves
// the A re-reads but has a single accumulator.
template <int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int NACC = BN_ == 128 ? 2 : 1;
    static constexpr int STAGES = BN_ == 128 ? 6 : 4;
    static constexpr int A_STAGE = BM * BK;
    static constexpr int B_STAGE = BN_ * BK;
    static constexpr int SFB_STAGE = (BN_ / 128) * 512;
    static constexpr uint32_t STAGE_TX = A_STAGE + B_STAGE + SFA_STAGE + SFB_STAGE;
    // TMEM: accumulators at [0, NACC*BN); stage s scales at SF0 + 16 s (A: 4
    // columns, B: BN/32 columns), so a stage's scale columns are rewritten
    // only after the MMAs that read them completed.
    static constexpr uint32_t SF0 = NACC * BN_;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
    static constexpr int NBAR = 2 * STAGES + 2 * NACC + 1;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
    static constexpr int OFF_GOFS = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = OFF_GOFS + (MAX_G + 1) * 4 + 1024;   // + alignment slack
    static_assert(SF0 + STAGES * TMEM_SF_STRIDE <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Params {
    int mode, epi, G;
    int N;
    int64_t M, K;
    int n_tiles;        // tiles along N
    int m_tiles;        // WGRAD: tiles along M per group
    const int32_t* gofs;
    const uint8_t* a_sf;
    const uint8_t* b_sf;
    int64_t a_sf_kstride, b_sf_kstride, b_sf_gstride;   // bytes
    __nv_bfloat16* d;
    __nv_bfloat16* d2;
    const __nv_bfloat16* aux;
    int32_t* err;
    uint64_t timeout_ns;
};

// ---------------------------------------------------------------- PTX ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Returns false when the CTA is aborting (timeout here or
// elsewhere in the CTA).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Params& p, volatile int* abort_flag) {
    uint64_t start = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (start == 0) {
                start = now;
            } else if (now - start > p.timeout_ns) {
                set_err(p.err, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128
// bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}
// Descriptor of a 32-row x 16-byte scale atom (no swizzle, 8-row core
// matrices of 128 contiguous bytes).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor: E4M3 x E4M3, fp32 accumulate, K-major A and B,
// E8M0 scales, M = 128, N = BN, scale byte `sf_id` of each 32-bit TMEM cell.
template <int BN>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
    return (sf_id << 4) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) | ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// 32 lanes x 32 columns of fp32 from TMEM (this warp's lane quarter).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 floats -> 32 bf16 (RNE) -> four 16-byte stores.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float* v) {
    uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = pack8(v + 8 * q);
}
__device__ __forceinline__ void load_row32(const __nv_bfloat16* src, float* v) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) unpack8(__ldg(s + q), v + 8 * q);
}

// ------------------------------------------------------------ schedule ----

struct Tile {
    int g;            // group of the B operand (FWD/DGRAD) / output group (WGRAD)
    int64_t a_row;    // first row of the A box
    int b_row;        // first row of the B boxes (BN consecutive rows)
    int64_t kbeg;     // first k-step (units of 128 along K)
    int nk;           // number of k-steps
    int64_t out_row;  // first output row
    int nt;           // tile index along N
};

__device__ __forceinline__ void band_decode(int64_t l, int64_t mtiles, int ntiles, int64_t& mt, int& nt) {
    const int64_t band_tiles = (int64_t)BAND * ntiles;
    const int64_t b = l / band_tiles;
    const int64_t rem = l - b * band_tiles;
    const int64_t m0 = b * BAND;
    const int64_t bw = min((int64_t)BAND, mtiles - m0);
    mt = m0 + rem % bw;
    nt = (int)(rem / bw);
}

__device__ __forceinline__ int find_group(const int* s_gofs, int G, int64_t row) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)s_gofs[mid] <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int BN>
__device__ __forceinline__ void get_tile(const Params& p, const int* s_gofs, int64_t total_mt, int64_t t, Tile& ti) {
    int64_t mt;
    int nt;
    if (p.mode != MOE_GEMM_WGRAD) {
        band_decode(t, total_mt, p.n_tiles, mt, nt);
        const int64_t row = mt * BM;
        ti.g = find_group(s_gofs, p.G, row);
        ti.a_row = row;
        ti.out_row = row;
        ti.kbeg = 0;
        ti.nk = (int)(p.K / BK);
    } else {
        const int64_t tpg = (int64_t)p.m_tiles * p.n_tiles;
        const int g = (int)(t / tpg);
        band_decode(t - (int64_t)g * tpg, p.m_tiles, p.n_tiles, mt, nt);
        ti.g = g;
        ti.a_row = mt * BM;
        ti.kbeg = s_gofs[g] / BK;
        ti.nk = (s_gofs[g + 1] - s_gofs[g]) / BK;
        ti.out_row = (int64_t)g * p.M + mt * BM;
    }
    ti.b_row = nt * BN;
    ti.nt = nt;
}

// --------------------------------------------------------------- kernel ----

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
    using C = Cfg<BN>;
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
    for (int i = threadIdx.x; i <= p.G; i += THREADS) s_gofs[i] = p.gofs[i];
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
            get_tile<BN>(p, s_gofs, total_mt, t, ti);
            const int gB = p.mode == MOE_GEMM_WGRAD ? 0 : ti.g;
            for (int ks = 0; ks < ti.nk; ++ks) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, p, abort_flag)) {
                    aborted = true;
                    break;
                }
                const int64_t kg = ti.kbeg + ks;
                const int kx = (int)(kg * BK);
                const uint32_t fb = full_bar(stage);
                mbar_expect_tx(fb, C::STAGE_TX);
                tma_load_2d(smem_u32(sA + stage * C::A_STAGE), &tmA, kx, (int)ti.a_row, fb);
                const uint8_t* sfa = p.a_sf + kg * p.a_sf_kstride + (ti.a_row / 128) * 512;
                const uint8_t* sfb = p.b_sf + (int64_t)gB * p.b_sf_gstride + kg * p.b_sf_kstride;
                bulk_load(smem_u32(sSFA + stage * SFA_STAGE), sfa, 512, fb);
#pragma unroll
                for (int h = 0; h < BN / 128; ++h) {
                    const int brow = ti.b_row + 128 * h;
                    tma_load_3d(smem_u32(sB + stage * C::B_STAGE + h * 16384), &tmB, kx, brow, gB, fb);
                    bulk_load(smem_u32(sSFB + stage * C::SFB_STAGE + h * 512), sfb + (int64_t)(brow / 128) * 512,
                              512, fb);
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
            get_tile<BN>(p, s_gofs, total_mt, t, ti);
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
                const uint32_t t_sfa = tmem_base + C::SF0 + TMEM_SF_STRIDE * stage;
                const uint32_t t_sfb = t_sfa + 4;
                tc_cp_sf(t_sfa, desc_sf(smem_u32(sSFA + stage * SFA_STAGE)));
#pragma unroll
                for (int h = 0; h < BN / 128; ++h)
                    tc_cp_sf(t_sfb + 4 * h, desc_sf(smem_u32(sSFB + stage * C::SFB_STAGE + 512 * h)));
                const uint64_t adesc = desc_sw128(smem_u32(sA + stage * C::A_STAGE));
                const uint64_t bdesc = desc_sw128(smem_u32(sB + stage * C::B_STAGE));
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk) {
                    // advance 32 bytes along K inside the 128-byte swizzled row
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
            get_tile<BN>(p, s_gofs, total_mt, t, ti);
            const int64_t row = ti.out_row + quarter * 32 + lane;
            if (ti.nk == 0) {   // WGRAD of an empty group: the gradient is zero
                float z[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) z[i] = 0.f;
                for (int c = 0; c < BN / 64; ++c)
                    store_row32(p.d + row * p.N + ti.nt * BN + half * (BN / 2) + 32 * c, z);
                continue;
            }
            if (!mbar_wait(tfull_bar(acc), acc_phase, p, abort_flag)) break;
            tc_fence_after();
            const uint32_t tacc = lane_base + (uint32_t)(acc * BN);
            float v[32];
            if (p.epi == MOE_EPI_SWIGLU) {
                // B rows interleave gate/up in 64-row chunks: accumulator
                // columns [128q, 128q+64) are gate, [128q+64, 128q+128) up
                const int64_t N = p.N, f = p.N / 2;
                for (int u = half * (BN / 128); u < (half + 1) * (BN / 128); ++u) {
                    const int q = u >> 1, c = u & 1;
                    float up[32], h[32];
                    tmem_ld32(tacc + 128 * q + 32 * c, v);
                    tmem_ld32(tacc + 128 * q + 64 + 32 * c, up);
                    const int64_t hcol = (int64_t)ti.nt * (BN / 2) + 64 * q + 32 * c;
                    store_row32(p.d + row * N + hcol, v);
                    store_row32(p.d + row * N + f + hcol, up);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float s = 1.f / (1.f + expf(-v[i]));
                        h[i] = v[i] * s * up[i];
                    }
                    store_row32(p.d2 + row * f + hcol, h);
                }
            } else if (p.epi == MOE_EPI_SWIGLU_BWD) {
                const int64_t N = p.N, ld = 2 * (int64_t)p.N;
                for (int c = 0; c < BN / 64; ++c) {
                    float g[32], u[32], dg[32], du[32];
                    const int col32 = half * (BN / 2) + 32 * c;
                    tmem_ld32(tacc + col32, v);          // dH
                    const int64_t col = (int64_t)ti.nt * BN + col32;
                    load_row32(p.aux + row * ld + col, g);
                    load_row32(p.aux + row * ld + N + col, u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float s = 1.f / (1.f + expf(-g[i]));
                        dg[i] = v[i] * u[i] * s * (1.f + g[i] * (1.f - s));
                        du[i] = v[i] * g[i] * s;
                    }
                    store_row32(p.d + row * ld + col, dg);
                    store_row32(p.d + row * ld + N + col, du);
                }
            } else {
                for (int c = 0; c < BN / 64; ++c) {
                    const int col32 = half * (BN / 2) + 32 * c;
                    tmem_ld32(tacc + col32, v);
                    store_row32(p.d + row * p.N + (int64_t)ti.nt * BN + col32, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
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

cudaError_t gemm_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gg::k_grouped_gemm<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gg::Cfg<128>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gg::k_grouped_gemm<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gg::Cfg<256>::SMEM_BYTES);
}

// Tile width used by grouped_gemm_mxfp8: 256 (one TMEM accumulator; on
// GB300 the 128-wide MMA is operand-bandwidth bound and ran at ~0.64x the
// 256-wide rate) unless the environment variable MOE_GEMM_BN=128 selects the
// double-buffered 128-wide tile (kept for measurement).
static int gemm_bn() {
    static int bn = [] {
        const char* e = getenv("MOE_GEMM_BN");
        return (e != nullptr && atoi(e) == 128) ? 128 : 256;
    }();
    return bn;
}

// rank-2/3 uint8 tensor map, 128x128 boxes, 128-byte swizzle
static bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes) {
    cuuint64_t gdim[3], gstr[2];
    cuuint32_t box[3] = {128, 128, 1}, estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
    for (int i = 0; i < rank - 1; ++i) gstr[i] = strides_bytes[i];
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), gdim, gstr,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t grouped_gemm_mxfp8(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                           const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G, int64_t M,
                                           int N, int64_t K, int epilogue, const void* epi_aux, void* d, void* d2,
                                           int32_t* err, void* stream) {
    using namespace gg;
    MOE_REQUIRE(mode == MOE_GEMM_FWD || mode == MOE_GEMM_DGRAD || mode == MOE_GEMM_WGRAD, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(a && a_sf && b && b_sf && gofs && d, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(G >= 1 && G <= MAX_G && M > 0 && N > 0 && K > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(M % 128 == 0 && K % BK == 0 && N % 128 == 0, MOE_ERR_UNSUPPORTED);
    const int BN = (gemm_bn() == 256 && N % 256 == 0) ? 256 : 128;
    MOE_REQUIRE(K <= 0x7FFFFF80LL && M <= 0x7FFFFF80LL, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(a) && moe_aligned16(b) && moe_aligned16(a_sf) && moe_aligned16(b_sf) &&
                    moe_aligned16(d) && (d2 == nullptr || moe_aligned16(d2)) &&
                    (epi_aux == nullptr || moe_aligned16(epi_aux)),
                MOE_ERR_ALIGNMENT);
    if (mode == MOE_GEMM_WGRAD) {
        MOE_REQUIRE(epilogue == MOE_EPI_NONE, MOE_ERR_INVALID_ARG);
    } else {
        MOE_REQUIRE(b_layout == MOE_B_GNK || b_layout == MOE_B_NGK, MOE_ERR_INVALID_ARG);
        MOE_REQUIRE(epilogue == MOE_EPI_NONE || epilogue == MOE_EPI_SWIGLU || epilogue == MOE_EPI_SWIGLU_BWD,
                    MOE_ERR_INVALID_ARG);
        if (epilogue == MOE_EPI_SWIGLU) MOE_REQUIRE(d2 != nullptr, MOE_ERR_INVALID_ARG);
        if (epilogue == MOE_EPI_SWIGLU_BWD) MOE_REQUIRE(epi_aux != nullptr, MOE_ERR_INVALID_ARG);
    }
    MOE_REQUIRE(device_initialized() && g_encode != nullptr, MOE_ERR_NOT_INITIALIZED);

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
    p.aux = (const __nv_bfloat16*)epi_aux;
    p.err = err;
    p.timeout_ns = 2000000000ull;   // 2 s per wait
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
    if (BN == 256)
        k_grouped_gemm<256><<<grid, THREADS, Cfg<256>::SMEM_BYTES, (cudaStream_t)stream>>>(tmA, tmB, p);
    else
        k_grouped_gemm<128><<<grid, THREADS, Cfg<128>::SMEM_BYTES, (cudaStream_t)stream>>>(tmA, tmB, p);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
