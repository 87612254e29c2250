// Shared pieces of the grouped MXFP8 GEMM kernels (1-SM and 2-SM): launch
// parameters, PTX wrappers for TMA / mbarrier / tcgen05, the tile schedule
// helpers and the fused epilogues.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128, BK = 128;             // BK in fp8 elements (= bytes)
constexpr int SFA_STAGE = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SF_STRIDE = 16;       // TMEM columns of scales per pipeline stage
constexpr int MAX_G = 1024;
constexpr int EPI_WARPS = 8;                  // two warps per TMEM lane quarter
// CTA-pair kernel, TMA-store epilogue: each epilogue warp stages 32-row x
// kEpiBoxCols-column bf16 boxes (64: 4 KB, 128-byte swizzle; 32: 2 KB,
// 64-byte swizzle, which leaves room for a sixth pipeline stage)
constexpr int kEpiBoxCols = 32;
constexpr int kEpiBoxBytes = 32 * kEpiBoxCols * 2;
constexpr int THREADS = 128 + 32 * EPI_WARPS;

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
    int band;           // m-tiles per raster band (consecutive tiles share the B tile)
    int group_bands;    // 1-SM FWD / DGRAD: bands restart at each group's first m-tile
    int tma_store;      // pair kernel, BN = 256, MOE_EPI_NONE: write D through the TMA (tensor map tmD)
    // WGRAD on the pair kernel: only the groups whose row count r passes
    // the filter (moe_gemm_opts_t: hi == 0: r >= lo; lo < hi: lo <= r < hi;
    // 0 < hi <= lo: r < hi or r >= lo); wg_filter = 0 when every group is
    // computed
    int wg_filter, wg_lo, wg_hi;
    // bf16 operands (kind::f16): the columns of D that exist (n_out <= N,
    // the rest of the tile is not stored) and D's row stride in elements
    int n_out;
    int64_t ldd;
    int k_ceil;         // bf16 operands: the last k-step may reach past K (TMA fills zeros)
    // MOE_EPI_SWIGLU: MXFP8 of h (NULL = not produced): rowwise codes
    // [M, N/2] + scale atoms, columnwise (transposed) codes [N/2, M] + atoms
    uint8_t* hq_r;
    uint8_t* hs_r;
    uint8_t* hq_c;
    uint8_t* hs_c;
    // NVFP4 operands: the per-tensor fp32 scales of A and B (device
    // pointers); the epilogue multiplies the accumulator by their product
    const float* alpha_a;
    const float* alpha_b;
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
// A waiting thread may sleep up to this long in one poll (it is woken when
// the phase completes), so idle warps do not take issue slots.
constexpr uint32_t kSuspendNs = 50000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Returns false when the CTA is aborting (timeout here or
// elsewhere in the CTA).
// Besides the time limit (p.timeout_ns of the global nanosecond timer) a
// wait gives up after kMaxSpin polls, so it ends even if the timer stood still.
constexpr uint32_t kMaxSpin = 1u << 22;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Params& p, volatile int* abort_flag) {
    uint64_t start = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
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

// TMA store of a shared-memory box (bulk-group completion) and its fences.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
                 "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk stores committed so far have finished reading shared memory
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// all but the most recent committed bulk store have finished reading shared memory
__device__ __forceinline__ void bulk_wait_group_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// the bulk stores committed so far are complete
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// this thread's shared-memory writes become visible to the TMA (async proxy)
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
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

// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B, fp32
// D, both K-major, M = 128, N = BN.
template <int BN>
__device__ __forceinline__ uint32_t make_idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::mxf4nvf4 with E2M1 A and B
// (format 1), UE4M3 block scales (scale format 0, scale_vec::4X: four
// 16-element blocks per K = 64 MMA, so the scale ids are 0), fp32 D, both
// K-major, M = 128, N = BN.
template <int BN>
__device__ __forceinline__ uint32_t make_idesc_nvf4() {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
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

// 32 lanes x 32 columns of 32-bit words from TMEM (this warp's lane
// quarter), without waiting: the registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }


// Two bf16 (RNE) packed into one word, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
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

__device__ __forceinline__ void band_decode(int64_t l, int64_t mtiles, int ntiles, int band, int64_t& mt, int& nt) {
    const int64_t band_tiles = (int64_t)band * ntiles;
    const int64_t b = l / band_tiles;
    const int64_t rem = l - b * band_tiles;
    const int64_t m0 = b * band;
    const int64_t bw = min((int64_t)band, mtiles - m0);
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

// 32 bytes (one L2 sector) per store.
__device__ __forceinline__ void st_global_v8(void* dst, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// ------------------------------------------------------------- epilogue ----

// MXFP8 of one 32-column block of h in the SwiGLU epilogue ([TE-JAX] "What
// specialized optimizations...": group-aware MXFP8 quantization; fused into
// the producing GEMM).  `ph` holds this thread's 32 bf16-rounded h values of
// row `row`, columns [hcol, hcol + 32) (hcol % 32 == 0), as 16 packed pairs;
// the warp's 32 lanes hold 32 consecutive rows starting at a multiple of 32.
// Rowwise: the block is this thread's own 32 values.  Columnwise: each
// column's block is the warp's 32 rows (tiles start at group offsets, which
// are multiples of 128, so a block never crosses a group), reduced with one
// warp max per column.  Codes, scales and layouts are those of
// mxfp8_gather_quantize for h.
__device__ __forceinline__ void h_quant_chunk(const Params& p, int64_t row, int64_t hcol, const uint32_t* ph,
                                              int lane) {
    const int64_t f = p.N / 2, M = p.M;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = __vmaxu2(m, ph[i] & 0x7FFF7FFFu);
    const uint32_t sb = e8m0_scale_byte(__uint_as_float(max(m & 0xFFFFu, m >> 16) << 16));
    const float inv = e8m0_inv_scale(sb);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = ph[2 * i], b = ph[2 * i + 1];
        const uint32_t lo = cvt_e4m3x2(__uint_as_float(a << 16) * inv, __uint_as_float(a & 0xFFFF0000u) * inv);
        const uint32_t hi = cvt_e4m3x2(__uint_as_float(b << 16) * inv, __uint_as_float(b & 0xFFFF0000u) * inv);
        q[i] = lo | (hi << 16);
    }
    st_global_v8(p.hq_r + row * f + hcol, q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
    const int64_t blk = hcol >> 5;
    p.hs_r[((blk >> 2) * (M >> 7) + (row >> 7)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (blk & 3)] =
        (uint8_t)sb;
    uint32_t my_sb = 0;      // scale of column hcol + lane
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t a = ph[i];
        const uint32_t s0 = e8m0_scale_byte(__uint_as_float(__reduce_max_sync(0xFFFFFFFFu, a & 0x7FFFu) << 16));
        const uint32_t s1 =
            e8m0_scale_byte(__uint_as_float(__reduce_max_sync(0xFFFFFFFFu, (a >> 16) & 0x7FFFu) << 16));
        if (lane == 2 * i) my_sb = s0;
        if (lane == 2 * i + 1) my_sb = s1;
        const uint32_t c = cvt_e4m3x2(__uint_as_float(a << 16) * e8m0_inv_scale(s0),
                                      __uint_as_float(a & 0xFFFF0000u) * e8m0_inv_scale(s1));
        p.hq_c[(hcol + 2 * i) * M + row] = (uint8_t)(c & 0xFFu);
        p.hq_c[(hcol + 2 * i + 1) * M + row] = (uint8_t)(c >> 8);
    }
    const int64_t col = hcol + lane, rb = (row - lane) >> 5;
    p.hs_c[((rb >> 2) * (f >> 7) + (col >> 7)) * 512 + (col & 31) * 16 + ((col >> 5) & 3) * 4 + (rb & 3)] =
        (uint8_t)my_sb;
}

// One TMEM accumulator of BN columns, 128 lanes: the calling warp owns lane
// quarter `quarter` (rows quarter*32 + lane of the tile) and column half
// `half` of the tile.  `row` is this thread's output row, `nt` the tile
// index along N.  Writes bf16 results with the fused activation.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t tacc, int64_t row, int nt, int half) {
    float v[32];
    if constexpr (EPI == MOE_EPI_SWIGLU) {
        // B rows interleave gate/up in 64-row chunks: accumulator columns
        // [128q, 128q+64) are gate, [128q+64, 128q+128) up
        const int64_t N = p.N, f = p.N / 2;
        for (int u = half * (BN / 128); u < (half + 1) * (BN / 128); ++u) {
            const int q = u >> 1, c = u & 1;
            float up[32], h[32];
            tmem_ld32(tacc + 128 * q + 32 * c, v);
            tmem_ld32(tacc + 128 * q + 64 + 32 * c, up);
            const int64_t hcol = (int64_t)nt * (BN / 2) + 64 * q + 32 * c;
            store_row32(p.d + row * N + hcol, v);
            store_row32(p.d + row * N + f + hcol, up);
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = v[i] * fast_sigmoid(v[i]) * up[i];
            if (p.d2 != nullptr) store_row32(p.d2 + row * f + hcol, h);
            if (p.hq_r != nullptr) {
                uint32_t ph[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) ph[i] = pack_bf16x2(h[2 * i], h[2 * i + 1]);
                h_quant_chunk(p, row, hcol, ph, (int)(threadIdx.x & 31));
            }
        }
    } else if constexpr (EPI == MOE_EPI_SWIGLU_BWD) {
        const int64_t N = p.N, ld = 2 * (int64_t)p.N;
        for (int c = 0; c < BN / 64; ++c) {
            float g[32], u[32], dg[32], du[32];
            const int col32 = half * (BN / 2) + 32 * c;
            tmem_ld32(tacc + col32, v);          // dH
            const int64_t col = (int64_t)nt * BN + col32;
            load_row32(p.aux + row * ld + col, g);
            load_row32(p.aux + row * ld + N + col, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                swiglu_bwd_pair(g[i], u[i], v[i], dg[i], du[i]);
            }
            store_row32(p.d + row * ld + col, dg);
            store_row32(p.d + row * ld + N + col, du);
        }
    } else if constexpr (EPI == MOE_EPI_NONE_F32) {
        float* out = reinterpret_cast<float*>(p.d) + row * p.ldd + (int64_t)nt * BN;
        for (int c = 0; c < BN / 64; ++c) {
            const int col32 = half * (BN / 2) + 32 * c;
            tmem_ld32(tacc + col32, v);
            uint32_t* o = reinterpret_cast<uint32_t*>(out + col32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (nt * BN + col32 + 8 * q < p.n_out)
                    st_global_v8(o + 8 * q, __float_as_uint(v[8 * q]), __float_as_uint(v[8 * q + 1]),
                                 __float_as_uint(v[8 * q + 2]), __float_as_uint(v[8 * q + 3]),
                                 __float_as_uint(v[8 * q + 4]), __float_as_uint(v[8 * q + 5]),
                                 __float_as_uint(v[8 * q + 6]), __float_as_uint(v[8 * q + 7]));
        }
    } else {
        for (int c = 0; c < BN / 64; ++c) {
            const int col32 = half * (BN / 2) + 32 * c;
            tmem_ld32(tacc + col32, v);
            store_row32(p.d + row * p.N + (int64_t)nt * BN + col32, v);
        }
    }
}


// Register-staged epilogue for 256-wide tiles: the calling thread drains
// its 128 accumulator columns (column half `half`) into registers as packed
// bf16 (two TMEM loads in flight per wait), calls release() so the MMA warp
// can reuse TMEM, and only then writes global memory, overlapped with the
// next tile's MMAs.  SwiGLU-backward has its own pipelined epilogue below.
// SCALED (NVFP4 operands, MOE_EPI_NONE / MOE_EPI_NONE_F32 only): every
// accumulator is multiplied by alpha_a * alpha_b before it is stored.
template <bool SCALED>
__device__ __forceinline__ void scale_acc(const Params& p, uint32_t* r) {
    if constexpr (SCALED) {
        const float al = __fmul_rn(__ldg(p.alpha_a), __ldg(p.alpha_b));
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), al));
    }
}

template <int EPI, bool SCALED = false, typename Release>
__device__ __forceinline__ void epilogue_tile_staged(const Params& p, uint32_t tacc, int64_t row, int nt, int half,
                                                     Release release) {
    static_assert(!SCALED || EPI == MOE_EPI_NONE || EPI == MOE_EPI_NONE_F32, "scaled epilogue: plain outputs only");
    uint32_t ra[32], rb[32];
    if constexpr (EPI == MOE_EPI_SWIGLU) {
        // units u = 2*half, 2*half+1: gate columns [128q + 32c, +32) and up
        // columns [128q + 64 + 32c, +32) with q = u / 2 = half, c = u % 2.
        // Chunk 0 is converted while chunk 1 is still in TMEM and written
        // after the release, so at most one chunk of fp32 is live.
        const int64_t N = p.N, f = p.N / 2;
        const int64_t hcol = (int64_t)nt * 128 + 64 * half;     // 64 h columns of this thread
        uint32_t* dg = reinterpret_cast<uint32_t*>(p.d + row * N + hcol);
        uint32_t* du = reinterpret_cast<uint32_t*>(p.d + row * N + f + hcol);
        uint32_t* dh = reinterpret_cast<uint32_t*>(p.d2 + row * f + hcol);
        uint32_t pg[16], pu[16], ph[16];
        auto convert = [&]() {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float g0 = __uint_as_float(ra[2 * i]), g1 = __uint_as_float(ra[2 * i + 1]);
                const float u0 = __uint_as_float(rb[2 * i]), u1 = __uint_as_float(rb[2 * i + 1]);
                pg[i] = pack_bf16x2(g0, g1);
                pu[i] = pack_bf16x2(u0, u1);
                ph[i] = pack_bf16x2(g0 * fast_sigmoid(g0) * u0, g1 * fast_sigmoid(g1) * u1);
            }
        };
        auto store = [&](int c) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int o = 16 * c + 8 * q;
                st_global_v8(dg + o, pg[8 * q], pg[8 * q + 1], pg[8 * q + 2], pg[8 * q + 3], pg[8 * q + 4],
                             pg[8 * q + 5], pg[8 * q + 6], pg[8 * q + 7]);
                st_global_v8(du + o, pu[8 * q], pu[8 * q + 1], pu[8 * q + 2], pu[8 * q + 3], pu[8 * q + 4],
                             pu[8 * q + 5], pu[8 * q + 6], pu[8 * q + 7]);
                if (p.d2 != nullptr)
                    st_global_v8(dh + o, ph[8 * q], ph[8 * q + 1], ph[8 * q + 2], ph[8 * q + 3], ph[8 * q + 4],
                                 ph[8 * q + 5], ph[8 * q + 6], ph[8 * q + 7]);
            }
        };
        tmem_ld32_issue(tacc + 128 * half, ra);
        tmem_ld32_issue(tacc + 128 * half + 64, rb);
        tmem_wait_ld();
        convert();
        tmem_ld32_issue(tacc + 128 * half + 32, ra);
        tmem_ld32_issue(tacc + 128 * half + 96, rb);
        tmem_wait_ld();
        release();
        store(0);
        uint32_t ph0[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) ph0[i] = ph[i];
        convert();
        store(1);
        if (p.hq_r != nullptr) {      // MXFP8 of h, after the stores, with no fp32 accumulator live
            const int lane = (int)(threadIdx.x & 31);
            h_quant_chunk(p, row, hcol, ph0, lane);
            h_quant_chunk(p, row, hcol + 32, ph, lane);
        }
    } else if constexpr (EPI == MOE_EPI_NONE_F32) {
        // fp32 out: each 32-column chunk is stored as it is drained; only
        // columns < n_out exist (row stride ldd), in 8-column groups
        const int col0 = nt * 256 + 128 * half;
        uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<float*>(p.d) + row * p.ldd + col0);
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
            tmem_ld32_issue(tacc + 128 * half + 32 * c, ra);
            tmem_ld32_issue(tacc + 128 * half + 32 * (c + 1), rb);
            tmem_wait_ld();
            if (c == 2) release();
            scale_acc<SCALED>(p, ra);
            scale_acc<SCALED>(p, rb);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (col0 + 32 * c + 8 * q < p.n_out)
                    st_global_v8(out + 32 * c + 8 * q, ra[8 * q], ra[8 * q + 1], ra[8 * q + 2], ra[8 * q + 3],
                                 ra[8 * q + 4], ra[8 * q + 5], ra[8 * q + 6], ra[8 * q + 7]);
                if (col0 + 32 * (c + 1) + 8 * q < p.n_out)
                    st_global_v8(out + 32 * (c + 1) + 8 * q, rb[8 * q], rb[8 * q + 1], rb[8 * q + 2], rb[8 * q + 3],
                                 rb[8 * q + 4], rb[8 * q + 5], rb[8 * q + 6], rb[8 * q + 7]);
            }
        }
    } else {
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
            tmem_ld32_issue(tacc + 128 * half + 32 * c, ra);
            tmem_ld32_issue(tacc + 128 * half + 32 * (c + 1), rb);
            tmem_wait_ld();
            if (c == 2) release();
            scale_acc<SCALED>(p, ra);
            scale_acc<SCALED>(p, rb);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                pk[16 * c + i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
                pk[16 * (c + 1) + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
            }
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.d + row * p.N + (int64_t)nt * 256 + 128 * half);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            st_global_v8(dst + 8 * q, pk[8 * q], pk[8 * q + 1], pk[8 * q + 2], pk[8 * q + 3], pk[8 * q + 4],
                         pk[8 * q + 5], pk[8 * q + 6], pk[8 * q + 7]);
    }
}

// TMA-store epilogue for 256-wide tiles without activation: the warp drains
// its 32 rows x 128 columns into registers as packed bf16 and releases TMEM
// (as epilogue_tile_staged), then writes 32 x kEpiBoxCols boxes through
// its staging buffer `buf` (kEpiBoxBytes, 1024-byte aligned, swizzled as
// the tensor map says) with TMA stores.  The warp's stores are
// asynchronous and the buffer is reused once the previous store has read
// it.  `row0` is the warp's first
// output row.
template <typename Release>
__device__ __forceinline__ void epilogue_tile_tma(const CUtensorMap* tmD, uint32_t buf, uint32_t tacc, int64_t row0,
                                                  int nt, int half, int lane, Release release) {
    uint32_t ra[32], rb[32], pk[64];
#pragma unroll
    for (int c = 0; c < 4; c += 2) {
        tmem_ld32_issue(tacc + 128 * half + 32 * c, ra);
        tmem_ld32_issue(tacc + 128 * half + 32 * (c + 1), rb);
        tmem_wait_ld();
        if (c == 2) release();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[16 * c + i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
            pk[16 * (c + 1) + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
        }
    }
    // box rows of kEpiBoxCols * 2 bytes; 16-byte chunk c of row r sits at
    // c ^ (r % 8) (128-byte swizzle) or c ^ ((r / 2) % 4) (64-byte swizzle),
    // conflict-free for the row-per-lane stores either way
    constexpr int CH = kEpiBoxCols / 8;                 // 16-byte chunks per row
    const uint32_t rowaddr = buf + (uint32_t)lane * (uint32_t)(kEpiBoxCols * 2);
    const uint32_t sw = CH == 8 ? (uint32_t)(lane & 7) : (uint32_t)((lane >> 1) & 3);
#pragma unroll
    for (int j = 0; j < 128 / kEpiBoxCols; ++j) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int w = (kEpiBoxCols / 2) * j + 4 * c;
            st_shared_v4(rowaddr + (((uint32_t)c ^ sw) << 4), pk[w], pk[w + 1], pk[w + 2], pk[w + 3]);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmD, buf, nt * 256 + 128 * half + kEpiBoxCols * j, (int)row0);
            bulk_commit_group();
        }
    }
}

// Zero fill of an empty group's 256-wide weight-gradient tile through the
// warp's own staging box: once the box's earlier stores have read it, the
// warp writes zeros into it and stores it four times (the 32-column boxes of
// its column half).  The next use of the box for data waits for these
// stores first, as it waits for any earlier one.
__device__ __forceinline__ void epilogue_zero_tma256(const CUtensorMap* tmD, uint32_t buf, int64_t row0, int nt,
                                                     int half, int lane) {
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    const uint32_t rowaddr = buf + (uint32_t)lane * (uint32_t)(kEpiBoxCols * 2);
#pragma unroll
    for (int c = 0; c < kEpiBoxCols / 8; ++c) st_shared_v4(rowaddr + 16u * c, 0u, 0u, 0u, 0u);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < 128 / kEpiBoxCols; ++j) {
            tma_store_2d(tmD, buf, nt * 256 + 128 * half + kEpiBoxCols * j, (int)row0);
            bulk_commit_group();
        }
    }
}

// TMA-store epilogue for the 224-wide weight-gradient tiles of the CTA-pair
// kernel (two accumulators, plain bf16 output).  The tile's 224 columns are
// seven 32-column chunks: the warps of column half 0 drain chunks 0-3, those
// of half 1 chunks 4-6, into packed bf16 registers; then TMEM is released
// and the chunks go out as 32 x 32 boxes through the warp's two staging
// buffers `buf` and `buf + kEpiBoxBytes` in turn, across tiles (`nbox`
// counts the warp's boxes, so consecutive boxes always use different
// buffers and a buffer is rewritten only once the store issued from it two
// boxes earlier has read it).  Boxes at or past column N (the last tile of
// an N that 224 does not divide) are not stored.
template <typename Release>
__device__ __forceinline__ void epilogue_tile_tma224(const CUtensorMap* tmD, uint32_t buf, uint32_t tacc,
                                                     int64_t row0, int nt, int half, int lane, int N,
                                                     uint32_t& nbox, Release release) {
    static_assert(kEpiBoxCols == 32, "224-wide tiles are stored as 32-column boxes");
    const int c0 = 4 * half;
    const int nch = half == 0 ? 4 : 3;
    uint32_t ra[32], rb[32], pk[64];
    tmem_ld32_issue(tacc + 32 * c0, ra);
    tmem_ld32_issue(tacc + 32 * (c0 + 1), rb);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        pk[i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
        pk[16 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
    }
    if (nch == 4) {
        tmem_ld32_issue(tacc + 32 * (c0 + 2), ra);
        tmem_ld32_issue(tacc + 32 * (c0 + 3), rb);
        tmem_wait_ld();
        release();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[32 + i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
            pk[48 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
        }
    } else {
        tmem_ld32_issue(tacc + 32 * (c0 + 2), ra);
        tmem_wait_ld();
        release();
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[32 + i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
    }
    constexpr int CH = kEpiBoxCols / 8;                 // 16-byte chunks per box row
    const uint32_t rowaddr = buf + (uint32_t)lane * (uint32_t)(kEpiBoxCols * 2);
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);    // 64-byte swizzle
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int col = nt * 224 + 32 * (c0 + j);
        if (j >= nch || col >= N) break;                // warp-uniform
        if (lane == 0) bulk_wait_group_read1();
        __syncwarp();
        const uint32_t bj = (nbox++ & 1u) * (uint32_t)kEpiBoxBytes;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int w = 16 * j + 4 * c;
            st_shared_v4(rowaddr + bj + (((uint32_t)c ^ sw) << 4), pk[w], pk[w + 1], pk[w + 2], pk[w + 3]);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmD, buf + bj, col, (int)row0);
            bulk_commit_group();
        }
    }
}

// SwiGLU-backward epilogue, software-pipelined: the bf16 gate/up values of
// a 32-column chunk (a_pre, global memory) are loaded one chunk ahead, the
// first chunk before the accumulator is ready (swiglu_bwd_prefetch), so the
// TMEM accumulator is held only for the TMEM loads and the arithmetic.
struct ApreChunk {
    uint4 g[4], u[4];   // 32 bf16 gate, 32 bf16 up
};
template <int BN>
__device__ __forceinline__ void swiglu_bwd_prefetch(const Params& p, int64_t row, int nt, int half, int c,
                                                    ApreChunk& a) {
    const int64_t N = p.N, ld = 2 * (int64_t)p.N;
    const int64_t col = (int64_t)nt * BN + half * (BN / 2) + 32 * c;
    const uint4* sg = reinterpret_cast<const uint4*>(p.aux + row * ld + col);
    const uint4* su = reinterpret_cast<const uint4*>(p.aux + row * ld + N + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        a.g[q] = __ldg(sg + q);
        a.u[q] = __ldg(su + q);
    }
}
// L2 prefetch of the gate/up values a thread's epilogue reads for a tile
// (issued one tile ahead, so that the loads of swiglu_bwd_prefetch hit L2).
template <int BN>
__device__ __forceinline__ void swiglu_bwd_prefetch_l2(const Params& p, int64_t row, int nt, int half) {
    const int64_t N = p.N, ld = 2 * (int64_t)p.N;
    const int64_t col = (int64_t)nt * BN + half * (BN / 2);
    const char* g = reinterpret_cast<const char*>(p.aux + row * ld + col);
    const char* u = reinterpret_cast<const char*>(p.aux + row * ld + N + col);
#pragma unroll
    for (int i = 0; i < BN; i += 128) {      // BN / 2 columns = BN bytes per operand
        asm volatile("prefetch.global.L2 [%0];" ::"l"(g + i));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(u + i));
    }
}
__device__ __forceinline__ uint32_t uint4_word(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
template <int BN, typename Release>
__device__ __forceinline__ void epilogue_swiglu_bwd(const Params& p, uint32_t tacc, int64_t row, int nt, int half,
                                                    Release release, ApreChunk& a) {
    constexpr int NC = BN / 64;             // 32-column chunks per thread
    const int64_t N = p.N, ld = 2 * (int64_t)p.N;
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        tmem_ld32_issue(tacc + half * (BN / 2) + 32 * c, r);     // dH
        tmem_wait_ld();
        if (c == NC - 1) release();
        ApreChunk nx;
        if (c + 1 < NC) swiglu_bwd_prefetch<BN>(p, row, nt, half, c + 1, nx);
        uint32_t pdg[16], pdu[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t gw = uint4_word(a.g[i >> 2], i & 3), uw = uint4_word(a.u[i >> 2], i & 3);
            float dg[2], du[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float g = __uint_as_float(e ? (gw & 0xFFFF0000u) : (gw << 16));
                const float u = __uint_as_float(e ? (uw & 0xFFFF0000u) : (uw << 16));
                const float dh = __uint_as_float(r[2 * i + e]);
                swiglu_bwd_pair(g, u, dh, dg[e], du[e]);
            }
            pdg[i] = pack_bf16x2(dg[0], dg[1]);
            pdu[i] = pack_bf16x2(du[0], du[1]);
        }
        const int64_t col = (int64_t)nt * BN + half * (BN / 2) + 32 * c;
        uint32_t* og = reinterpret_cast<uint32_t*>(p.d + row * ld + col);
        uint32_t* ou = reinterpret_cast<uint32_t*>(p.d + row * ld + N + col);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            st_global_v8(og + 8 * q, pdg[8 * q], pdg[8 * q + 1], pdg[8 * q + 2], pdg[8 * q + 3], pdg[8 * q + 4],
                         pdg[8 * q + 5], pdg[8 * q + 6], pdg[8 * q + 7]);
            st_global_v8(ou + 8 * q, pdu[8 * q], pdu[8 * q + 1], pdu[8 * q + 2], pdu[8 * q + 3], pdu[8 * q + 4],
                         pdu[8 * q + 5], pdu[8 * q + 6], pdu[8 * q + 7]);
        }
        if (c + 1 < NC) a = nx;
    }
}

// WGRAD of an empty group: the gradient is the empty sum, zero.
template <int BN>
__device__ __forceinline__ void epilogue_zero(const Params& p, int64_t row, int nt, int half) {
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0.f;
    for (int c = 0; c < BN / 64; ++c) store_row32(p.d + row * p.N + (int64_t)nt * BN + half * (BN / 2) + 32 * c, z);
}

// Zero fill of an empty group's weight-gradient tile through TMA stores of a
// shared-memory box of zeros (32 rows x kEpiBoxCols columns, written once at
// kernel start): the 32-column boxes of column half `half` of a BN-wide tile
// (224: chunks 0-3 and 4-6), boxes at or past column N skipped.  One lane
// issues the stores; they complete with the warp's other bulk stores.  (With
// many empty groups, as under skewed routing, per-thread zero stores took
// 1.3 ms more of the DeepSeek-V3 step's weight gradients.)
template <int BN>
__device__ __forceinline__ void epilogue_zero_tma(const CUtensorMap* tmD, uint32_t zbox, int64_t row0, int nt,
                                                  int half, int lane, int N) {
    static_assert(kEpiBoxCols == 32, "32-column zero boxes");
    const int c0 = 4 * half;
    const int nch = BN == 224 && half == 1 ? 3 : 4;
    if (lane == 0) {
        for (int j = 0; j < nch; ++j) {
            const int col = nt * BN + 32 * (c0 + j);
            if (col < N) {
                tma_store_2d(tmD, zbox, col, (int)row0);
                bulk_commit_group();
            }
        }
    }
    __syncwarp();
}


}  // namespace gg

// Host side (gemm.cu)
cudaError_t gemm_set_attributes_2sm();   // gemm2sm.cu
int gemm_max_clusters_2sm(int bn);        // co-resident CTA pairs for N = bn pair tiles
cudaError_t gemm_launch_2sm(int bn, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmSFA, const CUtensorMap& tmSFB, const CUtensorMap& tmD,
                            const gg::Params& p, int clusters, cudaStream_t stream);
cudaError_t gemm_launch_2sm_nvf4(int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const CUtensorMap& tmSFA, const CUtensorMap& tmSFB, const gg::Params& p,
                                 int clusters, cudaStream_t stream);
}  // namespace moe
