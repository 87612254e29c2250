// MXFP8 quantization: 1x32 blocks, E8M0 scales, E4M3 codes.
// [TE-JAX] "What specialized optimizations are required for dropless MoE?"
// (a group-aware MXFP8 quantization) and "Optimization 1" (MXFP8 block
// scaling); [CH1] "低精度格式的缩放机制" (per-block scaling, blocks of 32) and
// §1.1 (E4M3 = 1+4+3 bits).
//
// Both kernels work on 128x128 tiles so that one CTA produces exactly one
// 512-byte scale atom (the tensor core's native scale order, see moe.h) and
// writes it with one coalesced 512-byte store.
#include "common.cuh"

namespace moe {

constexpr int kQT = 128;   // tile edge

__device__ bool gofs_valid(const int32_t* gofs, int G, int64_t rows) {
    if (gofs[0] != 0) return false;
    for (int g = 0; g < G; ++g) {
        const int a = gofs[g], b = gofs[g + 1];
        if (b < a || (b & 127) != 0) return false;
    }
    return (int64_t)gofs[G] <= rows;
}

// Rowwise: tile = 128 rows x 128 cols.  256 threads; a thread owns 8
// consecutive elements, four neighbouring threads form one 32-element block.
// canon: scales in the canonical row-major [rows, cols / 32] layout instead
// of the atom layout.
__global__ void __launch_bounds__(256) k_quant_rows(const uint4* __restrict__ x, int64_t rows, int cols,
                                                    const int32_t* __restrict__ gofs, int G,
                                                    uint2* __restrict__ codes, uint8_t* __restrict__ scales,
                                                    int canon, int32_t* err) {
    __shared__ __align__(16) uint8_t s_atom[512];
    const int64_t r0 = (int64_t)blockIdx.y * kQT;
    const int c0 = blockIdx.x * kQT;
    if (gofs != nullptr && r0 >= (int64_t)gofs[G]) return;
    const int tc = threadIdx.x & 15;         // 16 threads per row (8 elements each)
    const int tr = threadIdx.x >> 4;         // 16 rows per pass
    const int cols8 = cols >> 3;
    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int64_t r = r0 + tr + 16 * p;
        v[p] = __ldg(x + r * cols8 + (c0 >> 3) + tc);
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(v[p], f);
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const uint32_t b = e8m0_scale_byte(amax);
        const float inv = e8m0_inv_scale(b);
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = cvt_e4m3x2(f[2 * i] * inv, f[2 * i + 1] * inv);
        const int rl = tr + 16 * p;          // local row
        const int64_t r = r0 + rl;
        codes[(r * cols + c0) / 8 + tc] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
        if ((tc & 3) == 0) {
            const int kb = tc >> 2;          // local block 0..3
            if (canon)
                scales[r * (cols / 32) + c0 / 32 + kb] = (uint8_t)b;
            else
                s_atom[(rl & 31) * 16 + ((rl >> 5) & 3) * 4 + kb] = (uint8_t)b;
        }
    }
    __syncthreads();
    if (!canon && threadIdx.x < 32) {
        const int64_t atom = (int64_t)(c0 / kQT) * (rows / kQT) + r0 / kQT;
        reinterpret_cast<uint4*>(scales + atom * 512)[threadIdx.x] = reinterpret_cast<const uint4*>(s_atom)[threadIdx.x];
    }
    (void)err;
}

// Columnwise, group-aware: a CTA owns 128 input columns (= 128 output rows)
// and kColTiles consecutive 128-row tiles (4 blocks of 32 rows each, all in
// one group because groups start at multiples of 128).  Output is
// transposed: codes [cols, rows]; each CTA writes kColTiles*128 contiguous
// bytes of each of its 128 output rows, and the CTAs that run together
// (consecutive blockIdx.x) continue the same rows, so the writes stream.
// With `glu`, output rows interleave the two column halves in 64-row chunks:
// output rows [128 j, 128 j + 64) are input columns [64 j, 64 j + 64) and
// rows [128 j + 64, 128 j + 128) are input columns [cols/2 + 64 j, ... + 64).
constexpr int kColTiles = 4;

// With batch_rows = Kg > 0 the input is G equal groups of Kg rows and the
// output is batched per group: codes [G][cols][Kg] (each group's transposed
// block contiguous) and scales in the atom layout of the [G*cols, Kg] matrix.
// canon: scales in the canonical row-major layout of the output matrix
// ([cols, rows], or [G * cols, batch_rows] batched) instead of the atoms.
__global__ void __launch_bounds__(256) k_quant_cols(const uint4* __restrict__ x, int64_t rows, int cols,
                                                    const int32_t* __restrict__ gofs, int G, int glu,
                                                    int64_t batch_rows, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ scales, int canon, int32_t* err) {
    // the input tile [row][col] and, after it has been consumed, the output
    // codes tile [col][row] share one buffer
    __shared__ __align__(16) uint8_t s_buf[kQT * (kQT + 8) * 2];
    __shared__ __align__(16) uint8_t s_atom[512];
    auto s_x = reinterpret_cast<uint16_t(*)[kQT + 8]>(s_buf);
    auto s_q = reinterpret_cast<uint8_t(*)[kQT + 16]>(s_buf);
    __shared__ int s_ok;
    const int ct = blockIdx.y;                       // column tile = output row tile
    const int c0 = ct * kQT;
    int64_t row_end = rows;
    if (gofs != nullptr) {
        if (threadIdx.x == 0) {
            const bool ok = gofs_valid(gofs, G, rows);
            s_ok = ok;
            if (!ok && blockIdx.x == 0 && blockIdx.y == 0) set_err(err, MOE_ERR_BAD_OFFSETS);
        }
        __syncthreads();
        if (!s_ok) return;
        row_end = (int64_t)gofs[G];
    }
    const int cols8 = cols >> 3;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int it = 0; it < kColTiles; ++it) {
        const int64_t r0 = ((int64_t)blockIdx.x * kColTiles + it) * kQT;
        if (r0 >= row_end) break;
        // load 128 x 128 bf16: 16 uint4 per row, 2048 uint4, 8 per thread
        uint4 v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int idx = threadIdx.x + 256 * p;
            const int rl = idx >> 4, cv = idx & 15;
            const int src8 = glu ? (cv < 8 ? 8 * ct + cv : (cols >> 4) + 8 * ct + cv - 8) : (c0 >> 3) + cv;
            v[p] = __ldg(x + (r0 + rl) * cols8 + src8);
        }
        __syncthreads();      // previous iteration is done with the buffer
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int idx = threadIdx.x + 256 * p;
            *reinterpret_cast<uint4*>(&s_x[idx >> 4][(idx & 15) * 8]) = v[p];
        }
        __syncthreads();
        // each thread: 2 (column, block) pairs; a warp covers 32 consecutive columns
        uint32_t w[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int pair = warp + 8 * h;        // 0..15
            const int col = (pair & 3) * 32 + lane;
            const int blk = pair >> 2;            // 32-row block 0..3
            float f[32];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                f[i] = bf16_bits_to_float(s_x[blk * 32 + i][col]);
                amax = fmaxf(amax, fabsf(f[i]));
            }
            const uint32_t b = e8m0_scale_byte(amax);
            const float inv = e8m0_inv_scale(b);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo = cvt_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv);
                const uint32_t hi = cvt_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv);
                w[h][i] = lo | (hi << 16);
            }
            if (canon) {
                // output row and 32-row block of this (column, block) pair
                int64_t orow, ob, kout;
                if (batch_rows > 0) {
                    const int64_t g = r0 / batch_rows;
                    orow = g * cols + c0 + col;
                    ob = (r0 - g * batch_rows) / 32 + blk;
                    kout = batch_rows;
                } else {
                    orow = c0 + col;
                    ob = r0 / 32 + blk;
                    kout = rows;
                }
                scales[orow * (kout / 32) + ob] = (uint8_t)b;
            } else {
                s_atom[(col & 31) * 16 + ((col >> 5) & 3) * 4 + blk] = (uint8_t)b;
            }
        }
        __syncthreads();     // every thread is done reading the input tile
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int pair = warp + 8 * h;
            const int col = (pair & 3) * 32 + lane;
            const int blk = pair >> 2;
            uint4* dst = reinterpret_cast<uint4*>(&s_q[col][blk * 32]);
            dst[0] = make_uint4(w[h][0], w[h][1], w[h][2], w[h][3]);
            dst[1] = make_uint4(w[h][4], w[h][5], w[h][6], w[h][7]);
        }
        __syncthreads();
        // write codes: output row (c0 + col), bytes [r0, r0 + 128): 8 uint4 per row
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int idx = threadIdx.x + 256 * p;    // 0..1023
            const int col = idx >> 3, cv = idx & 7;
            const uint4 q = *reinterpret_cast<const uint4*>(&s_q[col][cv * 16]);
            int64_t dst;
            if (batch_rows > 0) {
                const int64_t g = r0 / batch_rows, kk = r0 - g * batch_rows;
                dst = ((g * cols + c0 + col) * batch_rows) + kk + cv * 16;
            } else {
                dst = (int64_t)(c0 + col) * rows + r0 + cv * 16;
            }
            *reinterpret_cast<uint4*>(codes + dst) = q;
        }
        if (!canon && threadIdx.x < 32) {
            int64_t atom;
            if (batch_rows > 0) {
                const int64_t g = r0 / batch_rows, kk = r0 - g * batch_rows;
                atom = (kk / kQT) * ((int64_t)G * (cols / kQT)) + g * (cols / kQT) + ct;
            } else {
                atom = (r0 / kQT) * (int64_t)(cols / kQT) + ct;
            }
            reinterpret_cast<uint4*>(scales + atom * 512)[threadIdx.x] =
                reinterpret_cast<const uint4*>(s_atom)[threadIdx.x];
        }
    }
}

}  // namespace moe

using namespace moe;

// padded group offsets of an mxfp8_group_quantize output: gofs, or g * Kg
// for the batched axes
__global__ void k_padded_offsets(const int32_t* __restrict__ gofs, int G, int64_t batch_rows, int32_t* out) {
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g <= G; g += gridDim.x * blockDim.x)
        out[g] = batch_rows > 0 ? (int32_t)(g * batch_rows) : gofs[g];
}

extern "C" moe_status_t mxfp8_group_quantize_ex(const void* x, int64_t rows, int cols, int axis,
                                                const int32_t* gofs, int G, uint8_t* codes, uint8_t* scales,
                                                int32_t* padded_offsets, int scale_layout, int32_t* err,
                                                void* stream) {
    MOE_REQUIRE(x && codes && scales, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(scale_layout == MOE_SF_ATOMS || scale_layout == MOE_SF_CANONICAL, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows >= 0 && cols > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows % kQT == 0 && cols % kQT == 0, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(rows / kQT <= 65535 && cols / kQT <= 65535, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(axis == MOE_QUANT_ROWWISE || axis == MOE_QUANT_COLWISE_GROUPED || axis == MOE_QUANT_COLWISE_GLU ||
                    axis == MOE_QUANT_COLWISE_BATCHED || axis == MOE_QUANT_COLWISE_BATCHED_GLU,
                MOE_ERR_INVALID_ARG);
    const bool batched = axis == MOE_QUANT_COLWISE_BATCHED || axis == MOE_QUANT_COLWISE_BATCHED_GLU;
    if (batched) MOE_REQUIRE(G >= 1 && rows % G == 0 && (rows / G) % kQT == 0, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(gofs == nullptr || (G >= 1 && G <= 4096), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(padded_offsets == nullptr || batched || gofs != nullptr, MOE_ERR_INVALID_ARG);
    const int canon = scale_layout == MOE_SF_CANONICAL ? 1 : 0;
    MOE_REQUIRE(moe_aligned16(x) && moe_aligned16(codes) && moe_aligned16(scales), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    if (padded_offsets != nullptr) {
        k_padded_offsets<<<1, 256, 0, s>>>(gofs, G, batched ? rows / G : 0, padded_offsets);
        MOE_CHECK_LAUNCH();
    }
    if (rows == 0) return MOE_OK;
    if (axis == MOE_QUANT_ROWWISE) {
        dim3 grid(cols / kQT, (unsigned)(rows / kQT));
        k_quant_rows<<<grid, 256, 0, s>>>((const uint4*)x, rows, cols, gofs, G, (uint2*)codes, scales, canon, err);
    } else {
        dim3 grid((unsigned)((rows / kQT + kColTiles - 1) / kColTiles), cols / kQT);
        const int glu = (axis == MOE_QUANT_COLWISE_GLU || axis == MOE_QUANT_COLWISE_BATCHED_GLU) ? 1 : 0;
        // batched outputs use equal groups of rows / G rows (gofs, if given, only bounds the rows read)
        k_quant_cols<<<grid, 256, 0, s>>>((const uint4*)x, rows, cols, batched ? nullptr : gofs, G, glu,
                                          batched ? rows / G : 0, codes, scales, canon, err);
    }
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t mxfp8_group_quantize(const void* x, int64_t rows, int cols, int axis, const int32_t* gofs,
                                             int G, uint8_t* codes, uint8_t* scales, int32_t* err, void* stream) {
    return mxfp8_group_quantize_ex(x, rows, cols, axis, gofs, G, codes, scales, nullptr, MOE_SF_ATOMS, err, stream);
}

// ---------------------------------------------------------------------------
// Both axes from one read, optionally gathering the rows.
//
// Row s of the (virtual) permuted matrix is
//   src[row_id[s] / k] * row_w[row_id[s]]   (rounded to bf16 when scaled)
// or zero when row_id[s] < 0 (padding); with row_id == NULL it is src[s].
// This quantizes x_perm straight from x (the local half of dispatch,
// [TE-JAX] "Optimization 2") and dy_perm = w * dout straight from dout (the
// combine backward), so neither bf16 permuted matrix is written and read
// back; h and dA are read once for both axes.
//
// A CTA owns one 128-column tile and a run of kQBRowTiles 128-row tiles: it
// checks the group offsets once (in parallel), looks up the source row and
// weight of all its rows once, and streams its row tiles through a
// two-stage cp.async pipeline (the copy of tile i+1 is in flight while tile
// i is quantized; padding rows are zero-filled by the copy), three CTAs per
// SM, three CTA barriers per tile with router weights, two without.  Block
// maxima are taken on the packed
// bf16 bits (two values per instruction); a column block is read twice from
// shared memory (maximum, then codes) to keep registers low enough for three
// CTAs per SM.  Per tile it writes the rowwise codes and scale atom of its
// 128 rows and the columnwise (transposed) codes and atom of its 128
// columns; each 32-row block of a column is one 32-byte sector of the
// transposed output, stored from the registers of the lane that encoded it.
// Consecutive CTAs take consecutive row runs of the same column tile, so the CTAs
// resident at a time cover all rows of one or two column tiles: a gathered
// source row, read by up to k row tiles, is re-read from L2 (one column tile
// of x is 6 MB at T = 24576).
namespace moe {

constexpr int kQBThreads = 256;
constexpr int kQBRowTiles = 8;                      // row tiles per CTA (at most)
constexpr int kQBInBytes = kQT * kQT * 2;           // one bf16 tile, unpadded
constexpr int kQBSmem = 2 * kQBInBytes + 2 * 512 + 512 + kQBRowTiles * kQT * (4 + 4);

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, uint32_t nbytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(g), "r"(nbytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// amax of packed bf16 pairs, one instruction per word: each half of the
// result has the larger magnitude of the two inputs' halves (and the XOR
// of their signs, so mask the sign bits with 0x7FFF7FFF before use; the
// masked halves are bf16 bits of the block maxima).  Finite inputs.
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// 32 bytes to a 32-byte aligned global address in one instruction
__device__ __forceinline__ void st_global_32B(void* dst, const uint32_t* q) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(q[0]), "r"(q[1]),
                 "r"(q[2]), "r"(q[3]), "r"(q[4]), "r"(q[5]), "r"(q[6]), "r"(q[7])
                 : "memory");
}
__device__ __forceinline__ float bf16_bits_lo(uint32_t w) { return __uint_as_float(w << 16); }

// The scales of a 128-column tile of the transposed (columnwise) output,
// staged as one atom (column cl, blocks 0..3 at (cl % 32) * 16 +
// ((cl / 32) % 4) * 4), written in the tile-224 layout instead (moe.h):
// column c0 + cl is row c = c0 + cl of the [R, C] transposed matrix, in
// 224-row tile c / 224; its four block scales stay one 4-byte word.  One
// warp, four columns per lane.
__device__ __forceinline__ void store_col_scales_t224(uint8_t* sf_c, const uint8_t* s_atom, int64_t kb, int64_t c0,
                                                      int R, int lane) {
    const int64_t T = (R + 223) / 224;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int cl = lane + 32 * q;
        const int64_t c = c0 + cl;
        const int64_t t = c / 224;
        const int rp = (int)(c - 224 * t);
        const uint32_t w = *reinterpret_cast<const uint32_t*>(s_atom + (cl & 31) * 16 + ((cl >> 5) & 3) * 4);
        *reinterpret_cast<uint32_t*>(sf_c + (kb * T + t) * 1024 + (rp >> 7) * 512 + (rp & 31) * 16 +
                                     ((rp >> 5) & 3) * 4) = w;
    }
}
__device__ __forceinline__ float bf16_bits_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Scaling by 2^-e, two bf16 values per instruction.  The product of a bf16
// value and a power of two is exact whenever it is a normal bf16, and every
// element of a block scales to at most 448 in magnitude; a product below the
// smallest normal bf16 (2^-126) is far below half the smallest E4M3
// subnormal (2^-10), so it encodes as a signed zero either way.  The codes
// are therefore those of the fp32 product x * 2^-e.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// bf16x2 pair of 2^(127 - b) for the scale bytes of the low and high halves
// (the bf16 bits of e8m0_inv_scale)
__device__ __forceinline__ uint32_t inv_bf16x2(uint32_t b_lo, uint32_t b_hi) {
    return ((254u - b_lo) << 7) | ((254u - b_hi) << 23);
}
// E4M3 codes of the two (already scaled) bf16 values of a word, low in byte 0
__device__ __forceinline__ uint32_t e4m3x2_of(uint32_t w) { return cvt_e4m3x2(bf16_bits_lo(w), bf16_bits_hi(w)); }

__global__ void __launch_bounds__(kQBThreads, 3) k_quant_both(const uint16_t* __restrict__ src, int64_t src_rows,
                                                              int cols, int k, const int32_t* __restrict__ row_id,
                                                              const float* __restrict__ row_w,
                                                              const int32_t* __restrict__ gofs, int G,
                                                              int64_t rows, uint2* __restrict__ codes_r,
                                                              uint8_t* __restrict__ sf_r,
                                                              uint8_t* __restrict__ codes_c,
                                                              uint8_t* __restrict__ sf_c,
                                                              uint8_t* __restrict__ sf_c224,
                                                              int32_t* err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* s_in = reinterpret_cast<uint16_t*>(smem);                       // [2][128][128]
    uint8_t* s_atom_r = smem + 2 * kQBInBytes;                                // [2][512]
    uint8_t* s_atom_c = s_atom_r + 2 * 512;                                   // [512]
    int32_t* s_src = reinterpret_cast<int32_t*>(s_atom_c + 512);              // [kQBRowTiles * 128]
    float* s_w = reinterpret_cast<float*>(s_src + kQBRowTiles * kQT);         // [kQBRowTiles * 128]
    const int tid = threadIdx.x;
    const int ct = blockIdx.y;
    const int64_t rt0 = (int64_t)blockIdx.x * kQBRowTiles;
    const int ntiles = cols / kQT;

    // group offsets: gofs[0] == 0, monotone, multiples of 128, gofs[G] <= rows
    bool ok = true;
    for (int i = tid; i <= G; i += kQBThreads) {
        const int a = gofs[i];
        if ((a & 127) != 0 || (i == 0 && a != 0)) ok = false;
        if (i < G && gofs[i + 1] < a) ok = false;
        if (i == G && (int64_t)a > rows) ok = false;
    }
    if (!__syncthreads_and(ok)) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) set_err(err, MOE_ERR_BAD_OFFSETS);
        return;
    }
    const int nrt = (int)min((int64_t)kQBRowTiles, (int64_t)gofs[G] / kQT - rt0);   // row tiles below gofs[G]
    if (nrt <= 0) return;

    // source row and weight of every row of the CTA's row tiles, up front
    for (int j = tid; j < nrt * kQT; j += kQBThreads) {
        const int64_t s = rt0 * kQT + j;
        int64_t sr = s;
        float w = 1.f;
        if (row_id != nullptr) {
            const int id = row_id[s];
            sr = id >= 0 ? (int64_t)(id / k) : -1;
            if (sr >= src_rows) {              // not a row of src: report, read as zero
                set_err(err, MOE_ERR_INVALID_ARG);
                sr = -1;
            }
            if (sr >= 0 && row_w != nullptr) w = row_w[id];
        }
        s_src[j] = (int32_t)sr;                // < 2^31: checked on the host
        s_w[j] = w;
    }
    // Row/block assignment (copy and rowwise pass): a thread owns row qr
    // of the tile and its 32-element blocks qb and qb + 2 (4 x 16 bytes
    // each).  The 8 threads of a quarter warp hold rows qr + 32t (t = 0..3)
    // of blocks qb = 0, 1 (or 2, 3).  The tile sits in shared memory with
    // its 16-byte chunks swizzled by 32-row block: chunk c of row r is
    // stored at chunk c ^ ((r >> 5) & 3).  The rowwise 16-byte reads of a
    // quarter warp then fall on 8 distinct bank groups, and the columnwise
    // pass (one 32-row block per warp) reads with a per-thread constant
    // offset.
    const int qr = (tid >> 3) + 32 * (tid & 3), qb = (tid >> 2) & 1;
    const int qsw = (qr >> 5) & 3;
    // copy assignment (16 threads per row, 16 contiguous bytes each, so
    // every copy instruction reads whole 256-byte row segments): chunk p of
    // a thread = chunk tc of row tr + 16p
    const int tc = tid & 15, tr = tid >> 4;
    const uint32_t s_in_addr = (uint32_t)__cvta_generic_to_shared(s_in);
    auto issue = [&](int i) {
        const int buf = i & 1;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int rl = tr + 16 * p;
            const int64_t sr = s_src[i * kQT + rl];
            const uint16_t* g = src + (sr >= 0 ? sr : 0) * cols + (int64_t)ct * kQT + tc * 8;
            const int pc = tc ^ ((rl >> 5) & 3);
            cp_async16(s_in_addr + (uint32_t)(buf * kQBInBytes + (rl * kQT + pc * 8) * 2), g, sr >= 0 ? 16u : 0u);
        }
    };
    __syncthreads();                          // the gather plan is complete
    issue(0);
    cp_async_commit();
    const int lane = tid & 31, warp = tid >> 5;
    for (int i = 0; i < nrt; ++i) {
        const int b = i & 1;
        const int64_t r0 = (rt0 + i) * kQT;
        uint16_t* tile = s_in + b * (kQT * kQT);
        // the other buffer (tile i - 1) was released by the barrier that
        // ended tile i - 1: start tile i + 1 there
        if (i + 1 < nrt) issue(i + 1);
        cp_async_commit();
        cp_async_wait1();                     // this thread's copies of tile i have landed
        __syncthreads();                      // ... and every other thread's
        // rowwise, over this thread's own blocks (scaled in place first):
        // one 32-element block per step, so one scale per block and thread
        uint8_t* crow = reinterpret_cast<uint8_t*>(codes_r) + (r0 + qr) * cols + (int64_t)ct * kQT;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int qbu = qb + 2 * u;
            uint4 v[4];
            uint4* cp[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cp[j] = reinterpret_cast<uint4*>(tile + qr * kQT + (((4 * qbu + j) ^ qsw) * 8));
                v[j] = *cp[j];
            }
            if (row_w != nullptr) {
                const float w = s_w[i * kQT + qr];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float f[8];
                    unpack8(v[j], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] *= w;
                    v[j] = pack8(f);
                    *cp[j] = v[j];
                }
            }
            if (codes_r != nullptr) {
                uint32_t m = bf16x2_maxabs(bf16x2_maxabs(v[0].x, v[0].y), bf16x2_maxabs(v[0].z, v[0].w));
#pragma unroll
                for (int j = 1; j < 4; ++j)
                    m = bf16x2_maxabs(m, bf16x2_maxabs(bf16x2_maxabs(v[j].x, v[j].y), bf16x2_maxabs(v[j].z, v[j].w)));
                m &= 0x7FFF7FFFu;
                const uint32_t sb = e8m0_scale_byte(__uint_as_float(max(m & 0xFFFFu, m >> 16) << 16));
                const uint32_t s2 = inv_bf16x2(sb, sb);
                uint32_t q[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    q[2 * j] = e4m3x2_of(bf16x2_mul(v[j].x, s2)) | (e4m3x2_of(bf16x2_mul(v[j].y, s2)) << 16);
                    q[2 * j + 1] = e4m3x2_of(bf16x2_mul(v[j].z, s2)) | (e4m3x2_of(bf16x2_mul(v[j].w, s2)) << 16);
                }
                st_global_32B(crow + qbu * 32, q);   // one whole 32-byte sector
                s_atom_r[b * 512 + (qr & 31) * 16 + qsw * 4 + qbu] = (uint8_t)sb;
            }
        }
        // A: tile i, scaled in place by the router weights, is complete.
        // Without weights the rowwise pass writes nothing the columnwise
        // pass reads: the tile is complete since the barrier above.
        if (row_w != nullptr) __syncthreads();
        uint32_t w0[8], w1[8];
        const int blk = warp & 3;                       // 32-row block
        const int col = (warp >> 2) * 64 + 2 * lane;    // two columns per lane
        if (codes_c != nullptr) {
            // the block's rows are swizzled by blk: columns col, col + 1 sit
            // in chunk (col / 8) ^ blk
            const uint32_t* colp = reinterpret_cast<const uint32_t*>(tile + blk * 32 * kQT +
                                                                     (((col >> 3) ^ blk) << 3) + (col & 7));
            // pass 1: amax of both columns over the block, on packed bf16 bits,
            // in four independent chains
            uint32_t ma = 0, mb = 0, mc = 0, md = 0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                ma = bf16x2_maxabs(ma, colp[e * (kQT / 2)]);
                mb = bf16x2_maxabs(mb, colp[(e + 1) * (kQT / 2)]);
                mc = bf16x2_maxabs(mc, colp[(e + 2) * (kQT / 2)]);
                md = bf16x2_maxabs(md, colp[(e + 3) * (kQT / 2)]);
            }
            const uint32_t m = bf16x2_maxabs(bf16x2_maxabs(ma, mb), bf16x2_maxabs(mc, md)) & 0x7FFF7FFFu;
            const uint32_t b0 = e8m0_scale_byte(__uint_as_float((m & 0xFFFFu) << 16));
            const uint32_t b1 = e8m0_scale_byte(__uint_as_float(m & 0xFFFF0000u));
            const uint32_t s2 = inv_bf16x2(b0, b1);
            // pass 2: codes, two rows per conversion
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t v0 = bf16x2_mul(colp[(4 * e) * (kQT / 2)], s2);
                const uint32_t v1 = bf16x2_mul(colp[(4 * e + 1) * (kQT / 2)], s2);
                const uint32_t v2 = bf16x2_mul(colp[(4 * e + 2) * (kQT / 2)], s2);
                const uint32_t v3 = bf16x2_mul(colp[(4 * e + 3) * (kQT / 2)], s2);
                w0[e] = cvt_e4m3x2(bf16_bits_lo(v0), bf16_bits_lo(v1)) |
                        (cvt_e4m3x2(bf16_bits_lo(v2), bf16_bits_lo(v3)) << 16);
                w1[e] = cvt_e4m3x2(bf16_bits_hi(v0), bf16_bits_hi(v1)) |
                        (cvt_e4m3x2(bf16_bits_hi(v2), bf16_bits_hi(v3)) << 16);
            }
            s_atom_c[(col & 31) * 16 + ((col >> 5) & 3) * 4 + blk] = (uint8_t)b0;
            s_atom_c[((col + 1) & 31) * 16 + (((col + 1) >> 5) & 3) * 4 + blk] = (uint8_t)b1;
            // the 32 codes of each column's block are one 32-byte sector of the
            // transposed output: stored straight from registers
            uint8_t* dst = codes_c + ((int64_t)ct * kQT + col) * rows + r0 + 32 * blk;
            st_global_32B(dst, w0);
            st_global_32B(dst + rows, w1);
        }
        // B: every thread is done reading tile i (its buffer may be refilled)
        // and both atoms are complete
        __syncthreads();
        if (warp == 0) {
            if (codes_r != nullptr) {
                const int64_t atom = (int64_t)ct * (rows / kQT) + r0 / kQT;
                reinterpret_cast<uint4*>(sf_r + atom * 512)[lane] =
                    reinterpret_cast<const uint4*>(s_atom_r + b * 512)[lane];
            }
        } else if (warp == 1 || warp == 2) {
            // columnwise scales: the tile-224 layout (warp 1) and/or the atom
            // layout (warp 1 if it is the only one, else warp 2)
            const bool atoms = sf_c != nullptr && (warp == 2) == (sf_c224 != nullptr);
            if (warp == 1 && sf_c224 != nullptr)
                store_col_scales_t224(sf_c224, s_atom_c, r0 / kQT, (int64_t)ct * kQT, cols, lane);
            if (atoms) {
                const int64_t atom = (r0 / kQT) * (int64_t)ntiles + ct;
                reinterpret_cast<uint4*>(sf_c + atom * 512)[lane] = reinterpret_cast<const uint4*>(s_atom_c)[lane];
            }
        }
        // the atoms are rewritten no earlier than the next tile's barrier A
        // (s_atom_c) or two tiles on (s_atom_r, double-buffered)
    }
}

// ---------------------------------------------------------------------------
// SwiGLU backward fused with the two-axis quantization of its output.
//
// dA = [dgate | dup] ([M, 2f]) with dgate = dH*u*s*(1+g*(1-s)), dup = dH*g*s,
// s = sigmoid(g), from the dgrad GEMM's fp32 dH [M, f] and the forward's
// bf16 a_pre = [g | u] [M, 2f]; every element is rounded to bf16 and then
// quantized exactly as mxfp8_gather_quantize quantizes a stored dA (rowwise
// and group-columnwise), so dA never exists in bf16 in memory.  Moving this
// elementwise step out of the dgrad GEMM's epilogue frees that GEMM's single
// TMEM accumulator sooner; this pass has to touch dA anyway.
//
// A CTA owns one 128-column tile c0 of dH (hence output column tiles c0 of
// dgate and f + c0 of dup, which need the same dH, g and u) and a run of
// kQBRowTiles row tiles.  Per row tile each thread loads its eight 8-element
// chunks of dH, g and u (two chunks ahead of the one it computes: the pass
// streams from DRAM, and two CTAs per SM with 128 registers keep more bytes
// in flight than three with one chunk ahead), computes dgate and dup,
// quantizes them rowwise from registers and stages them in two
// shared-memory tiles for the columnwise blocks, done as in k_quant_both
// (the atoms double-buffered by tile parity, two CTA barriers per tile).
constexpr int kSBSmem = 2 * kQBInBytes + 8 * 512;

__device__ __forceinline__ uint2 quant_row_chunk(uint4 v, uint32_t& sb_out) {
    uint32_t m = bf16x2_maxabs(bf16x2_maxabs(v.x, v.y), bf16x2_maxabs(v.z, v.w));
    m = bf16x2_maxabs(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = bf16x2_maxabs(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2)) & 0x7FFF7FFFu;
    const uint32_t sb = e8m0_scale_byte(__uint_as_float(max(m & 0xFFFFu, m >> 16) << 16));
    const uint32_t s2 = inv_bf16x2(sb, sb);
    const uint32_t q0 = e4m3x2_of(bf16x2_mul(v.x, s2));
    const uint32_t q1 = e4m3x2_of(bf16x2_mul(v.y, s2));
    const uint32_t q2 = e4m3x2_of(bf16x2_mul(v.z, s2));
    const uint32_t q3 = e4m3x2_of(bf16x2_mul(v.w, s2));
    sb_out = sb;
    return make_uint2(q0 | (q1 << 16), q2 | (q3 << 16));
}

// columnwise block (32 rows `blk`, columns col and col + 1) of a bf16 tile in
// shared memory: codes of the two columns (8 words each) and scale bytes
__device__ __forceinline__ void quant_col_block(const uint16_t* tile, int blk, int col, uint32_t* w0, uint32_t* w1,
                                                uint32_t& b0, uint32_t& b1) {
    const uint32_t* colp = reinterpret_cast<const uint32_t*>(tile + blk * 32 * kQT + col);
    uint32_t m = 0;
#pragma unroll 8
    for (int e = 0; e < 32; ++e) m = bf16x2_maxabs(m, colp[e * (kQT / 2)]);
    m &= 0x7FFF7FFFu;
    b0 = e8m0_scale_byte(__uint_as_float((m & 0xFFFFu) << 16));
    b1 = e8m0_scale_byte(__uint_as_float(m & 0xFFFF0000u));
    const uint32_t s2 = inv_bf16x2(b0, b1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t v0 = bf16x2_mul(colp[(4 * e) * (kQT / 2)], s2);
        const uint32_t v1 = bf16x2_mul(colp[(4 * e + 1) * (kQT / 2)], s2);
        const uint32_t v2 = bf16x2_mul(colp[(4 * e + 2) * (kQT / 2)], s2);
        const uint32_t v3 = bf16x2_mul(colp[(4 * e + 3) * (kQT / 2)], s2);
        w0[e] = cvt_e4m3x2(bf16_bits_lo(v0), bf16_bits_lo(v1)) |
                (cvt_e4m3x2(bf16_bits_lo(v2), bf16_bits_lo(v3)) << 16);
        w1[e] = cvt_e4m3x2(bf16_bits_hi(v0), bf16_bits_hi(v1)) |
                (cvt_e4m3x2(bf16_bits_hi(v2), bf16_bits_hi(v3)) << 16);
    }
}

__global__ void __launch_bounds__(kQBThreads, 2) k_swiglu_bwd_quant(const float* __restrict__ dH,
                                                                    const uint16_t* __restrict__ a_pre, int f,
                                                                    const int32_t* __restrict__ gofs, int G,
                                                                    int64_t rows, uint16_t* __restrict__ dA,
                                                                    uint2* __restrict__ codes_r,
                                                                    uint8_t* __restrict__ sf_r,
                                                                    uint8_t* __restrict__ codes_c,
                                                                    uint8_t* __restrict__ sf_c,
                                                                    uint8_t* __restrict__ sf_c224,
                                                                    int32_t* err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* tiles = reinterpret_cast<uint16_t*>(smem);           // [2][128][128]: dgate, dup
    // atoms of the dgate / dup tiles, double-buffered by tile parity so the
    // next tile's passes may write while this tile's atoms are stored
    uint8_t* const s_atom_r0 = smem + 2 * kQBInBytes;              // [2 parities][2 tiles][512]
    uint8_t* const s_atom_c0 = s_atom_r0 + 4 * 512;                // [2 parities][2 tiles][512]
    const int tid = threadIdx.x;
    const int ct = blockIdx.y;                                     // column tile of dH / g / u
    const int64_t c0 = (int64_t)ct * kQT;
    const int64_t rt0 = (int64_t)blockIdx.x * kQBRowTiles;
    const int64_t F = f, F2 = 2 * (int64_t)f;
    const int out_tiles = (int)(F2 / kQT);
    auto octile = [&](int t) { return t == 0 ? ct : ct + f / kQT; };   // output column tiles: dgate, dup

    bool ok = true;
    for (int i = tid; i <= G; i += kQBThreads) {
        const int a = gofs[i];
        if ((a & 127) != 0 || (i == 0 && a != 0)) ok = false;
        if (i < G && gofs[i + 1] < a) ok = false;
        if (i == G && (int64_t)a > rows) ok = false;
    }
    if (!__syncthreads_and(ok)) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) set_err(err, MOE_ERR_BAD_OFFSETS);
        return;
    }
    const int nrt = (int)min((int64_t)kQBRowTiles, (int64_t)gofs[G] / kQT - rt0);
    if (nrt <= 0) return;

    const int tc = tid & 15, tr = tid >> 4;
    const int lane = tid & 31, warp = tid >> 5;
    // raw inputs of one chunk: 8 dH (fp32), 8 g and 8 u (bf16) of row
    // r0 + tr + 16p, columns c0 + tc*8 ...
    auto load = [&](int64_t r0, int p, float4& h0, float4& h1, uint4& gw, uint4& uw) {
        const int64_t r = r0 + tr + 16 * p;
        const float4* hp = reinterpret_cast<const float4*>(dH + r * F + c0 + tc * 8);
        h0 = __ldg(hp);
        h1 = __ldg(hp + 1);
        gw = __ldg(reinterpret_cast<const uint4*>(a_pre + r * F2 + c0 + tc * 8));
        uw = __ldg(reinterpret_cast<const uint4*>(a_pre + r * F2 + F + c0 + tc * 8));
    };
    // two chunks in flight: chunk p in set p & 1 while chunk p + 1 is loaded
    // in the other and chunk p + 2 into temporaries
    float4 H0[2], H1[2];
    uint4 GW[2], UW[2];
    for (int i = 0; i < nrt; ++i) {
        const int64_t r0 = (rt0 + i) * kQT;
        uint8_t* const s_atom_r = s_atom_r0 + (i & 1) * 1024;
        uint8_t* const s_atom_c = s_atom_c0 + (i & 1) * 1024;
        // dgate / dup of this thread's chunks: rowwise codes from registers,
        // bf16 values into the two tiles; the loads of chunks p + 1 and
        // p + 2 are in flight while chunk p is computed
        if (i == 0) {                         // later tiles: prefetched by the previous one
            load(r0, 0, H0[0], H1[0], GW[0], UW[0]);
            load(r0, 1, H0[1], H1[1], GW[1], UW[1]);
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int rl = tr + 16 * p;
            const int64_t r = r0 + rl;
            float4 nh0, nh1;
            uint4 ngw, nuw;
            if (p + 2 < 8) load(r0, p + 2, nh0, nh1, ngw, nuw);
            const float4 h0 = H0[p & 1], h1 = H1[p & 1];
            const uint4 gw = GW[p & 1], uw = UW[p & 1];
            float gf[8], uf[8], dg[8], du[8];
            const float hf[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
            unpack8(gw, gf);
            unpack8(uw, uf);
#pragma unroll
            for (int e = 0; e < 8; ++e) swiglu_bwd_pair(gf[e], uf[e], hf[e], dg[e], du[e]);
            const uint4 vg = pack8(dg), vu = pack8(du);
            if (dA != nullptr) {
                *reinterpret_cast<uint4*>(dA + r * F2 + c0 + tc * 8) = vg;
                *reinterpret_cast<uint4*>(dA + r * F2 + F + c0 + tc * 8) = vu;
            }
            uint32_t sg, su;
            const uint2 qg = quant_row_chunk(vg, sg);
            const uint2 qu = quant_row_chunk(vu, su);
            codes_r[(r * F2 + c0) / 8 + tc] = qg;
            codes_r[(r * F2 + F + c0) / 8 + tc] = qu;
            if ((tc & 3) == 0) {
                const int ab = (rl & 31) * 16 + ((rl >> 5) & 3) * 4 + (tc >> 2);
                s_atom_r[ab] = (uint8_t)sg;
                s_atom_r[512 + ab] = (uint8_t)su;
            }
            *reinterpret_cast<uint4*>(tiles + rl * kQT + tc * 8) = vg;
            *reinterpret_cast<uint4*>(tiles + kQT * kQT + rl * kQT + tc * 8) = vu;
            if (p + 2 < 8) {
                H0[p & 1] = nh0;
                H1[p & 1] = nh1;
                GW[p & 1] = ngw;
                UW[p & 1] = nuw;
            }
        }
        // the next tile's first two chunks are loaded while this tile's
        // columnwise blocks are quantized and stored
        if (i + 1 < nrt) {
            load(r0 + kQT, 0, H0[0], H1[0], GW[0], UW[0]);
            load(r0 + kQT, 1, H0[1], H1[1], GW[1], UW[1]);
        }
        __syncthreads();                      // A: both tiles complete
        const int blk = warp & 3;
        const int col = (warp >> 2) * 64 + 2 * lane;
        uint32_t wg0[8], wg1[8], wu0[8], wu1[8];
        uint32_t bg0, bg1, bu0, bu1;
        quant_col_block(tiles, blk, col, wg0, wg1, bg0, bg1);
        quant_col_block(tiles + kQT * kQT, blk, col, wu0, wu1, bu0, bu1);
        const int a0 = (col & 31) * 16 + ((col >> 5) & 3) * 4 + blk;
        const int a1 = ((col + 1) & 31) * 16 + (((col + 1) >> 5) & 3) * 4 + blk;
        s_atom_c[a0] = (uint8_t)bg0;
        s_atom_c[a1] = (uint8_t)bg1;
        s_atom_c[512 + a0] = (uint8_t)bu0;
        s_atom_c[512 + a1] = (uint8_t)bu1;
        {
            // each column's 32 codes of this block: one 32-byte sector of the
            // transposed output, stored straight from registers
            uint8_t* dg = codes_c + ((int64_t)octile(0) * kQT + col) * rows + r0 + 32 * blk;
            uint8_t* du = codes_c + ((int64_t)octile(1) * kQT + col) * rows + r0 + 32 * blk;
            st_global_32B(dg, wg0);
            st_global_32B(dg + rows, wg1);
            st_global_32B(du, wu0);
            st_global_32B(du + rows, wu1);
        }
        // B: both tiles are read (the next tile may overwrite them) and this
        // tile's atoms are complete
        __syncthreads();
        if (warp < 2) {
            const int t = warp;
            const int64_t atom = (int64_t)octile(t) * (rows / kQT) + r0 / kQT;
            reinterpret_cast<uint4*>(sf_r + atom * 512)[lane] = reinterpret_cast<const uint4*>(s_atom_r + t * 512)[lane];
        } else if (warp < 6) {
            // columnwise scales of output tile t: the tile-224 layout (warps
            // 2, 3) and/or the atom layout (warps 2, 3 if it is the only one,
            // else warps 4, 5)
            const int t = warp & 1;
            const bool atoms = sf_c != nullptr && (warp >= 4) == (sf_c224 != nullptr);
            if (warp < 4 && sf_c224 != nullptr)
                store_col_scales_t224(sf_c224, s_atom_c + t * 512, r0 / kQT, (int64_t)octile(t) * kQT, (int)F2, lane);
            if (atoms) {
                const int64_t atom = (r0 / kQT) * (int64_t)out_tiles + octile(t);
                reinterpret_cast<uint4*>(sf_c + atom * 512)[lane] =
                    reinterpret_cast<const uint4*>(s_atom_c + t * 512)[lane];
            }
        }
        // this tile's atoms are rewritten two tiles on (double-buffered)
    }
}

// Where the columnwise scales of a [rows, cols] quantization go (moe_sf_layout_t
// of the transposed [cols, rows] matrix): the atom layout, the tile-224 layout,
// or both, the tile-224 bytes first.
static void col_scale_outputs(uint8_t* scales_col, int layout, int64_t rows, int64_t cols, uint8_t*& atoms,
                              uint8_t*& t224) {
    atoms = t224 = nullptr;
    if (scales_col == nullptr) return;
    if (layout == MOE_SF_ATOMS) {
        atoms = scales_col;
    } else {
        t224 = scales_col;
        if (layout == MOE_SF_TILE224_AND_ATOMS) atoms = scales_col + (rows / kQT) * ((cols + 223) / 224) * 1024;
    }
}

cudaError_t quant_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(k_quant_both, cudaFuncAttributeMaxDynamicSharedMemorySize, kQBSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_swiglu_bwd_quant, cudaFuncAttributeMaxDynamicSharedMemorySize, kSBSmem);
}

}  // namespace moe

extern "C" moe_status_t mxfp8_gather_quantize_ex(const void* src, int64_t src_rows, int cols, int k,
                                                 const int32_t* row_id, const float* row_w, const int32_t* gofs,
                                                 int G, int64_t rows, uint8_t* codes_row, uint8_t* scales_row,
                                                 uint8_t* codes_col, uint8_t* scales_col, int col_sf_layout,
                                                 int32_t* err, void* stream) {
    using namespace moe;
    MOE_REQUIRE(col_sf_layout == MOE_SF_ATOMS || col_sf_layout == MOE_SF_TILE224 ||
                    col_sf_layout == MOE_SF_TILE224_AND_ATOMS,
                MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(src && gofs && G >= 1 && G <= 4096 && cols > 0 && rows > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(row_id != nullptr || row_w == nullptr, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(row_id == nullptr || (k >= 1 && src_rows >= 0 && src_rows <= 0x7FFFFFFF), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(row_id != nullptr || src_rows == rows, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE((codes_row != nullptr) == (scales_row != nullptr), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE((codes_col != nullptr) == (scales_col != nullptr), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(codes_row != nullptr || codes_col != nullptr, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows % kQT == 0 && cols % kQT == 0, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(cols / kQT <= 65535 && rows <= 0x7FFFFFFF, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(codes_row == nullptr || (reinterpret_cast<uintptr_t>(codes_row) & 31) == 0, MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(codes_col == nullptr || (reinterpret_cast<uintptr_t>(codes_col) & 31) == 0, MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(moe_aligned16(src) && (codes_row == nullptr || (moe_aligned16(codes_row) && moe_aligned16(scales_row))) &&
                    (codes_col == nullptr || (moe_aligned16(codes_col) && moe_aligned16(scales_col))),
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    const int64_t row_runs = (rows / kQT + kQBRowTiles - 1) / kQBRowTiles;
    MOE_REQUIRE(row_runs <= 0x7FFFFFFF, MOE_ERR_UNSUPPORTED);
    dim3 grid((unsigned)row_runs, (unsigned)(cols / kQT));
    uint8_t *sf_atoms = nullptr, *sf_t224 = nullptr;
    col_scale_outputs(scales_col, col_sf_layout, rows, cols, sf_atoms, sf_t224);
    k_quant_both<<<grid, kQBThreads, kQBSmem, (cudaStream_t)stream>>>((const uint16_t*)src, src_rows, cols, k, row_id,
                                                                     row_w, gofs, G, rows, (uint2*)codes_row,
                                                                     scales_row, codes_col, sf_atoms, sf_t224, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t mxfp8_gather_quantize(const void* src, int64_t src_rows, int cols, int k,
                                              const int32_t* row_id, const float* row_w, const int32_t* gofs, int G,
                                              int64_t rows, uint8_t* codes_row, uint8_t* scales_row,
                                              uint8_t* codes_col, uint8_t* scales_col, int32_t* err, void* stream) {
    return mxfp8_gather_quantize_ex(src, src_rows, cols, k, row_id, row_w, gofs, G, rows, codes_row, scales_row,
                                    codes_col, scales_col, MOE_SF_ATOMS, err, stream);
}

extern "C" moe_status_t mxfp8_swiglu_bwd_quantize_ex(const float* dH, const void* a_pre, int f,
                                                     const int32_t* gofs, int G, int64_t rows, void* dA,
                                                     uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                                                     uint8_t* scales_col, int col_sf_layout, int32_t* err,
                                                     void* stream) {
    using namespace moe;
    MOE_REQUIRE(col_sf_layout == MOE_SF_ATOMS || col_sf_layout == MOE_SF_TILE224 ||
                    col_sf_layout == MOE_SF_TILE224_AND_ATOMS,
                MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(dH && a_pre && gofs && codes_row && scales_row && codes_col && scales_col, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(G >= 1 && G <= 4096 && f > 0 && rows > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(f % kQT == 0 && rows % kQT == 0 && rows <= 0x7FFFFFFF && f / kQT <= 65535, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(dH) && moe_aligned16(a_pre) && moe_aligned16(dA) && moe_aligned16(codes_row) &&
                    moe_aligned16(scales_row) && (reinterpret_cast<uintptr_t>(codes_col) & 31) == 0 &&
                    moe_aligned16(scales_col),
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    const int64_t row_runs = (rows / kQT + kQBRowTiles - 1) / kQBRowTiles;
    dim3 grid((unsigned)row_runs, (unsigned)(f / kQT));
    uint8_t *sf_atoms = nullptr, *sf_t224 = nullptr;
    col_scale_outputs(scales_col, col_sf_layout, rows, 2 * (int64_t)f, sf_atoms, sf_t224);
    k_swiglu_bwd_quant<<<grid, kQBThreads, kSBSmem, (cudaStream_t)stream>>>(
        dH, (const uint16_t*)a_pre, f, gofs, G, rows, (uint16_t*)dA, (uint2*)codes_row, scales_row, codes_col,
        sf_atoms, sf_t224, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t mxfp8_swiglu_bwd_quantize(const float* dH, const void* a_pre, int f, const int32_t* gofs,
                                                  int G, int64_t rows, void* dA, uint8_t* codes_row,
                                                  uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                                                  int32_t* err, void* stream) {
    return mxfp8_swiglu_bwd_quantize_ex(dH, a_pre, f, gofs, G, rows, dA, codes_row, scales_row, codes_col,
                                        scales_col, MOE_SF_ATOMS, err, stream);
}
