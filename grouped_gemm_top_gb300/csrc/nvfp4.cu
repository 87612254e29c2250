// NVFP4 two-level quantization (sm_103a).
//
// [CH1] §1.1 precision table: FP4 is 4 bits, 1 sign + 2 exponent + 1
// mantissa (E2M1); "低精度格式的缩放机制": NVFP4 needs two scales, an E4M3
// scale per small block for the relative sizes inside it and one FP32 scale
// for the whole tensor's range.  [TE-JAX] "What is the training performance
// impact…": NVFP4 is the next format for the grouped expert GEMMs.
//
// Steps (all in fp32, each rounded to nearest):
//   s_t = amax / 2688, enc = 2688 / amax       (2688 = 6 x 448)
//   block of 16: t_b = (amax_b / 6) * enc, scale byte = E4M3(t_b) (RNE,
//                saturating), r_b = enc / E4M3 value
//   element:     code = E2M1(x * r_b) (RNE, saturating at 6)
// A block whose scale byte is 0 gets zero codes.  Two launches: the tensor
// amax (a reduction into a caller-owned word, zeroed first), then one pass
// that reads each row once and writes packed codes and scale atoms.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace nvf4 {

constexpr float kRange = 2688.0f;    // largest E2M1 (6) x largest E4M3 (448)

// Max |x| over a bf16 tensor, as the bf16 bits of the magnitude (for
// non-negative bf16 values the bit pattern orders like the value).
__global__ void __launch_bounds__(256) k_amax(const uint4* __restrict__ src, int64_t n16,
                                              uint32_t* __restrict__ amax_bits) {
    uint32_t m = 0;     // two packed bf16 magnitudes
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(src + i);
        m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    }
    uint32_t mm = max(m & 0xFFFFu, m >> 16);
    mm = __reduce_max_sync(0xffffffffu, mm);
    if ((threadIdx.x & 31) == 0 && mm != 0) atomicMax(amax_bits, mm);
}

// Value of an E4M3 byte (sign bit ignored: scales are non-negative).
__device__ __forceinline__ float e4m3_value(uint32_t byte) {
    const uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
    if (e == 0) return (float)m * 0x1p-9f;
    return __uint_as_float(((e + 120u) << 23) | (m << 20));     // (1 + m/8) * 2^(e - 7)
}

// Eight floats to eight E2M1 codes (RNE, saturating), element i in nibble i.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* f) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return r;
}

// One CTA per (256-column k-step, 128-row tile); thread t quantizes 128
// columns (8 blocks) of row t / 2 of the tile: 256 bytes read, 64 bytes of
// codes and two 4-byte scale words written.
__global__ void __launch_bounds__(256) k_quant(const __nv_bfloat16* __restrict__ src, int64_t rows, int cols,
                                               const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                                               uint8_t* __restrict__ scales, float* __restrict__ tensor_scale) {
    const float amax = bf16_bits_to_float(*amax_bits);
    const float enc = amax > 0.f ? __fdiv_rn(kRange, amax) : 0.f;
    const int tid = threadIdx.x, half = tid & 1;
    const int64_t r = (int64_t)blockIdx.y * 128 + (tid >> 1);
    const int64_t c0 = (int64_t)blockIdx.x * 256 + half * 128;
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *tensor_scale = amax > 0.f ? __fdiv_rn(amax, kRange) : 0.f;
    const uint4* in = reinterpret_cast<const uint4*>(src + r * cols + c0);
    uint32_t q[16];
    uint32_t sw[2] = {0u, 0u};
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        float f[16];
        unpack8(__ldg(in + 2 * b), f);
        unpack8(__ldg(in + 2 * b + 1), f + 8);
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
        uint32_t byte = 0u;
        float rb = 0.f;
        if (enc > 0.f) {
            const float tb = __fmul_rn(__fdiv_rn(am, 6.0f), enc);
            byte = cvt_e4m3x2(tb, 0.f) & 0x7Fu;
            if (byte != 0u) rb = __fdiv_rn(enc, e4m3_value(byte));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(f[i], rb);
        q[2 * b] = byte != 0u ? cvt_e2m1x8(f) : 0u;
        q[2 * b + 1] = byte != 0u ? cvt_e2m1x8(f + 8) : 0u;
        sw[b >> 2] |= byte << (8 * (b & 3));
    }
    uint4* o = reinterpret_cast<uint4*>(codes + r * (cols / 2) + c0 / 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = make_uint4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]);
    // scale atoms of this k-step: [k-step][row tile][4 atoms of 64 columns][512]
    const int64_t base = ((int64_t)blockIdx.x * (rows / 128) + blockIdx.y) * 2048 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        *reinterpret_cast<uint32_t*>(scales + base + (2 * half + j) * 512) = sw[j];
}

// Max |x| over the rows [0, lim) of a [rows, cols] bf16 matrix, lim =
// min(gofs[G], rows) read on the device (0 when the offsets are invalid).
__global__ void __launch_bounds__(256) k_amax_rows(const uint4* __restrict__ src, int cols, int64_t rows,
                                                   const int32_t* __restrict__ gofs, int G,
                                                   uint32_t* __restrict__ amax_bits) {
    const int64_t lim = min((int64_t)max(gofs[G], 0), rows);
    const int64_t n16 = lim * cols / 8;
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(src + i);
        m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
        m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    }
    uint32_t mm = max(m & 0xFFFFu, m >> 16);
    mm = __reduce_max_sync(0xffffffffu, mm);
    if ((threadIdx.x & 31) == 0 && mm != 0) atomicMax(amax_bits, mm);
}

// Group-aware columnwise quantization: blocks of 16 rows along each column
// (the contraction axis of the weight gradient).  Groups start at multiples
// of 128 rows, so no block crosses a group; rows >= gofs[G] count as zeros.
// One CTA per (64-column, 256-row) tile staged in shared memory; thread
// (c, q) quantizes rows [64 q, 64 q + 64) of column c: four blocks, 32 bytes
// of codes (transposed output) and one 4-byte scale word (one atom row).
__global__ void __launch_bounds__(256) k_quant_cols(const __nv_bfloat16* __restrict__ src, int64_t rows, int cols,
                                                    const int32_t* __restrict__ gofs, int G,
                                                    const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ scales, float* __restrict__ tensor_scale,
                                                    int32_t* __restrict__ err) {
    __shared__ __align__(16) uint16_t tile[256][64];
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    if (tid == 0) s_ok = 1;
    __syncthreads();
    // offsets: 0 first, monotone, multiples of 128, inside the buffer
    for (int g = tid; g < G; g += blockDim.x) {
        const int lo = gofs[g], hi = gofs[g + 1];
        if ((g == 0 && lo != 0) || hi < lo || (hi & 127) != 0 || (int64_t)hi > rows) s_ok = 0;
    }
    __syncthreads();
    const bool ok = s_ok != 0;
    if (!ok && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) set_err(err, MOE_ERR_BAD_OFFSETS);
    const int64_t lim = ok ? (int64_t)gofs[G] : 0;
    const float amax = ok ? bf16_bits_to_float(*amax_bits) : 0.f;
    const float enc = amax > 0.f ? __fdiv_rn(kRange, amax) : 0.f;
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *tensor_scale = amax > 0.f ? __fdiv_rn(amax, kRange) : 0.f;
    const int64_t r0 = (int64_t)blockIdx.y * 256;
    const int c0 = blockIdx.x * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 32 * i + (tid >> 3), ch = tid & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + r < lim) v = __ldg(reinterpret_cast<const uint4*>(src + (r0 + r) * cols + c0) + ch);
        *reinterpret_cast<uint4*>(&tile[r][8 * ch]) = v;
    }
    __syncthreads();
    const int c = tid & 63, q = tid >> 6;
    const int64_t cc = c0 + c;
    uint32_t qw[8];
    uint32_t sw = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = bf16_bits_to_float(tile[64 * q + 16 * b + i][c]);
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
        uint32_t byte = 0u;
        float rb = 0.f;
        if (enc > 0.f) {
            const float tb = __fmul_rn(__fdiv_rn(am, 6.0f), enc);
            byte = cvt_e4m3x2(tb, 0.f) & 0x7Fu;
            if (byte != 0u) rb = __fdiv_rn(enc, e4m3_value(byte));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(f[i], rb);
        qw[2 * b] = byte != 0u ? cvt_e2m1x8(f) : 0u;
        qw[2 * b + 1] = byte != 0u ? cvt_e2m1x8(f + 8) : 0u;
        sw |= byte << (8 * b);
    }
    uint4* o = reinterpret_cast<uint4*>(codes + cc * (rows / 2) + (r0 + 64 * q) / 2);
    o[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    o[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    // [256-row k-step][128-column tile of the transposed matrix][4 atoms][512]
    const int64_t off = ((int64_t)blockIdx.y * (cols / 128) + cc / 128) * 2048 + q * 512 + (cc & 31) * 16 +
                        ((cc >> 5) & 3) * 4;
    *reinterpret_cast<uint32_t*>(scales + off) = sw;
}

}  // namespace nvf4
}  // namespace moe

using namespace moe;

extern "C" int64_t nvfp4_sf_bytes(int64_t rows, int cols) {
    if (rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 256 != 0) return -1;
    return rows * (cols / 16);
}

extern "C" moe_status_t nvfp4_quantize(const void* src, int64_t rows, int cols, uint8_t* codes, uint8_t* scales,
                                       float* tensor_scale, uint32_t* amax_ws, int32_t* err, void* stream) {
    (void)err;
    MOE_REQUIRE(src && codes && scales && tensor_scale && amax_ws, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows > 0 && cols > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows % 128 == 0 && cols % 256 == 0 && rows / 128 <= 65535, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(src) && moe_aligned16(codes) && moe_aligned16(scales), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(amax_ws) & 3u) == 0 && (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) == 0,
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t n16 = rows * (int64_t)cols / 8;
    const int sms = device_sm_count();
    const int64_t want = (n16 + 255) / 256;
    const int grid = (int)std::min<int64_t>(want, (int64_t)(sms > 0 ? sms : 148) * 8);
    nvf4::k_amax<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), n16, amax_ws);
    nvf4::k_quant<<<dim3((unsigned)(cols / 256), (unsigned)(rows / 128)), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(src), rows, cols, amax_ws, codes, scales, tensor_scale);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t nvfp4_quantize_cols(const void* src, int64_t rows, int cols, const int32_t* gofs, int G,
                                            uint8_t* codes_t, uint8_t* scales_t, float* tensor_scale,
                                            uint32_t* amax_ws, int32_t* err, void* stream) {
    MOE_REQUIRE(src && gofs && codes_t && scales_t && tensor_scale && amax_ws, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows > 0 && cols > 0 && G >= 1 && G <= 4096, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows % 256 == 0 && cols % 128 == 0 && rows / 256 <= 65535 && rows <= 0x7FFFFF00LL,
                MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(src) && moe_aligned16(codes_t) && moe_aligned16(scales_t), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(amax_ws) & 3u) == 0 && (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) == 0,
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    const int sms = device_sm_count();
    const int64_t want = (rows * (int64_t)cols / 8 + 255) / 256;
    const int grid = (int)std::min<int64_t>(want, (int64_t)(sms > 0 ? sms : 148) * 8);
    nvf4::k_amax_rows<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), cols, rows, gofs, G, amax_ws);
    nvf4::k_quant_cols<<<dim3((unsigned)(cols / 64), (unsigned)(rows / 256)), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(src), rows, cols, gofs, G, amax_ws, codes_t, scales_t, tensor_scale,
        err);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

