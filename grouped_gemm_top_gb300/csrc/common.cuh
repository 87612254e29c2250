// Shared device/host helpers for libmoe (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Device-side error word: first error wins.
__device__ __forceinline__ void set_err(int32_t* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Unpack 8 bf16 held in a uint4 into floats.
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Round 8 floats to bf16 (nearest-even) and pack them into a uint4.
__device__ __forceinline__ uint4 pack8(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Byte offset of the scale of (row r, block b) in the atom layout of a
// matrix with `rows` rows (see moe.h).
__host__ __device__ __forceinline__ int64_t sf_atom_offset(int64_t r, int64_t b, int64_t rows) {
    return ((b >> 2) * (rows >> 7) + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

// E8M0 scale byte for a block whose largest magnitude is `amax` (a bf16 value
// held exactly in fp32): the smallest e with amax <= 448 * 2^e, byte e + 127,
// clamped to [0, 254]; zero and subnormal amax give byte 0.  For a normal
// amax = M * 2^q (M in [1, 2)): e = q - 8, plus one when M > 1.75.
__device__ __forceinline__ uint32_t e8m0_scale_byte(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int be = (int)((bits >> 23) & 0xFF);
    if (be == 0) return 0u;
    const uint32_t mant7 = (bits >> 16) & 0x7F;   // bf16 mantissa
    int b = be - 8 + (mant7 > 0x60 ? 1 : 0);
    b = b < 0 ? 0 : b;
    return (uint32_t)b;
}

// 2^-(b-127) as an fp32 (always a normal number for b in [0, 254]).
__device__ __forceinline__ float e8m0_inv_scale(uint32_t b) {
    return __uint_as_float((254u - b) << 23);
}

// sigmoid(x) with the fast exponential and division; x is clamped at -80
// so that 1 + exp(-x) stays finite (sigmoid(-80) ~ 2e-35).
__device__ __forceinline__ float fast_sigmoid(float x) {
    return __fdividef(1.f, 1.f + __expf(-fmaxf(x, -80.f)));
}

// SwiGLU backward of one element: h = g * sigmoid(g) * u, upstream dh:
// dg = dh * u * s * (1 + g * (1 - s)), du = dh * g * s with s = sigmoid(g).
// Shared by the GEMM epilogue and the fused quantization so both produce
// the same fp32 values.
__device__ __forceinline__ void swiglu_bwd_pair(float g, float u, float dh, float& dg, float& du) {
    const float s = fast_sigmoid(g);
    dg = dh * u * s * (1.f + g * (1.f - s));
    du = dh * g * s;
}

// Two fp32 -> two E4M3 bytes (round-to-nearest-even, saturate to +-448);
// the byte of `lo` is the low byte of the result.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Exclusive scan of one int per thread over a block of up to 1024 threads.
// Returns the exclusive prefix; *total gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        int x = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += n;
        }
        if (lane < nw) s_warp[lane] = x;   // inclusive over warps
    }
    __syncthreads();
    const int warp_base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[((blockDim.x + 31) >> 5) - 1];
    return warp_base + inc - v;
}

}  // namespace moe

// Host-side helpers (defined in api.cu).
namespace moe {
int device_sm_count();        // SM count of the current device (after moe_init)
bool device_initialized();
}  // namespace moe

#define MOE_CHECK_LAUNCH()                                   \
    do {                                                     \
        cudaError_t e_ = cudaGetLastError();                 \
        if (e_ != cudaSuccess) return MOE_ERR_CUDA;          \
    } while (0)

#define MOE_REQUIRE(cond, code)          \
    do {                                 \
        if (!(cond)) return (code);      \
    } while (0)

static inline bool moe_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
