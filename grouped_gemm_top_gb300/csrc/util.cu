// Library utilities outside the method's steps: the MXFP8 scale-layout
// conversion (atom layout <-> canonical row-major) and the write-only HBM
// stream that measures the ceiling of the write-heavy quantization kernels.
#include <algorithm>

#include "common.cuh"

namespace moe {

// One thread per scale byte; i runs over the canonical [rows, nb] matrix.
__global__ void __launch_bounds__(256) k_scale_layout(const uint8_t* __restrict__ src, int64_t rows, int nb,
                                                      int to_canonical, uint8_t* __restrict__ dst) {
    const int64_t n = rows * nb;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / nb, b = i - r * nb;
        const int64_t a = sf_atom_offset(r, b, rows);
        if (to_canonical)
            dst[i] = src[a];
        else
            dst[a] = src[i];
    }
}

// Write-only stream, method 0: 16-byte stores, four per loop trip.
__global__ void __launch_bounds__(256) k_fill_v4(uint4* __restrict__ dst, int64_t n16, uint32_t v) {
    const uint4 val = make_uint4(v, v, v, v);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        dst[i] = val;
        dst[i + stride] = val;
        dst[i + 2 * stride] = val;
        dst[i + 3 * stride] = val;
    }
    for (; i < n16; i += stride) dst[i] = val;
}

constexpr int kFillBulk = 32768;   // bytes per bulk copy (the CTA's shared buffer)

// Write-only stream, method 1: a shared-memory buffer filled once, written
// out by one thread with bulk asynchronous copies (at most 8 in flight).
__global__ void __launch_bounds__(128) k_fill_bulk(uint8_t* __restrict__ dst, int64_t bytes, uint32_t v) {
    extern __shared__ __align__(128) uint32_t s_buf[];
    for (int i = threadIdx.x; i < kFillBulk / 4; i += blockDim.x) s_buf[i] = v;
    // make the generic-proxy writes visible to the bulk copies (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x != 0) return;
    const uint32_t src = (uint32_t)__cvta_generic_to_shared(s_buf);
    for (int64_t off = (int64_t)blockIdx.x * kFillBulk; off < bytes; off += (int64_t)gridDim.x * kFillBulk) {
        const int64_t left = bytes - off;
        const uint32_t n = (uint32_t)(left < kFillBulk ? left : kFillBulk);
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst + off), "r"(src), "r"(n)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace moe

extern "C" moe_status_t mxfp8_scale_layout(const uint8_t* src, int64_t rows, int cols, int to_canonical, uint8_t* dst,
                                           void* stream) {
    using namespace moe;
    MOE_REQUIRE(src && dst && rows > 0 && cols > 0 && (to_canonical == 0 || to_canonical == 1), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(rows % 128 == 0 && cols % 128 == 0 && rows <= (1LL << 40), MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    const int nb = cols / 32;
    const int64_t n = rows * nb;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, cap > 0 ? cap : 1);
    k_scale_layout<<<grid, 256, 0, (cudaStream_t)stream>>>(src, rows, nb, to_canonical, dst);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_hbm_fill(void* dst, size_t bytes, uint32_t value, int method, void* stream) {
    using namespace moe;
    MOE_REQUIRE(dst && (method == 0 || method == 1), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(bytes % 16 == 0, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(moe_aligned16(dst), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (bytes == 0) return MOE_OK;
    const int sms = device_sm_count();
    MOE_REQUIRE(sms > 0, MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    if (method == 0) {
        const int64_t n16 = (int64_t)(bytes / 16);
        const int grid = (int)std::min<int64_t>((n16 + 255) / 256, (int64_t)sms * 8);
        k_fill_v4<<<grid, 256, 0, s>>>(static_cast<uint4*>(dst), n16, value);
    } else {
        const int64_t chunks = (int64_t)((bytes + kFillBulk - 1) / kFillBulk);
        const int grid = (int)std::min<int64_t>(chunks, (int64_t)sms * 2);
        k_fill_bulk<<<grid, 128, kFillBulk, s>>>(static_cast<uint8_t*>(dst), (int64_t)bytes, value);
    }
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
