// Router: top-k selection + weights + per-expert counts/offsets, and the
// router backward.  [TE-JAX] introduction (a trained router picks the top-k
// experts that process each token) and "Optimization 2" (the routing step
// runs as fused router kernels that map tokens to experts).
//
// One warp owns one token: lane l holds logits of experts l, l+32, ...; the
// k winners are found by k rounds of a warp argmax (ties -> lower index).
// Counts come from per-CTA histograms reduced by one small CTA, so they are
// deterministic and never leave the device.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace moe {

constexpr int kRouteTokPerCta = 128;
constexpr int kRouteThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Warp argmax over the not-yet-taken experts; returns the winner's (value,
// index) in every lane.  Ordering: larger value, then lower index.
template <int EPL>
__device__ __forceinline__ void warp_pick(const float (&v)[EPL], uint32_t taken, int lane, float& bv, int& bi) {
    bool have = false;
    bv = 0.f;
    bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        if (!((taken >> i) & 1u)) {
            const int e = lane + 32 * i;
            if (!have || v[i] > bv || (v[i] == bv && e < bi)) {
                bv = v[i];
                bi = e;
                have = true;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, o);
        const int oi = __shfl_xor_sync(kFull, bi, o);
        const int oh = __shfl_xor_sync(kFull, (int)have, o);
        if (oh && (!have || ov > bv || (ov == bv && oi < bi))) {
            bv = ov;
            bi = oi;
            have = true;
        }
    }
}

template <int EPL>
__global__ void __launch_bounds__(kRouteThreads) k_route_topk(const float* __restrict__ logits, int T, int E, int k,
                                                              int score, int normalize, int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w, int32_t* __restrict__ block_hist) {
    extern __shared__ int s_hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRouteTokPerCta;
    for (int tt = warp; tt < kRouteTokPerCta; tt += kRouteThreads / 32) {
        const int t = t0 + tt;
        if (t >= T) break;
        const float* row = logits + (size_t)t * E;
        float v[EPL];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? __ldg(row + e) : 0.f;
            if (e >= E) taken |= 1u << i;
        }
        int my_idx = 0;
        float my_val = 0.f;
        for (int r = 0; r < k; ++r) {
            float bv;
            int bi;
            warp_pick<EPL>(v, taken, lane, bv, bi);
            if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
            if (lane == r) {
                my_idx = bi;
                my_val = bv;
            }
        }
        const bool mine = lane < k;
        const float m = __shfl_sync(kFull, my_val, 0);   // largest logit overall
        float w;
        if (score == MOE_SCORE_SOFTMAX) {
            const float ex = mine ? expf(my_val - m) : 0.f;
            float den;
            if (normalize) {
                den = warp_sum(ex);
            } else {
                float part = 0.f;
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (!((lane + 32 * i) >= E)) part += expf(v[i] - m);
                den = warp_sum(part);
            }
            w = ex / den;
        } else {
            const float sg = mine ? 1.f / (1.f + expf(-my_val)) : 0.f;
            w = normalize ? sg / warp_sum(sg) : sg;
        }
        if (mine) {
            topk_idx[(size_t)t * k + lane] = my_idx;
            topk_w[(size_t)t * k + lane] = w;
            atomicAdd(&s_hist[my_idx], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[(size_t)blockIdx.x * E + e] = s_hist[e];
}

// counts[e] = sum over CTAs of the histograms; offsets = exclusive scan.
__global__ void __launch_bounds__(1024) k_route_offsets(const int32_t* __restrict__ block_hist, int nblk, int E,
                                                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    int c = 0;
    if (e < E)
        for (int b = 0; b < nblk; ++b) c += block_hist[(size_t)b * E + e];
    int total;
    const int ex = block_exclusive_scan(e < E ? c : 0, s_warp, &total);
    if (e < E) {
        counts[e] = c;
        offsets[e] = ex;
    }
    if (e == 0) offsets[E] = total;
}

template <int EPL>
__global__ void __launch_bounds__(kRouteThreads) k_route_bwd(const float* __restrict__ logits,
                                                             const int32_t* __restrict__ topk_idx,
                                                             const float* __restrict__ dw, int T, int E, int k,
                                                             int score, int normalize, float* __restrict__ dlogits,
                                                             int32_t* err) {
    const int warp = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int t = warp;
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    const bool mine = lane < k;
    int idx = mine ? topk_idx[(size_t)t * k + lane] : 0;
    if (mine && (idx < 0 || idx >= E)) {
        set_err(err, MOE_ERR_BAD_EXPERT);
        idx = 0;
    }
    const float g = mine ? dw[(size_t)t * k + lane] : 0.f;
    const float l = mine ? __ldg(row + idx) : 0.f;
    float out[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) out[i] = 0.f;
    float dl = 0.f;   // gradient for my chosen entry
    if (score == MOE_SCORE_SOFTMAX) {
        if (normalize) {
            const float m = warp_max(mine ? l : -INFINITY);
            const float ex = mine ? expf(l - m) : 0.f;
            const float w = ex / warp_sum(ex);
            const float inner = warp_sum(w * g);
            dl = w * (g - inner);
        } else {
            float v[EPL];
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                v[i] = e < E ? __ldg(row + e) : -INFINITY;
                m = fmaxf(m, v[i]);
            }
            m = warp_max(m);
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i < E) part += expf(v[i] - m);
            const float den = warp_sum(part);
            const float ps = mine ? expf(l - m) / den : 0.f;
            const float inner = warp_sum(ps * g);
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i < E) out[i] = -(expf(v[i] - m) / den) * inner;
            dl = ps * g;   // added on top of the -p*inner term below
        }
    } else {
        const float s = mine ? 1.f / (1.f + expf(-l)) : 0.f;
        if (normalize) {
            const float ssum = warp_sum(s);
            const float w = s / ssum;
            const float inner = warp_sum(w * g);
            dl = s * (1.f - s) / ssum * (g - inner);
        } else {
            dl = s * (1.f - s) * g;
        }
    }
    // scatter the k chosen gradients into the owning lanes
    for (int r = 0; r < k; ++r) {
        const int ir = __shfl_sync(kFull, idx, r);
        const float dr = __shfl_sync(kFull, dl, r);
        if ((ir & 31) == lane) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == (ir >> 5)) out[i] += dr;
        }
    }
    float* orow = dlogits + (size_t)t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) orow[e] = out[i];
    }
}

static int route_epl(int E) {
    const int need = (E + 31) / 32;
    int epl = 1;
    while (epl < need) epl <<= 1;
    return epl;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_workspace_size(int T, int E) {
    if (T < 0 || E <= 0) return 0;
    const size_t nblk = (size_t)(T + kRouteTokPerCta - 1) / kRouteTokPerCta;
    return (nblk > 0 ? nblk : 1) * (size_t)E * sizeof(int32_t);
}

#define MOE_ROUTE_DISPATCH(EPLV, KERNEL, GRID, BLOCK, SMEM, STREAM, ...) \
    switch (EPLV) {                                                     \
        case 1: KERNEL<1><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break;   \
        case 2: KERNEL<2><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break;   \
        case 4: KERNEL<4><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break;   \
        case 8: KERNEL<8><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break;   \
        case 16: KERNEL<16><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break; \
        default: KERNEL<32><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__); break; \
    }

extern "C" moe_status_t moe_route_topk(const float* logits, int T, int E, int k, int score, int normalize,
                                       int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                       void* ws, size_t ws_bytes, int32_t* err, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(score == MOE_SCORE_SOFTMAX || score == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(counts && offsets, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (logits && topk_idx && topk_w && ws), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(ws_bytes >= moe_route_workspace_size(T, E), MOE_ERR_WORKSPACE);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    const int nblk = (T + kRouteTokPerCta - 1) / kRouteTokPerCta;
    int32_t* hist = (int32_t*)ws;
    if (nblk > 0) {
        MOE_ROUTE_DISPATCH(route_epl(E), k_route_topk, nblk, kRouteThreads, E * sizeof(int), s, logits, T, E, k,
                           score, normalize, topk_idx, topk_w, hist);
        MOE_CHECK_LAUNCH();
    }
    k_route_offsets<<<1, 1024, 0, s>>>(hist, nblk, E, counts, offsets);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_route_bwd(const float* logits, const int32_t* topk_idx, const float* dw, int T, int E,
                                      int k, int score, int normalize, float* dlogits, int32_t* err, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(score == MOE_SCORE_SOFTMAX || score == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (logits && topk_idx && dw && dlogits), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (T == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const int warps_per_cta = kRouteThreads / 32;
    const int grid = (T + warps_per_cta - 1) / warps_per_cta;
    MOE_ROUTE_DISPATCH(route_epl(E), k_route_bwd, grid, kRouteThreads, 0, s, logits, topk_idx, dw, T, E, k, score,
                       normalize, dlogits, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// Shared experts: experts every token uses with weight 1 (DeepSeek-V3's
// shared expert).  They join the routed choices as choices k .. k+S-1 of
// every token (experts E .. E+S-1), so permute, the grouped GEMMs and the
// combine treat them like routed experts whose group holds every token.
namespace moe {

__global__ void k_append_shared(const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int k, int E,
                                int S, int32_t* __restrict__ idx2, float* __restrict__ w2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int k2 = k + S;
    if (i >= (int64_t)T * k2) return;
    const int64_t t = i / k2;
    const int j = (int)(i - t * k2);
    idx2[i] = j < k ? idx[t * k + j] : E + (j - k);
    w2[i] = j < k ? w[t * k + j] : 1.f;
}

__global__ void k_drop_shared(const float* __restrict__ dw2, int T, int k, int S, float* __restrict__ dw) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * k) return;
    const int64_t t = i / k;
    dw[i] = dw2[t * (k + S) + (i - t * k)];
}

}  // namespace moe

extern "C" moe_status_t moe_route_append_shared(const int32_t* topk_idx, const float* topk_w, int T, int k, int E,
                                                int n_shared, int32_t* idx_out, float* w_out, void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && E >= 1 && n_shared >= 1 && k + n_shared <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (topk_idx && topk_w && idx_out && w_out), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (T == 0) return MOE_OK;
    const int64_t n = (int64_t)T * (k + n_shared);
    moe::k_append_shared<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(topk_idx, topk_w, T, k, E,
                                                                                        n_shared, idx_out, w_out);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_route_drop_shared(const float* dw_all, int T, int k, int n_shared, float* dw,
                                              void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && n_shared >= 1 && k + n_shared <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (dw_all && dw), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (T == 0) return MOE_OK;
    const int64_t n = (int64_t)T * k;
    moe::k_drop_shared<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(dw_all, T, k, n_shared, dw);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_route_topk_noalloc: moe_route_topk without a caller workspace.
//
// Some callers have no way to give the library device memory: code behind a
// plugin or operator interface that passes only input and output pointers,
// processes whose device memory is owned by a fixed pool they cannot grow,
// and code that must not call cudaMalloc because it can synchronise the
// device or is not allowed while a stream is being captured.  For them the
// per-CTA expert histograms (the only scratch routing needs) live in this
// fixed device array, compiled into the library and kept by every GPU that
// loads it until the process exits.
namespace moe {
constexpr size_t kRouteScratchInts = (size_t)1 << 18;   // 1 MiB: ceil(T / 128) * E <= 262,144
static __device__ __align__(256) int32_t g_route_scratch[kRouteScratchInts];
static int32_t* g_route_scratch_dev[64] = {nullptr};     // device address of the array, per device
static std::mutex g_route_scratch_mu;

// moe_init drops the cached address, so the next call looks it up again in
// the context current then (after a device reset the old one is stale).
void route_scratch_forget(int device) {
    if (device < 0 || device >= 64) return;
    std::lock_guard<std::mutex> lock(g_route_scratch_mu);
    g_route_scratch_dev[device] = nullptr;
}
}  // namespace moe

extern "C" moe_status_t moe_route_topk_noalloc(const float* logits, int T, int E, int k, int score, int normalize,
                                               int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                               int32_t* err, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(score == MOE_SCORE_SOFTMAX || score == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(counts && offsets, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (logits && topk_idx && topk_w), MOE_ERR_INVALID_ARG);
    const int nblk = (T + kRouteTokPerCta - 1) / kRouteTokPerCta;
    // sizes whose histograms do not fit the fixed array are refused
    MOE_REQUIRE((size_t)nblk * (size_t)E <= kRouteScratchInts, MOE_ERR_WORKSPACE);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    int32_t* hist = nullptr;
    {
        // first call on this device since moe_init: host code cannot use the
        // array's name as a device pointer, so look its address up (device
        // current) and keep it
        std::lock_guard<std::mutex> lock(g_route_scratch_mu);
        if (g_route_scratch_dev[dev] == nullptr) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || ptr == nullptr) return MOE_ERR_CUDA;
            g_route_scratch_dev[dev] = static_cast<int32_t*>(ptr);
        }
        hist = g_route_scratch_dev[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    // every histogram entry read below is written first in the same call, so
    // what a previous call left in the array does not matter
    if (nblk > 0) {
        MOE_ROUTE_DISPATCH(route_epl(E), k_route_topk, nblk, kRouteThreads, E * sizeof(int), s, logits, T, E, k,
                           score, normalize, topk_idx, topk_w, hist);
        MOE_CHECK_LAUNCH();
    }
    k_route_offsets<<<1, 1024, 0, s>>>(hist, nblk, E, counts, offsets);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
