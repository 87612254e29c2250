// Local dispatch (permute into expert-grouped rows) and local combine
// (unpermute + router-weighted sum), plus the combine backward.
// [TE-JAX] "Optimization 2": dispatch permutes tokens to their experts
// (local reordering); combine returns them to token order and accumulates the
// per-expert results.  [CH1] §2.3.2: the combine is a sum weighted by the
// routing weights.
//
// Slots are deterministic: slot(t, j) = gofs[e] + rank of token t among the
// tokens routed to e.  A CTA of 128 tokens builds a 128-bit mask per expert
// (bit i = token i of the CTA chose e); the rank inside the CTA is a popcount
// of the lower bits, and a one-CTA scan over CTAs gives each CTA's base.
#include "common.cuh"

namespace moe {

constexpr int kPermTok = 128;        // tokens per rank CTA (4 mask words)
constexpr unsigned kFullMask = 0xFFFFFFFFu;

__global__ void __launch_bounds__(kPermTok) k_perm_rank(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                                                        int32_t* __restrict__ slot_of, int32_t* __restrict__ hist,
                                                        int32_t* err) {
    extern __shared__ uint32_t s_mask[];   // [E][4]
    for (int i = threadIdx.x; i < E * 4; i += blockDim.x) s_mask[i] = 0;
    __syncthreads();
    const int tl = threadIdx.x;
    const int t = blockIdx.x * kPermTok + tl;
    const uint32_t bit = 1u << (tl & 31);
    const int word = tl >> 5;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = topk_idx[(size_t)t * k + j];
            bool ok = e >= 0 && e < E;
            for (int j2 = 0; j2 < j && ok; ++j2) ok = topk_idx[(size_t)t * k + j2] != e;
            if (!ok) {
                set_err(err, MOE_ERR_BAD_EXPERT);
                continue;
            }
            atomicOr(&s_mask[e * 4 + word], bit);
        }
    }
    __syncthreads();
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = topk_idx[(size_t)t * k + j];
            // the same test as the mask pass: an expert out of range or named
            // a second time by this token gets no rank (slot -1), so no two
            // choices share a row
            bool ok = e >= 0 && e < E;
            for (int j2 = 0; j2 < j && ok; ++j2) ok = topk_idx[(size_t)t * k + j2] != e;
            int r = -1;
            if (ok) {
                r = __popc(s_mask[e * 4 + word] & (bit - 1u));
                for (int w = 0; w < word; ++w) r += __popc(s_mask[e * 4 + w]);
            }
            slot_of[(size_t)t * k + j] = r;   // rank inside this CTA; finished by k_perm_slot
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        hist[(size_t)blockIdx.x * E + e] = __popc(s_mask[e * 4]) + __popc(s_mask[e * 4 + 1]) +
                                           __popc(s_mask[e * 4 + 2]) + __popc(s_mask[e * 4 + 3]);
    }
}

// One CTA: per-expert scan over rank CTAs, padded group offsets, and -1 in
// the padding rows of row_id.
__global__ void __launch_bounds__(1024) k_perm_scan(const int32_t* __restrict__ hist, int nblk, int E,
                                                    int64_t row_cap, int32_t* __restrict__ base,
                                                    int32_t* __restrict__ gofs, int32_t* __restrict__ row_id,
                                                    int32_t* err) {
    __shared__ int s_warp[32];
    __shared__ int s_cnt[1024];
    __shared__ int s_off[1025];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int b = 0; b < nblk; ++b) {
            base[(size_t)b * E + e] = run;
            run += hist[(size_t)b * E + e];
        }
    }
    const int padded = (run + 127) & ~127;
    int total;
    const int ex = block_exclusive_scan(e < E ? padded : 0, s_warp, &total);
    if (e < E) {
        gofs[e] = ex;
        s_cnt[e] = run;
        s_off[e] = ex;
    }
    if (e == 0) {
        gofs[E] = total;
        s_off[E] = total;
        if ((int64_t)total > row_cap) set_err(err, MOE_ERR_CAPACITY);
    }
    __syncthreads();
    // padding rows: one warp per expert
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int g = warp; g < E; g += blockDim.x >> 5) {
        const int lo = s_off[g] + s_cnt[g], hi = s_off[g + 1];
        for (int r = lo + lane; r < hi; r += 32)
            if ((int64_t)r < row_cap) row_id[r] = -1;
    }
}

__global__ void k_perm_slot(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                            const int32_t* __restrict__ base, const int32_t* __restrict__ gofs, int64_t row_cap,
                            int32_t* __restrict__ slot_of, int32_t* __restrict__ row_id, int32_t* err) {
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= (int64_t)T * k) return;
    const int t = (int)(p / k);
    const int e = topk_idx[p];
    const int r = slot_of[p];
    if (e < 0 || e >= E || r < 0) {
        slot_of[p] = -1;
        return;
    }
    const int64_t slot = (int64_t)gofs[e] + base[(size_t)(t / kPermTok) * E + e] + r;
    if (slot >= row_cap) {
        set_err(err, MOE_ERR_CAPACITY);
        slot_of[p] = -1;
        return;
    }
    slot_of[p] = (int32_t)slot;
    row_id[slot] = (int32_t)p;
}

// x_perm[s] = x[row_id[s] / k] for s < gofs[E]; zeros for padding rows.
// One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) k_perm_gather(const uint4* __restrict__ x, int d8, int k,
                                                     const int32_t* __restrict__ row_id,
                                                     const int32_t* __restrict__ gofs_end, int64_t row_cap,
                                                     uint4* __restrict__ x_perm) {
    const int64_t rows = min((int64_t)*gofs_end, row_cap);
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t s = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); s < rows; s += nwarps) {
        const int id = row_id[s];
        uint4* dst = x_perm + s * d8;
        if (id >= 0) {
            const uint4* src = x + (int64_t)(id / k) * d8;
            int c = lane;
            for (; c + 96 < d8; c += 128) {
                const uint4 a0 = __ldg(src + c), a1 = __ldg(src + c + 32), a2 = __ldg(src + c + 64),
                            a3 = __ldg(src + c + 96);
                dst[c] = a0;
                dst[c + 32] = a1;
                dst[c + 64] = a2;
                dst[c + 96] = a3;
            }
            for (; c < d8; c += 32) dst[c] = __ldg(src + c);
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int c = lane; c < d8; c += 32) dst[c] = z;
        }
    }
}

// out[t] = sum_j w[t,j] * y[slot_of[t,j]] (fp32, j order); w == NULL -> 1.
__global__ void __launch_bounds__(128) k_combine(const uint4* __restrict__ y, const int32_t* __restrict__ slot_of,
                                                 const float* __restrict__ w, const float4* __restrict__ add, int d8,
                                                 int k, uint4* __restrict__ out) {
    const int t = blockIdx.x;
    __shared__ int s_slot[32];
    __shared__ float s_w[32];
    if (threadIdx.x < k) {
        s_slot[threadIdx.x] = slot_of[(size_t)t * k + threadIdx.x];
        s_w[threadIdx.x] = w ? w[(size_t)t * k + threadIdx.x] : 1.f;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < d8; c += blockDim.x) {
        float acc[8];
        if (add != nullptr) {           // fp32 addend first, then the k terms in j order
            const float4 a0 = __ldg(add + ((int64_t)t * d8 + c) * 2), a1 = __ldg(add + ((int64_t)t * d8 + c) * 2 + 1);
            acc[0] = a0.x; acc[1] = a0.y; acc[2] = a0.z; acc[3] = a0.w;
            acc[4] = a1.x; acc[5] = a1.y; acc[6] = a1.z; acc[7] = a1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        }
        for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const int s = j < k ? s_slot[j] : -1;
                v[jj] = s >= 0 ? __ldg(y + (int64_t)s * d8 + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                if (j < k && s_slot[j] >= 0) {
                    float f[8];
                    unpack8(v[jj], f);
                    const float wj = s_w[j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
                }
            }
        }
        out[(int64_t)t * d8 + c] = pack8(acc);
    }
}

// dy[slot(t,j)] = bf16(w[t,j] * dout[t]);  dw[t,j] = <dout[t], y[slot(t,j)]>.
__global__ void __launch_bounds__(128) k_combine_bwd(const uint4* __restrict__ dout, const uint4* __restrict__ y,
                                                     const int32_t* __restrict__ slot_of,
                                                     const float* __restrict__ w, int d8, int k,
                                                     uint4* __restrict__ dy, float* __restrict__ dw) {
    const int t = blockIdx.x;
    __shared__ int s_slot[32];
    __shared__ float s_w[32];
    __shared__ float s_red[8][4];
    if (threadIdx.x < k) {
        s_slot[threadIdx.x] = slot_of[(size_t)t * k + threadIdx.x];
        s_w[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j0 = 0; j0 < k; j0 += 8) {
        float part[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) part[jj] = 0.f;
        for (int c = threadIdx.x; c < d8; c += blockDim.x) {
            float g[8];
            unpack8(__ldg(dout + (int64_t)t * d8 + c), g);
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const int s = j < k ? s_slot[j] : -1;
                v[jj] = s >= 0 ? __ldg(y + (int64_t)s * d8 + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                if (j < k && s_slot[j] >= 0) {
                    float f[8], o[8];
                    unpack8(v[jj], f);
                    const float wj = s_w[j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        part[jj] = fmaf(g[i], f[i], part[jj]);
                        o[i] = wj * g[i];
                    }
                    if (dy != nullptr) dy[(int64_t)s_slot[j] * d8 + c] = pack8(o);
                }
            }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            float v = part[jj];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
            if (lane == 0) s_red[jj][warp] = v;
        }
        __syncthreads();
        if (threadIdx.x < 8 && j0 + threadIdx.x < k) {
            const int jj = threadIdx.x;
            const float tot = s_red[jj][0] + s_red[jj][1] + s_red[jj][2] + s_red[jj][3];
            dw[(size_t)t * k + j0 + jj] = tot;
        }
        __syncthreads();
    }
}

// Zero the padding rows (row_id == -1) below gofs[E].
__global__ void __launch_bounds__(256) k_zero_padding_rows(const int32_t* __restrict__ row_id,
                                                           const int32_t* __restrict__ gofs_end, int64_t row_cap,
                                                           int d8, uint4* __restrict__ buf) {
    const int64_t rows = min((int64_t)*gofs_end, row_cap);
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t s = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); s < rows; s += nwarps) {
        if (row_id[s] >= 0) continue;
        uint4* dst = buf + s * d8;
        for (int c = lane; c < d8; c += 32) dst[c] = z;
    }
}

static int rows_grid(int64_t row_cap) {
    const int64_t want = (row_cap + 7) / 8;     // 8 warps (rows) per CTA
    const int64_t cap = (int64_t)device_sm_count() * 16;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int E) {
    if (T < 0 || E <= 0) return 0;
    const size_t nblk = (size_t)(T + kPermTok - 1) / kPermTok;
    return 2 * (nblk > 0 ? nblk : 1) * (size_t)E * sizeof(int32_t);
}

extern "C" moe_status_t moe_permute(const void* x, int T, int d, int E, int k, const int32_t* topk_idx,
                                    int64_t row_cap, int32_t* gofs, int32_t* slot_of, int32_t* row_id, void* x_perm,
                                    void* ws, size_t ws_bytes, int32_t* err, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(x_perm == nullptr || d > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(gofs && (T == 0 || (topk_idx && slot_of && row_id && ws)), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(row_cap >= moe_row_capacity(T, E, k) && row_cap <= 0x7FFFFFFF, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(ws_bytes >= moe_permute_workspace_size(T, E), MOE_ERR_WORKSPACE);
    if (x_perm) {
        MOE_REQUIRE(x != nullptr, MOE_ERR_INVALID_ARG);
        MOE_REQUIRE(d % 8 == 0 && moe_aligned16(x) && moe_aligned16(x_perm), MOE_ERR_ALIGNMENT);
    }
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    const int nblk = (T + kPermTok - 1) / kPermTok;
    int32_t* hist = (int32_t*)ws;
    int32_t* base = hist + (size_t)(nblk > 0 ? nblk : 1) * E;
    if (nblk > 0) {
        k_perm_rank<<<nblk, kPermTok, (size_t)E * 4 * sizeof(uint32_t), s>>>(topk_idx, T, E, k, slot_of, hist, err);
        MOE_CHECK_LAUNCH();
    }
    k_perm_scan<<<1, 1024, 0, s>>>(hist, nblk, E, row_cap, base, gofs, row_id, err);
    MOE_CHECK_LAUNCH();
    if (T > 0) {
        const int64_t pairs = (int64_t)T * k;
        k_perm_slot<<<(unsigned)((pairs + 255) / 256), 256, 0, s>>>(topk_idx, T, E, k, base, gofs, row_cap, slot_of,
                                                                     row_id, err);
        MOE_CHECK_LAUNCH();
    }
    if (x_perm && T > 0) {
        k_perm_gather<<<rows_grid(row_cap), 256, 0, s>>>((const uint4*)x, d / 8, k, row_id, gofs + E, row_cap,
                                                         (uint4*)x_perm);
        MOE_CHECK_LAUNCH();
    }
    return MOE_OK;
}

extern "C" moe_status_t moe_unpermute_combine(const void* y_perm, const int32_t* slot_of, const float* topk_w, int T,
                                              int d, int k, void* out, int32_t* err, void* stream) {
    (void)err;
    MOE_REQUIRE(T >= 0 && d > 0 && k >= 1 && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (y_perm && slot_of && out), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(d % 8 == 0 && moe_aligned16(y_perm) && moe_aligned16(out), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (T == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    k_combine<<<T, 128, 0, s>>>((const uint4*)y_perm, slot_of, topk_w, nullptr, d / 8, k, (uint4*)out);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_unpermute_combine_add(const void* y_perm, const int32_t* slot_of, const float* topk_w,
                                                  const float* addend, int T, int d, int k, void* out, int32_t* err,
                                                  void* stream) {
    (void)err;
    MOE_REQUIRE(T >= 0 && d > 0 && k >= 1 && k <= 32, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (y_perm && slot_of && out && addend), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(d % 8 == 0 && moe_aligned16(y_perm) && moe_aligned16(out) && moe_aligned16(addend), MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    if (T == 0) return MOE_OK;
    k_combine<<<T, 128, 0, (cudaStream_t)stream>>>((const uint4*)y_perm, slot_of, topk_w, (const float4*)addend, d / 8,
                                                   k, (uint4*)out);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

// dst[c][r] = bf16(src[r][c]) (src bf16 or fp32): 32 x 32 tiles through
// shared memory, coalesced on both sides.
template <typename Src>
__global__ void __launch_bounds__(256) k_transpose(const Src* __restrict__ src, int64_t rows, int64_t cols,
                                                   uint16_t* __restrict__ dst) {
    __shared__ uint16_t tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        const int64_t r = r0 + ty + i, c = c0 + tx;
        uint16_t v = 0;
        if (r < rows && c < cols) {
            if constexpr (sizeof(Src) == 4) {
                __nv_bfloat16 b = __float2bfloat16_rn(src[r * cols + c]);
                v = *reinterpret_cast<uint16_t*>(&b);
            } else {
                v = src[r * cols + c];
            }
        }
        tile[ty + i][tx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        const int64_t c = c0 + ty + i, r = r0 + tx;
        if (c < cols && r < rows) dst[c * rows + r] = tile[tx][ty + i];
    }
}

extern "C" moe_status_t moe_transpose_bf16(const void* src, int src_fp32, int64_t rows, int64_t cols, void* dst,
                                           void* stream) {
    MOE_REQUIRE(src && dst && rows > 0 && cols > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE((rows + 31) / 32 <= 65535 && (cols + 31) / 32 <= 0x7FFFFFFF, MOE_ERR_UNSUPPORTED);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
    if (src_fp32)
        k_transpose<float><<<grid, 256, 0, (cudaStream_t)stream>>>((const float*)src, rows, cols, (uint16_t*)dst);
    else
        k_transpose<uint16_t><<<grid, 256, 0, (cudaStream_t)stream>>>((const uint16_t*)src, rows, cols,
                                                                      (uint16_t*)dst);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_combine_bwd(const void* dout, const void* y_perm, const int32_t* slot_of,
                                        const float* topk_w, const int32_t* row_id, const int32_t* gofs, int T, int d,
                                        int k, int E, int64_t row_cap, void* dy_perm, float* dw, int32_t* err,
                                        void* stream) {
    (void)err;
    MOE_REQUIRE(T >= 0 && d > 0 && k >= 1 && k <= 32 && E >= 1 && row_cap > 0, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(dy_perm == nullptr || (row_id && gofs), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(T == 0 || (dout && y_perm && slot_of && topk_w && dw), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(d % 8 == 0 && moe_aligned16(dy_perm) && (T == 0 || (moe_aligned16(dout) && moe_aligned16(y_perm))),
                MOE_ERR_ALIGNMENT);
    MOE_REQUIRE(device_initialized(), MOE_ERR_NOT_INITIALIZED);
    cudaStream_t s = (cudaStream_t)stream;
    if (T > 0) {
        k_combine_bwd<<<T, 128, 0, s>>>((const uint4*)dout, (const uint4*)y_perm, slot_of, topk_w, d / 8, k,
                                        (uint4*)dy_perm, dw);
        MOE_CHECK_LAUNCH();
    }
    if (dy_perm == nullptr) return MOE_OK;
    k_zero_padding_rows<<<rows_grid(row_cap), 256, 0, s>>>(row_id, gofs + E, row_cap, d / 8, (uint4*)dy_perm);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
