/*
 * moe.h -- C ABI of libmoe: the single-GPU hot path of dropless
 * Mixture-of-Experts training on GB300 (sm_103a).
 *
 * Sources (by page title and section):
 *   [TE-JAX] "NVIDIA Accelerates Dropless MoE Training in JAX Using Transformer
 *            Engine": "What specialized optimizations are required for
 *            dropless MoE?" (Figure 3), "Optimization 1: Grouped GEMM",
 *            "Optimization 2: Expert parallelism to integrate Dispatch and
 *            Combine".
 *   [CH1]    AI Systems Performance Engineering ch.1 ("第一章：介绍与 AI 系统
 *            概览"): §1.1 "数据精度" (FP8 E4M3 = 1+4+3 bits, FP4 = 1+2+1) and
 *            "低精度格式的缩放机制" (MXFP8: one scale per block of 32; NVFP4:
 *            an E4M3 scale per block plus an FP32 scale per tensor);
 *            §2.3.2 "MoE 推理优化" (combine = router-weighted sum; DeepSeek-V3's
 *            shared expert).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer is DEVICE memory owned by the caller unless stated.  The
 *   library never allocates, frees, synchronizes or copies to the host on
 *   these calls, so each one may be captured in a CUDA graph.  `stream` is a
 *   cudaStream_t (NULL = legacy default stream).  Grid sizes depend only on
 *   the host integers passed in and on the SM count, never on device data.
 * - Host-checkable problems (NULL pointers, sizes, 16-byte alignment,
 *   workspace too small) return a status synchronously and launch nothing.
 * - Problems found on the device (an expert index out of range, offsets that
 *   are not monotone or not multiples of 128, a bounded wait that ran out)
 *   are written once into the caller's int32 word `*err` with atomicCAS
 *   (first error wins; the caller zeroes it and reads it when it chooses).
 *   `err` may be NULL.  A kernel that detects such a problem skips the work
 *   it cannot do safely; it never traps.
 * - bf16 tensors are passed as void* (IEEE bfloat16, row-major).
 * - Per-expert token counts stay on the device; nothing here reads them on
 *   the host ([TE-JAX] "What specialized optimizations...": shapes must work
 *   when they are not visible to the CPU, to allow CUDA graphs).
 *
 * Row layout of the permuted (expert-grouped) buffers
 * ---------------------------------------------------
 * Group (expert) e occupies rows [gofs[e], gofs[e+1]) of every permuted
 * buffer, gofs[e] = sum_{h<e} ceil128(counts[h]).  Its first counts[e] rows
 * are the routed (token, choice) pairs in token order; the rest (< 128 rows)
 * are zero padding, so a 128-row GEMM tile never straddles two groups and a
 * 32-row quantization block never crosses a group boundary.  An empty group
 * has no rows.  Buffers are sized for moe_row_capacity(T, E, k) rows; rows at
 * or beyond gofs[E] are never read or written by any call (the transposed
 * NVFP4 output of nvfp4_quantize_cols states its own rule).
 *
 * MXFP8 tensors
 * -------------
 * codes: uint8 FP8 E4M3 (bias 7, max 448, S.1111.111 = NaN).
 * scales: uint8 E8M0 (value 2^(b-127)), one per block of 32 elements along
 * the quantized axis.  Scale rule: b = e + 127 with e the smallest integer
 * such that amax <= 448 * 2^e (clamped to [-127, 127]); an all-zero block has
 * b = 0.  Codes are round-to-nearest-even of x * 2^-e, sign kept.
 *
 * Scale layout ("atom layout", the tensor core's native order).  For a
 * quantized matrix Q with R rows (R % 128 == 0) whose rows are split into
 * 32-element blocks along C columns (C % 128 == 0), the scale of row r,
 * block b (= column / 32) is at byte
 *     ((b / 4) * (R / 128) + r / 128) * 512
 *       + (r % 32) * 16 + ((r / 32) % 4) * 4 + (b % 4)
 * i.e. one 512-byte atom per 128 rows x 4 blocks, atoms ordered by block
 * group first.  A columnwise-quantized matrix is stored transposed (Q = X^T)
 * and uses the same formula on Q.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL pointer or size out of range          */
    MOE_ERR_UNSUPPORTED = 2,   /* shape the kernels do not handle            */
    MOE_ERR_ALIGNMENT = 3,     /* pointer or stride not 16-byte aligned      */
    MOE_ERR_WORKSPACE = 4,     /* workspace too small                        */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime call failed                 */
    MOE_ERR_NOT_INITIALIZED = 6, /* moe_init was not called for this device  */
    /* device-side codes, written to *err */
    MOE_ERR_BAD_EXPERT = 16,   /* topk_idx outside [0, E) or repeated in a row */
    MOE_ERR_BAD_OFFSETS = 17,  /* group offsets not monotone / not 128-aligned /
                                  beyond the buffer                         */
    MOE_ERR_DEVICE_TIMEOUT = 18, /* a bounded wait inside a kernel gave up   */
    MOE_ERR_CAPACITY = 19      /* padded rows exceed the buffer capacity     */
} moe_status_t;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;
typedef enum {
    MOE_QUANT_ROWWISE = 0,
    MOE_QUANT_COLWISE_GROUPED = 1,
    MOE_QUANT_COLWISE_GLU = 2,
    MOE_QUANT_COLWISE_BATCHED = 3,
    MOE_QUANT_COLWISE_BATCHED_GLU = 4
} moe_quant_axis_t;
typedef enum { MOE_GEMM_FWD = 0, MOE_GEMM_DGRAD = 1, MOE_GEMM_WGRAD = 2 } moe_gemm_mode_t;
typedef enum { MOE_EPI_NONE = 0, MOE_EPI_SWIGLU = 1, MOE_EPI_SWIGLU_BWD = 2, MOE_EPI_NONE_F32 = 3 } moe_epilogue_t;
typedef enum {
    MOE_B_GNK = 0,  /* codes [G][N][K]: rowwise-quantized (scales: atom layout of
                       the [G*N, K] matrix)                                    */
    MOE_B_NGK = 1,  /* codes [N][G*K]: the columnwise (transposed) output of a
                       [G*K, N] weight with group offsets g*K (scales: atom
                       layout of the [N, G*K] matrix)                          */
    MOE_B_SF_TILE224 = 2  /* MOE_GEMM_WGRAD only: b's scales in the tile-224
                       layout (below); selects 256 x 224 CTA-pair tiles with
                       two TMEM accumulators per CTA                           */
} moe_b_layout_t;

/*
 * Scale layouts of a quantized matrix Q [R, C] (blocks of 32 along C):
 *   MOE_SF_ATOMS     the atom layout (above).
 *   MOE_SF_TILE224   rows in tiles of 224: for k-block kb (128 columns, 4
 *                    blocks) and row tile t (rows [224 t, 224 t + 224)),
 *                    1024 bytes at (kb * ceil(R / 224) + t) * 1024; inside, row
 *                    r' = r - 224 t, block b at
 *                        (r' / 128) * 512 + (r' % 32) * 16 + ((r' / 32) % 4) * 4
 *                          + (b % 4),
 *                    i.e. the atom layout of each tile on its own, two atoms
 *                    per tile (rows 224..255 of the second atom unused).
 *                    Size (C / 128) * ceil(R / 224) * 1024 bytes.  This is the
 *                    layout the 224-wide weight-gradient tiles read for their
 *                    right operand (MOE_B_SF_TILE224): a 224-row tile starts on
 *                    an atom of its own, which 224-row tiles of the plain atom
 *                    layout do not.
 *   MOE_SF_CANONICAL row-major [R, C / 32]: byte r * (C / 32) + b is the scale
 *                    of row r, block b (mxfp8_group_quantize_ex only; the
 *                    GEMMs read the atom layout, mxfp8_scale_layout converts).
 *   MOE_SF_TILE224_AND_ATOMS  both: the tile-224 layout in the first
 *                    (C / 128) * ceil(R / 224) * 1024 bytes, the atom layout
 *                    right after it (columnwise scales of
 *                    mxfp8_gather_quantize_ex and mxfp8_swiglu_bwd_quantize_ex
 *                    only), for weight gradients that run some groups on the
 *                    224-wide tiles and the others on 256-wide ones
 *                    (moe_gemm_opts_t.wgrad_rows_lo / _hi).
 */
typedef enum {
    MOE_SF_ATOMS = 0,
    MOE_SF_TILE224 = 1,
    MOE_SF_CANONICAL = 2,
    MOE_SF_TILE224_AND_ATOMS = 3
} moe_sf_layout_t;

/*
 * Grouped-GEMM kernel selection, per call (the *_ex entry points; the plain
 * entry points use MOE_GEMM_KERNEL_AUTO).  AUTO applies the library's own
 * rule, the kernel measured fastest for the call's mode and shape: WGRAD on
 * the CTA pair; plain-epilogue FWD/DGRAD with K <= 2048, >= 65,536 rows and
 * >= 512 rows per group on the CTA pair; everything else on the 1-SM kernel.
 * The other values force one kernel; every kernel computes the same
 * results (the parity tests run each of them).
 */
typedef enum {
    MOE_GEMM_KERNEL_AUTO = 0,
    MOE_GEMM_KERNEL_1SM = 1,       /* one CTA per 128 x 256 tile (128 x 128 if N % 256 != 0) */
    MOE_GEMM_KERNEL_1SM_N128 = 2,  /* one CTA per 128 x 128 tile, two TMEM accumulators */
    MOE_GEMM_KERNEL_PAIR = 3,      /* a CTA pair (tcgen05 cta_group::2) per 256 x 256 tile
                                      (256 x 128 if N % 256 != 0) */
    MOE_GEMM_KERNEL_PAIR_N128 = 4  /* a CTA pair per 256 x 128 tile, two accumulators per CTA */
} moe_gemm_kernel_t;

/*
 * Options of one grouped-GEMM call (NULL = all defaults).
 *   kernel           moe_gemm_kernel_t.  WGRAD with M % 256 != 0 runs on the
 *                    1-SM kernel whatever is asked, and so does any call if
 *                    no CTA pair fits on the device.  NVFP4 has no 128-wide
 *                    instances: 1SM_N128 runs as 1SM, PAIR_N128 as PAIR.
 *   band             m-tiles per raster band of the persistent tile order
 *                    (consecutive tiles walk the n-tiles of a band of m-tiles
 *                    that share them), 1..64; 0 = the kernel's measured
 *                    default.  On the 1-SM kernel the bands of the fp32
 *                    output (MOE_EPI_NONE_F32) restart at every group's first
 *                    m-tile; elsewhere they run across group boundaries.
 *   register_stores  1: the CTA-pair kernel's plain bf16 epilogue stores
 *                    from registers instead of staging through shared memory
 *                    for TMA stores; 0 = default (TMA stores).
 *   wgrad_rows_lo, wgrad_rows_hi
 *                    MOE_GEMM_WGRAD only: compute only the groups whose row
 *                    count r = gofs[g+1] - gofs[g] passes the filter
 *                      hi == 0:       r >= lo
 *                      lo < hi:       lo <= r < hi
 *                      0 < hi <= lo:  r < hi or r >= lo
 *                    and leave d[g] of every other group as it is.  Swapping
 *                    lo and hi gives the complement, so two calls cover every
 *                    group once, e.g. the mid-size groups on 224-wide tiles
 *                    (MOE_B_SF_TILE224) and the rest on 256-wide tiles.  The
 *                    choice is made on the device from gofs (no host round
 *                    trip).  0, 0 = every group; lo, hi >= 0.  Only the
 *                    CTA-pair kernels filter: a call that runs on the 1-SM
 *                    kernel (M % 256 != 0, MOE_GEMM_KERNEL_1SM*, NVFP4)
 *                    returns MOE_ERR_UNSUPPORTED, as does a filter on FWD or
 *                    DGRAD.
 * Values out of range return MOE_ERR_INVALID_ARG.
 */
typedef struct {
    int kernel;
    int band;
    int register_stores;
    int wgrad_rows_lo;
    int wgrad_rows_hi;
} moe_gemm_opts_t;

/* Calls that may take a workspace (moe_workspace_size). */
typedef enum {
    MOE_OP_ROUTE_TOPK = 0,
    MOE_OP_PERMUTE = 1,
    MOE_OP_GROUP_QUANTIZE = 2,
    MOE_OP_GATHER_QUANTIZE = 3,
    MOE_OP_GROUPED_GEMM = 4,
    MOE_OP_UNPERMUTE_COMBINE = 5,
    MOE_OP_COMBINE_BWD = 6,
    MOE_OP_ROUTE_BWD = 7
} moe_op_t;

/* Version of this ABI (major*100 + minor): 200.  2.0 grew moe_gemm_opts_t
 * by wgrad_rows_lo / wgrad_rows_hi (a caller built against the 1.x struct
 * passes too few bytes) and added MOE_SF_TILE224_AND_ATOMS. */
MOE_API int moe_abi_version(void);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(int status);

/* Select `device`, cache its SM count and set kernel attributes (large shared
 * memory).  Call it once per device before the first call on that device,
 * outside any stream capture.  Calling it again is harmless: every call
 * redoes the set-up in the context current at the time, so a process that
 * resets the device (cudaDeviceReset) calls moe_init again before using the
 * library.  The library works in the runtime API's primary context of each
 * device. */
MOE_API moe_status_t moe_init(int device);

/* Rows a permuted buffer needs: ceil128(T*k + 127*min(E, T*k)). */
MOE_API int64_t moe_row_capacity(int T, int E, int k);

/* Workspace bytes for moe_route_topk / moe_permute (device memory, any
 * content on entry, clobbered). */
MOE_API size_t moe_route_workspace_size(int T, int E);
MOE_API size_t moe_permute_workspace_size(int T, int E);

/*
 * moe_workspace_size -- device workspace bytes that call `op` (moe_op_t)
 * needs for a layer of T tokens, hidden size d, E expert groups (routed plus
 * shared), top-k and expert FFN width f.  Only MOE_OP_ROUTE_TOPK
 * (= moe_route_workspace_size(T, E)) and MOE_OP_PERMUTE
 * (= moe_permute_workspace_size(T, E)) take a workspace; every other op
 * returns 0 (its only scratch is the caller's outputs).  Returns (size_t)-1
 * for an unknown op or sizes out of range (T < 0, d, E, k or f < 1).  Host
 * only, no device call.
 */
MOE_API size_t moe_workspace_size(int op, int T, int d, int E, int k, int f);

/*
 * moe_route_topk -- the router's top-k ([TE-JAX] introduction: the router
 * picks k experts per token; "Optimization 2": routing runs as fused router
 * kernels).
 *   logits   [T, E] fp32.
 *   topk_idx [T, k] int32 out: the k largest logits per token, in
 *            descending order; equal logits go to the lower expert index.
 *   topk_w   [T, k] fp32 out: score = softmax over all E (score 0) or
 *            sigmoid (score 1); normalize != 0 divides by the sum over the
 *            k chosen.
 *   counts   [E] int32 out: pairs routed to each expert (sum = T*k).
 *   offsets  [E+1] int32 out: exclusive prefix sum of counts (unpadded).
 *   ws       >= moe_route_workspace_size(T, E) bytes.
 *   err      not written: routing has no device-side checks (finite logits
 *            are the caller's contract); may be NULL.
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0.
 */
MOE_API moe_status_t moe_route_topk(const float* logits, int T, int E, int k, int score, int normalize,
                            int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                            void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * moe_permute -- local half of dispatch ([TE-JAX] "Optimization 2": tokens
 * are permuted to their experts; local reordering part only).
 *   x          [T, d] bf16 (d % 8 == 0, 16-byte aligned).
 *   topk_idx   [T, k] int32 (from moe_route_topk or the caller).
 *   row_cap    rows of the permuted buffers, >= moe_row_capacity(T, E, k).
 *   gofs       [E+1] int32 out: padded group offsets (multiples of 128).
 *   slot_of    [T, k] int32 out: row of pair (t, j) in the permuted buffers,
 *              slot = gofs[e] + #{t' < t : e in topk_idx[t']} (token order).
 *   row_id     [row_cap] int32 out: t*k + j for the row of pair (t, j), -1
 *              for padding rows; rows >= gofs[E] untouched.
 *   x_perm     [row_cap, d] bf16 out (may be NULL): x_perm[slot_of[t,j]] =
 *              x[t]; padding rows are zero; rows >= gofs[E] untouched.
 *   ws         >= moe_permute_workspace_size(T, E) bytes.
 */
MOE_API moe_status_t moe_permute(const void* x, int T, int d, int E, int k, const int32_t* topk_idx,
                         int64_t row_cap, int32_t* gofs, int32_t* slot_of, int32_t* row_id,
                         void* x_perm, void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * mxfp8_group_quantize -- MXFP8 quantization, 1x32 blocks, E8M0 scales
 * ([TE-JAX] "What specialized optimizations...": a group-aware MXFP8
 * quantization; [CH1] "低精度格式的缩放机制").
 *   x      [rows, cols] bf16, rows % 128 == 0, cols % 128 == 0.
 *   axis   MOE_QUANT_ROWWISE: blocks along each row.  codes [rows, cols],
 *          scales in the atom layout of the [rows, cols] matrix.
 *          MOE_QUANT_COLWISE_GROUPED: blocks of 32 rows of one group along
 *          each column.  codes [cols, rows] (transposed), scales in the atom
 *          layout of that [cols, rows] matrix.  Each group's rows start at a
 *          multiple of 128, so blocks restart at every group boundary and
 *          the padding rows inside a group (zeros) pad its tail block.
 *          MOE_QUANT_COLWISE_GLU: as COLWISE_GROUPED, but the output rows
 *          interleave the two column halves in 64-row chunks: output rows
 *          [128j, 128j+64) are input columns [64j, 64j+64) and rows
 *          [128j+64, 128j+128) are input columns [cols/2+64j, cols/2+64j+64).
 *          This is the layout the SwiGLU epilogue of grouped_gemm_mxfp8
 *          expects for the fused gate/up weight (gate = first half).
 *          MOE_QUANT_COLWISE_BATCHED[_GLU]: for G equal groups of
 *          Kg = rows / G rows (a stack of per-expert weights [G][Kg][cols],
 *          Kg % 128 == 0): each group is quantized along its rows and stored
 *          transposed on its own, codes [G][cols][Kg] (row order interleaved
 *          as above for _GLU), scales in the atom layout of the
 *          [G*cols, Kg] matrix.  This is the MOE_B_GNK operand of
 *          grouped_gemm_mxfp8 built from a [G][K][N] weight; gofs is
 *          ignored.  (One expert's operand is contiguous, which on GB300
 *          halves the DRAM traffic of the forward GEMMs against MOE_B_NGK.)
 *   gofs   [G+1] int32 (device) or NULL.  If given, rows >= gofs[G] are not
 *          read and their codes/scales are not written; for the columnwise
 *          axis gofs is validated (monotone, multiples of 128, <= rows).
 */
MOE_API moe_status_t mxfp8_group_quantize(const void* x, int64_t rows, int cols, int axis,
                                  const int32_t* gofs, int G, uint8_t* codes, uint8_t* scales,
                                  int32_t* err, void* stream);
/*
 * mxfp8_group_quantize_ex -- mxfp8_group_quantize with the padded group
 * offsets as an output and the scale layout chosen.
 *   padded_offsets  [G+1] int32 out (device) or NULL: the first row of group
 *                   g in the blocked axis of the output, i.e. where its
 *                   blocks start (the column of the transposed columnwise
 *                   codes; the row of the rowwise codes).  For the grouped
 *                   axes these are gofs (the groups already start at
 *                   multiples of 128, see below); for the batched axes
 *                   g * rows / G.  Needs gofs unless the axis is batched.
 *   scale_layout    MOE_SF_ATOMS (as mxfp8_group_quantize) or
 *                   MOE_SF_CANONICAL: row-major [R, C / 32] for the output
 *                   matrix Q [R, C] quantized along C, where Q is [rows, cols]
 *                   for MOE_QUANT_ROWWISE, [cols, rows] for the columnwise
 *                   axes and [G * cols, rows / G] for the batched ones (the
 *                   same bytes as the atoms, placed in row order).
 */
MOE_API moe_status_t mxfp8_group_quantize_ex(const void* x, int64_t rows, int cols, int axis,
                                             const int32_t* gofs, int G, uint8_t* codes, uint8_t* scales,
                                             int32_t* padded_offsets, int scale_layout, int32_t* err,
                                             void* stream);
/*
 * Padded offsets of the group-aware columnwise output.  The plain definition
 * of the group-aware quantization pads group g's tail block and places the
 * group at sum_{h<g} ceil32(m_h) rows.  Here the permute already places
 * every group at a multiple of 128 rows (gofs, moe_permute), which is a
 * multiple of 32, with zero rows after its m_g routed rows: the padded
 * offsets of this output ARE gofs (mxfp8_group_quantize_ex writes them out
 * as padded_offsets).  Block j of group g covers rows gofs[g] + 32 j ..;
 * blocks past ceil32(m_g) rows of the group hold only zero rows (scale
 * byte 0, codes 0).
 *
 * Scale layout.  The hot path reads and writes scales in the atom layout
 * (the tensor cores' order, above), so no conversion runs there;
 * mxfp8_group_quantize_ex writes the canonical row-major [R, C / 32] layout
 * on request, and mxfp8_scale_layout converts between the two.
 */

/*
 * mxfp8_scale_layout -- converts the scales of a [rows, cols] matrix
 * quantized along cols between the atom layout and the canonical row-major
 * layout, where byte r * (cols / 32) + b is the scale of row r, block b.
 *   to_canonical 1: src = atoms, dst = canonical; 0: the reverse.
 *   src, dst     rows * cols / 32 bytes each (device), not overlapping.
 * rows % 128 == 0, cols % 128 == 0.  Pure data movement, one launch.
 */
MOE_API moe_status_t mxfp8_scale_layout(const uint8_t* src, int64_t rows, int cols, int to_canonical, uint8_t* dst,
                                        void* stream);

/*
 * mxfp8_gather_quantize -- the rowwise and the group-aware columnwise MXFP8
 * quantization of one (virtual) permuted matrix, from a single read of its
 * rows ([TE-JAX] "What specialized optimizations...": group-aware
 * quantization; "Optimization 2": the local permute feeding the grouped
 * GEMM).  Row s of the matrix P [rows, cols] is
 *   row_id == NULL:         P[s] = src[s]                 (src [rows, cols])
 *   row_id[s] < 0:          P[s] = 0                      (padding row)
 *   row_w == NULL:          P[s] = src[row_id[s] / k]     (src [T, cols])
 *   otherwise:              P[s] = bf16(row_w[row_id[s]] * src[row_id[s] / k])
 * so P is x_perm when src = x (a gather) and dy_perm of moe_combine_bwd
 * when src = dout and row_w = topk_w; neither is ever stored in bf16.
 *   src       [src_rows, cols] bf16, 16-byte aligned; cols % 128 == 0.
 *             Without row_id, src_rows must equal rows.
 *   row_id    [rows] int32 (from moe_permute) or NULL; k its tokens' top-k.
 *             An entry with row_id[s] / k >= src_rows (below gofs[G]) sets
 *             MOE_ERR_INVALID_ARG in *err and its row is read as zero.
 *   gofs      [G+1] int32 group offsets (multiples of 128, monotone,
 *             gofs[G] <= rows; validated, MOE_ERR_BAD_OFFSETS in *err and
 *             nothing written if not).  Rows >= gofs[G] are not read and
 *             their outputs are not written.
 *   rows      the row capacity, % 128 == 0.
 *   codes_row, scales_row   exactly MOE_QUANT_ROWWISE's output for P, or
 *             both NULL.
 *   codes_col, scales_col   exactly MOE_QUANT_COLWISE_GROUPED's output for
 *             P (codes [cols, rows]), or both NULL.  At least one pair.
 * All pointers are device pointers; outputs 16-byte aligned, codes_row and
 * codes_col 32-byte aligned (MOE_ERR_ALIGNMENT otherwise).
 */
MOE_API moe_status_t mxfp8_gather_quantize(const void* src, int64_t src_rows, int cols, int k,
                                   const int32_t* row_id,
                                   const float* row_w, const int32_t* gofs, int G, int64_t rows,
                                   uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col,
                                   uint8_t* scales_col, int32_t* err, void* stream);

/* mxfp8_gather_quantize with the layout of scales_col chosen (moe_sf_layout_t):
 * MOE_SF_TILE224 writes the columnwise scales in the tile-224 layout of the
 * [cols, rows] transposed matrix ((rows / 128) * ceil(cols / 224) * 1024
 * bytes; bytes of rows >= cols in the last tile are not written), the
 * right-operand scales of grouped_gemm_mxfp8 WGRAD with MOE_B_SF_TILE224;
 * MOE_SF_TILE224_AND_ATOMS writes that and, right after it, the atom layout
 * ((rows / 32) * cols more bytes).  The codes and the rowwise output are
 * unchanged; MOE_SF_CANONICAL is not accepted here (MOE_ERR_INVALID_ARG). */
MOE_API moe_status_t mxfp8_gather_quantize_ex(const void* src, int64_t src_rows, int cols, int k,
                                              const int32_t* row_id, const float* row_w, const int32_t* gofs, int G,
                                              int64_t rows, uint8_t* codes_row, uint8_t* scales_row,
                                              uint8_t* codes_col, uint8_t* scales_col, int col_sf_layout,
                                              int32_t* err, void* stream);

/*
 * mxfp8_swiglu_bwd_quantize -- the SwiGLU backward fused with the two-axis
 * MXFP8 quantization of its result ([TE-JAX] "What specialized
 * optimizations...": group-aware MXFP8 quantization; Figure 3's grouped MLP
 * run backward).  dA = [dgate | dup] [rows, 2f] with, per element,
 *   s = sigmoid(g), dgate = dH*u*s*(1 + g*(1 - s)), dup = dH*g*s
 * where [g | u] = a_pre, computed in fp32 and rounded to bf16; dA is then
 * quantized exactly as mxfp8_gather_quantize quantizes a stored [rows, 2f]
 * bf16 matrix (both axes, group-aware columnwise blocks).
 *   dH        [rows, f] fp32 (grouped_gemm_mxfp8 DGRAD with MOE_EPI_NONE_F32).
 *   a_pre     [rows, 2f] bf16 (the up/gate GEMM's result).
 *   dA        [rows, 2f] bf16 or NULL: the bf16 values, written only if given.
 *   gofs      as for mxfp8_gather_quantize; rows >= gofs[G] untouched.
 *   codes_row, scales_row, codes_col, scales_col   both axes, required.
 * f % 128 == 0, rows % 128 == 0, 16-byte aligned pointers (codes_col
 * 32-byte aligned).
 */
MOE_API moe_status_t mxfp8_swiglu_bwd_quantize(const float* dH, const void* a_pre, int f, const int32_t* gofs,
                                       int G, int64_t rows, void* dA, uint8_t* codes_row, uint8_t* scales_row,
                                       uint8_t* codes_col, uint8_t* scales_col, int32_t* err, void* stream);

/* mxfp8_swiglu_bwd_quantize with the layout of scales_col chosen, as for
 * mxfp8_gather_quantize_ex (the transposed matrix is [2f, rows]). */
MOE_API moe_status_t mxfp8_swiglu_bwd_quantize_ex(const float* dH, const void* a_pre, int f, const int32_t* gofs,
                                                  int G, int64_t rows, void* dA, uint8_t* codes_row,
                                                  uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                                                  int col_sf_layout, int32_t* err, void* stream);

/*
 * grouped_gemm_mxfp8 -- one launch for all experts' GEMMs, each over its own
 * rows only ([TE-JAX] "Optimization 1: Grouped GEMM"), MXFP8 block-scaled
 * operands, fp32 accumulation, bf16 output.  Group offsets are read on the
 * device (no host copy of counts).  K-major fp8 operands; K % 128 == 0.
 *
 * MOE_GEMM_FWD / MOE_GEMM_DGRAD (same kernel; dgrad passes the weight copy
 * quantized along the other axis):
 *   a, a_sf   [M, K] rowwise codes/scales of the permuted activations;
 *             M = row capacity (% 128 == 0); rows of group g are
 *             [gofs[g], gofs[g+1]).
 *   b, b_sf   the group weights B_g as [N, K] K-major blocks, b_layout.
 *   out       row r of group g: D[r, n] = sum_k A[r, k] * B_g[n, k].
 *   epilogue  MOE_EPI_NONE:       d = D [M, N] bf16.
 *             MOE_EPI_SWIGLU:     (fwd up/gate) N = 2f; B must be in the
 *                                 MOE_QUANT_COLWISE_GLU row order (gate and
 *                                 up rows interleaved in 64-row chunks, the
 *                                 gate is logical column n < f); d = a_pre
 *                                 [M, N] bf16 (the GEMM result), d2 = h
 *                                 [M, N/2] bf16, h = silu(gate) * up computed
 *                                 from the fp32 accumulators, in the
 *                                 logical [gate | up] column order.
 *             MOE_EPI_SWIGLU_BWD: (dgrad down) N = f, D = dH;
 *                                 epi_aux = a_pre [M, 2N] bf16; d = dA
 *                                 [M, 2N] bf16 = [dgate | dup] with
 *                                 dgate = dH*u*s*(1+g*(1-s)), dup = dH*g*s,
 *                                 s = sigmoid(g).
 *             MOE_EPI_NONE_F32:   d = D [M, N] fp32 (the accumulators as
 *                                 they are; e.g. dH for
 *                                 mxfp8_swiglu_bwd_quantize).
 *             N % 128 == 0 for every epilogue.
 * MOE_GEMM_WGRAD:
 *   a, a_sf   [M, K] columnwise codes (the transposed left operand, e.g.
 *             h^T); K = row capacity; group g contracts over columns
 *             [gofs[g], gofs[g+1]).
 *   b, b_sf   [N, K] columnwise codes of the right operand.  b_layout
 *             MOE_B_GNK or MOE_B_NGK: b_sf in the atom layout;
 *             MOE_B_SF_TILE224: b_sf in the tile-224 layout of the [N, K]
 *             matrix (M % 256 == 0 then; the call runs 256 x 224 CTA-pair
 *             tiles whatever the options ask, or returns MOE_ERR_UNSUPPORTED
 *             where no CTA pair fits).
 *   d         [G, M, N] bf16: d[g] = A_g * B_g^T over the group's rows;
 *             an empty group writes zeros.  M % 128 == 0, N % 128 == 0.
 * d, d2, epi_aux: 16-byte aligned.  Launch: one persistent CTA per SM.
 */
MOE_API moe_status_t grouped_gemm_mxfp8(int mode, const uint8_t* a, const uint8_t* a_sf,
                                const uint8_t* b, const uint8_t* b_sf, int b_layout,
                                const int32_t* gofs, int G, int64_t M, int N, int64_t K,
                                int epilogue, const void* epi_aux, void* d, void* d2,
                                int32_t* err, void* stream);

/* grouped_gemm_mxfp8 with per-call kernel options (moe_gemm_opts_t, may be
 * NULL = grouped_gemm_mxfp8). */
MOE_API moe_status_t grouped_gemm_mxfp8_ex(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                           const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G, int64_t M,
                                           int N, int64_t K, int epilogue, const void* epi_aux, void* d, void* d2,
                                           const moe_gemm_opts_t* opts, int32_t* err, void* stream);

/*
 * grouped_gemm_mxfp8_swiglu_quant -- the up/gate GEMM (MOE_GEMM_FWD,
 * MOE_EPI_SWIGLU) with the MXFP8 quantization of h fused into its epilogue
 * ([TE-JAX] "What specialized optimizations...": group-aware MXFP8
 * quantization; "What is the training performance impact...": quantization
 * fused with the GEMM is listed there as planned work).  Arguments as for
 * grouped_gemm_mxfp8 with mode FWD and epilogue SWIGLU (N % 256 == 0), and:
 *   a_pre        [M, N] bf16, written (the GEMM result).
 *   h            [M, N/2] bf16 or NULL: written only if given.
 *   h_codes_row, h_scales_row   exactly mxfp8_gather_quantize's rowwise
 *                output for h (codes [M, N/2], 32-byte aligned).
 *   h_codes_col, h_scales_col   exactly its columnwise output for h (codes
 *                [N/2, M]).
 * Every code is computed from the bf16-rounded h (the value `h` holds when
 * given).  Rows >= gofs[G] are not written.
 */
MOE_API moe_status_t grouped_gemm_mxfp8_swiglu_quant(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                             const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G,
                                             int64_t M, int N, int64_t K, void* a_pre, void* h,
                                             uint8_t* h_codes_row, uint8_t* h_scales_row, uint8_t* h_codes_col,
                                             uint8_t* h_scales_col, int32_t* err, void* stream);

/* grouped_gemm_mxfp8_swiglu_quant with per-call kernel options (may be NULL). */
MOE_API moe_status_t grouped_gemm_mxfp8_swiglu_quant_ex(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                                        const uint8_t* b_sf, int b_layout, const int32_t* gofs, int G,
                                                        int64_t M, int N, int64_t K, void* a_pre, void* h,
                                                        uint8_t* h_codes_row, uint8_t* h_scales_row,
                                                        uint8_t* h_codes_col, uint8_t* h_scales_col,
                                                        const moe_gemm_opts_t* opts, int32_t* err, void* stream);

/*
 * gemm_bf16_nt -- dense D = A * B^T with bf16 operands on the tensor cores
 * (tcgen05.mma kind::f16, fp32 accumulation): the router's GEMMs ([TE-JAX]
 * "Optimization 2": the fused router kernels assign tokens to experts from
 * the router's scores; the logits are x * W_r).
 *   a   [M, K] bf16 row-major (K contiguous); M % 128 == 0.
 *   b   [N, K] bf16 row-major; N % 8 == 0 (any N: columns are computed in
 *       256-wide tiles and the tile's columns >= N are not stored).
 *   d   [M, N] fp32 row-major, 32-byte aligned: D[m, n] = sum_k a[m,k] b[n,k].
 *   K % 8 == 0 (16-byte rows); a and b 16-byte aligned.
 */
MOE_API moe_status_t gemm_bf16_nt(const void* a, const void* b, int64_t M, int N, int64_t K, float* d, int32_t* err,
                          void* stream);

/*
 * moe_transpose_bf16 -- dst [cols, rows] bf16 = transpose of src [rows,
 * cols] (bf16, or fp32 rounded to bf16 nearest-even when src_fp32 != 0).
 * The router backward's K-major operands (x^T, dlogits^T).
 */
MOE_API moe_status_t moe_transpose_bf16(const void* src, int src_fp32, int64_t rows, int64_t cols, void* dst,
                                void* stream);

/*
 * moe_unpermute_combine_add -- moe_unpermute_combine plus an fp32 addend
 * [T, d] (16-byte aligned): out[t] = bf16(addend[t] + sum_j w[t,j] y[slot(t,j)]),
 * summed in fp32 in that order; the router's input gradient joins the
 * experts' here.
 */
MOE_API moe_status_t moe_unpermute_combine_add(const void* y_perm, const int32_t* slot_of, const float* topk_w,
                                       const float* addend, int T, int d, int k, void* out, int32_t* err,
                                       void* stream);

/*
 * moe_unpermute_combine -- local half of combine ([TE-JAX] "Optimization 2":
 * per-expert results are accumulated and restored to token order; [CH1]
 * §2.3.2: a sum weighted by the routing weights).
 *   out[t] = sum_{j<k} w[t, j] * y_perm[slot_of[t, j]]  (fp32 sum in j
 *   order, bf16 out).  topk_w == NULL means weights of 1 (the unpermute-sum
 *   used for dx).  y_perm [*, d] bf16, out [T, d] bf16, d % 8 == 0.
 */
MOE_API moe_status_t moe_unpermute_combine(const void* y_perm, const int32_t* slot_of, const float* topk_w,
                                   int T, int d, int k, void* out, int32_t* err, void* stream);

/*
 * moe_combine_bwd -- adjoint of the weighted combine of
 * moe_unpermute_combine ([TE-JAX] "Optimization 2" and [CH1] §2.3.2 define
 * the forward combine, a sum weighted by the routing weights; the pages give
 * no backward.  Reading: the backward of every step is the plain gradient of
 * its forward, with the MXFP8 quantization passed through as the identity,
 * and the product w * dout is rounded once to fp32 and then to bf16, the
 * activations' type).
 *   dy_perm[slot_of[t, j]] = bf16(w[t, j] * dout[t]); padding rows (row_id
 *   == -1, below gofs[E]) are written as zeros.
 *   dw[t, j] = <dout[t], y_perm[slot_of[t, j]]> (fp32).
 *   dy_perm may be NULL: only dw is computed (row_id and gofs may then be
 *   NULL too); mxfp8_gather_quantize then builds the quantized dy_perm
 *   straight from dout.
 */
MOE_API moe_status_t moe_combine_bwd(const void* dout, const void* y_perm, const int32_t* slot_of,
                             const float* topk_w, const int32_t* row_id, const int32_t* gofs,
                             int T, int d, int k, int E, int64_t row_cap, void* dy_perm, float* dw,
                             int32_t* err, void* stream);

/*
 * moe_route_bwd -- gradient of the routing weights with respect to the
 * logits (the backward of moe_route_topk's weights: [TE-JAX] introduction
 * and "Optimization 2" define the forward routing, the pages give no
 * backward.  Reading: the plain gradient of the forward scores; the top-k
 * selection itself is piecewise constant and has none).
 * dlogits [T, E] fp32 out (every entry written).
 *   softmax+normalize: dl_i = w_i (dw_i - sum_j w_j dw_j) on the chosen, 0 else
 *   softmax raw:       dl_m = p_m ([m chosen] dw_m - sum_j p_j dw_j) for all m
 *   sigmoid+normalize: dl_i = s_i (1-s_i) (dw_i - sum_j w_j dw_j) / sum s
 *   sigmoid raw:       dl_i = s_i (1-s_i) dw_i on the chosen, 0 else
 */
MOE_API moe_status_t moe_route_bwd(const float* logits, const int32_t* topk_idx, const float* dw,
                           int T, int E, int k, int score, int normalize, float* dlogits,
                           int32_t* err, void* stream);

/*
 * moe_route_append_shared -- shared experts (experts every token uses, with
 * weight 1; DeepSeek-V3 has one, [CH1] §2.3.2 MoE structure) as extra
 * choices: idx_out [T, k+S] = [topk_idx | E, E+1, .., E+S-1] and w_out
 * [T, k+S] = [topk_w | 1, .., 1] per token (S = n_shared).  Permute, the
 * grouped GEMMs (E+S groups) and the combine then need nothing else: each
 * shared expert's group holds every token, and its output joins the
 * combine with weight 1.  k + S <= 32.
 */
MOE_API moe_status_t moe_route_append_shared(const int32_t* topk_idx, const float* topk_w, int T, int k, int E,
                                     int n_shared, int32_t* idx_out, float* w_out, void* stream);

/*
 * moe_route_drop_shared -- dw [T, k] = the routed columns of dw_all [T, k+S]
 * (the shared choices' weights are constants; their dw is not used).
 */
MOE_API moe_status_t moe_route_drop_shared(const float* dw_all, int T, int k, int n_shared, float* dw, void* stream);

/*
 * moe_route_topk_noalloc -- moe_route_topk for callers that cannot allocate.
 * (The pages have no counterpart: this is a calling convention, not a step of
 * the method.)  Some callers cannot hand the library any device memory
 * beyond their inputs and outputs: code behind a plugin or operator
 * interface that passes only tensor pointers, processes whose device memory
 * belongs to a fixed pool they cannot grow, and code that must not call
 * cudaMalloc because it can synchronise the device or is not allowed while
 * a stream is being captured.  This entry point takes the same arguments as
 * moe_route_topk minus the workspace and computes the same results; its
 * scratch (one histogram of E counters per 128 tokens) is a fixed 1 MiB
 * device array inside the library, which every GPU that loads the library
 * keeps until the process exits.
 *   Limit: ceil(T / 128) * E <= 262144 (e.g. T = 131072 with E = 256);
 *   larger sizes return MOE_ERR_WORKSPACE without launching anything.
 *   It calls no allocator.  Its first call on a device after moe_init looks
 *   up the array's device address (cudaGetSymbolAddress) and keeps it; make
 *   that first call before any stream capture.  moe_init must have been
 *   called for the device (it drops the kept address, so after a device
 *   reset and a new moe_init the address is looked up again).
 *   err is not written (as for moe_route_topk); it may be NULL.
 *   Every call uses the same array, so calls that may overlap on the GPU
 *   (different streams, or several host threads) race with each other; order
 *   them on one stream.  The array keeps the previous call's contents, which
 *   is harmless: each call writes every entry it reads.
 */
MOE_API moe_status_t moe_route_topk_noalloc(const float* logits, int T, int E, int k, int score, int normalize,
                                            int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                            int32_t* err, void* stream);

/*
 * ---------------------------------------------------------------- NVFP4 --
 * [CH1] §1.1 precision table: FP4 is 4 bits, 1 sign + 2 exponent + 1
 * mantissa (E2M1, values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives);
 * "低精度格式的缩放机制": NVFP4 has two scales, an E4M3 scale per small
 * block and one FP32 scale per tensor.  [TE-JAX] "What is the training
 * performance impact…": NVFP4 is planned next for the expert GEMMs.
 * Block size 16 along the contraction axis (the tensor cores' NVFP4 MMA).
 *
 * Code layout: row-major [rows, cols / 2] bytes; element 2j of a row in the
 * low nibble of byte j, element 2j+1 in the high nibble.
 * Scale layout: 16-element block b of row r lives at byte
 *   ((b / 16) * (rows / 128) + r / 128) * 2048 + ((b / 4) % 4) * 512
 *   + (r % 32) * 16 + ((r / 32) % 4) * 4 + b % 4,
 * i.e. per 256-column k-step and 128-row tile four 512-byte atoms (one per
 * 64 columns) in the tensor cores' scale-factor layout.
 */

/* nvfp4_sf_bytes -- bytes of the scale array of a [rows, cols] matrix
 * (rows * cols / 16), or -1 unless rows % 128 == 0 and cols % 256 == 0. */
MOE_API int64_t nvfp4_sf_bytes(int64_t rows, int cols);

/*
 * nvfp4_quantize -- two-level NVFP4 of a bf16 matrix, blocks of 16 along
 * each row.  In fp32, each step rounded to nearest:
 *   amax = max |src|; s_t = amax / 2688; enc = 2688 / amax (2688 = 6 * 448)
 *   per block: t_b = (amax_b / 6) * enc; scale byte = E4M3(t_b), nearest,
 *              ties to even, saturating at 448; r_b = enc / E4M3 value
 *   per element: code = E2M1(x * r_b), nearest, ties to even, saturating at 6
 * so that x ~ E2M1(code) * scale * s_t.  A block whose scale byte is 0 gets
 * zero codes; an all-zero matrix gives s_t = 0.
 *   src           [rows, cols] bf16 row-major, 16-byte aligned; rows % 128
 *                 == 0, rows / 128 <= 65535, cols % 256 == 0.
 *   codes         [rows, cols / 2] bytes (layout above), written.
 *   scales        nvfp4_sf_bytes(rows, cols) bytes (layout above), written.
 *   tensor_scale  one float (device), written with s_t.
 *   amax_ws       one uint32 of device scratch (zeroed and used by the call;
 *                 calls that may overlap on the GPU need their own word).
 * Two launches (the amax reduction, then the quantization) after a 4-byte
 * memset; no allocation, no host sync.  err is unused (no device-side
 * checks); host-checkable errors are returned.
 */
MOE_API moe_status_t nvfp4_quantize(const void* src, int64_t rows, int cols, uint8_t* codes, uint8_t* scales,
                                    float* tensor_scale, uint32_t* amax_ws, int32_t* err, void* stream);

/*
 * nvfp4_quantize_cols -- group-aware columnwise NVFP4 of a row-permuted
 * bf16 matrix (the weight-gradient operands): blocks of 16 rows of one
 * group along each column, codes written transposed.  Groups start at
 * multiples of 128 rows (gofs as for the grouped GEMM), so no block
 * crosses a group; rows >= gofs[G] are quantized as zeros.  The tensor
 * amax, the fp32 steps and the rounding are those of nvfp4_quantize, over
 * rows [0, gofs[G]).
 *   src           [rows, cols] bf16, 16-byte aligned; rows % 256 == 0,
 *                 cols % 128 == 0.
 *   gofs, G       group offsets (device, G + 1 values, 1 <= G <= 4096):
 *                 gofs[0] == 0, monotone, multiples of 128, gofs[G] <= rows;
 *                 otherwise MOE_ERR_BAD_OFFSETS in err and zero output.
 *   codes_t       [cols, rows / 2] bytes: row c holds column c of src, two
 *                 rows per byte (row 2j in the low nibble).
 *   scales_t      nvfp4_sf_bytes(cols, rows) bytes: the scale layout above
 *                 for the [cols, rows] matrix.
 *   tensor_scale  one float (device), written; amax_ws one uint32 of
 *                 device scratch (zeroed and used by the call).
 */
MOE_API moe_status_t nvfp4_quantize_cols(const void* src, int64_t rows, int cols, const int32_t* gofs, int G,
                                         uint8_t* codes_t, uint8_t* scales_t, float* tensor_scale,
                                         uint32_t* amax_ws, int32_t* err, void* stream);

/*
 * grouped_gemm_nvfp4 -- the grouped GEMM of grouped_gemm_mxfp8 with NVFP4
 * operands on the tensor cores (tcgen05.mma kind::mxf4nvf4, UE4M3 block
 * scales, fp32 accumulation); the epilogue multiplies by a_scale * b_scale.
 * FWD / DGRAD: D[r, :] = A[r, :] * B_g^T for the rows r of group g.
 *   a, a_sf, a_scale   nvfp4_quantize output for A [M, K].
 *   b, b_sf, b_scale   nvfp4_quantize output for the [G * N, K] matrix whose
 *                      rows g*N .. g*N+N-1 are B_g ([G][N][K]; one tensor
 *                      scale for every expert's weights).
 *   gofs, G            0 = gofs[0], monotone, multiples of 128, gofs[G] <= M.
 *   d                  [M, N]; rows >= gofs[G] are not written.
 * WGRAD: D_g[m, n] = sum over the rows r of group g of A^T[r, m] B^T[r, n]
 * (the weight gradient; each group's contraction is its own rows).
 *   a, a_sf, a_scale   nvfp4_quantize_cols output for the row-permuted
 *                      [K, M] operand (codes [M, K / 2]).
 *   b, b_sf, b_scale   nvfp4_quantize_cols output for the [K, N] operand.
 *   gofs, G            as above with gofs[G] <= K; a group of an odd number
 *                      of 128-row tiles ends with a half 256-row k-step.
 *   d                  [G, M, N]; an empty group's D_g is written as zeros.
 * All modes: M % 128 == 0, N % 256 == 0, K % 256 == 0; epilogue
 * MOE_EPI_NONE (bf16 d) or, for FWD and DGRAD, MOE_EPI_NONE_F32 (fp32 d);
 * d 32-byte aligned;
 * bad offsets -> MOE_ERR_BAD_OFFSETS in err; every wait inside the kernel is
 * bounded (MOE_ERR_DEVICE_TIMEOUT in err).
 */
MOE_API moe_status_t grouped_gemm_nvfp4(int mode, const uint8_t* a, const uint8_t* a_sf, const float* a_scale,
                                        const uint8_t* b, const uint8_t* b_sf, const float* b_scale,
                                        const int32_t* gofs, int G, int64_t M, int N, int64_t K, int epilogue,
                                        void* d, int32_t* err, void* stream);

/* grouped_gemm_nvfp4 with per-call kernel options (may be NULL). */
MOE_API moe_status_t grouped_gemm_nvfp4_ex(int mode, const uint8_t* a, const uint8_t* a_sf, const float* a_scale,
                                           const uint8_t* b, const uint8_t* b_sf, const float* b_scale,
                                           const int32_t* gofs, int G, int64_t M, int N, int64_t K, int epilogue,
                                           void* d, const moe_gemm_opts_t* opts, int32_t* err, void* stream);

/*
 * moe_selftest_bounded_wait -- checks the failure path of the kernels'
 * bounded waits without a GPU fault: one thread waits, with the same
 * bounded wait the GEMM kernels use, on an mbarrier that nothing arrives
 * at.  After timeout_ns (1 ns .. 10 s) of the device's nanosecond timer, or
 * 2^22 polls, the wait gives up: *completed = 0 and MOE_ERR_DEVICE_TIMEOUT is
 * written into err (first error wins), and the kernel returns, so the
 * context stays usable.  err and completed are device int32 words.  (The
 * pages have no counterpart: this is a test hook of the library.)
 */
MOE_API moe_status_t moe_selftest_bounded_wait(uint64_t timeout_ns, int32_t* err, int32_t* completed, void* stream);

/*
 * moe_hbm_fill -- writes the 32-bit `value`, repeated, over `bytes` bytes at
 * dst: a write-only stream with no reads, the measuring stick for the
 * write-heavy quantization kernels (and a plain device memset).  (The pages
 * have no counterpart: this is a measuring tool of the library.)
 *   method 0: every thread stores 16-byte vectors (st.global.v4), 4 per
 *             loop trip, grid-stride over the buffer, 8 CTAs of 256
 *             threads per SM;
 *   method 1: each CTA fills a 32 KB shared-memory buffer once and writes it
 *             out with bulk asynchronous copies (cp.async.bulk
 *             .global.shared::cta) of 32 KB, grid-stride, one CTA per SM.
 * dst 16-byte aligned, bytes % 16 == 0.  One launch, no allocation.
 */
MOE_API moe_status_t moe_hbm_fill(void* dst, size_t bytes, uint32_t value, int method, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
