"""Plain, slow CPU oracle of the dropless-MoE training hot path (fp64, numpy).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  It shares no code, tables or helpers with the CUDA path in
``grouped_gemm_top_gb300/``; neither side imports the other.

Every function is the plain definition of one step of the method, written so
that a reader can check it against the pages by eye.  Sources, by page title:

* [TE-JAX] "NVIDIA Accelerates Dropless MoE Training in JAX Using Transformer
  Engine" (the English NVIDIA blog), sections "What are the challenges involved
  in MoE training?", "How is dropless MoE different from capacity-based MoE?",
  "What specialized optimizations are required for dropless MoE?" (Figure 3),
  "Optimization 1: Grouped GEMM" and "Optimization 2: Expert parallelism to
  integrate Dispatch and Combine".
* [CH1] "第一章：介绍与 AI 系统概览" (AI Systems Performance Engineering,
  chapter 1): §1.1 "数据精度" (the precision table and the FP32 storage worked
  example), "低精度格式的缩放机制" (MXFP8: one scale per block of 32),
  §2.3.2 "MoE 推理优化" (dispatch/combine table and figure: combine is a
  router-weighted sum), §4.1 "FlashAttention" (softmax worked example).

Where the pages are silent the plainest reading is taken; each such reading is
marked "Reading:" below.  Pins for every function live in
``tests/test_oracle_*.py``; no function here is "parity unpinned".

Conventions: floating point inputs are numpy arrays whose values are exactly
representable in the GPU input type (bf16 activations/weights, fp32 logits);
all arithmetic is fp64; outputs are fp64 unless they are integers or codes.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "MXFP8_BLOCK", "E4M3_MAX", "bf16_round", "e4m3_value", "E4M3_VALUES", "e4m3_encode", "e8m0_exponent",
    "e8m0_byte", "e8m0_value", "mxfp8_quantize_rows", "mxfp8_quantize_cols_grouped",
    "mxfp8_dequantize_rows", "mxfp8_dequantize_cols", "route_topk", "group_counts",
    "group_offsets", "aligned_group_offsets", "permute_slots", "permute", "fp32_round", "permute_scaled_bf16",
    "grouped_gemm", "grouped_gemm_wgrad", "swiglu", "swiglu_bwd", "combine",
    "combine_bwd", "route_bwd", "layer_forward", "layer_backward", "router_logits", "router_backward",
    "append_shared", "NVFP4_BLOCK", "E2M1_MAX", "e2m1_value", "E2M1_VALUES", "e2m1_encode", "nvfp4_tensor_scale",
    "nvfp4_quantize_rows", "nvfp4_dequantize_rows", "nvfp4_quantize_cols_grouped", "nvfp4_dequantize_cols",
]

MXFP8_BLOCK = 32          # [CH1] "低精度格式的缩放机制": one scale per group of 32
E4M3_MAX = 448.0


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def bf16_round(x):
    """Round fp64 values to the nearest bf16 value, ties to even.

    BF16 is 1 sign + 8 exponent + 7 mantissa bits ([CH1] §1.1 precision
    table), i.e. 8 significant bits for normal numbers with the same exponent
    range as FP32 ([CH1] FP32 storage example: bias 127).  Subnormal spacing
    is 2^-133; values that round beyond the largest finite bf16 become inf.
    Used only to state the output type of a GPU result (the GPU writes bf16).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    mant, expo = np.frexp(x[nz])               # x = mant * 2**expo, |mant| in [0.5, 1)
    # a normal bf16 with value in [2^(expo-1), 2^expo) has spacing 2^(expo-8)
    ulp_exp = np.maximum(expo - 8, -133)
    q = np.rint(np.ldexp(x[nz], -ulp_exp))     # np.rint rounds half to even
    r = np.ldexp(q, ulp_exp)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[nz] = r
    out[~nz] = x[~nz]                           # keeps the sign of zero
    return out


def e4m3_value(code: int) -> float:
    """Value of one FP8 E4M3 code: 1 sign, 4 exponent, 3 mantissa bits.

    The bit split is [CH1] §1.1 precision table ("E4M3: 1+4+3").  Reading (the
    pages give only the split): the OCP FP8 E4M3 definition -- exponent bias
    7 (2^(n-1)-1 as in the FP32 example), subnormals m/8 * 2^-6 at exponent
    field 0, no infinities, S.1111.111 is NaN, largest finite 448.
    """
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - 7)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_VALUES = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
_E4M3_POS = E4M3_VALUES[:127]     # codes 0x00..0x7E: finite, non-negative, increasing


def e4m3_encode(v):
    """Encode exact fp64 values to E4M3 codes: nearest value, ties to the even
    code, magnitudes above 448 saturate to 448, the sign bit is kept (so -0 and
    negatives that round to zero give 0x80).  Reading: round-to-nearest-even
    with saturation is the conversion the MXFP8 cast performs; NaN/Inf inputs
    are out of scope."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= E4M3_MAX, 126, code)
    sign = np.signbit(v).astype(np.int64)
    return (code.astype(np.int64) | (sign << 7)).astype(np.uint8)


def e8m0_exponent(amax):
    """Block scale exponent e for a block whose largest magnitude is amax.

    [CH1] "低精度格式的缩放机制": each block of 32 gets its own scale whose
    range is set by that block's values.  Reading (the pages do not give the
    rounding rule): e is the smallest integer with amax <= 448 * 2^e, so the
    largest element lands inside E4M3's range without saturating; e is clamped
    to the E8M0 range [-127, 127]; amax == 0 gives e = -127 (byte 0).
    """
    amax = np.asarray(amax, dtype=np.float64)
    e = np.full(amax.shape, -127, dtype=np.int64)
    nz = amax > 0
    guess = np.ceil(np.log2(amax[nz] / E4M3_MAX)).astype(np.int64)
    # make the inequality exact (log2 may be off by one near powers of two)
    for _ in range(2):
        too_small = amax[nz] > E4M3_MAX * np.ldexp(1.0, guess)
        guess = guess + too_small
        too_big = amax[nz] <= E4M3_MAX * np.ldexp(1.0, guess - 1)
        guess = guess - too_big
    e[nz] = guess
    return np.clip(e, -127, 127)


def e8m0_byte(amax):
    """E8M0 scale byte: unsigned, value 2^(b-127), 0xFF is NaN."""
    return (e8m0_exponent(amax) + 127).astype(np.uint8)


def e8m0_value(byte):
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


# --------------------------------------------------------------------------
# MXFP8 quantization ([TE-JAX] "What specialized optimizations...": a
# group-aware MXFP8 quantization; "Optimization 1": MXFP8 block scaling;
# [CH1] "低精度格式的缩放机制": per-block scaling, blocks of 32)
# --------------------------------------------------------------------------

def _quantize_blocks(blocks):
    """blocks [..., 32] exact fp64 -> (codes [..., 32] u8, scale byte [...] u8)."""
    amax = np.max(np.abs(blocks), axis=-1)
    e = e8m0_exponent(amax)
    scaled = blocks * np.ldexp(1.0, -e)[..., None]        # exact: power of two
    return e4m3_encode(scaled), (e + 127).astype(np.uint8)


def mxfp8_quantize_rows(x):
    """Rowwise MXFP8: blocks of 32 consecutive elements along each row
    (the contraction axis K of the next GEMM).  x [R, C], C % 32 == 0.
    Returns codes [R, C] u8 and scales [R, C/32] u8."""
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    assert C % MXFP8_BLOCK == 0
    codes, scales = _quantize_blocks(x.reshape(R, C // MXFP8_BLOCK, MXFP8_BLOCK))
    return codes.reshape(R, C), scales


def mxfp8_quantize_cols_grouped(x, offsets):
    """Group-aware columnwise MXFP8: blocks of 32 consecutive rows of ONE
    group, starting at the group's first row; a group's tail block is padded
    with zeros.  Group g occupies rows [offsets[g], offsets[g+1]).

    Reading: the padded layout puts group g at padded_offsets[g] =
    sum_{h<g} ceil32(m_h) so every block lies inside one group; an empty group
    occupies no rows.  The output is transposed (row c of the output is column
    c of x) because the block runs along x's rows.

    Returns codes [C, Rp] u8, scales [C, Rp/32] u8, padded_offsets [G+1].
    """
    x = np.asarray(x, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    C = x.shape[1]
    sizes = offsets[1:] - offsets[:-1]
    padded = np.concatenate([[0], np.cumsum((sizes + MXFP8_BLOCK - 1) // MXFP8_BLOCK * MXFP8_BLOCK)])
    Rp = int(padded[-1])
    xp = np.zeros((Rp, C), dtype=np.float64)
    for g in range(len(sizes)):
        xp[padded[g]:padded[g] + sizes[g]] = x[offsets[g]:offsets[g + 1]]
    blocks = xp.T.reshape(C, Rp // MXFP8_BLOCK, MXFP8_BLOCK)
    codes, scales = _quantize_blocks(blocks)
    return codes.reshape(C, Rp), scales, padded


def mxfp8_dequantize_rows(codes, scales):
    """Inverse of the rowwise layout: value = E4M3(code) * 2^(scale-127)."""
    codes = np.asarray(codes)
    R, C = codes.shape
    vals = E4M3_VALUES[codes.astype(np.int64)].reshape(R, C // MXFP8_BLOCK, MXFP8_BLOCK)
    return (vals * e8m0_value(scales)[..., None]).reshape(R, C)


def mxfp8_dequantize_cols(codes_t, scales_t):
    """Inverse of the columnwise layout: returns the [Rp, C] matrix."""
    return mxfp8_dequantize_rows(codes_t, scales_t).T


# --------------------------------------------------------------------------
# NVFP4 ([CH1] §1.1 precision table: FP4 is 4 bits, 1 sign + 2 exponent + 1
# mantissa; "低精度格式的缩放机制": NVFP4 scales in two levels, an E4M3 scale
# per small block for the relative sizes inside it and one FP32 scale for
# the whole tensor's range; [TE-JAX] "What is the training performance
# impact…": NVFP4 is planned next)
# --------------------------------------------------------------------------

NVFP4_BLOCK = 16    # Reading: the pages give no block size; 16 is the block the tensor cores' NVFP4 MMA scales
E2M1_MAX = 6.0


def e2m1_value(code: int) -> float:
    """Value of one FP4 E2M1 code: bit 3 sign, bits 2-1 exponent, bit 0
    mantissa ([CH1] §1.1: "FP4 4 (1+2+1)").  The exponent bias follows the
    rule of the pages' FP32 example, 2^(n-1) - 1 = 1.  Reading (the pages give
    only the split): as in E4M3, exponent field 0 holds the subnormals
    m/2 * 2^(1-1), and every code is finite (no inf/NaN), so the largest
    magnitude is 1.5 * 2^2 = 6."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = (m / 2.0) * 2.0 ** (1 - 1)
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


E2M1_VALUES = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E2M1_POS = E2M1_VALUES[:8]       # codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6


def e2m1_encode(v):
    """Encode exact fp64 values to E2M1 codes: nearest value, ties to the even
    code, magnitudes above 6 saturate to 6, the sign bit is kept (negatives
    that round to zero give 0x8).  Reading: the same round-to-nearest-even
    with saturation as the E4M3 cast."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    dlo = a - _E2M1_POS[lo]
    dhi = _E2M1_POS[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= E2M1_MAX, 7, code)
    sign = np.signbit(v).astype(np.int64)
    return (code.astype(np.int64) | (sign << 3)).astype(np.uint8)


def nvfp4_tensor_scale(amax):
    """Per-tensor FP32 scale s_t of a tensor whose largest magnitude is amax.
    Reading: the tensor-level scale maps the largest magnitude onto the top
    of the two-level range, 6 (E2M1) x 448 (E4M3), i.e. s_t = amax / 2688,
    computed in fp32 (it decides codes, so the oracle takes it in the
    kernel's precision).  amax == 0 gives s_t = 0."""
    return np.float32(np.float32(amax) / np.float32(E2M1_MAX * E4M3_MAX))


def nvfp4_quantize_rows(x):
    """Rowwise NVFP4 of x [R, C] (C % 16 == 0; exact bf16 values), blocks of
    16 consecutive elements along each row (the contraction axis).

    Steps, each rounded to fp32 where it decides a code (the kernel's
    precision; the order is a reading -- the pages give only the two levels):
      s_t = nvfp4_tensor_scale(max |x|)   (decode scale, fp32)
      enc = 2688 / max |x|                (encode factor, fp32)
      per block b: t_b = (amax_b / 6) * enc; scale byte = E4M3 of t_b
                   (nearest, ties to even, saturating at 448); its value s_b
                   r_b = enc / s_b
      per element: code = e2m1_encode(x * r_b)
    so that x ~ E2M1(code) * s_b * s_t.  A block whose scale byte is zero (its
    amax is negligible next to the tensor's) gets zero codes and dequantizes
    to zero; an all-zero tensor gives s_t = 0 and zero codes.

    Returns codes [R, C] u8 (one E2M1 code per element), scale bytes
    [R, C/16] u8 (E4M3) and s_t (np.float32)."""
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    assert C % NVFP4_BLOCK == 0
    f32 = np.float32
    amax_t = f32(np.max(np.abs(x)) if x.size else 0.0)
    st = nvfp4_tensor_scale(amax_t)
    blocks = x.reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    codes = np.zeros(blocks.shape, dtype=np.uint8)
    if st == 0:
        return codes.reshape(R, C), np.zeros((R, C // NVFP4_BLOCK), dtype=np.uint8), st
    enc = f32(f32(E2M1_MAX * E4M3_MAX) / amax_t)
    amax_b = np.max(np.abs(blocks), axis=-1).astype(f32)
    t_b = ((amax_b / f32(E2M1_MAX)).astype(f32) * enc).astype(f32)
    sbyte = e4m3_encode(t_b.astype(np.float64))
    live = sbyte != 0
    r_b = (enc / E4M3_VALUES[sbyte[live].astype(np.int64)].astype(f32)).astype(f32)
    y = (blocks[live].astype(f32) * r_b[:, None]).astype(f32)
    codes[live] = e2m1_encode(y.astype(np.float64))
    return codes.reshape(R, C), sbyte, st


def nvfp4_dequantize_rows(codes, scales, st):
    """value = E2M1(code) * E4M3(scale of its block) * s_t, in fp64."""
    codes = np.asarray(codes)
    R, C = codes.shape
    vals = E2M1_VALUES[codes.astype(np.int64)].reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    sb = E4M3_VALUES[np.asarray(scales).astype(np.int64)]
    return (vals * sb[..., None]).reshape(R, C) * float(st)


def nvfp4_quantize_cols_grouped(x, offsets):
    """Group-aware columnwise NVFP4 (the wgrad operands): blocks of 16
    consecutive rows of ONE group, starting at the group's first row, a
    group's tail block padded with zeros; one tensor scale for the whole
    matrix (the same s_t as the rowwise quantization of x).

    Reading: the group-aware layout of the MXFP8 columnwise quantization with
    the NVFP4 block of 16 (group g at padded_offsets[g] = sum_{h<g}
    ceil16(m_h)); every other step is nvfp4_quantize_rows applied to the
    transposed padded matrix, whose zero padding changes no block amax.

    Returns codes [C, Rp] u8 (one code per element, transposed), scales
    [C, Rp/16] u8, s_t and padded_offsets [G+1]."""
    x = np.asarray(x, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    C = x.shape[1]
    sizes = offsets[1:] - offsets[:-1]
    padded = np.concatenate([[0], np.cumsum((sizes + NVFP4_BLOCK - 1) // NVFP4_BLOCK * NVFP4_BLOCK)])
    Rp = int(padded[-1])
    xp = np.zeros((Rp, C), dtype=np.float64)
    for g in range(len(sizes)):
        xp[padded[g]:padded[g] + sizes[g]] = x[offsets[g]:offsets[g + 1]]
    codes, scales, st = nvfp4_quantize_rows(xp.T)
    return codes, scales, st, padded


def nvfp4_dequantize_cols(codes_t, scales_t, st):
    """Inverse of the columnwise layout: returns the [Rp, C] matrix."""
    return nvfp4_dequantize_rows(codes_t, scales_t, st).T


# --------------------------------------------------------------------------
# Routing ([TE-JAX] intro: a learned router picks the Top-K experts;
# "Optimization 2": the fused router kernels assign each token to its experts)
# --------------------------------------------------------------------------

def route_topk(logits, k, score="softmax", normalize=True):
    """Top-k expert selection and routing weights per token.

    logits [T, E] (fp32 values).  Selection is by logit, which equals
    selection by score since softmax and sigmoid are monotone.  Reading:
    ties go to the lower expert index, and the k choices are listed in
    descending score, then ascending index.

    Weights (fp64):
      softmax, normalize: softmax over all E, renormalised over the k chosen
      softmax, raw:       softmax probability of each chosen expert
      sigmoid, normalize: s = 1/(1+exp(-l)); w = s_chosen / sum(s_chosen)
      sigmoid, raw:       s_chosen
    Returns idx [T, k] int32 and w [T, k] fp64.
    """
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    assert 1 <= k <= E
    index = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((index, -l), axis=-1)      # primary: -logit; secondary: index
    idx = order[:, :k].astype(np.int32)
    chosen = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    if score == "softmax":
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)
        s = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    elif score == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-chosen))
    else:
        raise ValueError(score)
    w = s / s.sum(axis=1, keepdims=True) if normalize else s
    return idx, w


def group_counts(idx, E):
    """counts[e] = number of (token, choice) pairs routed to expert e.
    Dropless: every pair is kept, so sum(counts) == T*k ([TE-JAX] "How is
    dropless MoE different...")."""
    idx = np.asarray(idx)
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        counts[int(e)] += 1
    return counts


def group_offsets(counts):
    """offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]."""
    counts = np.asarray(counts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def aligned_group_offsets(counts, align):
    """Row layout of the permuted buffer: group e starts at
    gofs[e] = sum_{h<e} ceil_align(counts[h]).  With align == 1 this is the
    plain ragged layout.  Reading (a layout choice of the GPU path, stated in
    its header): align = 128, the GEMM tile height, so a tile never straddles
    two groups; rows [gofs[e] + counts[e], gofs[e+1]) are zero padding."""
    counts = np.asarray(counts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)]).astype(np.int64)


def permute_slots(idx, E, align=1):
    """Local half of dispatch ([TE-JAX] "Optimization 2": tokens are permuted
    into their experts' groups).  slot(t, j) = gofs[e] + #{t' < t : e in
    idx[t']} with e = idx[t, j].  Reading: the order inside a group is token
    order (stable), which makes the permutation unique.

    Returns slot_of [T, k] int64 and row_id [gofs[E]] int64 where
    row_id[slot(t, j)] = t*k + j and padding rows hold -1.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    counts = group_counts(idx, E)
    gofs = aligned_group_offsets(counts, align)
    fill = np.zeros(E, dtype=np.int64)
    slot_of = np.zeros((T, k), dtype=np.int64)
    row_id = np.full(int(gofs[-1]), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            s = gofs[e] + fill[e]
            fill[e] += 1
            slot_of[t, j] = s
            row_id[s] = t * k + j
    return slot_of, row_id


def permute(x, row_id, k):
    """x_perm[s] = x[row_id[s] // k]; padding rows (row_id == -1) are zero."""
    x = np.asarray(x, dtype=np.float64)
    row_id = np.asarray(row_id, dtype=np.int64)
    out = np.zeros((row_id.shape[0], x.shape[1]), dtype=np.float64)
    valid = row_id >= 0
    out[valid] = x[row_id[valid] // k]
    return out


def fp32_round(x):
    """Round fp64 values to the nearest fp32 value, ties to even (IEEE-754
    binary32: 24 significant bits); magnitudes beyond the fp32 range become
    inf, as the cast does."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def permute_scaled_bf16(src, row_id, k, w):
    """The permuted, router-weighted rows as stored in bf16:
    P[s] = bf16(fp32(w[t, j] * src[t])) with t*k + j = row_id[s], zero on
    padding rows.  This is the dy_perm of ``combine_bwd`` (src = dout) in
    the precision the step keeps it in.

    Reading: the pages fix neither the precision of dy_perm nor of the
    product; the activations of the step are bf16 and the routing weights
    fp32, so the product of an fp32 weight and a bf16 gradient is formed in
    fp32 (rounded once, ties to even) and stored as bf16 (rounded again).
    The second rounding decides MXFP8 codes, so it is part of the
    definition, not an error term."""
    src = np.asarray(src, dtype=np.float64)
    row_id = np.asarray(row_id, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64).reshape(-1)
    out = np.zeros((row_id.shape[0], src.shape[1]), dtype=np.float64)
    valid = row_id >= 0
    rid = row_id[valid]
    out[valid] = bf16_round(fp32_round(w[rid][:, None] * src[rid // k]))
    return out


# --------------------------------------------------------------------------
# Grouped GEMM ([TE-JAX] "Optimization 1: Grouped GEMM": all expert matmuls
# in one call, each with its actual token count, only valid-token regions)
# --------------------------------------------------------------------------

def grouped_gemm(A, B, offsets):
    """D[r, :] = A[r, :] @ B[g] for r in [offsets[g], offsets[g+1]).
    A [R, K], B [G, K, N].  Rows outside every group are left at zero.
    Serves fwd (B = W) and dgrad (B = W transposed per group)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    D = np.zeros((A.shape[0], B.shape[2]), dtype=np.float64)
    for g in range(B.shape[0]):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        if hi > lo:
            D[lo:hi] = A[lo:hi] @ B[g]
    return D


def grouped_gemm_wgrad(A, Gm, offsets):
    """dB[g] = A[rows of g].T @ Gm[rows of g]: the contraction runs over the
    group's rows (a ragged K).  Reading: an empty group's gradient is the
    empty sum, zero, and is written as such.  A [R, Ka], Gm [R, Nb] ->
    dB [G, Ka, Nb]."""
    A = np.asarray(A, dtype=np.float64)
    Gm = np.asarray(Gm, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    G = len(offsets) - 1
    dB = np.zeros((G, A.shape[1], Gm.shape[1]), dtype=np.float64)
    for g in range(G):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        if hi > lo:
            dB[g] = A[lo:hi].T @ Gm[lo:hi]
    return dB


# --------------------------------------------------------------------------
# SwiGLU expert activation.  Reading: the fused up/gate projection has the
# gate in columns [0, f) and the up projection in [f, 2f).
# --------------------------------------------------------------------------

def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def swiglu(a):
    a = np.asarray(a, dtype=np.float64)
    f = a.shape[1] // 2
    g, u = a[:, :f], a[:, f:]
    return g * _sigmoid(g) * u


def swiglu_bwd(a, dh):
    """Gradient of h = g*sigmoid(g)*u with respect to a = [g | u]."""
    a = np.asarray(a, dtype=np.float64)
    dh = np.asarray(dh, dtype=np.float64)
    f = a.shape[1] // 2
    g, u = a[:, :f], a[:, f:]
    sg = _sigmoid(g)
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    du = dh * g * sg
    return np.concatenate([dg, du], axis=1)


# --------------------------------------------------------------------------
# Combine ([TE-JAX] "Optimization 2": per-expert results are accumulated;
# [CH1] §2.3.2 dispatch/combine table and figure: a sum weighted by the
# routing weights, restoring the original token order)
# --------------------------------------------------------------------------

def combine(y_perm, slot_of, w=None):
    """out[t] = sum_{j=0}^{k-1} w[t, j] * y_perm[slot_of[t, j]], summed in
    j order; w = None means weights of one (the unpermute-sum of dgrad)."""
    y = np.asarray(y_perm, dtype=np.float64)
    slot_of = np.asarray(slot_of, dtype=np.int64)
    T, k = slot_of.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        wj = 1.0 if w is None else np.asarray(w, dtype=np.float64)[:, j:j + 1]
        out += wj * y[slot_of[:, j]]
    return out


def combine_bwd(dout, y_perm, slot_of, w, rows):
    """Adjoint of ``combine``: dy[slot(t,j)] = w[t,j] * dout[t] (other rows
    zero) and dw[t, j] = <dout[t], y_perm[slot(t,j)]>."""
    dout = np.asarray(dout, dtype=np.float64)
    y = np.asarray(y_perm, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    slot_of = np.asarray(slot_of, dtype=np.int64)
    T, k = slot_of.shape
    dy = np.zeros((rows, dout.shape[1]), dtype=np.float64)
    dw = np.zeros((T, k), dtype=np.float64)
    for j in range(k):
        dy[slot_of[:, j]] = w[:, j:j + 1] * dout
        dw[:, j] = np.sum(dout * y[slot_of[:, j]], axis=1)
    return dy, dw


def route_bwd(logits, idx, dw, score="softmax", normalize=True):
    """Gradient of the routing weights with respect to the logits (plain
    calculus on ``route_topk``'s weight formulas; the selection itself is
    piecewise constant).  Returns dlogits [T, E] fp64."""
    l = np.asarray(logits, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    dw = np.asarray(dw, dtype=np.float64)
    T, E = l.shape
    dl = np.zeros((T, E), dtype=np.float64)
    rows = np.arange(T)[:, None]
    if score == "softmax":
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)
        ps = np.take_along_axis(p, idx, axis=1)
        if normalize:
            w = ps / ps.sum(axis=1, keepdims=True)
            inner = np.sum(w * dw, axis=1, keepdims=True)
            dl[rows, idx] = w * (dw - inner)
        else:
            inner = np.sum(ps * dw, axis=1, keepdims=True)
            dl = -p * inner
            dl[rows, idx] += ps * dw
    elif score == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-np.take_along_axis(l, idx, axis=1)))
        if normalize:
            ssum = s.sum(axis=1, keepdims=True)
            w = s / ssum
            inner = np.sum(w * dw, axis=1, keepdims=True)
            dl[rows, idx] = s * (1.0 - s) / ssum * (dw - inner)
        else:
            dl[rows, idx] = s * (1.0 - s) * dw
    else:
        raise ValueError(score)
    return dl


# --------------------------------------------------------------------------
# Whole layer, unquantized fp64 (composition of the steps above; used to pin
# the backward formulas by finite differences)
# --------------------------------------------------------------------------

# --------------------------------------------------------------------------
# Router GEMM ([TE-JAX] "Optimization 2": the routing step is done by fused
# router kernels working from the router's scores.  Reading: the scores come
# from a learned linear router, logits = x W_r)
# --------------------------------------------------------------------------

def router_logits(x, Wr):
    """logits [T, E] = x [T, d] @ W_r [d, E].  Reading: the pages give no
    router arithmetic; the operands are the step's bf16 activations and bf16
    router weights, the product is exact in fp64 (the GPU accumulates in
    fp32 and stores fp32 logits)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(Wr, dtype=np.float64)


def router_backward(x, Wr, dlogits):
    """Gradients of ``router_logits``: dx_r = bf16(dlogits) @ W_r^T [T, d]
    and dW_r = x^T @ bf16(dlogits) [d, E].  Reading: the backward GEMMs take
    bf16 operands like the forward, so dlogits (fp32) is rounded to bf16
    (nearest even) once; the products are exact in fp64."""
    g = bf16_round(np.asarray(dlogits, dtype=np.float64))
    x = np.asarray(x, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    return g @ Wr.T, x.T @ g


def append_shared(idx, w, E, n_shared):
    """Shared experts (every token uses them with weight 1; DeepSeek-V3's
    shared expert, [CH1] §2.3.2) as extra choices: [idx | E .. E+S-1] and
    [w | 1 .. 1] per token.  Reading: a shared expert is an FFN of the same
    shape as a routed one whose output is added to the routed combine."""
    idx = np.asarray(idx, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64)
    T = idx.shape[0]
    sh = np.broadcast_to(E + np.arange(n_shared), (T, n_shared))
    return np.concatenate([idx, sh], axis=1), np.concatenate([w, np.ones((T, n_shared))], axis=1)


def layer_forward(x, logits, W1, W2, k, score="softmax", normalize=True, align=1, n_shared=0):
    """Dropless MoE layer, [TE-JAX] Figure 3: route, permute, grouped GEMM
    (up/gate), SwiGLU, grouped GEMM (down), combine.  W1 [E, d, 2f],
    W2 [E, f, d] (the last n_shared experts are shared experts, see
    ``append_shared``; logits cover the routed ones).  Returns out [T, d]
    and the saved activations."""
    E = W1.shape[0]
    idx, w = route_topk(logits, k, score, normalize)
    idx_all, w_all = append_shared(idx, w, E - n_shared, n_shared) if n_shared else (idx, w)
    k_all = k + n_shared
    slot_of, row_id = permute_slots(idx_all, E, align)
    gofs = aligned_group_offsets(group_counts(idx_all, E), align)
    xp = permute(x, row_id, k_all)
    a = grouped_gemm(xp, W1, gofs)
    h = swiglu(a)
    y = grouped_gemm(h, W2, gofs)
    out = combine(y, slot_of, w_all)
    saved = dict(idx=idx, w=w_all, slot_of=slot_of, row_id=row_id, gofs=gofs, xp=xp, a=a, h=h, y=y)
    return out, saved


def layer_backward(dout, logits, W1, W2, k, saved, score="softmax", normalize=True):
    """Backward of ``layer_forward`` (plain autograd, step by step)."""
    T = dout.shape[0]
    rows = saved["xp"].shape[0]
    dy, dw_all = combine_bwd(dout, saved["y"], saved["slot_of"], saved["w"], rows)
    dw = dw_all[:, :k]           # the shared choices' weights are constants
    dh = grouped_gemm(dy, np.transpose(W2, (0, 2, 1)), saved["gofs"])
    dW2 = grouped_gemm_wgrad(saved["h"], dy, saved["gofs"])
    da = swiglu_bwd(saved["a"], dh)
    dxp = grouped_gemm(da, np.transpose(W1, (0, 2, 1)), saved["gofs"])
    dW1 = grouped_gemm_wgrad(saved["xp"], da, saved["gofs"])
    dx = combine(dxp, saved["slot_of"], None)
    dlogits = route_bwd(logits, saved["idx"], dw, score, normalize)
    assert dx.shape[0] == T
    return dict(dx=dx, dlogits=dlogits, dW1=dW1, dW2=dW2, dy=dy, dw=dw, dh=dh, da=da, dxp=dxp)
