"""ctypes binding of libmoe.so: the same entry points as include/moe.h.

Argument marshalling only -- every step runs in the library's CUDA kernels.
Torch is used for device memory and the current stream.  If the shared
library is missing the import of this module fails loudly; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

# status codes (include/moe.h)
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_ALIGNMENT = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_CUDA = 5
MOE_ERR_NOT_INITIALIZED = 6
MOE_ERR_BAD_EXPERT = 16
MOE_ERR_BAD_OFFSETS = 17
MOE_ERR_DEVICE_TIMEOUT = 18
MOE_ERR_CAPACITY = 19

MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_QUANT_ROWWISE, MOE_QUANT_COLWISE_GROUPED, MOE_QUANT_COLWISE_GLU = 0, 1, 2
MOE_QUANT_COLWISE_BATCHED, MOE_QUANT_COLWISE_BATCHED_GLU = 3, 4
MOE_GEMM_FWD, MOE_GEMM_DGRAD, MOE_GEMM_WGRAD = 0, 1, 2
MOE_EPI_NONE, MOE_EPI_SWIGLU, MOE_EPI_SWIGLU_BWD, MOE_EPI_NONE_F32 = 0, 1, 2, 3
MOE_B_GNK, MOE_B_NGK, MOE_B_SF_TILE224 = 0, 1, 2
MOE_SF_ATOMS, MOE_SF_TILE224, MOE_SF_CANONICAL, MOE_SF_TILE224_AND_ATOMS = 0, 1, 2, 3
MOE_GEMM_KERNEL_AUTO, MOE_GEMM_KERNEL_1SM, MOE_GEMM_KERNEL_1SM_N128 = 0, 1, 2
MOE_GEMM_KERNEL_PAIR, MOE_GEMM_KERNEL_PAIR_N128 = 3, 4
(MOE_OP_ROUTE_TOPK, MOE_OP_PERMUTE, MOE_OP_GROUP_QUANTIZE, MOE_OP_GATHER_QUANTIZE, MOE_OP_GROUPED_GEMM,
 MOE_OP_UNPERMUTE_COMBINE, MOE_OP_COMBINE_BWD, MOE_OP_ROUTE_BWD) = range(8)

EXPORTS = [
    "moe_abi_version", "moe_status_string", "moe_init", "moe_row_capacity",
    "moe_route_workspace_size", "moe_permute_workspace_size", "moe_route_topk",
    "moe_permute", "mxfp8_group_quantize", "grouped_gemm_mxfp8",
    "moe_unpermute_combine", "moe_combine_bwd", "moe_route_bwd", "moe_route_topk_noalloc",
    "mxfp8_gather_quantize", "grouped_gemm_mxfp8_swiglu_quant", "mxfp8_swiglu_bwd_quantize",
    "gemm_bf16_nt", "moe_transpose_bf16", "moe_unpermute_combine_add", "moe_route_append_shared",
    "moe_route_drop_shared", "nvfp4_sf_bytes", "nvfp4_quantize", "grouped_gemm_nvfp4", "nvfp4_quantize_cols",
    "moe_selftest_bounded_wait", "moe_workspace_size", "mxfp8_scale_layout", "grouped_gemm_mxfp8_ex",
    "grouped_gemm_mxfp8_swiglu_quant_ex", "grouped_gemm_nvfp4_ex", "moe_hbm_fill", "mxfp8_gather_quantize_ex",
    "mxfp8_swiglu_bwd_quantize_ex", "mxfp8_group_quantize_ex",
]

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t


class GemmOpts(ctypes.Structure):
    """moe_gemm_opts_t (include/moe.h): per-call grouped-GEMM kernel choice."""
    _fields_ = [("kernel", ctypes.c_int), ("band", ctypes.c_int), ("register_stores", ctypes.c_int),
                ("wgrad_rows_lo", ctypes.c_int), ("wgrad_rows_hi", ctypes.c_int)]


_GEMM_KERNELS = {"auto": MOE_GEMM_KERNEL_AUTO, "1sm": MOE_GEMM_KERNEL_1SM, "1sm_n128": MOE_GEMM_KERNEL_1SM_N128,
                 "pair": MOE_GEMM_KERNEL_PAIR, "pair_n128": MOE_GEMM_KERNEL_PAIR_N128}


def gemm_opts(kernel="auto", band=0, register_stores=False, wgrad_rows=(0, 0)):
    """A GemmOpts for the opts= argument of the grouped-GEMM wrappers;
    kernel is one of "auto", "1sm", "1sm_n128", "pair", "pair_n128" (or the
    MOE_GEMM_KERNEL_* value); wgrad_rows = (lo, hi): WGRAD computes only the
    groups with lo <= rows and (hi == 0 or rows < hi)."""
    k = _GEMM_KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    lo, hi = wgrad_rows
    return GemmOpts(k, int(band), int(bool(register_stores)), int(lo), int(hi))


_SIGS = {
    "moe_abi_version": (_i32, []),
    "moe_status_string": (ctypes.c_char_p, [_i32]),
    "moe_init": (_i32, [_i32]),
    "moe_row_capacity": (_i64, [_i32, _i32, _i32]),
    "moe_route_workspace_size": (_sz, [_i32, _i32]),
    "moe_permute_workspace_size": (_sz, [_i32, _i32]),
    "moe_route_topk": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_permute": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "mxfp8_group_quantize": (_i32, [_vp, _i64, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp]),
    "mxfp8_group_quantize_ex": (_i32, [_vp, _i64, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp]),
    "mxfp8_gather_quantize": (_i32, [_vp, _i64, _i32, _i32, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp,
                                     _vp]),
    "gemm_bf16_nt": (_i32, [_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp]),
    "moe_route_append_shared": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_route_drop_shared": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp]),
    "moe_transpose_bf16": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
    "moe_unpermute_combine_add": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "mxfp8_swiglu_bwd_quantize": (_i32, [_vp, _vp, _i32, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "grouped_gemm_mxfp8_swiglu_quant": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i64, _vp, _vp, _vp,
                                               _vp, _vp, _vp, _vp, _vp]),
    "grouped_gemm_mxfp8": (_i32, [_i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i64, _i32, _vp, _vp,
                                  _vp, _vp, _vp]),
    "moe_unpermute_combine": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_combine_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _vp, _vp, _vp, _vp]),
    "moe_route_bwd": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_route_topk_noalloc": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_sf_bytes": (_i64, [_i64, _i32]),
    "moe_selftest_bounded_wait": (_i32, [ctypes.c_uint64, _vp, _vp, _vp]),
    "nvfp4_quantize": (_i32, [_vp, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_quantize_cols": (_i32, [_vp, _i64, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "grouped_gemm_nvfp4": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i64, _i32, _vp, _vp,
                                  _vp]),
    "moe_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "mxfp8_scale_layout": (_i32, [_vp, _i64, _i32, _i32, _vp, _vp]),
    "grouped_gemm_mxfp8_ex": (_i32, [_i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i64, _i32, _vp, _vp,
                                     _vp, _vp, _vp, _vp]),
    "grouped_gemm_mxfp8_swiglu_quant_ex": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i64, _vp, _vp,
                                                  _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "grouped_gemm_nvfp4_ex": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i64, _i32, _vp,
                                     _vp, _vp, _vp]),
    "moe_hbm_fill": (_i32, [_vp, _sz, ctypes.c_uint32, _i32, _vp]),
    "mxfp8_gather_quantize_ex": (_i32, [_vp, _i64, _i32, _i32, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _i32,
                                        _vp, _vp]),
    "mxfp8_swiglu_bwd_quantize_ex": (_i32, [_vp, _vp, _i32, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                            _vp]),
}


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so not found at {LIB_PATH}; build it with grouped_gemm_top_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def _check(fn, status):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _p(t):
    """Device pointer of a tensor (or None for NULL)."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------ entry points --

def moe_abi_version() -> int:
    return lib.moe_abi_version()


def moe_init(device: int = 0) -> None:
    _check("moe_init", lib.moe_init(int(device)))


def moe_row_capacity(T: int, E: int, k: int) -> int:
    return int(lib.moe_row_capacity(T, E, k))


def moe_route_workspace_size(T: int, E: int) -> int:
    return int(lib.moe_route_workspace_size(T, E))


def moe_permute_workspace_size(T: int, E: int) -> int:
    return int(lib.moe_permute_workspace_size(T, E))


def moe_workspace_size(op: int, T: int, d: int, E: int, k: int, f: int) -> int:
    """Workspace bytes of call `op` (MOE_OP_*); -1 for an unknown op or bad sizes."""
    v = int(lib.moe_workspace_size(int(op), int(T), int(d), int(E), int(k), int(f)))
    return -1 if v == ctypes.c_size_t(-1).value else v


def mxfp8_scale_layout(src, rows, cols, to_canonical=True, dst=None, stream=None):
    """Scales of a [rows, cols] matrix quantized along cols: atom layout ->
    canonical [rows, cols/32] (to_canonical) or back.  See include/moe.h."""
    dst = dst if dst is not None else _empty((rows * (cols // 32),), torch.uint8, src)
    _check("mxfp8_scale_layout", lib.mxfp8_scale_layout(_p(src), int(rows), int(cols), int(bool(to_canonical)),
                                                        _p(dst), _stream(stream)))
    return dst


def moe_hbm_fill(dst, value=0, method=0, stream=None):
    """Write the 32-bit value over all of dst's bytes (write-only stream)."""
    nbytes = dst.numel() * dst.element_size()
    _check("moe_hbm_fill", lib.moe_hbm_fill(_p(dst), nbytes, ctypes.c_uint32(int(value) & 0xFFFFFFFF).value,
                                            int(method), _stream(stream)))


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def moe_route_topk(logits, k, score=MOE_SCORE_SOFTMAX, normalize=True, topk_idx=None, topk_w=None,
                   counts=None, offsets=None, ws=None, err=None, stream=None):
    T, E = logits.shape
    topk_idx = topk_idx if topk_idx is not None else _empty((T, k), torch.int32, logits)
    topk_w = topk_w if topk_w is not None else _empty((T, k), torch.float32, logits)
    counts = counts if counts is not None else _empty((E,), torch.int32, logits)
    offsets = offsets if offsets is not None else _empty((E + 1,), torch.int32, logits)
    ws = ws if ws is not None else _empty((moe_route_workspace_size(T, E),), torch.uint8, logits)
    _check("moe_route_topk", lib.moe_route_topk(_p(logits), T, E, k, int(score), int(bool(normalize)),
                                                _p(topk_idx), _p(topk_w), _p(counts), _p(offsets), _p(ws),
                                                ws.numel(), _p(err), _stream(stream)))
    return topk_idx, topk_w, counts, offsets


def moe_permute(x, topk_idx, E, row_cap=None, gofs=None, slot_of=None, row_id=None, x_perm=None,
                want_x_perm=True, ws=None, err=None, stream=None):
    T, k = topk_idx.shape
    d = x.shape[1] if x is not None else 0
    row_cap = row_cap if row_cap is not None else moe_row_capacity(T, E, k)
    like = topk_idx
    gofs = gofs if gofs is not None else _empty((E + 1,), torch.int32, like)
    slot_of = slot_of if slot_of is not None else _empty((T, k), torch.int32, like)
    row_id = row_id if row_id is not None else _empty((row_cap,), torch.int32, like)
    if want_x_perm and x_perm is None:
        x_perm = _empty((row_cap, d), torch.bfloat16, like)
    ws = ws if ws is not None else _empty((moe_permute_workspace_size(T, E),), torch.uint8, like)
    _check("moe_permute", lib.moe_permute(_p(x), T, d, E, k, _p(topk_idx), row_cap, _p(gofs), _p(slot_of),
                                          _p(row_id), _p(x_perm) if want_x_perm else None, _p(ws), ws.numel(),
                                          _p(err), _stream(stream)))
    return gofs, slot_of, row_id, x_perm


def sf_bytes(rows: int, cols: int) -> int:
    """Bytes of the scale array of a [rows, cols] matrix quantized along cols."""
    return rows * (cols // 32)


def sf_bytes_tile224(rows: int, cols: int) -> int:
    """Bytes of the tile-224 scale layout of a [rows, cols] matrix quantized
    along cols (include/moe.h): (cols / 128) k-blocks of ceil(rows / 224)
    tiles of 1024 bytes."""
    return (cols // 128) * ((rows + 223) // 224) * 1024


def col_sf_bytes(layout: int, rows: int, cols: int) -> int:
    """Bytes of the columnwise scales of a [rows, cols] quantization (the
    transposed [cols, rows] matrix) in moe_sf_layout_t `layout`; for
    MOE_SF_TILE224_AND_ATOMS the atom layout starts at
    sf_bytes_tile224(cols, rows)."""
    if layout == MOE_SF_TILE224:
        return sf_bytes_tile224(cols, rows)
    if layout == MOE_SF_TILE224_AND_ATOMS:
        return sf_bytes_tile224(cols, rows) + sf_bytes(rows, cols)
    return sf_bytes(rows, cols)


def mxfp8_group_quantize(x, axis=MOE_QUANT_ROWWISE, gofs=None, G=0, codes=None, scales=None, err=None,
                         stream=None):
    """See include/moe.h.  Returns (codes, scales) with the scales in the
    atom layout."""
    rows, cols = x.shape
    if axis == MOE_QUANT_ROWWISE:
        codes = codes if codes is not None else _empty((rows, cols), torch.uint8, x)
    elif axis in (MOE_QUANT_COLWISE_BATCHED, MOE_QUANT_COLWISE_BATCHED_GLU):
        codes = codes if codes is not None else _empty((G, cols, rows // G), torch.uint8, x)
    else:
        codes = codes if codes is not None else _empty((cols, rows), torch.uint8, x)
    scales = scales if scales is not None else _empty((sf_bytes(rows, cols),), torch.uint8, x)
    _check("mxfp8_group_quantize", lib.mxfp8_group_quantize(_p(x), rows, cols, int(axis), _p(gofs), int(G),
                                                            _p(codes), _p(scales), _p(err), _stream(stream)))
    return codes, scales


def mxfp8_group_quantize_ex(x, axis=MOE_QUANT_ROWWISE, gofs=None, G=0, scale_layout=MOE_SF_CANONICAL,
                            want_padded_offsets=True, codes=None, scales=None, padded_offsets=None, err=None,
                            stream=None):
    """mxfp8_group_quantize with the scale layout chosen (MOE_SF_ATOMS or
    MOE_SF_CANONICAL, row-major [R, C / 32] of the output matrix) and the
    padded group offsets written out.  Returns (codes, scales,
    padded_offsets or None)."""
    rows, cols = x.shape
    if axis == MOE_QUANT_ROWWISE:
        codes = codes if codes is not None else _empty((rows, cols), torch.uint8, x)
    elif axis in (MOE_QUANT_COLWISE_BATCHED, MOE_QUANT_COLWISE_BATCHED_GLU):
        codes = codes if codes is not None else _empty((G, cols, rows // G), torch.uint8, x)
    else:
        codes = codes if codes is not None else _empty((cols, rows), torch.uint8, x)
    scales = scales if scales is not None else _empty((sf_bytes(rows, cols),), torch.uint8, x)
    if padded_offsets is None and want_padded_offsets:
        padded_offsets = _empty((int(G) + 1,), torch.int32, x)
    _check("mxfp8_group_quantize_ex",
           lib.mxfp8_group_quantize_ex(_p(x), rows, cols, int(axis), _p(gofs), int(G), _p(codes), _p(scales),
                                       _p(padded_offsets), int(scale_layout), _p(err), _stream(stream)))
    return codes, scales, padded_offsets


def mxfp8_gather_quantize(src, gofs, G, rows, row_id=None, k=1, row_w=None, rowwise=True, colwise=True,
                          codes_row=None, scales_row=None, codes_col=None, scales_col=None, err=None, stream=None,
                          col_sf_layout=MOE_SF_ATOMS):
    """Rowwise and/or group-aware columnwise MXFP8 codes of the permuted
    matrix whose row s is src[row_id[s] // k] (times row_w[row_id[s]]), or
    src[s] without row_id.  See include/moe.h (a given codes_row must be
    32-byte aligned, as fresh torch allocations are).  col_sf_layout
    MOE_SF_TILE224 writes the columnwise scales in the tile-224 layout,
    MOE_SF_TILE224_AND_ATOMS that and the atom layout after it
    (mxfp8_gather_quantize_ex).  Returns (codes_row, scales_row, codes_col,
    scales_col), None for an axis not asked for."""
    cols = src.shape[1]
    if rowwise:
        codes_row = codes_row if codes_row is not None else _empty((rows, cols), torch.uint8, src)
        scales_row = scales_row if scales_row is not None else _empty((sf_bytes(rows, cols),), torch.uint8, src)
    else:
        codes_row = scales_row = None
    if colwise:
        codes_col = codes_col if codes_col is not None else _empty((cols, rows), torch.uint8, src)
        nsc = col_sf_bytes(col_sf_layout, rows, cols)
        scales_col = scales_col if scales_col is not None else torch.zeros((nsc,), dtype=torch.uint8,
                                                                           device=src.device)
    else:
        codes_col = scales_col = None
    args = (_p(src), src.shape[0], cols, int(k), _p(row_id), _p(row_w), _p(gofs), int(G), int(rows), _p(codes_row),
            _p(scales_row), _p(codes_col), _p(scales_col))
    if col_sf_layout == MOE_SF_ATOMS:
        _check("mxfp8_gather_quantize", lib.mxfp8_gather_quantize(*args, _p(err), _stream(stream)))
    else:
        _check("mxfp8_gather_quantize_ex", lib.mxfp8_gather_quantize_ex(*args, int(col_sf_layout), _p(err),
                                                                        _stream(stream)))
    return codes_row, scales_row, codes_col, scales_col


def grouped_gemm_mxfp8(mode, a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, epilogue=MOE_EPI_NONE,
                       epi_aux=None, d=None, d2=None, err=None, stream=None, opts=None):
    """See include/moe.h.  Allocates d (and d2 for SwiGLU) when not given.
    opts: a GemmOpts (gemm_opts()) selects grouped_gemm_mxfp8_ex."""
    if d is None:
        if mode == MOE_GEMM_WGRAD:
            d = _empty((G, M, N), torch.bfloat16, a)
        elif epilogue == MOE_EPI_SWIGLU_BWD:
            d = _empty((M, 2 * N), torch.bfloat16, a)
        elif epilogue == MOE_EPI_NONE_F32:
            d = _empty((M, N), torch.float32, a)
        else:
            d = _empty((M, N), torch.bfloat16, a)
    if epilogue == MOE_EPI_SWIGLU and d2 is None:
        d2 = _empty((M, N // 2), torch.bfloat16, a)
    args = (int(mode), _p(a), _p(a_sf), _p(b), _p(b_sf), int(b_layout), _p(gofs), int(G), int(M), int(N), int(K),
            int(epilogue), _p(epi_aux), _p(d), _p(d2))
    if opts is None:
        _check("grouped_gemm_mxfp8", lib.grouped_gemm_mxfp8(*args, _p(err), _stream(stream)))
    else:
        _check("grouped_gemm_mxfp8_ex", lib.grouped_gemm_mxfp8_ex(*args, ctypes.byref(opts), _p(err),
                                                                  _stream(stream)))
    return (d, d2) if epilogue == MOE_EPI_SWIGLU else d


def mxfp8_swiglu_bwd_quantize(dH, a_pre, gofs, G, dA=None, want_dA=False, codes_row=None, scales_row=None,
                              codes_col=None, scales_col=None, err=None, stream=None, col_sf_layout=MOE_SF_ATOMS):
    """MXFP8 (both axes) of dA = SwiGLU-backward(a_pre, dH); dA itself in bf16
    only if want_dA or dA is given.  See include/moe.h.  Returns (dA or None,
    codes_row, scales_row, codes_col, scales_col)."""
    rows, f = dH.shape
    if dA is None and want_dA:
        dA = _empty((rows, 2 * f), torch.bfloat16, dH)
    codes_row = codes_row if codes_row is not None else _empty((rows, 2 * f), torch.uint8, dH)
    scales_row = scales_row if scales_row is not None else _empty((sf_bytes(rows, 2 * f),), torch.uint8, dH)
    codes_col = codes_col if codes_col is not None else _empty((2 * f, rows), torch.uint8, dH)
    nsc = col_sf_bytes(col_sf_layout, rows, 2 * f)
    scales_col = scales_col if scales_col is not None else torch.zeros((nsc,), dtype=torch.uint8, device=dH.device)
    args = (_p(dH), _p(a_pre), int(f), _p(gofs), int(G), int(rows), _p(dA), _p(codes_row), _p(scales_row),
            _p(codes_col), _p(scales_col))
    if col_sf_layout == MOE_SF_ATOMS:
        _check("mxfp8_swiglu_bwd_quantize", lib.mxfp8_swiglu_bwd_quantize(*args, _p(err), _stream(stream)))
    else:
        _check("mxfp8_swiglu_bwd_quantize_ex",
               lib.mxfp8_swiglu_bwd_quantize_ex(*args, int(col_sf_layout), _p(err), _stream(stream)))
    return dA, codes_row, scales_row, codes_col, scales_col


def grouped_gemm_mxfp8_swiglu_quant(a, a_sf, b, b_sf, b_layout, gofs, G, M, N, K, a_pre=None, h=None, want_h=False,
                                    h_codes_row=None, h_scales_row=None, h_codes_col=None, h_scales_col=None,
                                    err=None, stream=None, opts=None):
    """Up/gate GEMM with the SwiGLU epilogue writing a_pre [M, N] and the
    MXFP8 codes of h on both axes (h bf16 [M, N/2] only if want_h or h is
    given).  See include/moe.h.  Returns (a_pre, h or None, codes_row,
    scales_row, codes_col, scales_col)."""
    f = N // 2
    a_pre = a_pre if a_pre is not None else _empty((M, N), torch.bfloat16, a)
    if h is None and want_h:
        h = _empty((M, f), torch.bfloat16, a)
    h_codes_row = h_codes_row if h_codes_row is not None else _empty((M, f), torch.uint8, a)
    h_scales_row = h_scales_row if h_scales_row is not None else _empty((sf_bytes(M, f),), torch.uint8, a)
    h_codes_col = h_codes_col if h_codes_col is not None else _empty((f, M), torch.uint8, a)
    h_scales_col = h_scales_col if h_scales_col is not None else _empty((sf_bytes(M, f),), torch.uint8, a)
    args = (_p(a), _p(a_sf), _p(b), _p(b_sf), int(b_layout), _p(gofs), int(G), int(M), int(N), int(K), _p(a_pre),
            _p(h), _p(h_codes_row), _p(h_scales_row), _p(h_codes_col), _p(h_scales_col))
    if opts is None:
        _check("grouped_gemm_mxfp8_swiglu_quant",
               lib.grouped_gemm_mxfp8_swiglu_quant(*args, _p(err), _stream(stream)))
    else:
        _check("grouped_gemm_mxfp8_swiglu_quant_ex",
               lib.grouped_gemm_mxfp8_swiglu_quant_ex(*args, ctypes.byref(opts), _p(err), _stream(stream)))
    return a_pre, h, h_codes_row, h_scales_row, h_codes_col, h_scales_col


def moe_route_append_shared(topk_idx, topk_w, E, n_shared, idx_out=None, w_out=None, stream=None):
    """[T, k+S] choices: the routed ones, then the S shared experts E.. with weight 1."""
    T, k = topk_idx.shape
    idx_out = idx_out if idx_out is not None else _empty((T, k + n_shared), torch.int32, topk_idx)
    w_out = w_out if w_out is not None else _empty((T, k + n_shared), torch.float32, topk_idx)
    _check("moe_route_append_shared", lib.moe_route_append_shared(_p(topk_idx), _p(topk_w), T, k, int(E),
                                                                  int(n_shared), _p(idx_out), _p(w_out),
                                                                  _stream(stream)))
    return idx_out, w_out


def moe_route_drop_shared(dw_all, k, dw=None, stream=None):
    T, k2 = dw_all.shape
    dw = dw if dw is not None else _empty((T, k), torch.float32, dw_all)
    _check("moe_route_drop_shared", lib.moe_route_drop_shared(_p(dw_all), T, int(k), int(k2 - k), _p(dw),
                                                              _stream(stream)))
    return dw


def gemm_bf16_nt(a, b, d=None, err=None, stream=None):
    """d [M, N] fp32 = a [M, K] @ b [N, K]^T (bf16 operands).  See include/moe.h."""
    M, K = a.shape
    N = b.shape[0]
    d = d if d is not None else _empty((M, N), torch.float32, a)
    _check("gemm_bf16_nt", lib.gemm_bf16_nt(_p(a), _p(b), int(M), int(N), int(K), _p(d), _p(err), _stream(stream)))
    return d


def moe_transpose_bf16(src, dst=None, stream=None):
    """dst [cols, rows] bf16 = src [rows, cols]^T (src bf16 or fp32)."""
    rows, cols = src.shape
    dst = dst if dst is not None else _empty((cols, rows), torch.bfloat16, src)
    _check("moe_transpose_bf16", lib.moe_transpose_bf16(_p(src), int(src.dtype == torch.float32), int(rows),
                                                        int(cols), _p(dst), _stream(stream)))
    return dst


def moe_unpermute_combine_add(y_perm, slot_of, topk_w, addend, out=None, err=None, stream=None):
    T, k = slot_of.shape
    d = y_perm.shape[1]
    out = out if out is not None else _empty((T, d), torch.bfloat16, y_perm)
    _check("moe_unpermute_combine_add", lib.moe_unpermute_combine_add(_p(y_perm), _p(slot_of), _p(topk_w),
                                                                      _p(addend), T, d, k, _p(out), _p(err),
                                                                      _stream(stream)))
    return out


def moe_unpermute_combine(y_perm, slot_of, topk_w, out=None, err=None, stream=None):
    T, k = slot_of.shape
    d = y_perm.shape[1]
    out = out if out is not None else _empty((T, d), torch.bfloat16, y_perm)
    _check("moe_unpermute_combine", lib.moe_unpermute_combine(_p(y_perm), _p(slot_of), _p(topk_w), T, d, k,
                                                              _p(out), _p(err), _stream(stream)))
    return out


def moe_combine_bwd(dout, y_perm, slot_of, topk_w, row_id, gofs, E, dy_perm=None, dw=None, err=None, stream=None,
                    want_dy=True):
    """dy_perm (unless want_dy is False: then dw only, dy_perm is None) and dw."""
    T, k = slot_of.shape
    d = dout.shape[1]
    row_cap = row_id.shape[0] if row_id is not None else 0
    if want_dy:
        dy_perm = dy_perm if dy_perm is not None else _empty((row_cap, d), torch.bfloat16, dout)
    else:
        dy_perm = None
        row_cap = max(row_cap, 1)
    dw = dw if dw is not None else _empty((T, k), torch.float32, dout)
    _check("moe_combine_bwd", lib.moe_combine_bwd(_p(dout), _p(y_perm), _p(slot_of), _p(topk_w), _p(row_id),
                                                  _p(gofs), T, d, k, E, row_cap, _p(dy_perm), _p(dw), _p(err),
                                                  _stream(stream)))
    return dy_perm, dw


def moe_route_bwd(logits, topk_idx, dw, score=MOE_SCORE_SOFTMAX, normalize=True, dlogits=None, err=None,
                  stream=None):
    T, E = logits.shape
    k = topk_idx.shape[1]
    dlogits = dlogits if dlogits is not None else _empty((T, E), torch.float32, logits)
    _check("moe_route_bwd", lib.moe_route_bwd(_p(logits), _p(topk_idx), _p(dw), T, E, k, int(score),
                                              int(bool(normalize)), _p(dlogits), _p(err), _stream(stream)))
    return dlogits


def moe_route_topk_noalloc(logits, k, score=MOE_SCORE_SOFTMAX, normalize=True, topk_idx=None, topk_w=None,
                           counts=None, offsets=None, err=None, stream=None):
    """moe_route_topk for callers that cannot allocate device scratch: the
    library uses a fixed internal array instead of a workspace (limit
    ceil(T/128) * E <= 262144; calls must not overlap on the GPU).  The
    output tensors are allocated here only when not passed in."""
    T, E = logits.shape
    topk_idx = topk_idx if topk_idx is not None else _empty((T, k), torch.int32, logits)
    topk_w = topk_w if topk_w is not None else _empty((T, k), torch.float32, logits)
    counts = counts if counts is not None else _empty((E,), torch.int32, logits)
    offsets = offsets if offsets is not None else _empty((E + 1,), torch.int32, logits)
    _check("moe_route_topk_noalloc", lib.moe_route_topk_noalloc(_p(logits), T, E, k, int(score),
                                                                int(bool(normalize)), _p(topk_idx), _p(topk_w),
                                                                _p(counts), _p(offsets), _p(err), _stream(stream)))
    return topk_idx, topk_w, counts, offsets


def nvfp4_sf_bytes(rows: int, cols: int) -> int:
    return int(lib.nvfp4_sf_bytes(int(rows), int(cols)))


def nvfp4_quantize(x, codes=None, scales=None, tensor_scale=None, amax_ws=None, err=None, stream=None):
    """Two-level NVFP4 of bf16 x [rows, cols] (rows % 128, cols % 256).  See
    include/moe.h.  Returns (codes [rows, cols/2] u8, scales u8, tensor_scale
    float32 [1])."""
    rows, cols = x.shape
    codes = codes if codes is not None else _empty((rows, cols // 2), torch.uint8, x)
    scales = scales if scales is not None else _empty((max(nvfp4_sf_bytes(rows, cols), 0),), torch.uint8, x)
    tensor_scale = tensor_scale if tensor_scale is not None else _empty((1,), torch.float32, x)
    amax_ws = amax_ws if amax_ws is not None else _empty((1,), torch.int32, x)
    _check("nvfp4_quantize", lib.nvfp4_quantize(_p(x), int(rows), int(cols), _p(codes), _p(scales),
                                                _p(tensor_scale), _p(amax_ws), _p(err), _stream(stream)))
    return codes, scales, tensor_scale


def nvfp4_quantize_cols(x, gofs, G, codes_t=None, scales_t=None, tensor_scale=None, amax_ws=None, err=None,
                        stream=None):
    """Group-aware columnwise NVFP4 of bf16 x [rows, cols] (rows % 256, cols %
    128; groups at multiples of 128 rows).  See include/moe.h.  Returns
    (codes_t [cols, rows/2] u8, scales_t u8, tensor_scale float32 [1])."""
    rows, cols = x.shape
    codes_t = codes_t if codes_t is not None else _empty((cols, rows // 2), torch.uint8, x)
    scales_t = scales_t if scales_t is not None else _empty((max(nvfp4_sf_bytes(cols, rows), 0),), torch.uint8, x)
    tensor_scale = tensor_scale if tensor_scale is not None else _empty((1,), torch.float32, x)
    amax_ws = amax_ws if amax_ws is not None else _empty((1,), torch.int32, x)
    _check("nvfp4_quantize_cols", lib.nvfp4_quantize_cols(_p(x), int(rows), int(cols), _p(gofs), int(G),
                                                          _p(codes_t), _p(scales_t), _p(tensor_scale),
                                                          _p(amax_ws), _p(err), _stream(stream)))
    return codes_t, scales_t, tensor_scale


def grouped_gemm_nvfp4(mode, a, a_sf, a_scale, b, b_sf, b_scale, gofs, G, M, N, K, epilogue=MOE_EPI_NONE, d=None,
                       err=None, stream=None, opts=None):
    """See include/moe.h.  Allocates d when not given."""
    if d is None:
        shape = (G, M, N) if mode == MOE_GEMM_WGRAD else (M, N)
        d = _empty(shape, torch.float32 if epilogue == MOE_EPI_NONE_F32 else torch.bfloat16, a)
    args = (int(mode), _p(a), _p(a_sf), _p(a_scale), _p(b), _p(b_sf), _p(b_scale), _p(gofs), int(G), int(M), int(N),
            int(K), int(epilogue), _p(d))
    if opts is None:
        _check("grouped_gemm_nvfp4", lib.grouped_gemm_nvfp4(*args, _p(err), _stream(stream)))
    else:
        _check("grouped_gemm_nvfp4_ex", lib.grouped_gemm_nvfp4_ex(*args, ctypes.byref(opts), _p(err),
                                                                  _stream(stream)))
    return d


def moe_selftest_bounded_wait(timeout_ns, err, completed, stream=None):
    """A bounded wait on an mbarrier that nothing arrives at (include/moe.h)."""
    _check("moe_selftest_bounded_wait", lib.moe_selftest_bounded_wait(int(timeout_ns), _p(err), _p(completed),
                                                                      _stream(stream)))

