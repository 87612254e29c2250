"""Test-side helpers: layout conversions documented in include/moe.h and the
comparison rules of the parity tests.  No step of the method lives here."""
from __future__ import annotations

import functools
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402


def atoms_to_rowmajor(atoms, rows, cols):
    """Scale atoms (moe.h "atom layout") of a [rows, cols] matrix quantized
    along cols -> canonical [rows, cols/32] uint8."""
    atoms = np.asarray(atoms, dtype=np.uint8).reshape(-1)
    nb = cols // 32
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    off = ((b // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return atoms[off]


def atoms_rows_subset(atoms, rows, cols, row_idx):
    """Canonical scales of selected rows only."""
    atoms = np.asarray(atoms, dtype=np.uint8).reshape(-1)
    nb = cols // 32
    r = np.asarray(row_idx)[:, None]
    b = np.arange(nb)[None, :]
    off = ((b // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return atoms[off]


def atoms_block_range(atoms, rows, cols, b_lo, b_hi):
    """Canonical scales [rows, b_hi - b_lo] of blocks b_lo .. b_hi-1 of every
    row of a [rows, cols] matrix whose scales are in the atom layout."""
    atoms = np.asarray(atoms, dtype=np.uint8).reshape(-1)
    r = np.arange(rows)[:, None]
    b = np.arange(b_lo, b_hi)[None, :]
    off = ((b // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return atoms[off]


def rowmajor_to_tile224(canon):
    """Canonical scales [R, C/32] -> the tile-224 layout of include/moe.h
    (for k-block kb and 224-row tile t, 1024 bytes at (kb * T + t) * 1024,
    the atom layout of the tile's rows on their own; unused bytes zero)."""
    canon = np.asarray(canon, dtype=np.uint8)
    R, nb = canon.shape
    T = (R + 223) // 224
    out = np.zeros((nb // 4) * T * 1024, dtype=np.uint8)
    r = np.arange(R)[:, None]
    b = np.arange(nb)[None, :]
    t, rp = r // 224, r % 224
    off = ((b // 4) * T + t) * 1024 + (rp // 128) * 512 + (rp % 32) * 16 + ((rp // 32) % 4) * 4 + (b % 4)
    out[off] = canon
    return out


def tile224_to_rowmajor(buf, R, C):
    """Inverse of rowmajor_to_tile224 for a [R, C] matrix (C % 128 == 0)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    T = (R + 223) // 224
    r = np.arange(R)[:, None]
    b = np.arange(C // 32)[None, :]
    t, rp = r // 224, r % 224
    off = ((b // 4) * T + t) * 1024 + (rp // 128) * 512 + (rp % 32) * 16 + ((rp // 32) % 4) * 4 + (b % 4)
    return buf[off]


def tile224_block_range(buf, R, C, b_lo, b_hi, rows=None):
    """Canonical scales [len(rows), b_hi - b_lo] (rows default: all R) of
    blocks b_lo .. b_hi-1 of a [R, C] matrix whose scales are in the tile-224
    layout."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    T = (R + 223) // 224
    r = (np.arange(R) if rows is None else np.asarray(rows))[:, None]
    b = np.arange(b_lo, b_hi)[None, :]
    t, rp = r // 224, r % 224
    off = ((b // 4) * T + t) * 1024 + (rp // 128) * 512 + (rp % 32) * 16 + ((rp // 32) % 4) * 4 + (b % 4)
    return buf[off]


def colwise_scales_rowmajor(buf, C, M, tile224):
    """Canonical [C, M/32] scales of a columnwise (transposed) output [C, M]
    in the atom layout or, when tile224, the tile-224 layout."""
    return tile224_to_rowmajor(buf, C, M) if tile224 else atoms_to_rowmajor(buf, C, M)


def bf16_bits_of(t):
    """Bit patterns (numpy u16) of a bf16 torch tensor."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def assert_bf16_close(gpu, ref64, rel_frob=1e-3, elem=1e-2, what=""):
    """GPU bf16 result vs the fp64 oracle.

    Rule: relative Frobenius error <= 1e-3 against the oracle rounded once to
    the output type (bf16), and per element |gpu - ref| <= 1e-2 (|ref| +
    rms(ref)) against the unrounded fp64 oracle.
    """
    g = gpu if isinstance(gpu, np.ndarray) else to_np(gpu)
    ref64 = np.asarray(ref64, dtype=np.float64)
    assert g.shape == ref64.shape, (what, g.shape, ref64.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    nref = np.linalg.norm(ref64)
    if nref == 0:
        assert np.all(g == 0), f"{what}: expected zeros"
        return 0.0
    frob = np.linalg.norm(g - O.bf16_round(ref64)) / nref
    rms = np.sqrt(np.mean(ref64 ** 2))
    bad = np.abs(g - ref64) > elem * (np.abs(ref64) + rms)
    assert frob <= rel_frob, f"{what}: relative Frobenius error {frob:.3e} > {rel_frob}"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside 1e-2(|ref|+rms); first at "
                           f"{np.argwhere(bad)[0]}: gpu {g[tuple(np.argwhere(bad)[0])]} ref "
                           f"{ref64[tuple(np.argwhere(bad)[0])]}")
    return frob


def build_lib():
    from grouped_gemm_top_gb300 import build
    return build.build()


def deq_rows(codes, atoms, rows_total, cols, row_idx):
    """fp64 dequantized rows `row_idx` of a rowwise-quantized [rows_total,
    cols] matrix stored as codes + scale atoms (oracle dequantizer)."""
    codes = np.asarray(codes)
    row_idx = np.asarray(row_idx)
    sc = atoms_rows_subset(atoms, rows_total, cols, row_idx)
    return O.mxfp8_dequantize_rows(codes[row_idx], sc)


def gpu_ops():
    """Build (if needed), load and initialise libmoe on cuda:0."""
    build_lib()
    from grouped_gemm_top_gb300 import ops
    ops.moe_init(0)
    return ops


class KernelOps:
    """The ops module with every grouped-GEMM call bound to one kernel
    choice (moe_gemm_opts_t through the *_ex entry points), so a test file
    can run its whole GEMM suite once per kernel in one process."""
    GEMMS = ("grouped_gemm_mxfp8", "grouped_gemm_mxfp8_swiglu_quant", "grouped_gemm_nvfp4")

    def __init__(self, ops, kernel):
        self._ops = ops
        self.kernel = kernel
        self._opts = ops.gemm_opts(kernel)

    def __getattr__(self, name):
        v = getattr(self._ops, name)
        if name in self.GEMMS:
            return functools.partial(v, opts=self._opts)
        return v


def padded_layout(sizes, align=128):
    sizes = np.asarray(sizes, dtype=np.int64)
    gofs = np.concatenate([[0], np.cumsum((sizes + align - 1) // align * align)])
    return gofs


def assert_fp32_close(gpu, ref64, rel_frob=1e-5, what=""):
    """fp32 GPU result (no bf16 output rounding) vs the fp64 oracle:
    relative Frobenius error <= 1e-5 (fp32 accumulation order only)."""
    g = np.asarray(gpu if isinstance(gpu, np.ndarray) else gpu.double().cpu().numpy(), dtype=np.float64)
    ref64 = np.asarray(ref64, dtype=np.float64)
    assert g.shape == ref64.shape and np.all(np.isfinite(g)), what
    frob = np.linalg.norm(g - ref64) / max(np.linalg.norm(ref64), 1e-300)
    assert frob <= rel_frob, f"{what}: relative Frobenius error {frob:.3e} > {rel_frob}"
    return frob


def glu_perm(n):
    """Row r of a MOE_QUANT_COLWISE_GLU output holds input column glu_perm(n)[r]
    (moe.h: gate/up halves interleaved in 64-row chunks)."""
    r = np.arange(n)
    j, w = r // 128, r % 128
    return np.where(w < 64, 64 * j + w, n // 2 + 64 * j + (w - 64))


def batched_weight_operand(q, s, G, cols, Kg, glu=False):
    """Dequantize a MOE_QUANT_COLWISE_BATCHED[_GLU] operand (codes
    [G][cols][Kg], scales in the atom layout of [G*cols, Kg]) back to the
    logical weight [G, Kg, cols] (moe.h)."""
    qn = np.asarray(q).reshape(G * cols, Kg)
    sc = atoms_to_rowmajor(np.asarray(s), G * cols, Kg)
    deq = O.mxfp8_dequantize_rows(qn, sc).reshape(G, cols, Kg)
    perm = glu_perm(cols) if glu else np.arange(cols)
    out = np.empty_like(deq)
    out[:, perm, :] = deq
    return np.transpose(out, (0, 2, 1))
