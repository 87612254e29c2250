"""A process pool for the full-size parity checks: the oracle's MXFP8
quantization of whole tensors (both axes), cut into chunks and spread over
the host's cores.  Test infrastructure only; the arithmetic is the oracle's
(oracle.mxfp8_quantize_rows / mxfp8_quantize_cols_grouped), this module
only cuts the inputs into chunks and compares bytes.

The pool uses the "spawn" start method: a worker forked from a process that
has already used CUDA can hang.  Workers import numpy and the oracle only.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

CHUNK_ELEMS = 1 << 22


def bf16_bits(x64):
    """fp64 values that are exact bf16 numbers -> their bf16 bit patterns (u16)."""
    f32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def _from_bits(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _mismatch(want, got):
    want, got = np.asarray(want), np.asarray(got)
    if want.shape != got.shape:
        return (-1, f"shape {got.shape} != {want.shape}")
    bad = np.flatnonzero(want.reshape(-1) != got.reshape(-1))
    if len(bad) == 0:
        return (0, None)
    i = int(bad[0])
    return (len(bad), (np.unravel_index(i, want.shape), int(got.reshape(-1)[i]), int(want.reshape(-1)[i])))


def _rows_task(src_u16, codes, scales):
    import oracle as O
    q, s = O.mxfp8_quantize_rows(_from_bits(src_u16))
    return _mismatch(q, codes), _mismatch(s, scales)


def _cols_task(src_u16, gofs, codes_t, scales_t):
    import oracle as O
    q, s, padded = O.mxfp8_quantize_cols_grouped(_from_bits(src_u16), gofs)
    assert np.array_equal(padded, gofs)         # 128-row groups are their own padded layout
    return _mismatch(q, codes_t), _mismatch(s, scales_t)


class OraclePool:
    def __init__(self, workers=None):
        n = workers or min(16, os.cpu_count() or 1)
        self.workers = n
        self.ex = ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)

    def _run(self, tasks):
        """tasks: iterable of (label, fn, args); at most 2 x workers in flight.
        Returns the labels of the chunks that differ, with the first
        difference of each."""
        bad, pending = [], []

        def drain(limit):
            while len(pending) > limit:
                label, fut = pending.pop(0)
                for what, (n, first) in zip(("codes", "scales"), fut.result()):
                    if n != 0:
                        bad.append((label, what, n, first))

        for label, fn, args in tasks:
            pending.append((label, self.ex.submit(fn, *args)))
            drain(2 * self.workers)
        drain(0)
        return bad

    def check_both_axes(self, name, src_u16, gofs, codes_row, scales_row, codes_col, scales_col):
        """src_u16 [R, C]: the bf16 bits of the matrix the GPU quantized, R =
        gofs[-1] (whole 128-row groups, padding rows zero).  codes_row [R, C]
        and scales_row [R, C/32] (canonical) are the GPU's rowwise output;
        codes_col [C, R] and scales_col [C, R/32] its group-aware columnwise
        output.  Every byte is compared with the oracle's; returns a list of
        differences (empty when all match)."""
        R, C = src_u16.shape
        gofs = np.asarray(gofs, dtype=np.int64)
        assert int(gofs[0]) == 0 and int(gofs[-1]) == R

        def tasks():
            rstep = max(1, CHUNK_ELEMS // C)
            for r0 in range(0, R, rstep):
                r1 = min(R, r0 + rstep)
                yield ((name, "rows", r0, r1), _rows_task, (src_u16[r0:r1], codes_row[r0:r1], scales_row[r0:r1]))
            cstep = max(32, (CHUNK_ELEMS // max(R, 1)) // 32 * 32)
            for c0 in range(0, C, cstep):
                c1 = min(C, c0 + cstep)
                yield ((name, "cols", c0, c1), _cols_task,
                       (np.ascontiguousarray(src_u16[:, c0:c1]), gofs, codes_col[c0:c1], scales_col[c0:c1]))

        return self._run(tasks())
