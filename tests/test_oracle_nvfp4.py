"""Pins for the oracle's FP4 E2M1 format and two-level NVFP4 quantizer
(CPU only): the pages' format split (tests/golden/), the closed form of a
1+2+1 float, hand-worked blocks whose scales are exact, brute force over the
eight magnitudes, and the error bound the two scales imply."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float64)).bfloat16().double().numpy()


def test_e2m1_table_from_the_format_split():
    with open(os.path.join(GOLDEN, "precision_table.json")) as f:
        split = json.load(f)["formats"]["FP4_E2M1"]
    assert split == [1, 2, 1] and len(O.E2M1_VALUES) == 2 ** sum(split)
    # closed form of a 1+2+1 float, bias 1: largest 1.5 * 2^2, smallest
    # normal 2^0, the one subnormal 0.5 * 2^0
    pos = O.E2M1_VALUES[:8]
    assert pos.max() == O.E2M1_MAX == 6.0
    assert pos[2] == 1.0 and pos[1] == 0.5 and pos[0] == 0.0
    assert np.array_equal(pos, [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    assert np.array_equal(O.E2M1_VALUES[8:], -pos)


@pytest.mark.parametrize("v,code", [
    (0.25, 0x0), (0.26, 0x1), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
    (5.01, 0x7), (6.0, 0x7), (7.0, 0x7), (1e9, 0x7), (-0.1, 0x8), (-2.9, 0xD), (-100.0, 0xF), (0.0, 0x0),
])
def test_e2m1_encode_ties_even_and_saturates(v, code):
    assert int(O.e2m1_encode(np.array([v]))[0]) == code


def test_e2m1_encode_is_the_nearest_value_brute_force():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-7, 7, 5000), O.E2M1_VALUES, (O.E2M1_VALUES[:7] + O.E2M1_VALUES[1:8]) / 2])
    codes = O.e2m1_encode(v).astype(np.int64)
    got = O.E2M1_VALUES[codes]
    mags = O.E2M1_VALUES[:8]
    for x, c, g in zip(v, codes, got):
        d = np.abs(np.abs(x) - mags)
        best = d.min()
        assert abs(abs(x) - abs(g)) == best or (abs(x) > 6 and abs(g) == 6)
        if np.count_nonzero(d == best) == 2 and abs(x) <= 6:   # a tie picks the even code
            assert (c & 7) % 2 == 0
        assert (c >> 3) == int(np.signbit(x))


def test_nvfp4_worked_blocks_with_exact_scales():
    """amax 2688 = 6 * 448 makes s_t exactly 1; then a block with amax 12
    has s_b = 2 (exact) and codes x / 2, the block of the tensor maximum has
    s_b = 448, an all-zero block and a negligible one get scale byte 0."""
    x = np.zeros((2, 64))
    x[0, :16] = [2688.0, -448.0] + [0.0] * 14                     # s_b = 448: codes 6, -1
    x[0, 16:32] = 2.0 * O.E2M1_VALUES                              # amax 12 -> s_b = 2
    x[0, 48:64] = 2.0 ** -12                                       # t_b = 2^-12 / 6: rounds to zero
    x[1, :16] = 2.0 * O.E2M1_VALUES[::-1]                          # the same values, reversed
    x = _bf16(x)
    q, s, st = O.nvfp4_quantize_rows(x)
    assert st == np.float32(1.0)
    assert s[0, 0] == 0x7E and q[0, 0] == 0x7 and q[0, 1] == 0xA   # 448 and E2M1 codes of 6, -1
    assert O.E4M3_VALUES[s[0, 1]] == 2.0 and np.array_equal(q[0, 16:32], np.arange(16))
    assert s[0, 2] == 0 and s[0, 3] == 0 and not q[0, 32:].any()
    assert np.array_equal(q[1, :16], np.arange(16)[::-1])
    back = O.nvfp4_dequantize_rows(q, s, st)
    assert np.array_equal(back[:, :32], x[:, :32]) and not back[0, 32:].any()


def test_nvfp4_largest_block_scale_and_code():
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((16, 256)) * 3.0)
    q, s, st = O.nvfp4_quantize_rows(x)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert s[r, c // 16] == 0x7E                   # t_b = amax / 6 / (amax / 2688) = 448
    assert (q[r, c] & 7) == 7                      # the maximum itself is +-6
    assert st == np.float32(np.float32(np.abs(x).max()) / np.float32(2688.0))


@pytest.mark.parametrize("scale", [1e-6, 1.0, 3e4])
def test_nvfp4_error_bound(scale):
    """Every element is within s_b * s_t of its dequantized value: half the
    widest E2M1 spacing (4 -> 6) is 1, and saturation above 6 costs at most
    6 * 2^-4 (the E4M3 rounding of t_b) in the same units."""
    rng = np.random.default_rng(9)
    x = _bf16(rng.standard_normal((32, 128)) * scale * np.exp(rng.uniform(-3, 3, (32, 1))))
    q, s, st = O.nvfp4_quantize_rows(x)
    back = O.nvfp4_dequantize_rows(q, s, st)
    unit = np.repeat(O.E4M3_VALUES[s.astype(np.int64)], 16, axis=1) * float(st)
    assert np.all(np.abs(x - back) <= unit * (1.0 + 1e-9))
    rel = np.linalg.norm(x - back) / np.linalg.norm(x)
    assert rel < 0.15


def test_nvfp4_blocks_run_along_rows():
    """A block is 16 consecutive elements of one row: scaling one row's block
    changes only that block's scale byte."""
    rng = np.random.default_rng(2)
    x = _bf16(rng.standard_normal((4, 64)))
    y = x.copy()
    y[2, 16:32] *= 0.25                             # an exact power of two: the block's scale shrinks 4x
    _, sx, _ = O.nvfp4_quantize_rows(x)
    _, sy, _ = O.nvfp4_quantize_rows(y)
    diff = np.argwhere(sx != sy)
    assert diff.tolist() == [[2, 1]]


def test_nvfp4_zero_tensor():
    q, s, st = O.nvfp4_quantize_rows(np.zeros((2, 32)))
    assert st == 0 and not q.any() and not s.any()


def test_nvfp4_cols_grouped_reduces_to_rowwise_of_the_transpose():
    """With every group a multiple of 16 rows there is no padding: the
    columnwise codes are the rowwise codes of x transposed, with the same
    tensor scale as the rowwise quantization of x."""
    rng = np.random.default_rng(21)
    x = _bf16(rng.standard_normal((96, 32)) * np.exp(rng.uniform(-2, 2, (96, 1))))
    q, s, st, padded = O.nvfp4_quantize_cols_grouped(x, [0, 32, 32, 96])
    qr, sr, st_r = O.nvfp4_quantize_rows(x.T)
    assert np.array_equal(padded, [0, 32, 32, 96])
    assert np.array_equal(q, qr) and np.array_equal(s, sr) and st == st_r
    assert st == O.nvfp4_quantize_rows(x)[2]


def test_nvfp4_cols_grouped_blocks_restart_at_group_starts():
    """A group of 20 rows takes two blocks (16 + 4 rows, zero-padded to 16);
    the next group starts a fresh block: scaling its rows changes only its
    blocks' scale bytes, and the padding rows dequantize to zero."""
    rng = np.random.default_rng(8)
    x = _bf16(rng.standard_normal((36, 16)))
    x[0, 0] = 64.0                                   # the tensor maximum sits in group 0
    q, s, st, padded = O.nvfp4_quantize_cols_grouped(x, [0, 20, 36])
    assert np.array_equal(padded, [0, 32, 48]) and q.shape == (16, 48) and s.shape == (16, 3)
    back = O.nvfp4_dequantize_cols(q, s, st)
    assert not back[20:32].any()                     # padding of group 0's tail block
    y = x.copy()
    y[20:36] *= 0.5                                  # group 1 only (exact)
    _, s2, st2, _ = O.nvfp4_quantize_cols_grouped(y, [0, 20, 36])
    assert st2 == st
    assert np.array_equal(s2[:, :2], s[:, :2]) and not np.array_equal(s2[:, 2], s[:, 2])
    # every element within one unit (s_b * s_t) of its value
    unit = np.repeat(O.E4M3_VALUES[s.astype(np.int64)], 16, axis=1).T * float(st)
    xpad = np.zeros((48, 16))
    xpad[:20], xpad[32:48] = x[:20], x[20:36]
    assert np.all(np.abs(back - xpad) <= unit * (1 + 1e-9))
