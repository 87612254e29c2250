"""Pins for the oracle's number formats and MXFP8 quantizer (CPU only).

Each test ties the oracle to something other than itself: values printed on
the pages (tests/golden/), closed forms of the formats, a library conversion
(torch's float8 casts) or brute force over every representable value.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _all_bf16_values():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float().numpy()
    return v[np.isfinite(v)].astype(np.float64)


# ---------------------------------------------------------------- bf16 ----

def test_fp32_storage_example_pins_bias_and_bf16():
    g = _golden("fp32_storage_4p8125.json")
    e = int(g["exponent"], 2) - g["bias"]
    sig = 1 + int(g["mantissa"], 2) / 2 ** 23
    assert sig == g["significand"] and sig * 2 ** e == g["value"]
    # 4.8125 needs 6 fraction bits, so it is a bf16 value: bf16 keeps the
    # FP32 sign/exponent and the top 7 mantissa bits (precision table 1+8+7)
    assert O.bf16_round(np.array([g["value"]]))[0] == g["value"]
    bits16 = int(g["sign"] + g["exponent"] + g["mantissa"][:7], 2)
    assert torch.tensor([bits16], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item() == g["value"]
    # one more mantissa bit than bf16 holds gets rounded to even
    x = g["value"] + 2.0 ** (2 - 8)          # half a bf16 ulp above 4.8125 (ulp 2^-5 at [4,8))
    assert O.bf16_round(np.array([x]))[0] in (4.8125, 4.84375)


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000)),
        rng.standard_normal(1000) * 1e-39,                 # bf16 subnormals
        np.array([0.0, -0.0, 3.0e38, -3.4e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]),
    ])
    # torch converts fp64 through fp32 (two roundings), so compare on fp32
    # inputs, where its fp32 -> bf16 cast is a single round-to-nearest-even
    x = x.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    got = O.bf16_round(x)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- E4M3 ----

def test_e4m3_closed_forms():
    t = _golden("precision_table.json")
    assert t["formats"]["FP8_E4M3"] == [1, 4, 3]
    vals = O.E4M3_VALUES
    assert np.isnan(vals).sum() == 2 and np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert np.nanmax(vals) == 448.0 and vals[0x7E] == 448.0
    assert vals[0x01] == 2.0 ** -9            # smallest subnormal m/8 * 2^-6
    assert vals[0x08] == 2.0 ** -6            # smallest normal
    assert vals[0x38] == 1.0                  # exponent field 7 == bias
    assert vals[0x80] == 0.0 and math.copysign(1, vals[0x80]) < 0
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)           # codes are monotone in value
    assert np.array_equal(vals[0x80:0xFF], -vals[:0x7F])


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = O.E4M3_VALUES
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_encode_all_bf16_matches_torch_rne():
    v = _all_bf16_values()
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v)
    assert np.array_equal(got, ref)


def test_e4m3_encode_brute_force_nearest_even():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(-460, 460, 3000), rng.uniform(-0.02, 0.02, 3000),
                        (O.E4M3_VALUES[1:0x7E] + O.E4M3_VALUES[2:0x7F]) / 2])   # exact ties
    got = O.e4m3_encode(v)
    fin_codes = [c for c in range(256) if np.isfinite(O.E4M3_VALUES[c])]
    for x, c in zip(v, got):
        a = min(abs(x), 448.0)
        best = min(abs(a - O.E4M3_VALUES[cc]) for cc in fin_codes if cc < 0x80)
        cands = [cc for cc in range(0x7F) if abs(a - O.E4M3_VALUES[cc]) == best]
        want = [cc for cc in cands if cc % 2 == 0] if len(cands) > 1 else cands
        assert (c & 0x7F) == want[0]
        assert (c >> 7) == (1 if np.signbit(x) else 0)


# ---------------------------------------------------------------- E8M0 ----

def test_e8m0_decode_matches_torch():
    b = np.arange(256)
    ref = torch.from_numpy(b.astype(np.uint8)).view(torch.float8_e8m0fnu).double().numpy()
    got = O.e8m0_value(b)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_scale_rule_closed_form_on_every_bf16():
    """e = smallest integer with amax <= 448 * 2^e.  For a normal amax =
    M * 2^q (M in [1, 2)) that is q - 8 when M <= 1.75 and q - 7 otherwise."""
    v = _all_bf16_values()
    a = np.unique(np.abs(v[v != 0]))
    e = O.e8m0_exponent(a)
    mant, q = np.frexp(a)                      # a = mant * 2^q, mant in [0.5, 1)
    M, q = mant * 2, q - 1
    closed = np.where(M > 1.75, q - 7, q - 8)
    closed = np.clip(closed, -127, 127)
    assert np.array_equal(e, closed)
    # definition, checked directly where the clamp is inactive
    ok = e > -127
    assert np.all(a[ok] <= 448.0 * np.ldexp(1.0, e[ok]))
    assert np.all(a[ok] > 448.0 * np.ldexp(1.0, e[ok] - 1))
    assert O.e8m0_byte(np.array([0.0]))[0] == 0


@pytest.mark.parametrize("j", [-20, -1, 0, 3, 17])
def test_scale_rule_boundaries(j):
    s = 2.0 ** j
    ulp = 2.0 ** (8 + j - 7)               # bf16 spacing in [256, 512) * 2^j
    assert O.e8m0_exponent(np.array([448.0 * s]))[0] == j
    assert O.e8m0_exponent(np.array([448.0 * s + ulp]))[0] == j + 1
    assert O.e8m0_exponent(np.array([1.75 * s]))[0] == j - 8
    assert O.e8m0_exponent(np.array([1.875 * s]))[0] == j - 7


def test_scale_monotone_in_amax():
    rng = np.random.default_rng(2)
    a = np.sort(np.abs(rng.standard_normal(50000)) * np.exp(rng.uniform(-30, 30, 50000)))
    e = O.e8m0_exponent(a)
    assert np.all(np.diff(e) >= 0)


# ------------------------------------------------------- MXFP8 quantize ----

def test_mxfp8_block_is_32():
    assert _golden("precision_table.json")["mxfp8_block"] == O.MXFP8_BLOCK == 32


def _representable_blocks(rng, nblocks, j):
    """Blocks of E4M3 values times 2^j whose largest magnitude is in (224, 448]."""
    fin = np.array([c for c in range(256) if np.isfinite(O.E4M3_VALUES[c])])
    codes = rng.choice(fin, size=(nblocks, 32))
    big = np.array([c for c in fin if 224 < abs(O.E4M3_VALUES[c]) <= 448])
    codes[:, rng.integers(0, 32)] = rng.choice(big, size=nblocks)
    return O.E4M3_VALUES[codes] * 2.0 ** j, codes


@pytest.mark.parametrize("j", [-30, -9, 0, 5, 40])
def test_mxfp8_roundtrip_exact_on_representable(j):
    rng = np.random.default_rng(3 + j + 100)
    x, codes = _representable_blocks(rng, 64, j)
    q, s = O.mxfp8_quantize_rows(x.reshape(8, 256))
    assert np.all(s == j + 127)
    back = O.mxfp8_dequantize_rows(q, s)
    assert np.array_equal(back, x.reshape(8, 256))
    # the codes are the generating codes (up to the sign of zero)
    same = (q.reshape(64, 32) == codes) | ((O.E4M3_VALUES[codes] == 0) & ((q.reshape(64, 32) & 0x7F) == 0))
    assert np.all(same)


def test_mxfp8_rowwise_brute_force():
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((6, 96)) * 3).to(torch.bfloat16).double().numpy()
    x[0, :32] = 0.0                              # all-zero block -> scale byte 0, codes 0
    x[1, 32:64] *= 1e-30
    q, s = O.mxfp8_quantize_rows(x)
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    for r in range(6):
        for b in range(3):
            blk = x[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            if amax == 0:
                continue
            e = int(s[r, b]) - 127
            assert amax <= 448 * 2.0 ** e and not (amax <= 448 * 2.0 ** (e - 1) and e > -127)
            for i in range(32):
                y = blk[i] * 2.0 ** -e
                got = O.E4M3_VALUES[q[r, 32 * b + i]]
                err = abs(got - y)
                assert all(err <= abs(O.E4M3_VALUES[c] - y) for c in range(0x7F))


def test_colwise_grouped_blocks_restart_at_group_start():
    rng = np.random.default_rng(5)
    sizes = [5, 0, 40, 33, 64]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    x = torch.from_numpy(rng.standard_normal((offs[-1], 64))).to(torch.bfloat16).double().numpy()
    qt, st, padded = O.mxfp8_quantize_cols_grouped(x, offs)
    assert list(padded) == [0, 32, 32, 96, 160, 224]
    assert qt.shape == (64, 224) and st.shape == (64, 7)
    back = O.mxfp8_dequantize_cols(qt, st)
    for g in range(len(sizes)):
        pad_rows = back[padded[g] + sizes[g]:padded[g + 1]]
        assert np.all(pad_rows == 0)                     # zero padding
    # a group's codes depend only on its own rows
    x2 = x.copy()
    x2[offs[2]:offs[3]] *= 7.0
    qt2, st2, _ = O.mxfp8_quantize_cols_grouped(x2, offs)
    keep = np.r_[0:32, 96:224]
    assert np.array_equal(qt[:, keep], qt2[:, keep]) and np.array_equal(st[:, np.r_[0:1, 3:7]], st2[:, np.r_[0:1, 3:7]])
    # one aligned group reduces to the rowwise quantizer on the transpose
    x3 = torch.from_numpy(rng.standard_normal((160, 64))).to(torch.bfloat16).double().numpy()
    q1, s1, _ = O.mxfp8_quantize_cols_grouped(x3, np.array([0, 160]))
    qr, sr = O.mxfp8_quantize_rows(x3.T.copy())
    assert np.array_equal(q1, qr) and np.array_equal(s1, sr)
