"""Weight gradients split by group size (moe_gemm_opts_t wgrad_rows_lo /
wgrad_rows_hi): the groups in a row band on the 224-wide CTA-pair tiles
(right operand's scales in the tile-224 layout), the others (the filter
with lo and hi swapped) on the 256-wide tiles (atom layout), chosen on the
device from the offsets.  Each launch writes only its own groups; together
they equal the oracle's weight gradient, empty groups zero."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_bf16_close, atoms_to_rowmajor, gpu_ops, padded_layout, rowmajor_to_tile224
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _act(sizes, K, seed, row_cap=None):
    gofs = padded_layout(sizes)
    M = row_cap or int(gofs[-1]) + 128
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    src = synth.make_normal_bf16((int(sum(sizes)) + 1, K), seed, "cuda")
    r = 0
    for g, m in enumerate(sizes):
        x[gofs[g]:gofs[g] + m] = src[r:r + m]
        r += m
    return x, torch.tensor(gofs, dtype=torch.int32, device="cuda"), gofs


def _in_band(r, lo, hi):
    if hi == 0:
        return r >= lo
    return (lo <= r) & (r < hi) if lo < hi else (r < hi) | (r >= lo)


@pytest.mark.parametrize("sizes,Mo,No,band", [
    ([128, 0, 700, 2600, 5, 1200], 256, 512, (0, 1024)),      # 256 x 256 pair tiles for the rest
    ([128, 0, 700, 2600, 5, 1200], 256, 512, (512, 2048)),    # a band: the rest is below and above it
    ([3000, 0, 0, 64], 512, 896, (0, 2048)),                  # N % 256 != 0: the rest on 256 x 128 pair tiles
    ([300, 40], 256, 384, (0, 4096)),                         # everything in the band: the second launch idles
    ([2100, 2200], 256, 640, (0, 128)),                       # nothing in the band (no empty group)
    ([900, 0, 100, 5000], 256, 512, (128, 0)),                # an open band; the empty group goes with the rest
])
def test_wgrad_split_by_group_rows(ops, sizes, Mo, No, band):
    G = len(sizes)
    a, gofs_t, gofs = _act(sizes, Mo, seed=91)
    g_, _, _ = _act(sizes, No, seed=92, row_cap=a.shape[0])
    Kc = a.shape[0]
    aq, as_ = ops.mxfp8_group_quantize(a, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    gq, gs = ops.mxfp8_group_quantize(g_, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    torch.cuda.synchronize()
    G_can = atoms_to_rowmajor(gs.cpu().numpy(), No, Kc)
    gs224 = torch.from_numpy(rowmajor_to_tile224(G_can)).cuda()
    lo, hi = band
    small = _in_band(np.diff(gofs), lo, hi)       # the filter counts a group's padded rows
    d = torch.full((G, Mo, No), 3.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs224, ops.MOE_B_SF_TILE224, gofs_t, G, Mo, No, Kc,
                           d=d, err=err, opts=ops.gemm_opts(wgrad_rows=band))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for g in range(G):
        if not small[g]:
            assert torch.all(d[g] == 3.0), f"group {g} written by the band's launch"
    first = d.clone()
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs, ops.MOE_B_GNK, gofs_t, G, Mo, No, Kc, d=d, err=err,
                           opts=ops.gemm_opts(wgrad_rows=(hi, lo)))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for g in range(G):
        if small[g]:
            assert torch.equal(d[g], first[g]), f"group {g} written by the complement's launch"
    Rp = int(gofs[-1])
    Ah = O.mxfp8_dequantize_cols(aq.cpu().numpy()[:, :Rp], atoms_to_rowmajor(as_.cpu().numpy(), Mo, Kc)[:, :Rp // 32])
    Gh = O.mxfp8_dequantize_cols(gq.cpu().numpy()[:, :Rp], G_can[:, :Rp // 32])
    ref = O.grouped_gemm_wgrad(Ah, Gh, gofs)
    for g in range(G):
        if sizes[g] == 0:
            assert torch.all(d[g] == 0)
        else:
            assert_bf16_close(d[g], ref[g], what=f"split wgrad g={g} ({'224' if small[g] else '256'}-wide)")


def test_wgrad_filter_refused_where_unsupported(ops):
    """A group filter on FWD, or on a weight gradient that would run on the
    1-SM kernel (M % 256 != 0, or the 1-SM kernel asked for), is refused
    before anything runs."""
    sizes, Mo, No = [256, 128], 128, 256
    G = len(sizes)
    a, gofs_t, gofs = _act(sizes, Mo, seed=3)
    g_, _, _ = _act(sizes, No, seed=4, row_cap=a.shape[0])
    Kc = a.shape[0]
    aq, as_ = ops.mxfp8_group_quantize(a, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    gq, gs = ops.mxfp8_group_quantize(g_, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    d = torch.full((G, Mo, No), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoEError) as e:                    # M = 128: the 1-SM kernel
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs, ops.MOE_B_GNK, gofs_t, G, Mo, No, Kc, d=d,
                               opts=ops.gemm_opts(wgrad_rows=(200, 0)))
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    a2, _, _ = _act(sizes, 256, seed=5, row_cap=a.shape[0])
    aq2, as2 = ops.mxfp8_group_quantize(a2, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    d2 = torch.full((G, 256, No), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoEError) as e:                    # the 1-SM kernel asked for
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq2, as2, gq, gs, ops.MOE_B_GNK, gofs_t, G, 256, No, Kc, d=d2,
                               opts=ops.gemm_opts("1sm", wgrad_rows=(0, 200)))
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(d == 3.0) and torch.all(d2 == 3.0)
