"""The layer's two weight-gradient launches cover every group exactly once:
the 224-wide launch's filter and the 256-wide launch's (the complement,
lo and hi swapped) checked against the filter as include/moe.h defines it
(moe_gemm_opts_t wgrad_rows_lo / wgrad_rows_hi) on every padded row count."""
import pytest

from grouped_gemm_top_gb300.layer import WGRAD224_ROWS, wgrad_band_filters


def passes(r, lo, hi):
    """moe.h: hi == 0: r >= lo; lo < hi: lo <= r < hi; 0 < hi <= lo: r < hi or r >= lo."""
    if hi == 0:
        return r >= lo
    if lo < hi:
        return lo <= r < hi
    return r < hi or r >= lo


@pytest.mark.parametrize("band", [WGRAD224_ROWS, (0, 1024), (512, 0), (128, 0), (0, 128), (512, 640), (1, 2)])
def test_two_launches_cover_every_group_once(band):
    f224, f256 = wgrad_band_filters(*band)
    assert f224 == band
    for r in list(range(0, 40000, 128)) + [1, 127, 129, band[0], band[1], max(band[0] - 1, 0), band[1] + 1]:
        in224, in256 = passes(r, *f224), passes(r, *f256)
        assert in224 != in256, (band, r)
        lo, hi = band
        assert in224 == (r >= lo and (hi == 0 or r < hi)), (band, r)
