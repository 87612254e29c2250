"""CPU checks of the full-size parity machinery (parity_pool.OraclePool):
chunked over rows and columns and spread over worker processes, it must
report nothing for the oracle's own output and find a single changed byte
in either axis' codes or scales."""
import numpy as np

import oracle as O
from parity_pool import OraclePool, bf16_bits


def test_pool_agrees_with_the_oracle_and_finds_a_planted_byte(monkeypatch):
    import parity_pool
    monkeypatch.setattr(parity_pool, "CHUNK_ELEMS", 1 << 14)      # many chunks on a small matrix
    rng = np.random.default_rng(0)
    gofs = np.array([0, 128, 128, 384, 512])                      # an empty group
    R, C = int(gofs[-1]), 160
    x = O.bf16_round(rng.standard_normal((R, C)) * np.exp2(rng.integers(-6, 6, (R, 1))))
    x[200:256] = 0.0                                              # zero padding rows of a group
    src = bf16_bits(x)
    qr, sr = O.mxfp8_quantize_rows(x)
    qc, sc, _ = O.mxfp8_quantize_cols_grouped(x, gofs)
    pool = OraclePool(workers=2)
    try:
        assert pool.check_both_axes("x", src, gofs, qr, sr, qc, sc) == []
        for which in range(4):
            arrs = [a.copy() for a in (qr, sr, qc, sc)]
            a = arrs[which]
            a.reshape(-1)[a.size // 3] ^= 1
            bad = pool.check_both_axes("x", src, gofs, *arrs)
            assert len(bad) == 1 and bad[0][2] == 1
            assert bad[0][0][1] == ("rows" if which < 2 else "cols")
            assert bad[0][1] == ("codes" if which % 2 == 0 else "scales")
    finally:
        pool.close()
