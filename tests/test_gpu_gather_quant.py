"""mxfp8_gather_quantize vs the oracle: both MXFP8 axes of the permuted (and
router-weighted) rows, bit-exact codes and scales."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_bf16_close, atoms_rows_subset, atoms_to_rowmajor, gpu_ops, padded_layout, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _varied(rows, cols, seed):
    """bf16 rows spanning many binades, with zero and tiny rows."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, device="cuda")
    x = x * torch.exp2(torch.randint(-30, 30, (rows, 1), generator=g, device="cuda").float())
    x[0] = 0.0
    if rows > 2:
        x[2] *= 1e-36
    return x.to(torch.bfloat16)


def _routing(T, E, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits += (skew * -np.log1p(np.arange(E))).astype(np.float32)   # uneven load, some empty experts
    idx, w = O.route_topk(logits, k)
    slot_of, row_id = O.permute_slots(idx, E, 128)
    gofs = O.aligned_group_offsets(O.group_counts(idx, E), 128)
    return idx, w.astype(np.float32), slot_of, row_id, gofs


def _dev(a, dtype):
    return torch.tensor(np.ascontiguousarray(a), dtype=dtype, device="cuda")


def _check_axes(ops, P, gofs, rows, cols, res):
    """res = (codes_row, scales_row, codes_col, scales_col) of the GPU."""
    Rp = int(gofs[-1])
    cr, sr, cc, sc = res
    if cr is not None:
        rq, rs = O.mxfp8_quantize_rows(P)
        assert np.array_equal(cr[:Rp].cpu().numpy(), rq)
        assert np.array_equal(atoms_rows_subset(sr.cpu().numpy(), rows, cols, np.arange(Rp)), rs)
    if cc is not None:
        # groups start at multiples of 128 and their padding rows are zero,
        # so the oracle's per-group blocks line up with the GPU layout
        cq, cs, padded = O.mxfp8_quantize_cols_grouped(P, gofs)
        assert np.array_equal(padded, gofs)
        assert np.array_equal(cc[:, :Rp].cpu().numpy(), cq)
        assert np.array_equal(atoms_to_rowmajor(sc.cpu().numpy(), cols, rows)[:, :Rp // 32], cs)


@pytest.mark.parametrize("T,E,k,d,skew", [(1, 4, 2, 128, 0.0), (300, 8, 2, 256, 0.0), (1000, 16, 8, 512, 1.5),
                                          (64, 64, 8, 128, 3.0), (517, 32, 4, 1152, 0.5)])
def test_gather_both_axes(ops, T, E, k, d, skew):
    """x_perm quantized straight from x through row_id (oracle: permute,
    then each axis); ragged groups, empty groups, a single token."""
    idx, w, slot_of, row_id, gofs = _routing(T, E, k, seed=T + E, skew=skew)
    rows = ops.moe_row_capacity(T, E, k)
    rid = np.full(rows, -1, dtype=np.int64)
    rid[:len(row_id)] = row_id
    x = _varied(T, d, seed=T * 7 + d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = ops.mxfp8_gather_quantize(x, _dev(gofs, torch.int32), E, rows, row_id=_dev(rid, torch.int32), k=k,
                                    err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    P = O.permute(to_np(x), row_id, k)
    _check_axes(ops, P, gofs, rows, d, res)


@pytest.mark.parametrize("T,E,k,d", [(200, 8, 2, 256), (1000, 16, 8, 512), (33, 5, 3, 384)])
def test_gather_scaled_both_axes(ops, T, E, k, d):
    """dy_perm = bf16(fp32(w * dout)) quantized straight from dout (oracle:
    permute_scaled_bf16, then each axis)."""
    idx, w, slot_of, row_id, gofs = _routing(T, E, k, seed=3 * T + k)
    rows = ops.moe_row_capacity(T, E, k)
    rid = np.full(rows, -1, dtype=np.int64)
    rid[:len(row_id)] = row_id
    dout = _varied(T, d, seed=T + 11)
    res = ops.mxfp8_gather_quantize(dout, _dev(gofs, torch.int32), E, rows, row_id=_dev(rid, torch.int32), k=k,
                                    row_w=_dev(w, torch.float32))
    torch.cuda.synchronize()
    P = O.permute_scaled_bf16(to_np(dout), row_id, k, w.astype(np.float64))
    _check_axes(ops, P, gofs, rows, d, res)


def test_gather_scaled_double_rounding_case(ops):
    """The hand-worked fp32-then-bf16 rounding case of the oracle pins gives
    the same MXFP8 code on the GPU (E4M3 0x3A, not 0x3B)."""
    T, d, k = 1, 128, 1
    src = torch.zeros((T, d), dtype=torch.float32)
    src[0, 0] = float.fromhex("0x1.02p1")
    src[0, 1] = 512.0
    w = np.array([[float.fromhex("0x1.4e633ap-1")]], dtype=np.float32)
    row_id = np.array([0] + [-1] * 127)
    gofs = np.array([0, 128])
    res = ops.mxfp8_gather_quantize(src.to(torch.bfloat16).cuda(), _dev(gofs, torch.int32), 1, 128,
                                    row_id=_dev(row_id, torch.int32), k=k, row_w=_dev(w, torch.float32),
                                    colwise=False)
    torch.cuda.synchronize()
    assert int(res[0][0, 0].item()) == 0x3A
    P = O.permute_scaled_bf16(src.double().numpy(), row_id, k, w.astype(np.float64))
    _check_axes(ops, P, gofs, 128, d, res)


@pytest.mark.parametrize("sizes,cols", [([128], 128), ([5, 0, 130, 127, 1], 256), ([1000, 0, 300], 2048)])
def test_plain_both_axes_skip_tail(ops, sizes, cols):
    """Without row_id: both axes of src itself; rows >= gofs[G] are neither
    read (NaN there) nor written (sentinels survive)."""
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    rows = Rp + 256
    x = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    src = _varied(max(128, Rp), cols, seed=5 + cols)
    for g, m in enumerate(sizes):
        x[gofs[g]:gofs[g] + m] = src[gofs[g]:gofs[g] + m]
    x[Rp:] = float("nan")
    cr = torch.full((rows, cols), 0xAB, dtype=torch.uint8, device="cuda")
    sr = torch.full((rows * cols // 32,), 0xCD, dtype=torch.uint8, device="cuda")
    cc = torch.full((cols, rows), 0xAB, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows * cols // 32,), 0xCD, dtype=torch.uint8, device="cuda")
    res = ops.mxfp8_gather_quantize(x, _dev(gofs, torch.int32), len(sizes), rows, codes_row=cr, scales_row=sr,
                                    codes_col=cc, scales_col=sc)
    torch.cuda.synchronize()
    _check_axes(ops, to_np(x)[:Rp], gofs, rows, cols, res)
    assert torch.all(cr[Rp:] == 0xAB) and torch.all(cc[:, Rp:] == 0xAB)
    assert np.all(atoms_rows_subset(sr.cpu().numpy(), rows, cols, np.arange(Rp, rows)) == 0xCD)
    assert np.all(atoms_to_rowmajor(sc.cpu().numpy(), cols, rows)[:, Rp // 32:] == 0xCD)


def test_plain_both_axes_subnormal_blocks(ops):
    """Blocks whose elements are bf16 subnormals (scale byte 0: they scale by
    2^127 into the E4M3 normal range) and blocks of subnormals around a tiny
    normal maximum, on both axes; exact against the oracle."""
    rows, cols = 256, 256
    rng = np.random.default_rng(17)
    bits = (rng.integers(0x3C00, 0x4400, size=(rows, cols)) | (rng.integers(0, 2, size=(rows, cols)) << 15))
    sub = rng.integers(1, 0x80, size=(32, 32)) | (rng.integers(0, 2, size=(32, 32)) << 15)
    bits[0:32, 0:32] = sub                                   # all-subnormal blocks (rows and columns)
    bits[64:96, 64:96] = sub[::-1]
    for i in range(32):                                      # a tiny normal maximum in every row and column
        bits[64 + i, 64 + (5 * i) % 32] = 0x0380 | (int(rng.integers(0, 2)) << 15)   # 2^-120
    bits[128:160, 32:64] = sub.T                             # subnormals next to normal values
    x = torch.tensor(bits.astype(np.int32), dtype=torch.int32).to(torch.int16).view(torch.bfloat16).cuda()
    gofs = np.array([0, rows])
    res = ops.mxfp8_gather_quantize(x, _dev(gofs, torch.int32), 1, rows)
    torch.cuda.synchronize()
    P = to_np(x).astype(np.float64)
    assert np.count_nonzero((P != 0) & (np.abs(P) < 2.0 ** -126)) > 2000
    _check_axes(ops, P, gofs, rows, cols, res)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_single_axis(ops, rowwise, colwise):
    idx, w, slot_of, row_id, gofs = _routing(400, 8, 2, seed=21)
    rows = ops.moe_row_capacity(400, 8, 2)
    rid = np.full(rows, -1, dtype=np.int64)
    rid[:len(row_id)] = row_id
    x = _varied(400, 256, seed=22)
    res = ops.mxfp8_gather_quantize(x, _dev(gofs, torch.int32), 8, rows, row_id=_dev(rid, torch.int32), k=2,
                                    rowwise=rowwise, colwise=colwise)
    torch.cuda.synchronize()
    assert (res[0] is None) != rowwise and (res[2] is None) != colwise
    _check_axes(ops, O.permute(to_np(x), row_id, 2), gofs, rows, 256, res)


def test_rejects_bad_offsets(ops):
    x = _varied(256, 128, seed=9)
    cr = torch.full((256, 128), 0xAB, dtype=torch.uint8, device="cuda")
    sr = torch.full((256 * 4,), 0xCD, dtype=torch.uint8, device="cuda")
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384], [64, 128, 256]):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.mxfp8_gather_quantize(x, _dev(np.array(bad), torch.int32), 2, 256, colwise=False, codes_row=cr,
                                  scales_row=sr, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == ops.MOE_ERR_BAD_OFFSETS
        assert torch.all(cr == 0xAB) and torch.all(sr == 0xCD)


def test_host_argument_checks(ops):
    x = _varied(256, 128, seed=1)
    gofs = _dev(np.array([0, 256]), torch.int32)
    with pytest.raises(ops.MoEError):          # rows not a multiple of 128
        ops.mxfp8_gather_quantize(x, gofs, 1, 200)
    with pytest.raises(ops.MoEError):          # row_w without row_id
        ops.mxfp8_gather_quantize(x, gofs, 1, 256, row_w=torch.ones(256, device="cuda"))
    with pytest.raises(ops.MoEError):          # no output at all
        ops.mxfp8_gather_quantize(x, gofs, 1, 256, rowwise=False, colwise=False)


def test_row_id_beyond_src_is_reported(ops):
    """A row_id naming a token past src's rows is an error in *err; that row
    reads as zero and every other row is unaffected."""
    T, E, k, d = 100, 4, 2, 128
    idx, w, slot_of, row_id, gofs = _routing(T, E, k, seed=31)
    rows = ops.moe_row_capacity(T, E, k)
    rid = np.full(rows, -1, dtype=np.int64)
    rid[:len(row_id)] = row_id
    bad = int(slot_of[7, 1])
    rid[bad] = T * k + 3
    x = _varied(T, d, seed=32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = ops.mxfp8_gather_quantize(x, _dev(gofs, torch.int32), E, rows, row_id=_dev(rid, torch.int32), k=k,
                                    colwise=False, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ops.MOE_ERR_INVALID_ARG
    ref_rid = row_id.copy()
    ref_rid[bad] = -1
    _check_axes(ops, O.permute(to_np(x), ref_rid, k), gofs, rows, d, res)


@pytest.mark.parametrize("sizes,f", [([128], 128), ([5, 0, 130, 127, 1], 256), ([1000, 0, 300], 2048)])
def test_swiglu_bwd_quantize(ops, sizes, f):
    """dA = SwiGLU-backward(a_pre, dH) in bf16 against the oracle, its codes
    on both axes bit-exact against the oracle's quantization of that bf16
    dA; the same codes without dA written; rows beyond the groups neither
    read (NaN there) nor written."""
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    rows = Rp + 256
    g = torch.Generator(device="cuda")
    g.manual_seed(f + len(sizes))
    dH = torch.randn((rows, f), generator=g, device="cuda") * 3.0
    a_pre = (torch.randn((rows, 2 * f), generator=g, device="cuda") * 2.0).to(torch.bfloat16)
    dH[Rp:] = float("nan")
    a_pre[Rp:] = float("nan")
    gt = _dev(gofs, torch.int32)
    cr = torch.full((rows, 2 * f), 0xAB, dtype=torch.uint8, device="cuda")
    cc = torch.full((2 * f, rows), 0xAB, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dA, cr, sr, cc, sc = ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, gt, len(sizes), want_dA=True, codes_row=cr,
                                                       codes_col=cc, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.swiglu_bwd(to_np(a_pre[:Rp]), dH[:Rp].double().cpu().numpy())
    assert_bf16_close(dA[:Rp], ref, what="dA")
    _check_axes(ops, to_np(dA[:Rp]), gofs, rows, 2 * f, (cr, sr, cc, sc))
    assert torch.all(cr[Rp:] == 0xAB) and torch.all(cc[:, Rp:] == 0xAB)
    _, cr2, sr2, cc2, sc2 = ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, gt, len(sizes))
    torch.cuda.synchronize()
    assert torch.equal(cr2[:Rp], cr[:Rp]) and torch.equal(cc2[:, :Rp], cc[:, :Rp])
    assert np.array_equal(atoms_rows_subset(sr2.cpu().numpy(), rows, 2 * f, np.arange(Rp)),
                          atoms_rows_subset(sr.cpu().numpy(), rows, 2 * f, np.arange(Rp)))
    assert np.array_equal(atoms_to_rowmajor(sc2.cpu().numpy(), 2 * f, rows)[:, :Rp // 32],
                          atoms_to_rowmajor(sc.cpu().numpy(), 2 * f, rows)[:, :Rp // 32])


def test_swiglu_bwd_quantize_rejects_bad_offsets(ops):
    f, rows = 128, 256
    dH = torch.zeros((rows, f), device="cuda")
    a_pre = torch.zeros((rows, 2 * f), dtype=torch.bfloat16, device="cuda")
    cr = torch.full((rows, 2 * f), 0xAB, dtype=torch.uint8, device="cuda")
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384], [64, 128, 256]):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, _dev(np.array(bad), torch.int32), 2, codes_row=cr, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == ops.MOE_ERR_BAD_OFFSETS
        assert torch.all(cr == 0xAB)



@pytest.mark.parametrize("d", [128, 384, 896, 7168])
def test_gather_scaled_tile224_scales(ops, d):
    """The columnwise scales in the tile-224 layout (the weight gradients'
    right operand): the same bytes as the atom layout's, moved to the
    224-row tiles (ragged last tile for d = 128, 384), bit-exact against
    the oracle; codes unchanged; the bytes past the matrix's rows untouched."""
    from helpers import tile224_to_rowmajor
    T, E, k = 600, 8, 2
    idx, w, slot_of, row_id, gofs = _routing(T, E, k, 5, 0.5)
    Rp = int(gofs[-1])
    rows = Rp + 128
    x = _varied(T, d, 7)
    rid = np.full(rows, -1, dtype=np.int32)
    rid[:Rp] = row_id
    gt, rt, wt = _dev(gofs, torch.int32), _dev(rid, torch.int32), _dev(w, torch.float32)
    ref = ops.mxfp8_gather_quantize(x, gt, E, rows, rt, k, wt, True, True)
    nsc = ops.sf_bytes_tile224(d, rows)
    sc224 = torch.full((nsc,), 0xCD, dtype=torch.uint8, device="cuda")
    res = ops.mxfp8_gather_quantize(x, gt, E, rows, rt, k, wt, True, True, scales_col=sc224,
                                    col_sf_layout=ops.MOE_SF_TILE224)
    torch.cuda.synchronize()
    assert torch.equal(res[2][:, :Rp], ref[2][:, :Rp]) and torch.equal(res[0][:Rp], ref[0][:Rp])
    got = tile224_to_rowmajor(sc224.cpu().numpy(), d, rows)[:, :Rp // 32]
    assert np.array_equal(got, atoms_to_rowmajor(ref[3].cpu().numpy(), d, rows)[:, :Rp // 32])
    P = O.permute_scaled_bf16(to_np(x), row_id, k, w.astype(np.float64))
    _, cs, _ = O.mxfp8_quantize_cols_grouped(P, gofs)
    assert np.array_equal(got, cs)
    if d % 224:                  # rows of the last tile past d: never written
        T224 = (d + 223) // 224
        t = d // 224
        rp = np.arange(d - 224 * t, 224)
        off = (np.arange(Rp // 128)[:, None] * T224 + t) * 1024 + ((rp // 128) * 512 + (rp % 32) * 16 +
                                                                   ((rp // 32) % 4) * 4)[None, :]
        assert np.all(sc224.cpu().numpy()[off] == 0xCD)


def test_swiglu_bwd_tile224_scales(ops):
    """mxfp8_swiglu_bwd_quantize with the tile-224 columnwise scales: the
    atom layout's bytes, moved (2f = 512: a ragged last tile)."""
    from helpers import tile224_to_rowmajor
    sizes, f = [300, 0, 129], 256
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    rows = Rp + 128
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    dH = torch.randn((rows, f), generator=g, device="cuda")
    a_pre = torch.randn((rows, 2 * f), generator=g, device="cuda").to(torch.bfloat16)
    gt = _dev(gofs, torch.int32)
    _, cr, sr, cc, sc = ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, gt, len(sizes))
    _, cr2, sr2, cc2, sc2 = ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, gt, len(sizes),
                                                          col_sf_layout=ops.MOE_SF_TILE224)
    torch.cuda.synchronize()
    assert sc2.numel() == ops.sf_bytes_tile224(2 * f, rows)
    assert torch.equal(cc2[:, :Rp], cc[:, :Rp]) and torch.equal(cr2[:Rp], cr[:Rp])
    assert np.array_equal(tile224_to_rowmajor(sc2.cpu().numpy(), 2 * f, rows)[:, :Rp // 32],
                          atoms_to_rowmajor(sc.cpu().numpy(), 2 * f, rows)[:, :Rp // 32])


@pytest.mark.parametrize("d", [384, 7168])
def test_gather_scaled_both_scale_layouts(ops, d):
    """MOE_SF_TILE224_AND_ATOMS: the tile-224 bytes, then the atom layout,
    each bit-exact as the single-layout calls write them (same fill for the
    bytes neither writes); codes unchanged."""
    T, E, k = 600, 8, 2
    idx, w, slot_of, row_id, gofs = _routing(T, E, k, 5, 0.5)
    Rp = int(gofs[-1])
    rows = Rp + 128
    x = _varied(T, d, 11)
    rid = np.full(rows, -1, dtype=np.int32)
    rid[:Rp] = row_id
    gt, rt, wt = _dev(gofs, torch.int32), _dev(rid, torch.int32), _dev(w, torch.float32)
    n224, nat = ops.sf_bytes_tile224(d, rows), ops.sf_bytes(rows, d)
    assert ops.col_sf_bytes(ops.MOE_SF_TILE224_AND_ATOMS, rows, d) == n224 + nat

    def run(layout, n):
        sc = torch.full((n,), 0xCD, dtype=torch.uint8, device="cuda")
        r = ops.mxfp8_gather_quantize(x, gt, E, rows, rt, k, wt, True, True, scales_col=sc, col_sf_layout=layout)
        return r[0], r[2], sc

    q_at, qc_at, sc_at = run(ops.MOE_SF_ATOMS, nat)
    q_224, qc_224, sc_224 = run(ops.MOE_SF_TILE224, n224)
    q_b, qc_b, sc_b = run(ops.MOE_SF_TILE224_AND_ATOMS, n224 + nat)
    torch.cuda.synchronize()
    assert torch.equal(q_b[:Rp], q_at[:Rp]) and torch.equal(qc_b[:, :Rp], qc_at[:, :Rp])
    assert torch.equal(sc_b[:n224], sc_224)
    assert torch.equal(sc_b[n224:], sc_at)
    P = O.permute_scaled_bf16(to_np(x), row_id, k, w.astype(np.float64))
    _, cs, _ = O.mxfp8_quantize_cols_grouped(P, gofs)
    assert np.array_equal(atoms_to_rowmajor(sc_b[n224:].cpu().numpy(), d, rows)[:, :Rp // 32], cs)


def test_swiglu_bwd_both_scale_layouts(ops):
    """mxfp8_swiglu_bwd_quantize with MOE_SF_TILE224_AND_ATOMS: the
    tile-224 bytes, then the atom layout, as the single-layout calls write
    them."""
    sizes, f = [300, 0, 129, 700], 384
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    rows = Rp + 128
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    dH = torch.randn((rows, f), generator=g, device="cuda")
    a_pre = torch.randn((rows, 2 * f), generator=g, device="cuda").to(torch.bfloat16)
    gt = _dev(gofs, torch.int32)
    n224, nat = ops.sf_bytes_tile224(2 * f, rows), ops.sf_bytes(rows, 2 * f)

    def run(layout, n):
        sc = torch.full((n,), 0xCD, dtype=torch.uint8, device="cuda")
        _, cr, _, cc, _ = ops.mxfp8_swiglu_bwd_quantize(dH, a_pre, gt, len(sizes), scales_col=sc,
                                                        col_sf_layout=layout)
        return cr, cc, sc

    cr_at, cc_at, sc_at = run(ops.MOE_SF_ATOMS, nat)
    _, _, sc_224 = run(ops.MOE_SF_TILE224, n224)
    cr_b, cc_b, sc_b = run(ops.MOE_SF_TILE224_AND_ATOMS, n224 + nat)
    torch.cuda.synchronize()
    assert torch.equal(cr_b[:Rp], cr_at[:Rp]) and torch.equal(cc_b[:, :Rp], cc_at[:, :Rp])
    assert torch.equal(sc_b[:n224], sc_224)
    assert torch.equal(sc_b[n224:], sc_at)
