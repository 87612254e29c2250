"""Grouped MXFP8 GEMM (tcgen05) vs the fp64 oracle on the GPU's own
dequantized operands: fwd, dgrad (both weight layouts), wgrad, SwiGLU and
SwiGLU-backward epilogues, empty groups, padding rows, several tiles.  The
whole file runs once per kernel: the library's own choice ("auto"), the
1-SM kernel with 256- and 128-wide tiles, and the CTA-pair kernel with
256- and 128-wide tiles (chosen per call through moe_gemm_opts_t)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (KernelOps, assert_bf16_close, assert_fp32_close, atoms_rows_subset, atoms_to_rowmajor,
                     batched_weight_operand, glu_perm, gpu_ops, padded_layout, to_np)
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["auto", "1sm", "1sm_n128", "pair", "pair_n128"])
def ops(request):
    return KernelOps(gpu_ops(), request.param)


def _act(sizes, K, seed, row_cap=None):
    """Permuted-layout activations: group g holds sizes[g] random rows then
    zero padding up to a multiple of 128."""
    gofs = padded_layout(sizes)
    M = row_cap or int(gofs[-1]) + 128
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    src = synth.make_normal_bf16((int(sum(sizes)) + 1, K), seed, "cuda")
    r = 0
    for g, m in enumerate(sizes):
        x[gofs[g]:gofs[g] + m] = src[r:r + m]
        r += m
    return x, torch.tensor(gofs, dtype=torch.int32, device="cuda"), gofs


def _quant_rows(ops, x, gofs_t=None, G=0):
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE, gofs_t, G)
    rows, cols = x.shape
    codes = q.cpu().numpy()
    sc = atoms_to_rowmajor(s.cpu().numpy(), rows, cols)
    return q, s, O.mxfp8_dequantize_rows(codes, sc)


def _weights(ops, G, K, N, seed, layout, glu=False):
    """bf16 weights W [G, K, N]; returns the device operand (codes, scales)
    and the oracle's dequantized B [G, K, N] from those codes (in logical
    column order also for the gate/up-interleaved layout)."""
    W = synth.make_normal_bf16((G, K, N), seed, "cuda", std=0.5)
    Wv = W.reshape(G * K, N)
    if layout == ops.MOE_B_NGK:
        gofs = torch.arange(0, (G + 1) * K, K, dtype=torch.int32, device="cuda")
        axis = ops.MOE_QUANT_COLWISE_GLU if glu else ops.MOE_QUANT_COLWISE_GROUPED
        q, s = ops.mxfp8_group_quantize(Wv, axis, gofs, G)
        qn = q.cpu().numpy()                          # [N, G*K]
        sn = atoms_to_rowmajor(s.cpu().numpy(), N, G * K)
        perm = glu_perm(N) if glu else np.arange(N)
        # codes bit-exact against the oracle's group-aware columnwise quantizer
        rq, rs, _ = O.mxfp8_quantize_cols_grouped(to_np(Wv), np.arange(0, (G + 1) * K, K))
        assert np.array_equal(qn, rq[perm]) and np.array_equal(sn, rs[perm])
        deq = np.empty((N, G * K))
        deq[perm] = O.mxfp8_dequantize_rows(qn, sn)   # back to logical column order
        B = deq.T.reshape(G, K, N)
        return q, s, B
    # GNK from the [G][K][N] weight: per-group transposed blocks (batched)
    axis = ops.MOE_QUANT_COLWISE_BATCHED_GLU if glu else ops.MOE_QUANT_COLWISE_BATCHED
    q, s = ops.mxfp8_group_quantize(Wv, axis, None, G)
    B = batched_weight_operand(q.cpu().numpy(), s.cpu().numpy(), G, N, K, glu)
    return q, s, B


@pytest.mark.parametrize("sizes,K,N", [
    ([128], 128, 256),                    # one tile, one k-step
    ([300], 512, 256),                    # ragged rows, several k-steps
    ([128, 0, 256, 384], 512, 512),       # empty group, several m/n tiles
    ([5, 0, 130, 127, 1, 0], 256, 768),   # tiny groups, padding rows
    ([1000, 24], 1024, 1024),
    ([200, 90], 384, 384),                # N not a multiple of 256
])
def test_fwd_ngk(ops, sizes, K, N):
    G = len(sizes)
    x, gofs_t, gofs = _act(sizes, K, seed=11)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    bq, bs, B = _weights(ops, G, K, N, seed=12, layout=ops.MOE_B_NGK)
    d = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_NGK, gofs_t, G, M, N, K, d=d, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.grouped_gemm(A, B, gofs)
    Rp = int(gofs[-1])
    assert_bf16_close(d[:Rp], ref[:Rp], what="fwd")
    assert torch.all(d[Rp:] == 7.0)                        # rows outside every group untouched
    # padding rows of the activations are zero, so their outputs are zero
    for g, m in enumerate(sizes):
        assert torch.all(d[gofs[g] + m:gofs[g + 1]] == 0)


def test_fwd_max_groups(ops):
    """1024 groups (the largest G the kernels take), most of them empty or a
    few rows: the group offsets all fit the kernel's shared copy and every
    tile finds its group; G = 1025 is refused on the host."""
    rng = np.random.default_rng(5)
    G, K, N = 1024, 128, 256
    sizes = np.where(rng.random(G) < 0.7, 0, rng.integers(1, 40, G)).tolist()
    x, gofs_t, gofs = _act(sizes, K, seed=31)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    bq, bs, B = _weights(ops, G, K, N, seed=32, layout=ops.MOE_B_GNK)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_GNK, gofs_t, G, M, N, K, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    Rp = int(gofs[-1])
    assert_bf16_close(d[:Rp], O.grouped_gemm(A, B, gofs)[:Rp], what="fwd, 1024 groups")
    gofs2 = torch.cat([gofs_t, gofs_t[-1:]])
    with pytest.raises(ops.MoEError):
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_GNK, gofs2, G + 1, M, N, K, err=err)


@pytest.mark.parametrize("sizes,K,N", [([300, 0, 5], 512, 256), ([1000, 24], 1024, 768)])
def test_fwd_gnk_batched_weights(ops, sizes, K, N):
    G = len(sizes)
    x, gofs_t, gofs = _act(sizes, K, seed=71)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    bq, bs, B = _weights(ops, G, K, N, seed=72, layout=ops.MOE_B_GNK)
    d = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_GNK, gofs_t, G, M, N, K)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    assert_bf16_close(d[:Rp], O.grouped_gemm(A, B, gofs)[:Rp], what="fwd gnk")


@pytest.mark.parametrize("sizes,K,N", [([200, 0, 77], 512, 256), ([128, 128], 256, 512)])
def test_dgrad_gnk(ops, sizes, K, N):
    """DGRAD reads the weight copy quantized along the other axis: B_g is the
    [N, K] slice of a [G*N, K] rowwise-quantized matrix."""
    G = len(sizes)
    x, gofs_t, gofs = _act(sizes, K, seed=21)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    # weight stored [G, N, K] (rows N, quantized along K)
    W = synth.make_normal_bf16((G * N, K), 22, "cuda", std=0.5)
    wq, ws_ = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
    Wd = O.mxfp8_dequantize_rows(wq.cpu().numpy(), atoms_to_rowmajor(ws_.cpu().numpy(), G * N, K))
    B = np.transpose(Wd.reshape(G, N, K), (0, 2, 1))      # [G, K, N]
    d = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_DGRAD, xq, xs, wq, ws_, ops.MOE_B_GNK, gofs_t, G, M, N, K)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    assert_bf16_close(d[:Rp], O.grouped_gemm(A, B, gofs)[:Rp], what="dgrad")


@pytest.mark.parametrize("layout", [0, 1])       # MOE_B_GNK (batched weight quantization), MOE_B_NGK
@pytest.mark.parametrize("sizes,K,f", [([150, 0, 300], 512, 256), ([77, 500], 256, 128), ([129], 1024, 384)])
def test_swiglu_epilogue(ops, sizes, K, f, layout):
    G, N = len(sizes), 2 * f
    x, gofs_t, gofs = _act(sizes, K, seed=31)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    bq, bs, B = _weights(ops, G, K, N, seed=32, layout=layout, glu=True)
    a_pre, h = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, layout, gofs_t, G, M, N, K,
                                      ops.MOE_EPI_SWIGLU)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    ref = O.grouped_gemm(A, B, gofs)[:Rp]
    assert_bf16_close(a_pre[:Rp], ref, what="a_pre")
    assert_bf16_close(h[:Rp], O.swiglu(ref), what="h")


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("sizes,K,f", [([150, 0, 300], 512, 256), ([77, 500], 256, 128), ([129, 3], 1024, 384)])
def test_swiglu_quant_epilogue(ops, sizes, K, f, layout):
    """h's MXFP8 codes from the SwiGLU epilogue: bit-exact against the
    oracle's rowwise and group-aware columnwise quantization of the GPU's own
    bf16 h; the same codes whether or not h is also written; rows beyond the
    groups untouched."""
    G, N = len(sizes), 2 * f
    x, gofs_t, gofs = _act(sizes, K, seed=51)
    M = x.shape[0]
    xq, xs, A = _quant_rows(ops, x)
    bq, bs, B = _weights(ops, G, K, N, seed=52, layout=layout, glu=True)
    Rp = int(gofs[-1])
    sent = dict(h_codes_row=torch.full((M, f), 0xAB, dtype=torch.uint8, device="cuda"),
                h_codes_col=torch.full((f, M), 0xAB, dtype=torch.uint8, device="cuda"))
    a_pre, h, cr, sr, cc, sc = ops.grouped_gemm_mxfp8_swiglu_quant(xq, xs, bq, bs, layout, gofs_t, G, M, N, K,
                                                                    want_h=True, **sent)
    torch.cuda.synchronize()
    ref = O.grouped_gemm(A, B, gofs)[:Rp]
    assert_bf16_close(a_pre[:Rp], ref, what="a_pre")
    assert_bf16_close(h[:Rp], O.swiglu(ref), what="h")
    hn = to_np(h)[:Rp]
    rq, rs = O.mxfp8_quantize_rows(hn)
    assert np.array_equal(cr[:Rp].cpu().numpy(), rq)
    assert np.array_equal(atoms_rows_subset(sr.cpu().numpy(), M, f, np.arange(Rp)), rs)
    cq, cs, padded = O.mxfp8_quantize_cols_grouped(hn, gofs)
    assert np.array_equal(padded, gofs)
    assert np.array_equal(cc[:, :Rp].cpu().numpy(), cq)
    assert np.array_equal(atoms_to_rowmajor(sc.cpu().numpy(), f, M)[:, :Rp // 32], cs)
    assert torch.all(cr[Rp:] == 0xAB) and torch.all(cc[:, Rp:] == 0xAB)
    # without h: identical codes and scales
    a2, h2, cr2, sr2, cc2, sc2 = ops.grouped_gemm_mxfp8_swiglu_quant(xq, xs, bq, bs, layout, gofs_t, G, M, N, K)
    torch.cuda.synchronize()
    assert h2 is None
    assert torch.equal(a2[:Rp], a_pre[:Rp]) and torch.equal(cr2[:Rp], cr[:Rp]) and torch.equal(cc2[:, :Rp], cc[:, :Rp])
    assert np.array_equal(atoms_rows_subset(sr2.cpu().numpy(), M, f, np.arange(Rp)), rs)
    assert np.array_equal(atoms_to_rowmajor(sc2.cpu().numpy(), f, M)[:, :Rp // 32], cs)


@pytest.mark.parametrize("sizes,K,f", [([140, 260], 512, 256), ([300, 0, 5], 256, 384)])
def test_swiglu_bwd_epilogue(ops, sizes, K, f):
    G, N = len(sizes), f
    dy, gofs_t, gofs = _act(sizes, K, seed=41)
    M = dy.shape[0]
    dq, ds, A = _quant_rows(ops, dy)
    W = synth.make_normal_bf16((G * N, K), 42, "cuda", std=0.5)
    wq, ws_ = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
    Wd = O.mxfp8_dequantize_rows(wq.cpu().numpy(), atoms_to_rowmajor(ws_.cpu().numpy(), G * N, K))
    B = np.transpose(Wd.reshape(G, N, K), (0, 2, 1))
    a_pre = synth.make_normal_bf16((M, 2 * f), 43, "cuda", std=2.0)
    dA = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_DGRAD, dq, ds, wq, ws_, ops.MOE_B_GNK, gofs_t, G, M, N, K,
                                ops.MOE_EPI_SWIGLU_BWD, epi_aux=a_pre)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    dH = O.grouped_gemm(A, B, gofs)[:Rp]
    ref = O.swiglu_bwd(to_np(a_pre)[:Rp], dH)
    assert_bf16_close(dA[:Rp], ref, what="dA")


@pytest.mark.parametrize("sizes,K,N", [([140, 260], 512, 256), ([300, 0, 5], 256, 384), ([129], 1024, 2048)])
def test_dgrad_fp32_out(ops, sizes, K, N):
    """MOE_EPI_NONE_F32: the fp32 accumulators as they are (dH for the fused
    SwiGLU backward); rows beyond the groups untouched."""
    G = len(sizes)
    dy, gofs_t, gofs = _act(sizes, K, seed=45)
    M = dy.shape[0]
    dq, ds, A = _quant_rows(ops, dy)
    W = synth.make_normal_bf16((G * N, K), 46, "cuda", std=0.5)
    wq, ws_ = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
    Wd = O.mxfp8_dequantize_rows(wq.cpu().numpy(), atoms_to_rowmajor(ws_.cpu().numpy(), G * N, K))
    B = np.transpose(Wd.reshape(G, N, K), (0, 2, 1))
    d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_DGRAD, dq, ds, wq, ws_, ops.MOE_B_GNK, gofs_t, G, M, N, K,
                           ops.MOE_EPI_NONE_F32, d=d)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    assert_fp32_close(d[:Rp], O.grouped_gemm(A, B, gofs)[:Rp], what="dH fp32")
    assert torch.isnan(d[Rp:]).all()


@pytest.mark.parametrize("sizes,Mo,No", [([128, 0, 384], 256, 256), ([5, 130, 0, 64], 128, 512),
                                         ([900], 384, 768)])
def test_wgrad(ops, sizes, Mo, No):
    """dB_g = A_g^T G_g over the group's rows; the operands are the
    columnwise (transposed) codes; an empty group gives zeros."""
    G = len(sizes)
    a, gofs_t, gofs = _act(sizes, Mo, seed=51)
    g_, _, _ = _act(sizes, No, seed=52, row_cap=a.shape[0])
    Kc = a.shape[0]
    aq, as_ = ops.mxfp8_group_quantize(a, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    gq, gs = ops.mxfp8_group_quantize(g_, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    torch.cuda.synchronize()
    Rp = int(gofs[-1])
    aq_n, gq_n = aq.cpu().numpy()[:, :Rp], gq.cpu().numpy()[:, :Rp]
    # atoms of the [Mo, Kc] / [No, Kc] matrices; keep the first Rp columns
    A_sc = atoms_to_rowmajor(as_.cpu().numpy(), Mo, Kc)[:, :Rp // 32]
    G_sc = atoms_to_rowmajor(gs.cpu().numpy(), No, Kc)[:, :Rp // 32]
    rq, rs, _ = O.mxfp8_quantize_cols_grouped(to_np(a)[:Rp], gofs)
    assert np.array_equal(aq_n, rq) and np.array_equal(A_sc, rs)
    Ah = O.mxfp8_dequantize_cols(aq_n, A_sc)       # [Rp, Mo]
    Gh = O.mxfp8_dequantize_cols(gq_n, G_sc)       # [Rp, No]
    d = torch.full((G, Mo, No), 3.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs, 0, gofs_t, G, Mo, No, Kc, d=d, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.grouped_gemm_wgrad(Ah, Gh, gofs)
    for g in range(G):
        if sizes[g] == 0:
            assert torch.all(d[g] == 0)
        else:
            assert_bf16_close(d[g], ref[g], what=f"wgrad g={g}")
    if ops.kernel == "pair":
        # the pair kernel's register-staged stores write the same bytes as its TMA stores
        d2 = torch.full((G, Mo, No), 3.0, dtype=torch.bfloat16, device="cuda")
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs, 0, gofs_t, G, Mo, No, Kc, d=d2, err=err,
                               opts=ops.gemm_opts("pair", register_stores=True))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(d2, d)


@pytest.mark.parametrize("sizes,Mo,No", [([128, 0, 384], 256, 256), ([5, 130, 0, 64], 256, 512),
                                         ([900, 31], 512, 896), ([300], 256, 384), ([0, 0], 256, 4096)])
def test_wgrad_tile224(ops, sizes, Mo, No):
    """The weight gradient with b's scales in the tile-224 layout: 256 x 224
    CTA-pair tiles with two accumulators, whatever kernel the options ask
    for.  No = 384 and 4096 end in a partial 224-column tile (its columns
    past No are neither computed into d nor written); empty groups give
    zeros.  The scale bytes are the GPU quantizer's, moved to the tile-224
    layout on the host."""
    from helpers import rowmajor_to_tile224
    G = len(sizes)
    a, gofs_t, gofs = _act(sizes, Mo, seed=81)
    g_, _, _ = _act(sizes, No, seed=82, row_cap=a.shape[0])
    Kc = a.shape[0]
    aq, as_ = ops.mxfp8_group_quantize(a, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    gq, gs = ops.mxfp8_group_quantize(g_, ops.MOE_QUANT_COLWISE_GROUPED, gofs_t, G)
    torch.cuda.synchronize()
    G_can = atoms_to_rowmajor(gs.cpu().numpy(), No, Kc)
    gs224 = torch.from_numpy(rowmajor_to_tile224(G_can)).cuda()
    Rp = int(gofs[-1])
    d = torch.full((G, Mo, No), 3.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, aq, as_, gq, gs224, ops.MOE_B_SF_TILE224, gofs_t, G, Mo, No, Kc, d=d,
                           err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if Rp:
        Ah = O.mxfp8_dequantize_cols(aq.cpu().numpy()[:, :Rp],
                                     atoms_to_rowmajor(as_.cpu().numpy(), Mo, Kc)[:, :Rp // 32])
        Gh = O.mxfp8_dequantize_cols(gq.cpu().numpy()[:, :Rp], G_can[:, :Rp // 32])
        ref = O.grouped_gemm_wgrad(Ah, Gh, gofs)
    for g in range(G):
        if sizes[g] == 0:
            assert torch.all(d[g] == 0)
        else:
            assert_bf16_close(d[g], ref[g], what=f"wgrad tile-224 g={g}")


def test_bad_offsets_reported_not_faulting(ops):
    sizes, K, N = [128, 128], 128, 256
    x, gofs_t, gofs = _act(sizes, K, seed=61)
    M = x.shape[0]
    xq, xs, _ = _quant_rows(ops, x)
    bq, bs, _ = _weights(ops, 2, K, N, seed=62, layout=ops.MOE_B_NGK)
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, M + 128]):
        d = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        g_bad = torch.tensor(bad, dtype=torch.int32, device="cuda")
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_NGK, g_bad, 2, M, N, K, d=d, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == ops.MOE_ERR_BAD_OFFSETS
        assert torch.all(d == 5.0)
