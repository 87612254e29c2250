"""MXFP8 quantization kernels vs the oracle: bit-exact codes and scales."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import atoms_to_rowmajor, atoms_rows_subset, glu_perm, gpu_ops, padded_layout, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _varied(rows, cols, seed):
    """bf16 values whose 32-blocks span many binades, with zero blocks,
    negative zeros and tiny values."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, device="cuda")
    blk_scale = torch.exp2(torch.randint(-40, 40, (rows, cols // 32), generator=g, device="cuda").float())
    x = x * blk_scale.repeat_interleave(32, dim=1)
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, 32:64] *= 1e-36
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 512), (384, 7168)])
def test_rowwise_bit_exact(ops, rows, cols):
    x = _varied(rows, cols, seed=rows + cols)
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE)
    torch.cuda.synchronize()
    rq, rs = O.mxfp8_quantize_rows(to_np(x))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(atoms_to_rowmajor(s.cpu().numpy(), rows, cols), rs)


def test_rowwise_every_bf16_value_at_unit_scale(ops):
    """Every bf16 with |v| <= 448, in blocks whose max is 448 (scale 2^0): the
    codes are the E4M3 round-to-nearest-even of each value."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    v = bits[torch.isfinite(bits) & (bits.abs() <= 448)]
    n = v.numel()
    per = 31
    nblk = (n + per - 1) // per
    blocks = torch.zeros((nblk, 32))
    blocks[:, 0] = 448.0
    flat = torch.zeros(nblk * per)
    flat[:n] = v
    blocks[:, 1:] = flat.view(nblk, per)
    rows = ((nblk * 32 + 127) // 128 + 127) // 128 * 128
    x = torch.zeros(rows * 128)
    x[:nblk * 32] = blocks.reshape(-1)
    x = x.view(rows, 128).to(torch.bfloat16).cuda()
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE)
    torch.cuda.synchronize()
    rq, rs = O.mxfp8_quantize_rows(to_np(x))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(atoms_to_rowmajor(s.cpu().numpy(), rows, 128), rs)


def test_rowwise_skips_rows_beyond_groups(ops):
    x = _varied(512, 256, seed=3)
    gofs = torch.tensor([0, 128, 256], dtype=torch.int32, device="cuda")
    q = torch.full((512, 256), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((512 * 8,), 0xCD, dtype=torch.uint8, device="cuda")
    ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE, gofs, 2, q, s)
    torch.cuda.synchronize()
    rq, rs = O.mxfp8_quantize_rows(to_np(x)[:256])
    assert np.array_equal(q[:256].cpu().numpy(), rq)
    assert torch.all(q[256:] == 0xAB)
    assert np.array_equal(atoms_rows_subset(s.cpu().numpy(), 512, 256, np.arange(256)), rs)
    assert np.all(atoms_rows_subset(s.cpu().numpy(), 512, 256, np.arange(256, 512)) == 0xCD)


@pytest.mark.parametrize("sizes,cols", [([128], 128), ([5, 0, 130, 127, 1], 256), ([1000, 0, 300], 7168)])
def test_colwise_grouped_bit_exact(ops, sizes, cols):
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    rows = Rp + 256                                   # rows beyond the groups are not read
    x = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    src = _varied(max(128, (sum(sizes) + 127) // 128 * 128), cols, seed=7)
    r = 0
    for g, m in enumerate(sizes):
        x[gofs[g]:gofs[g] + m] = src[r:r + m]
        r += m
    x[Rp:] = float("nan")                              # must not be read
    gt = torch.tensor(gofs, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_COLWISE_GROUPED, gt, len(sizes), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle on the unpadded rows with the unpadded offsets: blocks restart at
    # every group start, tails are zero padded
    raw_offs = np.concatenate([[0], np.cumsum(sizes)])
    xr = np.concatenate([to_np(x)[gofs[g]:gofs[g] + m] for g, m in enumerate(sizes)])
    rq, rs, padded = O.mxfp8_quantize_cols_grouped(xr, raw_offs)
    # the oracle pads each group to 32, the GPU layout to 128: compare block by block
    qn = q.cpu().numpy()
    sn = atoms_to_rowmajor(s.cpu().numpy(), cols, rows)
    for g, m in enumerate(sizes):
        nb = (m + 31) // 32
        assert np.array_equal(qn[:, gofs[g]:gofs[g] + 32 * nb], rq[:, padded[g]:padded[g] + 32 * nb])
        assert np.array_equal(sn[:, gofs[g] // 32:gofs[g] // 32 + nb], rs[:, padded[g] // 32:padded[g] // 32 + nb])
        # whole padding blocks after the tail block are zero codes, scale byte 0
        assert np.all(qn[:, gofs[g] + 32 * nb:gofs[g + 1]] == 0)
        assert np.all(sn[:, gofs[g] // 32 + nb:gofs[g + 1] // 32] == 0)


def test_colwise_rejects_bad_offsets(ops):
    x = _varied(256, 128, seed=9)
    q = torch.full((128, 256), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((256 * 4,), 0xCD, dtype=torch.uint8, device="cuda")
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384], [64, 128, 256]):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.mxfp8_group_quantize(x, ops.MOE_QUANT_COLWISE_GROUPED,
                                 torch.tensor(bad, dtype=torch.int32, device="cuda"), 2, q, s, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == ops.MOE_ERR_BAD_OFFSETS
        assert torch.all(q == 0xAB) and torch.all(s == 0xCD)


@pytest.mark.parametrize("G,K,N", [(1, 128, 256), (4, 256, 512), (3, 128, 1152)])
def test_colwise_glu_interleaved_rows(ops, G, K, N):
    """The gate/up-interleaved columnwise layout is the plain columnwise
    quantization with output rows permuted (moe.h MOE_QUANT_COLWISE_GLU)."""
    x = _varied(G * K, N, seed=G + K)
    gofs = torch.arange(0, (G + 1) * K, K, dtype=torch.int32, device="cuda")
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_COLWISE_GLU, gofs, G)
    torch.cuda.synchronize()
    rq, rs, _ = O.mxfp8_quantize_cols_grouped(to_np(x), np.arange(0, (G + 1) * K, K))
    perm = glu_perm(N)
    assert np.array_equal(q.cpu().numpy(), rq[perm])
    assert np.array_equal(atoms_to_rowmajor(s.cpu().numpy(), N, G * K), rs[perm])


@pytest.mark.parametrize("G,K,N,glu", [(1, 128, 256, False), (4, 256, 512, True), (3, 384, 1152, False),
                                       (2, 128, 384, True)])
def test_colwise_batched_per_group_blocks(ops, G, K, N, glu):
    """Batched layout: group g's transposed block is contiguous, codes
    [G][N][K], scales in the atom layout of [G*N, K] (moe.h)."""
    x = _varied(G * K, N, seed=G * 7 + K)
    axis = ops.MOE_QUANT_COLWISE_BATCHED_GLU if glu else ops.MOE_QUANT_COLWISE_BATCHED
    q, s = ops.mxfp8_group_quantize(x, axis, None, G)
    torch.cuda.synchronize()
    assert tuple(q.shape) == (G, N, K)
    xn = to_np(x)
    qn = q.cpu().numpy()
    sn = atoms_to_rowmajor(s.cpu().numpy(), G * N, K).reshape(G, N, K // 32)
    perm = glu_perm(N) if glu else np.arange(N)
    for g in range(G):
        rq, rs, _ = O.mxfp8_quantize_cols_grouped(xn[g * K:(g + 1) * K], np.array([0, K]))
        assert np.array_equal(qn[g], rq[perm]) and np.array_equal(sn[g], rs[perm])


def test_ex_canonical_scales_and_padded_offsets(ops):
    """mxfp8_group_quantize_ex: the canonical row-major scales are the atom
    scales in row order (and the oracle's), the codes are unchanged, and the
    padded offsets of the grouped axes are the group offsets."""
    sizes, cols = [5, 0, 130, 127, 1], 256
    gofs = padded_layout(sizes)
    Rp = int(gofs[-1])
    x = torch.zeros((Rp, cols), dtype=torch.bfloat16, device="cuda")
    src = _varied(Rp, cols, seed=21)
    for g, m in enumerate(sizes):
        x[gofs[g]:gofs[g] + m] = src[gofs[g]:gofs[g] + m]
    gt = torch.tensor(gofs, dtype=torch.int32, device="cuda")
    G = len(sizes)
    for axis in (ops.MOE_QUANT_ROWWISE, ops.MOE_QUANT_COLWISE_GROUPED, ops.MOE_QUANT_COLWISE_GLU):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_at, s_at = ops.mxfp8_group_quantize(x, axis, gt, G, err=err)
        q_ca, s_ca, po = ops.mxfp8_group_quantize_ex(x, axis, gt, G, ops.MOE_SF_CANONICAL, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(q_at, q_ca)
        assert np.array_equal(po.cpu().numpy(), gofs)
        R, C = (Rp, cols) if axis == ops.MOE_QUANT_ROWWISE else (cols, Rp)
        assert np.array_equal(s_ca.cpu().numpy().reshape(R, C // 32), atoms_to_rowmajor(s_at.cpu().numpy(), R, C))
    _, rs = O.mxfp8_quantize_rows(to_np(x))
    _, s_ca, _ = ops.mxfp8_group_quantize_ex(x, ops.MOE_QUANT_ROWWISE, gt, G, ops.MOE_SF_CANONICAL)
    torch.cuda.synchronize()
    assert np.array_equal(s_ca.cpu().numpy().reshape(Rp, cols // 32), rs)


@pytest.mark.parametrize("glu", [False, True])
def test_ex_batched_canonical_and_offsets(ops, glu):
    G, K, N = 3, 256, 384
    x = _varied(G * K, N, seed=31)
    axis = ops.MOE_QUANT_COLWISE_BATCHED_GLU if glu else ops.MOE_QUANT_COLWISE_BATCHED
    q_at, s_at = ops.mxfp8_group_quantize(x, axis, None, G)
    q_ca, s_ca, po = ops.mxfp8_group_quantize_ex(x, axis, None, G, ops.MOE_SF_CANONICAL)
    torch.cuda.synchronize()
    assert torch.equal(q_at, q_ca)
    assert np.array_equal(po.cpu().numpy(), np.arange(0, (G + 1) * K, K))
    assert np.array_equal(s_ca.cpu().numpy().reshape(G * N, K // 32),
                          atoms_to_rowmajor(s_at.cpu().numpy(), G * N, K))
