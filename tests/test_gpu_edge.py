"""Degenerate inputs on the GPU: no tokens, every group empty, one token
choosing every expert."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import gpu_ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def test_zero_tokens(ops):
    """T = 0: routing gives all-zero counts and offsets, the permute all-zero
    group offsets, and the combine and router backward do nothing."""
    E, k, d = 8, 2, 256
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty((0, E), dtype=torch.float32, device="cuda")
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    idx, w, counts, offsets = ops.moe_route_topk(logits, k, counts=counts, offsets=offsets, err=err)
    gofs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    gofs, slot_of, row_id, _ = ops.moe_permute(None, idx, E, gofs=gofs, want_x_perm=False, err=err)
    out = ops.moe_unpermute_combine(torch.empty((0, d), dtype=torch.bfloat16, device="cuda"), slot_of, w, err=err)
    dl = torch.empty((0, E), dtype=torch.float32, device="cuda")
    ops.moe_route_bwd(logits, idx, torch.empty((0, k), dtype=torch.float32, device="cuda"), 0, True, dl, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.all(counts == 0) and torch.all(offsets == 0) and torch.all(gofs == 0)
    assert out.shape == (0, d)


def test_every_group_empty(ops):
    """Group offsets all zero: the forward GEMM writes nothing, the weight
    gradient is the empty sum (zero) for every group, and the two-axis
    quantization writes nothing."""
    G, M, N, K = 4, 256, 256, 128
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gofs = torch.zeros(G + 1, dtype=torch.int32, device="cuda")
    a = torch.zeros((128, K), dtype=torch.uint8, device="cuda")
    a_s = torch.zeros((128 * K // 32,), dtype=torch.uint8, device="cuda")
    b = torch.zeros((G, N, K), dtype=torch.uint8, device="cuda")
    b_s = torch.zeros((G * N * K // 32,), dtype=torch.uint8, device="cuda")
    d = torch.full((128, N), 3.0, dtype=torch.bfloat16, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, a, a_s, b, b_s, ops.MOE_B_GNK, gofs, G, 128, N, K, d=d, err=err)
    # WGRAD: A [M, rows] and B [N, rows] columnwise codes with rows = K (no rows in any group)
    at = torch.full((M, K), 0x38, dtype=torch.uint8, device="cuda")
    at_s = torch.full((M * K // 32,), 127, dtype=torch.uint8, device="cuda")
    bt = torch.full((N, K), 0x38, dtype=torch.uint8, device="cuda")
    bt_s = torch.full((N * K // 32,), 127, dtype=torch.uint8, device="cuda")
    dw = torch.full((G, M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, at, at_s, bt, bt_s, ops.MOE_B_GNK, gofs, G, M, N, K, d=dw, err=err)
    x = torch.ones((128, 256), dtype=torch.bfloat16, device="cuda")
    cr = torch.full((128, 256), 0xAB, dtype=torch.uint8, device="cuda")
    cc = torch.full((256, 128), 0xAB, dtype=torch.uint8, device="cuda")
    sr = torch.full((128 * 8,), 0xCD, dtype=torch.uint8, device="cuda")
    sc = torch.full((128 * 8,), 0xCD, dtype=torch.uint8, device="cuda")
    ops.mxfp8_gather_quantize(x, gofs, G, 128, codes_row=cr, scales_row=sr, codes_col=cc, scales_col=sc, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.all(d == 3.0)
    assert torch.all(dw == 0)
    assert torch.all(cr == 0xAB) and torch.all(cc == 0xAB) and torch.all(sr == 0xCD) and torch.all(sc == 0xCD)


@pytest.mark.parametrize("E", [1, 8, 32])
def test_one_token_chooses_every_expert(ops, E):
    """T = 1, k = E: every group holds exactly the one token (padded to 128
    rows), in expert order."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.randn((1, E), device="cuda")
    idx, w, counts, _ = ops.moe_route_topk(logits, E, ops.MOE_SCORE_SOFTMAX, True, err=err)
    gofs, slot_of, row_id, _ = ops.moe_permute(None, idx, E, want_x_perm=False, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ridx, rw = O.route_topk(logits.cpu().numpy(), E, "softmax", True)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert torch.all(counts == 1)
    assert np.array_equal(gofs.cpu().numpy(), np.arange(0, 128 * (E + 1), 128))
    r_slot, r_row = O.permute_slots(ridx, E, 128)
    assert np.array_equal(slot_of.cpu().numpy(), r_slot)
    assert np.array_equal(row_id.cpu().numpy()[:128 * E], r_row[:128 * E])
    assert abs(float(w.sum()) - 1.0) < 1e-6
